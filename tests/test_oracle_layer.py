"""Pins for the oracle's MoE layer and dense linear (CPU only).

  * brute force on tiny shapes: the oracle's per-token loop equals a dense
    numpy computation over fully dequantised weights (decoded here with an
    independent table + torch's e4m3 view), with no permutation involved;
  * special cases: E=1, k=1 equals the dense MLP bit-exactly; experts with
    all-zero codes contribute exactly zero; all-zero banks give out == 0;
  * invariants: permuting tokens permutes the outputs bit-exactly; doubling
    the up or the down weight_scale_2 doubles the output bit-exactly;
    W4A4 with x already on the NVFP4 grid gives the same h as W4A16;
    doubling a W4A4 input_scale (no block saturated or subnormal) keeps h.
"""
import numpy as np
import pytest
import torch

from oracle import calib
from serving_nvfp4_routed_gb300 import synth

E2M1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])


def _deq(codes, scales):
    c = np.asarray(codes)
    q = np.empty(c.shape[:-1] + (c.shape[-1] * 2,), np.uint8)
    q[..., 0::2] = c & 15
    q[..., 1::2] = c >> 4
    s = torch.from_numpy(np.ascontiguousarray(scales)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return E2M1[q] * np.repeat(s, 16, axis=-1)


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float64)).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()


def _f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _quant_bank(orc, banks):
    out = {}
    for name, w in banks.items():
        E = w.shape[0]
        res = [orc.quantize_tensor(synth.bf16_bits(w[e])) for e in range(E)]
        out[name] = (np.stack([r[0] for r in res]), np.stack([r[1] for r in res]),
                     np.array([r[2] for r in res], np.float32))
    return out


@pytest.fixture(scope="module")
def tiny(orc):
    s = synth.TINY
    inp = synth.moe_inputs(s, seed=1000)
    bank = _quant_bank(orc, dict(gate=inp["gate"], up=inp["up"], down=inp["down"]))
    xb = synth.bf16_bits(inp["x"])
    r = orc.route(inp["logits"].numpy(), s.k)
    return s, inp, bank, xb, r


def _brute(xf, ids, w, bank):
    """Dense per-token evaluation; no permutation, fp64 numpy matmuls."""
    T, d = xf.shape
    gq, gs, g2 = bank["gate"]
    uq, us, u2 = bank["up"]
    dq, ds, d2 = bank["down"]
    out = np.zeros((T, d))
    for t in range(T):
        acc = np.zeros(d)
        for j in range(ids.shape[1]):
            e = ids[t, j]
            G = _bf16(g2[e] * (_deq(gq[e], gs[e]) @ xf[t]))
            U = _bf16(u2[e] * (_deq(uq[e], us[e]) @ xf[t]))
            h = _bf16(G / (1 + np.exp(-G)) * U)
            acc += w[t, j] * (d2[e] * (_deq(dq[e], ds[e]) @ h))
        out[t] = _bf16(acc)
    return out


def test_tiny_layer_equals_brute_force(orc, tiny):
    s, inp, bank, xb, r = tiny
    out = orc.moe_layer("w4a16", xb, r["ids"], r["w"], bank)
    ref = _brute(_f32(xb).astype(np.float64), r["ids"], r["w"].astype(np.float64), bank)
    assert np.abs(ref).max() > 0
    same = np.mean(out == ref)
    assert same > 0.98, same
    np.testing.assert_allclose(out, ref, rtol=2 ** -7, atol=1e-6 * np.abs(ref).max())


def test_larger_shape_brute_force(orc):
    s = synth.MoEShape(T=5, d=128, E=3, k=2, F=64)
    inp = synth.moe_inputs(s, seed=77)
    bank = _quant_bank(orc, dict(gate=inp["gate"], up=inp["up"], down=inp["down"]))
    xb = synth.bf16_bits(inp["x"])
    r = orc.route(inp["logits"].numpy(), s.k)
    out = orc.moe_layer("w4a16", xb, r["ids"], r["w"], bank)
    ref = _brute(_f32(xb).astype(np.float64), r["ids"], r["w"].astype(np.float64), bank)
    np.testing.assert_allclose(out, ref, rtol=2 ** -7, atol=1e-6 * np.abs(ref).max())


def test_single_expert_equals_dense_mlp(orc):
    s = synth.MoEShape(T=6, d=128, E=1, k=1, F=64)
    inp = synth.moe_inputs(s, seed=5)
    bank = _quant_bank(orc, dict(gate=inp["gate"], up=inp["up"], down=inp["down"]))
    xb = synth.bf16_bits(inp["x"])
    r = orc.route(inp["logits"].numpy(), 1)
    assert np.all(r["w"] == 1.0)
    out = orc.moe_layer("w4a16", xb, r["ids"], r["w"], bank)
    g, u, dn = bank["gate"], bank["up"], bank["down"]
    h = orc.linear(xb, g[0][0], g[1][0], g[2][0], wup=(u[0][0], u[1][0], u[2][0]))
    hb = synth.bf16_bits(torch.from_numpy(h).to(torch.bfloat16))
    y = orc.linear(hb, dn[0][0], dn[1][0], dn[2][0])
    assert np.array_equal(out, y)


def test_zero_experts(orc, tiny):
    s, inp, bank, xb, r = tiny
    z = {k: (np.zeros_like(v[0]), v[1], v[2]) for k, v in bank.items()}
    assert not orc.moe_layer("w4a16", xb, r["ids"], r["w"], z).any()
    # zero only the down projection of expert e: tokens that route only elsewhere are unchanged
    e = int(r["ids"][0, 0])
    dq = bank["down"][0].copy()
    dq[e] = 0
    b2 = dict(bank, down=(dq, bank["down"][1], bank["down"][2]))
    out1 = orc.moe_layer("w4a16", xb, r["ids"], r["w"], bank)
    out2 = orc.moe_layer("w4a16", xb, r["ids"], r["w"], b2)
    for t in range(s.T):
        if e not in r["ids"][t]:
            assert np.array_equal(out1[t], out2[t])
    # token 0 with expert e removed = weighted sum of the other slot alone
    ids1 = r["ids"].copy()
    w1 = r["w"].copy()
    w1[0, 0] = 0.0
    out3 = orc.moe_layer("w4a16", xb, ids1, w1, bank)
    assert np.array_equal(out3[0], out2[0])


def test_token_permutation(orc, tiny):
    s, inp, bank, xb, r = tiny
    out = orc.moe_layer("w4a16", xb, r["ids"], r["w"], bank)
    p = np.array([2, 0, 3, 1])
    lg = inp["logits"].numpy()[p]
    r2 = orc.route(lg, s.k)
    out2 = orc.moe_layer("w4a16", xb[p], r2["ids"], r2["w"], bank)
    assert np.array_equal(out2, out[p])


def test_power_of_two_tensor_scales(orc, tiny):
    s, inp, bank, xb, r = tiny
    out = orc.moe_layer("w4a16", xb, r["ids"], r["w"], bank)
    b_up = dict(bank, up=(bank["up"][0], bank["up"][1], bank["up"][2] * 2))
    b_dn = dict(bank, down=(bank["down"][0], bank["down"][1], bank["down"][2] * 4))
    assert np.array_equal(orc.moe_layer("w4a16", xb, r["ids"], r["w"], b_up), 2 * out)
    assert np.array_equal(orc.moe_layer("w4a16", xb, r["ids"], r["w"], b_dn), 4 * out)


def test_w4a4_on_grid_x_matches_w4a16_h(orc, tiny):
    s, inp, bank, xb, r = tiny
    rng = np.random.default_rng(9)
    q = rng.integers(0, 16, size=(s.T, s.d)).astype(np.uint8)
    q.reshape(s.T, -1, 16)[:, :, 0] = 7
    sc = rng.integers(0x28, 0x60, size=(s.T, s.d // 16)).astype(np.uint8)
    gs = np.float32(2.0 ** -6)
    S = torch.from_numpy(sc).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    x = E2M1[q] * np.repeat(S, 16, axis=1) * float(gs)
    xg = synth.bf16_bits(torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16))
    assert np.array_equal(_f32(xg), x.astype(np.float32))
    E = s.E
    is13 = np.full(E, gs, np.float32)
    is2 = np.full(E, 1e-3, np.float32)
    _, h16 = orc.moe_layer("w4a16", xg, r["ids"], r["w"], bank, want_h=True)
    _, h4 = orc.moe_layer("w4a4", xg, r["ids"], r["w"], bank, is13=is13, is2=is2, want_h=True)
    assert np.array_equal(h16, h4)


def test_w4a4_input_scale_power_of_two(orc, tiny):
    s, inp, bank, xb, r = tiny
    amax = np.abs(_f32(xb)).max()
    is13 = np.full(s.E, np.float32(amax / 2688.0), np.float32)
    is2 = np.full(s.E, np.float32(0.05), np.float32)
    o1, h1 = orc.moe_layer("w4a4", xb, r["ids"], r["w"], bank, is13=is13, is2=is2, want_h=True)
    o2, h2 = orc.moe_layer("w4a4", xb, r["ids"], r["w"], bank, is13=is13 * 2, is2=is2, want_h=True)
    assert np.array_equal(h1, h2)
    assert np.array_equal(o1, o2)
    # and W4A4 is close to W4A16 (same layer, activations quantised)
    o16 = orc.moe_layer("w4a16", xb, r["ids"], r["w"], bank)
    rel = np.linalg.norm(o1 - o16) / np.linalg.norm(o16)
    assert 1e-3 < rel < 0.3


def test_linear_zero_and_shape(orc):
    x = synth.make_x(3, 64, seed=1)
    xb = synth.bf16_bits(x)
    w = synth.make_weights(1, 32, 64, seed=2)[0]
    q, sc, g = orc.quantize_tensor(synth.bf16_bits(w))
    y = orc.linear(xb, q, sc, g)
    ref = _bf16(g * (_deq(q, sc) @ _f32(xb).astype(np.float64).T).T)
    np.testing.assert_allclose(y, ref, rtol=2 ** -7)
    assert not orc.linear(xb, np.zeros_like(q), sc, g).any()


def test_calibration(orc, tiny):
    s, inp, bank, xb, r = tiny
    is13, is2 = calib.calibrate(xb, inp["logits"].numpy(), s.k, bank)
    assert is13.shape == (s.E,) and np.all(is13 > 0) and np.all(is2 > 0)
    used = np.unique(r["ids"])
    xf = _f32(xb)
    bam = np.abs(xf.reshape(s.T, -1, 16)).max(-1)
    for e in used:
        rows = [t for t in range(s.T) if e in r["ids"][t]]
        want = np.float32(np.percentile(bam[rows].reshape(-1), 99) * 1.05 / 2688.0)
        assert is13[e] == want
    unused = [e for e in range(s.E) if e not in used]
    if unused:
        allrows = np.concatenate([bam[[t for t in range(s.T) if e in r["ids"][t]]].reshape(-1) for e in used])
        assert is13[unused[0]] == np.float32(np.percentile(allrows, 99) * 1.05 / 2688.0)


def test_layer_percentile_policy():
    """The card's activation-scale policy: p99 everywhere, except w2 at
    p98 for layers 3-8 and p98.9 for layers 24-44; layers outside 3-44 are
    not converted."""
    for layer in range(3, 45):
        p13, p2 = calib.layer_percentiles(layer)
        assert p13 == 99.0
        assert p2 == (98.0 if layer <= 8 else 98.9 if layer >= 24 else 99.0)
    for bad in (0, 2, 45, 46):
        with pytest.raises(ValueError):
            calib.layer_percentiles(bad)


def test_calibration_w2_percentile_variants(orc, tiny):
    """w2 scales at the layer-specific percentiles equal the percentile of
    the same h-row block amaxes, recomputed here; a lower percentile never
    gives a larger scale; gate/up scales do not depend on it."""
    s, inp, bank, xb, r = tiny
    lg = inp["logits"].numpy()
    base13, base2 = calib.calibrate(xb, lg, s.k, bank)
    _, h = orc.moe_layer("w4a16", xb, r["ids"], r["w"], bank, want_h=True)
    bam = np.abs(h.astype(np.float32).reshape(s.T, s.k, -1, 16)).max(-1)  # [T, k, F/16]
    for layer in (5, 30):
        p13, p2 = calib.layer_percentiles(layer)
        is13, is2 = calib.calibrate(xb, lg, s.k, bank, pct13=p13, pct2=p2)
        assert np.array_equal(is13, base13)
        assert np.all(is2 <= base2)
        for e in np.unique(r["ids"]):
            sel = np.concatenate([bam[t, j] for t in range(s.T) for j in range(s.k) if r["ids"][t, j] == e])
            assert is2[e] == np.float32(np.percentile(sel, p2) * 1.05 / 2688.0)
