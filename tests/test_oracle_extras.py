"""Pins for the oracle's optional outputs (CPU only): the values before the
final bf16 rounding round to the oracle's outputs; the |term| sums equal a
numpy evaluation over the fully dequantised weights; h is the SwiGLU of the
rounded gate / up values; the W4A4 rows are the oracle's own quantisation
of x and h.  Also pins the tolerance helpers of the GPU tests on the
oracle's own values (they must accept the oracle's results and reject a
one-step miss far from a rounding midpoint)."""
import numpy as np
import torch

from gpu_util import (assert_h_in_interval, assert_out_close, bf16_key, h_interval, nvfp4_block_feasible,
                      round_bf16, unpack_codes)
from oracle import calib
from serving_nvfp4_routed_gb300 import synth
from test_oracle_layer import _deq, _f32, _quant_bank


def _setup(orc, seed=5, T=6, d=128, E=3, k=2, F=64):
    s = synth.MoEShape(T, d, E, k, F)
    inp = synth.moe_inputs(s, seed, outlier_frac=0.2)
    bank = _quant_bank(orc, dict(gate=inp["gate"], up=inp["up"], down=inp["down"]))
    xb = synth.bf16_bits(inp["x"])
    r = orc.route(inp["logits"].numpy(), k)
    return s, inp, bank, xb, r


def test_round_bf16_helper_matches_oracle(orc):
    rng = np.random.default_rng(1)
    v = rng.standard_normal(2000) * np.exp2(rng.integers(-20, 20, 2000))
    on_grid = round_bf16(v)
    ties = on_grid + np.ldexp(1.0, np.frexp(on_grid)[1] - 9)  # exact midpoints between bf16 neighbours
    for a in np.concatenate([v, ties]):
        assert round_bf16(a) == orc.round_bf16(float(a)), a
    k = bf16_key(np.array([1.0, 1.0078125, -0.0, 0.0, -1.0, -1.0078125, 2.0 ** -133], np.float32))
    assert k[1] - k[0] == 1 and k[2] == k[3] == 0 and k[5] == k[4] - 1 and k[6] == 1


def test_layer_extras(orc):
    s, inp, bank, xb, r = _setup(orc)
    ex = orc.moe_layer_ex("w4a16", xb, r["ids"], r["w"], bank)
    assert np.array_equal(ex["out"], orc.moe_layer("w4a16", xb, r["ids"], r["w"], bank))
    assert np.array_equal(round_bf16(ex["out_pre"]), ex["out"])
    xf = _f32(xb).astype(np.float64)
    gq, gs, g2 = bank["gate"]
    uq, us, u2 = bank["up"]
    dq, ds, d2 = bank["down"]
    for t in range(s.T):
        want_abs = np.zeros(s.d)
        for j in range(s.k):
            e = r["ids"][t, j]
            Wg, Wu, Wd = _deq(gq[e], gs[e]), _deq(uq[e], us[e]), _deq(dq[e], ds[e])
            np.testing.assert_allclose(ex["g_pre"][t, j], float(g2[e]) * (Wg @ xf[t]), rtol=1e-12, atol=1e-300)
            np.testing.assert_allclose(ex["g_abs"][t, j], float(g2[e]) * (np.abs(Wg) @ np.abs(xf[t])), rtol=1e-12)
            np.testing.assert_allclose(ex["u_abs"][t, j], float(u2[e]) * (np.abs(Wu) @ np.abs(xf[t])), rtol=1e-12)
            G, U = round_bf16(ex["g_pre"][t, j]), round_bf16(ex["u_pre"][t, j])
            assert np.array_equal(ex["h"][t, j], round_bf16(G / (1 + np.exp(-G)) * U))
            want_abs += abs(float(r["w"][t, j])) * float(d2[e]) * (np.abs(Wd) @ np.abs(ex["h"][t, j].astype(np.float64)))
        np.testing.assert_allclose(ex["out_abs"][t], want_abs, rtol=1e-12)
    assert np.all(ex["out_abs"] >= np.abs(ex["out_pre"]))


def test_layer_extras_w4a4_rows(orc):
    s, inp, bank, xb, r = _setup(orc, seed=9)
    is13, is2 = calib.calibrate(xb, inp["logits"].numpy(), s.k, bank)
    ex = orc.moe_layer_ex("w4a4", xb, r["ids"], r["w"], bank, is13=is13, is2=is2)
    assert np.array_equal(round_bf16(ex["out_pre"]), ex["out"])
    gs_rows = is13[r["ids"]].reshape(-1)
    xq, xs = orc.quantize_rows(np.repeat(xb, s.k, axis=0), gs_rows)
    assert np.array_equal(xq.reshape(ex["xq"].shape), ex["xq"]) and np.array_equal(xs.reshape(ex["xs"].shape), ex["xs"])
    hb = synth.bf16_bits(torch.from_numpy(ex["h"].reshape(-1, s.F)).to(torch.bfloat16))
    hq, hs = orc.quantize_rows(hb, is2[r["ids"]].reshape(-1))
    assert np.array_equal(hq.reshape(ex["hq"].shape), ex["hq"]) and np.array_equal(hs.reshape(ex["hs"].shape), ex["hs"])


def test_tolerance_helpers_accept_the_oracle_and_reject_a_real_miss(orc):
    s, inp, bank, xb, r = _setup(orc, seed=13, T=8)
    ex = orc.moe_layer_ex("w4a16", xb, r["ids"], r["w"], bank)
    lo, hi = h_interval(ex["g_pre"], ex["u_pre"], ex["g_abs"], ex["u_abs"], s.d, True)
    assert_h_in_interval(ex["h"], lo, hi)
    bound = 1e-6 * ex["out_abs"]
    assert_out_close(ex["out"], ex["out"], ex["out_pre"], bound)
    # a one-step miss on the largest element, whose exact value is not near a midpoint
    # (the bound is far below half a step there)
    out = ex["out"].astype(np.float64).copy()
    i = np.argmax(np.abs(out))
    step = np.ldexp(1.0, np.frexp(out.flat[i])[1] - 8)
    out.flat[i] += step
    mid = out.flat[i] - step / 2
    if abs(ex["out_pre"].flat[i] - mid) > bound.flat[i] and step > 2e-2 * np.sqrt(np.mean(ex["out"] ** 2)):
        try:
            assert_out_close(out, ex["out"], ex["out_pre"], bound)
        except AssertionError:
            pass
        else:
            raise AssertionError("a one-step miss far from the midpoint was accepted")


def test_block_feasibility_accepts_the_oracle_blocks(orc):
    s, inp, bank, xb, r = _setup(orc, seed=17)
    is13, is2 = calib.calibrate(xb, inp["logits"].numpy(), s.k, bank)
    ex = orc.moe_layer_ex("w4a4", xb, r["ids"], r["w"], bank, is13=is13, is2=is2)
    lo, hi = h_interval(ex["g_pre"], ex["u_pre"], ex["g_abs"], ex["u_abs"], s.d, False)
    codes = unpack_codes(ex["hq"])
    t, j = 0, 0
    e = r["ids"][t, j]
    for b in range(s.F // 16):
        sl = slice(16 * b, 16 * b + 16)
        assert nvfp4_block_feasible(orc, lo[t, j, sl], hi[t, j, sl], float(is2[e]), int(ex["hs"][t, j, b]),
                                    codes[t, j, sl])
    # a scale byte far above any reachable block maximum is rejected
    assert not nvfp4_block_feasible(orc, lo[t, j, :16], hi[t, j, :16], float(is2[e]), 0x7E, codes[t, j, :16])


def test_round_y_switch(orc):
    """y_pre is each pair's down projection (numpy over the dequantised
    weights); with the R3 switch the output is bf16 of the slot-ordered
    weighted sum of the bf16-rounded y, without it of the unrounded y."""
    s, inp, bank, xb, r = _setup(orc, seed=21)
    ex = orc.moe_layer_ex("w4a16", xb, r["ids"], r["w"], bank)
    ex3 = orc.moe_layer_ex("w4a16", xb, r["ids"], r["w"], bank, round_y=True)
    assert np.array_equal(ex["y_pre"], ex3["y_pre"]) and np.array_equal(ex["h"], ex3["h"])
    dq, ds, d2 = bank["down"]
    for t in range(s.T):
        acc = np.zeros(s.d)
        for j in range(s.k):
            e = r["ids"][t, j]
            Wd = _deq(dq[e], ds[e])
            y = float(d2[e]) * (Wd @ ex["h"][t, j].astype(np.float64))
            np.testing.assert_allclose(ex["y_pre"][t, j], y, rtol=1e-12, atol=1e-300)
            np.testing.assert_allclose(ex["y_abs"][t, j], float(d2[e]) * (np.abs(Wd) @ np.abs(ex["h"][t, j])),
                                       rtol=1e-12)
            acc = acc + float(r["w"][t, j]) * round_bf16(ex3["y_pre"][t, j])
        np.testing.assert_allclose(ex3["out_pre"][t], acc, rtol=1e-13, atol=1e-300)
    assert np.array_equal(round_bf16(ex3["out_pre"]), ex3["out"])
    assert not np.array_equal(ex["out_pre"], ex3["out_pre"])
