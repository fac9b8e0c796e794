"""GPU parity: NVFP4 weight recipe and static activation quantisation are
bit-exact against the oracle (codes, scales, weight_scale_2)."""
import numpy as np
import pytest
import torch

import serving_nvfp4_routed_gb300 as lib
from serving_nvfp4_routed_gb300 import synth

pytestmark = pytest.mark.gpu

E2M1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])


def _cmp_tensor(orc, w):
    q = lib.nvfp4_quantize_weights(w)
    for b in range(w.shape[0]):
        oc, os_, o2 = orc.quantize_tensor(synth.bf16_bits(w[b]))
        assert q.weight_scale_2[b].item() == o2
        assert np.array_equal(q.scales[b].cpu().numpy(), os_)
        gc = q.codes[b].cpu().numpy()
        bad = np.argwhere(gc != oc)
        assert bad.size == 0, (b, bad[:5], gc[tuple(bad[0])], oc[tuple(bad[0])])


@pytest.mark.parametrize("B,N,K,seed", [(1, 16, 16, 1), (3, 33, 48, 2), (2, 128, 256, 3), (1, 7, 4096, 4),
                                        (5, 96, 1536, 5)])
def test_weight_recipe_bit_exact(orc, B, N, K, seed):
    _cmp_tensor(orc, synth.make_weights(B, N, K, seed, device="cuda"))


def test_weight_recipe_ties_zero_and_extremes(orc):
    # on-grid blocks hitting every e2m1 tie with ws2 a power of two, plus a zero
    # tensor, a tensor of one nonzero value, and wide dynamic range
    rng = np.random.default_rng(11)
    N, K = 64, 256
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.0, 6.0, 0.5, 3.0, 4.0])
    t = rng.choice(ties, size=(N, K)) * rng.choice([-1, 1], size=(N, K))
    t.reshape(N, K // 16, 16)[:, :, 0] = 6.0
    s = rng.integers(0x20, 0x7E, size=(N, K // 16)).astype(np.uint8)
    s[0, 0] = 0x7E
    S = torch.from_numpy(s).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    v = t * np.repeat(S, 16, axis=1) * 2.0 ** -9
    w1 = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16)
    assert torch.equal(w1.double(), torch.from_numpy(v))
    w2 = torch.zeros(N, K, dtype=torch.bfloat16)
    w3 = torch.zeros(N, K, dtype=torch.bfloat16)
    w3[5, 17] = -3.0
    w4 = (torch.randn(N, K, generator=torch.Generator().manual_seed(3)) *
          torch.exp(torch.randn(N, K, generator=torch.Generator().manual_seed(4)) * 6)).to(torch.bfloat16)
    _cmp_tensor(orc, torch.stack([w1, w2, w3, w4]).cuda())


def test_weight_recipe_full_bank_sampled(orc):
    """The full decode bank (288 experts, gate [1536, 4096] and down [4096, 1536])
    quantised in one batched call; sampled experts checked bit-exact."""
    for (N, K) in ((1536, 4096), (4096, 1536)):
        w = synth.make_weights(288, N, K, seed=77, device="cuda")
        q = lib.nvfp4_quantize_weights(w)
        for e in (0, 131, 287):
            oc, os_, o2 = orc.quantize_tensor(synth.bf16_bits(w[e]))
            assert q.weight_scale_2[e].item() == o2
            assert np.array_equal(q.scales[e].cpu().numpy(), os_)
            assert np.array_equal(q.codes[e].cpu().numpy(), oc)
        del w, q
        torch.cuda.empty_cache()


@pytest.mark.parametrize("T,E,k,d,gs_kind", [(4, 8, 2, 256, "calib"), (64, 288, 8, 4096, "calib"),
                                             (33, 16, 4, 512, "tiny"), (17, 16, 3, 512, "huge"),
                                             (600, 288, 8, 1024, "calib"), (5, 16, 2, 1040, "calib"),
                                             (1250, 16, 8, 1040, "calib")])
def test_activation_quant_gathered_bit_exact(orc, T, E, k, d, gs_kind):
    x = synth.make_x(T, d, seed=T + d, device="cuda", outlier_frac=0.05)
    logits = synth.make_logits(T, E, seed=T, device="cuda")
    r = orc.route(logits.cpu().numpy(), k)
    xb = synth.bf16_bits(x)
    amax = np.abs((xb.astype(np.uint32) << 16).view(np.float32)).max()
    if gs_kind == "calib":
        gs = (np.linspace(0.2, 1.5, E) * amax / 2688.0).astype(np.float32)
    elif gs_kind == "tiny":
        gs = np.full(E, 1e-7, np.float32)
    else:
        gs = np.full(E, 1e3, np.float32)
    offs = r["offsets"]
    R = T * k
    row_exp = np.searchsorted(offs, np.arange(R), side="right") - 1
    src = r["row_to_slot"] // k
    oc, os_ = orc.quantize_rows(xb[src], gs[row_exp])
    gc, gsc = lib.nvfp4_quantize_act(x, torch.from_numpy(gs).cuda(), M=R,
                                     row_to_slot=torch.from_numpy(r["row_to_slot"]).cuda(), top_k=k,
                                     expert_offsets=torch.from_numpy(offs).cuda())
    assert np.array_equal(gsc.cpu().numpy(), os_)
    assert np.array_equal(gc.cpu().numpy(), oc)


def test_activation_quant_plain_rows(orc):
    x = synth.make_x(5, 64, seed=9, device="cuda")
    gs = np.array([0.01], np.float32)
    oc, os_ = orc.quantize_rows(synth.bf16_bits(x), np.repeat(gs, 5))
    gc, gsc = lib.nvfp4_quantize_act(x, torch.from_numpy(gs).cuda())
    assert np.array_equal(gc.cpu().numpy(), oc) and np.array_equal(gsc.cpu().numpy(), os_)


def test_activation_quant_quotients_near_every_boundary(orc):
    """Blocks whose quotients x / (S * gs) fall exactly on each e2m1 rounding
    boundary (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5) and within 1-4 fp32 ulp of
    it on either side: row t uses gs = 2^-6 * (1 + (t - 4) * 2^-23), so the
    kernel's reciprocal-multiply shortcut must defer to the exact quotient
    there.  Codes and scales bit-exact against the oracle."""
    E = T = 9
    d = 256
    base = np.array([6, .25, .75, 1.25, 1.75, 2.5, 3.5, 5, -.25, -.75, -1.25, -1.75, -2.5, -3.5, -5, -6])
    blocks = [base * 2.0 ** j for j in (0, -1, -2, 1)]
    row = np.concatenate([blocks[b % 4] for b in range(d // 16)]) * 2.0 ** -6
    x64 = np.tile(row, (T, 1))
    x = torch.from_numpy(x64).to(torch.bfloat16)
    assert torch.equal(x.double(), torch.from_numpy(x64))
    gs = np.array([2.0 ** -6 * (1 + (t - 4) * 2.0 ** -23) for t in range(T)], np.float32)
    offs = np.arange(E + 1, dtype=np.int32)
    rts = np.arange(T, dtype=np.int32)
    oc, os_ = orc.quantize_rows(synth.bf16_bits(x), gs)
    gc, gsc = lib.nvfp4_quantize_act(x.cuda(), torch.from_numpy(gs).cuda(), M=T,
                                     row_to_slot=torch.from_numpy(rts).cuda(), top_k=1,
                                     expert_offsets=torch.from_numpy(offs).cuda())
    assert np.array_equal(gsc.cpu().numpy(), os_)
    assert np.array_equal(gc.cpu().numpy(), oc)
    # the rows differ: the quotients sit on both sides of the boundaries
    assert len({bytes(oc[t]) for t in range(T)}) > 1
