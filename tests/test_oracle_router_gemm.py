"""Pins for the oracle's router GEMM (CPU only).

  * every element equals a plain Python loop over k of exact products of
    the bf16 values (fp64, k order) -- the definition written out again by
    hand, not a library call;
  * one-hot rows (x[t] = 1 at k = t, 0 elsewhere) return the router's
    column k exactly: a transposed operand or a wrong index fails it;
  * the |x w| sums are >= |logits| and equal the loop's.
"""
import numpy as np
import torch

from serving_nvfp4_routed_gb300 import synth


def _f(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_router_gemm_matches_a_hand_loop(orc):
    rng = np.random.default_rng(5)
    x = synth.bf16_bits(torch.from_numpy(rng.standard_normal((4, 37)).astype(np.float32)).to(torch.bfloat16))
    w = synth.bf16_bits(torch.from_numpy(rng.standard_normal((6, 37)).astype(np.float32)).to(torch.bfloat16))
    got, ab = orc.router_logits(x, w)
    xf, wf = _f(x), _f(w)
    for t in range(4):
        for e in range(6):
            s = a = 0.0
            for k in range(37):
                p = float(xf[t, k]) * float(wf[e, k])
                s += p
                a += abs(p)
            assert got[t, e] == s and ab[t, e] == a
    assert np.all(ab >= np.abs(got))


def test_router_gemm_one_hot_rows(orc):
    d, E = 64, 9
    w = synth.bf16_bits(synth.make_weights(1, E, d, seed=3, device="cpu")[0])
    x = np.zeros((d, d), np.uint16)
    x[np.arange(d), np.arange(d)] = 0x3F80  # bf16 1.0
    got, _ = orc.router_logits(x, w)
    assert np.array_equal(got, _f(w).T)
