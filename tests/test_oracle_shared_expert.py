"""Pins for the oracle's BF16 shared-expert MLP (CPU only).

  * a hand-worked token: G = 1, U = 2, h = bf16(silu(1) * 2) = 1.4609375,
    out = bf16(routed + h * wd);
  * a plain Python loop with torch's bf16 rounding at the same points
    (G, U, h, out) on random tiny shapes: equal bit for bit;
  * a zero down projection leaves the routed output unchanged.
"""
import math

import numpy as np
import torch


def _bf(v):
    return (np.asarray(v, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _f(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _rb(v):
    return float(torch.tensor(v, dtype=torch.float64).to(torch.bfloat16).to(torch.float64))


def test_shared_expert_hand_worked(orc):
    out = orc.shared_expert(_bf([[1, 2]]), _bf([[1, 0]]), _bf([[0, 1]]), _bf([[1], [2]]), _bf([[0.5, -1]]))
    h = _rb(2.0 / (1.0 + math.exp(-1.0)))
    assert h == 1.4609375
    assert out[0, 0] == _rb(0.5 + h) and out[0, 1] == _rb(-1 + 2 * h)


def test_shared_expert_matches_a_hand_loop(orc):
    rng = np.random.default_rng(9)
    T, d, Fs = 3, 5, 4
    x, wg, wu = (_bf(rng.standard_normal(s)) for s in ((T, d), (Fs, d), (Fs, d)))
    wd, r = _bf(rng.standard_normal((d, Fs))), _bf(rng.standard_normal((T, d)))
    got = orc.shared_expert(x, wg, wu, wd, r)
    X, G_, U_, D_, R_ = _f(x), _f(wg), _f(wu), _f(wd), _f(r)
    for t in range(T):
        h = []
        for f in range(Fs):
            g = u = 0.0
            for k in range(d):
                g += X[t, k] * G_[f, k]
                u += X[t, k] * U_[f, k]
            G, U = _rb(g), _rb(u)
            h.append(_rb(G / (1.0 + math.exp(-G)) * U))
        for n in range(d):
            y = 0.0
            for f in range(Fs):
                y += h[f] * D_[n, f]
            assert got[t, n] == _rb(R_[t, n] + y)


def test_shared_expert_zero_down_keeps_routed(orc):
    rng = np.random.default_rng(10)
    x, wg, wu = _bf(rng.standard_normal((2, 8))), _bf(rng.standard_normal((4, 8))), _bf(rng.standard_normal((4, 8)))
    r = _bf(rng.standard_normal((2, 8)))
    got = orc.shared_expert(x, wg, wu, np.zeros((8, 4), np.uint16), r)
    assert np.array_equal(got, _f(r).astype(np.float32))
