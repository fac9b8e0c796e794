"""GPU parity: the BF16 router GEMM (tcgen05, fp32 accumulate) against the
oracle's fp64 loop, within the bound any fp32 evaluation of the sum meets:
|logits - exact| <= d * 2^-24 * sum_k |x w|."""
import numpy as np
import pytest
import torch

import serving_nvfp4_routed_gb300 as lib
from serving_nvfp4_routed_gb300 import synth

pytestmark = pytest.mark.gpu


def _check(orc, x, w, rows=None):
    got = lib.moe_router_logits(x, w).cpu().double().numpy()
    xb = synth.bf16_bits(x)
    if rows is not None:
        xb, got = xb[rows], got[rows]
    ref, ab = orc.router_logits(xb, synth.bf16_bits(w))
    d = x.shape[1]
    bound = d * 2.0 ** -24 * ab + 1e-30
    bad = np.argwhere(np.abs(got - ref) > bound)
    assert bad.size == 0, (bad[:5], got[tuple(bad[0])], ref[tuple(bad[0])])
    return got, ref


@pytest.mark.parametrize("T,d,E", [(1, 4096, 288), (77, 4096, 288), (300, 256, 8), (130, 512, 33),
                                   (257, 1024, 500), (64, 64, 32), (129, 128, 512)])
def test_router_logits(orc, T, d, E):
    """Single and ragged token tiles, E padded to 32 columns, one or two
    MMA column blocks (E up to 512), k-stage counts below and above the ring."""
    x = synth.make_x(T, d, seed=T + d, device="cuda", outlier_frac=0.05)
    w = synth.make_weights(1, E, d, seed=E + 1, device="cuda")[0]
    _check(orc, x, w)


def test_router_logits_full_size_sampled(orc):
    """T=8192 tokens, d=4096, E=288 (the prompt configuration): sampled
    tokens from many 128-token tiles, the first and the last."""
    T, d, E = 8192, 4096, 288
    x = synth.make_x(T, d, seed=11, device="cuda", outlier_frac=0.05)
    w = synth.make_weights(1, E, d, seed=12, device="cuda")[0]
    rows = np.unique(np.append(np.random.default_rng(13).choice(T, 40, replace=False), [0, T - 1]))
    _check(orc, x, w, rows)


def test_router_then_route_matches_oracle_route(orc):
    """The fp32 logits feed moe_route_permute: its ids and weights equal the
    oracle's routing of the same fp32 logits, bit for bit."""
    T, d, E, k = 200, 1024, 64, 8
    x = synth.make_x(T, d, seed=21, device="cuda")
    w = synth.make_weights(1, E, d, seed=22, device="cuda")[0]
    lg = lib.moe_router_logits(x, w)
    r = lib.moe_route_permute(lg, k)
    ro = orc.route(lg.cpu().numpy(), k)
    assert np.array_equal(r["ids"].cpu().numpy(), ro["ids"])
    assert np.array_equal(r["row_to_slot"].cpu().numpy(), ro["row_to_slot"])
