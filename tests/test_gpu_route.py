"""GPU parity: routing ids, expert offsets and the stable permutation are
bit-exact against the oracle; routing weights within 1 fp32 ulp."""
import numpy as np
import pytest
import torch

import serving_nvfp4_routed_gb300 as lib
from serving_nvfp4_routed_gb300 import synth

pytestmark = pytest.mark.gpu


def _cmp(orc, logits, k):
    g = lib.moe_route_permute(logits, k)
    torch.cuda.synchronize()
    r = orc.route(logits.cpu().numpy(), k)
    assert np.array_equal(g["ids"].cpu().numpy(), r["ids"])
    assert np.array_equal(g["offsets"].cpu().numpy(), r["offsets"])
    assert np.array_equal(g["row_to_slot"].cpu().numpy(), r["row_to_slot"])
    assert np.array_equal(g["slot_to_row"].cpu().numpy(), r["slot_to_row"])
    _check_weights(logits.cpu().numpy(), r, g["w"].cpu().numpy(), k)
    return r


def _check_weights(lg, r, gw, k):
    """The GPU computes the renormalised softmax in fp32 (a_j = l_j - l_max
    rounded, expf within 2 ulp, a k-term fp32 sum, one division); the oracle
    in fp64.  Relative error bound of that fp32 evaluation:
    (|a_j| + max_i |a_i| + k + 8) * 2^-24."""
    sel = np.take_along_axis(lg.astype(np.float64), r["ids"].astype(np.int64), axis=1)
    with np.errstate(invalid="ignore"):
        a = np.abs(sel - sel[:, :1])
    a = np.where(np.isfinite(a), a, 0.0)
    bound = (a + a.max(axis=1, keepdims=True) + k + 8) * 2.0 ** -24
    ref = r["w"].astype(np.float64)
    err = np.abs(gw.astype(np.float64) - ref)
    assert np.all(err <= bound * np.maximum(ref, np.finfo(np.float32).tiny)), (err / np.maximum(ref, 1e-30)).max()


@pytest.mark.parametrize("T,E,k,kind", [(1, 288, 8, "normal"), (4, 8, 2, "normal"), (64, 288, 8, "normal"),
                                        (1023, 288, 8, "normal"), (1, 1024, 32, "normal"),
                                        (300, 1000, 3, "normal"), (50, 33, 32, "normal"),
                                        (4096, 288, 8, "normal"), (16384, 288, 8, "zipf"),
                                        (16384, 288, 8, "zipf_masked"), (5000, 64, 1, "normal")])
def test_route_matches_oracle(orc, T, E, k, kind):
    logits = synth.make_logits(T, E, seed=T * 7 + E, device="cuda", kind=kind)
    _cmp(orc, logits, k)


def test_route_ties_and_infinities(orc):
    lg = torch.zeros(40, 64)
    lg[10:20] = torch.randint(0, 3, (10, 64)).float()
    lg[20:30, ::2] = -float("inf")
    _cmp(orc, lg.cuda(), 8)
    _cmp(orc, torch.zeros(9000 // 8 + 3, 16).cuda(), 8)  # all ties, multi-block path


def test_route_empty():
    g = lib.moe_route_permute(torch.zeros(0, 16, device="cuda"), 2)
    assert g["ids"].numel() == 0
    assert torch.all(g["offsets"] == 0)
