"""GPU parity: routing ids, expert offsets and the stable permutation are
bit-exact against the oracle; routing weights within 1 fp32 ulp (both sides
evaluate the renormalised softmax in fp64 and round once to fp32, so they
can differ only where the fp64 value sits next to an fp32 midpoint)."""
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
    """Within 1 ulp of the oracle's fp32 weights (the pin asks for 2)."""
    ref = r["w"].astype(np.float32)
    got = gw.astype(np.float32)
    assert np.all(np.isfinite(got))
    ulp = np.spacing(np.maximum(np.abs(ref), np.finfo(np.float32).tiny))
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    assert np.all(err <= ulp), (err / ulp).max()
    return float(np.mean(got == ref))


@pytest.mark.parametrize("T,E,k,kind", [(1, 288, 8, "normal"), (4, 8, 2, "normal"), (64, 288, 8, "normal"),
                                        (1023, 288, 8, "normal"), (1, 1024, 32, "normal"),
                                        (300, 1000, 3, "normal"), (50, 33, 32, "normal"),
                                        (4096, 288, 8, "normal"), (16384, 288, 8, "zipf"),
                                        (16384, 288, 8, "zipf_masked"), (5000, 64, 1, "normal")])
def test_route_matches_oracle(orc, T, E, k, kind):
    logits = synth.make_logits(T, E, seed=T * 7 + E, device="cuda", kind=kind)
    _cmp(orc, logits, k)


def test_route_ties_and_infinities(orc):
    lg = torch.zeros(48, 64)
    lg[10:20] = torch.randint(0, 3, (10, 64)).float()
    lg[20:30, ::2] = -float("inf")
    lg[30, :] = -float("inf")             # every logit -inf: weights 1/k
    lg[31, 5] = float("inf")              # one +inf: weight 1 on it
    lg[32, [3, 9]] = float("inf")         # two +inf: 1/2 each
    lg[33, :40] = float("nan")            # NaN ranks as -inf
    lg[34, :] = float("nan")
    _cmp(orc, lg.cuda(), 8)
    r = orc.route(lg.numpy(), 8)
    assert np.allclose(r["w"][30], 1 / 8) and np.allclose(r["w"][34], 1 / 8)
    assert r["w"][31, 0] == 1.0 and r["ids"][31, 0] == 5 and not r["w"][31, 1:].any()
    assert np.all(r["w"][32, :2] == 0.5) and list(r["ids"][32, :2]) == [3, 9]
    assert r["ids"][33].min() >= 40
    _cmp(orc, torch.zeros(9000 // 8 + 3, 16).cuda(), 8)  # all ties, multi-block path


def test_route_empty():
    g = lib.moe_route_permute(torch.zeros(0, 16, device="cuda"), 2)
    assert g["ids"].numel() == 0
    assert torch.all(g["offsets"] == 0)
