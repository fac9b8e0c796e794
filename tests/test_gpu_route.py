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
    np.testing.assert_array_max_ulp(g["w"].cpu().numpy(), r["w"], maxulp=1)
    return r


@pytest.mark.parametrize("T,E,k,kind", [(1, 288, 8, "normal"), (4, 8, 2, "normal"), (64, 288, 8, "normal"),
                                        (1023, 288, 8, "normal"), (1, 1024, 32, "normal"),
                                        (300, 1000, 3, "normal"), (50, 33, 33, "normal"),
                                        (4096, 288, 8, "normal"), (16384, 288, 8, "zipf"),
                                        (16384, 288, 8, "zipf_masked"), (5000, 64, 1, "normal")])
def test_route_matches_oracle(orc, T, E, k, kind):
    logits = synth.make_logits(T, E, seed=T * 7 + E, device="cuda", kind=kind)
    _cmp(orc, logits, k)


def test_route_ties_and_infinities(orc):
    lg = torch.zeros(40, 64)
    lg[10:20] = torch.randint(0, 3, (10, 64)).float()
    lg[20:30, ::2] = -float("inf")
    lg[30:40, 5] = float("inf")
    _cmp(orc, lg.cuda(), 8)
    _cmp(orc, torch.zeros(9000 // 8 + 3, 16).cuda(), 8)  # all ties, multi-block path


def test_route_empty():
    g = lib.moe_route_permute(torch.zeros(0, 16, device="cuda"), 2)
    assert g["ids"].numel() == 0
    assert torch.all(g["offsets"] == 0)
