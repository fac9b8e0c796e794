"""Failure detection without a GPU fault: a library kernel waits on a barrier
that nothing arrives on; its bounded wait must give up, report
NVFP4_ERR_TIMEOUT (7) through the status word and return normally, leaving
the context usable for the next layer call."""
import numpy as np
import pytest
import torch

import serving_nvfp4_routed_gb300 as lib
from serving_nvfp4_routed_gb300 import synth

from gpu_util import OracleBank, gpu_bank
from layer_check import check_layer

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(orc):
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    lib.selftest_bounded_wait(st)
    torch.cuda.synchronize()
    assert st[0].item() == 7  # NVFP4_ERR_TIMEOUT
    assert lib.status_string(7) != ""
    # the context still runs the layer correctly afterwards
    s = synth.TINY
    inp = synth.moe_inputs(s, 77, device="cuda")
    banks = {k: inp[k] for k in ("gate", "up", "down")}
    ws = lib.moe_workspace(s.T, s.E, s.k, s.d, s.F, "w4a16", "cuda")
    out = lib.nvfp4_moe_w4a16(inp["x"], inp["logits"], s.k, gpu_bank(lib, banks), ws=ws)
    check_layer(orc, "w4a16", inp["x"], inp["logits"], s.k, OracleBank(orc, banks).get(), out, ws,
                np.arange(s.T, dtype=np.int32), what="after timeout")
