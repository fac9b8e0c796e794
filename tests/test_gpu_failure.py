"""Failure detection without a GPU fault: a library kernel waits on a barrier
that nothing arrives on; its bounded wait must give up, report
NVFP4_ERR_TIMEOUT (7) through the status word and return normally, leaving
the context usable for the next layer call."""
import numpy as np
import pytest
import torch

import serving_nvfp4_routed_gb300 as lib
from serving_nvfp4_routed_gb300 import synth

from gpu_util import assert_layer_close, bf16_to_f32, gpu_bank, oracle_bank

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
    out = lib.nvfp4_moe_w4a16(inp["x"], inp["logits"], s.k, gpu_bank(lib, banks))
    r = orc.route(inp["logits"].cpu().numpy(), s.k)
    ref = orc.moe_layer("w4a16", synth.bf16_bits(inp["x"]), r["ids"], r["w"], oracle_bank(orc, banks))
    assert_layer_close(bf16_to_f32(out), ref, "after timeout")
