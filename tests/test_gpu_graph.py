"""The layer calls are CUDA-graph capturable (no host sync, no allocation,
device-side work counters reset inside the graph): a call captured once and
replayed on new inputs copied into the captured buffers gives the result of
an eager call -- bit for bit on the prompt path (slot-ordered combine), and
against the oracle on the decode path (arrival-order combine)."""
import numpy as np
import pytest
import torch

import serving_nvfp4_routed_gb300 as lib
from serving_nvfp4_routed_gb300 import synth

from gpu_util import OracleBank
from layer_check import check_layer

pytestmark = pytest.mark.gpu


def _capture(run, x_s, lg_s):
    out = run(x_s, lg_s)  # first call outside the capture (one-time kernel setup)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            run(x_s, lg_s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g, out


@pytest.mark.parametrize("path,mode", [("tc", "w4a16"), ("tc", "w4a4"), ("gemv", "w4a16")])
def test_layer_graph_replay(orc, path, mode):
    lib.set_kernel_choice(path)
    try:
        _graph_case(orc, path, mode)
    finally:
        lib.set_kernel_choice("auto")


def _graph_case(orc, path, mode):
    T, E, k, d, F = 256, 16, 4, 512, 256
    s = synth.MoEShape(T, d, E, k, F)
    inp = synth.moe_inputs(s, 41, device="cuda", outlier_frac=0.05)
    banks = dict(gate=inp["gate"], up=inp["up"], down=inp["down"])
    gw = lib.MoEWeights(*(lib.nvfp4_quantize_weights(banks[n]) for n in ("gate", "up", "down")))
    is13 = torch.full((E,), 0.004, device="cuda")
    is2 = torch.full((E,), 0.001, device="cuda")
    out = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    ws = lib.moe_workspace(T, E, k, d, F, mode, "cuda")
    if mode == "w4a16":
        run = lambda xx, ll: lib.nvfp4_moe_w4a16(xx, ll, k, gw, out=out, ws=ws)
    else:
        run = lambda xx, ll: lib.nvfp4_moe_w4a4(xx, ll, k, gw, is13, is2, out=out, ws=ws)
    x_s, lg_s = inp["x"].clone(), inp["logits"].clone()
    g, _ = _capture(run, x_s, lg_s)
    # a second batch through the graph
    x2 = synth.make_x(T, d, seed=42, device="cuda", outlier_frac=0.05)
    lg2 = synth.make_logits(T, E, seed=43, device="cuda")
    x_s.copy_(x2)
    lg_s.copy_(lg2)
    g.replay()
    torch.cuda.synchronize()
    got = out.clone()
    if path == "tc":
        eager = run(x2, lg2).clone()
        assert torch.equal(got.view(torch.int16), eager.view(torch.int16))
    else:
        ob = OracleBank(orc, banks).get()
        check_layer(orc, "w4a16", x2, lg2, k, ob, got, ws, np.arange(T, dtype=np.int32), what="graph replay")
