"""GPU parity: the BF16 shared-expert MLP (tcgen05 bf16 GEMMs) added to a
routed output, against the oracle with the same rounding points (G, U, h,
out): the kernel's h inside the interval of the error model, the output
within the layer tolerance or a justified bf16 neighbour (tests/gpu_util.py)."""
import numpy as np
import pytest
import torch

import serving_nvfp4_routed_gb300 as lib
from serving_nvfp4_routed_gb300 import synth

from gpu_util import (OracleBank, U32, assert_h_in_interval, assert_out_close, bf16_to_f32, gamma, gpu_bank,
                      h_interval)
from layer_check import check_layer

pytestmark = pytest.mark.gpu


def _check_shared(orc, x, wg, wu, wd, routed, out, ws, what):
    T, d = x.shape
    Fs = wg.shape[0]
    ex = orc.shared_expert_ex(synth.bf16_bits(x), synth.bf16_bits(wg), synth.bf16_bits(wu), synth.bf16_bits(wd),
                              synth.bf16_bits(routed))
    hk = bf16_to_f32(ws[:T * Fs * 2].view(torch.bfloat16).view(T, Fs)).astype(np.float64)
    lo, hi = h_interval(ex["g_pre"], ex["u_pre"], ex["g_abs"], ex["u_abs"], d, True)
    assert_h_in_interval(hk, lo, hi, f"{what}: h")
    dh = np.abs(hk - ex["h"])
    wdf = np.abs(bf16_to_f32(wd).astype(np.float64))
    bound = gamma(Fs) * ex["out_abs"] + 2 * U32 * np.abs(ex["out_pre"]) + dh @ wdf.T
    return assert_out_close(bf16_to_f32(out), ex["out"], ex["out_pre"], bound, what)


@pytest.mark.parametrize("T,d,Fs", [(1, 256, 128), (24, 2048, 512), (100, 512, 256), (300, 1024, 384),
                                    (129, 4096, 1536), (64, 4096, 1536), (1280, 2048, 256)])
def test_shared_expert(orc, T, d, Fs):
    """Single and ragged token tiles, one and several weight tiles in both
    GEMMs, K from 128 to 4096.  The small batches run the narrow tiles (the
    weight rows as the MMA's M, 16, 32, 64 or 128 tokens as its N: T = 1,
    24, 64 and the rest; K split over clusters of 1 to 8 CTAs), the last
    case (ten 128-token tiles) the wide ones."""
    x = synth.make_x(T, d, seed=T + d, device="cuda", outlier_frac=0.05)
    wg = synth.make_weights(1, Fs, d, seed=Fs + 1, device="cuda")[0]
    wu = synth.make_weights(1, Fs, d, seed=Fs + 2, device="cuda")[0] * 2
    wd = synth.make_weights(1, d, Fs, seed=Fs + 3, device="cuda")[0]
    routed = synth.make_x(T, d, seed=T + d + 1, device="cuda")
    out = routed.clone()
    ws = torch.empty(max(16, lib.load().moe_shared_expert_workspace_size(T, Fs)), dtype=torch.uint8, device="cuda")
    lib.moe_shared_expert(x, wg, wu, wd, out, ws=ws)
    torch.cuda.synchronize()
    _check_shared(orc, x, wg, wu, wd, routed, out, ws, "shared expert")


def test_routed_layer_then_shared_expert(orc):
    """The MoE block end to end on the library: router GEMM -> routed W4A16
    layer -> shared expert; checked against the oracle step by step on the
    library's own intermediate results."""
    T, d, E, k, F, Fs = 64, 512, 16, 4, 256, 256
    s = synth.MoEShape(T, d, E, k, F)
    inp = synth.moe_inputs(s, 31, device="cuda")
    banks = dict(gate=inp["gate"], up=inp["up"], down=inp["down"])
    gw = gpu_bank(lib, banks)
    wr = synth.make_weights(1, E, d, seed=32, device="cuda")[0]
    logits = lib.moe_router_logits(inp["x"], wr)
    ws = lib.moe_workspace(T, E, k, d, F, "w4a16", "cuda")
    routed = lib.nvfp4_moe_w4a16(inp["x"], logits, k, gw, ws=ws)
    ob = OracleBank(orc, banks).get()
    check_layer(orc, "w4a16", inp["x"], logits, k, ob, routed, ws, np.arange(T, dtype=np.int32), what="routed")
    wg, wu = (synth.make_weights(1, Fs, d, seed=33 + i, device="cuda")[0] for i in range(2))
    wd = synth.make_weights(1, d, Fs, seed=35, device="cuda")[0]
    out = routed.clone()
    wss = torch.empty(max(16, lib.load().moe_shared_expert_workspace_size(T, Fs)), dtype=torch.uint8, device="cuda")
    lib.moe_shared_expert(inp["x"], wg, wu, wd, out, ws=wss)
    torch.cuda.synchronize()
    _check_shared(orc, inp["x"], wg, wu, wd, routed, out, wss, "block")


def test_shared_expert_deterministic():
    """The narrow tiles' split-K sums their partials in rank order: the same
    output bits on every call (decode size, K split over clusters)."""
    T, d, Fs = 64, 4096, 1536
    x = synth.make_x(T, d, seed=7, device="cuda", outlier_frac=0.05)
    wg = synth.make_weights(1, Fs, d, seed=8, device="cuda")[0]
    wu = synth.make_weights(1, Fs, d, seed=9, device="cuda")[0]
    wd = synth.make_weights(1, d, Fs, seed=10, device="cuda")[0]
    routed = synth.make_x(T, d, seed=11, device="cuda")
    ws = torch.empty(max(16, lib.load().moe_shared_expert_workspace_size(T, Fs)), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(3):
        out = routed.clone()
        lib.moe_shared_expert(x, wg, wu, wd, out, ws=ws)
        outs.append(out)
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
