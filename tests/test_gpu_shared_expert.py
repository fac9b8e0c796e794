"""GPU parity: the BF16 shared-expert MLP (tcgen05 bf16 GEMMs) added to a
routed output, against the oracle with the same rounding points (G, U, h,
out), within the layer tolerance."""
import numpy as np
import pytest
import torch

import serving_nvfp4_routed_gb300 as lib
from serving_nvfp4_routed_gb300 import synth

from gpu_util import assert_layer_close, bf16_to_f32

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,d,Fs", [(1, 256, 128), (100, 512, 256), (300, 1024, 384), (129, 4096, 1536),
                                    (1280, 2048, 256)])
def test_shared_expert(orc, T, d, Fs):
    """Single and ragged token tiles, one and several column tiles in both
    GEMMs, K from 128 to 4096; the small batches run 64-wide tiles, the last
    case (ten token tiles) the 256-wide ones."""
    x = synth.make_x(T, d, seed=T + d, device="cuda", outlier_frac=0.05)
    wg = synth.make_weights(1, Fs, d, seed=Fs + 1, device="cuda")[0]
    wu = synth.make_weights(1, Fs, d, seed=Fs + 2, device="cuda")[0] * 2
    wd = synth.make_weights(1, d, Fs, seed=Fs + 3, device="cuda")[0]
    routed = synth.make_x(T, d, seed=T + d + 1, device="cuda")
    ref = orc.shared_expert(synth.bf16_bits(x), synth.bf16_bits(wg), synth.bf16_bits(wu), synth.bf16_bits(wd),
                            synth.bf16_bits(routed))
    out = routed.clone()
    lib.moe_shared_expert(x, wg, wu, wd, out)
    assert_layer_close(bf16_to_f32(out), ref, "shared expert")


def test_routed_layer_then_shared_expert(orc):
    """The MoE block end to end on the library: router GEMM -> routed W4A16
    layer -> shared expert; checked against the oracle step by step on the
    library's own intermediate results."""
    T, d, E, k, F, Fs = 64, 512, 16, 4, 256, 256
    s = synth.MoEShape(T, d, E, k, F)
    inp = synth.moe_inputs(s, 31, device="cuda")
    from gpu_util import gpu_bank, oracle_bank
    banks = dict(gate=inp["gate"], up=inp["up"], down=inp["down"])
    gw = gpu_bank(lib, banks)
    wr = synth.make_weights(1, E, d, seed=32, device="cuda")[0]
    logits = lib.moe_router_logits(inp["x"], wr)
    routed = lib.nvfp4_moe_w4a16(inp["x"], logits, k, gw)
    r = orc.route(logits.cpu().numpy(), k)
    ob = oracle_bank(orc, banks, np.arange(E))
    ref_routed = orc.moe_layer("w4a16", synth.bf16_bits(inp["x"]), r["ids"], r["w"], ob)
    assert_layer_close(bf16_to_f32(routed), ref_routed, "routed")
    wg, wu = (synth.make_weights(1, Fs, d, seed=33 + i, device="cuda")[0] for i in range(2))
    wd = synth.make_weights(1, d, Fs, seed=35, device="cuda")[0]
    out = routed.clone()
    lib.moe_shared_expert(inp["x"], wg, wu, wd, out)
    ref = orc.shared_expert(synth.bf16_bits(inp["x"]), synth.bf16_bits(wg), synth.bf16_bits(wu),
                            synth.bf16_bits(wd), synth.bf16_bits(routed))
    assert_layer_close(bf16_to_f32(out), ref, "block")
