"""nvfp4_quantize_weights_noalloc: the weight recipe for callers that cannot
allocate device memory (it keeps its scratch in a fixed array inside the
library).  Called through the C ABI and compared with
nvfp4_quantize_weights on two calls in a row -- the second call must not see
the first call's scratch.  The outputs are codes, e4m3 scales and fp32
weight_scale_2, so the comparison is exact.  This file is collected last."""
import ctypes

import numpy as np
import pytest
import torch

import serving_nvfp4_routed_gb300 as lib
from serving_nvfp4_routed_gb300 import _lib, synth

pytestmark = pytest.mark.gpu


def _noalloc(w):
    L = _lib.load()
    B, N, K = w.shape
    codes = torch.empty(B, N, K // 2, dtype=torch.uint8, device=w.device)
    scales = torch.empty(B, N, K // 16, dtype=torch.uint8, device=w.device)
    ws2 = torch.empty(B, dtype=torch.float32, device=w.device)
    st = L.nvfp4_quantize_weights_noalloc(ctypes.c_void_p(w.data_ptr()), B, N, K, ctypes.c_void_p(codes.data_ptr()),
                                          ctypes.c_void_p(scales.data_ptr()), ctypes.c_void_p(ws2.data_ptr()),
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, _lib.STATUS.get(st, st)
    return codes, scales, ws2


def test_noalloc_matches_workspace_entry_point_twice():
    # first call: large values; second call: much smaller ones, so stale
    # running maxima from the first call would change every scale
    w1 = synth.make_weights(5, 96, 512, seed=71, device="cuda") * 50
    w2 = synth.make_weights(3, 128, 256, seed=72, device="cuda")
    for w in (w1, w2):
        c, s, g = _noalloc(w)
        ref = lib.nvfp4_quantize_weights(w)
        torch.cuda.synchronize()
        assert torch.equal(g, ref.weight_scale_2)
        assert torch.equal(s, ref.scales)
        assert torch.equal(c, ref.codes)


def test_noalloc_rejects_batch_beyond_limit():
    L = _lib.load()
    limit = L.nvfp4_quantize_weights_noalloc_max_batch()
    assert limit == 4096
    p = ctypes.c_void_p(0x10000)
    assert L.nvfp4_quantize_weights_noalloc(p, limit + 1, 16, 16, p, p, p, None) == 2  # NVFP4_ERR_SHAPE
