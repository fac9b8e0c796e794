"""The C ABI: the library builds, loads, exports every declared symbol, and
rejects bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

from serving_nvfp4_routed_gb300 import _lib
from serving_nvfp4_routed_gb300 import build as nvbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    nvbuild.build()
    return _lib.load()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(\w+)\s*\([^;{]*\)\s*;", src))
    return names - {"if", "while", "for", "return", "sizeof"}


def test_every_declared_symbol_is_exported(L):
    decl = _declared()
    assert {"nvfp4_quantize_weights", "nvfp4_quantize_act", "moe_route_permute", "nvfp4_moe_w4a16",
            "nvfp4_moe_w4a4", "nvfp4_linear"} <= decl
    for name in decl:
        assert hasattr(L, name), name
    assert set(_lib.EXPORTS) == decl


def test_status_strings(L):
    for code, name in _lib.STATUS.items():
        assert _lib.status_string(code) == name


def test_workspace_sizes(L):
    s16 = L.nvfp4_moe_workspace_size(64, 288, 8, 4096, 1536, 0)
    s4 = L.nvfp4_moe_workspace_size(64, 288, 8, 4096, 1536, 1)
    R = 64 * 8
    assert s16 >= R * 1536 * 2 + 64 * 4096 * 4
    assert s4 >= R * (4096 // 2 + 4096 // 16)
    assert L.nvfp4_moe_workspace_size(64, 288, 8, 4096, 1536, 2) == 0
    assert L.moe_route_permute_workspace_size(16384, 288, 8) > 0
    assert L.nvfp4_quantize_weights_workspace_size(288, 1536, 4096) >= 288 * 4


def _fake(addr=0x10000):
    return ctypes.c_void_p(addr)


def _moew(E=8, d=256, F=128, addr=0x20000):
    w = _lib._W(addr, addr, addr)
    return _lib._MoEW(w, w, w, E, d, F)


def test_moe_host_validation(L):
    big = 1 << 40
    p = _fake()
    mw = _moew()
    call = lambda T, k, w=mw, x=p, out=p, ws=p, wsb=big: L.nvfp4_moe_w4a16(x, T, p, k, ctypes.byref(w), out, ws,
                                                                            wsb, None, None)
    assert call(0, 2) == 0                       # T = 0 is a no-op
    assert call(4, 0) == 2                       # top_k < 1
    assert call(4, 9) == 2                       # top_k > E
    assert call(4, 2, w=_moew(d=96)) == 2        # d % 64
    assert call(4, 2, w=_moew(F=100)) == 2       # F % 64
    assert call(4, 2, w=_moew(E=2000)) == 2      # E > 1024
    assert call(4, 2, x=None) == 1               # NULL x
    assert call(4, 2, x=_fake(0x10008)) == 3     # misaligned x
    assert call(4, 2, wsb=16) == 4               # workspace too small
    assert L.nvfp4_moe_w4a16(p, -1, p, 2, ctypes.byref(mw), p, p, big, None, None) == 1
    assert L.nvfp4_moe_w4a4(p, 4, p, 2, ctypes.byref(mw), None, p, p, p, big, None, None) == 1


def test_other_host_validation(L):
    p = _fake()
    big = 1 << 40
    assert L.nvfp4_quantize_weights(p, 1, 4, 24, p, p, p, p, big, None) == 2  # K % 16
    assert L.nvfp4_quantize_weights(p, 1, 4, 32, p, p, p, p, 0, None) == 4
    assert L.nvfp4_quantize_weights(_fake(0x10004), 1, 4, 32, p, p, p, p, big, None) == 3
    assert L.nvfp4_quantize_weights(None, 1, 4, 32, p, p, p, p, big, None) == 1
    assert L.nvfp4_quantize_weights(p, 0, 4, 32, p, p, p, p, 0, None) == 0
    assert L.nvfp4_quantize_weights(p, 65536, 4, 32, p, p, p, p, big, None) == 2  # one grid row per tensor
    assert L.nvfp4_quantize_weights_noalloc(p, 4097, 4, 32, p, p, p, None) == 2  # beyond the fixed scratch
    assert L.nvfp4_quantize_weights_noalloc(p, 1, 4, 24, p, p, p, None) == 2
    assert L.nvfp4_set_kernel_choice(5) == 1 and L.nvfp4_set_kernel_choice(-1) == 1
    assert L.nvfp4_set_kernel_choice(2) == 0 and L.nvfp4_set_kernel_choice(0) == 0
    assert L.nvfp4_quantize_act(p, 4, 40, None, 1, p, None, 0, p, p, None) == 2
    assert L.nvfp4_quantize_act(p, 4, 32, p, 0, p, None, 0, p, p, None) == 1
    assert L.moe_route_permute(p, 4, 8, 9, p, p, p, p, p, p, big, None) == 2
    assert L.moe_route_permute(p, 4, 2000, 8, p, p, p, p, p, p, big, None) == 2
    assert L.moe_route_permute(p, 4, 8, 2, p, p, p, p, p, p, 0, None) == 4
    assert L.moe_router_logits(p, 4, 100, p, 8, p, None, None) == 2  # d % 64
    assert L.moe_router_logits(p, 4, 128, p, 600, p, None, None) == 2  # E > 512
    assert L.moe_router_logits(p, -1, 128, p, 8, p, None, None) == 1
    assert L.moe_router_logits(None, 4, 128, p, 8, p, None, None) == 1
    assert L.moe_router_logits(_fake(0x10004), 4, 128, p, 8, p, None, None) == 3
    assert L.moe_router_logits(p, 0, 128, p, 8, p, None, None) == 0  # no-op
    assert L.moe_shared_expert(p, 4, 384, p, p, p, 128, p, p, big, None, None) == 2  # d % 256
    assert L.moe_shared_expert(p, 4, 256, p, p, p, 192, p, p, big, None, None) == 2  # Fs % 128
    assert L.moe_shared_expert(p, 4, 256, p, p, p, 128, p, p, 0, None, None) == 4
    assert L.moe_shared_expert(p, 0, 256, p, p, p, 128, p, p, 0, None, None) == 0  # no-op
    w = _lib._W(0x20000, 0x20000, 0x20000)
    assert L.nvfp4_linear(p, 4, 96, ctypes.byref(w), 16, None, p, p, big, None) == 2
    assert L.nvfp4_linear(p, 4, 64, ctypes.byref(w), 24, None, p, p, big, None) == 2
    assert L.nvfp4_linear(p, 4, 64, ctypes.byref(w), 16, None, p, p, 0, None) == 4
    assert L.nvfp4_linear(p, 0, 64, ctypes.byref(w), 16, None, p, p, 0, None) == 0


def test_no_cpu_path():
    import torch

    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        _lib.nvfp4_quantize_weights(x)
