"""CPU oracle for the NVFP4 routed-expert MoE layer -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` leg
of ``bench.py`` may import this module.  The product (the CUDA library and its
binding) never does, and nothing here imports the product.

This file is argument marshalling (numpy <-> C) around ``nvfp4_oracle.c``,
which holds the arithmetic; see that file's header for the sources and the
rounding points.  ``build()`` compiles the C file with gcc (no fast-math, no
FMA contraction) into ``oracle/_build/``.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build", platform.machine())
_SO = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library (host gcc, OpenMP)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _P(t):
    return ctypes.POINTER(t)


class _LayerExtras(ctypes.Structure):
    """Mirror of orc_layer_extras (optional outputs of orc_moe_layer_ex)."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("out_pre", "out_abs", "g_pre", "u_pre", "g_abs", "u_abs", "h",
                                                 "xq", "xs", "hq", "hs", "y_pre", "y_abs")]


def bind(L):
    """Declare the C signatures on a loaded oracle library."""
    i64, i32, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_float
    vp = ctypes.c_void_p
    L.orc_round_bf16.argtypes = [ctypes.c_double]
    L.orc_round_bf16.restype = ctypes.c_double
    L.orc_e2m1_decode.argtypes = [i32]
    L.orc_e2m1_decode.restype = ctypes.c_double
    L.orc_e2m1_encode.argtypes = [f32]
    L.orc_e2m1_encode.restype = i32
    L.orc_e4m3_decode.argtypes = [i32]
    L.orc_e4m3_decode.restype = ctypes.c_double
    L.orc_e4m3_encode_nonneg.argtypes = [f32]
    L.orc_e4m3_encode_nonneg.restype = i32
    L.orc_quantize_tensor.argtypes = [vp, i64, i64, vp, vp, vp]
    L.orc_quantize_rows.argtypes = [vp, i64, i64, vp, vp, vp]
    L.orc_dequantize.argtypes = [vp, vp, i64, i64, vp]
    L.orc_route.argtypes = [vp, i64, i32, i32, vp, vp, vp, vp, vp]
    L.orc_router_logits.argtypes = [vp, i64, i64, vp, i64, vp, vp]
    L.orc_shared_expert.argtypes = [vp, i64, i64, vp, vp, vp, i64, vp, vp]
    L.orc_shared_expert_ex.argtypes = [vp, i64, i64, vp, vp, vp, i64, vp, vp] + [vp] * 7
    L.orc_moe_layer.argtypes = [i32, vp, i64, i64, i64, i32, i32, vp, vp,
                                vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                vp, vp, vp, i64, vp, vp]
    L.orc_moe_layer_ex.argtypes = [i32, vp, i64, i64, i64, i32, i32, vp, vp,
                                   vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                   vp, vp, i32, vp, i64, vp, ctypes.POINTER(_LayerExtras)]
    L.orc_linear.argtypes = [vp, i64, i64, vp, vp, f32, i64, vp, vp, f32, vp]
    L.orc_linear_ex.argtypes = [vp, i64, i64, vp, vp, f32, i64, vp, vp, f32, vp, vp, vp, vp, vp, vp]
    L.orc_num_threads.restype = i32
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(ctypes.CDLL(build()))
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# codecs
# --------------------------------------------------------------------------
def e2m1_decode(code: int) -> float:
    return lib().orc_e2m1_decode(int(code))


def e2m1_encode(v: float) -> int:
    return lib().orc_e2m1_encode(float(v))


def e4m3_decode(b: int) -> float:
    return lib().orc_e4m3_decode(int(b))


def e4m3_encode(v: float) -> int:
    return lib().orc_e4m3_encode_nonneg(float(v))


def round_bf16(v: float) -> float:
    return lib().orc_round_bf16(float(v))


def num_threads() -> int:
    return lib().orc_num_threads()


# --------------------------------------------------------------------------
# quantisation
# --------------------------------------------------------------------------
def quantize_tensor(w_bf16_bits: np.ndarray):
    """ModelOpt NVFP4 recipe on one [N, K] tensor given as uint16 bf16 bits.

    Returns (codes uint8 [N, K/2], scales uint8 [N, K/16], weight_scale_2 float32).
    """
    w = _c(w_bf16_bits, np.uint16)
    N, K = w.shape
    codes = np.zeros((N, K // 2), np.uint8)
    scales = np.zeros((N, K // 16), np.uint8)
    ws2 = np.zeros(1, np.float32)
    lib().orc_quantize_tensor(_ptr(w), N, K, _ptr(codes), _ptr(scales), _ptr(ws2))
    return codes, scales, np.float32(ws2[0])


def quantize_rows(x_bf16_bits: np.ndarray, gs_per_row: np.ndarray):
    """Static-scale NVFP4 quantisation of each row r with tensor scale gs[r]."""
    x = _c(x_bf16_bits, np.uint16)
    M, K = x.shape
    gs = _c(gs_per_row, np.float32)
    assert gs.shape == (M,)
    codes = np.zeros((M, K // 2), np.uint8)
    scales = np.zeros((M, K // 16), np.uint8)
    lib().orc_quantize_rows(_ptr(x), M, K, _ptr(gs), _ptr(codes), _ptr(scales))
    return codes, scales


def dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """dec(q) * dec(s) in fp64, without the tensor scale, shape [N, K]."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    N = codes.shape[0]
    K = codes.shape[1] * 2
    out = np.zeros((N, K), np.float64)
    lib().orc_dequantize(_ptr(codes), _ptr(scales), N, K, _ptr(out))
    return out


# --------------------------------------------------------------------------
# routing
# --------------------------------------------------------------------------
def router_logits(x_bf16_bits: np.ndarray, w_bf16_bits: np.ndarray):
    """fp64 logits [T, E] = x @ w^T of bf16 bit patterns x [T, d], w [E, d],
    and sum_k |x w| per element (the error-bound scale of an fp32 sum)."""
    x = _c(x_bf16_bits, np.uint16)
    w = _c(w_bf16_bits, np.uint16)
    T, d = x.shape
    E = w.shape[0]
    out = np.zeros((T, E), np.float64)
    absum = np.zeros((T, E), np.float64)
    lib().orc_router_logits(_ptr(x), T, d, _ptr(w), E, _ptr(out), _ptr(absum))
    return out, absum


def route(logits: np.ndarray, top_k: int):
    """Softmax/top-k/renormalise, then the stable permutation by expert.

    Returns dict(ids [T,k] i32, w [T,k] f32, offsets [E+1] i32,
    row_to_slot [T*k] i32, slot_to_row [T*k] i32).
    """
    lg = _c(logits, np.float32)
    T, E = lg.shape
    ids = np.zeros((T, top_k), np.int32)
    w = np.zeros((T, top_k), np.float32)
    offsets = np.zeros(E + 1, np.int32)
    r2s = np.zeros(T * top_k, np.int32)
    s2r = np.zeros(T * top_k, np.int32)
    lib().orc_route(_ptr(lg), T, E, top_k, _ptr(ids), _ptr(w), _ptr(offsets), _ptr(r2s), _ptr(s2r))
    return dict(ids=ids, w=w, offsets=offsets, row_to_slot=r2s, slot_to_row=s2r)


# --------------------------------------------------------------------------
# the layer
# --------------------------------------------------------------------------
def moe_layer(mode: str, x_bf16_bits, ids, w, bank, tokens=None, is13=None, is2=None,
              want_h: bool = False):
    """Routed-expert layer for ``tokens`` (default: all).

    ``bank`` is a dict with gate/up/down entries, each (codes, scales, ws2)
    stacked over experts: gate/up codes [E, F, d/2], down codes [E, d, F/2].
    Returns out float32 [n_tokens, d] (bf16 values), and h [n, k, F] if asked.
    """
    x = _c(x_bf16_bits, np.uint16)
    T, d = x.shape
    ids = _c(ids, np.int32)
    w = _c(w, np.float32)
    k = ids.shape[1]
    gq, gs, g2 = bank["gate"]
    uq, us, u2 = bank["up"]
    dq, ds, d2 = bank["down"]
    E, F = gq.shape[0], gq.shape[1]
    arrs = [_c(a, np.uint8) for a in (gq, gs, uq, us, dq, ds)]
    ws2s = [_c(a, np.float32) for a in (g2, u2, d2)]
    if tokens is None:
        tokens = np.arange(T, dtype=np.int32)
    tokens = _c(tokens, np.int32)
    n = tokens.shape[0]
    m = 0 if mode == "w4a16" else 1
    if m == 1:
        is13 = _c(is13, np.float32)
        is2 = _c(is2, np.float32)
    out = np.zeros((n, d), np.float32)
    h = np.zeros((n, k, F), np.float32) if want_h else None
    lib().orc_moe_layer(m, _ptr(x), T, d, F, E, k, _ptr(ids), _ptr(w),
                        _ptr(arrs[0]), _ptr(arrs[1]), _ptr(ws2s[0]),
                        _ptr(arrs[2]), _ptr(arrs[3]), _ptr(ws2s[1]),
                        _ptr(arrs[4]), _ptr(arrs[5]), _ptr(ws2s[2]),
                        _ptr(is13) if m == 1 else None, _ptr(is2) if m == 1 else None,
                        _ptr(tokens), n, _ptr(out), _ptr(h))
    return (out, h) if want_h else out


def moe_layer_ex(mode: str, x_bf16_bits, ids, w, bank, tokens=None, is13=None, is2=None, round_y=False):
    """The layer for ``tokens`` with every optional output (see
    ``orc_moe_layer_ex``): dict with out [n, d] (bf16 values), out_pre and
    out_abs [n, d] fp64, g_pre / u_pre / g_abs / u_abs [n, k, F] fp64,
    h [n, k, F], y_pre / y_abs [n, k, d] fp64, and for W4A4 the pairs'
    NVFP4 rows xq [n, k, d/2], xs [n, k, d/16], hq [n, k, F/2],
    hs [n, k, F/16].  round_y: each Y rounded to bf16 before the weighted
    sum (the R3 rounding point of the prompt-shaped path)."""
    x = _c(x_bf16_bits, np.uint16)
    T, d = x.shape
    ids = _c(ids, np.int32)
    w = _c(w, np.float32)
    k = ids.shape[1]
    gq, gs, g2 = bank["gate"]
    uq, us, u2 = bank["up"]
    dq, ds, d2 = bank["down"]
    E, F = gq.shape[0], gq.shape[1]
    arrs = [_c(a, np.uint8) for a in (gq, gs, uq, us, dq, ds)]
    ws2s = [_c(a, np.float32) for a in (g2, u2, d2)]
    if tokens is None:
        tokens = np.arange(T, dtype=np.int32)
    tokens = _c(tokens, np.int32)
    n = tokens.shape[0]
    m = 0 if mode == "w4a16" else 1
    if m == 1:
        is13 = _c(is13, np.float32)
        is2 = _c(is2, np.float32)
    r = dict(out=np.zeros((n, d), np.float32), out_pre=np.zeros((n, d)), out_abs=np.zeros((n, d)),
             g_pre=np.zeros((n, k, F)), u_pre=np.zeros((n, k, F)), g_abs=np.zeros((n, k, F)),
             u_abs=np.zeros((n, k, F)), h=np.zeros((n, k, F), np.float32), y_pre=np.zeros((n, k, d)),
             y_abs=np.zeros((n, k, d)))
    if m == 1:
        r.update(xq=np.zeros((n, k, d // 2), np.uint8), xs=np.zeros((n, k, d // 16), np.uint8),
                 hq=np.zeros((n, k, F // 2), np.uint8), hs=np.zeros((n, k, F // 16), np.uint8))
    ex = _LayerExtras(*[_ptr(r.get(nm)) for nm, _ in _LayerExtras._fields_])
    lib().orc_moe_layer_ex(m, _ptr(x), T, d, F, E, k, _ptr(ids), _ptr(w),
                           _ptr(arrs[0]), _ptr(arrs[1]), _ptr(ws2s[0]),
                           _ptr(arrs[2]), _ptr(arrs[3]), _ptr(ws2s[1]),
                           _ptr(arrs[4]), _ptr(arrs[5]), _ptr(ws2s[2]),
                           _ptr(is13) if m == 1 else None, _ptr(is2) if m == 1 else None, 1 if round_y else 0,
                           _ptr(tokens), n, _ptr(r["out"]), ctypes.byref(ex))
    return r


def shared_expert(x_bf16_bits, wg_bits, wu_bits, wd_bits, routed_bf16_bits):
    """BF16 shared-expert MLP added to the routed output, fp32 [T, d] of
    bf16 values: bf16(routed + bf16(silu(bf16 xWg^T) * bf16 xWu^T) Wd^T)."""
    x = _c(x_bf16_bits, np.uint16)
    wg, wu, wd = (_c(w, np.uint16) for w in (wg_bits, wu_bits, wd_bits))
    r = _c(routed_bf16_bits, np.uint16)
    T, d = x.shape
    Fs = wg.shape[0]
    out = np.zeros((T, d), np.float32)
    lib().orc_shared_expert(_ptr(x), T, d, _ptr(wg), _ptr(wu), _ptr(wd), Fs, _ptr(r), _ptr(out))
    return out


def shared_expert_ex(x_bf16_bits, wg_bits, wu_bits, wd_bits, routed_bf16_bits):
    """``shared_expert`` with its optional outputs: dict with out, out_pre,
    out_abs [T, d] and g_pre, u_pre, g_abs, u_abs, h [T, Fs]."""
    x = _c(x_bf16_bits, np.uint16)
    wg, wu, wd = (_c(w, np.uint16) for w in (wg_bits, wu_bits, wd_bits))
    rt = _c(routed_bf16_bits, np.uint16)
    T, d = x.shape
    Fs = wg.shape[0]
    r = dict(out=np.zeros((T, d), np.float32), out_pre=np.zeros((T, d)), out_abs=np.zeros((T, d)),
             g_pre=np.zeros((T, Fs)), u_pre=np.zeros((T, Fs)), g_abs=np.zeros((T, Fs)), u_abs=np.zeros((T, Fs)),
             h=np.zeros((T, Fs), np.float32))
    lib().orc_shared_expert_ex(_ptr(x), T, d, _ptr(wg), _ptr(wu), _ptr(wd), Fs, _ptr(rt), _ptr(r["out"]),
                               *[_ptr(r[n]) for n in ("out_pre", "out_abs", "g_pre", "u_pre", "g_abs", "u_abs",
                                                      "h")])
    return r


def linear(x_bf16_bits, wq, ws, ws2, wup=None):
    """Dense NVFP4 linear; with ``wup`` = (codes, scales, ws2) it returns
    bf16(silu(bf16 G) * bf16 U) instead of bf16(ws2 * x W^T)."""
    x = _c(x_bf16_bits, np.uint16)
    M, K = x.shape
    wq = _c(wq, np.uint8)
    ws = _c(ws, np.uint8)
    N = wq.shape[0]
    out = np.zeros((M, N), np.float32)
    if wup is not None:
        uq, us, u2 = _c(wup[0], np.uint8), _c(wup[1], np.uint8), float(wup[2])
    else:
        uq = us = None
        u2 = 0.0
    lib().orc_linear(_ptr(x), M, K, _ptr(wq), _ptr(ws), float(ws2), N, _ptr(uq), _ptr(us), u2,
                     _ptr(out))
    return out


def linear_ex(x_bf16_bits, wq, ws, ws2, wup=None):
    """``linear`` with its optional outputs: dict with out [M, N] (bf16
    values), pre (before the final rounding), g_pre / g_abs and, with
    ``wup``, u_pre / u_abs, all [M, N] fp64."""
    x = _c(x_bf16_bits, np.uint16)
    M, K = x.shape
    wq = _c(wq, np.uint8)
    ws = _c(ws, np.uint8)
    N = wq.shape[0]
    r = dict(out=np.zeros((M, N), np.float32), pre=np.zeros((M, N)), g_pre=np.zeros((M, N)),
             g_abs=np.zeros((M, N)))
    if wup is not None:
        uq, us, u2 = _c(wup[0], np.uint8), _c(wup[1], np.uint8), float(wup[2])
        r.update(u_pre=np.zeros((M, N)), u_abs=np.zeros((M, N)))
    else:
        uq = us = None
        u2 = 0.0
    lib().orc_linear_ex(_ptr(x), M, K, _ptr(wq), _ptr(ws), float(ws2), N, _ptr(uq), _ptr(us), u2,
                        _ptr(r["out"]), _ptr(r["pre"]), _ptr(r["g_pre"]), _ptr(r.get("u_pre")),
                        _ptr(r["g_abs"]), _ptr(r.get("u_abs")))
    return r
