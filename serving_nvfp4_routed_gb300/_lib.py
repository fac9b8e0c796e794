"""Thin Python binding of libnvfp4moe (ctypes).

Argument marshalling only: torch supplies device memory and the current CUDA
stream; every step of the layer runs in the library's CUDA kernels.  There is
no CPU fallback: if the shared library is missing or the tensors are not on
a CUDA device, the calls raise.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import platform
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", platform.machine(), "libnvfp4moe.so")

STATUS = {0: "NVFP4_OK", 1: "NVFP4_ERR_INVALID_ARG", 2: "NVFP4_ERR_SHAPE", 3: "NVFP4_ERR_ALIGN",
          4: "NVFP4_ERR_WORKSPACE", 5: "NVFP4_ERR_UNSUPPORTED", 6: "NVFP4_ERR_CUDA",
          7: "NVFP4_ERR_TIMEOUT", 8: "NVFP4_ERR_DEVICE_INPUT"}

EXPORTS = ("nvfp4_quantize_weights", "nvfp4_quantize_weights_workspace_size", "nvfp4_quantize_act",
           "moe_route_permute", "moe_route_permute_workspace_size", "nvfp4_moe_w4a16", "nvfp4_moe_w4a4",
           "nvfp4_moe_workspace_size", "nvfp4_moe_workspace_views", "nvfp4_moe_workspace_intermediates",
           "nvfp4_set_kernel_choice", "nvfp4_linear",
           "nvfp4_linear_workspace_size", "nvfp4_status_string", "nvfp4_launch_count",
           "nvfp4_profile_enable", "nvfp4_profile_collect", "nvfp4_quantize_weights_noalloc",
           "nvfp4_quantize_weights_noalloc_max_batch", "nvfp4_selftest_bounded_wait", "moe_router_logits",
           "moe_shared_expert", "moe_shared_expert_workspace_size", "moe_gather_rows", "moe_combine_rows")


class Nvfp4Error(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} returned {STATUS.get(code, code)}")
        self.code = code


class _W(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("weight_scale_2", ctypes.c_void_p)]


class _MoEW(ctypes.Structure):
    _fields_ = [("gate", _W), ("up", _W), ("down", _W), ("E", ctypes.c_int), ("d", ctypes.c_int),
                ("F", ctypes.c_int)]


_lib = None
_lock = threading.Lock()


def load(path: str = LIB_PATH):
    """Load the shared library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise ImportError(f"libnvfp4moe is not built ({path}); run serving_nvfp4_routed_gb300/build.py")
        L = ctypes.CDLL(path)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.nvfp4_quantize_weights.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, sz, vp]
        L.nvfp4_quantize_weights_workspace_size.argtypes = [i32, i32, i32]
        L.nvfp4_quantize_weights_workspace_size.restype = sz
        L.nvfp4_quantize_weights_noalloc.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp]
        L.nvfp4_quantize_weights_noalloc_max_batch.restype = i32
        L.nvfp4_quantize_act.argtypes = [vp, i32, i32, vp, i32, vp, vp, i32, vp, vp, vp]
        L.moe_route_permute.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp]
        L.moe_route_permute_workspace_size.argtypes = [i32, i32, i32]
        L.moe_route_permute_workspace_size.restype = sz
        L.nvfp4_moe_w4a16.argtypes = [vp, i32, vp, i32, ctypes.POINTER(_MoEW), vp, vp, sz, vp, vp]
        L.nvfp4_moe_w4a4.argtypes = [vp, i32, vp, i32, ctypes.POINTER(_MoEW), vp, vp, vp, vp, sz, vp, vp]
        L.nvfp4_moe_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
        L.nvfp4_moe_workspace_size.restype = sz
        L.nvfp4_moe_workspace_views.argtypes = [vp, i32, i32, i32, i32, i32, i32] + [ctypes.POINTER(vp)] * 5
        L.nvfp4_moe_workspace_intermediates.argtypes = [vp, i32, i32, i32, i32, i32, i32] + [ctypes.POINTER(vp)] * 5
        L.nvfp4_set_kernel_choice.argtypes = [i32]
        L.moe_gather_rows.argtypes = [vp, i32, i32, vp, i32, vp, i32, vp, vp, vp]
        L.moe_combine_rows.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp]
        L.nvfp4_linear.argtypes = [vp, i32, i32, ctypes.POINTER(_W), i32, ctypes.POINTER(_W), vp, vp, sz, vp]
        L.nvfp4_linear_workspace_size.argtypes = [i32, i32, i32]
        L.nvfp4_linear_workspace_size.restype = sz
        L.nvfp4_status_string.argtypes = [i32]
        L.nvfp4_status_string.restype = ctypes.c_char_p
        L.nvfp4_launch_count.restype = ctypes.c_uint64
        L.nvfp4_selftest_bounded_wait.argtypes = [vp, vp]
        L.moe_router_logits.argtypes = [vp, i32, i32, vp, i32, vp, vp, vp]
        L.moe_shared_expert.argtypes = [vp, i32, i32, vp, vp, vp, i32, vp, vp, sz, vp, vp]
        L.moe_shared_expert_workspace_size.argtypes = [i32, i32]
        L.moe_shared_expert_workspace_size.restype = sz
        L.nvfp4_profile_enable.argtypes = [i32]
        L.nvfp4_profile_collect.argtypes = [i32, ctypes.c_char_p, ctypes.POINTER(i32),
                                            ctypes.POINTER(ctypes.c_double)]
        L.nvfp4_profile_collect.restype = i32
        _lib = L
        return L


def _check(fn, code):
    if code != 0:
        raise Nvfp4Error(fn, code)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("libnvfp4moe takes CUDA tensors only (no CPU path)")


def _empty(shape, dtype, device):
    return torch.empty(shape, dtype=dtype, device=device)


# ---------------------------------------------------------------------------
@dataclasses.dataclass
class NVFP4Tensor:
    """Stacked NVFP4 tensors: codes [E, N, K/2] u8, scales [E, N, K/16] u8 (e4m3
    bits), weight_scale_2 [E] f32."""
    codes: torch.Tensor
    scales: torch.Tensor
    weight_scale_2: torch.Tensor

    def _c(self):
        return _W(self.codes.data_ptr(), self.scales.data_ptr(), self.weight_scale_2.data_ptr())


@dataclasses.dataclass
class MoEWeights:
    gate: NVFP4Tensor
    up: NVFP4Tensor
    down: NVFP4Tensor

    @property
    def E(self):
        return self.gate.codes.shape[0]

    @property
    def F(self):
        return self.gate.codes.shape[1]

    @property
    def d(self):
        return self.gate.codes.shape[2] * 2

    def _c(self):
        return _MoEW(self.gate._c(), self.up._c(), self.down._c(), self.E, self.d, self.F)


# ---------------------------------------------------------------------------
def nvfp4_quantize_weights(w: torch.Tensor, stream=None) -> NVFP4Tensor:
    """ModelOpt NVFP4 recipe on bf16 [N, K] or [batch, N, K] (one tensor scale per batch entry)."""
    L = load()
    _cuda(w)
    w3 = w.unsqueeze(0) if w.dim() == 2 else w
    w3 = w3.contiguous()
    B, N, K = w3.shape
    codes = _empty((B, N, K // 2), torch.uint8, w.device)
    scales = _empty((B, N, K // 16), torch.uint8, w.device)
    ws2 = _empty((B,), torch.float32, w.device)
    wsb = L.nvfp4_quantize_weights_workspace_size(B, N, K)
    ws = _empty((max(wsb, 16),), torch.uint8, w.device)
    _check("nvfp4_quantize_weights",
           L.nvfp4_quantize_weights(_p(w3.view(torch.int16)), B, N, K, _p(codes), _p(scales), _p(ws2), _p(ws),
                                    wsb, _stream(stream)))
    return NVFP4Tensor(codes, scales, ws2)


def nvfp4_quantize_act(x: torch.Tensor, input_scale: torch.Tensor, M: int | None = None,
                       row_to_slot: torch.Tensor | None = None, top_k: int = 1,
                       expert_offsets: torch.Tensor | None = None, stream=None):
    """Static-scale NVFP4 quantisation of (optionally gathered) rows of bf16 x."""
    L = load()
    _cuda(x, input_scale, row_to_slot, expert_offsets)
    x = x.contiguous()
    K = x.shape[-1]
    if M is None:
        M = row_to_slot.numel() if row_to_slot is not None else x.shape[0]
    codes = _empty((M, K // 2), torch.uint8, x.device)
    scales = _empty((M, K // 16), torch.uint8, x.device)
    E = 0 if expert_offsets is None else expert_offsets.numel() - 1
    _check("nvfp4_quantize_act",
           L.nvfp4_quantize_act(_p(x.view(torch.int16)), M, K, _p(row_to_slot), top_k, _p(input_scale),
                                _p(expert_offsets), E, _p(codes), _p(scales), _stream(stream)))
    return codes, scales


def moe_router_logits(x: torch.Tensor, w_router: torch.Tensor, out=None, d_status=None, stream=None) -> torch.Tensor:
    """fp32 logits [T, E] = x [T, d] (bf16) @ w_router [E, d] (bf16)^T."""
    L = load()
    _cuda(x, w_router)
    x, w_router = x.contiguous(), w_router.contiguous()
    T, d = x.shape
    E = w_router.shape[0]
    if out is None:
        out = _empty((T, E), torch.float32, x.device)
    _check("moe_router_logits",
           L.moe_router_logits(_p(x), T, d, _p(w_router), E, _p(out), _p(d_status) if d_status is not None else None,
                               _stream(stream)))
    return out


def moe_shared_expert(x: torch.Tensor, w_gate: torch.Tensor, w_up: torch.Tensor, w_down: torch.Tensor,
                      out: torch.Tensor, ws=None, d_status=None, stream=None) -> torch.Tensor:
    """out[T, d] (bf16, the routed layer's result) += the BF16 shared-expert
    MLP of x [T, d]: bf16(silu(bf16 x Wg^T) * bf16 x Wu^T) Wd^T, in place."""
    L = load()
    _cuda(x, w_gate, w_up, w_down, out)
    x, w_gate, w_up, w_down = (t.contiguous() for t in (x, w_gate, w_up, w_down))
    assert out.is_contiguous()
    T, d = x.shape
    Fs = w_gate.shape[0]
    wsb = L.moe_shared_expert_workspace_size(T, Fs)
    if ws is None:
        ws = _empty((max(wsb, 16),), torch.uint8, x.device)
    _check("moe_shared_expert",
           L.moe_shared_expert(_p(x), T, d, _p(w_gate), _p(w_up), _p(w_down), Fs, _p(out), _p(ws), ws.numel(),
                               _p(d_status) if d_status is not None else None, _stream(stream)))
    return out


def moe_route_permute(logits: torch.Tensor, top_k: int, stream=None) -> dict:
    L = load()
    _cuda(logits)
    logits = logits.contiguous()
    T, E = logits.shape
    dev = logits.device
    R = T * top_k
    out = dict(ids=_empty((T, top_k), torch.int32, dev), w=_empty((T, top_k), torch.float32, dev),
               offsets=_empty((E + 1,), torch.int32, dev), row_to_slot=_empty((max(R, 1),), torch.int32, dev),
               slot_to_row=_empty((max(R, 1),), torch.int32, dev))
    wsb = L.moe_route_permute_workspace_size(T, E, top_k)
    ws = _empty((max(wsb, 16),), torch.uint8, dev)
    _check("moe_route_permute",
           L.moe_route_permute(_p(logits), T, E, top_k, _p(out["ids"]), _p(out["w"]), _p(out["offsets"]),
                               _p(out["row_to_slot"]), _p(out["slot_to_row"]), _p(ws), wsb, _stream(stream)))
    out["row_to_slot"] = out["row_to_slot"][:R]
    out["slot_to_row"] = out["slot_to_row"][:R]
    return out


def moe_gather_rows(x: torch.Tensor, row_to_slot: torch.Tensor, top_k: int, expert_offsets=None, stream=None):
    """Routed rows in the permutation's order: rows[r] = x[row_to_slot[r] // top_k]
    (bf16 [R, d]), and with expert_offsets the expert of each row (int32 [R])."""
    L = load()
    _cuda(x, row_to_slot, expert_offsets)
    x = x.contiguous()
    T, d = x.shape
    R = T * top_k
    rows = _empty((R, d), torch.bfloat16, x.device)
    eor = _empty((max(R, 1),), torch.int32, x.device) if expert_offsets is not None else None
    E = 0 if expert_offsets is None else expert_offsets.numel() - 1
    _check("moe_gather_rows",
           L.moe_gather_rows(_p(x.view(torch.int16)), T, d, _p(row_to_slot), top_k, _p(expert_offsets), E,
                             _p(rows.view(torch.int16)), _p(eor), _stream(stream)))
    return rows, (eor[:R] if eor is not None else None)


def moe_combine_rows(y: torch.Tensor, slot_to_row: torch.Tensor, topk_w: torch.Tensor, T: int, top_k: int,
                     out=None, stream=None):
    """out[t] = bf16(sum_j topk_w[t, j] * y[slot_to_row[t * k + j]]), fp32 in slot order."""
    L = load()
    _cuda(y, slot_to_row, topk_w, out)
    y = y.contiguous()
    d = y.shape[1]
    if out is None:
        out = _empty((T, d), torch.bfloat16, y.device)
    _check("moe_combine_rows",
           L.moe_combine_rows(_p(y.view(torch.int16)), _p(slot_to_row), _p(topk_w.contiguous()), T, top_k, d,
                              _p(out.view(torch.int16)), _stream(stream)))
    return out


def moe_workspace_size(T, E, top_k, d, F, mode: str) -> int:
    return load().nvfp4_moe_workspace_size(T, E, top_k, d, F, 0 if mode == "w4a16" else 1)


def moe_workspace(T, E, top_k, d, F, mode, device) -> torch.Tensor:
    return _empty((max(moe_workspace_size(T, E, top_k, d, F, mode), 16),), torch.uint8, device)


def moe_workspace_views(ws: torch.Tensor, T, E, top_k, d, F, mode) -> dict:
    """Tensor views of the routing arrays inside an MoE workspace."""
    L = load()
    ptrs = [ctypes.c_void_p() for _ in range(5)]
    _check("nvfp4_moe_workspace_views",
           L.nvfp4_moe_workspace_views(_p(ws), T, E, top_k, d, F, 0 if mode == "w4a16" else 1,
                                       *[ctypes.byref(p) for p in ptrs]))
    base = ws.data_ptr()
    R = T * top_k

    def view(p, n, dtype):
        off = p.value - base
        esz = torch.tensor([], dtype=dtype).element_size()
        return ws[off:off + n * esz].view(dtype)

    return dict(ids=view(ptrs[0], R, torch.int32).view(T, top_k), w=view(ptrs[1], R, torch.float32).view(T, top_k),
                offsets=view(ptrs[2], E + 1, torch.int32), row_to_slot=view(ptrs[3], R, torch.int32),
                slot_to_row=view(ptrs[4], R, torch.int32))


def moe_workspace_intermediates(ws: torch.Tensor, T, E, top_k, d, F, mode) -> dict:
    """Tensor views of the per-row intermediates inside an MoE workspace
    (rows in the permuted, expert-contiguous order): W4A16 h [R, F] bf16;
    W4A4 xq [R, d/2], xs [R, d/16], hq [R, F/2], hs [R, F/16] uint8."""
    L = load()
    ptrs = [ctypes.c_void_p() for _ in range(5)]
    m = 0 if mode == "w4a16" else 1
    _check("nvfp4_moe_workspace_intermediates",
           L.nvfp4_moe_workspace_intermediates(_p(ws), T, E, top_k, d, F, m, *[ctypes.byref(p) for p in ptrs]))
    base = ws.data_ptr()
    R = T * top_k

    def view(p, shape, dtype):
        n = 1
        for v in shape:
            n *= v
        esz = torch.tensor([], dtype=dtype).element_size()
        off = p.value - base
        return ws[off:off + n * esz].view(dtype).view(*shape)

    if m == 0:
        return dict(h=view(ptrs[0], (R, F), torch.bfloat16))
    return dict(xq=view(ptrs[1], (R, d // 2), torch.uint8), xs=view(ptrs[2], (R, d // 16), torch.uint8),
                hq=view(ptrs[3], (R, F // 2), torch.uint8), hs=view(ptrs[4], (R, F // 16), torch.uint8))


KERNEL_CHOICE = {"auto": 0, "gemv": 1, "tc": 2, "gemv_split": 3, "gemv_fused": 4}


def set_kernel_choice(choice: str = "auto") -> None:
    """Which kernels later layer / linear calls run: "auto" (by shape),
    "gemv" (decode-shaped), "tc" (prompt-shaped tensor-core kernels where
    the shapes allow them), or one form of the decode-shaped layer:
    "gemv_split" (gate/up and down as two launches) or "gemv_fused" (one
    persistent launch, d and F multiples of 256).  Process-wide; for tests
    and measurements."""
    _check("nvfp4_set_kernel_choice", load().nvfp4_set_kernel_choice(KERNEL_CHOICE[choice]))


def _moe(mode, x, logits, top_k, weights: MoEWeights, is13=None, is2=None, out=None, ws=None,
         d_status=None, stream=None):
    L = load()
    _cuda(x, logits, is13, is2, out, ws, d_status)
    x = x.contiguous()
    T, d = x.shape
    if out is None:
        out = _empty((T, d), torch.bfloat16, x.device)
    wsb = moe_workspace_size(T, weights.E, top_k, d, weights.F, mode)
    if ws is None:
        ws = _empty((max(wsb, 16),), torch.uint8, x.device)
    cw = weights._c()
    lg = None if logits is None else logits.contiguous()
    if mode == "w4a16":
        code = L.nvfp4_moe_w4a16(_p(x.view(torch.int16)), T, _p(lg), top_k, ctypes.byref(cw),
                                 _p(out.view(torch.int16)), _p(ws), ws.numel(), _p(d_status), _stream(stream))
    else:
        code = L.nvfp4_moe_w4a4(_p(x.view(torch.int16)), T, _p(lg), top_k, ctypes.byref(cw), _p(is13), _p(is2),
                                _p(out.view(torch.int16)), _p(ws), ws.numel(), _p(d_status), _stream(stream))
    _check(f"nvfp4_moe_{mode}", code)
    return out


def nvfp4_moe_w4a16(x, logits, top_k, weights, out=None, ws=None, d_status=None, stream=None):
    return _moe("w4a16", x, logits, top_k, weights, out=out, ws=ws, d_status=d_status, stream=stream)


def nvfp4_moe_w4a4(x, logits, top_k, weights, input_scale_w13, input_scale_w2, out=None, ws=None, d_status=None,
                   stream=None):
    return _moe("w4a4", x, logits, top_k, weights, input_scale_w13, input_scale_w2, out=out, ws=ws,
                d_status=d_status, stream=stream)


def nvfp4_linear(x, w: NVFP4Tensor, w_up: NVFP4Tensor | None = None, out=None, ws=None, stream=None):
    L = load()
    _cuda(x, out, ws)
    x = x.contiguous()
    M, K = x.shape
    N = w.codes.shape[-2]
    if out is None:
        out = _empty((M, N), torch.bfloat16, x.device)
    wsb = L.nvfp4_linear_workspace_size(M, K, N)
    if ws is None:
        ws = _empty((max(wsb, 16),), torch.uint8, x.device)
    cw = w._c()
    cu = w_up._c() if w_up is not None else None
    _check("nvfp4_linear",
           L.nvfp4_linear(_p(x.view(torch.int16)), M, K, ctypes.byref(cw), N,
                          ctypes.byref(cu) if cu is not None else None, _p(out.view(torch.int16)), _p(ws),
                          ws.numel(), _stream(stream)))
    return out


def status_string(code: int) -> str:
    return load().nvfp4_status_string(int(code)).decode()


def launch_count() -> int:
    return int(load().nvfp4_launch_count())


def selftest_bounded_wait(d_status, stream=None) -> None:
    """Launch the library's bounded-wait self-test: a barrier nothing arrives
    on; the kernel gives up after about 2 s and writes NVFP4_ERR_TIMEOUT (7)
    into d_status (an int32 CUDA tensor)."""
    _cuda(d_status)
    _check("nvfp4_selftest_bounded_wait", load().nvfp4_selftest_bounded_wait(_p(d_status), _stream(stream)))


def profile_enable(on: bool = True):
    load().nvfp4_profile_enable(1 if on else 0)


def profile_collect(max_names: int = 64) -> dict:
    L = load()
    names = ctypes.create_string_buffer(64 * max_names)
    launches = (ctypes.c_int * max_names)()
    ms = (ctypes.c_double * max_names)()
    n = L.nvfp4_profile_collect(max_names, names, launches, ms)
    out = {}
    for i in range(n):
        nm = names.raw[64 * i:64 * (i + 1)].split(b"\0", 1)[0].decode()
        out[nm] = (int(launches[i]), float(ms[i]))
    return out
