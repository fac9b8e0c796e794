"""Benchmark of the NVFP4 routed-expert MoE layer on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one call of the layer (route + permutation, gate/up + SwiGLU,
down + weighted combine) over one batch of seeded synthetic tokens whose
inputs are already resident in HBM.  The default workload is the
decode-shaped layer (288 experts, top-8, d=4096, ffn=1536) at T=64; the
line also carries a sweep over T in {1, 8, 32, 64} and, under "workloads",
the W4A4 decode-shaped layer at T=64 and the prompt-shaped layers (W4A16
T=4096; W4A4 T=8192 with calibrated static scales; skewed Zipf(1.2)
popularity at T=16384, with and without a third of the experts masked, both
modes) and the dense NVFP4 MLP, each with its own
device time, end-to-end time, kernel split and binding roofline.  The L2 is flushed (a
256 MB write) between timed steps, outside the timed events.

Under torchrun every rank runs its own batch on its own GPU (no collective
on the data path); the reported time is the max over ranks and the value
counts the tokens of all ranks ("weak" scaling).

--impl reference times the CPU oracle (the plain C restatement used by the
tests) on the machine's host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from serving_nvfp4_routed_gb300 import synth  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
EXPERT_BYTES = lambda d, F: 3 * d * F * 9 // 16  # codes (1/2 B) + e4m3 scales (1/16 B) per weight


# ---------------------------------------------------------------------------
# distributed helpers (host logic; tested with gloo on CPU)
# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, device=None) -> float:
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def aggregate(units_per_rank: float, ms_per_rank: float, world: int, device=None):
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    ms = reduce_max(ms_per_rank, device)
    return units_per_rank * world / (ms / 1e3), ms


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
WORKLOADS = {
    "decode1": (synth.decode(1), "w4a16", "normal", 0.0),
    "decode8": (synth.decode(8), "w4a16", "normal", 0.0),
    "decode32": (synth.decode(32), "w4a16", "normal", 0.0),
    "decode64": (synth.decode(64), "w4a16", "normal", 0.0),
    "decode64_w4a4": (synth.decode(64), "w4a4", "normal", 0.0),
    "prefill_w4a16": (synth.PREFILL_W4A16, "w4a16", "normal", 0.05),
    "prefill_w4a4": (synth.PREFILL_W4A4, "w4a4", "normal", 0.05),
    "skew_w4a16": (synth.SKEW, "w4a16", "zipf", 0.0),
    "skew_w4a4": (synth.SKEW, "w4a4", "zipf", 0.0),
    "skew_masked_w4a16": (synth.SKEW, "w4a16", "zipf_masked", 0.0),
    "skew_masked_w4a4": (synth.SKEW, "w4a4", "zipf_masked", 0.0),
    "dense": (None, "w4a16", "dense", 0.05),
    # small prompt-shaped cases for full-metric ncu captures (not bench lines)
    "prompt_small_w4a16": (synth.PROMPT_SMALL, "w4a16", "normal", 0.05),
    "prompt_small_w4a4": (synth.PROMPT_SMALL, "w4a4", "normal", 0.05),
}


def peaks():
    try:
        p = json.load(open(PEAKS_FILE))
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


KERNEL_SOURCES = {
    "gemv": ("moe_gemv.cu", "gemv.cuh", "tc_ptx.cuh", "common.cuh", "internal.cuh"),
    "decode": ("moe_decode.cu", "decode.cuh", "tc_ptx.cuh", "common.cuh", "internal.cuh"),
    "tc": ("moe_tc.cu", "tc.cuh", "tc_ptx.cuh", "common.cuh", "internal.cuh"),
    "tcm": ("moe_tcm.cu", "tc.cuh", "tc_ptx.cuh", "common.cuh", "internal.cuh"),
    "tcq": ("moe_tcq.cu", "tc.cuh", "tc_ptx.cuh", "common.cuh", "internal.cuh"),
}
# nominal dense FP4 : BF16 tensor rate (13.5 : 2.25 PFLOP/s); the FP4 peak is
# the measured bf16 peak times this ratio
FP4_BF16_RATIO = 6.0


def _code_only(text: str) -> str:
    """Source text without // comments, trailing blanks and empty lines
    (a comment edit does not change a kernel)."""
    out = []
    for line in text.splitlines():
        i = line.find("//")
        while i >= 0 and line.count('"', 0, i) % 2 == 1:  # inside a string literal
            i = line.find("//", i + 2)
        if i >= 0:
            line = line[:i]
        line = line.rstrip()
        if line:
            out.append(line)
    return "\n".join(out)


def kernel_source_hash(kernel: str):
    """Hash of the code of the source files a kernel is built from (its
    recorded DRAM traffic is only reported while that code is unchanged)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "serving_nvfp4_routed_gb300", "csrc")
    family = "decode" if "gateup_down" in kernel else kernel.split("_")[0]
    for fn in KERNEL_SOURCES[family if family in KERNEL_SOURCES else "gemv"]:
        h.update(_code_only(open(os.path.join(csrc, fn)).read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    try:
        t = json.load(open(TRAFFIC_FILE))
        ent = t[kernel][workload]
        if ent.get("source_hash") == kernel_source_hash(kernel):
            return float(ent["bytes_per_launch"])
    except Exception:
        pass
    return None


def calibrate_scales(lib, w, shape, device, seed, n=1024, pct=99.0, margin=1.05):
    """Static W4A4 input scales of a layer (W4A4 model card, "Quantization
    boundary": calibrated static activation scales, p99 with a 5 % margin),
    computed with the library itself once, outside any timed region: a
    seeded n-token draw of the layer's input distribution (N(0,1) rows, 5 %
    of them x 8; normal router logits) runs through the W4A16 layer; per
    expert and projection, the percentile (linear interpolation) of the
    16-block maxima of the rows routed to it -- x rows for gate/up, the
    layer's own h rows for down -- times 1.05 / 2688.  Experts the draw does
    not reach take the percentile over all rows of that projection."""
    s = shape
    x = synth.make_x(n, s.d, seed, device, outlier_frac=0.05)
    lg = synth.make_logits(n, s.E, seed + 1, device)
    ws = lib.moe_workspace(n, s.E, s.k, s.d, s.F, "w4a16", device)
    lib.nvfp4_moe_w4a16(x, lg, s.k, w, ws=ws)
    v = lib.moe_workspace_views(ws, n, s.E, s.k, s.d, s.F, "w4a16")
    h = lib.moe_workspace_intermediates(ws, n, s.E, s.k, s.d, s.F, "w4a16")["h"]
    R = n * s.k
    offs = v["offsets"].cpu().tolist()
    rows = x[v["row_to_slot"].long() // s.k]
    bx = rows.float().abs().view(R, s.d // 16, 16).amax(-1).double()
    bh = h.float().abs().view(R, s.F // 16, 16).amax(-1).double()
    q = pct / 100.0

    def scales(b):
        fb = torch.quantile(b.reshape(-1), q).item()
        out = []
        for e in range(s.E):
            seg = b[offs[e]:offs[e + 1]]
            p = torch.quantile(seg.reshape(-1), q).item() if seg.numel() else fb
            out.append(p * margin / 2688.0)
        return torch.tensor(out, dtype=torch.float32, device=device)

    return scales(bx), scales(bh)


class Layer:
    """Resident weights + a rotation of input batches for one workload."""

    def __init__(self, name, lib, device, seed, n_batches=4):
        self.name = name
        self.shape, self.mode, self.kind, self.outlier = WORKLOADS[name]
        s = self.shape
        self.lib = lib
        self.device = device
        banks = {}
        for nm, (N, K), sd in (("gate", (s.F, s.d), 3), ("up", (s.F, s.d), 4), ("down", (s.d, s.F), 5)):
            w = synth.make_weights(s.E, N, K, seed * 10 + sd, device)
            banks[nm] = lib.nvfp4_quantize_weights(w)
            del w
        torch.cuda.empty_cache()
        self.w = lib.MoEWeights(banks["gate"], banks["up"], banks["down"])
        self.batches = []
        for b in range(n_batches):
            x = synth.make_x(s.T, s.d, seed * 100 + 2 * b, device, self.outlier)
            lg = synth.make_logits(s.T, s.E, seed * 100 + 2 * b + 1, device, self.kind)
            self.batches.append((x, lg))
        self.is13 = self.is2 = None
        if self.mode == "w4a4":
            self.is13, self.is2 = calibrate_scales(lib, self.w, s, device, seed * 100 + 99)
        self.ws = lib.moe_workspace(s.T, s.E, s.k, s.d, s.F, self.mode, device)
        self.out = torch.empty(s.T, s.d, dtype=torch.bfloat16, device=device)

    def step(self, i, x=None, lg=None):
        if x is None:
            x, lg = self.batches[i % len(self.batches)]
        s = self.shape
        if self.mode == "w4a16":
            return self.lib.nvfp4_moe_w4a16(x, lg, s.k, self.w, out=self.out, ws=self.ws)
        return self.lib.nvfp4_moe_w4a4(x, lg, s.k, self.w, self.is13, self.is2, out=self.out, ws=self.ws)

    def touched_experts(self, i):
        s = self.shape
        self.step(i)
        v = self.lib.moe_workspace_views(self.ws, s.T, s.E, s.k, s.d, s.F, self.mode)
        counts = torch.diff(v["offsets"]).cpu()
        return int((counts > 0).sum().item())

    def mean_touched(self, start, steps):
        """Touched experts averaged over the batches that `steps` steps from
        `start` run (each batch routes to its own expert set)."""
        per = [self.touched_experts(b) for b in range(len(self.batches))]
        return statistics.mean(per[(start + i) % len(per)] for i in range(steps)), per

    def algorithmic_bytes(self, touched):
        s = self.shape
        R = s.T * s.k
        w = touched * EXPERT_BYTES(s.d, s.F)
        io = s.T * s.d * 2 + s.T * s.E * 4 + s.T * s.d * 2
        return w + io, R

    def gateup_bytes(self, touched):
        s = self.shape
        R = s.T * s.k
        w = touched * 2 * s.F * s.d * 9 // 16
        if self.mode == "w4a16":
            act = s.T * s.d * 2 + R * s.F * 2
        else:
            act = R * s.d * 9 // 16 + R * s.F * 9 // 16
        return w + act

    def flops(self):
        s = self.shape
        return 6.0 * s.T * s.k * s.d * s.F


class DenseLayer:
    """Dense NVFP4 MLP (gate and up with different tensor scales, SwiGLU,
    down): two nvfp4_linear calls per step."""

    def __init__(self, name, lib, device, seed, n_batches=2):
        self.name = name
        d, F, M = synth.DENSE["d"], synth.DENSE["F"], synth.DENSE["M"]
        self.shape = synth.MoEShape(M, d, 1, 1, F)
        self.mode = "w4a16"
        self.kind = "dense"
        self.lib = lib
        self.device = device
        self.wg = lib.nvfp4_quantize_weights(synth.make_weights(1, F, d, seed * 10 + 3, device)[0])
        self.wu = lib.nvfp4_quantize_weights(synth.make_weights(1, F, d, seed * 10 + 4, device)[0] * 2)
        self.wd = lib.nvfp4_quantize_weights(synth.make_weights(1, d, F, seed * 10 + 5, device)[0])
        torch.cuda.empty_cache()
        self.batches = [(synth.make_x(M, d, seed * 100 + 2 * b, device, 0.05), None) for b in range(n_batches)]
        self.h = torch.empty(M, F, dtype=torch.bfloat16, device=device)
        self.out = torch.empty(M, d, dtype=torch.bfloat16, device=device)
        self.ws1 = torch.empty(lib.load().nvfp4_linear_workspace_size(M, d, F), dtype=torch.uint8, device=device)
        self.ws2 = torch.empty(lib.load().nvfp4_linear_workspace_size(M, F, d), dtype=torch.uint8, device=device)
        self.is13 = self.is2 = None

    def step(self, i, x=None, lg=None):
        if x is None:
            x = self.batches[i % len(self.batches)][0]
        self.lib.nvfp4_linear(x, self.wg, self.wu, out=self.h, ws=self.ws1)
        return self.lib.nvfp4_linear(self.h, self.wd, out=self.out, ws=self.ws2)

    def touched_experts(self, i):
        return 1

    def mean_touched(self, start, steps):
        return 1, [1]

    def algorithmic_bytes(self, touched):
        s = self.shape
        return 3 * s.d * s.F * 9 // 16 + 2 * s.T * s.d * 2, s.T

    def flops(self):
        s = self.shape
        return 6.0 * s.T * s.d * s.F


def time_steps(layer, steps, flush, start=0):
    """Per-step CUDA-event time (ms) of `steps` calls, L2 flushed between."""
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        if flush is not None:
            flush.fill_(i & 0xFF)
        evs[i][0].record(stream)
        layer.step(start + i)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def time_router(layer, steps, flush):
    """The BF16 router GEMM for the workload's tokens (d -> E logits), timed
    like the layer (CUDA events per call, L2 flushed between calls).  It is
    the step before the layer and reported beside it, not inside `value`:
    the metric takes the router's logits as given."""
    s = layer.shape
    dev = layer.device
    w = synth.make_weights(1, s.E, s.d, 777, dev)[0]
    out = torch.empty(s.T, s.E, dtype=torch.float32, device=dev)
    x = layer.batches[0][0]
    for _ in range(3):
        layer.lib.moe_router_logits(x, w, out=out)
    stream = torch.cuda.current_stream()
    ts = []
    for i in range(steps):
        if flush is not None:
            flush.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        layer.lib.moe_router_logits(x, w, out=out)
        b.record(stream)
        ts.append((a, b))
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ts)
    flops = 2.0 * s.T * s.d * s.E
    nbytes = s.T * s.d * 2 + s.E * s.d * 2 + s.T * s.E * 4
    return {"ms_per_call": ms, "tflops": flops / (ms / 1e3) / 1e12, "gbs": nbytes / (ms / 1e3) / 1e9,
            "T": s.T, "d": s.d, "E": s.E}


def time_graph(layer, steps, flush):
    """One layer call captured in a CUDA graph (inputs in the captured
    buffers), replayed `steps` times: CUDA events per replay, L2 flushed
    between replays.  The same work as a step, without host launch gaps."""
    x_s, lg_s = (t.clone() for t in layer.batches[0])
    layer.step(0, x_s, lg_s)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            layer.step(0, x_s, lg_s)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ts = []
    for i in range(steps):
        x, lg = layer.batches[(i + 1) % len(layer.batches)]
        x_s.copy_(x)
        lg_s.copy_(lg)
        if flush is not None:
            flush.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        ts.append((a, b))
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ts)
    return {"ms_per_step": ms, "tokens_per_s": layer.shape.T / (ms / 1e3)}


def time_shared(layer, steps, flush):
    """The BF16 shared-expert MLP for the workload's tokens (ffn taken equal
    to the routed experts': the pages give none), added into the layer's
    output buffer; CUDA events per call, L2 flushed between calls.  Reported
    beside the layer line, not inside `value`."""
    s = layer.shape
    dev = layer.device
    Fs = s.F
    wg, wu = (synth.make_weights(1, Fs, s.d, 779 + i, dev)[0] for i in range(2))
    wd = synth.make_weights(1, s.d, Fs, 781, dev)[0]
    x = layer.batches[0][0]
    out = torch.zeros(s.T, s.d, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(16, layer.lib.load().moe_shared_expert_workspace_size(s.T, Fs)), dtype=torch.uint8,
                     device=dev)
    for _ in range(3):
        layer.lib.moe_shared_expert(x, wg, wu, wd, out, ws=ws)
    stream = torch.cuda.current_stream()
    ts = []
    for i in range(steps):
        if flush is not None:
            flush.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        layer.lib.moe_shared_expert(x, wg, wu, wd, out, ws=ws)
        b.record(stream)
        ts.append((a, b))
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ts)
    flops = 2.0 * s.T * s.d * Fs * 3
    return {"ms_per_call": ms, "tflops": flops / (ms / 1e3) / 1e12, "T": s.T, "d": s.d, "ffn": Fs}


def time_recipe(layer, flush, reps=3):
    """The ModelOpt weight recipe (a load-time step, not inside `value`) on
    one projection bank of the workload, [E, ffn, d] bf16: CUDA events per
    call, L2 flushed between calls.  Algorithmic bytes: the bf16 weights read
    once, the codes and scales written (2 + 1/2 + 1/16 bytes per weight)."""
    s = layer.shape
    dev = layer.device
    w = synth.make_weights(s.E, s.F, s.d, 778, dev)
    layer.lib.nvfp4_quantize_weights(w)
    stream = torch.cuda.current_stream()
    ts = []
    for i in range(reps):
        if flush is not None:
            flush.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        q = layer.lib.nvfp4_quantize_weights(w)
        b.record(stream)
        ts.append((a, b))
        del q
    torch.cuda.synchronize()
    del w
    torch.cuda.empty_cache()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ts)
    n = s.E * s.F * s.d
    nbytes = n * 2 + n // 2 + n // 16
    return {"ms_per_bank": ms, "gbs": nbytes / (ms / 1e3) / 1e9, "weights": n,
            "algorithmic_bytes": nbytes, "passes": "amax pass + block pass (the bf16 bank is read twice)"}


def time_e2e(layer, steps, flush):
    """Same metric with host buffers: pinned H2D of x and logits, the layer,
    D2H of the output, all inside the timed events."""
    s = layer.shape
    hx = [b[0].cpu().pin_memory() for b in layer.batches]
    hl = [b[1].cpu().pin_memory() if b[1] is not None else None for b in layer.batches]
    dx = torch.empty_like(layer.batches[0][0])
    dl = torch.empty_like(layer.batches[0][1]) if layer.batches[0][1] is not None else None
    hout = torch.empty(s.T, s.d, dtype=torch.bfloat16).pin_memory()
    stream = torch.cuda.current_stream()
    times = []
    for i in range(steps):
        if flush is not None:
            flush.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dx.copy_(hx[i % len(hx)], non_blocking=True)
        if dl is not None:
            dl.copy_(hl[i % len(hl)], non_blocking=True)
        out = layer.step(i, dx, dl)
        hout.copy_(out, non_blocking=True)
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b))
    h2d = dx.numel() * dx.element_size() + (dl.numel() * dl.element_size() if dl is not None else 0)
    d2h = hout.numel() * hout.element_size()
    return statistics.mean(times), h2d, d2h


def oracle_timing_scales(x, E):
    """Static input scales for timing the oracle on W4A4 workloads: p99 of
    the batch's 16-block maxima x 1.05 / 2688 for every expert, and a fixed
    down-side scale.  The oracle takes no input from the library, and the
    scales only move saturation, not the oracle's work."""
    bam = np.abs(x[: min(1024, x.shape[0])].float().cpu().numpy()).reshape(-1, 16).max(1)
    is13 = np.full(E, np.percentile(bam, 99) * 1.05 / 2688.0, np.float32)
    is2 = np.full(E, 4.0 * 1.05 / 2688.0, np.float32)
    return is13, is2


def cpu_baseline(layer, seed, n_tokens=8, min_seconds=10.0):
    """The oracle (plain C, fp64, OpenMP on the host cores) on a bounded
    sample of the workload: `n_tokens` tokens of the first batch in a seeded
    order, the call repeated until at least `min_seconds` of oracle time.
    The weights of the sampled tokens' experts are quantised by the oracle
    itself first (untimed: load-time work, not part of a layer call)."""
    from oracle import oracle as orc

    s = layer.shape
    x, lg = layer.batches[0]
    r = orc.route(lg.cpu().numpy(), s.k)
    xb = synth.bf16_bits(x)
    rng = np.random.default_rng(seed)
    tok = np.sort(rng.permutation(s.T)[: min(n_tokens, s.T)]).astype(np.int32)
    experts = np.unique(r["ids"][tok])
    ob = {}
    for nm, (N, K), sd in (("gate", (s.F, s.d), 3), ("up", (s.F, s.d), 4), ("down", (s.d, s.F), 5)):
        w = synth.make_weights(s.E, N, K, seed * 10 + sd, layer.device)
        codes = np.zeros((s.E, N, K // 2), np.uint8)
        scales = np.zeros((s.E, N, K // 16), np.uint8)
        ws2 = np.zeros(s.E, np.float32)
        for e in experts:
            codes[e], scales[e], ws2[e] = orc.quantize_tensor(synth.bf16_bits(w[int(e)]))
        ob[nm] = (codes, scales, ws2)
        del w
    torch.cuda.empty_cache()
    is13 = is2 = None
    if layer.mode == "w4a4":
        is13, is2 = oracle_timing_scales(x, s.E)
    reps = 0
    t0 = time.perf_counter()
    while True:
        orc.moe_layer(layer.mode, xb, r["ids"], r["w"], ob, tokens=tok, is13=is13, is2=is2)
        reps += 1
        elapsed = time.perf_counter() - t0
        if elapsed >= min_seconds:
            break
    return {"value": len(tok) * reps / elapsed, "unit": "tokens/s", "cores": orc.num_threads(), "kind": "oracle",
            "sample": f"{len(tok)} of the {s.T} tokens of the {layer.name} batch (seeded choice), the call "
                      f"repeated {reps} times: {elapsed:.1f} s of oracle time over {len(tok) * s.k} (token, expert) "
                      f"pairs per call; expert weights quantised by the oracle beforehand, untimed"}


def workload_config(layer, flush_mb):
    s = layer.shape
    if layer.kind == "dense":
        return {"workload": f"dense: NVFP4 MLP d={s.d} ffn={s.F} M={s.T}, gate/up with their own tensor scales, "
                            "SwiGLU, down (two nvfp4_linear calls)",
                "M": s.T, "d": s.d, "ffn": s.F, "mode": "w4a16",
                "l2": f"flushed between steps ({flush_mb} MB write), outside the timed events",
                "parallelism": "independent replicas (one batch per GPU)"}
    desc = {"w4a16": "W4A16", "w4a4": "W4A4"}[layer.mode]
    cfg = {"workload": f"{layer.name}: routed-expert NVFP4 layer {desc}, E={s.E} top-{s.k} d={s.d} "
                       f"ffn={s.F} T={s.T}, logits {layer.kind}",
           "T": s.T, "E": s.E, "top_k": s.k, "d": s.d, "ffn": s.F, "mode": layer.mode,
           "l2": f"flushed between steps ({flush_mb} MB write), outside the timed events",
           "parallelism": "independent replicas (one batch per GPU)"}
    if layer.mode == "w4a4":
        cfg["input_scale"] = ("per expert and projection: p99 of the routed rows' 16-block maxima x 1.05 / 2688 "
                              "over a seeded 1024-token draw (h rows from the library's W4A16 layer)")
    return cfg


def kernel_roofline(layer, dom, dom_ms, touched, hbm, bf16, peak_kind, workload):
    """The binding roofline of the dominant kernel's launches: algorithmic
    bytes (touched experts' weights read once, the A rows, the output rows)
    over the measured copy bandwidth, or algorithmic flops over the tensor
    peak -- whichever floor is longer; the other is reported beside it."""
    s_ = layer.shape
    R = s_.T * s_.k if layer.kind != "dense" else s_.T
    if dom.startswith(("tc_", "tcm_", "tcq_")):
        nproj = 2 if "gateup" in dom else 1
        dom_flops = 2.0 * R * s_.d * s_.F * nproj
        achieved = dom_flops / (dom_ms / 1e3) / 1e12
        fp4 = dom.startswith("tcq_")
        peak = bf16 * FP4_BF16_RATIO if fp4 else bf16
        kind = (f"{peak_kind} bf16 dense x nominal FP4/BF16 ratio {FP4_BF16_RATIO:g}, burst" if fp4
                else f"{peak_kind} bf16 dense (f16 runs at the same rate), burst")
        if layer.kind == "dense":
            dom_bytes = (2 if nproj == 2 else 1) * s_.d * s_.F * 9 // 16 + s_.T * (s_.d + s_.F) * 2
        elif nproj == 2:
            dom_bytes = layer.gateup_bytes(touched)
        else:
            a_bytes = R * s_.F * (2 if layer.mode == "w4a16" else 9 / 16)
            dom_bytes = int(touched * s_.d * s_.F * 9 // 16 + a_bytes + s_.T * s_.d * 2)
        bytes_gbs = dom_bytes / (dom_ms / 1e3) / 1e9
        if dom_bytes / hbm > dom_flops / (peak * 1e3):
            return {"bound": "hbm", "kernel": dom, "achieved": bytes_gbs, "peak": hbm, "unit": "GB/s",
                    "frac": bytes_gbs / hbm, "peak_kind": f"{peak_kind} (copy bandwidth, burst)",
                    "traffic": recorded_traffic(dom, workload), "algorithmic_bytes_per_launch": dom_bytes,
                    "tensor": {"achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                               "peak_kind": kind, "algorithmic_flops_per_launch": dom_flops}}
        return {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "peak_kind": kind, "traffic": recorded_traffic(dom, workload),
                "algorithmic_flops_per_launch": dom_flops,
                "hbm": {"achieved": bytes_gbs, "peak": hbm, "unit": "GB/s", "frac": bytes_gbs / hbm,
                        "algorithmic_bytes_per_launch": dom_bytes}}
    if "gateup_down" in dom:
        # the whole decode-shaped layer in one launch: every touched expert's
        # three projections, x in, out and the routing arrays
        dom_bytes = layer.algorithmic_bytes(touched)[0]
    elif dom.startswith("gemv_down"):
        dom_bytes = touched * s_.d * s_.F * 9 // 16 + (R * s_.F * 2 if layer.mode == "w4a16" else R * s_.F * 9 // 16)
    else:
        dom_bytes = layer.gateup_bytes(touched)
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    return {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "peak_kind": f"{peak_kind} (copy bandwidth, burst)",
            "traffic": recorded_traffic(dom, workload), "algorithmic_bytes_per_launch": dom_bytes}


def measure(layer, lib, args, flush, hbm, bf16, peak_kind, steps, world=1, dev=None):
    """Time `steps` layer steps (CUDA events, L2 flushed between steps) with
    the SM clocks sampled, then the same steps with per-launch events for
    the kernel split, then the end-to-end variant with host buffers."""
    for i in range(args.warmup):
        layer.step(i)
    torch.cuda.synchronize()
    touched, per_batch = layer.mean_touched(0, steps)
    launches0 = lib.launch_count()
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        times = time_steps(layer, steps, flush)
    torch.cuda.synchronize()
    barrier()
    launches = lib.launch_count() - launches0
    ms = statistics.mean(times)
    value, ms_max = aggregate(layer.shape.T, ms, world, dev)
    if args.lean:
        # only the timed steps (for profiler captures): no per-launch events, no host-buffer run
        return {"value": value, "ms_per_step": ms_max, "times_ms": times, "launches": launches, "kernels": {},
                "roofline": {"touched_experts": touched}, "clocks": clk.summary(), "e2e": None}
    lib.profile_enable(True)
    time_steps(layer, steps, flush)
    lib.profile_enable(False)
    prof = lib.profile_collect()
    e2e_ms, h2d, d2h = time_e2e(layer, max(3, steps), flush)
    e2e_value, _ = aggregate(layer.shape.T, e2e_ms, world, dev)
    kernels = {k: {"launches": v[0], "ms_per_launch": v[1] / max(1, v[0])} for k, v in prof.items()}
    dom = max(kernels, key=lambda k: kernels[k]["ms_per_launch"] * kernels[k]["launches"]) if kernels else "?"
    dom_ms = kernels.get(dom, {"ms_per_launch": float("nan")})["ms_per_launch"]
    roof = kernel_roofline(layer, dom, dom_ms, touched, hbm, bf16, peak_kind, layer.name)
    total_bytes, R = layer.algorithmic_bytes(touched)
    layer_gbs = total_bytes / (ms / 1e3) / 1e9
    layer_tflops = layer.flops() / (ms / 1e3) / 1e12
    fp4 = layer.mode == "w4a4" and any(k.startswith("tcq_") for k in kernels)
    tpeak = bf16 * FP4_BF16_RATIO if fp4 else bf16
    # the layer's own floor: the longer of its HBM and tensor floors
    floor_ms = max(total_bytes / hbm / 1e6, layer.flops() / (tpeak * 1e9))
    roof.update({"layer_gbs": layer_gbs, "layer_frac_hbm": layer_gbs / hbm, "layer_tflops": layer_tflops,
                 "layer_frac_bf16": layer_tflops / bf16, "layer_frac_tensor": layer_tflops / tpeak,
                 "layer_tensor_peak": "fp4 (measured bf16 x 6)" if fp4 else "bf16",
                 "layer_floor_ms": floor_ms, "layer_frac_of_floor": floor_ms / ms,
                 "touched_experts": touched, "touched_experts_per_batch": per_batch})
    return {"value": value, "ms_per_step": ms_max, "times_ms": times, "launches": launches, "kernels": kernels,
            "roofline": roof, "clocks": clk.summary(),
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms}}


def dtype_of(layer, kernels):
    if layer.mode == "w4a16":
        return "e2m1+e4m3 weights, f16 mma, f32 accumulate"
    if any(k.startswith("tcq_") for k in kernels):
        return "e2m1+e4m3 weights and activations, block-scaled fp4 mma, f32 accumulate"
    return "e2m1+e4m3 weights and activations, f16 mma, f32 accumulate"


PROMPT_WORKLOADS = ("prefill_w4a16", "prefill_w4a4", "skew_w4a16", "skew_w4a4", "skew_masked_w4a16",
                    "skew_masked_w4a4", "dense")
# other layers measured beside the headline in the default run (decode steps)
EXTRA_DECODE_WORKLOADS = ("decode64_w4a4",)


def run_ours(args):
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    from serving_nvfp4_routed_gb300 import build as nvbuild

    if rank == 0:
        nvbuild.build()
    barrier()
    import serving_nvfp4_routed_gb300 as lib

    lib.set_kernel_choice({"auto": "auto", "split": "gemv_split", "fused": "gemv_fused"}[args.decode_form])
    hbm, bf16, peak_kind = peaks()
    flush_mb = 256
    flush = torch.empty(flush_mb << 20, dtype=torch.uint8, device=dev)
    seed = 1001 + 17 * rank
    layer = (DenseLayer if args.workload == "dense" else Layer)(args.workload, lib, dev, seed)
    m = measure(layer, lib, args, flush, hbm, bf16, peak_kind, args.steps, world, dev)

    line = {
        "metric": "MoE-layer tokens/s",
        "value": m["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": m["ms_per_step"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": dtype_of(layer, m["kernels"]),
        "data": "synthetic (seeded N(0,1) x and logits, N(0,0.02) bf16 weights quantised by the library)",
        "config": dict(workload_config(layer, flush_mb), decode_form=args.decode_form),
        "roofline": m["roofline"],
        "kernels": m["kernels"],
        "e2e": m["e2e"],
        "gpu_launches": m["launches"],
        "clocks": m["clocks"],
    }
    if layer.kind != "dense" and not args.lean:
        line["router_gemm"] = time_router(layer, max(3, args.steps), flush)
        line["graph_replay"] = time_graph(layer, max(3, args.steps), flush)
        recipe = time_recipe(layer, flush)
        recipe["frac_hbm"] = recipe["gbs"] / hbm
        line["weight_recipe"] = recipe
        shared = time_shared(layer, max(3, args.steps), flush)
        shared["frac_bf16"] = shared["tflops"] / bf16
        line["shared_expert"] = shared
    if args.sweep and args.workload == "decode64":
        sweep = {"decode64": {"tokens_per_s": m["value"] / world, "ms": m["ms_per_step"],
                              "layer_frac": m["roofline"]["layer_frac_hbm"]}}
        for T in synth.DECODE_T:
            if T == 64:
                continue
            sl = Layer(f"decode{T}", lib, dev, seed + T)
            ms_ = measure(sl, lib, args, flush, hbm, bf16, peak_kind, args.steps)
            sweep[f"decode{T}"] = {"tokens_per_s": T / (ms_["ms_per_step"] / 1e3), "ms": ms_["ms_per_step"],
                                   "touched_experts": ms_["roofline"]["touched_experts"],
                                   "layer_gbs": ms_["roofline"]["layer_gbs"],
                                   "layer_frac": ms_["roofline"]["layer_frac_hbm"],
                                   "kernels": ms_["kernels"], "e2e": ms_["e2e"], "clocks": ms_["clocks"]}
            del sl
            torch.cuda.empty_cache()
        line["sweep"] = sweep
    if rank == 0 and not args.no_cpu_baseline and layer.kind != "dense":
        line["cpu_baseline"] = cpu_baseline(layer, seed, n_tokens=args.cpu_tokens)
    del layer
    torch.cuda.empty_cache()
    if args.workloads and args.workload == "decode64":
        # the prompt-shaped half of the metric: the other configurations,
        # each measured the same way (fewer steps: each step is milliseconds)
        lib.set_kernel_choice("auto")
        wl = {}
        for name in EXTRA_DECODE_WORKLOADS + PROMPT_WORKLOADS:
            lay = (DenseLayer if name == "dense" else Layer)(name, lib, dev, seed + 7)
            n_steps = args.steps if name in EXTRA_DECODE_WORKLOADS else min(args.steps, args.prompt_steps)
            res = measure(lay, lib, args, flush, hbm, bf16, peak_kind, n_steps, world, dev)
            res.pop("times_ms")
            res["tokens_per_s"] = res.pop("value")
            res["config"] = workload_config(lay, flush_mb)
            res["dtype"] = dtype_of(lay, res["kernels"])
            wl[name] = res
            del lay
            torch.cuda.empty_cache()
        line["workloads"] = wl
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def run_reference(args):
    world, rank, local = dist_env()
    if rank != 0:
        return
    from oracle import oracle as orc

    orc.build()
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    shape, mode, kind, outlier = WORKLOADS[args.workload]
    seed = 1001
    x = synth.make_x(shape.T, shape.d, seed * 100, dev, outlier)
    lg = synth.make_logits(shape.T, shape.E, seed * 100 + 1, dev, kind)
    r = orc.route(lg.cpu().numpy(), shape.k)
    xb = synth.bf16_bits(x)
    gen = {nm: (N, K, sd) for nm, (N, K), sd in
           (("gate", (shape.F, shape.d), 3), ("up", (shape.F, shape.d), 4), ("down", (shape.d, shape.F), 5))}
    per_step = max(1, min(shape.T, args.ref_tokens))
    rng = np.random.default_rng(seed)
    tok_all = rng.permutation(shape.T)[: per_step * (args.warmup + args.steps)] % shape.T
    experts = np.unique(r["ids"][tok_all])
    ob = {}
    for nm, (N, K, sd) in gen.items():
        w = synth.make_weights(shape.E, N, K, seed * 10 + sd, dev)
        codes = np.zeros((shape.E, N, K // 2), np.uint8)
        scales = np.zeros((shape.E, N, K // 16), np.uint8)
        ws2 = np.zeros(shape.E, np.float32)
        for e in experts:
            codes[e], scales[e], ws2[e] = orc.quantize_tensor(synth.bf16_bits(w[int(e)]))
        ob[nm] = (codes, scales, ws2)
        del w
    is13 = is2 = None
    if mode == "w4a4":
        is13, is2 = oracle_timing_scales(x, shape.E)
    times = []
    for i in range(args.warmup + args.steps):
        tok = np.sort(tok_all[i * per_step:(i + 1) * per_step]).astype(np.int32)
        t0 = time.perf_counter()
        orc.moe_layer(mode, xb, r["ids"], r["w"], ob, tokens=tok, is13=is13, is2=is2)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    ms = statistics.mean(times) * 1e3
    value = per_step / (ms / 1e3)
    cores = orc.num_threads()
    line = {"impl": "reference", "metric": "MoE-layer tokens/s",
            "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64 (CPU oracle)", "data": "synthetic",
            "config": {"workload": f"{args.workload} (same seeds and shapes as the GPU arm)", "T": shape.T,
                       "E": shape.E, "top_k": shape.k, "d": shape.d, "ffn": shape.F, "mode": mode},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{per_step} tokens per step of the {shape.T}-token batch"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="decode64")
    ap.add_argument("--no-sweep", dest="sweep", action="store_false")
    ap.add_argument("--no-workloads", dest="workloads", action="store_false",
                    help="skip the prompt-shaped and dense workloads of the default run")
    ap.add_argument("--prompt-steps", type=int, default=10)
    ap.add_argument("--lean", action="store_true",
                    help="time the layer steps only (no kernel split, host-buffer run or side timings): for "
                         "profiler captures, whose launch list then holds the warm-up, the touched-expert count "
                         "(one step per input batch) and the timed steps")
    ap.add_argument("--decode-form", choices=("auto", "split", "fused"), default="auto",
                    help="decode-shaped layer as the library picks it, as two launches, or as one")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-tokens", type=int, default=8)
    ap.add_argument("--ref-tokens", type=int, default=4)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
