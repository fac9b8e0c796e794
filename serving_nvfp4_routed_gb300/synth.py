"""Seeded synthetic inputs for the routed-expert NVFP4 MoE layer.

This module only draws random numbers: it holds none of the layer's
arithmetic (no quantisation, routing or matmul), so the CUDA path and the CPU
oracle can both be fed from it without sharing any of the method.

Workloads (shapes from the GLM-5.3-Flash routed-expert layer: 288 experts per
layer with gate_proj/up_proj/down_proj, top-8, hidden 4096, expert ffn 1536;
model card "GLM-5.3-Flash-NVFP4-W4A4-Experts", "Quantization boundary"):

  tiny      T=4,     d=256,  E=8,   k=2, F=128    x ~ N(0,1), logits ~ N(0,1)
  decode    T in {1,8,32,64}, d=4096, E=288, k=8, F=1536
  prefill   T=4096 (W4A16) / 8192 (W4A4), 5 % of rows of x scaled x8
  skew      T=16384, logits = Gumbel-perturbed Zipf(1.2) log-weights over a
            seeded permutation of the experts; the "masked" variant sets a
            seeded third of the experts to -inf so that they receive no rows
  dense     M=8192, d=4096, F=12288 (gate/up drawn independently, so their
            tensor scales differ)
Weights are bf16 ~ N(0, 0.02) (quantised to NVFP4 by the library under test
or by the oracle, never here).
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class MoEShape:
    T: int
    d: int
    E: int
    k: int
    F: int


TINY = MoEShape(T=4, d=256, E=8, k=2, F=128)
DECODE_T = (1, 8, 32, 64)


def decode(T: int) -> MoEShape:
    return MoEShape(T=T, d=4096, E=288, k=8, F=1536)


PREFILL_W4A16 = MoEShape(T=4096, d=4096, E=288, k=8, F=1536)
PREFILL_W4A4 = MoEShape(T=8192, d=4096, E=288, k=8, F=1536)
# a smaller prompt-shaped layer (about 128 routed rows per expert) for
# full-metric profiler captures, whose replay cost grows with device memory
PROMPT_SMALL = MoEShape(T=1024, d=4096, E=64, k=8, F=1536)
SKEW = MoEShape(T=16384, d=4096, E=288, k=8, F=1536)
DENSE = dict(M=8192, d=4096, F=12288)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_x(T: int, d: int, seed: int, device="cpu", outlier_frac: float = 0.0,
           outlier_scale: float = 8.0) -> torch.Tensor:
    """bf16 [T, d] ~ N(0,1); a seeded ``outlier_frac`` of the rows is scaled."""
    g = _gen(seed, device)
    x = torch.randn(T, d, generator=g, device=device, dtype=torch.float32)
    if outlier_frac > 0 and T > 0:
        n_out = max(1, int(round(outlier_frac * T)))
        rows = torch.randperm(T, generator=g, device=device)[:n_out]
        x[rows] *= outlier_scale
    return x.to(torch.bfloat16)


def make_logits(T: int, E: int, seed: int, device="cpu", kind: str = "normal",
                zipf_s: float = 1.2, masked_frac: float = 1.0 / 3.0) -> torch.Tensor:
    """fp32 router logits [T, E].

    normal: N(0,1) (uniform expert choice in expectation).
    zipf:   -s*ln(rank(e)) + Gumbel noise, rank from a seeded permutation, so
            that top-k of the logits is a draw without replacement from the
            Zipf(s) popularity.
    zipf_masked: as zipf, with a seeded ``masked_frac`` of experts at -inf.
    """
    g = _gen(seed, device)
    if kind == "normal":
        return torch.randn(T, E, generator=g, device=device, dtype=torch.float32)
    perm = torch.randperm(E, generator=g, device=device)
    rank = torch.empty(E, device=device, dtype=torch.float32)
    rank[perm] = torch.arange(1, E + 1, device=device, dtype=torch.float32)
    logw = -zipf_s * torch.log(rank)
    u = torch.rand(T, E, generator=g, device=device, dtype=torch.float32).clamp_(1e-12, 1 - 1e-7)
    gumbel = -torch.log(-torch.log(u))
    lg = logw[None, :] + gumbel
    if kind == "zipf_masked":
        n_mask = int(round(masked_frac * E))
        masked = torch.randperm(E, generator=g, device=device)[:n_mask]
        lg[:, masked] = -math.inf
    elif kind != "zipf":
        raise ValueError(kind)
    return lg.contiguous()


def make_weights(E: int, N: int, K: int, seed: int, device="cpu", std: float = 0.02,
                 chunk: int = 16) -> torch.Tensor:
    """bf16 [E, N, K] ~ N(0, std), drawn expert-chunk by expert-chunk."""
    g = _gen(seed, device)
    w = torch.empty(E, N, K, device=device, dtype=torch.bfloat16)
    for e0 in range(0, E, chunk):
        e1 = min(E, e0 + chunk)
        w[e0:e1] = (torch.randn(e1 - e0, N, K, generator=g, device=device,
                                dtype=torch.float32) * std).to(torch.bfloat16)
    return w


def moe_inputs(shape: MoEShape, seed: int, device="cpu", outlier_frac: float = 0.0,
               logits_kind: str = "normal"):
    """x, logits and the three bf16 weight banks for one routed layer."""
    return dict(
        x=make_x(shape.T, shape.d, seed * 10 + 1, device, outlier_frac),
        logits=make_logits(shape.T, shape.E, seed * 10 + 2, device, logits_kind),
        gate=make_weights(shape.E, shape.F, shape.d, seed * 10 + 3, device),
        up=make_weights(shape.E, shape.F, shape.d, seed * 10 + 4, device),
        down=make_weights(shape.E, shape.d, shape.F, seed * 10 + 5, device),
    )


def bf16_bits(t: torch.Tensor):
    """uint16 numpy view of a bf16 tensor (on the host)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")
