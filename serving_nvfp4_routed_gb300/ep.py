"""Expert-parallel routed layer over the ranks of a torch.distributed group.

W4A4 model card "GLM-5.3-Flash-NVFP4-W4A4-Experts", "Validation": the routed
experts run expert-parallel across GPUs (EP4 next to TP4); TensorFold issue
#308, "What the branch does": the grouped kernel takes the routed rows
expert by expert.  Each rank holds the NVFP4 banks of a contiguous range of
experts and routes its own tokens.  One layer call on every rank:

  1. route its tokens and permute the routed rows by expert
     (moe_route_permute): the rows owned by each rank are then contiguous;
  2. gather those rows in that order, with each row's expert
     (moe_gather_rows);
  3. exchange the row counts, then the rows and their experts
     (all_to_all_single);
  4. run its own experts over the rows it received: the layer with the
     routing given (each row one slot of weight 1), i.e. bf16(y) per row;
  5. send the rows back (all_to_all_single, counts reversed);
  6. combine: each token's k rows weighted and summed in slot order
     (moe_combine_rows).

The arithmetic is that of the prompt-shaped path on one GPU -- each routed
row's y rounded to bf16, the weighted sum in fp32 in slot order -- for any
number of ranks and any split of the experts.  The host reads the per-expert
row counts of step 1 to size the exchange (E + 1 integers per call).

The device work of steps 1, 2, 4 and 6 goes through `ops` (the library by
default); the exchange through `torch.distributed` (NCCL between GPUs).
"""
from __future__ import annotations

import numpy as np
import torch

from . import _lib


def expert_range(E: int, world: int, rank: int) -> tuple[int, int]:
    """Experts [lo, hi) of `rank` when E experts are split over `world`
    ranks in contiguous ranges whose sizes differ by at most one."""
    return rank * E // world, (rank + 1) * E // world


def split_counts(offsets, E: int, world: int) -> list[int]:
    """Routed rows owned by each rank, from the permutation's expert
    offsets [E + 1] (the rows of rank q are offsets[lo_q] .. offsets[hi_q])."""
    o = np.asarray(offsets)
    return [int(o[expert_range(E, world, q)[1]] - o[expert_range(E, world, q)[0]]) for q in range(world)]


class LibraryOps:
    """The device side of one rank on the library's kernels."""

    def __init__(self, local_weights: _lib.MoEWeights):
        self.w = local_weights

    def route(self, logits, top_k):
        return _lib.moe_route_permute(logits, top_k)

    def gather(self, x, route, top_k):
        return _lib.moe_gather_rows(x, route["row_to_slot"], top_k, route["offsets"])

    def experts(self, rows, local_ids, mode, is13=None, is2=None):
        """The rank's experts over `rows` [n, d], row i routed (alone, with
        weight 1) to local expert local_ids[i]: bf16(y) per row."""
        n, d = rows.shape
        if n == 0:
            return torch.empty(0, d, dtype=torch.bfloat16, device=rows.device)
        w = self.w
        ws = _lib.moe_workspace(n, w.E, 1, d, w.F, mode, rows.device)
        v = _lib.moe_workspace_views(ws, n, w.E, 1, d, w.F, mode)
        v["ids"].copy_(local_ids.view(n, 1).to(torch.int32))
        v["w"].fill_(1.0)
        if mode == "w4a16":
            return _lib.nvfp4_moe_w4a16(rows, None, 1, w, ws=ws)
        return _lib.nvfp4_moe_w4a4(rows, None, 1, w, is13, is2, ws=ws)

    def combine(self, y, route, T, top_k):
        return _lib.moe_combine_rows(y, route["slot_to_row"], route["w"], T, top_k)


def _all_to_all(out, inp, out_splits, in_splits, group):
    import torch.distributed as dist

    dist.all_to_all_single(out, inp, out_splits, in_splits, group=group)


class ExpertParallelMoE:
    """The routed layer on one rank of an expert-parallel group.

    `ops` holds this rank's experts [lo, hi) (expert_range(E, world, rank))
    and runs the device steps; `exchange(out, inp, out_splits, in_splits)`
    moves rows between ranks (all_to_all_single of the group by default)."""

    def __init__(self, ops, E: int, rank: int, world: int, group=None, exchange=None):
        self.ops = ops
        self.E, self.rank, self.world = E, rank, world
        self.lo, self.hi = expert_range(E, world, rank)
        self.group = group
        self.exchange = exchange or (lambda o, i, os_, is_: _all_to_all(o, i, os_, is_, group))

    # -- the three phases, usable on their own (a single-process driver can
    # -- stand in for the exchange between them)
    def dispatch(self, x, logits, top_k):
        """Steps 1-2: returns (rows in send order, their experts, rows per
        destination rank, routing state for finish())."""
        route = self.ops.route(logits, top_k)
        rows, experts = self.ops.gather(x, route, top_k)
        send = split_counts(route["offsets"].cpu().numpy(), self.E, self.world)
        return rows, experts, send, dict(route=route, T=x.shape[0], k=top_k)

    def compute(self, rows, experts, mode, is13=None, is2=None):
        """Step 4 on the rows received (global expert ids in [lo, hi))."""
        local = experts.to(torch.int64) - self.lo
        if local.numel():
            assert int(local.min()) >= 0 and int(local.max()) < self.hi - self.lo, "rows sent to the wrong rank"
        s13 = None if is13 is None else is13[self.lo:self.hi].contiguous()
        s2 = None if is2 is None else is2[self.lo:self.hi].contiguous()
        return self.ops.experts(rows, local, mode, s13, s2)

    def finish(self, y, state):
        """Step 6 on the rows returned (in this rank's send order)."""
        return self.ops.combine(y, state["route"], state["T"], state["k"])

    def __call__(self, x, logits, top_k, mode="w4a16", is13=None, is2=None):
        rows, experts, send, state = self.dispatch(x, logits, top_k)
        dev = rows.device
        cnt = torch.tensor(send, dtype=torch.int64, device=dev)
        got = torch.empty(self.world, dtype=torch.int64, device=dev)
        self.exchange(got, cnt, None, None)
        recv = [int(v) for v in got.cpu().tolist()]
        d = rows.shape[1]
        rrows = torch.empty(sum(recv), d, dtype=rows.dtype, device=dev)
        rexp = torch.empty(sum(recv), dtype=experts.dtype, device=dev)
        self.exchange(rrows, rows, recv, send)
        self.exchange(rexp, experts, recv, send)
        y = self.compute(rrows, rexp, mode, is13, is2)
        back = torch.empty(rows.shape[0], d, dtype=y.dtype, device=dev)
        self.exchange(back, y.contiguous(), send, recv)
        return self.finish(back, state)
