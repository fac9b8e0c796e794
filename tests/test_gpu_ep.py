"""The expert-parallel layer's device steps on the library's kernels.

Two ranks are emulated in one process on one GPU: each rank's dispatch,
expert compute and combine run on its own experts and tokens, and the rows
move between the "ranks" by tensor copies (no kernel of one rank waits on
another's).  With the prompt-shaped kernels, each routed row's y depends
only on its own data and is kept in bf16 before the slot-ordered combine,
so every rank's output must equal, bit for bit, the single-GPU layer on the
same tokens (itself checked against the oracle elsewhere).  The real
distributed path is run on a one-rank NCCL group the same way."""
import os
import socket

import pytest
import torch

import serving_nvfp4_routed_gb300 as lib
from serving_nvfp4_routed_gb300 import synth
from serving_nvfp4_routed_gb300.ep import ExpertParallelMoE, LibraryOps, expert_range

pytestmark = pytest.mark.gpu


def _banks(s, seed):
    inp = synth.moe_inputs(s, seed, device="cuda")
    return {n: inp[n] for n in ("gate", "up", "down")}


def _local(banks, lo, hi):
    q = {n: lib.nvfp4_quantize_weights(banks[n][lo:hi].contiguous()) for n in banks}
    return lib.MoEWeights(q["gate"], q["up"], q["down"])


def _emulate(eps, xs, lgs, k, mode, is13=None, is2=None):
    world = len(eps)
    disp = [ep.dispatch(x, lg, k) for ep, x, lg in zip(eps, xs, lgs)]
    rows = [torch.split(dd[0], dd[2]) for dd in disp]
    exps = [torch.split(dd[1], dd[2]) for dd in disp]
    back = []
    for q in range(world):
        y = eps[q].compute(torch.cat([rows[p][q] for p in range(world)]),
                           torch.cat([exps[p][q] for p in range(world)]), mode, is13, is2)
        back.append(torch.split(y, [disp[p][2][q] for p in range(world)]))
    return [eps[p].finish(torch.cat([back[q][p] for q in range(world)]), disp[p][3]) for p in range(world)]


@pytest.mark.parametrize("mode,E", [("w4a16", 16), ("w4a4", 16), ("w4a16", 13)])
def test_two_emulated_ranks_equal_single_gpu(mode, E):
    s = synth.MoEShape(T=300, d=512, E=E, k=4, F=256)
    banks = _banks(s, 800 + E)
    full = lib.MoEWeights(*(lib.nvfp4_quantize_weights(banks[n]) for n in ("gate", "up", "down")))
    xs = [synth.make_x(s.T + 37 * r, s.d, 810 + r, "cuda", outlier_frac=0.05) for r in range(2)]
    lgs = [synth.make_logits(s.T + 37 * r, E, 820 + r, "cuda") for r in range(2)]
    is13 = is2 = None
    if mode == "w4a4":
        is13 = torch.full((E,), 4.0 * 1.05 / 2688, device="cuda")
        is2 = torch.full((E,), 1.0 * 1.05 / 2688, device="cuda")
    eps = [ExpertParallelMoE(LibraryOps(_local(banks, *expert_range(E, 2, r))), E, r, 2) for r in range(2)]
    lib.set_kernel_choice("tc")
    try:
        outs = _emulate(eps, xs, lgs, s.k, mode, is13, is2)
        for r in range(2):
            if mode == "w4a16":
                ref = lib.nvfp4_moe_w4a16(xs[r], lgs[r], s.k, full)
            else:
                ref = lib.nvfp4_moe_w4a4(xs[r], lgs[r], s.k, full, is13, is2)
            assert torch.equal(outs[r].view(torch.int16), ref.view(torch.int16)), f"rank {r}"
    finally:
        lib.set_kernel_choice("auto")


def test_one_rank_nccl_group():
    import torch.distributed as dist

    if not dist.is_nccl_available():
        pytest.skip("no NCCL")
    sock = socket.socket()
    sock.bind(("127.0.0.1", 0))
    port = sock.getsockname()[1]
    sock.close()
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", torch.cuda.current_device()))
    try:
        s = synth.MoEShape(T=256, d=512, E=8, k=2, F=256)
        banks = _banks(s, 830)
        w = _local(banks, 0, s.E)
        x = synth.make_x(s.T, s.d, 831, "cuda")
        lg = synth.make_logits(s.T, s.E, 832, "cuda")
        lib.set_kernel_choice("tc")
        try:
            out = ExpertParallelMoE(LibraryOps(w), s.E, 0, 1)(x, lg, s.k)
            ref = lib.nvfp4_moe_w4a16(x, lg, s.k, w)
        finally:
            lib.set_kernel_choice("auto")
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    finally:
        dist.destroy_process_group()
