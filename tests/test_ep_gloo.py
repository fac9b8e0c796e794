"""The expert-parallel layer (serving_nvfp4_routed_gb300/ep.py) on two
ranks of a gloo group on the CPU: the experts split over the ranks, each
rank routes its own tokens, rows go to the owning rank and back through
all_to_all_single, and each rank's output equals, bit for bit, the
single-process oracle with every routed row's y rounded to bf16 (the
arithmetic the expert-parallel layer keeps).  The ranks' device steps are
the oracle's (tests/ep_util.py): the test covers the partition, the
dispatch and combine index arithmetic and the exchange."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from serving_nvfp4_routed_gb300.ep import expert_range, split_counts


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_partition_and_counts():
    for E, world in ((8, 2), (7, 2), (288, 4), (5, 3), (3, 3)):
        r = [expert_range(E, world, q) for q in range(world)]
        assert r[0][0] == 0 and r[-1][1] == E
        assert all(r[q][1] == r[q + 1][0] for q in range(world - 1))
        assert max(h - l for l, h in r) - min(h - l for l, h in r) <= 1
    offs = np.array([0, 3, 3, 7, 9, 9, 12])
    assert split_counts(offs, 6, 2) == [7, 5]
    assert split_counts(offs, 6, 3) == [3, 6, 3]


def _worker(rank, world, port, E, mode, masked, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import sys
        sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
        from ep_util import OracleOps, slice_bank
        from oracle import calib
        from oracle import oracle as orc
        from serving_nvfp4_routed_gb300 import synth
        from serving_nvfp4_routed_gb300.ep import ExpertParallelMoE

        s = synth.MoEShape(T=6, d=256, E=E, k=2, F=128)
        inp = synth.moe_inputs(s, 500)  # the same weights on every rank
        bank = {}
        for name in ("gate", "up", "down"):
            res = [orc.quantize_tensor(synth.bf16_bits(inp[name][e])) for e in range(E)]
            bank[name] = (np.stack([r[0] for r in res]), np.stack([r[1] for r in res]),
                          np.array([r[2] for r in res], np.float32))
        x = synth.make_x(s.T + rank, s.d, 600 + rank, outlier_frac=0.2)  # each rank its own tokens
        logits = synth.make_logits(s.T + rank, E, 700 + rank)
        if masked:  # no token is routed to the last rank's experts
            lo, hi = expert_range(E, world, world - 1)
            logits[:, lo:hi] = -float("inf")
        is13 = is2 = None
        if mode == "w4a4":
            a, b = calib.calibrate(synth.bf16_bits(inp["x"]), inp["logits"].numpy(), s.k, bank)
            is13, is2 = torch.from_numpy(a), torch.from_numpy(b)
        lo, hi = expert_range(E, world, rank)
        ep = ExpertParallelMoE(OracleOps(orc, slice_bank(bank, lo, hi)), E, rank, world)
        out = ep(x, logits, s.k, mode, is13, is2)
        r = orc.route(logits.numpy(), s.k)
        ref = orc.moe_layer_ex(mode, synth.bf16_bits(x), r["ids"], r["w"], bank,
                               is13=None if is13 is None else is13.numpy(),
                               is2=None if is2 is None else is2.numpy(), round_y=True)["out"]
        q.put((rank, bool(np.array_equal(out.float().numpy(), ref)), float(np.abs(ref).max())))
    except Exception as exc:  # report instead of hanging the other rank
        q.put((rank, repr(exc), 0.0))
        raise
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("E,mode,masked", [(8, "w4a16", False), (7, "w4a16", False), (8, "w4a4", False),
                                           (8, "w4a16", True)])
def test_two_rank_expert_parallel_layer(E, mode, masked):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, E, mode, masked, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    for rank, ok, amax in res:
        assert ok is True, f"rank {rank}: {ok}"
        assert amax > 0
