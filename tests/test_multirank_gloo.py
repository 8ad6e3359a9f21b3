"""The bench's multi-GPU host logic, on CPU ranks over gloo (world size 2).

With N GPUs every rank runs its own virtual-rank problem (weak scaling, no
data-path collective); the only cross-rank steps are the barrier, the max
over ranks of the timed region, and rank 0 alone printing. These run here
with the gloo backend; nothing needs a GPU.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, local = bench.dist_env()
    times = [1.5, 4.25]
    got = bench.max_over_ranks(times[rank])
    dist.barrier()
    # the reference arm: rank 0 alone runs the oracle; the others return at once
    class A:
        steps, warmup, ref_budget = 1, 0, 0.5
    rc = bench.run_reference(A) if rank != 0 else 0
    out[rank] = (w, r, local, got, bench.rank_seed(rank), rc)
    dist.destroy_process_group()


def test_two_ranks_over_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(world):
        w, rr, local, got, seed, rc = out[r]
        assert (w, rr, local) == (world, r, r)
        assert got == 4.25          # every rank sees the slowest rank's time
        assert rc == 0
    assert out[0][4] != out[1][4]   # each GPU draws its own problem


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0) == 3.0
    assert bench.busbw_gbs(8 << 20, 8, 1e-3) == pytest.approx((8 << 20) / 1e-3 * 2 * 7 / 8 / 1e9)
