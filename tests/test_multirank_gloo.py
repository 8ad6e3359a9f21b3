"""The bench's multi-GPU host logic, on CPU ranks over gloo (world size 2).

With N GPUs one AllReduce problem is split by element range: every GPU
reduces its own contiguous part of all n virtual ranks' buffers (weak
scaling: the problem grows with N, each part stays the single-GPU
workload), with no data-path collective; the only cross-rank steps are the
barrier, the max over ranks of the timed region, and rank 0 alone
printing. These run here with the gloo backend, and each rank runs the
oracle on its part in place of the GPU; nothing needs a GPU.
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


def _shard_worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from oracle import ring
    from ring_allreduce_reduction_gb300 import build
    build.build()
    from ring_allreduce_reduction_gb300 import vrccl
    from ring_allreduce_reduction_gb300.workloads import make_inputs
    n, per_gpu, C, K = 4, 5003, 3, 64
    total, off, ln = bench.shard_of(vrccl, per_gpu, "float32", world, rank)
    # integer-valued fp32 inputs: sums are exact, so the whole problem has
    # one correct answer whatever each shard's schedule
    x = make_inputs(n, ln, "float32", "int_uniform", seed=bench.rank_seed(rank), lo=-8, hi=8)
    y = ring.ring_allreduce(x, "sum", "float32", C, K)
    parts = [None] * world
    dist.all_gather_object(parts, (off, ln, x, y))
    if rank == 0:
        out["parts"] = parts
        out["total"] = total
    dist.destroy_process_group()


def test_element_range_shards_over_gloo():
    """Two ranks each reduce their part of one 4-rank problem (the oracle
    standing in for the GPU). The parts tile the buffer in order on 16-byte
    boundaries, the concatenated result is the closed form of the
    concatenated inputs, and each part is the ring's association for its
    own schedule."""
    import numpy as np
    sys.path.insert(0, ROOT)
    from oracle import ring
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_shard_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    parts, total = out["parts"], out["total"]
    pos = 0
    for off, ln, _, _ in parts:
        assert off == pos and (off * 4) % 16 == 0
        pos += ln
    assert pos == total
    x = np.concatenate([p[2] for p in parts], axis=1)
    y = np.concatenate([p[3] for p in parts], axis=1)
    assert np.array_equal(y, np.broadcast_to(x.astype(np.float64).sum(axis=0).astype(np.float32), y.shape))
    for off, ln, xs, ys in parts:
        assert np.array_equal(ys[0], ring.ring_predict(xs, "sum", "float32", 3, 64))


def test_shard_ranges_tile_the_buffer():
    """vrcclShardRange (host only): contiguous parts in shard order, each
    starting on a 16-byte boundary, covering [0, count) exactly; empty
    trailing parts when the count is small."""
    sys.path.insert(0, ROOT)
    from ring_allreduce_reduction_gb300 import build
    build.build()
    from ring_allreduce_reduction_gb300 import vrccl
    for dtype, E in (("float32", 4), ("bfloat16", 2), ("int8", 1), ("float64", 8)):
        for count in (0, 1, 7, 100, 4097, 1 << 20, 3 * (1 << 20) + 5):
            for N in (1, 2, 3, 8, 72):
                pos = 0
                for s in range(N):
                    off, ln = vrccl.vrcclShardRange(count, dtype, N, s)
                    assert off == pos or (ln == 0 and off == count)
                    assert (off * E) % 16 == 0 or off == count
                    pos = off + ln
                assert pos == count
    with pytest.raises(vrccl.VrcclError):
        vrccl.vrcclShardRange(10, "float32", 2, 2)
