"""GPU parity of the one-shot AllReduce.

The one-shot reads all n inputs of an element at once and writes all n
outputs, folding in the ring's association order for the channel count and
chunk it reports. So it must equal, bit for bit, the oracle's ring step
machine replaying that schedule, and the ring kernel itself when both run
with the same channel count and chunk.
"""
import numpy as np
import pytest

from oracle import closed_form, ring as oring
from ring_allreduce_reduction_gb300.workloads import ELEM_SIZE, make_inputs
from tests.gpu_harness import run

pytestmark = pytest.mark.gpu

DT = ["int32", "float32", "bfloat16", "float16"]
OPS = ["sum", "prod", "max", "min", "avg"]


@pytest.fixture(scope="module")
def v():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ring_allreduce_reduction_gb300 import build
    build.build()
    from ring_allreduce_reduction_gb300 import vrccl
    return vrccl


def _inputs(n, count, dtype, op, seed=0):
    if dtype == "int32":
        return make_inputs(n, count, dtype, "int_uniform", seed=seed, lo=-2**20, hi=2**20)
    if op == "prod":
        return make_inputs(n, count, dtype, "uniform", seed=seed, lo=0.5, hi=2.0)
    return make_inputs(n, count, dtype, "normal", seed=seed)


def _same_bits(a, b):
    return np.array_equal(np.ascontiguousarray(a).view(np.uint8), np.ascontiguousarray(b).view(np.uint8))


@pytest.mark.parametrize("n", [1, 2, 5, 8])
def test_oneshot_equals_ring_and_oracle_every_dtype_and_op(v, n):
    """Forced schedule (3 channels, 256-byte chunk): several loops, a short
    last loop, a ragged tail shorter than one 16-byte vector."""
    comm = v.vrcclCommInit(n, 4)
    try:
        v.vrcclCommSetSchedule(comm, 3, 256)
        for dtype in DT:
            count = 3001 if ELEM_SIZE[dtype] == 4 else 6003
            for op in OPS:
                x = _inputs(n, count, dtype, op, seed=n + len(op))
                y1, s1, b1 = run(v, comm, x, dtype, op, "oneshot", "simple")
                assert s1["algo"] == "oneshot" and s1["nchannels"] == 3
                y2, s2, _ = run(v, comm, x, dtype, op, "ring", "simple")
                assert (s2["nchannels"], s2["chunk_elems"]) == (s1["nchannels"], s1["chunk_elems"])
                assert _same_bits(y1, y2), (dtype, op)
                ref = oring.ring_allreduce(x, op, dtype, s1["nchannels"], s1["chunk_elems"])
                assert _same_bits(y1, ref), (dtype, op)
                ok, worst = closed_form.check(y1[0], x, op, dtype)
                assert ok, worst
                assert b1.canaries_intact()
    finally:
        v.vrcclCommDestroy(comm)


@pytest.mark.parametrize("count", [0, 1, 3, 4, 5, 1000, 65536 + 7])
def test_oneshot_small_and_ragged_counts_inplace(v, count):
    n = 6
    comm = v.vrcclCommInit(n, 8)
    try:
        if count == 0:  # nothing to do: success, nothing launched, no schedule recorded
            from tests.gpu_harness import Buffers
            b = Buffers(np.zeros((n, 0), dtype=np.float32), "float32")
            v.vrcclAllReduce(b.send_ptrs(), b.recv_ptrs(), 0, "float32", "sum", "oneshot", "simple", comm)
            assert b.canaries_intact()
            return
        for inplace in (False, True):
            x = _inputs(n, count, "float32", "sum", seed=count)
            y, s, b = run(v, comm, x, "float32", "sum", "oneshot", "auto", inplace=inplace)
            ref = oring.ring_allreduce(x, "sum", "float32", s["nchannels"], s["chunk_elems"])
            assert _same_bits(y, ref)
            assert b.canaries_intact()
    finally:
        v.vrcclCommDestroy(comm)


@pytest.mark.parametrize("n", [16, 72])
def test_oneshot_many_ranks(v, n):
    """More ranks than one load group (8): the fold runs in several groups."""
    comm = v.vrcclCommInit(n, 4)
    try:
        x = _inputs(n, 40000 + 4, "bfloat16", "sum", seed=n)
        y, s, b = run(v, comm, x, "bfloat16", "sum", "oneshot", "simple")
        ref = oring.ring_allreduce(x, "sum", "bfloat16", s["nchannels"], s["chunk_elems"])
        assert _same_bits(y, ref) and b.canaries_intact()
    finally:
        v.vrcclCommDestroy(comm)


def test_oneshot_full_size_matches_ring(v):
    """n=8, 256 MiB fp32 per rank: the ring's own schedule, forced on the
    one-shot, gives the same 2 GiB of results (compared on the device);
    sampled outputs match the oracle's predictor."""
    import torch
    n, count = 8, (256 << 20) // 4
    x = make_inputs(n, count, "float32", "uniform", seed=1000)
    send = torch.from_numpy(x).to("cuda:0")
    r1 = torch.empty_like(send)
    r2 = torch.empty_like(send)
    comm = v.vrcclCommInit(n, 32)
    try:
        v.vrcclAllReduce([send[r] for r in range(n)], [r1[r] for r in range(n)], count, "float32", "sum", "ring",
                         "simple", comm)
        s = v.vrcclCommGetLastSchedule(comm)
        v.vrcclCommSetSchedule(comm, s["nchannels"], s["chunk_elems"] * 4)
        v.vrcclAllReduce([send[r] for r in range(n)], [r2[r] for r in range(n)], count, "float32", "sum",
                         "oneshot", "simple", comm)
        torch.cuda.synchronize()
        s2 = v.vrcclCommGetLastSchedule(comm)
        assert (s2["nchannels"], s2["chunk_elems"]) == (s["nchannels"], s["chunk_elems"])
        assert torch.equal(r1.view(torch.int32), r2.view(torch.int32))
        for r in range(1, n):
            assert torch.equal(r2[r], r2[0])
        idx = np.unique(np.concatenate([np.random.default_rng(5).choice(count, 100_000, replace=False),
                                        [0, count - 1]]))
        got = r2[0].cpu().numpy()[idx]
        ref = oring.ring_predict(x, "sum", "float32", s["nchannels"], s["chunk_elems"], idx)
        assert _same_bits(got, ref)
        assert v.vrcclCommGetAsyncError(comm) == 0
    finally:
        v.vrcclCommDestroy(comm)
