"""vrcclAllReduceNoAlloc against vrcclAllReduce, on the GPU, through the C ABI.

The allocation-free entry point serves callers that cannot allocate device
memory when they need the reduction (a memory-pool manager owns the device,
or cudaMalloc's implicit synchronisation is not acceptable on the path).
Its scratch is a static device array shared by all calls, so this checks
two calls in a row (the second one starts from what the first left behind)
and calls of other shapes, each against the communicator path run with the
same schedule and against the oracle's ring association for that schedule
(so the two paths cannot drift from the method together). This file sorts
last so that a run stopping at the first failure has already run every
other test.
"""
import numpy as np
import pytest

from oracle import closed_form, ring as oring
from ring_allreduce_reduction_gb300.workloads import make_inputs
from tests.gpu_harness import Buffers

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def v():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ring_allreduce_reduction_gb300 import build
    build.build()
    from ring_allreduce_reduction_gb300 import vrccl
    return vrccl


def _channels(n):
    return max(1, min(4, 32 // n))


def _reference(v, x, dtype, op, inplace=False):
    """The communicator path with the schedule the no-alloc call uses."""
    n, count = x.shape
    comm = v.vrcclCommInit(n, 4)
    try:
        v.vrcclCommSetSchedule(comm, _channels(n), 262144)
        b = Buffers(x, dtype, inplace=inplace)
        v.vrcclAllReduce(b.send_ptrs(), b.recv_ptrs(), count, dtype, op, "ring", "simple", comm)
        y = b.result()
        assert v.vrcclCommGetAsyncError(comm) == 0
        return y
    finally:
        v.vrcclCommDestroy(comm)


def _no_alloc(v, x, dtype, op, inplace=False):
    n, count = x.shape
    b = Buffers(x, dtype, inplace=inplace)
    v.vrcclAllReduceNoAlloc(b.send_ptrs(), b.recv_ptrs(), count, n, dtype, op)
    y = b.result()
    assert b.canaries_intact()
    return y


def _same(y, ref, x, dtype, op):
    # identical schedule -> identical bits (tolerance 0), and within the
    # closed-form tolerance every parity test uses
    assert np.array_equal(y.view(np.uint8), ref.view(np.uint8))
    for r in range(1, y.shape[0]):
        assert np.array_equal(y[r].view(np.uint8), y[0].view(np.uint8))
    ok, worst = closed_form.check(y[0], x, op, dtype)
    assert ok, worst
    # the oracle's ring order for the no-alloc schedule (chunk 256 KiB)
    E = y.dtype.itemsize
    pred = oring.ring_predict(x, op, dtype, _channels(x.shape[0]), 262144 // E)
    assert np.array_equal(y[0].view(np.uint8), np.ascontiguousarray(pred).view(np.uint8))


def test_no_alloc_matches_communicator_path(v):
    x = make_inputs(8, 3_000_001, "float32", "normal", seed=21)
    ref = _reference(v, x, "float32", "sum")
    for _ in range(2):  # two calls in a row on the shared scratch
        _same(_no_alloc(v, x, "float32", "sum"), ref, x, "float32", "sum")
    x2 = make_inputs(5, 200_003, "bfloat16", "normal", seed=22)
    _same(_no_alloc(v, x2, "bfloat16", "avg"), _reference(v, x2, "bfloat16", "avg"), x2, "bfloat16", "avg")


@pytest.mark.parametrize("n,count,dtype,op,inplace", [
    (32, 100_003, "float32", "sum", False),   # one channel, all 32 edges of the scratch
    (1, 4_099, "float32", "sum", False),      # a single rank: the copy
    (8, 250_001, "int32", "avg", False),      # integer avg: the post-op divide
    (6, 77_777, "float16", "max", True),      # in place
])
def test_no_alloc_edge_cases(v, n, count, dtype, op, inplace):
    if dtype == "int32":
        x = make_inputs(n, count, dtype, "int_uniform", seed=24, lo=-2**20, hi=2**20)
    else:
        x = make_inputs(n, count, dtype, "normal", seed=24)
    ref = _reference(v, x, dtype, op, inplace=inplace)
    for _ in range(2):
        _same(_no_alloc(v, x, dtype, op, inplace=inplace), ref, x, dtype, op)


def test_no_alloc_rejects_overlapping_buffers(v):
    x = make_inputs(4, 1024, "float32", "normal", seed=25)
    b = Buffers(x, "float32")
    recv = [p + 16 for p in b.send_ptrs()]  # each recv buffer overlaps its own send buffer
    with pytest.raises(v.VrcclError, match="InvalidArgument"):
        v.vrcclAllReduceNoAlloc(b.send_ptrs(), recv, 1024, 4, "float32", "sum")


def test_no_alloc_rejects_more_ranks_than_its_scratch_holds(v):
    x = make_inputs(33, 64, "float32", "normal", seed=23)
    b = Buffers(x, "float32")
    with pytest.raises(v.VrcclError, match="InvalidUsage"):
        v.vrcclAllReduceNoAlloc(b.send_ptrs(), b.recv_ptrs(), 64, 33, "float32", "sum")
