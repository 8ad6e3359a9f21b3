"""The element-range split of one problem over several GPUs, emulated on
one GPU: the parts run one after another, each on a communicator of its
own (nothing waits across parts), and each part's result must be the
oracle's ring association for the schedule that part ran; the parts
concatenated must equal the closed form where the sum is exact."""
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


@pytest.mark.parametrize("nshards,count,dtype", [(2, 1_000_003, "float32"), (3, 250_001, "bfloat16"),
                                                  (8, 77_777, "float32")])
def test_parts_of_one_problem(v, nshards, count, dtype):
    n = 8
    if dtype == "float32":
        x = make_inputs(n, count, dtype, "int_uniform", seed=nshards, lo=-8, hi=8)  # exact sums
    else:
        x = make_inputs(n, count, dtype, "normal", seed=nshards)
    y = np.empty_like(x)
    pos = 0
    for s in range(nshards):
        off, ln = v.vrcclShardRange(count, dtype, nshards, s)
        assert off == pos
        pos += ln
        if ln == 0:
            continue
        part = np.ascontiguousarray(x[:, off:off + ln])
        comm = v.vrcclCommInit(n, 32)
        try:
            b = Buffers(part, dtype)
            v.vrcclAllReduce(b.send_ptrs(), b.recv_ptrs(), ln, dtype, "sum", "ring", "auto", comm)
            got = b.result()
            sched = v.vrcclCommGetLastSchedule(comm)
            assert v.vrcclCommGetAsyncError(comm) == 0
        finally:
            v.vrcclCommDestroy(comm)
        assert b.canaries_intact()
        ref = oring.ring_allreduce(part, "sum", dtype, sched["nchannels"], sched["chunk_elems"])
        assert np.array_equal(got.view(np.uint8), ref.view(np.uint8)), (s, sched)
        y[:, off:off + ln] = got
    assert pos == count
    ok, worst = closed_form.check(y[0], x, "sum", dtype)
    assert ok, worst
    if dtype == "float32":
        assert np.array_equal(y[0], x.astype(np.float64).sum(axis=0).astype(np.float32))
