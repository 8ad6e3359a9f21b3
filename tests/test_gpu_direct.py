"""GPU parity of the two all-gather forms of the ring / Simple AllReduce
(vrcclCommSetDirect): through the ranks' recv buffers (the default) and
through the FIFOs. Both must give the oracle's bits for every type, op,
rank count, ragged end and in place; switching between the two forms on
one communicator must keep both correct."""
import numpy as np
import pytest

from oracle import closed_form, ring as oring
from ring_allreduce_reduction_gb300.workloads import ELEM_SIZE, make_inputs
from tests.gpu_harness import run

pytestmark = pytest.mark.gpu

DT = ["int32", "float32", "bfloat16", "float16", "int8", "uint8", "int64", "float64"]
OPS = ["sum", "prod", "max", "min", "avg"]
INT_RANGE = {"int32": (-2**20, 2**20), "int8": (-128, 127), "uint8": (0, 255), "int64": (-2**62, 2**62)}
COUNT = {1: 12007, 2: 6003, 4: 3001, 8: 1501}  # a ragged end shorter than 16 bytes


@pytest.fixture(scope="module")
def v():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ring_allreduce_reduction_gb300 import build
    build.build()
    from ring_allreduce_reduction_gb300 import vrccl
    return vrccl


def _inputs(n, count, dtype, op, seed=0):
    if dtype in INT_RANGE:
        lo, hi = INT_RANGE[dtype]
        return make_inputs(n, count, dtype, "int_uniform", seed=seed, lo=lo, hi=hi)
    if op == "prod":
        return make_inputs(n, count, dtype, "uniform", seed=seed, lo=0.5, hi=2.0)
    return make_inputs(n, count, dtype, "normal", seed=seed)


def _same(a, b):
    return np.array_equal(np.ascontiguousarray(a).view(np.uint8), np.ascontiguousarray(b).view(np.uint8))


@pytest.mark.parametrize("direct", [True, False])
@pytest.mark.parametrize("n", [2, 3, 5, 8])
def test_direct_every_dtype_and_op(v, n, direct):
    """3 channels, 256-byte chunks: several loops, a short last loop, a
    ragged end shorter than 16 bytes; both all-gather forms."""
    comm = v.vrcclCommInit(n, 4)
    try:
        v.vrcclCommSetSchedule(comm, 3, 256)
        v.vrcclCommSetDirect(comm, direct)
        for dtype in DT:
            count = COUNT[ELEM_SIZE[dtype]]
            for op in OPS:
                x = _inputs(n, count, dtype, op, seed=n + len(op))
                y, s, b = run(v, comm, x, dtype, op, "ring", "simple")
                ref = oring.ring_allreduce(x, op, dtype, s["nchannels"], s["chunk_elems"])
                assert _same(y, ref), (dtype, op)
                ok, worst = closed_form.check(y[0], x, op, dtype)
                assert ok, worst
                assert b.canaries_intact()
        assert v.vrcclCommGetAsyncError(comm) == 0
    finally:
        v.vrcclCommDestroy(comm)


@pytest.mark.parametrize("count", [1, 4, 7, 4096, 65536 * 3 + 5])
def test_direct_inplace_and_mode_switches(v, count):
    n = 6
    comm = v.vrcclCommInit(n, 8)
    try:
        for it, (direct, inplace) in enumerate([(True, False), (True, True), (False, True), (True, False),
                                                (False, False), (True, True)]):
            v.vrcclCommSetDirect(comm, direct)
            x = _inputs(n, count, "bfloat16", "sum", seed=it)
            y, s, b = run(v, comm, x, "bfloat16", "sum", "ring", "simple", inplace=inplace)
            ref = oring.ring_allreduce(x, "sum", "bfloat16", s["nchannels"], s["chunk_elems"])
            assert _same(y, ref), (it, direct, inplace)
            assert b.canaries_intact()
        assert v.vrcclCommGetAsyncError(comm) == 0
    finally:
        v.vrcclCommDestroy(comm)


@pytest.mark.parametrize("n", [2, 3, 8])
def test_direct_counters_across_launches(v, n):
    """The direct in-edge counts carry from launch to launch (the last
    step's slices are passed over and only counted): many launches of
    different sizes and channel counts on one communicator stay exact."""
    rng = np.random.default_rng(n)
    comm = v.vrcclCommInit(n, 8)
    try:
        v.vrcclCommSetDirect(comm, True)
        for k in range(12):
            count = int(rng.integers(1, 200_000))
            v.vrcclCommSetSchedule(comm, int(rng.integers(1, 9)), int(rng.choice([256, 4096, 0])))
            x = _inputs(n, count, "float32", "sum", seed=k)
            y, s, b = run(v, comm, x, "float32", "sum", "ring", "simple")
            ref = oring.ring_allreduce(x, "sum", "float32", s["nchannels"], s["chunk_elems"])
            assert _same(y, ref), (k, count, s)
            assert b.canaries_intact()
        assert v.vrcclCommGetAsyncError(comm) == 0
    finally:
        v.vrcclCommDestroy(comm)


@pytest.mark.parametrize("n", [16, 32])
def test_direct_many_ranks(v, n):
    comm = v.vrcclCommInit(n, 8)
    try:
        v.vrcclCommSetDirect(comm, True)
        x = _inputs(n, 300_001, "float32", "sum", seed=n)
        y, s, b = run(v, comm, x, "float32", "sum", "ring", "simple")
        ref = oring.ring_allreduce(x, "sum", "float32", s["nchannels"], s["chunk_elems"])
        assert _same(y, ref) and b.canaries_intact()
    finally:
        v.vrcclCommDestroy(comm)


def test_direct_full_size_matches_fifo_form(v):
    """The bench workload (n=8, 256 MiB fp32 per rank): the direct and FIFO
    forms give the same 2 GiB of results, compared on the device; sampled
    outputs match the oracle's predictor."""
    import torch
    n, count = 8, (256 << 20) // 4
    x = make_inputs(n, count, "float32", "uniform", seed=1000)
    send = torch.from_numpy(x).to("cuda:0")
    r1 = torch.empty_like(send)
    r2 = torch.empty_like(send)
    comm = v.vrcclCommInit(n, 32)
    try:
        v.vrcclCommSetDirect(comm, False)
        v.vrcclAllReduce([send[r] for r in range(n)], [r1[r] for r in range(n)], count, "float32", "sum", "ring",
                         "simple", comm)
        s1 = v.vrcclCommGetLastSchedule(comm)
        v.vrcclCommSetDirect(comm, True)
        v.vrcclAllReduce([send[r] for r in range(n)], [r2[r] for r in range(n)], count, "float32", "sum", "ring",
                         "simple", comm)
        torch.cuda.synchronize()
        assert v.vrcclCommGetLastSchedule(comm) == s1
        assert v.vrcclCommGetAsyncError(comm) == 0
        assert torch.equal(r1.view(torch.int32), r2.view(torch.int32))
        idx = np.unique(np.concatenate([np.random.default_rng(9).choice(count, 100_000, replace=False),
                                        [0, count - 1]]))
        got = r2[3].cpu().numpy()[idx]
        assert _same(got, oring.ring_predict(x, "sum", "float32", s1["nchannels"], s1["chunk_elems"], idx))
    finally:
        v.vrcclCommDestroy(comm)
