"""GPU parity of the int8, uint8, int64 and float64 paths: every
algorithm, protocol and op against the oracle replaying the reported
schedule (bit for bit), the order-free closed form, identical recv
buffers and intact canaries; the phases, groups and the one-shot too."""
import numpy as np
import pytest

from oracle import closed_form, phases, ring as oring, tree as otree
from ring_allreduce_reduction_gb300.workloads import ELEM_SIZE, STORAGE, make_inputs
from tests.gpu_harness import run

pytestmark = pytest.mark.gpu

NEW = ["int8", "uint8", "int64", "float64"]
OPS = ["sum", "prod", "max", "min", "avg"]
RANGE = {"int8": (-128, 127), "uint8": (0, 255), "int64": (-2**62, 2**62)}


@pytest.fixture(scope="module")
def v():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ring_allreduce_reduction_gb300 import build
    build.build()
    from ring_allreduce_reduction_gb300 import vrccl
    return vrccl


def _inputs(n, count, dtype, op, seed=0):
    if dtype in RANGE:
        lo, hi = RANGE[dtype]
        return make_inputs(n, count, dtype, "int_uniform", seed=seed, lo=lo, hi=hi)
    if op == "prod":
        return make_inputs(n, count, dtype, "uniform", seed=seed, lo=0.5, hi=2.0)
    return make_inputs(n, count, dtype, "normal", seed=seed)


def _oracle(x, dtype, op, s):
    if s["algo"] == "tree":
        return otree.tree_allreduce(x, op, dtype, s["nchannels"])
    return oring.ring_allreduce(x, op, dtype, s["nchannels"], s["chunk_elems"])


def _parity(x, y, dtype, op, s):
    for r in range(1, x.shape[0]):
        assert np.array_equal(y[r].view(np.uint8), y[0].view(np.uint8)), f"rank {r} differs"
    ref = _oracle(x, dtype, op, s)
    bad = np.nonzero(y[0].view(np.uint8) != ref[0].view(np.uint8))[0]
    assert bad.size == 0, f"{bad.size} bytes differ from the oracle, first at {bad[:8]} ({s})"
    ok, worst = closed_form.check(y[0], x, op, dtype)
    assert ok, worst


def _count(dtype):
    # several loops of 256-byte chunks over 3 channels, and a ragged end
    return {1: 12003, 8: 1501}[ELEM_SIZE[dtype]]


@pytest.mark.parametrize("proto", ["simple", "ll", "ll128"])
@pytest.mark.parametrize("algo", ["ring", "tree"])
@pytest.mark.parametrize("n", [2, 5, 8])
def test_every_new_dtype_and_op(v, proto, algo, n):
    comm = v.vrcclCommInit(n, 4)
    try:
        v.vrcclCommSetSchedule(comm, 3, 256)
        for dtype in NEW:
            for op in OPS:
                x = _inputs(n, _count(dtype), dtype, op, seed=n + len(op))
                y, s, b = run(v, comm, x, dtype, op, algo, proto)
                assert s["algo"] == algo and s["proto"] == proto
                _parity(x, y, dtype, op, s)
                assert b.canaries_intact(), (dtype, op)
        assert v.vrcclCommGetAsyncError(comm) == 0
    finally:
        v.vrcclCommDestroy(comm)


@pytest.mark.parametrize("dtype", NEW)
def test_new_dtypes_default_schedules_and_in_place(v, dtype):
    """algo / protocol auto at small, middle and large sizes (the tuning
    table's shapes, LL128's wide kernels included), in place at one size."""
    n = 8
    comm = v.vrcclCommInit(n, 32)
    try:
        E = ELEM_SIZE[dtype]
        for nbytes, algo, proto, ops in ((1000, "auto", "auto", ("sum", "max", "avg")),
                                         (1 << 20, "auto", "auto", ("sum", "max", "avg")),
                                         (3 << 20, "ring", "ll128", ("sum",)), (3 << 20, "tree", "ll128", ("sum",)),
                                         (24 << 20, "auto", "auto", ("sum",)), (24 << 20, "tree", "simple", ("avg",))):
            count = nbytes // E + 3
            for op in ops:
                x = _inputs(n, count, dtype, op, seed=nbytes % 97)
                y, s, b = run(v, comm, x, dtype, op, algo, proto, inplace=(nbytes == 1 << 20))
                _parity(x, y, dtype, op, s)
                assert b.canaries_intact()
        assert v.vrcclCommGetAsyncError(comm) == 0
    finally:
        v.vrcclCommDestroy(comm)


@pytest.mark.parametrize("dtype", NEW)
def test_new_dtypes_oneshot(v, dtype):
    n = 6
    comm = v.vrcclCommInit(n, 8)
    try:
        for op in OPS:
            x = _inputs(n, 40_000 + 5, dtype, op, seed=3)
            y, s, b = run(v, comm, x, dtype, op, "oneshot", "simple")
            ref = oring.ring_allreduce(x, op, dtype, s["nchannels"], s["chunk_elems"])
            assert np.array_equal(y.view(np.uint8), ref.view(np.uint8)), op
            assert b.canaries_intact()
        assert v.vrcclCommGetAsyncError(comm) == 0
    finally:
        v.vrcclCommDestroy(comm)


@pytest.mark.parametrize("proto", ["simple", "ll", "ll128"])
def test_new_dtypes_phases(v, proto):
    """ReduceScatter of every op and AllGather, blocks of whole 16-byte units."""
    import torch
    n = 5
    comm = v.vrcclCommInit(n, 4)
    try:
        for dtype in NEW:
            E = ELEM_SIZE[dtype]
            blk = 16 * 301 // E
            for op in OPS:
                x = _inputs(n, n * blk, dtype, op, seed=11)
                xs = torch.from_numpy(np.ascontiguousarray(x).view(np.uint8)).to("cuda:0")
                out = torch.empty((n, blk * E), dtype=torch.uint8, device="cuda:0")
                v.vrcclReduceScatter([xs[r] for r in range(n)], [out[r] for r in range(n)], blk, dtype, op, proto, comm)
                torch.cuda.synchronize()
                y = out.cpu().numpy().view(STORAGE[dtype])
                ref = phases.ring_reduce_scatter(x, op, dtype)
                assert np.array_equal(y.view(np.uint8), ref.view(np.uint8)), (dtype, op)
            x = _inputs(n, blk, dtype, "sum", seed=12)
            xs = torch.from_numpy(np.ascontiguousarray(x).view(np.uint8)).to("cuda:0")
            out = torch.empty((n, n * blk * E), dtype=torch.uint8, device="cuda:0")
            v.vrcclAllGather([xs[r] for r in range(n)], [out[r] for r in range(n)], blk, dtype, proto, comm)
            torch.cuda.synchronize()
            assert np.array_equal(out.cpu().numpy(), np.ascontiguousarray(phases.ring_all_gather(x)).view(
                np.uint8).reshape(n, -1)), dtype
        assert v.vrcclCommGetAsyncError(comm) == 0
    finally:
        v.vrcclCommDestroy(comm)


def test_new_dtypes_in_one_group(v):
    """A group mixing the new types with each other and with fp32: every
    call bit-exact under the schedule reported for it."""
    import torch
    n = 8
    comm = v.vrcclCommInit(n, 32)
    try:
        spec = [("int8", "sum", 100_000), ("uint8", "max", 70_001), ("int64", "avg", 30_000),
                ("float64", "sum", 50_000), ("float64", "prod", 9_999), ("float32", "sum", 40_000)]
        data = []
        v.vrcclGroupStart()
        for i, (dt, op, cnt) in enumerate(spec):
            x = _inputs(n, cnt, dt, op, seed=i)
            E = ELEM_SIZE[dt]
            row = -(-cnt * E // 256) * 256
            h = np.zeros((n, row), dtype=np.uint8)
            h[:, :cnt * E] = np.ascontiguousarray(x).view(np.uint8).reshape(n, -1)
            a = torch.from_numpy(h).to("cuda:0")
            b = torch.empty_like(a)
            data.append((dt, op, cnt, x, a, b))
            v.vrcclAllReduce([a[r] for r in range(n)], [b[r] for r in range(n)], cnt, dt, op, "auto", "auto", comm)
        v.vrcclGroupEnd()
        torch.cuda.synchronize()
        assert v.vrcclCommGetAsyncError(comm) == 0
        for i, (dt, op, cnt, x, a, b) in enumerate(data):
            s = v.vrcclCommGetGroupSchedule(comm, i)
            y = np.ascontiguousarray(b.cpu().numpy()[:, :cnt * ELEM_SIZE[dt]]).view(STORAGE[dt])
            ref = _oracle(x, dt, op, s)
            assert np.array_equal(y.view(np.uint8), ref.view(np.uint8)), (dt, op, s)
    finally:
        v.vrcclCommDestroy(comm)


@pytest.mark.parametrize("algo", ["ring", "tree"])
def test_new_dtypes_ll128_wide_kernels(v, algo):
    """Four channels and 8 MiB per rank leave every agent many whole LL128
    slices, so the wide LL128 kernels of types 4-7 run."""
    n = 8
    comm = v.vrcclCommInit(n, 4)
    try:
        v.vrcclCommSetSchedule(comm, 4, 0)
        for dtype in NEW:
            count = (8 << 20) // ELEM_SIZE[dtype] + 5
            x = _inputs(n, count, dtype, "sum", seed=21)
            y, s, b = run(v, comm, x, dtype, "sum", algo, "ll128")
            assert s["proto"] == "ll128" and s["nchannels"] == 4
            _parity(x, y, dtype, "sum", s)
            assert b.canaries_intact()
        assert v.vrcclCommGetAsyncError(comm) == 0
    finally:
        v.vrcclCommDestroy(comm)
