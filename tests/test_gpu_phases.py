"""GPU parity of the standalone ReduceScatter and AllGather against the oracle.

ReduceScatter results must be bit-identical to the oracle's reduce-scatter
step machine (the association depends only on the block, so no schedule
parameter enters) and within the closed-form bound; AllGather results must
be the concatenation of the send buffers, bit for bit. Canary bytes around
every buffer must survive.
"""
import ctypes

import numpy as np
import pytest

from oracle import closed_form, phases, ring as oring
from ring_allreduce_reduction_gb300.workloads import ELEM_SIZE, STORAGE, make_inputs

pytestmark = pytest.mark.gpu

DT = ["int32", "float32", "bfloat16", "float16"]
OPS = ["sum", "prod", "max", "min", "avg"]
GUARD = 256
CANARY = 0xA5


@pytest.fixture(scope="module")
def v():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ring_allreduce_reduction_gb300 import build
    build.build()
    from ring_allreduce_reduction_gb300 import vrccl
    return vrccl


class Rows:
    """n rows of `nbytes` data each, with canary guards, on cuda:0."""

    def __init__(self, n, nbytes, data=None):
        import torch
        self.n, self.nbytes = n, nbytes
        self.row = (nbytes + 2 * GUARD + 255) // 256 * 256
        host = np.full((n, self.row), CANARY, dtype=np.uint8)
        if data is not None:
            host[:, GUARD:GUARD + nbytes] = np.ascontiguousarray(data).view(np.uint8).reshape(n, -1)
        self.t = torch.from_numpy(host).to("cuda:0")

    def ptr(self, r, byte_off=0):
        return self.t.data_ptr() + r * self.row + GUARD + byte_off

    def data(self, dtype):
        import torch
        torch.cuda.synchronize()
        h = self.t.cpu().numpy()
        return np.ascontiguousarray(h[:, GUARD:GUARD + self.nbytes]).view(STORAGE[dtype]).reshape(self.n, -1)

    def canaries(self):
        import torch
        torch.cuda.synchronize()
        h = self.t.cpu().numpy()
        return bool(np.all(h[:, :GUARD] == CANARY) and np.all(h[:, GUARD + self.nbytes:] == CANARY))


INT_RANGE = {"int32": (-2**20, 2**20), "int8": (-128, 127), "uint8": (0, 255), "int64": (-2**62, 2**62)}


def _inputs(n, count, dtype, op, seed=0):
    if dtype in INT_RANGE:
        lo, hi = INT_RANGE[dtype]
        return make_inputs(n, count, dtype, "int_uniform", seed=seed, lo=lo, hi=hi)
    if op == "prod":
        return make_inputs(n, count, dtype, "uniform", seed=seed, lo=0.5, hi=2.0)
    return make_inputs(n, count, dtype, "normal", seed=seed)


def _rs(v, comm, x, dtype, op, proto, inplace=False):
    n, total = x.shape
    b = total // n
    E = ELEM_SIZE[dtype]
    send = Rows(n, total * E, x)
    if inplace:
        recv_ptrs = [send.ptr(r, r * b * E) for r in range(n)]
        recv = None
    else:
        recv = Rows(n, b * E)
        recv_ptrs = [recv.ptr(r) for r in range(n)]
    v.vrcclReduceScatter([send.ptr(r) for r in range(n)], recv_ptrs, b, dtype, op, proto, comm)
    if inplace:
        full = send.data(dtype)
        y = np.stack([full[r, r * b:(r + 1) * b] for r in range(n)])
        ok = send.canaries()
    else:
        y = recv.data(dtype)
        ok = recv.canaries() and send.canaries()
        assert np.array_equal(send.data(dtype).view(np.uint8), x.view(np.uint8)), "send buffers changed"
    return y, ok


def _check_rs(x, y, dtype, op):
    n, total = x.shape
    b = total // n
    ref = phases.ring_reduce_scatter(x, op, dtype)
    bad = np.nonzero(y.view(np.uint8) != ref.view(np.uint8))
    assert bad[0].size == 0, f"{bad[0].size} bytes differ from the oracle, first at rank/byte {bad[0][0]}/{bad[1][0]}"
    for r in range(n):
        ok, worst = closed_form.check(y[r], x[:, r * b:(r + 1) * b], op, dtype)
        assert ok, (r, worst)


@pytest.mark.parametrize("proto", ["simple", "ll", "ll128"])
def test_reduce_scatter_every_dtype_and_op(v, proto):
    """n=5, 3 channels, a 256-byte chunk: several loops, a short last loop
    and channels of unequal length within each block."""
    n = 5
    comm = v.vrcclCommInit(n, 4)
    try:
        v.vrcclCommSetSchedule(comm, 3, 256)
        for dtype in DT:
            b = 1000 if ELEM_SIZE[dtype] == 4 else 1992
            for op in OPS:
                x = _inputs(n, n * b, dtype, op, seed=len(op))
                y, ok = _rs(v, comm, x, dtype, op, proto)
                _check_rs(x, y, dtype, op)
                assert ok, "canary overwritten"
                s = v.vrcclCommGetLastSchedule(comm)
                assert s["algo"] == "ring" and s["proto"] == proto and s["nchannels"] == 3
        assert v.vrcclCommGetAsyncError(comm) == 0
    finally:
        v.vrcclCommDestroy(comm)


@pytest.mark.parametrize("n", [2, 3, 8, 16])
@pytest.mark.parametrize("proto", ["simple", "ll", "ll128", "auto"])
def test_reduce_scatter_ranks_and_inplace(v, n, proto):
    comm = v.vrcclCommInit(n, 8)
    try:
        for inplace in (False, True):
            x = _inputs(n, n * 4100, "float32", "sum", seed=n)
            y, ok = _rs(v, comm, x, "float32", "sum", proto, inplace)
            _check_rs(x, y, "float32", "sum")
            assert ok
            x = _inputs(n, n * 4096, "bfloat16", "avg", seed=n + 1)
            y, ok = _rs(v, comm, x, "bfloat16", "avg", proto, inplace)
            _check_rs(x, y, "bfloat16", "avg")
            assert ok
    finally:
        v.vrcclCommDestroy(comm)


def _ag(v, comm, x, dtype, proto, inplace=False):
    n, b = x.shape
    E = ELEM_SIZE[dtype]
    recv = Rows(n, n * b * E)
    if inplace:  # each rank's block already sits at its place in the recv buffer
        import torch
        host = recv.t.cpu().numpy()
        for r in range(n):
            host[r, GUARD + r * b * E:GUARD + (r + 1) * b * E] = x[r].view(np.uint8)
        recv.t.copy_(torch.from_numpy(host))
        send_ptrs = [recv.ptr(r, r * b * E) for r in range(n)]
        send = None
    else:
        send = Rows(n, b * E, x)
        send_ptrs = [send.ptr(r) for r in range(n)]
    v.vrcclAllGather(send_ptrs, [recv.ptr(r) for r in range(n)], b, dtype, proto, comm)
    y = recv.data(dtype)
    ok = recv.canaries() and (send is None or send.canaries())
    return y, ok


@pytest.mark.parametrize("proto", ["simple", "ll", "ll128", "auto"])
@pytest.mark.parametrize("n", [2, 5, 8])
def test_all_gather_is_the_concatenation(v, proto, n):
    comm = v.vrcclCommInit(n, 4)
    try:
        for dtype, b in (("bfloat16", 8 * 777), ("float32", 4 * 1001), ("int32", 4)):
            for inplace in (False, True):
                x = _inputs(n, b, dtype, "sum", seed=b)
                y, ok = _ag(v, comm, x, dtype, proto, inplace)
                want = phases.ring_all_gather(x)
                assert np.array_equal(y.view(np.uint8), want.view(np.uint8)), (dtype, inplace)
                assert ok
    finally:
        v.vrcclCommDestroy(comm)


@pytest.mark.parametrize("direct", [True, False])
@pytest.mark.parametrize("n", [2, 3, 5, 8])
def test_all_gather_both_forms(v, n, direct):
    """Simple AllGather with its blocks moved through the recv buffers (the
    default) and through the FIFOs: 3 channels and 256-byte chunks (several
    loops and a short last one), 1-, 2-, 4- and 8-byte types, in place and
    not, several launches on one communicator."""
    comm = v.vrcclCommInit(n, 4)
    try:
        v.vrcclCommSetDirect(comm, direct)
        v.vrcclCommSetSchedule(comm, 3, 256)
        for dtype, b in (("bfloat16", 8 * 777), ("float32", 4 * 1001), ("int8", 16 * 301), ("float64", 2 * 999)):
            for inplace in (False, True):
                x = _inputs(n, b, dtype, "sum", seed=b + n)
                y, ok = _ag(v, comm, x, dtype, "simple", inplace)
                want = phases.ring_all_gather(x)
                assert np.array_equal(y.view(np.uint8), want.view(np.uint8)), (dtype, inplace)
                assert ok
        assert v.vrcclCommGetAsyncError(comm) == 0
    finally:
        v.vrcclCommDestroy(comm)


def test_one_rank_and_empty_and_misaligned(v):
    import torch
    comm = v.vrcclCommInit(1, 2)
    try:
        x = make_inputs(1, 1001, "float16", "normal", seed=1)  # 2002 bytes: one rank needs no block rule
        y, ok = _rs(v, comm, x, "float16", "avg", "simple")
        assert np.array_equal(y.view(np.uint8), phases.ring_reduce_scatter(x, "avg", "float16").view(np.uint8))
        y, ok2 = _ag(v, comm, x, "float16", "ll")
        assert np.array_equal(y.view(np.uint8), x.view(np.uint8)) and ok and ok2
    finally:
        v.vrcclCommDestroy(comm)
    comm = v.vrcclCommInit(4, 2)
    try:
        buf = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda:0")
        p = [buf.data_ptr() + r * 4096 for r in range(4)]
        q = [buf.data_ptr() + 32768 + r * 4096 for r in range(4)]
        v.vrcclReduceScatter(p, q, 0, "float32", "sum", "simple", comm)   # empty: nothing launched
        v.vrcclAllGather(p, q, 0, "float32", "simple", comm)
        code = v.raw_call("vrcclReduceScatter", (ctypes.c_void_p * 4)(*p), (ctypes.c_void_p * 4)(*q), 6, 1, 0, 0,
                          comm, None)
        assert code == 1, "a 24-byte block must be rejected"
        code = v.raw_call("vrcclAllGather", (ctypes.c_void_p * 4)(*p), (ctypes.c_void_p * 4)(*q), 3, 2, 0,
                          comm, None)
        assert code == 1, "a 6-byte block must be rejected"
        # overlapping blocks: recv buffers of 4 x 1 KiB starting 1 KiB apart in the send rows
        code = v.raw_call("vrcclAllGather", (ctypes.c_void_p * 4)(*p), (ctypes.c_void_p * 4)(*p), 256, 1, 0,
                          comm, None)
        assert code == 1, "overlapping buffers must be rejected"
        torch.cuda.synchronize()
        assert v.vrcclCommGetAsyncError(comm) == 0
    finally:
        v.vrcclCommDestroy(comm)


def test_collectives_share_one_communicator(v):
    """AllReduce, ReduceScatter and AllGather interleaved on one communicator
    and stream, every protocol: the FIFO counters and LL flags carry over
    from one kind of launch to the next."""
    import torch
    n = 6
    comm = v.vrcclCommInit(n, 4)
    try:
        for it in range(3):
            for proto in ("ll", "simple", "ll128"):
                x = _inputs(n, n * 2048, "float32", "sum", seed=it)
                y, ok = _rs(v, comm, x, "float32", "sum", proto)
                _check_rs(x, y, "float32", "sum")
                g, ok2 = _ag(v, comm, y, "float32", proto)
                assert np.array_equal(g.view(np.uint8), phases.ring_all_gather(y).view(np.uint8))
                xa = _inputs(n, 5000, "bfloat16", "sum", seed=it + 7)
                send = torch.from_numpy(xa.view(np.int16)).to("cuda:0")
                recv = torch.empty_like(send)
                v.vrcclAllReduce([send[r] for r in range(n)], [recv[r] for r in range(n)], 5000, "bfloat16", "sum",
                                 "ring", proto, comm)
                sched = v.vrcclCommGetLastSchedule(comm)
                ref = oring.ring_allreduce(xa, "sum", "bfloat16", sched["nchannels"], sched["chunk_elems"])
                assert np.array_equal(recv.cpu().numpy().view(np.uint16), ref.view(np.uint16))
                assert ok and ok2
        assert v.vrcclCommGetAsyncError(comm) == 0
    finally:
        v.vrcclCommDestroy(comm)


def test_reduce_scatter_full_size_sampled(v):
    """n=8, 256 MiB fp32 send buffer per rank (32 MiB blocks), sum, Simple,
    channel count chosen by the library; sampled outputs bit-exact."""
    import torch
    n, b = 8, (32 << 20) // 4
    x = make_inputs(n, n * b, "float32", "uniform", seed=21)
    send = torch.from_numpy(x).to("cuda:0")
    recv = torch.empty((n, b), dtype=torch.float32, device="cuda:0")
    comm = v.vrcclCommInit(n, 32)
    try:
        v.vrcclReduceScatter([send[r] for r in range(n)], [recv[r] for r in range(n)], b, "float32", "sum",
                             "simple", comm)
        torch.cuda.synchronize()
        assert v.vrcclCommGetAsyncError(comm) == 0
        idx = np.unique(np.concatenate([np.random.default_rng(0).choice(b, 100_000, replace=False), [0, b - 1]]))
        for r in range(n):
            got = recv[r].cpu().numpy()[idx]
            ref = phases.reduce_scatter_predict(x, "sum", "float32", r, idx)
            assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), r
        # then the AllGather of those blocks: every recv buffer equals the blocks in order, on the device
        out = torch.empty((n, n * b), dtype=torch.float32, device="cuda:0")
        v.vrcclAllGather([recv[r] for r in range(n)], [out[r] for r in range(n)], b, "float32", "simple", comm)
        torch.cuda.synchronize()
        flat = recv.reshape(-1)
        for r in range(n):
            assert torch.equal(out[r], flat), r
        assert v.vrcclCommGetAsyncError(comm) == 0
    finally:
        v.vrcclCommDestroy(comm)
