"""GPU parity: the sm_103a path through the C ABI against the CPU oracle.

Floating results must be bit-identical to the oracle replaying the same
schedule (the library reports its channel count and chunk size); integer
results must also equal the order-free closed form; every result must be
within the stated tolerance of the float64 value; all n recv buffers must
be identical; canaries around every buffer must be untouched.
"""
import numpy as np
import pytest

from oracle import closed_form, ring as oring, tree as otree
from ring_allreduce_reduction_gb300.workloads import ELEM_SIZE, STORAGE, make_inputs
from tests.gpu_harness import Buffers, run

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


def _oracle(x, dtype, op, sched):
    if sched["algo"] == "tree":
        return otree.tree_allreduce(x, op, dtype, sched["nchannels"])
    return oring.ring_allreduce(x, op, dtype, sched["nchannels"], sched["chunk_elems"])


def _assert_parity(x, y, dtype, op, sched):
    n = x.shape[0]
    for r in range(1, n):
        assert np.array_equal(y[r].view(np.uint8), y[0].view(np.uint8)), f"rank {r} differs from rank 0"
    ref = _oracle(x, dtype, op, sched)
    bad = np.nonzero(y[0].view(np.uint8) != ref[0].view(np.uint8))[0]
    assert bad.size == 0, f"{bad.size} bytes differ from the oracle, first at byte {bad[:8]} ({sched})"
    ok, worst = closed_form.check(y[0], x, op, dtype)
    assert ok, f"outside tolerance: worst ratio {worst}"


def test_config_small_exact(v):
    """n=4, 4096 fp32 integers in [-8, 8], one channel, ring, Simple, sum:
    exact, so equal to the closed form whatever the order."""
    x = make_inputs(4, 4096, "float32", "int_uniform", seed=0, lo=-8, hi=8)
    comm = v.vrcclCommInit(4, 1)
    try:
        y, sched, b = run(v, comm, x, "float32", "sum", "ring", "simple")
        assert sched["nchannels"] == 1 and sched["algo"] == "ring" and sched["proto"] == "simple"
        assert np.array_equal(y[0].astype(np.float64), x.astype(np.float64).sum(axis=0))
        _assert_parity(x, y, "float32", "sum", sched)
        assert b.canaries_intact()
    finally:
        v.vrcclCommDestroy(comm)


@pytest.mark.parametrize("proto", ["simple", "ll", "ll128"])
@pytest.mark.parametrize("algo", ["ring", "tree"])
def test_every_dtype_and_op(v, proto, algo):
    """n=5 (odd), 3 channels, a chunk of 256 bytes (several loops and a
    short tail loop), a ragged count."""
    n = 5
    comm = v.vrcclCommInit(n, 4)
    try:
        v.vrcclCommSetSchedule(comm, 3, 256)
        for dtype in DT:
            for op in OPS:
                count = 3001 if ELEM_SIZE[dtype] == 2 else 2999
                x = _inputs(n, count, dtype, op, seed=10 * DT.index(dtype) + OPS.index(op))
                y, sched, b = run(v, comm, x, dtype, op, algo, proto)
                assert sched["algo"] == algo and sched["proto"] == proto and sched["nchannels"] == 3
                _assert_parity(x, y, dtype, op, sched)
                assert b.canaries_intact(), (dtype, op)
        assert v.vrcclCommGetAsyncError(comm) == 0
    finally:
        v.vrcclCommDestroy(comm)


@pytest.mark.parametrize("n", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("proto", ["simple", "ll", "ll128"])
def test_shapes_and_edges(v, n, proto):
    """Counts below n, below one 16-byte unit, around unit and line
    boundaries, several channels (some empty)."""
    comm = v.vrcclCommInit(n, 8)
    try:
        for dtype in ("float32", "bfloat16"):
            for count in (1, 3, 7, 8, 15, 16, 17, 31, 61, 120, 1000, 4097):
                for nch in (1, 3, 8):
                    v.vrcclCommSetSchedule(comm, nch, 0)
                    x = _inputs(n, count, dtype, "sum", seed=count)
                    for algo in ("ring", "tree"):
                        y, sched, b = run(v, comm, x, dtype, "sum", algo, proto)
                        _assert_parity(x, y, dtype, "sum", sched)
                        assert b.canaries_intact()
    finally:
        v.vrcclCommDestroy(comm)


@pytest.mark.parametrize("proto", ["simple", "ll", "ll128"])
def test_in_place(v, proto):
    n = 6
    comm = v.vrcclCommInit(n, 4)
    try:
        v.vrcclCommSetSchedule(comm, 2, 512)
        for algo in ("ring", "tree"):
            x = _inputs(n, 5003, "float32", "sum", seed=3)
            y, sched, b = run(v, comm, x, "float32", "sum", algo, proto, inplace=True)
            _assert_parity(x, y, "float32", "sum", sched)
            assert b.canaries_intact()
    finally:
        v.vrcclCommDestroy(comm)


def test_repeated_calls_keep_fifo_state(v):
    """Step counters and LL flags persist across launches on one
    communicator: many calls of changing size and protocol stay correct."""
    n = 4
    comm = v.vrcclCommInit(n, 4)
    try:
        rng = np.random.default_rng(5)
        for it in range(40):
            proto = ["simple", "ll", "ll128"][it % 3]
            algo = ["ring", "tree"][(it // 3) % 2]
            count = int(rng.integers(1, 20000))
            v.vrcclCommSetSchedule(comm, int(rng.integers(1, 5)), 0)
            x = _inputs(n, count, "bfloat16", "sum", seed=it)
            y, sched, _ = run(v, comm, x, "bfloat16", "sum", algo, proto)
            _assert_parity(x, y, "bfloat16", "sum", sched)
    finally:
        v.vrcclCommDestroy(comm)


@pytest.mark.parametrize("proto", ["simple", "ll", "ll128"])
def test_many_loops_wrap_the_fifo(v, proto):
    """n=8, 2^20 fp32 per rank, 4 channels, small chunks: hundreds of FIFO
    steps per edge, so every slot is reused many times."""
    n, count = 8, 1 << 20
    comm = v.vrcclCommInit(n, 4)
    try:
        v.vrcclCommSetSchedule(comm, 4, 4096)
        x = _inputs(n, count, "float32", "sum", seed=9)
        y, sched, b = run(v, comm, x, "float32", "sum", "ring", proto)
        assert sched["chunk_elems"] == 1024
        _assert_parity(x, y, "float32", "sum", sched)
        assert b.canaries_intact()
    finally:
        v.vrcclCommDestroy(comm)


def test_tree_large_rank_counts(v):
    for n in (16, 32, 72):
        comm = v.vrcclCommInit(n, 2)
        try:
            x = _inputs(n, 20000, "float32", "sum", seed=n)
            for proto in ("simple", "ll128"):
                y, sched, _ = run(v, comm, x, "float32", "sum", "tree", proto)
                _assert_parity(x, y, "float32", "sum", sched)
            y, sched, _ = run(v, comm, x, "float32", "sum", "ring", "simple")
            _assert_parity(x, y, "float32", "sum", sched)
        finally:
            v.vrcclCommDestroy(comm)


def test_page_example_first_element(v):
    """The single-process AllReduce example: 32M floats per rank, element 0
    of rank i is i, the rest 0; every recv buffer starts with n(n-1)/2."""
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "allreduce_example.json")) as f:
        fx = json.load(f)
    import torch
    count = fx["example_count"]
    for case in fx["cases"]:
        n = case["n"]
        if n > 8:
            continue
        comm = v.vrcclCommInit(n, 32)
        try:
            send = torch.zeros((n, count), dtype=torch.float32, device="cuda:0")
            send[:, 0] = torch.arange(n, dtype=torch.float32, device="cuda:0")
            recv = torch.full((n, count), -1.0, dtype=torch.float32, device="cuda:0")
            v.vrcclAllReduce([send[r] for r in range(n)], [recv[r] for r in range(n)], count, "float32", "sum",
                             "auto", "auto", comm)
            torch.cuda.synchronize()
            assert torch.all(recv[:, 0] == case["expected_first"])
            assert torch.count_nonzero(recv[:, 1:]).item() == 0
        finally:
            v.vrcclCommDestroy(comm)


def test_count_zero_touches_nothing(v):
    comm = v.vrcclCommInit(3, 2)
    try:
        x = _inputs(3, 64, "float32", "sum")
        b = Buffers(x, "float32")
        v.vrcclAllReduce(b.send_ptrs(), b.recv_ptrs(), 0, "float32", "sum", "ring", "simple", comm)
        import torch
        torch.cuda.synchronize()
        assert np.all(b.recv.cpu().numpy() == 0xA5)
    finally:
        v.vrcclCommDestroy(comm)


def test_argument_errors(v):
    comm = v.vrcclCommInit(2, 2)
    try:
        x = _inputs(2, 64, "float32", "sum")
        b = Buffers(x, "float32")
        s, r = b.send_ptrs(), b.recv_ptrs()
        with pytest.raises(v.VrcclError, match="InvalidArgument"):
            v.vrcclAllReduce([s[0] + 4, s[1]], r, 64, "float32", "sum", "ring", "simple", comm)
        with pytest.raises(v.VrcclError, match="InvalidArgument"):  # rank 1's output overlaps rank 0's input
            v.vrcclAllReduce(s, [r[0], s[0] + 16], 64, "float32", "sum", "ring", "simple", comm)
        with pytest.raises(v.VrcclError, match="InvalidArgument"):
            v.vrcclAllReduce(s, r, 64, len(v.DTYPES), "sum", "ring", "simple", comm)  # past the last type
        with pytest.raises(v.VrcclError, match="InvalidArgument"):
            v.vrcclCommSetSchedule(comm, 3, 0)  # more channels than the communicator has
    finally:
        v.vrcclCommDestroy(comm)


@pytest.mark.parametrize("proto", ["simple", "ll", "ll128"])
def test_timeout_is_reported_not_hung(v, proto):
    """An agent that stops (a flag nothing will set) makes its peers' waits
    run out: the launch ends, the status says vrcclTimeout, the
    communicator refuses further work, and the GPU context stays usable."""
    import torch
    n = 4
    comm = v.vrcclCommInit(n, 2)
    try:
        v.vrcclCommSetTimeout(comm, 300)
        v.vrcclCommSetSchedule(comm, 2, 0)
        v.vrcclCommInjectFault(comm, 1, 0, 2)
        x = _inputs(n, 50000, "float32", "sum")
        b = Buffers(x, "float32")
        v.vrcclAllReduce(b.send_ptrs(), b.recv_ptrs(), b.count, "float32", "sum", "ring", proto, comm)
        torch.cuda.synchronize()
        assert v.RESULTS[v.vrcclCommGetAsyncError(comm)] == "vrcclTimeout"
        info = v.vrcclCommGetErrorInfo(comm)
        assert 0 <= info["rank"] < n and 0 <= info["channel"] < 2
        with pytest.raises(v.VrcclError, match="InvalidUsage"):
            v.vrcclAllReduce(b.send_ptrs(), b.recv_ptrs(), b.count, "float32", "sum", "ring", proto, comm)
    finally:
        v.vrcclCommDestroy(comm)
    # the device is fine: a fresh communicator works
    comm = v.vrcclCommInit(n, 2)
    try:
        x = _inputs(n, 1000, "float32", "sum")
        y, sched, _ = run(v, comm, x, "float32", "sum", "ring", proto)
        _assert_parity(x, y, "float32", "sum", sched)
    finally:
        v.vrcclCommDestroy(comm)


def test_abort(v):
    import torch
    comm = v.vrcclCommInit(3, 1)
    try:
        v.vrcclCommAbort(comm)
        x = _inputs(3, 100, "float32", "sum")
        b = Buffers(x, "float32")
        with pytest.raises(v.VrcclError, match="InvalidUsage"):
            v.vrcclAllReduce(b.send_ptrs(), b.recv_ptrs(), b.count, "float32", "sum", "ring", "simple", comm)
        torch.cuda.synchronize()
        assert v.RESULTS[v.vrcclCommGetAsyncError(comm)] == "vrcclAborted"
    finally:
        v.vrcclCommDestroy(comm)


def _hostile_2byte(n, count, dtype, seed):
    """Bit patterns of the type drawn over every exponent (NaN and infinity
    excluded), a quarter of them subnormal, with zeros of both signs and
    values next to the largest finite one; summing them rounds at every
    exponent distance, overflows to infinity and meets subnormals."""
    g = np.random.default_rng(seed)
    if dtype == "bfloat16":
        exp_bits, man_bits, max_finite = 8, 7, 0x7F7F
    else:
        exp_bits, man_bits, max_finite = 5, 10, 0x7BFF
    emax = (1 << exp_bits) - 1
    sign = g.integers(0, 2, (n, count), dtype=np.uint16) << 15
    exp = g.integers(0, emax, (n, count), dtype=np.uint16)          # emax excluded: no inf/NaN
    exp = np.where(g.random((n, count)) < 0.25, 0, exp).astype(np.uint16)  # subnormals and zeros
    man = g.integers(0, 1 << man_bits, (n, count), dtype=np.uint16)
    bits = (sign | (exp << man_bits) | man).astype(np.uint16)
    pick = g.random((n, count))
    bits = np.where(pick < 0.03, (sign | max_finite).astype(np.uint16), bits)
    bits = np.where((pick >= 0.03) & (pick < 0.05), sign, bits)  # +0 / -0
    return np.ascontiguousarray(bits.astype(np.uint16)).view(STORAGE[dtype])


@pytest.mark.parametrize("dtype", ["bfloat16", "float16"])
@pytest.mark.parametrize("op", ["sum", "avg"])
def test_two_byte_sums_on_hostile_values(v, dtype, op):
    """The packed 2-byte add must give the oracle's bits (binary32 add, then
    round to nearest even) at every exponent distance, on subnormals, signed
    zeros and overflow, for every schedule that reduces."""
    n, count = 8, 20000
    x = _hostile_2byte(n, count, dtype, seed={"bfloat16": 10, "float16": 20}[dtype] + len(op))
    comm = v.vrcclCommInit(n, 4)
    try:
        v.vrcclCommSetSchedule(comm, 3, 512)
        for algo, proto in (("ring", "simple"), ("ring", "ll"), ("ring", "ll128"), ("tree", "simple"),
                            ("tree", "ll"), ("oneshot", "simple")):
            y, sched, b = run(v, comm, x, dtype, op, algo, proto)
            ref = (otree.tree_allreduce(x, op, dtype, sched["nchannels"]) if sched["algo"] == "tree" else
                   oring.ring_allreduce(x, op, dtype, sched["nchannels"], sched["chunk_elems"]))
            # bits must match, except that any NaN equals any NaN (the tree can add
            # +inf and -inf partial sums; NaN payloads are not part of the result)
            exp_mask, man_mask = (0x7F80, 0x007F) if dtype == "bfloat16" else (0x7C00, 0x03FF)
            yu, ru = y.view(np.uint16), ref.view(np.uint16)
            nan_y = ((yu & exp_mask) == exp_mask) & ((yu & man_mask) != 0)
            nan_r = ((ru & exp_mask) == exp_mask) & ((ru & man_mask) != 0)
            bad = np.nonzero((yu != ru) & ~(nan_y & nan_r))
            assert bad[0].size == 0, (algo, proto, bad[0].size, y.view(np.uint16)[bad][:4], ref.view(np.uint16)[bad][:4])
            assert b.canaries_intact()
    finally:
        v.vrcclCommDestroy(comm)


@pytest.mark.parametrize("algo", ["ring", "tree"])
def test_ll128_long_slices(v, algo):
    """LL128 with several whole slices per agent (the wide kernels: four
    groups of lines per warp and pass), every type and a ragged end."""
    n = 5
    comm = v.vrcclCommInit(n, 4)
    try:
        v.vrcclCommSetSchedule(comm, 2, 0)
        for dtype, op in (("float32", "sum"), ("bfloat16", "avg"), ("float16", "max"), ("int32", "prod")):
            count = 400_003 if ELEM_SIZE[dtype] == 4 else 800_011
            x = _inputs(n, count, dtype, op, seed=count % 97)
            for inplace in (False, True):
                y, sched, b = run(v, comm, x, dtype, op, algo, "ll128", inplace=inplace)
                assert sched["proto"] == "ll128" and sched["nchannels"] == 2
                _assert_parity(x, y, dtype, op, sched)
                assert b.canaries_intact()
        assert v.vrcclCommGetAsyncError(comm) == 0
    finally:
        v.vrcclCommDestroy(comm)


@pytest.mark.parametrize("proto", ["simple", "ll", "ll128"])
@pytest.mark.parametrize("algo", ["ring", "tree"])
def test_maximum_rank_count(v, algo, proto):
    """n = VRCCL_MAX_RANKS (128): 255 primitives per ring loop, trees of
    depth 7, a ragged count; one channel (a tree channel is 255 agents)."""
    n = v.MAX_RANKS
    comm = v.vrcclCommInit(n, 2)
    try:
        v.vrcclCommSetSchedule(comm, 1, 0)
        x = _inputs(n, 5003, "float32", "sum", seed=128)
        y, sched, b = run(v, comm, x, "float32", "sum", algo, proto)
        assert sched["nchannels"] == 1
        _assert_parity(x, y, "float32", "sum", sched)
        assert b.canaries_intact()
        xi = _inputs(n, 777, "int32", "avg", seed=129)
        y, sched, b = run(v, comm, xi, "int32", "avg", algo, proto)
        _assert_parity(xi, y, "int32", "avg", sched)
        assert v.vrcclCommGetAsyncError(comm) == 0
    finally:
        v.vrcclCommDestroy(comm)
