"""Pins of the ReduceScatter / AllGather oracle (``oracle.phases``). No GPU.

What fixes them, other than the oracle itself:

* the closed form: block r of the ReduceScatter result is the elementwise
  op over every rank's block r (exact for int32, within the stated bound
  for floats); every AllGather recv buffer is the concatenation of the
  send buffers, bit for bit;
* brute force on tiny inputs: each ReduceScatter element is a left fold
  over all n ranks, each once, in ring order from the rank after the
  block's owner;
* the decomposition the pages state: the AllReduce is the reduce-scatter
  phase followed by the all-gather phase. For one channel and a chunk of
  count/n elements, a loop's n chunks are exactly the n blocks, so the
  AllReduce step machine of ``oracle.ring`` (separate code) must give the
  same bits as AllGather(ReduceScatter(x));
* step and payload counts: n-1 sends per rank per phase, (n-1) n b FIFO
  elements in all.
"""
import numpy as np
import pytest

from oracle import closed_form, phases, ring
from ring_allreduce_reduction_gb300.workloads import ELEM_SIZE, make_inputs
from tests.test_oracle_pins import _flatten_left_chain, _sym_combine

OPS = ["sum", "prod", "max", "min", "avg"]
DTYPES = ["int32", "float32", "bfloat16", "float16", "int8", "uint8", "int64", "float64"]
INT_RANGE = {"int32": (-2**20, 2**20), "int8": (-128, 127), "uint8": (0, 255), "int64": (-2**62, 2**62)}


def _inputs(n, count, dtype, op, seed):
    if dtype in INT_RANGE:
        lo, hi = INT_RANGE[dtype]
        return make_inputs(n, count, dtype, "int_uniform", seed=seed, lo=lo, hi=hi)
    if op == "prod":
        return make_inputs(n, count, dtype, "uniform", seed=seed, lo=0.5, hi=2.0)
    return make_inputs(n, count, dtype, "normal", seed=seed)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("n", [1, 2, 3, 5, 8])
def test_reduce_scatter_matches_closed_form(dtype, op, n):
    b = 257
    x = _inputs(n, n * b, dtype, op, seed=n)
    y = phases.ring_reduce_scatter(x, op, dtype)
    assert y.shape == (n, b) and y.dtype == x.dtype
    for r in range(n):
        ok, worst = closed_form.check(y[r], x[:, r * b:(r + 1) * b], op, dtype)
        assert ok, (r, worst)
        if dtype in INT_RANGE:
            assert np.array_equal(y[r], closed_form.exact(x[:, r * b:(r + 1) * b], op, dtype))
        # the predictor is a second route to the same bits
        p = phases.reduce_scatter_predict(x, op, dtype, r)
        assert np.array_equal(p.view(np.uint8), y[r].view(np.uint8))


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6])
def test_reduce_scatter_symbolic_association(n):
    for b in (0, 1, 3):
        local = []
        for r in range(n):
            a = np.empty(n * b, dtype=object)
            a[:] = [r] * (n * b)
            local.append(a)
        stats = {}
        out = phases.reduce_scatter_machine(local, _sym_combine, lambda v: v, stats)
        for r in range(n):
            assert len(out[r]) == b
            for i in range(b):
                seq = _flatten_left_chain(out[r][i])
                assert seq == [(r + 1 + t) % n for t in range(n)], (r, out[r][i])
        if n > 1:
            assert stats["sends"] == [n - 1] * n
            assert stats["fifo_elems"] == n * (n - 1) * b


@pytest.mark.parametrize("n", [1, 2, 3, 7])
def test_all_gather_is_concatenation(n):
    b = 37
    x = make_inputs(n, b, "bfloat16", "normal", seed=4)
    stats = {}
    y = phases.ring_all_gather(x, stats)
    want = np.concatenate([x[q] for q in range(n)])
    for r in range(n):
        assert np.array_equal(y[r].view(np.uint8), want.view(np.uint8))
    if n > 1:
        assert stats["sends"] == [n - 1] * n
        assert stats["fifo_elems"] == n * (n - 1) * b


@pytest.mark.parametrize("dtype,op", [("float32", "sum"), ("bfloat16", "sum"), ("float16", "avg"),
                                      ("bfloat16", "max"), ("int32", "avg"), ("float32", "prod"),
                                      ("int8", "prod"), ("uint8", "avg"), ("int64", "sum"), ("float64", "avg")])
@pytest.mark.parametrize("n", [2, 3, 5, 8])
def test_allreduce_is_reduce_scatter_then_all_gather(dtype, op, n):
    """One channel, chunk = count/n (a multiple of 16 bytes): the AllReduce
    loop's chunks are the blocks, so the two step machines must agree."""
    a = 16 // ELEM_SIZE[dtype]
    b = 24 * a
    x = _inputs(n, n * b, dtype, op, seed=11 + n)
    ar = ring.ring_allreduce(x, op, dtype, 1, b)
    rs = phases.ring_reduce_scatter(x, op, dtype)
    ag = phases.ring_all_gather(rs)
    assert np.array_equal(ag.view(np.uint8), ar.view(np.uint8))


def test_float_order_is_the_ring_order():
    """Cancellation-prone fp32: the association is visible in the bits, and a
    fold that starts at the block's owner (the other rotation) differs."""
    n, b = 8, 4096
    x = make_inputs(n, n * b, "float32", "uniform", seed=3)
    y = phases.ring_reduce_scatter(x, "sum", "float32")
    r = 5
    blk = x[:, r * b:(r + 1) * b]
    other = blk[r].copy()
    for t in range(1, n):
        other = (other + blk[(r + t) % n]).astype(np.float32)
    assert not np.array_equal(other, y[r])
    ring_order = blk[(r + 1) % n].copy()
    for t in range(2, n + 1):
        ring_order = (ring_order + blk[(r + t) % n]).astype(np.float32)
    assert np.array_equal(ring_order, y[r])


def test_closed_form_catches_a_dropped_block_term():
    """A planted mistake in the oracle (one rank's term left out) must fail
    the closed-form check that pins it."""
    n, b = 4, 64
    x = _inputs(n, n * b, "float32", "sum", seed=5)
    y = phases.ring_reduce_scatter(x, "sum", "float32")
    bad = y.copy()
    bad[2] = (bad[2] - x[1, 2 * b:3 * b]).astype(np.float32)
    ok, _ = closed_form.check(bad[2], x[:, 2 * b:3 * b], "sum", "float32")
    assert not ok
    ok, _ = closed_form.check(y[2], x[:, 2 * b:3 * b], "sum", "float32")
    assert ok
