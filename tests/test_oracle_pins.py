"""Pins of the CPU oracle against things other than itself.

Closed forms, brute force on tiny inputs, invariants, library routines and
the worked examples the pages print (``tests/golden/``). No GPU.
"""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import closed_form, numerics as nm, ring, schedule, tree
from ring_allreduce_reduction_gb300.workloads import ELEM_SIZE, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- numerics

def test_bf16_round_is_nearest_even_by_brute_force():
    """Every result is one of the two bf16 neighbours, the nearer one, and
    the even one on a tie -- checked in float64 from the definition."""
    g = np.random.default_rng(1)
    y = np.concatenate([
        g.standard_normal(20000).astype(np.float32),
        (g.standard_normal(2000) * 1e30).astype(np.float32),
        (g.standard_normal(2000) * 1e-38).astype(np.float32),  # subnormals
        # exact ties: upper half + 0x8000 in the lower half
        ((g.integers(0, 0x7F7F, 2000).astype(np.uint32) << 16) | 0x8000).view(np.float32),
    ])
    b = nm.bf16_round(y)
    hi = (y.view(np.uint32) >> 16).astype(np.uint32)
    lo_n = (hi << 16).view(np.float32).astype(np.float64)
    up_n = ((hi + 1) << 16).view(np.float32).astype(np.float64)
    got = (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    y64 = y.astype(np.float64)
    d_lo, d_up = np.abs(y64 - lo_n), np.abs(y64 - up_n)
    expect_up = (d_up < d_lo) | ((d_up == d_lo) & ((hi & 1) == 1))
    assert np.array_equal(got, np.where(expect_up, up_n, lo_n))


def test_bf16_round_matches_torch_conversion():
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(2)
    y = np.concatenate([g.standard_normal(50000), g.standard_normal(5000) * 3e38]).clip(-3.4e38, 3.4e38).astype(np.float32)
    ref = torch.from_numpy(y).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(nm.bf16_round(y), ref)


def test_fp16_and_bf16_sum_step_matches_torch_fp32_then_round():
    """One reduction step is binary32 op + one rounding: compare with torch
    doing the same through its own conversion routines."""
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(3)
    for dtype, tdt in (("float16", torch.float16), ("bfloat16", torch.bfloat16)):
        a = make_inputs(1, 4096, dtype, "normal", seed=4)[0]
        b = make_inputs(1, 4096, dtype, "normal", seed=5)[0]
        ta = torch.from_numpy(a.view(np.int16)).view(tdt) if dtype == "bfloat16" else torch.from_numpy(a)
        tb = torch.from_numpy(b.view(np.int16)).view(tdt) if dtype == "bfloat16" else torch.from_numpy(b)
        for op, f in (("sum", torch.add), ("prod", torch.mul)):
            ref = f(ta.float(), tb.float()).to(tdt)
            ref = ref.view(torch.int16).numpy().view(np.uint16) if dtype == "bfloat16" else ref.numpy()
            got = nm.combine(op, a, b, dtype)
            assert np.array_equal(got.view(np.uint16), np.asarray(ref).view(np.uint16)), (dtype, op)
    del g


def test_int32_ops_wrap_and_truncating_avg():
    fx = _golden("operand_order.json")["int_avg"]
    x = np.array(fx["inputs"], dtype=np.int32).reshape(fx["n"], 1)
    y = ring.ring_allreduce(x, "avg", "int32", 1, 4)
    assert int(y[0, 0]) == fx["expected"]
    a = np.array([2**31 - 1, -2**31, 70000], dtype=np.int32)
    b = np.array([1, -1, 70000], dtype=np.int32)
    assert nm.combine("sum", a, b, "int32").tolist() == [-2**31, 2**31 - 1, 140000]
    assert nm.combine("prod", a, b, "int32").tolist() == [2**31 - 1, -2**31, (70000 * 70000) % 2**32 - 2**32 if (70000 * 70000) % 2**32 >= 2**31 else (70000 * 70000) % 2**32]


# ---------------------------------------------------------------- schedule

@pytest.mark.parametrize("count", [0, 1, 3, 4, 5, 63, 64, 65, 1000, 4096, 4099])
@pytest.mark.parametrize("nch", [1, 2, 3, 7, 32])
@pytest.mark.parametrize("elem", [4, 2])
def test_channel_ranges_tile_and_align(count, nch, elem):
    r = schedule.channel_ranges(count, nch, elem)
    assert len(r) == nch
    pos = 0
    for lo, hi in r:
        assert lo == pos and hi >= lo
        assert (lo * elem) % 16 == 0 or lo == count
        pos = hi
    assert pos == count
    sizes = [hi - lo for lo, hi in r]
    assert all(s1 >= s2 for s1, s2 in zip(sizes, sizes[1:]))  # leading channels are the full ones


def test_channel_ranges_page_example():
    """[Deep Dive §2.2]: 4 channels, channel 0 takes 0..count/4-1, channel 1
    count/4..count/2-1, and so on."""
    count = 4096
    assert schedule.channel_ranges(count, 4, 4) == [(0, 1024), (1024, 2048), (2048, 3072), (3072, 4096)]


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("elem", [4, 2])
def test_ring_loops_by_brute_force(n, elem):
    """Full loops use K; a tail loop uses the smallest 16-byte multiple k
    with n*k >= remaining (found by search, not by the formula); the n
    chunks tile the loop in order, each starting 16-byte aligned."""
    a = 16 // elem
    for K in (a, 2 * a, 5 * a):
        for ch_count in range(0, 3 * n * K + 2 * a + 1):
            pos = 0
            for off, k, chunks in schedule.ring_loops(ch_count, n, K, elem):
                assert off == pos
                rem = ch_count - off
                if rem >= n * K:
                    assert k == K
                else:
                    k_search = next(c for c in itertools.count(a, a) if n * c >= rem)
                    assert k == k_search
                for j, (lo, hi) in enumerate(chunks):
                    assert lo <= hi
                    assert (lo - off) == min(rem, j * k)
                    assert (lo * elem) % 16 == 0 or lo == ch_count
                    assert lo == (chunks[j - 1][1] if j else off)
                pos = chunks[-1][1]
            assert pos == ch_count


def test_build_ring_checks():
    assert schedule.build_ring(schedule.ring_next(8)) == list(range(8))
    assert schedule.build_ring(schedule.ring_next(8), start=3) == [3, 4, 5, 6, 7, 0, 1, 2]
    with pytest.raises(ValueError, match="loop back"):
        schedule.build_ring([1, 0, 2])
    with pytest.raises(ValueError, match="loop back|contain"):
        schedule.build_ring([1, 2, 1])


def test_dtree_matches_page_figure_n8():
    fx = _golden("dtree_n8.json")
    n = fx["n"]
    t0 = [schedule.get_dtree(n, r)[0] for r in range(n)]
    t1 = [schedule.get_dtree(n, r)[1] for r in range(n)]
    assert [t[0] for t in t0] == fx["tree0_parent"]
    assert [t[0] for t in t1] == fx["tree1_parent"]
    internal0 = sorted(r for r in range(n) if any(c != -1 for c in t0[r][1:]))
    internal1 = sorted(r for r in range(n) if any(c != -1 for c in t1[r][1:]))
    assert internal0 == fx["tree0_internal"] and internal1 == fx["tree1_internal"]
    for ex in fx["bit_examples"]:
        u, d0, d1 = schedule.get_btree(n, ex["rank"])
        assert u == ex["parent"]
        assert sorted(c for c in (d0, d1) if c != -1) == ex["children"]
    two = fx["two_ranks"]
    assert [schedule.get_dtree(2, r)[0][0] for r in range(2)] == two["tree0_parent"]
    assert [schedule.get_dtree(2, r)[1][0] for r in range(2)] == two["tree1_parent"]


@pytest.mark.parametrize("n", list(range(1, 40)) + [64, 72, 100, 128])
def test_dtree_is_two_valid_complementary_trees(n):
    for which in (0, 1):
        links = tree.tree_links(n, which)  # raises if inconsistent
        for r, (_u, d0, d1) in enumerate(links):
            assert d0 == -1 or d0 < n and d1 == -1 or d1 < n
    if n % 2 == 0 and n > 1:
        # even n: tree 1 is the mirror of tree 0
        for r in range(n):
            u0 = schedule.get_dtree(n, n - 1 - r)[0][0]
            u1 = schedule.get_dtree(n, r)[1][0]
            assert u1 == (-1 if u0 == -1 else n - 1 - u0)


def test_channel_tree_map():
    assert [schedule.channel_tree(c, 1) for c in range(1)] == [0]
    assert [schedule.channel_tree(c, 24) for c in (0, 11, 12, 23)] == [0, 0, 1, 1]
    assert [schedule.channel_tree(c, 3) for c in range(3)] == [0, 0, 1]


# ---------------------------------------------------------------- ring oracle

def _sym_leaves(n, count):
    out = []
    for r in range(n):
        a = np.empty(count, dtype=object)
        for i in range(count):
            a[i] = r
        out.append(a)
    return out


def _sym_combine(a, b):
    out = np.empty(len(a), dtype=object)
    for i in range(len(a)):
        out[i] = (a[i], b[i])
    return out


def _flatten_left_chain(t):
    """A left fold ((r1, r2), r3)... -> [r1, r2, r3, ...]; None if not a left chain."""
    seq = []
    while isinstance(t, tuple):
        if isinstance(t[1], tuple):
            return None
        seq.append(t[1])
        t = t[0]
    seq.append(t)
    return seq[::-1]


@pytest.mark.parametrize("n", [2, 3, 4, 5, 6])
@pytest.mark.parametrize("nch", [1, 2, 3])
def test_ring_symbolic_association(n, nch):
    """Brute force: every output element is a left fold over all n ranks,
    each once, in ring order, starting at the rank after the chunk's
    owner; chunks appear in loop order; all ranks get the same tree."""
    elem = 4
    a = 16 // elem
    for K in (a, 2 * a):
        for count in range(0, 3 * n * a + 5):
            stats = {}
            outs = ring.ring_machine(_sym_leaves(n, count), _sym_combine, lambda v: v, count, nch, K,
                                     elem, stats, out_factory=lambda r: np.empty(count, dtype=object))
            for r in range(1, n):
                assert all(outs[r][i] == outs[0][i] for i in range(count))
            j_pred = ring.chunk_index(np.arange(count), count, n, nch, K, elem)
            for lo, hi in schedule.channel_ranges(count, nch, elem):
                for off, k, chunks in schedule.ring_loops(hi - lo, n, K, elem):
                    for j, (clo, chi) in enumerate(chunks):
                        for i in range(lo + clo, lo + chi):
                            seq = _flatten_left_chain(outs[0][i])
                            assert seq is not None, outs[0][i]
                            assert sorted(seq) == list(range(n))
                            assert seq == [(j + 1 + t) % n for t in range(n)]
                            assert j_pred[i] == j
            # invariants: 2n-1 primitives and 2(n-1) sends per loop per rank;
            # FIFO payload = 2(n-1) * count elements over all ranks
            assert stats["primitives"] == [stats["loops"] * (2 * n - 1)] * n
            assert stats["sends"] == [stats["loops"] * 2 * (n - 1)] * n
            assert stats["fifo_elems"] == 2 * (n - 1) * count
            assert stats["max_fifo_depth"] <= 2


def test_ring_walkthrough_step_counts():
    fx = _golden("ring_walkthrough_n4.json")
    # One "element" of the walkthrough is one 16-byte unit here (4 floats):
    # chunk boundaries are 16-byte aligned, so 4 parts need 16 floats.
    n, cnt = fx["n"], fx["elements_per_rank"] * 4
    stats = {}
    x = make_inputs(n, cnt, "float32", "int_uniform", lo=-8, hi=8)
    ring.ring_allreduce(x, "sum", "float32", 1, 4, stats)
    assert stats["loops"] == 1
    steps = len(fx["reduce_scatter_steps"]) + len(fx["all_gather_steps"])
    assert stats["primitives"] == [steps] * n
    assert stats["sends"] == [fx["sends_per_rank_per_loop"]] * n
    # after the reduce-scatter steps every rank holds a distinct finished part
    outs = ring.ring_machine(_sym_leaves(n, cnt), _sym_combine, lambda v: v, cnt, 1, 4, 4,
                             out_factory=lambda r: np.empty(cnt, dtype=object))
    finisher = [_flatten_left_chain(outs[0][i])[-1] for i in range(0, cnt, 4)]
    assert sorted(finisher) == list(range(n))


def test_operand_order_fixture():
    fx = _golden("operand_order.json")
    conv = lambda v: np.float32(0.0) if v == "+0" else (np.float32(-0.0) if v == "-0" else np.float32(v))  # noqa
    x = np.stack([np.array([conv(v) for v in fx["x0"]], dtype=np.float32),
                  np.array([conv(v) for v in fx["x1"]], dtype=np.float32)])
    for op in ("max", "min"):
        y = ring.ring_allreduce(x, op, "float32", fx["nchannels"], fx["chunk_elems"])
        assert int(np.signbit(y[0, 0])) == fx[f"expected_{op}_sign_bit_elem0"]
        assert int(np.signbit(y[0, 4])) == fx[f"expected_{op}_sign_bit_elem4"]
        assert np.array_equal(y[0], y[1])


def test_allreduce_example_first_element():
    fx = _golden("allreduce_example.json")
    for case in fx["cases"]:
        n = case["n"]
        count = 4096 + 3
        x = make_inputs(n, count, fx["dtype"], "rank_first")
        y = ring.ring_allreduce(x, fx["op"], fx["dtype"], 2, 64)
        assert np.all(y[:, 0] == case["expected_first"])
        assert np.all(y[:, 1:] == 0)


OPS = ["sum", "prod", "max", "min", "avg"]


ALL_DTYPES = ["int32", "float32", "bfloat16", "float16", "int8", "uint8", "int64", "float64"]
INT_RANGE = {"int32": (-2**20, 2**20), "int8": (-128, 127), "uint8": (0, 255), "int64": (-2**62, 2**62)}


@pytest.mark.parametrize("dtype", ALL_DTYPES)
@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("n", [1, 2, 3, 5, 8])
def test_ring_matches_closed_form(dtype, op, n):
    count = 1000 + n
    if dtype in INT_RANGE:
        lo, hi = INT_RANGE[dtype]
        x = make_inputs(n, count, dtype, "int_uniform", seed=7, lo=lo, hi=hi)
    elif op == "prod":
        x = make_inputs(n, count, dtype, "uniform", seed=7, lo=0.5, hi=2.0)
    else:
        x = make_inputs(n, count, dtype, "normal", seed=7)
    K = 4 * (16 // ELEM_SIZE[dtype])
    y = ring.ring_allreduce(x, op, dtype, 3, K)
    for r in range(1, n):
        assert np.array_equal(y[r].view(np.uint8), y[0].view(np.uint8))
    ok, worst = closed_form.check(y[0], x, op, dtype)
    assert ok, worst
    # the predictor is a second route to the same bits
    p = ring.ring_predict(x, op, dtype, 3, K)
    assert np.array_equal(p.view(np.uint8), y[0].view(np.uint8))


def test_integer_valued_fp32_is_exact():
    """n=4, 4096 integers in [-8, 8] stored as fp32: every partial sum is an
    integer below 2^24, so any order gives the float64 sum exactly."""
    x = make_inputs(4, 4096, "float32", "int_uniform", seed=0, lo=-8, hi=8)
    y = ring.ring_allreduce(x, "sum", "float32", 1, 1024)
    assert np.array_equal(y[0].astype(np.float64), x.astype(np.float64).sum(axis=0))


def test_float_order_matters_and_predictor_tracks_it():
    """With cancellation-prone fp32 data the ring order is visible in the
    bits: a different chunk size changes some results, and the predictor
    follows each choice exactly."""
    x = make_inputs(8, 4096, "float32", "uniform", seed=3)
    y1 = ring.ring_allreduce(x, "sum", "float32", 1, 64)[0]
    y2 = ring.ring_allreduce(x, "sum", "float32", 1, 128)[0]
    assert not np.array_equal(y1, y2)
    assert np.array_equal(ring.ring_predict(x, "sum", "float32", 1, 64), y1)
    assert np.array_equal(ring.ring_predict(x, "sum", "float32", 1, 128), y2)


def test_predictor_on_sampled_indices():
    x = make_inputs(8, 100003, "bfloat16", "normal", seed=11)
    full = ring.ring_allreduce(x, "sum", "bfloat16", 5, 512)[0]
    idx = np.random.default_rng(0).choice(100003, 5000, replace=False)
    assert np.array_equal(ring.ring_predict(x, "sum", "bfloat16", 5, 512, idx), full[idx])


# ---------------------------------------------------------------- tree oracle

def _tree_expected(links, r):
    u, d0, d1 = links[r]
    t = r
    for c in (d0, d1):
        if c != -1:
            t = (t, _tree_expected(links, c))
    return t


@pytest.mark.parametrize("n", [2, 3, 4, 5, 7, 8, 9])
@pytest.mark.parametrize("nch", [1, 2, 3])
def test_tree_symbolic_association(n, nch):
    count = 40
    outs = [np.empty(count, dtype=object) for _ in range(n)]
    leaves = _sym_leaves(n, count)
    for ch, (lo, hi) in enumerate(schedule.channel_ranges(count, nch, 4)):
        if hi > lo:
            links = tree.tree_links(n, schedule.channel_tree(ch, nch))
            tree.tree_machine(leaves, _sym_combine, lambda v: v, links, slice(lo, hi), outs)
            root = next(r for r in range(n) if links[r][0] == -1)
            want = _tree_expected(links, root)
            for r in range(n):
                assert all(outs[r][i] == want for i in range(lo, hi))


@pytest.mark.parametrize("dtype", ALL_DTYPES)
@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("n", [1, 2, 3, 8, 16])
def test_tree_matches_closed_form(dtype, op, n):
    count = 777
    if dtype in INT_RANGE:
        lo, hi = INT_RANGE[dtype]
        x = make_inputs(n, count, dtype, "int_uniform", seed=9, lo=lo, hi=hi)
    elif op == "prod":
        x = make_inputs(n, count, dtype, "uniform", seed=9, lo=0.5, hi=2.0)
    else:
        x = make_inputs(n, count, dtype, "normal", seed=9)
    y = tree.tree_allreduce(x, op, dtype, 4)
    for r in range(1, n):
        assert np.array_equal(y[r].view(np.uint8), y[0].view(np.uint8))
    ok, worst = closed_form.check(y[0], x, op, dtype)
    assert ok, worst


def test_closed_form_catches_a_dropped_term():
    """Sanity of the checker itself: leaving out one rank's contribution is
    far outside every tolerance."""
    x = make_inputs(8, 512, "float32", "normal", seed=1)
    y = ring.ring_allreduce(x, "sum", "float32", 1, 64)[0]
    bad = (y - x[3]).astype(np.float32)
    assert closed_form.check(y, x, "sum", "float32")[0]
    assert not closed_form.check(bad, x, "sum", "float32")[0]
