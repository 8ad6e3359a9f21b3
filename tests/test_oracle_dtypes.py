"""Pins of the oracle's arithmetic for int8, uint8, int64 and float64
against definitions computed another way: exhaustive Python-integer
arithmetic modulo 2^8, Python integers modulo 2^64, exact rationals
rounded once to binary64, and the closed form with a planted mistake.
No GPU."""
import fractions
import itertools

import numpy as np
import pytest

from oracle import closed_form, numerics as nm, ring, tree
from ring_allreduce_reduction_gb300.workloads import make_inputs


def _wrap(v, bits, signed):
    v %= 1 << bits
    return v - (1 << bits) if signed and v >= 1 << (bits - 1) else v


@pytest.mark.parametrize("dtype,signed", [("int8", True), ("uint8", False)])
def test_byte_ops_exhaustively(dtype, signed):
    """All 65536 operand pairs of each op against Python integers."""
    vals = list(range(-128, 128)) if signed else list(range(256))
    pairs = list(itertools.product(vals, vals))
    st = np.int8 if signed else np.uint8
    a = np.array([p[0] for p in pairs], dtype=st)
    b = np.array([p[1] for p in pairs], dtype=st)
    for op, f in (("sum", lambda x, y: x + y), ("prod", lambda x, y: x * y), ("max", max), ("min", min)):
        got = nm.combine(op, a, b, dtype).astype(np.int64).tolist()
        want = [_wrap(f(x, y), 8, signed) for x, y in pairs]
        assert got == want, op


def test_int64_ops_wrap_like_python_integers():
    g = np.random.default_rng(5)
    a = g.integers(-2**63, 2**63 - 1, size=4000, dtype=np.int64, endpoint=True)
    b = g.integers(-2**63, 2**63 - 1, size=4000, dtype=np.int64, endpoint=True)
    a[:4] = [2**63 - 1, -2**63, -1, 0]
    b[:4] = [1, -1, -2**63, 2**63 - 1]
    for op, f in (("sum", lambda x, y: x + y), ("prod", lambda x, y: x * y), ("max", max), ("min", min)):
        got = nm.combine(op, a, b, "int64").tolist()
        want = [_wrap(f(int(x), int(y)), 64, True) for x, y in zip(a, b)]
        assert got == want, op


@pytest.mark.parametrize("n", [1, 2, 3, 7, 8, 128])
def test_integer_avg_truncates_toward_zero(n):
    """Post-op against exact integer division rounded toward zero, at the
    edges of every integer type (including the most negative value)."""
    for dtype, bits, signed in (("int8", 8, True), ("uint8", 8, False), ("int32", 32, True), ("int64", 64, True)):
        lo, hi = (-(1 << (bits - 1)), (1 << (bits - 1)) - 1) if signed else (0, (1 << bits) - 1)
        ys = sorted(y for y in {lo, lo + 1, -7, -1, 0, 1, 7, hi - 1, hi} if lo <= y <= hi)
        st = nm.INT_TYPES[dtype][0]
        got = nm.postop(np.array(ys, dtype=st), "avg", dtype, n).astype(np.int64).tolist()
        want = [abs(y) // n * (1 if y >= 0 else -1) for y in ys]
        assert got == want, dtype


def _round_to_double(q: fractions.Fraction) -> float:
    return float(q)  # correctly rounded, ties to even


def test_float64_ops_are_one_binary64_rounding_of_the_exact_result():
    g = np.random.default_rng(11)
    a = g.standard_normal(3000) * np.exp2(g.integers(-40, 40, size=3000))
    b = g.standard_normal(3000) * np.exp2(g.integers(-40, 40, size=3000))
    a[:3] = [1.0, 0.0, -0.0]
    b[:3] = [2.0 ** -53, -0.0, 0.0]
    s = nm.combine("sum", a, b, "float64")
    p = nm.combine("prod", a, b, "float64")
    for i in range(len(a)):
        fa, fb = fractions.Fraction(float(a[i])), fractions.Fraction(float(b[i]))
        assert s[i] == _round_to_double(fa + fb) or (s[i] == 0 and fa + fb == 0)
        assert p[i] == _round_to_double(fa * fb) or (p[i] == 0 and fa * fb == 0)
    # ties keep the running value: +0 against -0 keeps a
    assert np.signbit(nm.combine("max", np.array([0.0]), np.array([-0.0]), "float64"))[0] == False  # noqa: E712
    assert np.signbit(nm.combine("max", np.array([-0.0]), np.array([0.0]), "float64"))[0] == True  # noqa: E712


def test_float64_avg_prescale_is_binary64():
    """The float64 pre-scale multiplies by the binary64 1/n, one rounding:
    for n = 3 it differs from the binary32 scale the 4-byte types use."""
    x = np.array([1.0, 3.0, -6.0])
    got = nm.prescale(x, "avg", "float64", 3)
    want = [_round_to_double(fractions.Fraction(v) * fractions.Fraction(1.0 / 3.0)) for v in x]
    assert got.tolist() == want
    assert float(np.float32(1) / np.float32(3)) != 1.0 / 3.0


@pytest.mark.parametrize("dtype", ["int8", "uint8", "int64", "float64"])
def test_closed_form_catches_a_dropped_term(dtype):
    n = 8
    if dtype == "float64":
        x = make_inputs(n, 512, dtype, "normal", seed=2)
    else:
        lo, hi = {"int8": (-128, 127), "uint8": (0, 255), "int64": (-2**62, 2**62)}[dtype]
        x = make_inputs(n, 512, dtype, "int_uniform", seed=2, lo=lo, hi=hi)
    y = ring.ring_allreduce(x, "sum", dtype, 2, 64)[0]
    assert closed_form.check(y, x, "sum", dtype)[0]
    bad = nm.combine("sum", y, (-x[3].astype(np.float64)).astype(x.dtype) if dtype == "float64" else
                     (np.zeros_like(x[3]) - x[3]), dtype)
    assert not closed_form.check(bad, x, "sum", dtype)[0]


def test_float64_sum_tolerance_is_tight_enough_to_see_fp32_rounding():
    """A result rounded through binary32 once fails the float64 bound."""
    x = make_inputs(8, 4096, "float64", "normal", seed=4)
    y = ring.ring_allreduce(x, "sum", "float64", 1, 128)[0]
    assert closed_form.check(y, x, "sum", "float64")[0]
    assert not closed_form.check(y.astype(np.float32).astype(np.float64), x, "sum", "float64")[0]


@pytest.mark.parametrize("dtype", ["int8", "uint8", "int64", "float64"])
def test_ring_and_tree_agree_where_the_order_does_not_matter(dtype):
    n = 6
    if dtype == "float64":
        x = make_inputs(n, 999, dtype, "int_uniform", seed=3, lo=-1000, hi=1000).astype(np.float64)
    else:
        lo, hi = {"int8": (-128, 127), "uint8": (0, 255), "int64": (-2**62, 2**62)}[dtype]
        x = make_inputs(n, 999, dtype, "int_uniform", seed=3, lo=lo, hi=hi)
    for op in ("sum", "max", "min", "avg") if dtype != "float64" else ("sum", "max", "min"):
        yr = ring.ring_allreduce(x, op, dtype, 3, 128 // x.itemsize)
        yt = tree.tree_allreduce(x, op, dtype, 3)
        assert np.array_equal(yr, yt), op
