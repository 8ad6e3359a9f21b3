"""Pins of the oracle's avg pre-scale for float32, bfloat16 and float16,
computed from the definition without the oracle's own arithmetic.

avg is not an op the pages define; the reading taken is that each input is
multiplied once by the binary32 number nearest to 1/n, the product is
rounded to binary32 (round to nearest, ties to even), and that value is
rounded once more to the element type before it enters the ring's sum.
Here every step is done with exact rationals (``fractions.Fraction``) and
a brute-force nearest-neighbour search over representable values, so a
wrong scale (for instance 1/(n+1)), a skipped rounding or a rounding the
wrong way fails these tests. A second test checks whole avg AllReduces of
positive inputs against the mean of the *unscaled* inputs. No GPU.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import numerics as nm, ring, tree
from ring_allreduce_reduction_gb300.workloads import make_inputs

NS = (2, 3, 5, 7, 8, 72)


def _nearest(q: Fraction, cands):
    """The candidate nearest to q; on a tie the one whose bit pattern is
    even. cands: (exact value, bit pattern, stored value)."""
    best = None
    for val, bits, stored in cands:
        d = abs(val - q)
        key = (d, bits & 1)
        if best is None or key < best[0]:
            best = (key, stored)
    return best[1]


def _f32_neighbours(q: Fraction):
    c = np.float32(float(q))
    out = []
    for v in (np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))):
        v = np.float32(v)
        out.append((Fraction(float(v)), int(np.array(v).view(np.uint32)), v))
    return out


def round_to_binary32(q: Fraction) -> np.float32:
    return _nearest(q, _f32_neighbours(q))


def round_binary32_to_type(v: np.float32, dtype: str):
    """One more rounding, binary32 -> the element type (storage form)."""
    q = Fraction(float(v))
    if dtype == "float32":
        return v
    if dtype == "float16":
        c = np.float16(float(v))
        cands = []
        for w in (np.nextafter(c, np.float16(-np.inf)), c, np.nextafter(c, np.float16(np.inf))):
            w = np.float16(w)
            cands.append((Fraction(float(w)), int(np.array(w).view(np.uint16)), w))
        return _nearest(q, cands)
    # bfloat16: the upper half of a binary32 pattern; try the pattern of v
    # truncated and its two neighbours
    p = int(np.array(v).view(np.uint32)) >> 16
    cands = []
    for b in (p - 1, p, p + 1):
        if 0 <= b <= 0xFFFF and (b & 0x7F80) != 0x7F80:
            val = np.array(b << 16, dtype=np.uint32).view(np.float32)[()]
            cands.append((Fraction(float(val)), b, np.uint16(b)))
    return _nearest(q, cands)


def exact_value(x, dtype: str) -> Fraction:
    if dtype == "bfloat16":
        return Fraction(float(np.array(int(x) << 16, dtype=np.uint32).view(np.float32)[()]))
    return Fraction(float(x))


def expected_prescaled(xs, dtype: str, n: int) -> np.ndarray:
    s = round_to_binary32(Fraction(1, n))
    out = [round_binary32_to_type(round_to_binary32(exact_value(x, dtype) * Fraction(float(s))), dtype) for x in xs]
    return np.array(out, dtype={"bfloat16": np.uint16, "float16": np.float16, "float32": np.float32}[dtype])


def _bits(a):
    a = np.ascontiguousarray(a)
    return a.view({2: np.uint16, 4: np.uint32}[a.dtype.itemsize])


@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "float16"])
@pytest.mark.parametrize("n", NS)
def test_avg_prescale_from_exact_rationals(dtype, n):
    x = make_inputs(1, 600, dtype, "normal", seed=40 + n)[0]
    # values whose products land near rounding boundaries of the type:
    # powers of two and their neighbours, and numbers with a full mantissa
    extra = {"float32": np.array([1.0, 3.0, 1.5, 0.7, 1e-30, 6e37, 2.0 ** -120], dtype=np.float32),
             "float16": np.array([1.0, 3.0, 1.5, 65504.0, 6.1e-5, 2.0 ** -20, 0.333], dtype=np.float16),
             "bfloat16": np.array([0x3F80, 0x4040, 0x3FC0, 0x7F7F, 0x0080, 0x0001, 0x3EAB], dtype=np.uint16)}[dtype]
    x = np.concatenate([x[x != 0] if dtype != "bfloat16" else x[(x & 0x7FFF) != 0], extra])
    got = nm.prescale(x, "avg", dtype, n)
    want = expected_prescaled(x, dtype, n)
    assert np.array_equal(_bits(got), _bits(want))


def test_avg_scale_is_the_binary32_nearest_to_one_over_n():
    for n in (*NS, 1, 6, 10, 100, 127, 128):
        assert nm.avg_scale(n) == round_to_binary32(Fraction(1, n)), n


@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "float16"])
@pytest.mark.parametrize("n", [2, 3, 5, 8])
def test_avg_allreduce_is_the_mean_of_unscaled_inputs(dtype, n):
    """A whole avg AllReduce (ring and tree) of positive inputs against the
    mean of the inputs as given, before any scaling: per element
    |y - mean| <= tol * mean, tol = fp32 1e-5, bf16 (n+1) 2^-8, fp16
    (n+1) 2^-11 (the pre-scale's own rounding is inside that bound)."""
    x = make_inputs(n, 4096, dtype, "uniform", seed=7, lo=0.5, hi=2.0)
    vals = np.stack([[float(exact_value(v, dtype)) for v in row] for row in x])
    mean = vals.sum(axis=0) / n
    tol = {"float32": 1e-5, "bfloat16": (n + 1) * 2.0 ** -8, "float16": (n + 1) * 2.0 ** -11}[dtype]
    for y in (ring.ring_allreduce(x, "avg", dtype, 3, 256), tree.tree_allreduce(x, "avg", dtype, 2)):
        got = np.array([float(exact_value(v, dtype)) for v in y[0]])
        assert np.all(np.abs(got - mean) <= tol * mean)
