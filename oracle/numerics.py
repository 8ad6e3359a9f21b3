"""Element arithmetic of the oracle (test infrastructure only).

Storage forms: int32 -> np.int32, float32 -> np.float32, float16 ->
np.float16, bfloat16 -> np.uint16 holding the bf16 bit pattern, int8 ->
np.int8, uint8 -> np.uint8, int64 -> np.int64, float64 -> np.float64.

One reduction step ``combine(op, a, b)`` is, for the 2- and 4-byte floating
types, the op in IEEE binary32 with round-to-nearest-even, then one
rounding to the storage type (round-to-nearest-even); for float64 the op in
binary64 (round-to-nearest-even). The pages leave the intermediate
precision open: NCCL's FIFOs carry the user's dtype, so every hop of the
ring stores (and therefore rounds to) that dtype [Architecture §7.2, the
FIFO carries user data; Deep Dive §2.4]. Integer types: sum and prod wrap
modulo 2^bits; max and min compare as signed (int8, int32, int64) or
unsigned (uint8).

Operand order: ``a`` is the running value (what arrived from the previous
rank in the ring, or the node's own accumulator in the tree) and ``b`` the
other operand. ``max(a, b) = b if b > a else a`` and ``min(a, b) = b if
b < a else a``, so a tie (including +0 against -0) keeps ``a``.

avg is not on the pages: for the 2- and 4-byte floating types every input
is multiplied once by ``s = 1.0f / n`` (binary32, RNE) and rounded to the
storage type before it enters the sum; for float64 by ``1.0 / n`` in
binary64. For the integer types the wrapped sum is divided by n with
truncation toward zero once, where the ring finishes a chunk (the post-op
of the last reduce-scatter step, [Architecture §9.4]).
"""
from __future__ import annotations

import numpy as np

OPS = ("sum", "prod", "max", "min", "avg")
FLOAT_TYPES = ("float32", "float16", "bfloat16", "float64")
# integer types: (storage type, unsigned type of the same width)
INT_TYPES = {"int32": (np.int32, np.uint32), "int8": (np.int8, np.uint8), "uint8": (np.uint8, np.uint8),
             "int64": (np.int64, np.uint64)}


def to_f32(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of a storage array to binary32."""
    if dtype == "float32":
        return np.asarray(x, dtype=np.float32)
    if dtype == "float16":
        return np.asarray(x, dtype=np.float16).astype(np.float32)
    if dtype == "bfloat16":
        return (np.asarray(x, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    raise ValueError(dtype)


def bf16_round(y: np.ndarray) -> np.ndarray:
    """binary32 -> bf16 bits, round to nearest, ties to even.

    A bf16 number is the upper half of a binary32 pattern. The two bf16
    neighbours of y are its upper half ``hi`` (toward zero) and ``hi + 1``
    (away from zero); the lower 16 bits say where y sits between them:
    above half way -> round away, exactly half way -> pick the neighbour
    whose last mantissa bit is 0. A carry out of the mantissa moves into
    the exponent, which is the correct next binade (and gives inf past the
    largest finite value). NaNs stay NaN (quiet bit forced).
    """
    u = np.ascontiguousarray(y, dtype=np.float32).view(np.uint32)
    hi = (u >> 16).astype(np.uint32)
    lo = u & np.uint32(0xFFFF)
    up = (lo > 0x8000) | ((lo == 0x8000) & ((hi & 1) == 1))
    out = hi + up.astype(np.uint32)
    nan = ((u & np.uint32(0x7F800000)) == np.uint32(0x7F800000)) & ((u & np.uint32(0x007FFFFF)) != 0)
    out = np.where(nan, hi | np.uint32(0x40), out)
    return out.astype(np.uint16)


def from_f32(y: np.ndarray, dtype: str) -> np.ndarray:
    """binary32 -> storage type, round to nearest even."""
    if dtype == "float32":
        return np.asarray(y, dtype=np.float32)
    if dtype == "float16":
        return np.asarray(y, dtype=np.float32).astype(np.float16)
    if dtype == "bfloat16":
        return bf16_round(y)
    raise ValueError(dtype)


def combine(op: str, a: np.ndarray, b: np.ndarray, dtype: str) -> np.ndarray:
    """One reduction step ``op(a, b)``; ``a`` is the running value."""
    if op == "avg":
        op = "sum"  # the pre-scale / post-op are applied outside
    if dtype in INT_TYPES:
        st, ut = INT_TYPES[dtype]
        shape = np.broadcast_shapes(np.shape(a), np.shape(b))
        ua = np.atleast_1d(np.asarray(a, dtype=st)).view(ut)
        ub = np.atleast_1d(np.asarray(b, dtype=st)).view(ut)
        if op == "sum":
            return (ua + ub).view(st).reshape(shape)  # unsigned arrays wrap modulo 2^bits
        if op == "prod":
            return (ua * ub).view(st).reshape(shape)
        a = np.asarray(a, dtype=st)
        b = np.asarray(b, dtype=st)
        if op == "max":
            return np.where(b > a, b, a)
        if op == "min":
            return np.where(b < a, b, a)
        raise ValueError(op)
    if dtype == "float64":
        fa = np.asarray(a, dtype=np.float64)
        fb = np.asarray(b, dtype=np.float64)
        if op == "sum":
            return fa + fb
        if op == "prod":
            return fa * fb
        if op == "max":
            return np.where(fb > fa, fb, fa)
        if op == "min":
            return np.where(fb < fa, fb, fa)
        raise ValueError(op)
    fa = to_f32(a, dtype)
    fb = to_f32(b, dtype)
    if op == "sum":
        return from_f32(fa + fb, dtype)
    if op == "prod":
        return from_f32(fa * fb, dtype)
    if op == "max":
        return np.where(fb > fa, b, a)
    if op == "min":
        return np.where(fb < fa, b, a)
    raise ValueError(op)


def avg_scale(n: int) -> np.float32:
    """The avg pre-scale factor ``1.0f / n`` in binary32."""
    return np.float32(1.0) / np.float32(n)


def prescale(x: np.ndarray, op: str, dtype: str, n: int) -> np.ndarray:
    """The value a rank feeds into the reduction for its own input x.

    Identity except for floating avg, where it is ``rnd(float(x) * (1/n))``
    (binary32 scale and product for the 2- and 4-byte types, binary64 for
    float64).
    """
    if op != "avg" or dtype in INT_TYPES:
        return np.asarray(x)
    if dtype == "float64":
        return np.asarray(x, dtype=np.float64) * (np.float64(1.0) / np.float64(n))
    return from_f32(to_f32(x, dtype) * avg_scale(n), dtype)


def trunc_div(y: np.ndarray, n: int) -> np.ndarray:
    """Integer division truncating toward zero, without overflow for any
    64-bit y (floor quotient, plus one where a negative y left a
    remainder)."""
    y64 = np.asarray(y, dtype=np.int64)
    q = y64 // n
    return q + ((y64 < 0) & (y64 % n != 0)).astype(np.int64)


def postop(y: np.ndarray, op: str, dtype: str, n: int) -> np.ndarray:
    """Applied once to a finished chunk: integer avg divides by n,
    truncating toward zero."""
    if op != "avg" or dtype not in INT_TYPES:
        return y
    st = INT_TYPES[dtype][0]
    if dtype == "uint8":
        return (np.asarray(y, dtype=np.uint8).astype(np.int64) // n).astype(np.uint8)
    return trunc_div(np.asarray(y, dtype=st), n).astype(st)
