"""Order-free definition of AllReduce and the error bounds it is held to.

Test infrastructure only. Every rank's output must be the elementwise op
over all n inputs; the example program of [Deep Dive §1.3] checks exactly
this (first element of every recv buffer = 0 + 1 + ... + (n-1)).

* integer types (int8, uint8, int32, int64): sum and prod modulo 2^bits,
  max/min (signed, unsigned for uint8), avg = wrapped sum divided by n with
  truncation toward zero. These are exact and order-free, so any schedule
  must match them bit for bit.
* floating types: the exact value of the op over the dtype-exact inputs
  (pre-scaled by ``1/n`` and rounded to the dtype for avg, the same
  operands the schedule adds), computed in float64 for the 2- and 4-byte
  types and in extended precision (numpy longdouble, at least 64 mantissa
  bits) for float64. Bounds, per element, with ``u``-scale tolerances of
  fp32 1e-5, bf16 (n+1) 2^-8, fp16 (n+1) 2^-11 and fp64 (n+1) 2^-53:
  sum/avg ``|y - s| <= tol * sum_i |x_i|`` (the recursive-summation bound,
  safe under cancellation); prod ``|y - p| <= tol * |p|``; max/min exact.
"""
from __future__ import annotations

import numpy as np

from . import numerics as nm

_BITS = {"int8": 8, "uint8": 8, "int32": 32, "int64": 64}


def tolerance(dtype: str, n: int) -> float:
    if dtype == "float32":
        return 1e-5
    if dtype == "bfloat16":
        return (n + 1) * 2.0 ** -8
    if dtype == "float16":
        return (n + 1) * 2.0 ** -11
    if dtype == "float64":
        return (n + 1) * 2.0 ** -53
    return 0.0


def _wide(dtype: str):
    return np.longdouble if dtype == "float64" else np.float64


def operands(inputs: np.ndarray, op: str, dtype: str) -> np.ndarray:
    """The per-rank operands: exact integers (int64, or uint64 for the
    64-bit wrap) for integer types; exact reals in float64 (longdouble for
    float64) for floating types."""
    n = inputs.shape[0]
    if dtype in nm.INT_TYPES:
        return np.asarray(inputs, dtype=np.int64)
    pre = np.stack([nm.prescale(inputs[r], op, dtype, n) for r in range(n)]) if n else inputs
    if dtype == "float64":
        return np.asarray(pre, dtype=np.float64).astype(np.longdouble)
    return nm.to_f32(pre, dtype).astype(np.float64)


def exact(inputs: np.ndarray, op: str, dtype: str) -> np.ndarray:
    """The closed form: exact wrapped integers for integer types, float64
    (longdouble for float64) for floating types."""
    n = inputs.shape[0]
    x = operands(inputs, op, dtype)
    if dtype in nm.INT_TYPES:
        st = nm.INT_TYPES[dtype][0]
        bits = _BITS[dtype]
        if op == "max":
            return x.max(axis=0).astype(st)
        if op == "min":
            return x.min(axis=0).astype(st)
        u = x.view(np.uint64) if bits == 64 else (x % (1 << bits)).astype(np.uint64)
        if op in ("sum", "avg"):
            acc = u.sum(axis=0, dtype=np.uint64)  # wraps modulo 2^64
        elif op == "prod":
            acc = np.ones(x.shape[1], dtype=np.uint64)
            for r in range(n):
                acc = acc * u[r]  # wraps modulo 2^64; the low `bits` bits are the product modulo 2^bits
        else:
            raise ValueError(op)
        if bits < 64:
            acc = acc % np.uint64(1 << bits)
        signed = dtype != "uint8"
        if bits == 64:
            s = acc.view(np.int64)
        else:
            s = acc.astype(np.int64)
            if signed:
                s = np.where(s >= (1 << (bits - 1)), s - (1 << bits), s)
        if op == "avg":
            s = nm.trunc_div(s, n) if signed else s // n
        return s.astype(st)
    if op in ("sum", "avg"):
        return x.sum(axis=0)
    if op == "prod":
        return np.prod(x, axis=0)
    if op == "max":
        return x.max(axis=0)
    if op == "min":
        return x.min(axis=0)
    raise ValueError(op)


def bound(inputs: np.ndarray, op: str, dtype: str) -> np.ndarray:
    """Allowed per-element absolute error for a floating result."""
    n = inputs.shape[0]
    x = operands(inputs, op, dtype)
    tol = tolerance(dtype, n)
    if op in ("sum", "avg"):
        return tol * np.abs(x).sum(axis=0)
    if op == "prod":
        return tol * np.abs(np.prod(x, axis=0))
    return np.zeros(x.shape[1])


def check(result: np.ndarray, inputs: np.ndarray, op: str, dtype: str) -> tuple[bool, float]:
    """(within bounds?, worst excess ratio) of a ``[count]`` result row."""
    ref = exact(inputs, op, dtype)
    if dtype in nm.INT_TYPES:
        ok = np.array_equal(np.asarray(result, dtype=nm.INT_TYPES[dtype][0]), ref)
        return ok, 0.0 if ok else float("inf")
    if dtype == "float64":
        y = np.asarray(result, dtype=np.float64).astype(np.longdouble)
    else:
        y = nm.to_f32(result, dtype).astype(np.float64)
    err = np.abs(y - ref)
    b = bound(inputs, op, dtype)
    if op in ("max", "min"):
        ok = bool(np.all(err == 0))
        return ok, 0.0 if ok else float("inf")
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(b > 0, err / b, np.where(err > 0, np.inf, 0.0))
    worst = float(ratio.max()) if ratio.size else 0.0
    return worst <= 1.0, worst
