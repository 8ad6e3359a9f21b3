"""Order-free definition of AllReduce and the error bounds it is held to.

Test infrastructure only. Every rank's output must be the elementwise op
over all n inputs; the example program of [Deep Dive §1.3] checks exactly
this (first element of every recv buffer = 0 + 1 + ... + (n-1)).

* int32: sum and prod modulo 2^32, max/min, avg = wrapped sum divided by n
  with truncation toward zero. These are exact and order-free, so any
  schedule must match them bit for bit.
* floating types: the float64 value of the op over the dtype-exact inputs
  (pre-scaled by ``1/n`` and rounded to the dtype for avg, the same
  operands the schedule adds). Bounds, per element, with ``u``-scale
  tolerances of fp32 1e-5, bf16 (n+1) 2^-8, fp16 (n+1) 2^-11:
  sum/avg ``|y - s64| <= tol * sum_i |x_i|`` (the recursive-summation
  bound, safe under cancellation); prod ``|y - p64| <= tol * |p64|``;
  max/min exact.
"""
from __future__ import annotations

import numpy as np

from . import numerics as nm


def tolerance(dtype: str, n: int) -> float:
    if dtype == "float32":
        return 1e-5
    if dtype == "bfloat16":
        return (n + 1) * 2.0 ** -8
    if dtype == "float16":
        return (n + 1) * 2.0 ** -11
    return 0.0


def operands(inputs: np.ndarray, op: str, dtype: str) -> np.ndarray:
    """The per-rank operands as float64 (floats) or int64 (int32)."""
    n = inputs.shape[0]
    if dtype == "int32":
        return np.asarray(inputs, dtype=np.int64)
    pre = np.stack([nm.prescale(inputs[r], op, dtype, n) for r in range(n)]) if n else inputs
    return nm.to_f32(pre, dtype).astype(np.float64)


def exact(inputs: np.ndarray, op: str, dtype: str) -> np.ndarray:
    """The closed form: float64 for floats, exact wrapped int32 for int32."""
    n = inputs.shape[0]
    x = operands(inputs, op, dtype)
    if dtype == "int32":
        m = np.uint64(1 << 32)
        u = (x % (1 << 32)).astype(np.uint64)
        if op in ("sum", "avg"):
            acc = u.sum(axis=0, dtype=np.uint64) % m
        elif op == "prod":
            acc = np.ones(x.shape[1], dtype=np.uint64)
            for r in range(n):
                acc = (acc * u[r]) % m  # both factors < 2^32: the product fits 64 bits
        elif op == "max":
            return x.max(axis=0).astype(np.int32)
        elif op == "min":
            return x.min(axis=0).astype(np.int32)
        else:
            raise ValueError(op)
        s = acc.astype(np.int64)
        s = np.where(s >= (1 << 31), s - (1 << 32), s)
        if op == "avg":
            s = (np.abs(s) // n) * np.sign(s)
        return s.astype(np.int32)
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
    if dtype == "int32":
        ok = np.array_equal(np.asarray(result, dtype=np.int32), ref)
        return ok, 0.0 if ok else float("inf")
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
