"""Seeded synthetic inputs for the virtual-rank AllReduce.

This module only draws random numbers and lays them out; it holds none of
the reduction arithmetic, so both the CUDA path (through the tests and
``bench.py``) and the CPU oracle can take their inputs from it.

Each virtual rank r gets its own numpy Generator, spawned from one
``SeedSequence(seed)``: ``default_rng(SeedSequence(seed).spawn(n)[r])``.
The result is one ``[n, count]`` array in the *storage* representation of
the dtype:

=========  ==================  =========================================
dtype      numpy array dtype   meaning of one element
=========  ==================  =========================================
int32      ``np.int32``        the value
float32    ``np.float32``      the value
float16    ``np.float16``      the value
bfloat16   ``np.uint16``       the bf16 bit pattern (sign, 8-bit
                               exponent, 7-bit mantissa)
int8       ``np.int8``         the value
uint8      ``np.uint8``        the value
int64      ``np.int64``        the value
float64    ``np.float64``      the value
=========  ==================  =========================================

Real-valued draws are binary32 for the 2- and 4-byte floating types and
binary64 for float64.

bf16 values are made by keeping the upper 16 bits of a float32 draw
(truncation toward zero). That is a recipe for drawing inputs, not a
rounding step of the method; integer-valued draws survive it exactly.
"""
from __future__ import annotations

import numpy as np

DTYPES = ("int32", "float32", "bfloat16", "float16", "int8", "uint8", "int64", "float64")
ELEM_SIZE = {"int32": 4, "float32": 4, "bfloat16": 2, "float16": 2, "int8": 1, "uint8": 1, "int64": 8,
             "float64": 8}
STORAGE = {"int32": np.int32, "float32": np.float32, "bfloat16": np.uint16,
           "float16": np.float16, "int8": np.int8, "uint8": np.uint8, "int64": np.int64,
           "float64": np.float64}
INT_TYPES = ("int32", "int8", "uint8", "int64")


def rank_generators(n: int, seed: int = 0) -> list[np.random.Generator]:
    """One independent generator per virtual rank."""
    return [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(n)]


def _bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _store(vals: np.ndarray, dtype: str) -> np.ndarray:
    if dtype in INT_TYPES:
        return vals.astype(STORAGE[dtype])
    if dtype == "float64":
        return vals.astype(np.float64)
    if dtype == "float32":
        return vals.astype(np.float32)
    if dtype == "float16":
        return vals.astype(np.float32).astype(np.float16)
    if dtype == "bfloat16":
        return _bf16_bits_from_f32(vals.astype(np.float32))
    raise ValueError(f"unknown dtype {dtype!r}")


def make_inputs(n: int, count: int, dtype: str, dist: str = "uniform", seed: int = 0,
                lo: float = -1.0, hi: float = 1.0, std: float = 1.0) -> np.ndarray:
    """Return an ``[n, count]`` array of per-rank inputs in storage form.

    dist:
      * ``"int_uniform"``: integers uniform in ``[lo, hi]`` inclusive.
      * ``"uniform"``: reals uniform in ``[lo, hi)``.
      * ``"normal"``: reals normal with mean 0 and standard deviation ``std``.
      * ``"rank_first"``: element 0 of rank r is r, every other element is 0
        (the verification pattern of the single-process AllReduce example).
    """
    if dtype not in STORAGE:
        raise ValueError(f"unknown dtype {dtype!r}")
    out = np.empty((n, count), dtype=STORAGE[dtype])
    if dist == "rank_first":
        vals = np.zeros((n, count), dtype=np.float64)
        if count:
            vals[:, 0] = np.arange(n)
        return _store(vals, dtype)
    for r, g in enumerate(rank_generators(n, seed)):
        if dist == "int_uniform":
            v = g.integers(int(lo), int(hi), size=count, endpoint=True, dtype=np.int64)
            out[r] = _store(v, dtype)
        elif dist == "uniform":
            if dtype in INT_TYPES:
                raise ValueError(f"use int_uniform for {dtype}")
            if dtype == "float64":
                v = g.random(count) * (hi - lo) + lo
            else:
                v = g.random(count, dtype=np.float32) * np.float32(hi - lo) + np.float32(lo)
            out[r] = _store(v, dtype)
        elif dist == "normal":
            if dtype in INT_TYPES:
                raise ValueError(f"use int_uniform for {dtype}")
            if dtype == "float64":
                v = g.standard_normal(count) * std
            else:
                v = g.standard_normal(count, dtype=np.float32) * np.float32(std)
            out[r] = _store(v, dtype)
        else:
            raise ValueError(f"unknown dist {dist!r}")
    return out


def bucket_sizes(total_bytes: int, ntensors: int, lo_bytes: int, hi_bytes: int,
                 seed: int = 0, align: int = 16) -> list[int]:
    """Sizes (bytes) of a gradient bucket made of ``ntensors`` tensors.

    Sizes are drawn log-uniform in ``[lo_bytes, hi_bytes]``, rescaled so
    they add up to ``total_bytes``, rounded down to ``align`` bytes, and
    the last tensor takes the remainder.
    """
    g = np.random.default_rng(np.random.SeedSequence(seed))
    raw = np.exp(g.uniform(np.log(lo_bytes), np.log(hi_bytes), size=ntensors))
    raw *= total_bytes / raw.sum()
    sizes = [max(align, int(s) // align * align) for s in raw[:-1]]
    sizes.append(total_bytes - sum(sizes))
    if sizes[-1] <= 0:
        raise ValueError("bucket rescaling left no room for the last tensor")
    return sizes
