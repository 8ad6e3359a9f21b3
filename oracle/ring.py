"""Ring AllReduce oracle (test infrastructure only).

Two independent routes to the same bits:

* ``ring_allreduce`` replays the ring as a step machine. Every channel runs
  its loops; in every loop each rank executes the 2n-1 primitives of
  runRing [Architecture §9.4, device-side primitives]:

  ====  ===========================  ====================================
  p     primitive                    chunk handled by rank r
  ====  ===========================  ====================================
  0     send                         (r - 1) mod n
  1..   recv, reduce, send           (r - 1 - p) mod n      (n-2 times)
  n-1   recv, reduce, copy, send     r      (post-op; result is final)
  n..   recv, copy, send             (r - (p - n + 1)) mod n (n-2 times)
  2n-2  recv, copy                   (r + 1) mod n
  ====  ===========================  ====================================

  The chunk index follows ``chunkId = (ringIndex + n - 1 - chunkStage) mod
  n`` of RingARAlgorithm::getNextSendAddr [Deep Dive §2.3]: rank r sends
  chunk r-1 at stage 0 and holds the finished chunk r after n-1 stages.
  (The prose walkthrough beside it rotates the other way, "rank 0 sends
  element 0"; the code is followed.) Each rank-to-next edge is an explicit
  FIFO; a received value is the running value ``a`` of ``combine(op, a,
  local)``. Ranks move in lock-step, one primitive at a time, which is one
  legal interleaving of the real, asynchronous ring; the result does not
  depend on the interleaving.

* ``ring_predict`` writes the resulting association down directly: an
  element of chunk j ends up as
  ``op(...op(op(x[j+1], x[j+2]), x[j+3])..., x[j])`` (indices mod n), with
  its own, vectorised copy of the chunk addressing. It evaluates any set
  of sampled indices, which is how the full-size GPU runs are checked.
"""
from __future__ import annotations

from collections import deque

import numpy as np

from . import numerics as nm
from .schedule import align_up, ceil_div, channel_ranges, ring_loops

ELEM_SIZE = {"int32": 4, "float32": 4, "bfloat16": 2, "float16": 2, "int8": 1, "uint8": 1, "int64": 8,
             "float64": 8}


def ring_machine(local, combine_fn, post_fn, count: int, nchannels: int, chunk_elems: int,
                 elem_size: int, stats: dict | None = None, out_factory=None):
    """Step machine over per-rank value arrays ``local[r]`` (already pre-scaled).

    ``combine_fn(a, b)`` is one reduction step with ``a`` the received value;
    ``post_fn(v)`` is the post-op applied where a chunk becomes final.
    Returns the n output arrays. ``stats`` (optional) collects the number of
    primitives and FIFO payload elements per rank.
    """
    n = len(local)
    make = out_factory or (lambda r: np.empty_like(local[r]))
    out = [make(r) for r in range(n)]
    if stats is not None:
        stats.setdefault("primitives", [0] * n)
        stats.setdefault("sends", [0] * n)
        stats.setdefault("fifo_elems", 0)
        stats.setdefault("loops", 0)
        stats.setdefault("max_fifo_depth", 0)
    if n == 1:
        out[0][:] = post_fn(local[0][:])
        return out
    for lo, hi in channel_ranges(count, nchannels, elem_size):
        for _off, _k, chunks in ring_loops(hi - lo, n, chunk_elems, elem_size):
            if stats is not None:
                stats["loops"] += 1
            sl = [slice(lo + a, lo + b) for a, b in chunks]
            fifo = [deque() for _ in range(n)]  # fifo[r]: edge r -> r+1

            def send(r, c, v):
                fifo[r].append((c, v))
                if stats is not None:
                    stats["sends"][r] += 1
                    stats["fifo_elems"] += len(v)
                    stats["max_fifo_depth"] = max(stats["max_fifo_depth"], len(fifo[r]))

            def recv(r, c):
                got_c, v = fifo[(r - 1) % n].popleft()
                if got_c != c:
                    raise AssertionError(f"rank {r} expected chunk {c}, FIFO holds {got_c}")
                return v

            for p in range(2 * n - 1):
                for r in range(n):
                    if stats is not None:
                        stats["primitives"][r] += 1
                    if p == 0:
                        c = (r - 1) % n
                        send(r, c, local[r][sl[c]])
                    elif p <= n - 2:
                        c = (r - 1 - p) % n
                        send(r, c, combine_fn(recv(r, c), local[r][sl[c]]))
                    elif p == n - 1:
                        c = r
                        v = post_fn(combine_fn(recv(r, c), local[r][sl[c]]))
                        out[r][sl[c]] = v
                        send(r, c, v)
                    elif p <= 2 * n - 3:
                        c = (r - (p - n + 1)) % n
                        v = recv(r, c)
                        out[r][sl[c]] = v
                        send(r, c, v)
                    else:
                        c = (r + 1) % n
                        out[r][sl[c]] = recv(r, c)
            if any(fifo):
                raise AssertionError("FIFO not drained at the end of a loop")
    return out


def ring_allreduce(inputs: np.ndarray, op: str, dtype: str, nchannels: int, chunk_elems: int,
                   stats: dict | None = None) -> np.ndarray:
    """Ring AllReduce of ``inputs`` (``[n, count]``, storage form).

    Returns ``[n, count]``: the recv buffer of every virtual rank.
    """
    inputs = np.asarray(inputs)
    n, count = inputs.shape
    local = [nm.prescale(inputs[r], op, dtype, n) for r in range(n)]
    out = ring_machine(local,
                       lambda a, b: nm.combine(op, a, b, dtype),
                       lambda v: nm.postop(v, op, dtype, n),
                       count, nchannels, chunk_elems, ELEM_SIZE[dtype], stats,
                       out_factory=lambda r: np.empty(count, dtype=inputs.dtype))
    return np.stack(out) if n else inputs.copy()


def chunk_index(idx: np.ndarray, count: int, n: int, nchannels: int, chunk_elems: int,
                elem_size: int) -> np.ndarray:
    """Chunk index j (0..n-1) of each element index, vectorised.

    A second, independent statement of the channel partition and the loop
    chunking (see ``schedule.channel_ranges`` / ``schedule.ring_loops``).
    """
    a = 16 // elem_size
    idx = np.asarray(idx, dtype=np.int64)
    part = align_up(ceil_div(count, nchannels), a) if count else 1
    ch = idx // part
    ch_lo = ch * part
    ch_count = np.minimum(count, ch_lo + part) - ch_lo
    within = idx - ch_lo
    loop = n * chunk_elems
    loop_off = (within // loop) * loop
    rem = ch_count - loop_off
    tail_k = ((rem + n - 1) // n + a - 1) // a * a
    k = np.where(rem >= loop, chunk_elems, tail_k)
    return (within - loop_off) // k


def ring_predict(inputs: np.ndarray, op: str, dtype: str, nchannels: int, chunk_elems: int,
                 idx: np.ndarray | None = None) -> np.ndarray:
    """Result of the ring at element indices ``idx`` (all if None)."""
    inputs = np.asarray(inputs)
    n, count = inputs.shape
    if idx is None:
        idx = np.arange(count, dtype=np.int64)
    idx = np.asarray(idx, dtype=np.int64)
    if n == 1:
        return nm.postop(nm.prescale(inputs[0, idx], op, dtype, 1), op, dtype, 1)
    j = chunk_index(idx, count, n, nchannels, chunk_elems, ELEM_SIZE[dtype])
    acc = nm.prescale(inputs[(j + 1) % n, idx], op, dtype, n)
    for i in range(2, n + 1):
        nxt = nm.prescale(inputs[(j + i) % n, idx], op, dtype, n)
        acc = nm.combine(op, acc, nxt, dtype)
    return nm.postop(acc, op, dtype, n)
