"""The two phases of the ring as standalone collectives (test infrastructure only).

[Deep Dive §2.3] walks the ring AllReduce as a reduce-scatter phase
followed by an all-gather phase, each n-1 steps per loop, which is why a
loop takes 2(n-1) steps. Run alone, the phases are the ReduceScatter and
AllGather collectives. The pages describe them only as phases, so their
buffer contract is read as NCCL's: with block size b,

* ReduceScatter: rank r's send buffer holds n blocks of b elements; its
  recv buffer (b elements) receives the reduction of every rank's block r.
* AllGather: rank r's send buffer holds b elements; block q of every
  rank's recv buffer (n blocks) receives rank q's send buffer.

The chunk a rank handles at each step follows the AllReduce ring
(RingARAlgorithm::getNextSendAddr, [Deep Dive §2.3]): in the reduce-scatter
phase rank r sends block r-1 first, adds its own contribution to the
block it receives, and holds the finished block r after n-1 steps; in the
all-gather phase rank r starts from its own block and, at step p,
receives block r-p. So an element of block c of the ReduceScatter result
is ``op(...op(op(x[c+1], x[c+2]), x[c+3])..., x[c])`` (indices mod n).

Channels and chunks only cut each block into pieces that travel the same
way: an element's association depends on its block alone. The step
machines below therefore move whole blocks, one loop, one channel.
"""
from __future__ import annotations

from collections import deque

import numpy as np

from . import numerics as nm


def _machine(n, nsteps, first, step, stats):
    """Lock-step ring of n ranks with an explicit FIFO per edge r -> r+1.

    ``first(r)`` gives (block, value) rank r sends at step 0;
    ``step(r, p, block, value)`` consumes what arrived at step p and
    returns the value to forward, or None at the last step.
    """
    fifo = [deque() for _ in range(n)]
    if stats is not None:
        stats.setdefault("sends", [0] * n)
        stats.setdefault("fifo_elems", 0)
    for p in range(nsteps):
        for r in range(n):
            if p == 0:
                c, v = first(r)
            else:
                c_in, v_in = fifo[(r - 1) % n].popleft()
                c, v = c_in, step(r, p, c_in, v_in)
            if v is not None:
                fifo[r].append((c, v))
                if stats is not None:
                    stats["sends"][r] += 1
                    stats["fifo_elems"] += len(v)
    if any(fifo):
        raise AssertionError("FIFO not drained at the end of the phase")


def reduce_scatter_machine(local, combine_fn, post_fn, stats: dict | None = None):
    """The reduce-scatter phase over per-rank arrays ``local[r]`` (n blocks
    of b values each, already pre-scaled); returns rank r's finished block r
    for every r. ``combine_fn(a, b)`` is one reduction step with ``a`` the
    received value; ``post_fn`` is applied where a block becomes final.
    """
    n = len(local)
    b = len(local[0]) // n
    blk = lambda r, c: local[r][c * b:(c + 1) * b]  # noqa: E731
    out = [None] * n
    if n == 1:
        out[0] = post_fn(local[0])
        return out

    def step(r, p, c, v):
        if c != (r - 1 - p) % n:
            raise AssertionError(f"rank {r} step {p}: FIFO holds block {c}")
        acc = combine_fn(v, blk(r, c))
        if p == n - 1:  # block r is final (recvReduceCopy with postOp)
            out[r] = post_fn(acc)
            return None
        return acc

    _machine(n, n, lambda r: ((r - 1) % n, blk(r, (r - 1) % n)), step, stats)
    return out


def ring_reduce_scatter(inputs: np.ndarray, op: str, dtype: str, stats: dict | None = None) -> np.ndarray:
    """ReduceScatter of ``inputs`` ([n, n*b], storage form) -> [n, b].

    The avg pre-scale and the integer avg post-op are those of the
    AllReduce (``numerics.prescale`` / ``numerics.postop``).
    """
    inputs = np.asarray(inputs)
    n, total = inputs.shape
    if total % max(n, 1):
        raise ValueError("send buffers must hold n blocks")
    local = [nm.prescale(inputs[r], op, dtype, n) for r in range(n)]
    res = reduce_scatter_machine(local, lambda a, b: nm.combine(op, a, b, dtype),
                                 lambda v: nm.postop(v, op, dtype, n), stats)
    return np.stack([np.asarray(v, dtype=inputs.dtype) for v in res]) if n else inputs.copy()


def ring_all_gather(inputs: np.ndarray, stats: dict | None = None) -> np.ndarray:
    """AllGather of ``inputs`` ([n, b], any storage type) -> [n, n*b]; a bitwise copy."""
    inputs = np.asarray(inputs)
    n, b = inputs.shape
    out = np.empty((n, n * b), dtype=inputs.dtype)
    for r in range(n):  # step 0: every rank places its own block
        out[r, r * b:(r + 1) * b] = inputs[r]
    if n == 1:
        return out

    def step(r, p, c, v):
        if c != (r - p) % n:
            raise AssertionError(f"rank {r} step {p}: FIFO holds block {c}")
        out[r, c * b:(c + 1) * b] = v
        return v if p < n - 1 else None

    _machine(n, n, lambda r: (r, inputs[r]), step, stats)
    return out


def reduce_scatter_predict(inputs: np.ndarray, op: str, dtype: str, rank: int,
                           idx: np.ndarray | None = None) -> np.ndarray:
    """Rank ``rank``'s ReduceScatter result at element indices ``idx`` of its block.

    The association written out directly: start from rank+1's element of
    block ``rank`` and fold in ranks rank+2, ..., rank (mod n).
    """
    inputs = np.asarray(inputs)
    n, total = inputs.shape
    b = total // n
    if idx is None:
        idx = np.arange(b, dtype=np.int64)
    col = rank * b + np.asarray(idx, dtype=np.int64)
    if n == 1:
        return nm.postop(nm.prescale(inputs[0, col], op, dtype, 1), op, dtype, 1)
    acc = nm.prescale(inputs[(rank + 1) % n, col], op, dtype, n)
    for i in range(2, n + 1):
        acc = nm.combine(op, acc, nm.prescale(inputs[(rank + i) % n, col], op, dtype, n), dtype)
    return nm.postop(acc, op, dtype, n)
