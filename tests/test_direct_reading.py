"""The direct all-gather's data flow, checked on the CPU from the schedule.

In the direct form (runRing's direct primitives, "NCCL architecture:
topology, channels, algorithms and protocols" §9.4) the step that finishes
a chunk writes it into its own recv buffer and the next rank's, each later
all-gather step forwards the chunk the predecessor wrote into this rank's
recv buffer on to the next rank's, and the last step has nothing to do (its
chunk is already in place), so it is passed over and only counted. The
kernels rely on three facts of the ring's chunk order ("NCCL Source Code
Deep Dive" §2.3, getNextSendAddr), checked here for many shapes with the
oracle's loop and chunk rules:

* the k-th slice a rank sends directly is the k-th slice its successor
  receives directly or passes over: same chunk, same position, same length
  (so one counter per edge, advanced by both ends, pairs them up);
* over a launch the two counts are equal (the receiver's count, run plus
  passed over, seeds the next launch);
* every chunk of every rank's recv buffer is written exactly once: by the
  rank itself when it finishes the chunk, or by its predecessor.
"""
import itertools

import numpy as np
import pytest

from oracle import schedule


def _chunk_at(n: int, r: int, p: int) -> int:
    """Chunk handled by rank r at primitive p of a loop (2n - 1 primitives):
    send r-1, then recvReduceSend r-1-p, recvReduceCopySend r (final),
    recvCopySend r-(p-n+1), recv r+1 (all mod n)."""
    if p == 0:
        return (r - 1) % n
    if p <= n - 2:
        return (r - 1 - p) % n
    if p == n - 1:
        return r
    if p <= 2 * n - 3:
        return (r - (p - n + 1)) % n
    return (r + 1) % n


def _direct_slices(n, r, ch_count, chunk_elems, elem_size, slice_elems):
    """(sent, received-or-passed, finished) of rank r on one channel:
    lists of (lo, hi) element ranges in the order the rank handles them."""
    sent, recvd, own = [], [], []
    for _, _, chunks in schedule.ring_loops(ch_count, n, chunk_elems, elem_size):
        for p in range(2 * n - 1):
            lo, hi = chunks[_chunk_at(n, r, p)]
            slices = [(s, min(s + slice_elems, hi)) for s in range(lo, hi, slice_elems)]
            if n - 1 <= p <= 2 * n - 3:
                sent += slices                  # written into the next rank's recv buffer
            if p >= n:
                recvd += slices                 # forwarded on, or (last step) passed over
            if p == n - 1:
                own += slices                   # finished here, written to the own buffer too
    return sent, recvd, own


SHAPES = list(itertools.product([2, 3, 5, 8], [4, 2], [1, 3]))


@pytest.mark.parametrize("n,elem_size,nchannels", SHAPES)
def test_direct_edges_pair_up_and_cover_every_chunk(n, elem_size, nchannels):
    rng = np.random.default_rng(n * 100 + elem_size * 10 + nchannels)
    a = 16 // elem_size
    for _ in range(6):
        count = int(rng.integers(1, 40_000))
        chunk = int(rng.choice([1, 4, 16, 64])) * a
        slice_elems = int(rng.choice([1, 2, 8])) * a
        for lo, hi in schedule.channel_ranges(count, nchannels, elem_size):
            ch = hi - lo
            per = [_direct_slices(n, r, ch, chunk, elem_size, slice_elems) for r in range(n)]
            for r in range(n):
                sent = per[r][0]
                recvd = per[(r + 1) % n][1]
                assert sent == recvd, (n, r, count, chunk, slice_elems)
            for r in range(n):
                cover = np.zeros(ch, dtype=np.int64)
                for s, e in per[r][2] + per[(r - 1) % n][0]:
                    cover[s:e] += 1
                assert np.all(cover == 1), (n, r, count, chunk, slice_elems)


def test_a_mistaken_order_is_caught():
    """The check has teeth: forwarding the chunk of the wrong step (one too
    early) breaks the pairing."""
    n, es, a = 5, 4, 4
    ch, chunk, sl = 3001, 16 * a, 2 * a

    def shifted(r):
        sent = []
        for _, _, chunks in schedule.ring_loops(ch, n, chunk, es):
            for p in range(2 * n - 1):
                if n - 2 <= p <= 2 * n - 4:  # the mistake: one primitive early
                    lo, hi = chunks[_chunk_at(n, r, p)]
                    sent += [(s, min(s + sl, hi)) for s in range(lo, hi, sl)]
        return sent

    good = [_direct_slices(n, r, ch, chunk, es, sl) for r in range(n)]
    assert any(shifted(r) != good[(r + 1) % n][1] for r in range(n))
