"""Schedules of the AllReduce: who handles which elements, in which order.

Test infrastructure only (see the package docstring for the sources).

Notation: n ranks, C channels, E bytes per element, A = 16 / E elements per
16 bytes, K chunk size in elements (a multiple of A).
"""
from __future__ import annotations


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def align_up(a: int, b: int) -> int:
    return ceil_div(a, b) * b


def channel_ranges(count: int, nchannels: int, elem_size: int) -> list[tuple[int, int]]:
    """Element range ``[lo, hi)`` of each channel.

    The data is cut into nChannels contiguous parts, channel c taking the
    c-th part, and channels run independently with no synchronisation
    between them [Deep Dive §2.2, "Step 3: Data Splitting";
    Architecture §6.3]. Reading of the page's ``count / nChannels``: each
    part is ``P = alignUp(ceil(count / C), A)`` elements, so every
    channel starts on a 16-byte boundary; the last parts may be short or
    empty.
    """
    if nchannels < 1:
        raise ValueError("nchannels must be >= 1")
    a = 16 // elem_size
    part = align_up(ceil_div(count, nchannels), a) if count else 0
    out = []
    for c in range(nchannels):
        lo = min(count, c * part)
        hi = min(count, (c + 1) * part)
        out.append((lo, hi))
    return out


def ring_loops(ch_count: int, nranks: int, chunk_elems: int, elem_size: int):
    """Loops and chunks of one channel's range, relative to its start.

    Follows RingARAlgorithm::getNextSendAddr [Deep Dive §2.3]: one loop
    covers ``n * K`` elements, one chunk per rank. When fewer than
    ``n * K`` elements remain, the chunk size shrinks to the number of
    remaining elements divided by n, rounded up to whole 16-byte units,
    and a chunk's element count is what is left after its offset (zero
    for chunks past the end).

    Yields ``(loop_offset, k, chunks)`` with ``chunks[j] = (lo, hi)``,
    ``lo <= hi``, relative to the channel start.
    """
    a = 16 // elem_size
    if chunk_elems <= 0 or chunk_elems % a:
        raise ValueError("chunk size must be a positive multiple of 16 bytes")
    loop = nranks * chunk_elems
    off = 0
    while off < ch_count:
        rem = ch_count - off
        k = chunk_elems if rem >= loop else align_up(ceil_div(rem, nranks), a)
        chunks = []
        for j in range(nranks):
            lo = off + min(rem, j * k)
            hi = off + min(rem, (j + 1) * k)
            chunks.append((lo, hi))
        yield off, k, chunks
        off += loop


def ring_next(nranks: int) -> list[int]:
    """The ring used for virtual ranks: rank r sends to r + 1 (mod n).

    This is the ring the pages show for eight ranks on one node, 0 -> 1 ->
    ... -> 7 -> 0 [Deep Dive ch.4, ncclBuildRings walkthrough].
    """
    return [(r + 1) % nranks for r in range(nranks)]


def build_ring(next_of: list[int], start: int = 0) -> list[int]:
    """Follow ``next`` from ``start`` n times; reject rings that do not close
    or miss a rank (the two checks of ncclBuildRings, [Deep Dive ch.4])."""
    n = len(next_of)
    seen = [False] * n
    order = []
    cur = start
    for _ in range(n):
        if not 0 <= cur < n:
            raise ValueError(f"ring leaves the rank range at {cur}")
        seen[cur] = True
        order.append(cur)
        cur = next_of[cur]
    if cur != start:
        raise ValueError(f"ring does not loop back to start ({cur} != {start})")
    missing = [r for r in range(n) if not seen[r]]
    if missing:
        raise ValueError(f"ring does not contain rank {missing[0]}")
    return order


def get_btree(nranks: int, rank: int) -> tuple[int, int, int]:
    """(parent, child0, child1) of ``rank`` in the bit-built binary tree.

    From ncclGetBtree [Deep Dive ch.4; Architecture §5.4]: b is the lowest
    set bit of the rank; the parent clears b and sets the next bit up,
    falling back to just clearing b when that leaves the rank range; the
    children are rank -/+ b/2, the upper one pulled down (the page's loop
    halves the offset one iteration late) until it is inside the range.
    Rank 0 is the root and has one child, the highest power of two below
    n. -1 means "none".
    """
    bit = 1
    while bit < nranks:
        if bit & rank:
            break
        bit <<= 1
    if rank == 0:
        return -1, -1, (bit >> 1) if nranks > 1 else -1
    up = (rank ^ bit) | (bit << 1)
    if up >= nranks:
        up = rank ^ bit
    lowbit = bit >> 1
    down0 = -1 if lowbit == 0 else rank - lowbit
    down1 = -1 if lowbit == 0 else rank + lowbit
    while down1 >= nranks:
        down1 = -1 if lowbit == 0 else rank + lowbit
        lowbit >>= 1
    return up, down0, down1


def get_dtree(nranks: int, rank: int) -> tuple[tuple[int, int, int], tuple[int, int, int]]:
    """The two trees of the double binary tree for ``rank``.

    From ncclGetDtree [Deep Dive ch.4 / Japanese edition ch.4, "odd rank
    handling"; Architecture §5.4]: tree 0 is the binary tree; tree 1 is its
    mirror ``r -> n-1-r`` when n is even, and its shift by one when n is
    odd. The odd-n body is elided on the pages; the reading used here is
    the plain one: build the binary tree for ``(r - 1) mod n`` and map every
    rank u it names to ``(u + 1) mod n``.
    """
    t0 = get_btree(nranks, rank)
    if nranks % 2 == 1:
        u, d0, d1 = get_btree(nranks, (rank - 1 + nranks) % nranks)
        f = lambda v: -1 if v == -1 else (v + 1) % nranks  # noqa: E731
    else:
        u, d0, d1 = get_btree(nranks, nranks - 1 - rank)
        f = lambda v: -1 if v == -1 else nranks - 1 - v  # noqa: E731
    return t0, (f(u), f(d0), f(d1))


def channel_tree(ch: int, nchannels: int) -> int:
    """Which of the two trees channel ``ch`` runs.

    NCCL doubles its channels and gives the second copy of each the other
    tree [Architecture §5.3, channel duplication; the INFO log of §10 shows
    channel 12 of 24 on tree 1]. Reading: the first ``ceil(C/2)`` channels
    run tree 0, the rest tree 1 (one channel -> tree 0 only).
    """
    return 0 if ch < ceil_div(nchannels, 2) else 1
