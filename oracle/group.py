"""How a group's AllReduces are aggregated (test infrastructure only).

[Architecture §9.2] (ncclPrepareTasks) and [Deep Dive (Japanese edition)
ch.6, "step 2" and "step 3"]: the collectives registered between
ncclGroupStart and ncclGroupEnd are put into buckets by (function,
reduction op, data type); the sorter hands each bucket's tasks out by size,
largest first; tasks of a bucket whose sizes lie within 4x of each other are
aggregated and looked up in the tuning table together ("ten 1 MB
all_reduces in one group are timed as ten 1 MB operations in a pipeline",
numPipeOps = 10).

The printed loop (``aggEnd->trafficBytes < 4*aggBeg->trafficBytes``) read
against a largest-first order would take every task of a bucket; the prose
of both pages says "within 4x". Reading taken: a run starts at its largest
task and takes the following tasks (in largest-first order, equal sizes in
call order) while the run's largest is less than 4x the candidate.

Which calls may be grouped at all is the library's choice: AllReduces on
the ring (algo ring or auto); the protocol the caller asked for is part of
the bucket key, since a run is launched with one protocol.
"""
from __future__ import annotations


def aggregate(tasks):
    """Runs of a group.

    ``tasks``: list of ``(key, size)`` in call order; ``key`` is any hashable
    bucket key, ``size`` the per-rank byte (or element) count.
    Returns a list of runs, each a list of call indices, buckets in order
    of their first call, runs of a bucket largest first.
    """
    buckets: dict = {}
    order = []
    for i, (key, _size) in enumerate(tasks):
        if key not in buckets:
            buckets[key] = []
            order.append(key)
        buckets[key].append(i)
    runs = []
    for key in order:
        idx = sorted(buckets[key], key=lambda i: (-tasks[i][1], i))
        start = 0
        while start < len(idx):
            first = tasks[idx[start]][1]
            end = start + 1
            while end < len(idx) and first < 4 * tasks[idx[end]][1]:
                end += 1
            runs.append(idx[start:end])
            start = end
    return runs
