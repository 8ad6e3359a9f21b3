"""Double-binary-tree AllReduce oracle (test infrastructure only).

The tree AllReduce reduces up the tree to the root, which then broadcasts
the result back down [Architecture §7.1 (Tree) and §9.4 (runTreeUpDown /
runTreeSplit)]. Each channel runs one of the two trees of the double binary
tree [Architecture §5.3-§5.4; Deep Dive ch.4]; see
``schedule.channel_tree`` for the channel-to-tree reading.

Readings where the pages are silent:

* order inside a node: the node's own (pre-scaled) value is the running
  value, then the value from child ``down[0]``, then from ``down[1]``:
  ``v = op(op(x_r, v_down0), v_down1)``;
* the integer avg post-op is applied once, at the root.

The result depends on the tree and this order only, not on how the
channel's range is cut into chunks, so no chunk size enters here.
"""
from __future__ import annotations

import numpy as np

from . import numerics as nm
from .schedule import channel_ranges, channel_tree, get_dtree

ELEM_SIZE = {"int32": 4, "float32": 4, "bfloat16": 2, "float16": 2, "int8": 1, "uint8": 1, "int64": 8,
             "float64": 8}


def tree_links(nranks: int, which: int) -> list[tuple[int, int, int]]:
    """(parent, child0, child1) for every rank in tree ``which``, checked
    for consistency (each child names its parent, one root, all reachable)."""
    links = [get_dtree(nranks, r)[which] for r in range(nranks)]
    roots = [r for r, (u, _, _) in enumerate(links) if u == -1]
    if len(roots) != 1:
        raise AssertionError(f"tree {which} of {nranks} has roots {roots}")
    for r, (u, d0, d1) in enumerate(links):
        for c in (d0, d1):
            if c != -1 and links[c][0] != r:
                raise AssertionError(f"rank {c} is a child of {r} but names parent {links[c][0]}")
        if u != -1 and r not in links[u][1:]:
            raise AssertionError(f"rank {r} names parent {u}, which does not list it")
    seen, stack = set(), [roots[0]]
    while stack:
        r = stack.pop()
        seen.add(r)
        stack.extend(c for c in links[r][1:] if c != -1)
    if len(seen) != nranks:
        raise AssertionError(f"tree {which} of {nranks} reaches only {len(seen)} ranks")
    return links


def tree_machine(local, combine_fn, post_fn, links, sl, out):
    """Reduce up / broadcast down over one slice ``sl`` of every rank."""
    n = len(local)
    depth = [0] * n
    for r in range(n):
        u, d = links[r][0], 0
        while u != -1:
            d += 1
            u = links[u][0]
        depth[r] = d
    up_val = {}
    for r in sorted(range(n), key=lambda q: -depth[q]):  # children before parents
        acc = local[r][sl]
        for c in links[r][1:]:
            if c != -1:
                acc = combine_fn(acc, up_val.pop(c))
        up_val[r] = acc
    root = next(r for r in range(n) if links[r][0] == -1)
    y = post_fn(up_val.pop(root))
    for r in sorted(range(n), key=lambda q: depth[q]):  # parents before children
        out[r][sl] = y
    return out


def tree_allreduce(inputs: np.ndarray, op: str, dtype: str, nchannels: int) -> np.ndarray:
    """Double-binary-tree AllReduce of ``inputs`` (``[n, count]``)."""
    inputs = np.asarray(inputs)
    n, count = inputs.shape
    local = [nm.prescale(inputs[r], op, dtype, n) for r in range(n)]
    out = [np.empty(count, dtype=inputs.dtype) for _ in range(n)]
    if n == 1:
        out[0][:] = nm.postop(local[0], op, dtype, 1)
        return np.stack(out)
    trees = [tree_links(n, 0), tree_links(n, 1)]
    for ch, (lo, hi) in enumerate(channel_ranges(count, nchannels, ELEM_SIZE[dtype])):
        if hi == lo:
            continue
        tree_machine(local, lambda a, b: nm.combine(op, a, b, dtype),
                     lambda v: nm.postop(v, op, dtype, n),
                     trees[channel_tree(ch, nchannels)], slice(lo, hi), out)
    return np.stack(out)
