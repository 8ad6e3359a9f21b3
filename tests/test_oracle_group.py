"""Pins of the group aggregation rule (``oracle.group``). No GPU."""
import itertools
import random

import pytest

from oracle import group


def test_page_example_ten_equal_allreduces_form_one_run():
    """Ten 1 MB all_reduces in one group are looked up together
    ("NCCL architecture ...", §9.2: numPipeOps = 10)."""
    runs = group.aggregate([("ar", 1 << 20)] * 10)
    assert runs == [list(range(10))]


def test_four_times_boundary():
    # the run's largest must be below 4x the candidate
    assert group.aggregate([("k", 4000), ("k", 1000)]) == [[0], [1]]
    assert group.aggregate([("k", 3999), ("k", 1000)]) == [[0, 1]]
    # largest first, whatever the call order
    assert group.aggregate([("k", 10), ("k", 100), ("k", 30)]) == [[1, 2], [0]]


def test_buckets_never_mix():
    runs = group.aggregate([("a", 100), ("b", 100), ("a", 90), ("b", 95)])
    assert runs == [[0, 2], [1, 3]]


def _check_characterisation(tasks, runs):
    """The greedy runs are the unique partition with: runs inside one bucket,
    contiguous in largest-first order, every member within 4x of the run's
    first, and the task after a run not within 4x of that run's first."""
    seen = sorted(i for r in runs for i in r)
    assert seen == list(range(len(tasks)))
    by_key = {}
    for i, (k, s) in enumerate(tasks):
        by_key.setdefault(k, []).append(i)
    for k, members in by_key.items():
        order = sorted(members, key=lambda i: (-tasks[i][1], i))
        mine = [r for r in runs if tasks[r[0]][0] == k]
        assert [i for r in mine for i in r] == order
        for a, r in enumerate(mine):
            first = tasks[r[0]][1]
            assert all(tasks[i][0] == k for i in r)
            assert all(first < 4 * tasks[i][1] for i in r)
            if a + 1 < len(mine):
                assert not first < 4 * tasks[mine[a + 1][0]][1]


@pytest.mark.parametrize("seed", range(20))
def test_random_groups_by_characterisation(seed):
    rnd = random.Random(seed)
    tasks = [(rnd.choice("xyz"), int(2 ** rnd.uniform(10, 26))) for _ in range(rnd.randint(1, 60))]
    _check_characterisation(tasks, group.aggregate(tasks))


def test_brute_force_small():
    """Every size tuple over a small alphabet: the greedy runs satisfy the
    characterisation (which fixes them uniquely)."""
    for n in range(1, 6):
        for sizes in itertools.product([1, 3, 4, 12, 16, 50], repeat=n):
            tasks = [("k", s) for s in sizes]
            _check_characterisation(tasks, group.aggregate(tasks))
