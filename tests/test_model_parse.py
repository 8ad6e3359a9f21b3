"""The pages' tuning model and the NCCL_ALGO / NCCL_PROTO list syntax, in the
library (vrcclModelPredict, vrcclParseList), against the values and
examples the pages print (tests/golden/). No GPU."""
import json
import os

import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def v():
    pytest.importorskip("torch")
    from ring_allreduce_reduction_gb300 import build
    build.build()
    from ring_allreduce_reduction_gb300 import vrccl
    return vrccl


def _close(got, want, whole=False):
    # the page rounds to 0.1, or to whole units where the fixture says so
    return abs(got - want) <= (0.5 if whole else 0.06)


def _predict(v, case, nbytes=1, ops=1):
    nr, nn, nch, bw_intra, bw_inter, hw, arch = case["graph"]
    return v.vrcclModelPredict(nr, nn, nch, bw_intra, case["algo"], case["proto"], nbytes, ops, bw_inter=bw_inter,
                               hw_intra=hw, arch=arch)


def test_model_reproduces_the_pages_worked_numbers(v):
    fx = json.load(open(os.path.join(GOLDEN, "tuning_model.json")))
    for case in fx["cases"]:
        p = _predict(v, case, case.get("bytes", 1))
        whole = case.get("whole_units", [])
        if "lat" in case:
            assert _close(p["lat_us"], case["lat"], "lat" in whole), (case["what"], p)
        if "algbw" in case:
            assert _close(p["algbw_gbs"], case["algbw"], "algbw" in whole), (case["what"], p)
        if "time" in case:
            assert abs(p["time_us"] - case["time"]) <= 0.01 * case["time"], (case["what"], p)


def test_model_crossover_machine_three(v):
    """Tree+Simple and Ring+Simple cross near 533 MB on the 32-node machine."""
    fx = json.load(open(os.path.join(GOLDEN, "tuning_model.json")))
    ring = next(c for c in fx["cases"] if c["what"] == "machine three Ring+Simple")
    tree = next(c for c in fx["cases"] if c["what"] == "machine three Tree+Simple")
    lo, hi = 1 << 20, 1 << 34
    while hi - lo > 1 << 16:
        mid = (lo + hi) // 2
        if _predict(v, tree, mid)["time_us"] < _predict(v, ring, mid)["time_us"]:
            lo = mid
        else:
            hi = mid
    assert abs(lo - fx["crossover_machine_three_bytes"]) <= 0.02 * fx["crossover_machine_three_bytes"]


def test_model_structure(v):
    """Properties the formulas fix: time = latency + bytes / bandwidth; the
    ring pays the latency once per pipelined operation, the tree once; the
    ring's steps grow with 2(n-1), the tree's with the depth."""
    p1 = v.vrcclModelPredict(8, 1, 16, 24.0, "ring", "simple", 1 << 30)
    assert abs(p1["time_us"] - (p1["lat_us"] + (1 << 30) / (1000 * p1["algbw_gbs"]))) < 1e-3 * p1["time_us"]
    r4 = v.vrcclModelPredict(8, 1, 16, 24.0, "ring", "ll", 1 << 20, 4)
    r1 = v.vrcclModelPredict(8, 1, 16, 24.0, "ring", "ll", 1 << 20, 1)
    assert abs((r4["time_us"] - r1["time_us"]) - 3 * r1["lat_us"]) < 1e-2
    t4 = v.vrcclModelPredict(8, 1, 16, 24.0, "tree", "ll", 1 << 20, 4)
    t1 = v.vrcclModelPredict(8, 1, 16, 24.0, "tree", "ll", 1 << 20, 1)
    assert abs(t4["time_us"] - t1["time_us"]) < 1e-3
    a = v.vrcclModelPredict(8, 1, 16, 24.0, "ring", "simple", 1)["lat_us"]
    b = v.vrcclModelPredict(16, 1, 16, 24.0, "ring", "simple", 1)["lat_us"]
    assert abs((b - a) - 16 * 3.4) < 1e-3  # 2(16-1) - 2(8-1) = 16 more NVLink steps of 3.4 us
    with pytest.raises(v.VrcclError):
        v.vrcclModelPredict(8, 3, 16, 24.0, "ring", "simple", 1)  # 8 ranks do not split over 3 nodes


def test_parse_list_page_examples(v):
    fx = json.load(open(os.path.join(GOLDEN, "parse_list.json")))
    for case in fx["cases"]:
        got = v.vrcclParseList(case["spec"], case["kind"])
        for fn, names in case["expect"].items():
            assert sorted(got[fn]) == sorted(names), (case["spec"], fn, got[fn])
    for kind, spec in fx["unrecognized"]:
        with pytest.raises(v.VrcclError):
            v.vrcclParseList(spec, kind)


def test_parse_list_rules(v):
    everything = v.vrcclParseList(None, "proto")
    assert all(sorted(x) == ["ll", "ll128", "simple"] for x in everything.values())
    assert v.vrcclParseList("", "algo")["allreduce"] == v.PARSE_NAMES[0]
    assert v.vrcclParseList("SIMPLE", "proto")["allgather"] == ["simple"]          # case-insensitive
    assert v.vrcclParseList("^ring", "algo")["allreduce"] == [n for n in v.PARSE_NAMES[0] if n != "ring"]
    got = v.vrcclParseList(" ll , ll128 ; reducescatter : simple ", "proto")  # spaces around tokens
    assert got["reducescatter"] == ["simple"] and got["allreduce"] == ["ll", "ll128"]


def test_compare_prints_the_shipped_table_beside_the_model(v):
    from ring_allreduce_reduction_gb300 import tune
    path = os.path.join(os.path.dirname(GOLDEN), "..", "ring_allreduce_reduction_gb300", "tuning", "gb300_n8.txt")
    recs = tune.read_table(path)
    rows, graph = tune.compare(recs)
    assert [r["bytes"] for r in rows] == sorted({r["bytes"] for r in recs})
    assert graph["bw_link_gbs"] > 0 and graph["channels"] >= 1
    # the link bandwidth is fitted at the largest size, where the model's
    # latency term is small: the ratio there is just under 1
    last = rows[-1]
    assert last["measured"][:2] == ("ring", "simple") and 0.85 < last["ratio"] <= 1.0
    assert all(r["ratio"] > 0 for r in rows)
