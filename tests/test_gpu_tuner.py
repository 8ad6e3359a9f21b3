"""The measured tuner: "auto" takes the table's fastest entry at the nearest
measured size, among the entries the caller left free. Through the C ABI."""
import os

import numpy as np
import pytest

from oracle import ring as oring, tree as otree
from ring_allreduce_reduction_gb300.workloads import make_inputs
from tests.gpu_harness import run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def v():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ring_allreduce_reduction_gb300 import build
    build.build()
    from ring_allreduce_reduction_gb300 import vrccl
    return vrccl


def _check(x, y, sched):
    if sched["algo"] == "tree":
        ref = otree.tree_allreduce(x, "sum", "float32", sched["nchannels"])
    else:
        ref = oring.ring_allreduce(x, "sum", "float32", sched["nchannels"], sched["chunk_elems"])
    assert np.array_equal(y.view(np.uint32), ref.view(np.uint32))


def test_auto_follows_the_measured_table(v, tmp_path):
    n = 5
    table = tmp_path / "table.txt"
    # nranks algo proto channels log2bytes sliceBytes us ; 2^18 B = 65536 floats
    table.write_text("# synthetic\n"
                     "5 0 0 2 18 16384 10.0\n"   # ring simple C=2
                     "5 1 2 3 18 30720 5.0\n"    # tree ll128 C=3  <- fastest overall
                     "5 0 1 1 18 8192 7.0\n"     # ring ll C=1     <- fastest ring
                     "5 0 0 4 10 16384 1.0\n"    # another size: must not be picked
                     "7 0 0 1 18 16384 0.5\n")   # another rank count: ignored
    comm = v.vrcclCommInit(n, 4)
    try:
        assert v.vrcclCommLoadTuning(comm, str(table)) == 4
        x = make_inputs(n, 70000, "float32", "normal", seed=3)  # 280000 B: nearest measured size 2^18
        for algo, proto, want in (("auto", "auto", ("tree", "ll128", 3)),
                                  ("auto", "simple", ("ring", "simple", 2)),
                                  ("ring", "auto", ("ring", "ll", 1))):
            y, sched, _ = run(v, comm, x, "float32", "sum", algo, proto)
            assert (sched["algo"], sched["proto"], sched["nchannels"]) == want, (algo, proto, sched)
            _check(x, y, sched)
    finally:
        v.vrcclCommDestroy(comm)


@pytest.mark.parametrize("n", [4, 8, 16, 32, 72])
def test_shipped_tables_drive_auto(v, n, monkeypatch, capfd):
    """Every configured rank count has a shipped table: "auto" takes the
    row the table rule names (the host mirror in tune.table_choice), the
    decision line says the choice was measured, and the result is the
    oracle's."""
    from ring_allreduce_reduction_gb300 import tune, vrccl
    path = os.path.join(os.path.dirname(vrccl.LIB_PATH), "tuning", f"gb300_n{n}.txt")
    assert os.path.exists(path)
    rows = tune.read_table(path)
    monkeypatch.setenv("VRCCL_DEBUG", "INFO")
    comm = v.vrcclCommInit(n, 64)
    try:
        for count in (64, 1 << 14, 1 << 17, 64, 70):  # repeated and same-bucket sizes: the kept choices
            x = make_inputs(n, count, "float32", "normal", seed=4)
            y, sched, _ = run(v, comm, x, "float32", "sum", "auto", "auto")
            want = tune.table_choice(rows, n, count * 4, 4)
            assert (sched["algo"], sched["proto"]) == (want["algo"], want["proto"]), (count, sched, want)
            _check(x, y, sched)
        err = capfd.readouterr().err
        lines = [ln for ln in err.splitlines() if "VRCCL INFO AllReduce" in ln]
        assert len(lines) == 5 and all("tuning measured (4-byte rows" in ln for ln in lines), lines
    finally:
        v.vrcclCommDestroy(comm)


def test_env_lists_steer_auto(v, monkeypatch):
    """VRCCL_ALGO / VRCCL_PROTO in NCCL's list syntax, read when the
    communicator is made: per-collective restrictions, exclusions, and
    NCCL's "no algorithm available" when nothing is left."""
    import torch
    n = 8
    x = torch.randn((n, 1 << 16), device="cuda:0")
    y = torch.empty_like(x)
    rs = torch.empty((n, (1 << 16) // n), device="cuda:0")

    def ar(comm):
        v.vrcclAllReduce([x[r] for r in range(n)], [y[r] for r in range(n)], 1 << 16, "float32", "sum", "auto",
                         "auto", comm)
        return v.vrcclCommGetLastSchedule(comm)

    def red_scat(comm):
        v.vrcclReduceScatter([x[r] for r in range(n)], [rs[r] for r in range(n)], (1 << 16) // n, "float32", "sum",
                             "auto", comm)
        return v.vrcclCommGetLastSchedule(comm)

    monkeypatch.setenv("VRCCL_ALGO", "ring;allreduce:tree")
    monkeypatch.setenv("VRCCL_PROTO", "^ll;allreduce:LL128")
    comm = v.vrcclCommInit(n, 8)
    try:
        s = ar(comm)
        assert (s["algo"], s["proto"]) == ("tree", "ll128")
        s = red_scat(comm)
        assert s["algo"] == "ring" and s["proto"] in ("simple", "ll128")
        s = v.vrcclAllReduce([x[r] for r in range(n)], [y[r] for r in range(n)], 1 << 16, "float32", "sum", "ring",
                             "simple", comm)  # an explicit choice overrides the lists
        s = v.vrcclCommGetLastSchedule(comm)
        assert (s["algo"], s["proto"]) == ("ring", "simple")
        torch.cuda.synchronize()
        assert v.vrcclCommGetAsyncError(comm) == 0
    finally:
        v.vrcclCommDestroy(comm)
    monkeypatch.setenv("VRCCL_ALGO", "tree")  # the phases have only the ring
    monkeypatch.delenv("VRCCL_PROTO")
    comm = v.vrcclCommInit(n, 8)
    try:
        assert ar(comm)["algo"] == "tree"
        with pytest.raises(v.VrcclError) as e:
            red_scat(comm)
        assert e.value.name == "vrcclInvalidUsage"
    finally:
        v.vrcclCommDestroy(comm)
    monkeypatch.setenv("VRCCL_ALGO", "ring,torus")
    with pytest.raises(v.VrcclError) as e:
        v.vrcclCommInit(n, 8)
    assert e.value.name == "vrcclInvalidArgument"


def test_element_size_picks_its_own_rows(v, tmp_path, monkeypatch, capfd):
    """A table keyed by element size: a bf16 call and an fp32 call of the
    same byte size take their own rows; a type the table has no rows for
    takes the rows of the nearest measured element size. The decision line
    (VRCCL_DEBUG=INFO) names the rows used."""
    n = 5
    table = tmp_path / "table.txt"
    # nranks algo proto channels log2bytes sliceBytes us elementBytes; 2^18 B per rank
    table.write_text("5 1 2 3 18 30720 5.0 2\n"    # bf16: tree ll128 C=3
                     "5 0 0 2 18 16384 9.0 2\n"
                     "5 0 0 2 18 16384 4.0 4\n"    # fp32: ring simple C=2
                     "5 1 2 3 18 30720 6.0 4\n")
    monkeypatch.setenv("VRCCL_DEBUG", "INFO")
    comm = v.vrcclCommInit(n, 4)
    try:
        assert v.vrcclCommLoadTuning(comm, str(table)) == 4
        for dtype, count, want in (("bfloat16", 1 << 17, ("tree", "ll128", 3)),
                                   ("float32", 1 << 16, ("ring", "simple", 2)),
                                   ("int8", 1 << 18, ("tree", "ll128", 3)),      # nearest rows: 2-byte
                                   ("float64", 1 << 15, ("ring", "simple", 2))):  # nearest rows: 4-byte
            if dtype == "int8":
                x = make_inputs(n, count, dtype, "int_uniform", seed=5, lo=-128, hi=127)
            else:
                x = make_inputs(n, count, dtype, "normal", seed=5)
            y, sched, _ = run(v, comm, x, dtype, "sum", "auto", "auto")
            assert (sched["algo"], sched["proto"], sched["nchannels"]) == want, (dtype, sched)
            if sched["algo"] == "tree":
                ref = otree.tree_allreduce(x, "sum", dtype, sched["nchannels"])
            else:
                ref = oring.ring_allreduce(x, "sum", dtype, sched["nchannels"], sched["chunk_elems"])
            assert np.array_equal(y.view(np.uint8), ref.view(np.uint8)), dtype
        err = capfd.readouterr().err
        lines = [ln for ln in err.splitlines() if "VRCCL INFO AllReduce" in ln]
        assert len(lines) == 4
        assert "measured (2-byte rows, 2^18 B)" in lines[0] and "measured (4-byte rows, 2^18 B)" in lines[1]
        assert "measured (2-byte rows" in lines[2] and "measured (4-byte rows" in lines[3]
    finally:
        v.vrcclCommDestroy(comm)
