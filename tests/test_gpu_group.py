"""GPU parity of grouped calls (vrcclGroupStart / vrcclGroupEnd).

Every call of a group must give the bits the oracle gives for that call
alone under the schedule the library reports for it
(vrcclCommGetGroupSchedule); calls that the pages' aggregation rule puts in
one run must share a launch, and no others.
"""
import numpy as np
import pytest

from oracle import group as ogroup, phases, ring as oring, tree as otree
from ring_allreduce_reduction_gb300.workloads import ELEM_SIZE, STORAGE, bucket_sizes, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def v():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ring_allreduce_reduction_gb300 import build
    build.build()
    from ring_allreduce_reduction_gb300 import vrccl
    return vrccl


def _dev(x, dtype):
    """[n, count] on the device, every row starting on a 256-byte boundary
    (rows padded; the result is a view of the first `count` columns)."""
    import torch
    n, count = x.shape
    E = ELEM_SIZE[dtype]
    pad = max(-(-count * E // 256) * 256 // E, 256 // E)
    h = np.zeros((n, pad), dtype=np.int16 if E == 2 else x.dtype)
    h[:, :count] = np.ascontiguousarray(x).view(np.int16) if E == 2 else x
    return torch.from_numpy(h).to("cuda:0")[:, :count]


def _empty(t):
    import torch
    return torch.empty((t.shape[0], t.stride(0)), dtype=t.dtype, device=t.device)[:, :t.shape[1]]


def _host(t, dtype):
    import torch
    torch.cuda.synchronize()
    return np.ascontiguousarray(t.cpu().numpy()).view(STORAGE[dtype])


def _same(a, b):
    return np.array_equal(np.ascontiguousarray(a).view(np.uint8), np.ascontiguousarray(b).view(np.uint8))


def _oracle_ar(x, dtype, op, s):
    if s["algo"] == "tree":
        return otree.tree_allreduce(x, op, dtype, s["nchannels"])
    return oring.ring_allreduce(x, op, dtype, s["nchannels"], s["chunk_elems"])


@pytest.mark.parametrize("direct", [True, False])
def test_mixed_group_matches_oracle_and_aggregation_rule(v, direct):
    """Both all-gather forms: through the recv buffers (the default; every
    call's buffers are separate tensors, so the next rank's buffer of a task
    sits at its own offset) and through the FIFOs."""
    import torch
    n = 8
    comm = v.vrcclCommInit(n, 32)
    try:
        v.vrcclCommSetDirect(comm, direct)
        spec = [  # (dtype, op, count, algo, proto)
            ("float32", "sum", 300_000, "auto", "auto"),
            ("float32", "sum", 100_001, "ring", "auto"),      # within 4x of the first: same run
            ("float32", "sum", 50_000, "auto", "auto"),       # not within 4x of 300k: next run
            ("bfloat16", "avg", 70_000, "auto", "auto"),      # another bucket
            ("float32", "sum", 20_000, "auto", "auto"),       # 50k run
            ("float32", "sum", 7_000, "auto", "ll"),          # forced protocol: its own bucket
            ("float32", "sum", 6_000, "auto", "ll"),
            ("float32", "sum", 9_000, "tree", "auto"),        # tree: runs alone
            ("int32", "max", 0, "auto", "auto"),              # nothing to do
            ("bfloat16", "avg", 40_000, "auto", "auto"),
        ]
        xs, ins, outs = [], [], []
        for i, (dt, op, cnt, algo, proto) in enumerate(spec):
            x = make_inputs(n, cnt, dt, "normal" if dt != "int32" else "int_uniform", seed=i, **(
                {"lo": -100, "hi": 100} if dt == "int32" else {}))
            xs.append(x)
            ins.append(_dev(x, dt))
            outs.append(_empty(ins[-1]))
        # one reduce-scatter and one all-gather in the same group
        xrs = make_inputs(n, n * 1024, "float32", "normal", seed=99)
        rs_in = _dev(xrs, "float32")
        rs_out = torch.empty((n, 1024), dtype=torch.float32, device="cuda:0")
        xag = make_inputs(n, 2048, "bfloat16", "normal", seed=98)
        ag_in = _dev(xag, "bfloat16")
        ag_out = torch.empty((n, n * 2048), dtype=torch.int16, device="cuda:0")

        v.vrcclGroupStart()
        for i, (dt, op, cnt, algo, proto) in enumerate(spec):
            v.vrcclAllReduce([ins[i][r] for r in range(n)], [outs[i][r] for r in range(n)], cnt, dt, op, algo,
                             proto, comm)
        v.vrcclReduceScatter([rs_in[r] for r in range(n)], [rs_out[r] for r in range(n)], 1024, "float32", "sum",
                             "auto", comm)
        v.vrcclAllGather([ag_in[r] for r in range(n)], [ag_out[r] for r in range(n)], 2048, "bfloat16", "auto",
                         comm)
        v.vrcclGroupEnd()
        torch.cuda.synchronize()
        assert v.vrcclCommGetAsyncError(comm) == 0

        scheds = {}
        for i, (dt, op, cnt, algo, proto) in enumerate(spec):
            if cnt == 0:
                with pytest.raises(v.VrcclError):
                    v.vrcclCommGetGroupSchedule(comm, i)
                continue
            s = v.vrcclCommGetGroupSchedule(comm, i)
            scheds[i] = s
            y = _host(outs[i], dt)
            ref = _oracle_ar(xs[i], dt, op, s)
            assert _same(y, ref), (i, s)
            if algo == "tree":
                assert s["algo"] == "tree"
        y = _host(rs_out, "float32")
        assert _same(y, phases.ring_reduce_scatter(xrs, "sum", "float32"))
        y = ag_out.cpu().numpy().view(np.uint16)
        assert _same(y, phases.ring_all_gather(xag))

        # the aggregation: ring-able calls (ring/auto, count > 0) keyed by (type, op, requested proto)
        ringable = [i for i, sp in enumerate(spec) if sp[2] > 0 and sp[3] in ("ring", "auto")]
        tasks = [((spec[i][0], spec[i][1], spec[i][4]), spec[i][2]) for i in ringable]
        runs = [[ringable[j] for j in run] for run in ogroup.aggregate(tasks)]
        launch_of = {i: scheds[i]["launch"] for i in ringable}
        for run in runs:  # a run is scheduled as a whole: one launch
            assert len({launch_of[i] for i in run}) == 1, run
        # runs with the same launch shape may share a launch; calls of
        # different runs never share one unless their whole runs do
        for a in runs:
            for b in runs:
                if launch_of[a[0]] == launch_of[b[0]]:
                    assert scheds[a[0]]["proto"] == scheds[b[0]]["proto"]
        assert len(set(launch_of.values())) <= len(runs)
        assert [2, 4] in runs and [0, 1] in runs
    finally:
        v.vrcclCommDestroy(comm)


def test_gradient_bucket_as_224_grouped_calls(v):
    """The bf16 gradient bucket as 224 AllReduce calls in one group, each on
    its own slice of a flat buffer (avg, algo and protocol auto): every
    tensor bit-exact to the oracle under its reported schedule. Scaled to
    64 MiB per rank so the oracle checks every element."""
    import torch
    n, total = 8, 64 << 20
    sizes = bucket_sizes(total, 224, 256, 4 << 20, seed=0, align=16)
    count = total // 2
    x = make_inputs(n, count, "bfloat16", "normal", seed=7, std=1e-3)
    send = _dev(x, "bfloat16")
    recv = torch.empty_like(send)
    comm = v.vrcclCommInit(n, 32)
    try:
        offs = np.concatenate([[0], np.cumsum(sizes)]) // 2
        v.vrcclGroupStart()
        for t in range(224):
            a, b = int(offs[t]), int(offs[t + 1])
            v.vrcclAllReduce([send[r, a:b] for r in range(n)], [recv[r, a:b] for r in range(n)], b - a, "bfloat16",
                             "avg", "auto", "auto", comm)
        v.vrcclGroupEnd()
        y = _host(recv, "bfloat16")
        assert v.vrcclCommGetAsyncError(comm) == 0
        launches = set()
        for t in range(224):
            a, b = int(offs[t]), int(offs[t + 1])
            s = v.vrcclCommGetGroupSchedule(comm, t)
            launches.add(s["launch"])
            ref = oring.ring_allreduce(x[:, a:b], "avg", "bfloat16", s["nchannels"], s["chunk_elems"])
            assert _same(y[:, a:b], ref), (t, s)
        tasks = [("bf16avg", int(sz)) for sz in sizes]
        assert len(launches) <= len(ogroup.aggregate(tasks)) + 224 * 8 // 1536 + 1
        assert len(launches) < 12, "224 calls should need only a few launches"
    finally:
        v.vrcclCommDestroy(comm)


def test_group_rules(v):
    import torch
    n = 4
    comm = v.vrcclCommInit(n, 4)
    try:
        x = torch.zeros((n, 4096), dtype=torch.float32, device="cuda:0")
        y = torch.zeros_like(x)
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        v.vrcclGroupStart()
        v.vrcclAllReduce([x[r] for r in range(n)], [y[r] for r in range(n)], 4096, "float32", "sum", "ring",
                         "simple", comm, s1)
        with pytest.raises(v.VrcclError):  # a second stream for the same communicator
            v.vrcclAllReduce([x[r] for r in range(n)], [y[r] for r in range(n)], 4096, "float32", "sum", "ring",
                             "simple", comm, s2)
        v.vrcclGroupStart()  # nested
        v.vrcclGroupEnd()
        v.vrcclGroupEnd()
        torch.cuda.synchronize()
        assert v.vrcclCommGetGroupSchedule(comm, 0)["launch"] == 0
        with pytest.raises(v.VrcclError):
            v.vrcclCommGetGroupSchedule(comm, 1)
        with pytest.raises(v.VrcclError):
            v.vrcclGroupEnd()
        assert v.vrcclCommGetAsyncError(comm) == 0
    finally:
        v.vrcclCommDestroy(comm)


def test_group_over_two_communicators_and_many_tasks(v):
    """Two communicators in one group, and more calls than one launch's
    parameter block holds (the run is split into several launches)."""
    import torch
    comms = [v.vrcclCommInit(4, 8), v.vrcclCommInit(16, 4)]
    try:
        data = []
        v.vrcclGroupStart()
        for ci, comm in enumerate(comms):
            n = 4 if ci == 0 else 16
            ntask = 200 if ci == 0 else 100  # 200 calls x 4 ranks > one launch's 128 tasks
            for t in range(ntask):
                cnt = 1000 + 37 * (t % 5)
                x = make_inputs(n, cnt, "float32", "normal", seed=1000 * ci + t)
                a = _dev(x, "float32")
                b = _empty(a)
                data.append((ci, t, x, a, b))
                v.vrcclAllReduce([a[r] for r in range(n)], [b[r] for r in range(n)], cnt, "float32", "sum", "auto",
                                 "auto", comm)
        v.vrcclGroupEnd()
        torch.cuda.synchronize()
        launches = [set(), set()]
        for ci, t, x, a, b in data:
            s = v.vrcclCommGetGroupSchedule(comms[ci], t)
            launches[ci].add(s["launch"])
            assert _same(_host(b, "float32"), _oracle_ar(x, "float32", "sum", s)), (ci, t, s)
        assert len(launches[0]) >= 2
        for c in comms:
            assert v.vrcclCommGetAsyncError(c) == 0
    finally:
        for c in comms:
            v.vrcclCommDestroy(c)
