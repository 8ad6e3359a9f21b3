"""Collectives captured in a CUDA graph and replayed: the FIFO counters and
flags live in device memory and run on across replays, so every replay must
give the oracle's bits (new inputs are copied in before each replay)."""
import numpy as np
import pytest

from oracle import phases, ring as oring
from ring_allreduce_reduction_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def v():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ring_allreduce_reduction_gb300 import build
    build.build()
    from ring_allreduce_reduction_gb300 import vrccl
    return vrccl


def test_graph_replays_match_the_oracle(v):
    import torch
    n, count = 8, 100_000
    comm = v.vrcclCommInit(n, 8)
    try:
        v.vrcclCommSetSchedule(comm, 4, 0)
        send = torch.zeros((n, count), dtype=torch.float32, device="cuda:0")
        outs = {p: torch.empty_like(send) for p in ("simple", "ll", "ll128")}
        rs_out = torch.empty((n, count // n), dtype=torch.float32, device="cuda:0")
        scheds = {}
        for p in outs:  # warm the schedule (and the library's occupancy cache) outside the capture
            v.vrcclAllReduce([send[r] for r in range(n)], [outs[p][r] for r in range(n)], count, "float32", "sum",
                             "ring", p, comm)
            scheds[p] = v.vrcclCommGetLastSchedule(comm)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        with torch.cuda.graph(g, stream=side):
            s = torch.cuda.current_stream()
            for p in outs:
                v.vrcclAllReduce([send[r] for r in range(n)], [outs[p][r] for r in range(n)], count, "float32",
                                 "sum", "ring", p, comm, s)
            v.vrcclReduceScatter([send[r] for r in range(n)], [rs_out[r] for r in range(n)], count // n, "float32",
                                 "sum", "simple", comm, s)
        for rep in range(4):
            x = make_inputs(n, count, "float32", "normal", seed=rep)
            send.copy_(torch.from_numpy(x))
            g.replay()
            torch.cuda.synchronize()
            for p, out in outs.items():
                ref = oring.ring_allreduce(x, "sum", "float32", scheds[p]["nchannels"], scheds[p]["chunk_elems"])
                assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32)), (rep, p)
            ref = phases.ring_reduce_scatter(x, "sum", "float32")
            assert np.array_equal(rs_out.cpu().numpy().view(np.uint32), ref.view(np.uint32)), rep
        assert v.vrcclCommGetAsyncError(comm) == 0
    finally:
        v.vrcclCommDestroy(comm)
