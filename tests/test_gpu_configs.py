"""GPU parity at the shapes of two benchmark configurations, and a stress
run of the flag protocols.

* The latency configuration: n = 8 virtual ranks, bf16 values normal(0, 1),
  ops sum / max / min, protocols LL, LL128 and Simple, every power-of-two
  per-rank size from 8 B to 4 MiB, ring and tree -- every output element
  bit-exact to the oracle under the schedule the library reports.
* The bandwidth configuration's channel sweep: n = 8, fp32 uniform [-1, 1)
  and int32 uniform [-2^20, 2^20], sum, ring, Simple, forced channel counts
  1, 4 and 32 at 16 MiB and 256 MiB per rank, sampled against the oracle's
  association predictor.
* LL and LL128 stress: many launches of random sizes and channel counts at
  n = 8 and n = 72 on one communicator, so the flags run on across launches
  (an LL line is one 16-byte store carrying data and flags, an LL128 line
  one warp store of eight 16-byte pieces with the flag in the last; a
  reader that saw a torn line would show up here as a wrong bit).
"""
import numpy as np
import pytest

from oracle import closed_form, ring as oring
from ring_allreduce_reduction_gb300.workloads import STORAGE, make_inputs
from tests.gpu_harness import Buffers
from tests.test_gpu_fullsize import _sampled_check, _tree_sampled

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def v():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from ring_allreduce_reduction_gb300 import build
    build.build()
    from ring_allreduce_reduction_gb300 import vrccl
    return vrccl


def _all_indices_ref(x, op, dtype, sched):
    idx = np.arange(x.shape[1])
    if sched["algo"] == "ring":
        return oring.ring_predict(x, op, dtype, sched["nchannels"], sched["chunk_elems"], idx)
    return _tree_sampled(x, op, dtype, sched["nchannels"], idx)


@pytest.mark.parametrize("algo", ["ring", "tree"])
@pytest.mark.parametrize("proto", ["ll", "ll128", "simple"])
def test_latency_config_bf16_n8(v, algo, proto):
    n = 8
    comm = v.vrcclCommInit(n, 32)
    try:
        for lg in range(3, 23):  # 8 B .. 4 MiB per rank
            count = (1 << lg) // 2
            for op in ("sum", "max", "min"):
                x = make_inputs(n, count, "bfloat16", "normal", seed=100 + lg)
                b = Buffers(x, "bfloat16")
                v.vrcclAllReduce(b.send_ptrs(), b.recv_ptrs(), count, "bfloat16", op, algo, proto, comm)
                y = b.result()
                sched = v.vrcclCommGetLastSchedule(comm)
                assert sched["algo"] == algo and sched["proto"] == proto
                for r in range(1, n):
                    assert np.array_equal(y[r], y[0]), (lg, op, r)
                ref = _all_indices_ref(x, op, "bfloat16", sched)
                bad = np.nonzero(y[0] != ref)[0]
                assert bad.size == 0, (lg, op, sched, bad[:5])
                ok, worst = closed_form.check(y[0], x, op, "bfloat16")
                assert ok, (lg, op, worst)
                assert b.canaries_intact(), (lg, op)
        assert v.vrcclCommGetAsyncError(comm) == 0
    finally:
        v.vrcclCommDestroy(comm)


@pytest.mark.parametrize("dtype", ["float32", "int32"])
@pytest.mark.parametrize("mib", [16, 256])
def test_bandwidth_config_channel_sweep(v, dtype, mib):
    import torch
    n, count = 8, (mib << 20) // 4
    if dtype == "int32":
        x = make_inputs(n, count, dtype, "int_uniform", seed=mib, lo=-2**20, hi=2**20)
    else:
        x = make_inputs(n, count, dtype, "uniform", seed=mib)
    send = torch.from_numpy(x).to("cuda:0")
    recv = torch.empty_like(send)
    comm = v.vrcclCommInit(n, 32)
    try:
        for C in (1, 4, 32):
            v.vrcclCommSetSchedule(comm, C, 0)
            recv.fill_(0)
            v.vrcclAllReduce([send[r] for r in range(n)], [recv[r] for r in range(n)], count, dtype, "sum", "ring",
                             "simple", comm)
            torch.cuda.synchronize()
            sched = _sampled_check(v, comm, x, recv, dtype, "sum", seed=C)
            assert sched["nchannels"] == C and sched["proto"] == "simple"
    finally:
        v.vrcclCommDestroy(comm)


@pytest.mark.parametrize("n", [8, 72])
def test_flag_protocols_stress(v, n):
    rng = np.random.default_rng(n)
    comm = v.vrcclCommInit(n, 16)
    try:
        for k in range(40):
            proto = ("ll", "ll128")[k % 2]
            algo = ("ring", "tree")[(k // 2) % 2]
            dtype = ("float32", "bfloat16", "int32")[k % 3]
            count = int(rng.integers(1, (1 << 18) // (4 if n == 72 else 1)))
            C = int(rng.integers(1, 9))
            v.vrcclCommSetSchedule(comm, C, 0)
            if dtype == "int32":
                x = make_inputs(n, count, dtype, "int_uniform", seed=k, lo=-2**20, hi=2**20)
            else:
                x = make_inputs(n, count, dtype, "normal", seed=k)
            b = Buffers(x, dtype)
            v.vrcclAllReduce(b.send_ptrs(), b.recv_ptrs(), count, dtype, "sum", algo, proto, comm)
            y = b.result()
            sched = v.vrcclCommGetLastSchedule(comm)
            for r in range(1, n):
                assert np.array_equal(y[r].view(np.uint8), y[0].view(np.uint8)), (k, r)
            ref = _all_indices_ref(x, "sum", dtype, sched)
            assert np.array_equal(y[0].view(np.uint8), ref.view(STORAGE[dtype]).view(np.uint8)), (k, sched, count)
            assert b.canaries_intact(), k
        assert v.vrcclCommGetAsyncError(comm) == 0
    finally:
        v.vrcclCommDestroy(comm)
