"""Benchmark: virtual-rank ring AllReduce on one GB300 (busbw and HBM GB/s).

One step = one AllReduce of the whole workload through the C ABI: n = 8
virtual ranks, 256 MiB of fp32 per rank (2 GiB in, 2 GiB out -- far larger
than the 129 MB L2, so no flush is needed between steps), op sum, ring,
Simple protocol, channel count from the library's schedule rule.

Reported (one JSON line on rank 0):
  value     busbw = algbw * 2(n-1)/n, algbw = bytes per rank / time, summed
            over GPUs (weak scaling: every GPU runs its own n virtual ranks)
  roofline  essential HBM bytes 2 n S per launch (read n inputs, write n
            outputs) / kernel time, against MEASURED_PEAKS.json's hbm_gbs
  e2e       the same metric with pinned host buffers: H2D of the inputs,
            the AllReduce, D2H of the outputs, every step; pipelined (the
            buffers in 8 pieces, upload / AllReduce / download overlapping
            on three streams), with the serial form beside it
  cpu_baseline  the CPU oracle replaying the same schedule on a bounded
            sample of the workload, on the host cores
`--impl reference` times that oracle alone (the reference arm).
`--coll reduce_scatter|all_gather` times one of the ring's two phases run
alone on the same n, dtype and 256 MiB per-rank buffer (ReduceScatter: the
send buffer; AllGather: the recv buffer) instead of the AllReduce.

Launch: python bench.py [--gpus N] [--steps K] [--warmup W]; for N > 1 under
torchrun (one process per GPU, RANK/LOCAL_RANK/WORLD_SIZE from the env).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = {
    "name": "n8_fp32_sum_ring_simple_256MiB",
    "nranks": 8,
    "dtype": "float32",
    "bytes_per_rank": 256 << 20,
    "op": "sum",
    "algo": "ring",
    "proto": "simple",
    "max_channels": 32,
}
METRIC = "allreduce busbw (n=8 virtual ranks, 256 MiB/rank fp32 sum, ring Simple)"
COLL_METRIC = {
    "allreduce": METRIC,
    "reduce_scatter": "reduce_scatter busbw (n=8 virtual ranks, 256 MiB/rank send fp32 sum, ring Simple)",
    "all_gather": "all_gather busbw (n=8 virtual ranks, 256 MiB/rank recv fp32, ring Simple)",
}
ELEM = {"int32": 4, "float32": 4, "bfloat16": 2, "float16": 2}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, device="cpu") -> float:
    """The largest value of x over all ranks of the process group (x itself
    without one): the job's time is its slowest rank's."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(rank: int) -> int:
    """The seed of GPU `rank`'s inputs: its shard of the one problem (or,
    for the bucket and the phases, its own problem) is drawn from it."""
    return 1000 + rank


def shard_of(v, count_per_gpu: int, dtype: str, world: int, rank: int):
    """One problem split over the GPUs by element range (weak scaling: the
    problem grows with the GPU count, each GPU's part stays the single-GPU
    workload). Returns (global count per virtual rank, this GPU's first
    element, its element count); the split is the library's
    vrcclShardRange. The global input is the concatenation of the shards'
    inputs, each drawn from its GPU's seed."""
    total = count_per_gpu * world
    off, ln = v.vrcclShardRange(total, dtype, world, rank)
    return total, off, ln


def busbw_gbs(bytes_per_rank: int, n: int, seconds: float, coll: str = "allreduce") -> float:
    """busbw = algbw * 2(n-1)/n with algbw = S / t ("NCCL architecture ...",
    introduction: the ring moves 2(n-1)/n * S per rank). Each phase alone
    moves half of that, (n-1)/n * S per rank, with S the per-rank buffer
    that holds all n blocks."""
    if n == 1:
        return bytes_per_rank / seconds / 1e9
    f = 2 if coll == "allreduce" else 1
    return bytes_per_rank / seconds * f * (n - 1) / n / 1e9


KERNEL_SOURCES = os.path.join(ROOT, "ring_allreduce_reduction_gb300", "csrc")
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "ring_simple_n8_fp32_256MiB.md")


def kernel_sources_sha256() -> str:
    """Hash of the sources the profiled kernel (the Simple-protocol ring) is
    compiled from: its translation unit, the device headers and the shared
    layout header. It ties an ncu summary to the kernel it measured; host
    code and the other kernels' translation units do not enter."""
    import hashlib
    h = hashlib.sha256()
    for f in sorted(os.listdir(KERNEL_SOURCES)):
        if f.endswith(".cuh") or f == "kernels_simple.cu" or f == "vrccl_internal.h":
            with open(os.path.join(KERNEL_SOURCES, f), "rb") as fh:
                h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()


def profiled_traffic(bytes_per_rank: int):
    """DRAM bytes per launch from the committed ncu summary, if it measured
    the current kernel sources (else None). The summary holds lines
    `kernel_sources_sha256: <hex>` and `dram_bytes_per_launch_<bytes>: <n>`."""
    try:
        with open(PROFILE_SUMMARY) as f:
            txt = f.read()
    except OSError:
        return None
    kv = {}
    for ln in txt.splitlines():
        ln = ln.strip().strip("`")
        if ":" in ln:
            k, _, val = ln.partition(":")
            kv[k.strip()] = val.strip()
    if kv.get("kernel_sources_sha256") != kernel_sources_sha256():
        return None
    val = kv.get(f"dram_bytes_per_launch_{bytes_per_rank}")
    return int(float(val)) if val else None


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---- the CPU oracle on the host cores: channels are independent ranges
# ("NCCL architecture ...", §6.3), so each worker process runs the oracle,
# unchanged, on one channel's part of every rank's buffer with one channel
# (the loops of a channel are cut relative to its own start, so the part's
# result is the whole run's). Inputs and outputs sit in shared memory.
_POOL_STATE = {}


def _pool_attach(in_name, out_name, shape, np_dtype):
    from multiprocessing import shared_memory
    shm_in = shared_memory.SharedMemory(name=in_name)
    shm_out = shared_memory.SharedMemory(name=out_name)
    _POOL_STATE.update(shm_in=shm_in, shm_out=shm_out,
                       x=np.ndarray(shape, dtype=np_dtype, buffer=shm_in.buf),
                       y=np.ndarray(shape, dtype=np_dtype, buffer=shm_out.buf))


def _pool_channel(task):
    from oracle import ring as oring
    lo, hi, op, dtype, chunk = task
    x, y = _POOL_STATE["x"], _POOL_STATE["y"]
    if hi > lo:
        y[:, lo:hi] = oring.ring_allreduce(np.ascontiguousarray(x[:, lo:hi]), op, dtype, 1, chunk)
    return hi - lo


class ParallelOracle:
    """The ring oracle over the channels of one schedule, one worker
    process per host core (at most one per channel)."""

    def __init__(self, x: np.ndarray, dtype: str, op: str, nch: int, chunk: int):
        import multiprocessing as mp
        from multiprocessing import shared_memory
        from oracle import schedule
        self.shape, self.np_dtype = x.shape, x.dtype
        self.shm_in = shared_memory.SharedMemory(create=True, size=max(1, x.nbytes))
        self.shm_out = shared_memory.SharedMemory(create=True, size=max(1, x.nbytes))
        np.ndarray(x.shape, dtype=x.dtype, buffer=self.shm_in.buf)[...] = x
        self.y = np.ndarray(x.shape, dtype=x.dtype, buffer=self.shm_out.buf)
        ranges = schedule.channel_ranges(x.shape[1], nch, ELEM[dtype])
        self.tasks = [(lo, hi, op, dtype, chunk) for lo, hi in ranges]
        self.cores = max(1, min(len(self.tasks), os.cpu_count() or 1))
        self.pool = mp.get_context("spawn").Pool(self.cores, initializer=_pool_attach,
                                                 initargs=(self.shm_in.name, self.shm_out.name, x.shape, x.dtype))
        self.pool.map(_pool_channel, [(0, 0, op, dtype, chunk)] * self.cores)  # workers up before timing

    def run(self) -> np.ndarray:
        self.pool.map(_pool_channel, self.tasks, chunksize=1)
        return self.y

    def close(self):
        self.pool.close()
        self.pool.join()
        for shm in (self.shm_in, self.shm_out):
            shm.close()
            shm.unlink()


def cpu_baseline(x: np.ndarray, dtype: str, op: str, nch: int, chunk_elems: int, min_seconds: float = 10.0,
                 coll: str = "allreduce") -> dict:
    """The oracle as it stands on the bench's own inputs, replaying the
    schedule the GPU ran (same channels and chunk) on the host cores (one
    process per channel, up to the core count), repeated until about
    `min_seconds` of wall time (at most 40 runs). The phases run on one
    core (their oracle has no channels)."""
    from oracle import phases
    n, count = x.shape
    par = None
    if coll == "allreduce":
        par = ParallelOracle(x, dtype, op, nch, chunk_elems)
        run, cores = par.run, par.cores
    else:
        run = {"reduce_scatter": lambda: phases.ring_reduce_scatter(x, op, dtype),
               "all_gather": lambda: phases.ring_all_gather(x)}[coll]
        cores = 1
    times = []
    try:
        while True:
            t0 = time.perf_counter()
            run()
            times.append(time.perf_counter() - t0)
            if sum(times) >= min_seconds or len(times) >= 40:
                break
    finally:
        if par is not None:
            par.close()
    dt = statistics.mean(times)
    S = count * ELEM[dtype] * (n if coll == "all_gather" else 1)
    how = (f"numpy step machine, one process per channel on {cores} host cores" if par is not None
           else "numpy step machine, one thread")
    return {"value": round(busbw_gbs(S, n, dt, coll), 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"the whole workload: n={n} x {count} {dtype} per rank send buffer, {coll}, {nch} channels, "
                      f"chunk {chunk_elems} elements; {how}; {len(times)} run(s), mean {dt:.2f} s"}


def run_reference(args) -> int:
    """Reference arm: the CPU oracle on the host cores (rank 0 only). Each
    step is a bounded sample of the workload (same n, dtype, op, ring order),
    sized from a calibration run so the whole run takes about
    args.ref_budget seconds."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    W = WORKLOAD
    n, dtype = W["nranks"], W["dtype"]
    from oracle import ring as oring
    from ring_allreduce_reduction_gb300.workloads import make_inputs
    # the schedule the GPU arm runs: the shipped tuning table's row for this
    # workload (ring, Simple), chunk = VRCCL_STEPS/2 slices of the row's slice
    from ring_allreduce_reduction_gb300.tune import read_table, table_choice
    tpath = os.path.join(ROOT, "ring_allreduce_reduction_gb300", "tuning", f"gb300_n{n}.txt")
    row = table_choice(read_table(tpath), n, W["bytes_per_rank"], ELEM[dtype], ("ring",), ("simple",),
                       W["max_channels"]) if os.path.exists(tpath) else None
    nch, chunk = (row["channels"], row["slice_bytes"] * 8 // ELEM[dtype]) if row else (1, 65536)
    probe = 1 << 20
    xp = make_inputs(n, probe, dtype, "uniform", seed=0)
    t0 = time.perf_counter()
    oring.ring_allreduce(xp, W["op"], dtype, nch, chunk)
    cores = max(1, min(nch, os.cpu_count() or 1))
    per_elem = (time.perf_counter() - t0) / probe / cores  # roughly: the channels run on `cores` processes
    per_step = args.ref_budget / max(1, args.steps + args.warmup)
    full = W["bytes_per_rank"] // ELEM[dtype]
    count = int(min(full, max(1 << 16, per_step / max(per_elem, 1e-12)))) // 4 * 4
    x = make_inputs(n, count, dtype, "uniform", seed=0)
    par = ParallelOracle(x, dtype, W["op"], nch, chunk)
    try:
        for _ in range(args.warmup):
            par.run()
        times = []
        for _ in range(args.steps):
            t0 = time.perf_counter()
            par.run()
            times.append(time.perf_counter() - t0)
    finally:
        par.close()
    S = count * ELEM[dtype]
    mean = statistics.mean(times)
    v = busbw_gbs(S, n, mean)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * mean, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": W["name"], "nranks": n, "bytes_per_rank": W["bytes_per_rank"],
                   "sample_bytes_per_rank": S, "op": W["op"], "algo": "ring", "channels": nch,
                   "chunk_elems": chunk},
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": par.cores, "kind": "oracle",
                         "sample": f"per step n={n} x {count} {dtype} per rank ({S >> 20} MiB/rank) of the "
                                   f"{W['bytes_per_rank'] >> 20} MiB/rank workload; numpy step machine, one "
                                   f"process per channel on {par.cores} host cores"},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


BUCKET = {"nranks": 8, "dtype": "bfloat16", "bytes_per_rank": 1 << 30, "ntensors": 224, "lo": 4 << 10,
          "hi": 64 << 20, "op": "avg", "max_channels": 32}


def run_bucket(args) -> int:
    """The gradient bucket: n = 8, 1 GiB of bf16 per rank made of 224
    tensors of log-uniform sizes in [4 KiB, 64 MiB], op avg, algo and
    protocol auto; one step reduces the whole bucket, as one flat call
    (`flat`), as 224 calls in one group (`group`) or as 224 separate calls
    (`separate`)."""
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    from ring_allreduce_reduction_gb300 import build
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        torch.distributed.barrier()
    from ring_allreduce_reduction_gb300 import vrccl as v
    from ring_allreduce_reduction_gb300.workloads import bucket_sizes, make_inputs
    B = BUCKET
    n, S = B["nranks"], B["bytes_per_rank"]
    sizes = bucket_sizes(S, B["ntensors"], B["lo"], B["hi"], seed=0, align=16)
    offs = np.concatenate([[0], np.cumsum(sizes)]) // 2
    x = make_inputs(n, S // 2, "bfloat16", "normal", seed=rank_seed(rank), std=1e-3)
    send = torch.from_numpy(x.view(np.int16)).cuda()
    recv = torch.empty_like(send)
    comm = v.vrcclCommInit(n, B["max_channels"])
    stream = torch.cuda.current_stream()
    views = [([send[r, int(a):int(b)] for r in range(n)], [recv[r, int(a):int(b)] for r in range(n)], int(b - a))
             for a, b in zip(offs[:-1], offs[1:])]

    def step():
        if args.bucket == "flat":
            v.vrcclAllReduce([send[r] for r in range(n)], [recv[r] for r in range(n)], S // 2, "bfloat16",
                             B["op"], "auto", "auto", comm, stream)
            return
        if args.bucket == "group":
            v.vrcclGroupStart()
        for sp, rp, cnt in views:
            v.vrcclAllReduce(sp, rp, cnt, "bfloat16", B["op"], "auto", "auto", comm, stream)
        if args.bucket == "group":
            v.vrcclGroupEnd()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if args.bucket == "flat":
        launches = 1
    elif args.bucket == "group":
        launches = 1 + max(v.vrcclCommGetGroupSchedule(comm, t)["launch"] for t in range(len(views)))
    else:
        launches = len(views)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
    err = v.vrcclCommGetAsyncError(comm)
    if err:
        raise RuntimeError(f"device error in the timed region: {v.RESULTS[err]}")
    ms = max_over_ranks(t0.elapsed_time(t1) / args.steps, "cuda")
    value = busbw_gbs(S, n, ms / 1e3) * world
    peak, peak_kind = measured_peak()
    achieved = 2 * n * S / (ms / 1e3) / 1e9
    v.vrcclCommDestroy(comm)
    if rank != 0:
        return 0
    line = {
        "metric": f"allreduce busbw (n=8 virtual ranks, bf16 1 GiB/rank bucket of 224 tensors, avg, auto; "
                  f"{args.bucket})",
        "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"n8_bf16_avg_bucket224_1GiB_{args.bucket}", "nranks": n, "bytes_per_rank": S,
                   "tensors": len(views), "launches_per_step": launches,
                   "l2": "inputs larger than L2 (8 GiB in, 8 GiB out); no flush"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": None,
                     "peak_kind": f"{peak_kind} hbm_gbs (burst copy)",
                     "algorithmic_bytes_per_step": 2 * n * S, "note": "whole step, all launches"},
        "gpu_launches": launches * args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def _host(x: np.ndarray) -> np.ndarray:
    """bf16 storage (uint16 bit patterns) as int16, which torch moves and
    pins like any 2-byte type."""
    return x.view(np.int16) if x.dtype == np.uint16 else x


def verify_download(x: np.ndarray, out: np.ndarray, op: str, dtype: str, nch: int, chunk: int, seed: int = 0,
                    samples: int = 200_000) -> bool:
    """Part of the CPU-baseline leg: a downloaded e2e result against the
    oracle's ring association for the schedule that ran, on sampled
    elements of every rank's buffer (and every rank equal to rank 0 there)."""
    from oracle import ring as oring
    n, count = x.shape
    idx = np.unique(np.concatenate([np.random.default_rng(seed).choice(count, min(samples, count), replace=False),
                                    [0, count - 1]]))
    ref = oring.ring_predict(x, op, dtype, nch, chunk, idx)
    return all(np.array_equal(out[r][idx].view(np.uint8), ref.view(np.uint8)) for r in range(n))


def run_e2e(v, comm, x, recv, send, step, n, count, dtype, W, coll, world, stream, steps):
    """The same metric end to end with pinned host buffers, in two forms,
    both timed; the faster is reported, the other kept beside it.

    serial     every step uploads the inputs, runs the collective and
               downloads the result on one stream;
    pipelined  (AllReduce) the buffers in 8 pieces, piece k+1's upload,
               piece k's AllReduce and piece k-1's download overlapping on
               three streams (the two copy directions run on separate copy
               engines).
    Returns the e2e record and, per form, the downloaded result with the
    schedule it ran, which the CPU-baseline leg checks against the oracle."""
    import torch
    S = count * ELEM[dtype]
    forms = {}
    host_in = torch.from_numpy(_host(x)).pin_memory()
    host_out = torch.empty(recv.shape, dtype=recv.dtype).pin_memory()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        send.copy_(host_in, non_blocking=True)
        step()
        host_out.copy_(recv, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, "cuda")
    sched = v.vrcclCommGetLastSchedule(comm)
    downloads = {}
    if coll == "allreduce":
        downloads["serial"] = [(x, host_out.numpy(), sched["nchannels"], sched["chunk_elems"])]
    forms["serial"] = {"value": round(busbw_gbs(S, n, ms / 1e3, coll) * world, 3), "ms_per_step": round(ms, 3),
                       "h2d_bytes_per_step": host_in.numel() * host_in.element_size(),
                       "d2h_bytes_per_step": host_out.numel() * host_out.element_size(), "verified": None,
                       "form": "serial: upload, AllReduce, download on one stream"}
    del host_in
    if coll == "allreduce" and count % 8 == 0:
        K, pc = 8, count // 8
        hin = torch.from_numpy(_host(x)).reshape(n, K, pc).permute(1, 0, 2).contiguous().pin_memory()  # [K, n, pc]
        hout = torch.empty(hin.shape, dtype=hin.dtype).pin_memory()
        dsend = torch.empty(hin.shape, dtype=hin.dtype, device="cuda")
        drecv = torch.empty_like(dsend)
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(K)]
        ev_red = [torch.cuda.Event() for _ in range(K)]
        ev_out = [torch.cuda.Event() for _ in range(K)]
        for k in range(K):  # events start completed
            ev_red[k].record(stream)
            ev_out[k].record(stream)

        def pipe_step():
            for k in range(K):
                s_in.wait_event(ev_red[k])  # the previous step's AllReduce of piece k read dsend[k]
                with torch.cuda.stream(s_in):
                    dsend[k].copy_(hin[k], non_blocking=True)
                ev_in[k].record(s_in)
                stream.wait_event(ev_in[k])
                stream.wait_event(ev_out[k])  # the previous step's download of drecv[k]
                v.vrcclAllReduce([dsend[k, r] for r in range(n)], [drecv[k, r] for r in range(n)], pc, dtype,
                                 W["op"], W["algo"], W["proto"], comm, stream)
                ev_red[k].record(stream)
                s_out.wait_event(ev_red[k])
                with torch.cuda.stream(s_out):
                    hout[k].copy_(drecv[k], non_blocking=True)
                ev_out[k].record(s_out)

        pipe_step()
        torch.cuda.synchronize()
        p0 = torch.cuda.Event(enable_timing=True)
        p1 = torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        for _ in range(steps):
            pipe_step()
        stream.wait_event(ev_out[K - 1])
        p1.record(stream)
        torch.cuda.synchronize()
        pms = max_over_ranks(p0.elapsed_time(p1) / steps, "cuda")
        ps = v.vrcclCommGetLastSchedule(comm)
        xk = x.reshape(n, K, pc)
        hk = hout.numpy()  # [K, n, pc]
        downloads["pipelined"] = [(np.ascontiguousarray(xk[:, k]), hk[k], ps["nchannels"], ps["chunk_elems"])
                                  for k in range(K)]
        forms["pipelined"] = {"value": round(busbw_gbs(S, n, pms / 1e3, coll) * world, 3),
                              "ms_per_step": round(pms, 3), "h2d_bytes_per_step": hin.numel() * hin.element_size(),
                              "d2h_bytes_per_step": hout.numel() * hout.element_size(), "verified": None,
                              "form": f"pipelined: {K} pieces of {pc} elements per rank, upload / AllReduce / "
                                      f"download on three streams"}
        del hin, dsend, drecv
    best = min(forms, key=lambda f: forms[f]["ms_per_step"])
    e2e = {"value": forms[best]["value"], "unit": "GB/s", "h2d_bytes_per_step": forms[best]["h2d_bytes_per_step"],
           "d2h_bytes_per_step": forms[best]["d2h_bytes_per_step"], "ms_per_step": forms[best]["ms_per_step"],
           "form": best, "verified": None, "forms": forms}
    return e2e, downloads


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--ref-budget", type=float, default=150.0, help="seconds the reference arm aims to take")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffers) leg")
    ap.add_argument("--coll", default="allreduce", choices=["allreduce", "reduce_scatter", "all_gather"],
                    help="allreduce (the workload), or one of its two ring phases run alone")
    ap.add_argument("--algo", default="ring", choices=["ring", "tree", "oneshot"],
                    help="allreduce only: the schedule timed (the workload's is the ring)")
    ap.add_argument("--no-bound", action="store_true", help="skip timing the one-shot bound beside the ring")
    ap.add_argument("--fifo", action="store_true",
                    help="ring AllReduce / AllGather with the all-gather through the FIFOs (the library's default "
                         "runs it through the recv buffers)")
    ap.add_argument("--bucket", default="", choices=["", "flat", "group", "separate"],
                    help="time the 224-tensor bf16 gradient bucket instead of the workload")
    ap.add_argument("--proto", default="", choices=["", "simple", "ll", "ll128"],
                    help="profiling only: another protocol than the workload's (named in config)")
    ap.add_argument("--dtype", default="", choices=["", "float32", "bfloat16"],
                    help="profiling only: another element type than the workload's (named in config)")
    ap.add_argument("--op", default="", choices=["", "sum", "prod", "max", "min", "avg"],
                    help="profiling only: another reduction op than the workload's (named in config)")
    ap.add_argument("--bytes-per-rank", type=int, default=0,
                    help="profiling only: a smaller per-rank size than the workload's (reported in config)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.bucket:
        return run_bucket(args)

    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    from ring_allreduce_reduction_gb300 import build
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        torch.distributed.barrier()
    from ring_allreduce_reduction_gb300 import vrccl as v
    from ring_allreduce_reduction_gb300.workloads import make_inputs

    W = dict(WORKLOAD)
    coll = args.coll
    if coll != "allreduce":
        W["name"] = W["name"].replace("_sum_", "_sum_" + coll + "_")
    elif args.algo != "ring":
        W["algo"] = args.algo
        W["name"] = W["name"].replace("_ring_", "_" + args.algo + "_")
    if args.proto and args.proto != W["proto"]:
        W["proto"] = args.proto
        W["name"] = W["name"].replace("_simple_", "_" + args.proto + "_")
    if args.dtype and args.dtype != W["dtype"]:
        W["dtype"] = args.dtype
        W["name"] = W["name"].replace("_fp32_", "_bf16_" if args.dtype == "bfloat16" else "_" + args.dtype + "_")
    if args.op and args.op != W["op"]:
        W["name"] = W["name"].replace("_" + W["op"] + "_", "_" + args.op + "_")
        W["op"] = args.op
    if args.bytes_per_rank:
        W["bytes_per_rank"] = args.bytes_per_rank
        W["name"] += f" (profiling size {args.bytes_per_rank} B/rank)"
    n, dtype = W["nranks"], W["dtype"]
    S = W["bytes_per_rank"]
    count = S // ELEM[dtype]           # elements of the per-rank buffer that holds all n blocks
    block = count // n                 # phases: elements per block
    shard = None
    if coll == "allreduce" and world > 1:
        # one AllReduce problem of world x S per virtual rank, split by
        # element range: this GPU reduces its part of every rank's buffer
        total, off, count = shard_of(v, count, dtype, world, rank)
        shard = {"global_count_per_rank": total, "offset": off, "count": count}
    x = make_inputs(n, block if coll == "all_gather" else count, dtype, "uniform", seed=rank_seed(rank))
    send = torch.from_numpy(_host(x)).cuda()
    recv = torch.empty((n, block) if coll == "reduce_scatter" else (n, count), dtype=send.dtype, device=send.device)
    sp, rp = [send[r] for r in range(n)], [recv[r] for r in range(n)]
    comm = v.vrcclCommInit(n, W["max_channels"])
    if args.fifo:
        v.vrcclCommSetDirect(comm, False)
        W["name"] += "_fifo"
    stream = torch.cuda.current_stream()

    def step():
        if coll == "allreduce":
            v.vrcclAllReduce(sp, rp, count, dtype, W["op"], W["algo"], W["proto"], comm, stream)
        elif coll == "reduce_scatter":
            v.vrcclReduceScatter(sp, rp, block, dtype, W["op"], W["proto"], comm, stream)
        else:
            v.vrcclAllGather(sp, rp, block, dtype, W["proto"], comm, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sched = v.vrcclCommGetLastSchedule(comm)
    shape = v.vrcclCommGetLaunchShape(comm)
    err = v.vrcclCommGetAsyncError(comm)
    if err:
        raise RuntimeError(f"device error during warm-up: {v.RESULTS[err]}")

    # ---- timed region: device-resident inputs
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    total_ms = t_start.elapsed_time(t_end)
    kern_ms = [a.elapsed_time(b) for a, b in ev]
    err = v.vrcclCommGetAsyncError(comm)
    if err:
        raise RuntimeError(f"device error in the timed region: {v.RESULTS[err]}")
    total_ms = max_over_ranks(total_ms, "cuda")
    ms_step = total_ms / args.steps
    value = busbw_gbs(S, n, ms_step / 1e3, coll) * world

    # roofline of the one kernel: essential bytes / mean launch time. The
    # AllReduce reads n inputs and writes n outputs (2 n S); a phase reads
    # and writes n S + S (n full buffers one way, n blocks the other).
    algo_bytes = 2 * n * S if coll == "allreduce" else (n + 1) * S
    mean_kern_s = statistics.mean(kern_ms) / 1e3
    peak, peak_kind = measured_peak()
    achieved = algo_bytes / mean_kern_s / 1e9
    traffic = (profiled_traffic(S) if coll == "allreduce" and not args.fifo and W["algo"] == "ring"
               and W["proto"] == "simple" and dtype == "float32" else None)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_kind": f"{peak_kind} hbm_gbs (burst copy)",
                "algorithmic_bytes_per_launch": algo_bytes}
    if traffic:
        # achieved DRAM GB/s: the ncu-measured DRAM bytes of one launch over
        # the live mean launch time, against the measured and the nominal peak
        dram = traffic / mean_kern_s / 1e9
        roofline.update({"dram_gbs": round(dram, 1), "dram_frac": round(dram / peak, 4),
                         "dram_frac_of_8tbs": round(dram / 8000.0, 4)})

    # ---- end to end through the public API with pinned host buffers
    e2e, downloads = None, {}
    if not args.no_e2e:
        e2e, downloads = run_e2e(v, comm, x, recv, send, step, n, count, dtype, W, coll, world, stream,
                                 args.e2e_steps)

    # ---- the one-shot bound on the same buffers and schedule: every input
    # read once, every output written once, the ring's association order
    bound = None
    if coll == "allreduce" and W["algo"] == "ring" and not args.no_bound:
        v.vrcclCommSetSchedule(comm, sched["nchannels"], sched["chunk_elems"] * ELEM[dtype])
        for _ in range(3):
            v.vrcclAllReduce(sp, rp, count, dtype, W["op"], "oneshot", "simple", comm, stream)
        nb = max(3, min(args.steps, 50))
        b0 = torch.cuda.Event(enable_timing=True)
        b1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        b0.record(stream)
        for _ in range(nb):
            v.vrcclAllReduce(sp, rp, count, dtype, W["op"], "oneshot", "simple", comm, stream)
        b1.record(stream)
        torch.cuda.synchronize()
        bms = b0.elapsed_time(b1) / nb
        v.vrcclCommSetSchedule(comm, 0, 0)
        bach = 2 * n * S / (bms / 1e3) / 1e9
        bound = {"algo": "oneshot", "ms_per_step": round(bms, 4), "achieved": round(bach, 1), "unit": "GB/s",
                 "frac": round(bach / peak, 4), "ring_time_over_bound": round(ms_step / bms, 3),
                 "launches": nb + 3}

    v.vrcclCommDestroy(comm)
    if rank != 0:
        return 0
    cpu = None
    if not args.no_cpu:
        cpu = cpu_baseline(x, dtype, W["op"], sched["nchannels"], sched["chunk_elems"], coll=coll)
        # the e2e downloads against the oracle (sampled, per piece)
        for form, pieces in downloads.items():
            per = max(1, 200_000 // len(pieces))
            e2e["forms"][form]["verified"] = all(
                verify_download(xi, yi, W["op"], dtype, nch, ck, seed=k, samples=per)
                for k, (xi, yi, nch, ck) in enumerate(pieces))
        if e2e is not None:
            e2e["verified"] = e2e["forms"][e2e["form"]]["verified"]
        downloads.clear()
    line = {
        "metric": COLL_METRIC[coll], "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": {"float32": "f32", "bfloat16": "bf16"}[dtype], "data": "synthetic",
        "config": {"workload": W["name"], "coll": coll, "nranks": n, "bytes_per_rank": S, "count": count,
                   "op": W["op"],
                   "algo": sched["algo"], "proto": sched["proto"], "channels": sched["nchannels"],
                   "chunk_elems": sched["chunk_elems"], "blocks": shape["blocks"], "threads": shape["threads"],
                   "slice_elems": shape["slice_elems"],
                   "allgather": ("none (one-shot)" if sched["algo"] == "oneshot" else
                                 "through the FIFOs" if args.fifo or coll == "reduce_scatter" or sched["algo"] != "ring"
                                 or sched["proto"] != "simple" else "through the recv buffers (direct)"),
                   "l2": "inputs larger than L2 (n*S = 2 GiB in, 2 GiB out); no flush",
                   "algbw_gbs": round(S / (ms_step / 1e3) / 1e9 * world, 3),
                   "parallelism": (f"one problem split over {world} GPUs by element range (vrcclShardRange); "
                                   f"no data-path collective" if shard else
                                   f"{world} independent problems" if world > 1 else "single GPU"),
                   "shard_rank0": shard},
        "kernel_ms": {"p10": round(float(np.percentile(kern_ms, 10)), 4),
                      "p50": round(float(np.percentile(kern_ms, 50)), 4),
                      "p90": round(float(np.percentile(kern_ms, 90)), 4)},
        "roofline": roofline,
        "oneshot_bound": bound,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
