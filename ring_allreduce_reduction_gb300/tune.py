"""Measure the auto-tuning table on this GPU, through the C ABI.

NCCL fills its tuning tables from model constants and takes the smallest
predicted time T = latency + bytes / bandwidth per (algorithm, protocol)
("NCCL architecture: topology, channels, algorithms and protocols", §8.2).
Here every (algo, proto, channels) candidate is timed at every power-of-two
message size, and the table records the measured microseconds per call;
``vrcclCommLoadTuning`` (or ``VRCCL_TUNE_FILE``) makes "auto" pick the
measured minimum at the nearest size.

Usage (on the GPU):
    python -m ring_allreduce_reduction_gb300.tune --nranks 8 --dtype bfloat16 \\
        --min-bytes 8 --max-bytes 4194304 --out table.txt

Table format (one entry per line, '#' comments):
    nranks algo proto channels log2bytes sliceBytes microseconds elementBytes
(the library also reads lines without the last field, as rows for every
element size). ``--append`` adds a sweep's rows to an existing table, so
one table holds the sweeps of several element types.

    python -m ring_allreduce_reduction_gb300.tune --compare table.txt
prints a table beside the pages' analytic model (no GPU needed).
"""
from __future__ import annotations

import argparse
import os
import sys
import time

import torch

ELEM = {"int32": 4, "float32": 4, "bfloat16": 2, "float16": 2, "int8": 1, "uint8": 1, "int64": 8, "float64": 8}
TORCH = {"int32": torch.int32, "float32": torch.float32, "bfloat16": torch.bfloat16, "float16": torch.float16,
         "int8": torch.int8, "uint8": torch.uint8, "int64": torch.int64, "float64": torch.float64}


def time_call(v, comm, sp, rp, count, dtype, op, algo, proto, iters, warmup, stream) -> float:
    """Mean microseconds per call over `iters` back-to-back calls on one stream."""
    for _ in range(warmup):
        v.vrcclAllReduce(sp, rp, count, dtype, op, algo, proto, comm, stream)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(iters):
        v.vrcclAllReduce(sp, rp, count, dtype, op, algo, proto, comm, stream)
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) * 1e3 / iters


def time_graph(v, comm, sp, rp, count, dtype, op, algo, proto, calls, reps, stream) -> float:
    """Mean microseconds per call with `calls` calls captured in one CUDA
    graph and the graph replayed `reps` times: the device-side latency,
    without the host's launch overhead. (A replay does not run the host's
    LL/LL128 flag-wrap accounting; `calls * reps` stays far below the 2^31
    steps after which a flag could repeat.)"""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        cap = torch.cuda.current_stream()
        for _ in range(calls):
            v.vrcclAllReduce(sp, rp, count, dtype, op, algo, proto, comm, cap)
    g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (calls * reps)


def sweep(nranks: int, dtype: str, sizes: list[int], protos: list[str], algos: list[str], channels: list[int],
          op: str = "sum", max_channels: int = 32, iters: int = 30, warmup: int = 3, log=print,
          graph: bool = False) -> list[dict]:
    """Time every candidate at every size; returns one record per point."""
    from ring_allreduce_reduction_gb300 import vrccl as v
    E = ELEM[dtype]
    maxcount = max(sizes) // E
    pad = (maxcount + 15) // 16 * 16
    send = torch.zeros((nranks, pad), dtype=TORCH[dtype], device="cuda")
    if dtype in ("int32", "int8", "uint8", "int64"):
        send.random_(0, 100)
    else:
        send.uniform_(-1, 1)
    recv = torch.empty_like(send)
    sp = [send[r] for r in range(nranks)]
    rp = [recv[r] for r in range(nranks)]
    comm = v.vrcclCommInit(nranks, max_channels)
    stream = torch.cuda.current_stream()
    out = []
    try:
        for nbytes in sizes:
            count = max(1, nbytes // E)
            for algo in algos:
                if algo == "tree" and nranks == 1:
                    continue
                for proto in protos:
                    for nch in channels:
                        if nch > max_channels:
                            continue
                        v.vrcclCommSetSchedule(comm, nch, 0)
                        try:
                            it = iters if nbytes <= (1 << 24) else max(3, iters // 10)
                            us = time_call(v, comm, sp, rp, count, dtype, op, algo, proto, it, warmup, stream)
                            if graph:  # the same point, 1000 calls per graph replay
                                us = time_graph(v, comm, sp, rp, count, dtype, op, algo, proto, 1000, 3, stream)
                        except v.VrcclError as e:  # a shape this GPU cannot hold at once
                            log(f"# skip n={nranks} {algo}/{proto} C={nch} {nbytes} B: {e}")
                            continue
                        sched = v.vrcclCommGetLastSchedule(comm)
                        shape = v.vrcclCommGetLaunchShape(comm)
                        rec = {"nranks": nranks, "dtype": dtype, "bytes": count * E, "algo": algo, "proto": proto,
                               "channels": sched["nchannels"], "chunk_elems": sched["chunk_elems"],
                               "slice_bytes": shape["slice_elems"] * E, "us": us,
                               "busbw_gbs": count * E / (us * 1e-6) * (2 * (nranks - 1) / nranks if nranks > 1 else 1)
                               / 1e9}
                        out.append(rec)
                        log(f"n={nranks} {dtype} {count * E:>11d} B {algo:4s} {proto:6s} C={sched['nchannels']:2d} "
                            f"{us:10.2f} us  busbw {rec['busbw_gbs']:8.2f} GB/s")
        err = v.vrcclCommGetAsyncError(comm)
        if err:
            raise RuntimeError(f"device error during the sweep: {v.RESULTS[err]}")
    finally:
        v.vrcclCommDestroy(comm)
    return out


def write_table(records: list[dict], path: str, header: str = "", append: bool = False) -> None:
    alg = {"ring": 0, "tree": 1}
    pro = {"simple": 0, "ll": 1, "ll128": 2}
    fresh = not (append and os.path.exists(path))
    with open(path, "w" if fresh else "a") as f:
        if fresh:
            f.write("# vrccl tuning table: nranks algo proto channels log2bytes sliceBytes microseconds "
                    "elementBytes\n")
        if header:
            for ln in header.splitlines():
                f.write(f"# {ln}\n")
        for r in records:
            log2 = max(0, int(r["bytes"]).bit_length() - 1)
            f.write(f"{r['nranks']} {alg[r['algo']]} {pro[r['proto']]} {r['channels']} {log2} {r['slice_bytes']} "
                    f"{r['us']:.3f} {ELEM[r['dtype']] if 'dtype' in r else 0}\n")


def read_table(path: str) -> list[dict]:
    alg = {0: "ring", 1: "tree"}
    pro = {0: "simple", 1: "ll", 2: "ll128"}
    recs = []
    for ln in open(path):
        ln = ln.split("#", 1)[0].split()
        if len(ln) in (7, 8):
            n, a, p, c, lg, sl, us = ln[:7]
            recs.append({"nranks": int(n), "algo": alg[int(a)], "proto": pro[int(p)], "channels": int(c),
                         "bytes": 1 << int(lg), "slice_bytes": int(sl), "us": float(us),
                         "esize": int(ln[7]) if len(ln) == 8 else 0})
    return recs


def table_choice(recs: list[dict], nranks: int, nbytes: int, esize: int, algos=("ring", "tree"),
                 protos=("simple", "ll", "ll128"), max_channels: int = 64) -> dict | None:
    """The row the library's tuner takes for a call (host only, for tools
    that need the schedule without a GPU): the rows of the call's element
    size (else rows for any size, else the nearest measured element size),
    the nearest measured power-of-two size, the fastest row there. None
    if the table has no eligible row."""
    import math
    el = [r for r in recs if r["nranks"] == nranks and r["channels"] <= max_channels and r["algo"] in algos
          and r["proto"] in protos]
    if not el:
        return None
    sizes = {r.get("esize", 0) for r in el}
    if esize in sizes:
        g = esize
    elif 0 in sizes:
        g = 0
    else:
        g = min(sizes, key=lambda e: (abs(math.log2(e) - math.log2(esize)), -e))
    el = [r for r in el if r.get("esize", 0) == g]
    b = max(0, int(nbytes).bit_length() - 1)
    if b < 62 and nbytes - (1 << b) > (1 << (b + 1)) - nbytes:
        b += 1
    want = 1 << b
    d = min(abs(r["bytes"].bit_length() - want.bit_length()) for r in el)
    here = [r for r in el if abs(r["bytes"].bit_length() - want.bit_length()) == d]
    return min(here, key=lambda r: r["us"])


def compare(recs: list[dict], arch: str = "blackwell", hw: str = "nvlink") -> list[dict]:
    """The measured table beside the pages' model (vrcclModelPredict), as
    the pages' log reader sets NCCL's printed tuning table against measured
    times. The model's one free input is the per-channel link bandwidth:
    here the ring/Simple bus bandwidth per channel at the table's largest
    size. Returns one row per size: the measured best, the model's best and
    the ratio measured / model for the measured best's (algo, proto)."""
    from ring_allreduce_reduction_gb300 import vrccl as v
    n = recs[0]["nranks"]
    big = max(r["bytes"] for r in recs)
    simple = [r for r in recs if r["bytes"] == big and r["algo"] == "ring" and r["proto"] == "simple"]
    best_big = min(simple, key=lambda r: r["us"])
    C = best_big["channels"]
    busbw = big / (best_big["us"] * 1e-6) * 2 * (n - 1) / n / 1e9
    bw_link = busbw / C
    rows = []
    for size in sorted({r["bytes"] for r in recs}):
        here = [r for r in recs if r["bytes"] == size]
        meas = min(here, key=lambda r: r["us"])
        model = {}
        for a in ("ring", "tree"):
            for p in ("simple", "ll", "ll128"):
                model[(a, p)] = v.vrcclModelPredict(n, 1, C, bw_link, a, p, size, arch=arch, hw_intra=hw)["time_us"]
        mbest = min(model, key=model.get)
        rows.append({"bytes": size, "measured": (meas["algo"], meas["proto"], meas["channels"], meas["us"]),
                     "model": (mbest[0], mbest[1], model[mbest]),
                     "ratio": meas["us"] / model[(meas["algo"], meas["proto"])]})
    return rows, {"nranks": n, "channels": C, "bw_link_gbs": bw_link, "arch": arch, "hw": hw}


def print_compare(rows, graph) -> None:
    print(f"# measured table vs the pages' model: {graph['nranks']} ranks, {graph['channels']} channels x "
          f"{graph['bw_link_gbs']:.1f} GB/s (fitted), {graph['hw']} latencies, {graph['arch']} constants")
    print(f"{'bytes':>12} | {'measured best':>28} | {'model best':>24} | measured/model")
    for r in rows:
        a, p, c, us = r["measured"]
        ma, mp, mus = r["model"]
        print(f"{r['bytes']:>12} | {a + '/' + p + ' C=' + str(c):>17} {us:9.1f} us | {ma + '/' + mp:>13} "
              f"{mus:8.1f} us | {r['ratio']:6.2f}")


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--compare", default="", help="print a measured table beside the pages' model and exit")
    ap.add_argument("--nranks", type=int, default=8)
    ap.add_argument("--dtype", default="bfloat16", choices=list(ELEM))
    ap.add_argument("--op", default="sum")
    ap.add_argument("--min-bytes", type=int, default=8)
    ap.add_argument("--max-bytes", type=int, default=4 << 20)
    ap.add_argument("--protos", default="simple,ll,ll128")
    ap.add_argument("--algos", default="ring,tree")
    ap.add_argument("--channels", default="1,2,4,8,16,32")
    ap.add_argument("--max-channels", type=int, default=32)
    ap.add_argument("--iters", type=int, default=30)
    ap.add_argument("--out", default="")
    ap.add_argument("--append", action="store_true", help="add the rows to the --out table instead of replacing it")
    ap.add_argument("--json", default="")
    ap.add_argument("--graph", action="store_true",
                    help="time 1000 calls captured in a CUDA graph per point (device latency, no launch overhead)")
    args = ap.parse_args()
    if args.compare:
        rows, graph = compare(read_table(args.compare))
        print_compare(rows, graph)
        return 0
    sizes, b = [], args.min_bytes
    while b <= args.max_bytes:
        sizes.append(b)
        b *= 2
    t0 = time.time()
    recs = sweep(args.nranks, args.dtype, sizes, args.protos.split(","), args.algos.split(","),
                 [int(c) for c in args.channels.split(",")], args.op, args.max_channels, args.iters,
                 graph=args.graph)
    if args.out:
        write_table(recs, args.out, header=f"measured on {torch.cuda.get_device_name()} in {time.time() - t0:.0f} s, "
                                           f"dtype {args.dtype}, op {args.op}", append=args.append)
    if args.json:
        import json
        with open(args.json, "w") as f:
            json.dump(recs, f)
    return 0


if __name__ == "__main__":
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    sys.exit(main())
