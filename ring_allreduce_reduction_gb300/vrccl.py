"""Python binding of libvrccl.so: the C entry points under the same names.

Argument marshalling only -- every step of the AllReduce runs in the
library's sm_103a kernels. Buffers may be given as torch tensors (their
``data_ptr()`` is passed) or as raw integer device addresses; streams as
``torch.cuda.Stream``, a raw ``cudaStream_t`` integer, or None (the current
torch stream).

Importing this module loads ``libvrccl.so`` and raises ImportError if it has
not been built (``python -m ring_allreduce_reduction_gb300.build``): there
is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import torch  # noqa: F401  (loads the CUDA runtime the library links against)

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libvrccl.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is missing: build it with `python -m ring_allreduce_reduction_gb300.build`")
_lib = ctypes.CDLL(_LIB_PATH)

RESULTS = ["vrcclSuccess", "vrcclInvalidArgument", "vrcclInvalidUsage", "vrcclInternalError",
           "vrcclCudaError", "vrcclTimeout", "vrcclAborted"]
DTYPES = {"int32": 0, "float32": 1, "bfloat16": 2, "float16": 3, "int8": 4, "uint8": 5, "int64": 6, "float64": 7}
OPS = {"sum": 0, "prod": 1, "max": 2, "min": 3, "avg": 4}
ALGOS = {"ring": 0, "tree": 1, "auto": 2, "oneshot": 3}
PROTOS = {"simple": 0, "ll": 1, "ll128": 2, "auto": 3}
ALGO_NAMES = {v: k for k, v in ALGOS.items()}
PROTO_NAMES = {v: k for k, v in PROTOS.items()}
ELEM_SIZE = {"int32": 4, "float32": 4, "bfloat16": 2, "float16": 2, "int8": 1, "uint8": 1, "int64": 8, "float64": 8}
MAX_RANKS = 128
MAX_CHANNELS = 64
STEPS = 16

_TORCH_DTYPES = {torch.int32: "int32", torch.float32: "float32", torch.bfloat16: "bfloat16",
                 torch.float16: "float16", torch.int8: "int8", torch.uint8: "uint8", torch.int64: "int64",
                 torch.float64: "float64"}

_c_int_p = ctypes.POINTER(ctypes.c_int)
_sig = {
    "vrcclCommInit": [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int, ctypes.c_int],
    "vrcclAllReduce": [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t,
                       ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p],
    "vrcclReduceScatter": [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t,
                           ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p],
    "vrcclAllGather": [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t,
                       ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p],
    "vrcclGroupStart": [],
    "vrcclGroupEnd": [],
    "vrcclCommGetGroupSchedule": [ctypes.c_void_p, ctypes.c_int, _c_int_p, _c_int_p, _c_int_p,
                                  ctypes.POINTER(ctypes.c_size_t), _c_int_p],
    "vrcclParseList": [ctypes.c_char_p, ctypes.c_int, ctypes.POINTER(ctypes.c_uint)],
    "vrcclModelPredict": [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_size_t, ctypes.c_int,
                          ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float),
                          ctypes.POINTER(ctypes.c_float)],
    "vrcclCommSetDirect": [ctypes.c_void_p, ctypes.c_int],
    "vrcclCommSetSchedule": [ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t],
    "vrcclCommGetLastSchedule": [ctypes.c_void_p, _c_int_p, _c_int_p, _c_int_p, ctypes.POINTER(ctypes.c_size_t)],
    "vrcclCommGetAsyncError": [ctypes.c_void_p, _c_int_p],
    "vrcclCommGetErrorInfo": [ctypes.c_void_p, _c_int_p, _c_int_p, ctypes.POINTER(ctypes.c_uint64)],
    "vrcclCommSetTimeout": [ctypes.c_void_p, ctypes.c_uint64],
    "vrcclCommAbort": [ctypes.c_void_p],
    "vrcclCommDestroy": [ctypes.c_void_p],
    "vrcclCommCount": [ctypes.c_void_p, _c_int_p],
    "vrcclCommInjectFault": [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int],
    "vrcclCommGetLaunchShape": [ctypes.c_void_p, _c_int_p, _c_int_p, _c_int_p],
    "vrcclCommLoadTuning": [ctypes.c_void_p, ctypes.c_char_p, _c_int_p],
    "vrcclShardRange": [ctypes.c_size_t, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t),
                        ctypes.POINTER(ctypes.c_size_t)],
    "vrcclAllReduceNoAlloc": [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t,
                              ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p],
}
for _name, _args in _sig.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_int
_lib.vrcclGetErrorString.argtypes = [ctypes.c_int]
_lib.vrcclGetErrorString.restype = ctypes.c_char_p


class VrcclError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        self.name = RESULTS[code] if 0 <= code < len(RESULTS) else str(code)
        super().__init__(f"{where}: {self.name} ({vrcclGetErrorString(code)})")


def _check(code: int, where: str) -> None:
    if code != 0:
        raise VrcclError(code, where)


def _ptr(x) -> int:
    if isinstance(x, torch.Tensor):
        return x.data_ptr()
    return int(x)


def _stream(s) -> int | None:
    if s is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, torch.cuda.Stream):
        return s.cuda_stream
    return int(s)


def _enum(table: dict, v, what: str) -> int:
    if isinstance(v, int):
        return v
    if isinstance(v, torch.dtype) and table is DTYPES:
        v = _TORCH_DTYPES[v]
    try:
        return table[v]
    except KeyError:
        raise ValueError(f"unknown {what} {v!r}") from None


def vrcclGetErrorString(code: int) -> str:
    return _lib.vrcclGetErrorString(code).decode()


def vrcclCommInit(nranks: int, nchannels: int) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check(_lib.vrcclCommInit(ctypes.byref(h), nranks, nchannels), "vrcclCommInit")
    return h


def vrcclAllReduce(sendbufs, recvbufs, count: int, dtype, op, algo="ring", proto="simple", comm=None,
                   stream=None) -> None:
    n = len(sendbufs)
    S = (ctypes.c_void_p * n)(*[_ptr(b) for b in sendbufs])
    R = (ctypes.c_void_p * len(recvbufs))(*[_ptr(b) for b in recvbufs])
    _check(_lib.vrcclAllReduce(S, R, count, _enum(DTYPES, dtype, "dtype"), _enum(OPS, op, "op"),
                               _enum(ALGOS, algo, "algo"), _enum(PROTOS, proto, "proto"), comm,
                               _stream(stream)), "vrcclAllReduce")


def vrcclReduceScatter(sendbufs, recvbufs, recvcount: int, dtype, op, proto="simple", comm=None,
                       stream=None) -> None:
    S = (ctypes.c_void_p * len(sendbufs))(*[_ptr(b) for b in sendbufs])
    R = (ctypes.c_void_p * len(recvbufs))(*[_ptr(b) for b in recvbufs])
    _check(_lib.vrcclReduceScatter(S, R, recvcount, _enum(DTYPES, dtype, "dtype"), _enum(OPS, op, "op"),
                                   _enum(PROTOS, proto, "proto"), comm, _stream(stream)), "vrcclReduceScatter")


def vrcclAllGather(sendbufs, recvbufs, sendcount: int, dtype, proto="simple", comm=None, stream=None) -> None:
    S = (ctypes.c_void_p * len(sendbufs))(*[_ptr(b) for b in sendbufs])
    R = (ctypes.c_void_p * len(recvbufs))(*[_ptr(b) for b in recvbufs])
    _check(_lib.vrcclAllGather(S, R, sendcount, _enum(DTYPES, dtype, "dtype"), _enum(PROTOS, proto, "proto"), comm,
                               _stream(stream)), "vrcclAllGather")


def vrcclAllReduceNoAlloc(sendbufs, recvbufs, count: int, nranks: int, dtype, op, stream=None) -> None:
    """The allocation-free ring/Simple AllReduce (see include/vrccl.h)."""
    S = (ctypes.c_void_p * len(sendbufs))(*[_ptr(b) for b in sendbufs])
    R = (ctypes.c_void_p * len(recvbufs))(*[_ptr(b) for b in recvbufs])
    _check(_lib.vrcclAllReduceNoAlloc(S, R, count, nranks, _enum(DTYPES, dtype, "dtype"), _enum(OPS, op, "op"),
                                      _stream(stream)), "vrcclAllReduceNoAlloc")


def vrcclShardRange(count: int, dtype, nshards: int, shard: int) -> tuple[int, int]:
    """(offset, length) of GPU `shard`'s part of a problem split over
    `nshards` GPUs by element range (host only; see include/vrccl.h)."""
    off, ln = ctypes.c_size_t(), ctypes.c_size_t()
    _check(_lib.vrcclShardRange(count, _enum(DTYPES, dtype, "dtype"), nshards, shard, ctypes.byref(off),
                                ctypes.byref(ln)), "vrcclShardRange")
    return off.value, ln.value


def vrcclGroupStart() -> None:
    _check(_lib.vrcclGroupStart(), "vrcclGroupStart")


def vrcclGroupEnd() -> None:
    _check(_lib.vrcclGroupEnd(), "vrcclGroupEnd")


def vrcclCommGetGroupSchedule(comm, index: int) -> dict:
    a, p, c, l = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    k = ctypes.c_size_t()
    _check(_lib.vrcclCommGetGroupSchedule(comm, index, ctypes.byref(a), ctypes.byref(p), ctypes.byref(c),
                                          ctypes.byref(k), ctypes.byref(l)), "vrcclCommGetGroupSchedule")
    return {"algo": ALGO_NAMES[a.value], "proto": PROTO_NAMES[p.value], "nchannels": c.value,
            "chunk_elems": k.value, "launch": l.value}


PARSE_FUNCS = ["broadcast", "reduce", "allgather", "reducescatter", "allreduce"]
PARSE_NAMES = {0: ["tree", "ring", "collnetdirect", "collnetchain", "nvls", "nvlstree", "pat"],
               1: ["ll", "ll128", "simple"]}


class _ModelGraph(ctypes.Structure):
    _fields_ = [("nranks", ctypes.c_int), ("nnodes", ctypes.c_int), ("nchannels", ctypes.c_int),
                ("bwIntra", ctypes.c_float), ("bwInter", ctypes.c_float), ("latencyInter", ctypes.c_float),
                ("hwIntra", ctypes.c_int), ("arch", ctypes.c_int)]


def vrcclParseList(spec, kind: str) -> dict:
    """{function: sorted list of allowed names}; kind "algo" or "proto"."""
    k = {"algo": 0, "proto": 1}[kind]
    masks = (ctypes.c_uint * 5)()
    _check(_lib.vrcclParseList(None if spec is None else spec.encode(), k, masks), "vrcclParseList")
    return {f: [nm for i, nm in enumerate(PARSE_NAMES[k]) if masks[j] >> i & 1] for j, f in enumerate(PARSE_FUNCS)}


def vrcclModelPredict(nranks: int, nnodes: int, nchannels: int, bw_intra: float, algo, proto, nbytes: int,
                      num_pipe_ops: int = 1, bw_inter: float = 0.0, latency_inter: float = 0.0, hw_intra: str = "nvlink",
                      arch: str = "hopper") -> dict:
    g = _ModelGraph(nranks, nnodes, nchannels, bw_intra, bw_inter, latency_inter,
                    {"nvlink": 0, "pci": 1}[hw_intra], {"volta": 0, "ampere": 1, "hopper": 2, "blackwell": 3}[arch])
    lat, bw, t = ctypes.c_float(), ctypes.c_float(), ctypes.c_float()
    _check(_lib.vrcclModelPredict(ctypes.byref(g), _enum(ALGOS, algo, "algo"), _enum(PROTOS, proto, "proto"), nbytes,
                                  num_pipe_ops, ctypes.byref(lat), ctypes.byref(bw), ctypes.byref(t)),
           "vrcclModelPredict")
    return {"lat_us": lat.value, "algbw_gbs": bw.value, "time_us": t.value}


def vrcclCommSetDirect(comm, enable: bool) -> None:
    _check(_lib.vrcclCommSetDirect(comm, 1 if enable else 0), "vrcclCommSetDirect")


def vrcclCommSetSchedule(comm, nchannels: int = 0, chunkBytes: int = 0) -> None:
    _check(_lib.vrcclCommSetSchedule(comm, nchannels, chunkBytes), "vrcclCommSetSchedule")


def vrcclCommGetLastSchedule(comm) -> dict:
    a, p, c = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    k = ctypes.c_size_t()
    _check(_lib.vrcclCommGetLastSchedule(comm, ctypes.byref(a), ctypes.byref(p), ctypes.byref(c),
                                         ctypes.byref(k)), "vrcclCommGetLastSchedule")
    return {"algo": ALGO_NAMES[a.value], "proto": PROTO_NAMES[p.value], "nchannels": c.value,
            "chunk_elems": k.value}


def vrcclCommGetLaunchShape(comm) -> dict:
    b, t, s = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(_lib.vrcclCommGetLaunchShape(comm, ctypes.byref(b), ctypes.byref(t), ctypes.byref(s)),
           "vrcclCommGetLaunchShape")
    return {"blocks": b.value, "threads": t.value, "slice_elems": s.value}


def vrcclCommGetAsyncError(comm) -> int:
    e = ctypes.c_int()
    _check(_lib.vrcclCommGetAsyncError(comm, ctypes.byref(e)), "vrcclCommGetAsyncError")
    return e.value


def vrcclCommGetErrorInfo(comm) -> dict:
    r, c = ctypes.c_int(), ctypes.c_int()
    s = ctypes.c_uint64()
    _check(_lib.vrcclCommGetErrorInfo(comm, ctypes.byref(r), ctypes.byref(c), ctypes.byref(s)),
           "vrcclCommGetErrorInfo")
    return {"rank": r.value, "channel": c.value, "step": s.value}


def vrcclCommSetTimeout(comm, timeoutMs: int) -> None:
    _check(_lib.vrcclCommSetTimeout(comm, timeoutMs), "vrcclCommSetTimeout")


def vrcclCommAbort(comm) -> None:
    _check(_lib.vrcclCommAbort(comm), "vrcclCommAbort")


def vrcclCommDestroy(comm) -> None:
    _check(_lib.vrcclCommDestroy(comm), "vrcclCommDestroy")


def vrcclCommCount(comm) -> int:
    n = ctypes.c_int()
    _check(_lib.vrcclCommCount(comm, ctypes.byref(n)), "vrcclCommCount")
    return n.value


def vrcclCommInjectFault(comm, rank: int, channel: int = 0, afterSteps: int = 0) -> None:
    _check(_lib.vrcclCommInjectFault(comm, rank, channel, afterSteps), "vrcclCommInjectFault")


def vrcclCommLoadTuning(comm, path: str) -> int:
    k = ctypes.c_int()
    _check(_lib.vrcclCommLoadTuning(comm, path.encode(), ctypes.byref(k)), "vrcclCommLoadTuning")
    return k.value


def raw_call(name: str, *args) -> int:
    """Call a C entry point by name and return its raw result code (tests)."""
    return getattr(_lib, name)(*args)


LIB = _lib
LIB_PATH = _LIB_PATH
