"""The C-ABI library: builds, loads, exports every declared entry point, and
rejects bad arguments on the host before touching the GPU. No GPU needed."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vrccl.h")


@pytest.fixture(scope="module")
def lib():
    from ring_allreduce_reduction_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:vrcclResult_t|const char\*)\s+(vrccl\w+)\s*\(", txt, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared()
    for must in ("vrcclCommInit", "vrcclAllReduce", "vrcclCommGetLastSchedule", "vrcclCommGetAsyncError",
                 "vrcclCommAbort", "vrcclCommDestroy", "vrcclGetErrorString"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared():
        assert hasattr(lib, name), f"{name} declared in include/vrccl.h but not exported"


def test_error_strings(lib):
    lib.vrcclGetErrorString.restype = ctypes.c_char_p
    assert lib.vrcclGetErrorString(0) == b"no error"
    assert lib.vrcclGetErrorString(5) == b"device wait timed out"
    assert lib.vrcclGetErrorString(99) == b"unknown result code"


def test_host_side_argument_checks(lib):
    h = ctypes.c_void_p()
    assert lib.vrcclCommInit(None, 4, 1) == 1
    assert lib.vrcclCommInit(ctypes.byref(h), 0, 1) == 1
    assert lib.vrcclCommInit(ctypes.byref(h), 129, 1) == 1
    assert lib.vrcclCommInit(ctypes.byref(h), 4, 0) == 1
    assert lib.vrcclCommInit(ctypes.byref(h), 4, 65) == 1
    assert lib.vrcclAllReduce(None, None, 1, 0, 0, 0, 0, None, None) == 1
    bogus = ctypes.create_string_buffer(4096)  # not a communicator: the magic check rejects it
    assert lib.vrcclAllReduce(None, None, 1, 0, 0, 0, 0, bogus, None) == 1
    assert lib.vrcclReduceScatter(None, None, 4, 0, 0, 0, None, None) == 1
    assert lib.vrcclAllGather(None, None, 4, 0, 0, None, None) == 1
    assert lib.vrcclReduceScatter(None, None, 4, 0, 0, 0, bogus, None) == 1
    assert lib.vrcclAllGather(None, None, 4, 0, 0, bogus, None) == 1
    assert lib.vrcclCommDestroy(None) == 0
    assert lib.vrcclCommDestroy(bogus) == 1
    assert lib.vrcclCommAbort(bogus) == 1
    assert lib.vrcclCommCount(bogus, None) == 1


def test_binding_names_match_the_c_names():
    torch = pytest.importorskip("torch")  # noqa: F841
    from ring_allreduce_reduction_gb300 import build
    build.build()
    from ring_allreduce_reduction_gb300 import vrccl
    for name in declared():
        assert hasattr(vrccl, name), f"binding lacks {name}"


def test_tuning_table_writer_format(tmp_path):
    """tune.write_table emits the line format the library parses:
    nranks algo proto channels log2bytes sliceBytes microseconds
    elementBytes; --append adds rows under the first header."""
    pytest.importorskip("torch")
    from ring_allreduce_reduction_gb300.tune import read_table, write_table
    recs = [{"nranks": 8, "dtype": "bfloat16", "algo": "tree", "proto": "ll128", "channels": 3, "bytes": 1 << 20,
             "slice_bytes": 30720, "us": 12.5}]
    p = tmp_path / "t.txt"
    write_table(recs, str(p), header="x")
    write_table([dict(recs[0], dtype="float32", us=7.25)], str(p), header="y", append=True)
    rows = [ln.split() for ln in p.read_text().splitlines() if not ln.startswith("#")]
    assert rows == [["8", "1", "2", "3", "20", "30720", "12.500", "2"], ["8", "1", "2", "3", "20", "30720", "7.250", "4"]]
    assert [r["esize"] for r in read_table(str(p))] == [2, 4]


def test_shipped_tuning_tables_parse():
    d = os.path.join(ROOT, "ring_allreduce_reduction_gb300", "tuning")
    tables = sorted(f for f in os.listdir(d) if re.fullmatch(r"gb300_n\d+\.txt", f))
    assert "gb300_n8.txt" in tables
    for f in tables:
        nr = int(re.findall(r"\d+", f)[1])
        rows = [ln.split() for ln in open(os.path.join(d, f)) if ln.strip() and not ln.startswith("#")]
        assert len(rows) > 50, f
        for r in rows:
            assert len(r) in (7, 8), (f, r)
            n, algo, proto, ch, lg, sl = map(int, r[:6])
            assert n == nr and algo in (0, 1) and proto in (0, 1, 2) and 1 <= ch <= 64 and 0 <= lg < 40 and sl > 0
            assert float(r[6]) > 0
            assert len(r) == 7 or int(r[7]) in (1, 2, 4, 8)


def test_binding_constants_match_the_header():
    """The Python binding's copies of the header's macros and enums agree."""
    pytest.importorskip("torch")
    from ring_allreduce_reduction_gb300 import build
    build.build()
    from ring_allreduce_reduction_gb300 import vrccl
    txt = open(HEADER).read()
    macro = {m: int(v) for m, v in re.findall(r"#define\s+(VRCCL_\w+)\s+(\d+)", txt)}
    assert vrccl.MAX_RANKS == macro["VRCCL_MAX_RANKS"]
    assert vrccl.MAX_CHANNELS == macro["VRCCL_MAX_CHANNELS"]
    assert vrccl.STEPS == macro["VRCCL_STEPS"]

    def enum_body(first):
        body = re.search(r"typedef enum\s*\{([^}]*" + first + r"[^}]*)\}", txt).group(1)
        body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
        names, val = [], -1
        for item in [x.strip() for x in body.split(",") if x.strip()]:
            name, _, rhs = item.partition("=")
            val = int(rhs) if rhs.strip() else val + 1
            names.append((name.strip(), val))
        return dict(names)

    dt = enum_body("vrcclInt32")
    assert {k: dt["vrccl" + {"int32": "Int32", "float32": "Float32", "bfloat16": "Bfloat16",
                             "float16": "Float16", "int8": "Int8", "uint8": "Uint8", "int64": "Int64",
                             "float64": "Float64"}[k]] for k in vrccl.DTYPES} == vrccl.DTYPES
    assert len(vrccl.DTYPES) == dt["vrcclNumTypes"]
    from ring_allreduce_reduction_gb300 import workloads
    assert set(workloads.DTYPES) == set(vrccl.DTYPES) and workloads.ELEM_SIZE == vrccl.ELEM_SIZE
    ops = enum_body("vrcclSum")
    assert {k: ops["vrccl" + k.capitalize()] for k in vrccl.OPS} == vrccl.OPS
    res = enum_body("vrcclSuccess")
    assert [res[name] for name in vrccl.RESULTS] == list(range(len(vrccl.RESULTS)))


def test_group_depth_on_the_host(lib):
    """Group bookkeeping needs no GPU: an unmatched end is refused, nested
    empty groups succeed."""
    assert lib.vrcclGroupEnd() == 2
    assert lib.vrcclGroupStart() == 0
    assert lib.vrcclGroupStart() == 0
    assert lib.vrcclGroupEnd() == 0
    assert lib.vrcclGroupEnd() == 0
    assert lib.vrcclGroupEnd() == 2
    bogus = ctypes.create_string_buffer(4096)
    assert lib.vrcclCommGetGroupSchedule(bogus, 0, None, None, None, None, None) == 1


def test_no_alloc_host_checks(lib):
    """vrcclAllReduceNoAlloc refuses bad arguments before touching a GPU:
    too many ranks, misaligned pointers, and buffers that overlap other
    than in place (the pointers below are never dereferenced)."""
    P = ctypes.c_void_p
    base = 1 << 40

    def call(send, recv, count, n, dtype=1, op=0):
        s = (P * n)(*send)
        r = (P * n)(*recv)
        return lib.vrcclAllReduceNoAlloc(s, r, ctypes.c_size_t(count), n, dtype, op, None)

    n, count = 4, 1024  # 4 KiB per rank
    send = [base + i * 8192 for i in range(n)]
    assert call([base] * 33, [base + 8192] * 33, count, 33) == 2                      # beyond the scratch
    assert call([s + 8 for s in send], send, count, n) == 1                          # misaligned
    assert call(send, [s + 4096 - 16 for s in send], count, n) == 1                  # recv overlaps a send buffer
    assert call(send, [base + 65536] * n, count, n) == 1                             # recv buffers overlap each other
    assert call(send, send, 0, n) == 0                                               # count 0: nothing to do
    assert call([], [], count, 0) == 1                                               # no ranks
    assert call(send, send, count, n, dtype=8) == 1                                  # bad type


def test_table_choice_mirrors_the_rule():
    """tune.table_choice, the host mirror of the library's rule: rows of the
    call's element size, else rows for any size, else the nearest measured
    element size (ties to the larger); then the nearest power-of-two size
    and the fastest row there."""
    pytest.importorskip("torch")
    from ring_allreduce_reduction_gb300.tune import table_choice
    def row(algo, proto, ch, lg, us, es):
        return {"nranks": 5, "algo": algo, "proto": proto, "channels": ch, "bytes": 1 << lg, "slice_bytes": 16384,
                "us": us, "esize": es}
    t = [row("tree", "ll128", 3, 18, 5.0, 2), row("ring", "simple", 2, 18, 9.0, 2),
         row("ring", "simple", 2, 18, 4.0, 4), row("tree", "ll128", 3, 18, 6.0, 4),
         row("ring", "ll", 1, 10, 1.0, 4)]
    pick = lambda **kw: (lambda r: (r["algo"], r["proto"], r["channels"]))(table_choice(t, **kw))
    assert pick(nranks=5, nbytes=1 << 18, esize=2) == ("tree", "ll128", 3)
    assert pick(nranks=5, nbytes=1 << 18, esize=4) == ("ring", "simple", 2)
    assert pick(nranks=5, nbytes=1 << 18, esize=1) == ("tree", "ll128", 3)      # nearest: 2-byte rows
    assert pick(nranks=5, nbytes=1 << 18, esize=8) == ("ring", "simple", 2)     # nearest: 4-byte rows
    assert pick(nranks=5, nbytes=300 << 10, esize=4) == ("ring", "simple", 2)   # nearest size 2^18
    assert pick(nranks=5, nbytes=1000, esize=4) == ("ring", "ll", 1)
    assert pick(nranks=5, nbytes=1 << 18, esize=4, protos=("ll128",)) == ("tree", "ll128", 3)
    assert table_choice(t, nranks=6, nbytes=1 << 18, esize=4) is None
