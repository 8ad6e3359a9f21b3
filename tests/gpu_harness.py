"""Device-buffer plumbing for the GPU tests (torch allocates, libvrccl computes).

Each virtual rank's buffer is a 256-byte-aligned row of one uint8 tensor,
with canary bytes before and after it, so any out-of-bounds write by a
kernel shows up as a changed canary.
"""
from __future__ import annotations

import numpy as np
import torch

from ring_allreduce_reduction_gb300.workloads import ELEM_SIZE, STORAGE

GUARD = 256
CANARY = 0xA5


def _row_bytes(count: int, dtype: str) -> int:
    return (count * ELEM_SIZE[dtype] + 2 * GUARD + 255) // 256 * 256


class Buffers:
    """n send rows and n recv rows on cuda:0, each [GUARD | data | GUARD...]."""

    def __init__(self, x: np.ndarray, dtype: str, inplace: bool = False, device: str = "cuda:0"):
        self.n, self.count = x.shape
        self.dtype = dtype
        self.nbytes = self.count * ELEM_SIZE[dtype]
        self.row = _row_bytes(self.count, dtype)
        host = np.full((self.n, self.row), CANARY, dtype=np.uint8)
        host[:, GUARD:GUARD + self.nbytes] = np.ascontiguousarray(x).view(np.uint8).reshape(self.n, -1)
        self.send = torch.from_numpy(host).to(device)
        self.inplace = inplace
        self.recv = self.send if inplace else torch.full((self.n, self.row), CANARY, dtype=torch.uint8,
                                                           device=device)

    def send_ptrs(self):
        base = self.send.data_ptr()
        return [base + r * self.row + GUARD for r in range(self.n)]

    def recv_ptrs(self):
        base = self.recv.data_ptr()
        return [base + r * self.row + GUARD for r in range(self.n)]

    def result(self) -> np.ndarray:
        torch.cuda.synchronize()
        h = self.recv.cpu().numpy()
        return np.ascontiguousarray(h[:, GUARD:GUARD + self.nbytes]).view(STORAGE[self.dtype]).reshape(
            self.n, self.count)

    def canaries_intact(self) -> bool:
        torch.cuda.synchronize()
        h = self.recv.cpu().numpy()
        ok = np.all(h[:, :GUARD] == CANARY) and np.all(h[:, GUARD + self.nbytes:] == CANARY)
        if not self.inplace:
            s = self.send.cpu().numpy()
            ok = ok and np.all(s[:, :GUARD] == CANARY) and np.all(s[:, GUARD + self.nbytes:] == CANARY)
        return bool(ok)


def run(v, comm, x: np.ndarray, dtype: str, op: str, algo: str, proto: str, inplace: bool = False):
    """One AllReduce through the C ABI; returns (result [n, count], schedule, buffers)."""
    b = Buffers(x, dtype, inplace=inplace)
    v.vrcclAllReduce(b.send_ptrs(), b.recv_ptrs(), b.count, dtype, op, algo, proto, comm)
    y = b.result()
    return y, v.vrcclCommGetLastSchedule(comm), b
