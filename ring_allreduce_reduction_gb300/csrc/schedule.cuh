// Slice sequences of one agent. Every role of an agent (and the agent on
// the other end of each FIFO) walks the same deterministic sequence, so no
// schedule state is shared between threads.
#pragma once

#include "engine.cuh"

namespace vrccl {

struct SliceDesc {
  long long pos;  // element offset within the channel
  int nelem;
  int flags;
};

// Ring: per loop of n chunks, runRing's 2n-1 primitives ("NCCL architecture:
// topology, channels, algorithms and protocols", §9.4); primitive p of rank
// r handles chunk
//   p = 0          send               r-1
//   p = 1..n-2     recvReduceSend     r-1-p
//   p = n-1        recvReduceCopySend r        (post-op, final)
//   p = n..2n-3    recvCopySend       r-(p-n+1)
//   p = 2n-2       recv               r+1            (all mod n)
// i.e. chunkId = (ringIndex + n - 1 - chunkStage) mod n of
// RingARAlgorithm::getNextSendAddr ("NCCL Source Code Deep Dive", §2.3).
// A loop covers n*K elements; a shorter remainder uses chunks of
// alignUp(ceil(rem/n), 16 bytes). A chunk is cut into slices of at most
// `slice` elements, one FIFO step each. With n == 1 the sequence is a copy.
struct RingIter {
  int n, r;
  long long chCount, K, A, slice;
  long long off, rem, k, s, cHi;
  int p, flags;
  bool started;

  __device__ __forceinline__ void init(int n_, int r_, long long chCount_, long long K_, long long A_,
                                       long long slice_) {
    n = n_;
    r = r_;
    chCount = chCount_;
    K = K_;
    A = A_;
    slice = slice_;
    started = false;
    s = cHi = 0;
    p = 0;
    off = 0;
    flags = 0;
  }
  __device__ __forceinline__ void setChunk() {
    int c;
    if (p == 0) {
      c = (r - 1 + n) % n;
      flags = F_IN | F_SEND;
    } else if (p <= n - 2) {
      c = ((r - 1 - p) % n + n) % n;
      flags = F_IN | F_RECV | F_SEND;
    } else if (p == n - 1) {
      c = r;
      flags = F_IN | F_RECV | F_POST | F_OUT | F_SEND;
    } else if (p <= 2 * n - 3) {
      c = ((r - (p - n + 1)) % n + n) % n;
      flags = F_RECV | F_OUT | F_SEND;
    } else {
      c = (r + 1) % n;
      flags = F_RECV | F_OUT;
    }
    const long long cLo = min(rem, (long long)c * k);
    cHi = off + min(rem, (long long)(c + 1) * k);
    s = off + cLo;
  }
  __device__ __forceinline__ void setLoop() {
    rem = chCount - off;
    const long long loop = (long long)n * K;
    k = rem >= loop ? K : ((rem + n - 1) / n + A - 1) / A * A;
  }
  __device__ __forceinline__ bool next(SliceDesc& d) {
    if (n == 1) {  // single rank: the local copy
      if (!started) {
        started = true;
        s = 0;
      }
      if (s >= chCount) return false;
      d.pos = s;
      d.nelem = (int)min(slice, chCount - s);
      d.flags = F_IN | F_OUT | F_POST;
      s += slice;
      return true;
    }
    while (true) {
      if (s < cHi) {
        d.pos = s;
        d.nelem = (int)min(slice, cHi - s);
        d.flags = flags;
        s += slice;
        return true;
      }
      if (!started) {
        started = true;
        if (chCount <= 0) return false;
        off = 0;
        p = 0;
        setLoop();
      } else if (++p == 2 * n - 1) {
        off += (long long)n * K;
        if (off >= chCount) return false;
        p = 0;
        setLoop();
      }
      setChunk();
    }
  }
};

// Tree: the channel's range in slices, every slice with the role's flags.
struct TreeIter {
  long long chCount, slice, s;
  int flags;
  __device__ __forceinline__ void init(long long chCount_, long long slice_, int flags_) {
    chCount = chCount_;
    slice = slice_;
    flags = flags_;
    s = 0;
  }
  __device__ __forceinline__ bool next(SliceDesc& d) {
    if (s >= chCount) return false;
    d.pos = s;
    d.nelem = (int)min(slice, chCount - s);
    d.flags = flags;
    s += slice;
    return true;
  }
};

}  // namespace vrccl
