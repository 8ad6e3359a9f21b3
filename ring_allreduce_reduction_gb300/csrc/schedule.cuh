// Slice sequences of one agent. Every role of an agent (and the agent on
// the other end of each FIFO) walks the same deterministic sequence, so no
// schedule state is shared between threads.
#pragma once

#include "engine.cuh"

namespace vrccl {

struct SliceDesc {
  long long inPos;   // element offset of the slice in this agent's send buffer
  long long outPos;  // element offset of the slice in this agent's recv buffer
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
//
// The two phases run alone ("NCCL Source Code Deep Dive", §2.3 walks the
// AllReduce as a reduce-scatter phase and an all-gather phase of n-1 steps
// each) use the same chunk order on blocks instead of loop chunks. The
// channel range [lo, lo + chCount) is then a range within a block of `blk`
// elements, a loop takes K elements of every block, and chunk c of a loop
// lives in block c:
//   ReduceScatter  p = 0 send c = r-1; p = 1..n-2 recvReduceSend c = r-1-p;
//                  p = n-1 recvReduceCopy (post-op) c = r -> recv buffer
//   AllGather      p = 0 copySend c = r (own send buffer -> block r);
//                  p = 1..n-2 recvCopySend c = r-p; p = n-1 recv c = r+1
struct RingIter {
  int n, r, coll;
  long long chCount, K, A, slice, lo, blk;
  long long off, rem, k;                // loop offset and remainder; chunk size of the loop
  long long inBase, outBase, len, s;    // current chunk: slices [s, len) from the two bases
  int p, nprim, flags;
  bool started;

  __device__ __forceinline__ void init(int n_, int r_, int coll_, long long lo_, long long chCount_, long long blk_,
                                       long long K_, long long A_, long long slice_) {
    n = n_;
    r = r_;
    coll = coll_;
    lo = lo_;
    chCount = chCount_;
    blk = blk_;
    K = K_;
    A = A_;
    slice = slice_;
    nprim = coll == kAllReduce ? 2 * n - 1 : n;
    started = false;
    s = len = 0;
    inBase = outBase = 0;
    p = 0;
    off = 0;
    flags = 0;
  }
  __device__ __forceinline__ static int mod(int x, int m) { return ((x % m) + m) % m; }
  __device__ __forceinline__ void setChunk() {
    int c;
    if (coll == kAllReduce) {
      if (p == 0) {
        c = mod(r - 1, n);
        flags = F_IN | F_SEND;
      } else if (p <= n - 2) {
        c = mod(r - 1 - p, n);
        flags = F_IN | F_RECV | F_SEND;
      } else if (p == n - 1) {
        c = r;
        flags = F_IN | F_RECV | F_POST | F_OUT | F_SEND;
      } else if (p <= 2 * n - 3) {
        c = mod(r - (p - n + 1), n);
        flags = F_RECV | F_OUT | F_SEND;
      } else {
        c = mod(r + 1, n);
        flags = F_RECV | F_OUT;
      }
      const long long cLo = min(rem, (long long)c * k);
      len = min(rem, (long long)(c + 1) * k) - cLo;
      inBase = outBase = lo + off + cLo;
    } else if (coll == kReduceScatter) {
      c = p == n - 1 ? r : mod(r - 1 - p, n);
      flags = p == 0 ? (F_IN | F_SEND) : p < n - 1 ? (F_IN | F_RECV | F_SEND) : (F_IN | F_RECV | F_POST | F_OUT);
      len = k;
      inBase = (long long)c * blk + lo + off;
      outBase = lo + off;
    } else {
      c = mod(r - p, n);
      flags = p == 0 ? (F_IN | F_OUT | F_SEND) : p < n - 1 ? (F_RECV | F_OUT | F_SEND) : (F_RECV | F_OUT);
      len = k;
      inBase = lo + off;
      outBase = (long long)c * blk + lo + off;
    }
    s = 0;
  }
  __device__ __forceinline__ void setLoop() {
    rem = chCount - off;
    if (coll == kAllReduce) {
      const long long loop = (long long)n * K;
      k = rem >= loop ? K : ((rem + n - 1) / n + A - 1) / A * A;
    } else {
      k = min(rem, K);
    }
  }
  __device__ __forceinline__ bool next(SliceDesc& d) {
    if (n == 1) {  // single rank: the local copy
      if (!started) {
        started = true;
        s = 0;
      }
      if (s >= chCount) return false;
      d.inPos = d.outPos = lo + s;
      d.nelem = (int)min(slice, chCount - s);
      d.flags = F_IN | F_OUT | F_POST;
      s += slice;
      return true;
    }
    while (true) {
      if (s < len) {
        d.inPos = inBase + s;
        d.outPos = outBase + s;
        d.nelem = (int)min(slice, len - s);
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
      } else if (++p == nprim) {
        off += coll == kAllReduce ? (long long)n * K : K;
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
  long long lo, chCount, slice, s;
  int flags;
  __device__ __forceinline__ void init(long long lo_, long long chCount_, long long slice_, int flags_) {
    lo = lo_;
    chCount = chCount_;
    slice = slice_;
    flags = flags_;
    s = 0;
  }
  __device__ __forceinline__ bool next(SliceDesc& d) {
    if (s >= chCount) return false;
    d.inPos = d.outPos = lo + s;
    d.nelem = (int)min(slice, chCount - s);
    d.flags = flags;
    s += slice;
    return true;
  }
};

}  // namespace vrccl
