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
// Positions are element offsets from the start of the rank's buffers; the
// channel's range starts at `lo`.
//
// direct (Simple): the directRecvCopyDirectSend form of the same primitives
// for ranks that can address each other's buffers: the all-gather moves
// through the recv buffers. The step that finishes chunk r writes it to
// this rank's recv buffer and into the next rank's; an all-gather step
// takes the chunk from this rank's recv buffer (where the predecessor wrote
// it) and writes it into the next rank's. The last step has nothing left
// to do: its slices are passed over and only counted (dskip), so they take
// no stage of the pipeline (measured on the 256 MiB fp32 ring, n = 8:
// 1.484 -> 1.394 ms for the direct form).
struct RingIter {
  int n, r;
  long long lo, chCount, K, A, slice;
  long long off, rem, k, s, cHi;
  long long dskip;  // direct: slices of the last steps passed over so far
  int p, flags;
  bool started, direct;

  __device__ __forceinline__ void init(int n_, int r_, long long lo_, long long chCount_, long long K_, long long A_,
                                       long long slice_, bool direct_ = false) {
    n = n_;
    r = r_;
    direct = direct_;
    lo = lo_;
    chCount = chCount_;
    K = K_;
    A = A_;
    slice = slice_;
    started = false;
    s = cHi = 0;
    dskip = 0;
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
      flags = F_IN | F_RECV | F_POST | F_OUT | (direct ? F_DSEND : F_SEND);
    } else if (p <= 2 * n - 3) {
      c = ((r - (p - n + 1)) % n + n) % n;
      flags = direct ? (F_DRECV | F_DSEND) : (F_RECV | F_OUT | F_SEND);
    } else {
      c = (r + 1) % n;
      flags = F_RECV | F_OUT;
    }
    const long long cLo = min(rem, (long long)c * k);
    cHi = off + min(rem, (long long)(c + 1) * k);
    s = off + cLo;
    if (direct && p == 2 * n - 2) {  // the chunk is already in place
      if (cHi > s) dskip += (cHi - s + slice - 1) / slice;
      s = cHi;
    }
  }
  // direct: slices passed over so far, and where a slice sits in the next
  // rank's recv buffer relative to its position here (the same place)
  __device__ __forceinline__ long long skippedDirect() const { return dskip; }
  __device__ __forceinline__ long long nextShift() const { return 0; }
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
      d.inPos = d.outPos = lo + s;
      d.nelem = (int)min(slice, chCount - s);
      d.flags = F_IN | F_OUT | F_POST;
      s += slice;
      return true;
    }
    while (true) {
      if (s < cHi) {
        d.inPos = d.outPos = lo + s;
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

// The two phases run alone ("NCCL Source Code Deep Dive", §2.3 walks the
// AllReduce as a reduce-scatter phase and an all-gather phase of n-1 steps
// each) use the ring's chunk order on blocks instead of loop chunks. The
// channel range [lo, lo + chCount) is a range within a block of `blk`
// elements; a loop takes K elements of every block, and chunk c of a loop
// lives in block c:
//   ReduceScatter  p = 0 send c = r-1; p = 1..n-2 recvReduceSend c = r-1-p;
//                  p = n-1 recvReduceCopy (post-op) c = r -> recv buffer
//   AllGather      p = 0 copySend c = r (own send buffer -> block r);
//                  p = 1..n-2 recvCopySend c = r-p; p = n-1 recv c = r+1
// (n > 1; one rank runs the AllReduce copy instead).
// direct (AllGather, Simple): as the ring's direct all-gather, each block
// moves through the recv buffers: step 0 writes the own block to this
// rank's recv buffer and into the next rank's, each later step forwards
// the block the predecessor wrote here into the next rank's recv buffer,
// and the last step's slices are passed over and only counted (dskip).
struct PhaseIter {
  int n, r;
  bool gather, direct;
  long long lo, chCount, blk, K, slice;
  long long off, len, inBase, outBase, s;
  long long dskip;  // direct: slices of the last steps passed over so far
  int p, flags;
  bool started;

  __device__ __forceinline__ void init(int n_, int r_, bool gather_, long long lo_, long long chCount_,
                                       long long blk_, long long K_, long long slice_, bool direct_ = false) {
    n = n_;
    r = r_;
    gather = gather_;
    direct = direct_ && gather_;
    dskip = 0;
    lo = lo_;
    chCount = chCount_;
    blk = blk_;
    K = K_;
    slice = slice_;
    started = false;
    off = len = inBase = outBase = s = 0;
    p = 0;
    flags = 0;
  }
  __device__ __forceinline__ long long skippedDirect() const { return dskip; }
  __device__ __forceinline__ long long nextShift() const { return 0; }
  __device__ __forceinline__ void setChunk() {
    int c;
    if (!gather) {
      c = p == n - 1 ? r : ((r - 1 - p) % n + n) % n;
      flags = p == 0 ? (F_IN | F_SEND) : p < n - 1 ? (F_IN | F_RECV | F_SEND) : (F_IN | F_RECV | F_POST | F_OUT);
      inBase = (long long)c * blk + lo + off;
      outBase = lo + off;
    } else {
      c = ((r - p) % n + n) % n;
      if (direct)
        flags = p == 0 ? (F_IN | F_OUT | F_DSEND) : (F_DRECV | F_DSEND);
      else
        flags = p == 0 ? (F_IN | F_OUT | F_SEND) : p < n - 1 ? (F_RECV | F_OUT | F_SEND) : (F_RECV | F_OUT);
      inBase = lo + off;
      outBase = (long long)c * blk + lo + off;
    }
    s = 0;
    if (direct && p == n - 1) {  // the block is already in place
      if (len > 0) dskip += (len + slice - 1) / slice;
      s = len;
    }
  }
  __device__ __forceinline__ bool next(SliceDesc& d) {
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
      } else if (++p == n) {
        off += K;
        if (off >= chCount) return false;
        p = 0;
      }
      len = min(chCount - off, K);
      setChunk();
    }
  }
};

// Tree: the channel's range in slices, every slice with the role's flags.
struct TreeIter {
  long long lo, chCount, slice, s;
  int flags;
  __device__ __forceinline__ long long skippedDirect() const { return 0; }
  __device__ __forceinline__ long long nextShift() const { return 0; }
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
