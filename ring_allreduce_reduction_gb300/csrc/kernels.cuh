// The two schedules, as kernels: one CTA per agent, all agents of a launch
// co-resident (cooperative launch), so every wait is on a running peer.
#pragma once

#include "simple_pipe.cuh"

namespace vrccl {

__device__ __forceinline__ unsigned long long alignUpU(unsigned long long x, unsigned long long a) {
  return (x + a - 1) / a * a;
}

// Channel ch owns elements [lo, hi): parts of alignUp(ceil(count/C), A)
// elements, one per channel, in channel order ("NCCL Source Code Deep Dive",
// §2.2, "Step 3: Data Splitting").
template <typename S>
__device__ __forceinline__ void channelRange(unsigned long long count, int C, int ch, unsigned long long& lo,
                                             unsigned long long& hi) {
  constexpr unsigned long long A = 16 / sizeof(S);
  const unsigned long long part = count ? alignUpU((count + C - 1) / C, A) : 0;
  lo = min(count, part * (unsigned long long)ch);
  hi = min(count, lo + part);
}

// ---------------------------------------------------------------------- ring
// Agent (rank r, channel ch) = block r + n * ch. Per loop of n chunks it
// runs runRing's 2n-1 primitives ("NCCL architecture ...", §9.4):
//   p = 0          send              chunk r-1
//   p = 1..n-2     recvReduceSend    chunk r-1-p
//   p = n-1        recvReduceCopySend (post-op) chunk r   -> final
//   p = n..2n-3    recvCopySend      chunk r-(p-n+1)
//   p = 2n-2       recv              chunk r+1            (all mod n)
// which is chunkId = (ringIndex + n - 1 - chunkStage) mod n of
// RingARAlgorithm::getNextSendAddr ("NCCL Source Code Deep Dive", §2.3).
// The loop covers n*K elements; a shorter remainder uses chunks of
// alignUp(ceil(rem/n), 16 bytes). A chunk moves as slices of at most
// sliceElems elements, one FIFO step each.
// One ring agent's slice sequence through its protocol.
template <int PROTO, int DT, int OP, bool DIRECT = false, class Args, class It>
__device__ __forceinline__ void ringAgent(const Args& a, Agent& ag, It& it, const char* in, char* out) {
  using S = typename Ty<DT>::S;
  constexpr long long E = sizeof(S);
  if constexpr (PROTO == kSimple) {
    simplePipeline<DT, OP, false, DIRECT>(a, ag, it, in, out);
  } else {
    llBegin();
    SliceDesc d;
    while (it.next(d))
      if (!runSlice<PROTO, DT, OP, false>(a, ag, in + d.inPos * E, out + d.outPos * E, d.nelem, d.flags)) return;
    ag.finish(a.comm);
  }
}

template <int PROTO, int DT, int OP>
__global__ void __launch_bounds__(maxAgentThreads(PROTO)) ringKernel(const __grid_constant__ KArgs a) {
  using S = typename Ty<DT>::S;
  constexpr long long E = sizeof(S);
  const int n = a.nranks;
  const int r = blockIdx.x % n, ch = blockIdx.x / n;
  const DevComm& c = a.comm;
  if (aborted(c)) return;
  // AllReduce: channels split the buffer; the phases: channels split a
  // block, and every loop visits the same range of each block. A launch
  // runs one of the two slice sequences.
  unsigned long long lo, hi;
  channelRange<S>(a.count, a.nchannels, ch, lo, hi);
  const char* in = reinterpret_cast<const char*>(a.send[r]);
  char* out = reinterpret_cast<char*>(a.recv[r]);

  Agent ag;
  ag.init(c, wireProto(PROTO), r, ch);
  if (n > 1) {
    ag.addRecv(c, ringEdge(ch, (r - 1 + n) % n, n));
    ag.addSend(c, ringEdge(ch, r, n));
  }
  const bool direct = PROTO == kSimple && a.direct && (a.coll == kAllReduce || a.coll == kAllGather) && n > 1;
  if (direct) ag.addDirect(c, ringEdge(ch, (r - 1 + n) % n, n), ringEdge(ch, r, n));
  if (a.coll == kAllReduce || n == 1) {
    RingIter it;
    it.init(n, r, (long long)lo, (long long)(hi - lo), a.chunkElems, 16 / E, a.sliceElems, direct);
    if constexpr (PROTO == kSimple) {
      if (direct)
        ringAgent<PROTO, DT, OP, true>(a, ag, it, in, out);
      else
        ringAgent<PROTO, DT, OP, false>(a, ag, it, in, out);
    } else {
      ringAgent<PROTO, DT, OP>(a, ag, it, in, out);
    }
  } else {
    PhaseIter it;
    it.init(n, r, a.coll == kAllGather, (long long)lo, (long long)(hi - lo), (long long)a.count, a.chunkElems,
            a.sliceElems, direct);
    if constexpr (PROTO == kSimple) {
      if (direct)
        ringAgent<PROTO, DT, OP, true>(a, ag, it, in, out);
      else
        ringAgent<PROTO, DT, OP, false>(a, ag, it, in, out);
    } else {
      ringAgent<PROTO, DT, OP>(a, ag, it, in, out);
    }
  }
}

// ---------------------------------------------------------------------- tree
// ncclGetBtree / ncclGetDtree ("NCCL Source Code Deep Dive", ch.4;
// "NCCL architecture ...", §5.4): tree 0 is the bit-built binary tree, tree 1
// its mirror (even n) or its shift by one (odd n).
__host__ __device__ inline void getBtree(int n, int rank, int& up, int& d0, int& d1) {
  int bit = 1;
  while (bit < n) {
    if (bit & rank) break;
    bit <<= 1;
  }
  if (rank == 0) {
    up = -1;
    d0 = -1;
    d1 = n > 1 ? bit >> 1 : -1;
    return;
  }
  up = (rank ^ bit) | (bit << 1);
  if (up >= n) up = rank ^ bit;
  int lowbit = bit >> 1;
  d0 = lowbit == 0 ? -1 : rank - lowbit;
  d1 = lowbit == 0 ? -1 : rank + lowbit;
  while (d1 >= n) {  // the upper child is pulled into range one halving late
    d1 = lowbit == 0 ? -1 : rank + lowbit;
    lowbit >>= 1;
  }
}

__host__ __device__ inline void getTree(int n, int which, int rank, int& up, int& d0, int& d1) {
  if (which == 0) {
    getBtree(n, rank, up, d0, d1);
    return;
  }
  if (n % 2 == 1) {
    getBtree(n, (rank - 1 + n) % n, up, d0, d1);
    up = up == -1 ? -1 : (up + 1) % n;
    d0 = d0 == -1 ? -1 : (d0 + 1) % n;
    d1 = d1 == -1 ? -1 : (d1 + 1) % n;
  } else {
    getBtree(n, n - 1 - rank, up, d0, d1);
    up = up == -1 ? -1 : n - 1 - up;
    d0 = d0 == -1 ? -1 : n - 1 - d0;
    d1 = d1 == -1 ? -1 : n - 1 - d1;
  }
}

__host__ __device__ inline int treeRoot(int n, int which) {
  for (int r = 0; r < n; ++r) {
    int u, d0, d1;
    getTree(n, which, r, u, d0, d1);
    if (u == -1) return r;
  }
  return 0;
}

// The first ceil(C/2) channels run tree 0, the others tree 1 (NCCL gives the
// duplicated half of its channels the second tree, "NCCL architecture ...",
// §5.3).
__host__ __device__ inline int channelTree(int ch, int C) { return ch < (C + 1) / 2 ? 0 : 1; }

// Agents per channel: n "up" agents (the root's one does up and down) and
// n-1 "down" agents, as runTreeSplit splits a rank's threads between the
// two directions ("NCCL architecture ...", §9.4). Up agent of rank r:
// receive from down[0], down[1], reduce own-first, send to the parent.
// Root: same, then post-op, write the result and send it down. Down agent:
// receive from the parent, write the result, forward to the children.
template <int PROTO, int DT, int OP>
__global__ void __launch_bounds__(maxAgentThreads(PROTO)) treeKernel(const __grid_constant__ KArgs a) {
  using S = typename Ty<DT>::S;
  constexpr long long E = sizeof(S);
  const int n = a.nranks;
  const int per = 2 * n - 1;
  const int ch = blockIdx.x / per, i = blockIdx.x % per;
  const DevComm& c = a.comm;
  if (aborted(c)) return;
  const int which = channelTree(ch, a.nchannels);
  const int root = treeRoot(n, which);
  const bool downRole = i >= n;
  const int rank = downRole ? ((i - n) < root ? (i - n) : (i - n) + 1) : i;
  int up, d0, d1;
  getTree(n, which, rank, up, d0, d1);
  const int maxCh = c.maxChannels;

  Agent ag;
  ag.init(c, wireProto(PROTO), rank, ch);
  int flags;
  if (!downRole) {
    if (d0 >= 0) ag.addRecv(c, treeUpEdge(ch, d0, n, maxCh));
    if (d1 >= 0) ag.addRecv(c, treeUpEdge(ch, d1, n, maxCh));
    if (up >= 0) {
      ag.addSend(c, treeUpEdge(ch, rank, n, maxCh));
      flags = F_IN | F_SEND;
    } else {
      if (d0 >= 0) ag.addSend(c, treeDownEdge(ch, d0, n, maxCh));
      if (d1 >= 0) ag.addSend(c, treeDownEdge(ch, d1, n, maxCh));
      flags = F_IN | F_POST | F_OUT | (ag.nsend ? F_SEND : 0);
    }
    if (ag.nrecv) flags |= F_RECV;
  } else {
    ag.addRecv(c, treeDownEdge(ch, rank, n, maxCh));
    if (d0 >= 0) ag.addSend(c, treeDownEdge(ch, d0, n, maxCh));
    if (d1 >= 0) ag.addSend(c, treeDownEdge(ch, d1, n, maxCh));
    flags = F_RECV | F_OUT | (ag.nsend ? F_SEND : 0);
  }

  unsigned long long lo, hi;
  channelRange<S>(a.count, a.nchannels, ch, lo, hi);
  const char* in = reinterpret_cast<const char*>(a.send[rank]);
  char* out = reinterpret_cast<char*>(a.recv[rank]);
  TreeIter it;
  it.init((long long)lo, (long long)(hi - lo), a.sliceElems, flags);
  if constexpr (PROTO == kSimple) {
    simplePipeline<DT, OP, true>(a, ag, it, in, out);
  } else {
    llBegin();
    SliceDesc d;
    while (it.next(d))
      if (!runSlice<PROTO, DT, OP, true>(a, ag, in + d.inPos * E, out + d.outPos * E, d.nelem, d.flags)) return;
    ag.finish(c);
  }
}

// Explicit instantiation of every op of element types D0 .. D0+3 (or of all
// eight) for one protocol: rows of the kernel table.
#define VRCCL_KERNEL_DT_ROW(PROTO, ALGO_KERNEL, DT)                                                   \
  {(const void*)ALGO_KERNEL<PROTO, DT, 0>, (const void*)ALGO_KERNEL<PROTO, DT, 1>,                   \
   (const void*)ALGO_KERNEL<PROTO, DT, 2>, (const void*)ALGO_KERNEL<PROTO, DT, 3>,                   \
   (const void*)ALGO_KERNEL<PROTO, DT, 4>}
#define VRCCL_KERNEL_ROWS4(PROTO, ALGO_KERNEL, D0)                                                    \
  {VRCCL_KERNEL_DT_ROW(PROTO, ALGO_KERNEL, D0), VRCCL_KERNEL_DT_ROW(PROTO, ALGO_KERNEL, D0 + 1),     \
   VRCCL_KERNEL_DT_ROW(PROTO, ALGO_KERNEL, D0 + 2), VRCCL_KERNEL_DT_ROW(PROTO, ALGO_KERNEL, D0 + 3)}
#define VRCCL_KERNEL_ROWS8(PROTO, ALGO_KERNEL)                                                        \
  {VRCCL_KERNEL_DT_ROW(PROTO, ALGO_KERNEL, 0), VRCCL_KERNEL_DT_ROW(PROTO, ALGO_KERNEL, 1),           \
   VRCCL_KERNEL_DT_ROW(PROTO, ALGO_KERNEL, 2), VRCCL_KERNEL_DT_ROW(PROTO, ALGO_KERNEL, 3),           \
   VRCCL_KERNEL_DT_ROW(PROTO, ALGO_KERNEL, 4), VRCCL_KERNEL_DT_ROW(PROTO, ALGO_KERNEL, 5),           \
   VRCCL_KERNEL_DT_ROW(PROTO, ALGO_KERNEL, 6), VRCCL_KERNEL_DT_ROW(PROTO, ALGO_KERNEL, 7)}

}  // namespace vrccl
