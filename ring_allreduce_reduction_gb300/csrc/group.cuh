// Grouped AllReduce: one launch runs a list of ring AllReduces of one type
// and op. Each channel's agents walk the tasks that use their channel in
// task order, so the two ends of every ring edge see the same sequence of
// slices and the FIFO counters simply continue from task to task; so do
// the direct all-gather's counters (Simple), whose forwarded chunks land in
// the next rank's buffer of the same task.
#pragma once

#include "kernels.cuh"

namespace vrccl {

// The slices of every task on one channel, as element offsets from the
// rank's buffers of task 0 (all buffers are 16-byte aligned, so every
// difference is a whole number of elements).
template <typename S>
struct GroupRingIter {
  const GroupArgs* g;
  int n, r, ch, t;
  long long K, slice;
  const char* in0;
  const char* out0;
  RingIter it;
  long long dIn, dOut;
  long long dNext;     // direct: next rank's task buffer against its task-0 one, less dOut (elements)
  long long skipDone;  // direct: slices passed over in finished tasks
  bool live, direct;

  __device__ __forceinline__ void init(const GroupArgs* g_, int n_, int r_, int ch_) {
    g = g_;
    n = n_;
    r = r_;
    ch = ch_;
    t = -1;
    K = g->chunkElems;
    slice = g->sliceElems;
    in0 = reinterpret_cast<const char*>(g->send[r]);
    out0 = reinterpret_cast<const char*>(g->recv[r]);
    dIn = dOut = dNext = skipDone = 0;
    live = false;
    direct = g->direct != 0 && n > 1;
  }
  __device__ __forceinline__ long long skippedDirect() const { return skipDone + (live ? it.dskip : 0); }
  __device__ __forceinline__ long long nextShift() const { return dNext; }
  __device__ __forceinline__ bool nextTask() {
    const int C = g->nchannels;
    while (++t < g->ntasks) {
      const GroupTask& T = g->task[t];
      const int j = (ch - T.chLo + C) % C;  // this channel's index within the task
      if (j >= T.nch) continue;
      unsigned long long lo, hi;
      channelRange<S>(T.count, T.nch, j, lo, hi);
      it.init(n, r, (long long)lo, (long long)(hi - lo), K, 16 / (long long)sizeof(S), slice, direct);
      dIn = (reinterpret_cast<const char*>(g->send[t * n + r]) - in0) / (long long)sizeof(S);
      dOut = (reinterpret_cast<const char*>(g->recv[t * n + r]) - out0) / (long long)sizeof(S);
      const int r1 = (r + 1) % n;
      dNext = (reinterpret_cast<const char*>(g->recv[t * n + r1]) - reinterpret_cast<const char*>(g->recv[r1])) /
                  (long long)sizeof(S) - dOut;
      return true;
    }
    return false;
  }
  __device__ __forceinline__ bool next(SliceDesc& d) {
    while (true) {
      if (live && it.next(d)) {
        d.inPos += dIn;
        d.outPos += dOut;
        return true;
      }
      if (live) skipDone += it.dskip;
      live = false;
      if (!nextTask()) return false;
      live = true;
    }
  }
};

template <int PROTO, int DT, int OP>
__global__ void __launch_bounds__(maxAgentThreads(PROTO)) groupRingKernel(const __grid_constant__ GroupArgs g) {
  using S = typename Ty<DT>::S;
  const int n = g.nranks;
  const int r = blockIdx.x % n, ch = blockIdx.x / n;
  const DevComm& c = g.comm;
  if (aborted(c)) return;
  Agent ag;
  ag.init(c, PROTO, r, ch);
  if (n > 1) {
    ag.addRecv(c, ringEdge(ch, (r - 1 + n) % n, n));
    ag.addSend(c, ringEdge(ch, r, n));
  }
  GroupRingIter<S> it;
  it.init(&g, n, r, ch);
  const char* in = reinterpret_cast<const char*>(g.send[r]);
  char* out = reinterpret_cast<char*>(g.recv[r]);
  if constexpr (PROTO == kSimple) {
    if (it.direct) {
      ag.addDirect(c, ringEdge(ch, (r - 1 + n) % n, n), ringEdge(ch, r, n));
      ringAgent<PROTO, DT, OP, true>(g, ag, it, in, out);
    } else {
      ringAgent<PROTO, DT, OP, false>(g, ag, it, in, out);
    }
  } else {
    ringAgent<PROTO, DT, OP>(g, ag, it, in, out);
  }
}

#define VRCCL_GROUP_ROW(PROTO, DT)                                                          \
  {(const void*)groupRingKernel<PROTO, DT, 0>, (const void*)groupRingKernel<PROTO, DT, 1>, \
   (const void*)groupRingKernel<PROTO, DT, 2>, (const void*)groupRingKernel<PROTO, DT, 3>, \
   (const void*)groupRingKernel<PROTO, DT, 4>}
#define VRCCL_GROUP_TABLE(PROTO)                                                                 \
  {VRCCL_GROUP_ROW(PROTO, 0), VRCCL_GROUP_ROW(PROTO, 1), VRCCL_GROUP_ROW(PROTO, 2), VRCCL_GROUP_ROW(PROTO, 3), \
   VRCCL_GROUP_ROW(PROTO, 4), VRCCL_GROUP_ROW(PROTO, 5), VRCCL_GROUP_ROW(PROTO, 6), VRCCL_GROUP_ROW(PROTO, 7)}

}  // namespace vrccl
