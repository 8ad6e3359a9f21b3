// Simple protocol as a warp-specialised pipeline.
//
// The Simple wire format is unchanged: a slot of raw elements, published by
// raising the edge's tail counter once the whole slot is written, drained
// by raising its head counter ("NCCL architecture: topology, channels,
// algorithms and protocols", §6.5 and §7.2). What changes is how one agent
// (CTA) moves its slices:
//
//   warp 0, one thread   input producer: as soon as stage q % S of the
//                        shared-memory ring is free it bulk-copies (TMA,
//                        cp.async.bulk) the agent's input slice q into it.
//   warp 1, one thread   FIFO producer: waits until the out-edge slot of
//                        slice q is drained and its in-edge slot filled
//                        (cached flag values cover several slices per
//                        poll), then, once stage q % S is free, bulk-copies
//                        the received slot(s) next to the input; in the
//                        direct all-gather, the chunk the predecessor wrote
//                        into this rank's recv buffer instead.
//   warp 2, one thread   publisher: once every consumer warp is past a run
//                        of slices it publishes them with one gpu-scope fence
//                        and the new tail (sent) and head (drained) counters.
//   warps 3..W+2         consumers. They wait for the stage, reduce from
//                        shared memory, store the result to the out-edge
//                        slot, the recv buffer and/or (direct) the next
//                        rank's recv buffer, free the stage and report the
//                        slice done. They never fence at gpu scope, so no
//                        consumer waits for the memory system.
//
// So the producer keeps up to S slices of input and FIFO data in flight
// while consumers work, and no CTA-wide barrier is taken per slice.
#pragma once

#include "schedule.cuh"

namespace vrccl {

struct PipeShared {
  unsigned long long fullIn[kMaxStages];    // input producer's copies landed
  unsigned long long fullFifo[kMaxStages];  // FIFO producer's copies landed
  unsigned long long empty[kMaxStages];
  unsigned prog[kMaxConsumerWarps];  // slices finished by each consumer warp
  int abort;
};

// Bounded wait on a shared-memory barrier phase; false = give up.
__device__ __forceinline__ bool pipeWait(const DevComm& c, const Agent& ag, PipeShared* sh,
                                         unsigned long long* bar, unsigned parity) {
  Spin sp(15u);
  while (!mbarTryWait(bar, parity)) {
    if (*reinterpret_cast<volatile int*>(&sh->abort)) return false;
    if (sp.tick(c, ag.rank, ag.ch, 4, 0)) return false;
  }
  return true;
}

// Waits (bounded) until every bulk copy this thread issued into the stage
// ring has landed; a CTA must not exit with copies into its shared memory in
// flight.
__device__ __forceinline__ void drainStages(const DevComm& c, unsigned long long* full, const int* lastUse,
                                            int nst) {
  for (int i = 0; i < nst; ++i) {
    if (lastUse[i] < 0) continue;
    const unsigned long long t0 = globalTimer();
    while (!mbarTryWait(&full[i], lastUse[i] & 1)) {
      if (globalTimer() - t0 > c.timeoutNs) break;
    }
  }
}

// The consumers' vector loop over one slice. The ring compiles it once per
// combination of "reads its input" (IN) and "reads a received value" (RV),
// so the loop carries no per-vector test of the slice's kind (measured on
// the 256 MiB fp32 ring, n = 8: sum 1.086 -> 1.081 ms with the FIFO
// all-gather, avg 1.462 -> 1.084 ms, the direct all-gather 1.394 -> 0.887
// ms). The tree keeps one loop for every kind (IN = RV = false below
// means "decided per vector"): split like the ring's it measured slower
// (256 MiB, n = 8: 2.36 -> 2.61 ms).
template <int DT, int OP, bool TREE, bool DIRECT, bool IN, bool RV>
__device__ __forceinline__ void consumeVectors(int ct, int CT, int nv, const char* sIn, const char* sR0, const char* sR1,
                                               int post, int nrecv, float scale, int n, char* dst0, char* dst1,
                                               char* dnx, char* o, unsigned long long keep) {
  // TREE: post carries the slice's flags, decided per vector
  const int flags = TREE ? post : (IN ? F_IN : 0) | (RV ? F_RECV : 0) | post;
  const int nr = TREE ? nrecv : (RV ? 1 : 0);
  const bool rdIn = TREE ? (flags & F_IN) != 0 : IN;
  const bool rdR0 = TREE ? (flags & F_RECV) && nr > 0 : RV;
  for (int i = ct; i < nv; i += CT) {
    const size_t b = size_t(i) * 16;
    uint4 xv = make_uint4(0, 0, 0, 0), r0v = xv, r1v = xv;
    if (rdIn) xv = *reinterpret_cast<const uint4*>(sIn + b);
    if (rdR0) r0v = *reinterpret_cast<const uint4*>(sR0 + b);
    if constexpr (TREE)
      if (rdR0 && nr > 1) r1v = *reinterpret_cast<const uint4*>(sR1 + b);
    uint32_t x[4] = {xv.x, xv.y, xv.z, xv.w}, r0[4] = {r0v.x, r0v.y, r0v.z, r0v.w},
             r1[4] = {r1v.x, r1v.y, r1v.z, r1v.w}, acc[4];
    reduceWords<DT, OP, TREE, 4>(acc, x, r0, r1, flags, nr, scale, n);
    const uint4 av = make_uint4(acc[0], acc[1], acc[2], acc[3]);
    if (dst0) stFifoHint16(dst0 + b, av, keep);
    if (dst1) stFifoHint16(dst1 + b, av, keep);
    if constexpr (DIRECT)
      if (dnx) stFifo16(dnx + b, av);
    if (o) stStream16(o + b, av);
  }
}

// DIRECT: the ring's all-gather through the recv buffers (F_DRECV /
// F_DSEND slices); a separate instantiation, so the FIFO form carries none
// of its per-slice work. The in-edge's count of direct slices received is
// the slices run (ag.drstep) plus those passed over (it.skippedDirect()).
template <int DT, int OP, bool TREE, bool DIRECT = false, class Args, class It>
__device__ void simplePipeline(const Args& a, Agent& ag, It it, const char* in, char* out) {
  using S = typename Ty<DT>::S;
  constexpr int E = sizeof(S);
  constexpr int V = 16 / E;
  constexpr int NBUF = TREE ? 3 : 2;  // own input + up to (NBUF-1) received slots
  extern __shared__ __align__(128) char smemDyn[];
  __shared__ PipeShared sh;
  const DevComm& c = a.comm;
  // Buffers of one stage: the ring's input and received slot; for a tree
  // agent those its role uses (its input if it reads it, one slot per
  // in-edge). The block's dynamic shared memory, a.stages stages of NBUF
  // slices, is cut into as many of this agent's stages as fit (at most
  // kMaxStages), so down agents and leaves get deeper pipelines than the
  // two-child agents the launch was sized for.
  int inBuf = 1, nbuf = NBUF;
  if constexpr (TREE) {
    inBuf = (it.flags & F_IN) ? 1 : 0;
    nbuf = max(1, inBuf + ag.nrecv);
  }
  const int NST = TREE ? min(kMaxStages, a.stages * NBUF / nbuf) : a.stages;
  const size_t sliceBytes = size_t(a.sliceElems) * E;
  const int W = (blockDim.x >> 5) - 3;  // consumer warps
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbarInit(&sh.fullIn[i], 1);
      mbarInit(&sh.fullFifo[i], 1);
      mbarInit(&sh.empty[i], W);
    }
    for (int w = 0; w < W; ++w) sh.prog[w] = 0;
    sh.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------- input producer
    // Streams this agent's own input slices into the stage ring as soon as
    // a stage is free; it never waits on another agent.
    if (lane != 0) return;
    int lastUse[kMaxStages];
    for (int i = 0; i < NST; ++i) lastUse[i] = -1;
    // A second walk of the same sequence, a.prefetch slices ahead, pulls
    // future input slices into L2 so the stage copies hit L2, not HBM.
    It ahead = it;
    SliceDesc pd;
    bool pmore = a.prefetch > 0;
    for (int k = 0; k < a.prefetch && pmore; ++k) {
      pmore = ahead.next(pd);
      if (pmore && (pd.flags & F_IN) && pd.nelem * E >= 16) bulkPrefetchL2(in + pd.inPos * E, unsigned(pd.nelem * E / 16 * 16));
    }
    SliceDesc d;
    int st = 0, ph = 0;  // next stage and its phase (no division per slice)
    bool ok = true;
    const unsigned long long once = evictFirstPolicy();
    while (it.next(d)) {
      if (pmore && (pmore = ahead.next(pd)) && (pd.flags & F_IN) && pd.nelem * E >= 16)
        bulkPrefetchL2(in + pd.inPos * E, unsigned(pd.nelem * E / 16 * 16));
      if (!pipeWait(c, ag, &sh, &sh.empty[st], ph ^ 1)) {
        ok = false;
        break;
      }
      const unsigned inBytes = (d.flags & F_IN) ? unsigned(d.nelem * E / 16 * 16) : 0u;
      if (inBytes) {
        lastUse[st] = ph;
        mbarExpectTx(&sh.fullIn[st], inBytes);
        bulkLoadOnce(smemDyn + size_t(st) * nbuf * sliceBytes, in + d.inPos * E, inBytes, &sh.fullIn[st], once);
      }
      mbarArrive(&sh.fullIn[st]);
      if (++st == NST) {
        st = 0;
        ph ^= 1;
      }
    }
    if (!ok) {
      *reinterpret_cast<volatile int*>(&sh.abort) = 1;
      drainStages(c, sh.fullIn, lastUse, NST);
    }
    return;
  }

  if (warp == 1) {
    // -------------------------------------------------- FIFO producer
    // For each slice: wait until the out-edge slot is drained and the
    // in-edge slot is filled (cached flag values cover several slices per
    // poll), then bulk-copy the received slot(s) into the stage.
    if (lane != 0) return;
    unsigned long long headSeen[2] = {0, 0}, tailSeen[2] = {0, 0}, dtailSeen = 0;
    // A forwarded chunk's recv lines are final output once copied here:
    // tagged evict-first, they leave L2 ahead of the FIFO lines still to be
    // read (256 MiB fp32 ring, n = 8: 0.893 -> 0.872 ms).
    const unsigned long long fwdPolicy = DIRECT ? evictFirstPolicy() : 0ull;
    int lastUse[kMaxStages];
    for (int i = 0; i < NST; ++i) lastUse[i] = -1;
    SliceDesc d;
    int st = 0, ph = 0;  // next stage and its phase
    bool ok = true;
    while (it.next(d)) {
      if (ag.faultNow(c)) {
        ok = false;
        break;
      }
      // The flags first: they do not depend on the stage, so their polls
      // overlap the consumers' work on the stage (measured: 1.127 -> 1.088
      // ms on the 256 MiB fp32 ring against waiting for the stage first).
      const unsigned rvBytes = unsigned((d.nelem * E + 15) / 16 * 16);
      if (d.flags & F_SEND) {
        for (int i = 0; i < ag.nsend && ok; ++i) {
          const unsigned long long need = ag.sstep[i] + 1;
          if (need > (unsigned long long)kSteps)
            ok = flagAtLeast(c, ag, &c.ctrl[kSimple][ag.se[i]].head, need - kSteps, headSeen[i], 1);
        }
      }
      bool fresh = false;
      if (ok && (d.flags & F_RECV)) {
        for (int i = 0; i < ag.nrecv && ok; ++i) {
          const unsigned long long before = tailSeen[i];
          ok = flagAtLeast(c, ag, &c.ctrl[kSimple][ag.re[i]].tail, ag.rstep[i] + 1, tailSeen[i], 0);
          fresh |= tailSeen[i] != before;
        }
      }
      if (ok && !pipeWait(c, ag, &sh, &sh.empty[st], ph ^ 1)) {
        ok = false;
        break;
      }
      if (ok && (d.flags & F_RECV)) {
        char* buf = smemDyn + size_t(st) * nbuf * sliceBytes;
        if (fresh) fenceProxyAsync();
        for (int i = 0; i < ag.nrecv; ++i) {
          lastUse[st] = ph;
          mbarExpectTx(&sh.fullFifo[st], rvBytes);
          bulkLoad(buf + size_t(inBuf + i) * sliceBytes, ag.slot(c, ag.re[i], ag.rstep[i]), rvBytes,
                   &sh.fullFifo[st]);
        }
      }
      if (DIRECT && ok && (d.flags & F_DRECV) && (d.flags & F_DSEND)) {
        // Direct: the predecessor wrote this slice into this rank's recv
        // buffer; take its whole 16-byte units (the ragged end of the
        // buffer is read element by element, never past the buffer).
        const unsigned long long before = dtailSeen;
        ok = flagAtLeast(c, ag, &c.dctrl[ag.dre].tail, ag.drstep + it.skippedDirect() + 1, dtailSeen, 0);
        const unsigned dBytes = unsigned(d.nelem * E / 16 * 16);
        if (ok && dBytes) {
          if (dtailSeen != before) fenceProxyAsync();
          lastUse[st] = ph;
          mbarExpectTx(&sh.fullFifo[st], dBytes);
          bulkLoadOnce(smemDyn + size_t(st) * nbuf * sliceBytes + size_t(inBuf) * sliceBytes, out + d.outPos * E,
                       dBytes, &sh.fullFifo[st], fwdPolicy);
        }
      }
      // On failure the consumers are told before this arrival, so the stage
      // it may complete is never published.
      if (!ok) *reinterpret_cast<volatile int*>(&sh.abort) = 1;
      mbarArrive(&sh.fullFifo[st]);
      if (!ok) break;
      ag.advance(d.flags);
      if constexpr (DIRECT) ag.advanceDirect(d.flags);
      if (++st == NST) {
        st = 0;
        ph ^= 1;
      }
    }
    if (!ok) {
      *reinterpret_cast<volatile int*>(&sh.abort) = 1;
      drainStages(c, sh.fullFifo, lastUse, NST);
    }
    return;
  }

  if (warp == 2) {
    // ------------------------------------------------------- publisher
    // Slices are complete once every consumer warp has moved past them.
    // Whatever has completed since the last pass is published at once:
    // one gpu-scope fence (cumulative over the consumers' stores, which the
    // CTA-scope acquire below ordered before it), then the new tail of each
    // out-edge and head of each in-edge.
    if (lane != 0) return;
    SliceDesc d;
    long long q = 0;  // slices published so far
    bool more = it.next(d);
    Spin sp(15u);
    while (more) {
      unsigned done = 0xffffffffu;
      for (int w = 0; w < W; ++w) {
        unsigned v;
        asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smemAddr(&sh.prog[w])) : "memory");
        done = min(done, v);
      }
      if ((long long)done <= q) {
        if (*reinterpret_cast<volatile int*>(&sh.abort) || sp.tick(c, ag.rank, ag.ch, 4, 0)) return;
        continue;
      }
      bool send = false, recv = false;
      int anyDirect = 0;
      while (more && q < (long long)done) {
        send |= (d.flags & F_SEND) != 0;
        recv |= (d.flags & F_RECV) != 0;
        ag.advance(d.flags);
        if constexpr (DIRECT) {
          anyDirect |= d.flags;
          ag.advanceDirect(d.flags);
        }
        ++q;
        more = it.next(d);
      }
      if (send || recv || (DIRECT && (anyDirect & F_DSEND))) {
        fenceAcqRelGpu();
        if (send)
          for (int i = 0; i < ag.nsend; ++i) redMaxRelaxed(&c.ctrl[kSimple][ag.se[i]].tail, ag.sstep[i]);
        if (recv)
          for (int i = 0; i < ag.nrecv; ++i) redMaxRelaxed(&c.ctrl[kSimple][ag.re[i]].head, ag.rstep[i]);
        if constexpr (DIRECT) {
          if (anyDirect & F_DSEND) redMaxRelaxed(&c.dctrl[ag.dse].tail, ag.dsstep);
        }
      }
    }
    // The direct in-edge's head is read only at the next launch's start
    // (it seeds that launch's count), so it is written once, complete.
    if constexpr (DIRECT) redMaxRelaxed(&c.dctrl[ag.dre].head, ag.drstep + it.skippedDirect());
    return;
  }

  // -------------------------------------------------------------- consumers
  const int ct = threadIdx.x - 96, CT = W * 32;
  const int cw = warp - 3;
  // FIFO slots are stored evict-last: they must survive in L2 until their
  // receiver reads them (256 MiB fp32 ring, n = 8: 0.872 -> 0.859 ms with
  // the direct all-gather, 1.091 -> 1.088 ms with FIFOs only)
  const unsigned long long keep = evictLastPolicy();
  char* const nextOut = DIRECT ? reinterpret_cast<char*>(a.recv[(ag.rank + 1) % a.nranks]) : nullptr;
  SliceDesc d;
  unsigned q = 0;      // slices done
  int st = 0, ph = 0;  // stage and phase
  while (it.next(d)) {
    if (!pipeWait(c, ag, &sh, &sh.fullIn[st], ph)) return;
    if (!pipeWait(c, ag, &sh, &sh.fullFifo[st], ph)) return;
    if (*reinterpret_cast<volatile int*>(&sh.abort)) return;
    const char* buf = smemDyn + size_t(st) * nbuf * sliceBytes;
    const char* sIn = buf;
    const char* sR0 = buf + size_t(inBuf) * sliceBytes;
    const char* sR1 = sR0 + sliceBytes;
    const bool rv = (d.flags & F_RECV) && ag.nrecv > 0;
    const bool drv = DIRECT && (d.flags & F_DRECV) && (d.flags & F_DSEND);  // staged from own recv buffer
    const int rf = d.flags | (drv ? F_RECV : 0);  // the reduction sees a received value
    char* dst0 = (d.flags & F_SEND) && ag.nsend > 0 ? ag.slot(c, ag.se[0], ag.sstep[0]) : nullptr;
    char* dst1 = (d.flags & F_SEND) && ag.nsend > 1 ? ag.slot(c, ag.se[1], ag.sstep[1]) : nullptr;
    char* dnx = DIRECT && (d.flags & F_DSEND) ? nextOut + (d.outPos + it.nextShift()) * E : nullptr;
    char* o = out + d.outPos * E;
    const int nv = d.nelem / V;
    {
      char* const ov = (d.flags & F_OUT) ? o : nullptr;
      const int post = d.flags & F_POST;
      const bool inF = d.flags & F_IN, rvF = rv || drv;
      if constexpr (TREE)
        consumeVectors<DT, OP, TREE, DIRECT, false, false>(ct, CT, nv, sIn, sR0, sR1, rf, ag.nrecv, a.scale,
                                                           a.nranks, dst0, dst1, dnx, ov, keep);
      else if (inF && rvF)
        consumeVectors<DT, OP, TREE, DIRECT, true, true>(ct, CT, nv, sIn, sR0, sR1, post, ag.nrecv, a.scale,
                                                         a.nranks, dst0, dst1, dnx, ov, keep);
      else if (inF)
        consumeVectors<DT, OP, TREE, DIRECT, true, false>(ct, CT, nv, sIn, sR0, sR1, post, ag.nrecv, a.scale,
                                                          a.nranks, dst0, dst1, dnx, ov, keep);
      else if (rvF)
        consumeVectors<DT, OP, TREE, DIRECT, false, true>(ct, CT, nv, sIn, sR0, sR1, post, ag.nrecv, a.scale,
                                                          a.nranks, dst0, dst1, dnx, ov, keep);
      else
        consumeVectors<DT, OP, TREE, DIRECT, false, false>(ct, CT, nv, sIn, sR0, sR1, post, ag.nrecv, a.scale,
                                                           a.nranks, dst0, dst1, dnx, ov, keep);
    }
    for (int j = nv * V + ct; j < d.nelem; j += CT) {  // ragged end of the user buffer
      S x = (d.flags & F_IN) ? reinterpret_cast<const S*>(in + d.inPos * E)[j] : S(0);
      S r0 = rv ? reinterpret_cast<const S*>(sR0)[j] : drv ? reinterpret_cast<const S*>(o)[j] : S(0);
      S r1 = (rv && ag.nrecv > 1) ? reinterpret_cast<const S*>(sR1)[j] : S(0);
      S v = reduceElem<DT, OP, TREE>(x, r0, r1, rf, ag.nrecv, a.scale, a.nranks);
      if (dst0) reinterpret_cast<S*>(dst0)[j] = v;
      if (dst1) reinterpret_cast<S*>(dst1)[j] = v;
      if (dnx) reinterpret_cast<S*>(dnx)[j] = v;
      if (d.flags & F_OUT) reinterpret_cast<S*>(o)[j] = v;
    }
    if (rv) {
      // The received slot(s) now sit in shared memory and the sender will
      // rewrite them: drop their L2 lines instead of letting them be written
      // back to HBM. The report below orders this before the head that
      // lets the sender reuse the slot.
      const int lines = (d.nelem * E + 127) / 128;
      for (int i = 0; i < ag.nrecv; ++i) {
        const char* slotp = ag.slot(c, ag.re[i], ag.rstep[i]);
        for (int l = ct; l < lines; l += CT) discardL2(slotp + size_t(l) * 128);
      }
    }
    __syncwarp();
    if (lane == 0) {
      // Free the stage (its shared memory has been read), then report the
      // slice done; the release orders this warp's stores before the report.
      mbarArrive(&sh.empty[st]);
      asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smemAddr(&sh.prog[cw])), "r"(q + 1)
                   : "memory");
    }
    ag.advance(d.flags);
    if constexpr (DIRECT) ag.advanceDirect(d.flags);
    if (++st == NST) {
      st = 0;
      ph ^= 1;
    }
    ++q;
  }
}

}  // namespace vrccl
