// The agent engine: one CTA is one agent, i.e. one virtual rank working one
// channel (ring) or one role of one rank in one tree (tree). An agent runs
// a fixed sequence of FIFO steps ("slices"); each slice receives from up
// to two in-edges, reduces with the agent's own input, and sends on up to
// two out-edges and/or writes the agent's recv buffer -- the primitives of
// "NCCL architecture: topology, channels, algorithms and protocols", §9.4
// (send / recvReduceSend / recvReduceCopySend / recvCopySend / recv, with
// Fan = receive/send arity: ring 1/1, tree up to 2/1 and 1/2).
//
// Flow control is NCCL's head/tail credit scheme of §6.5 of the same page:
// a sender may fill slot `step % VRCCL_STEPS` once the receiver's head
// shows the slot drained (head + VRCCL_STEPS > step). How the receiver
// learns that data is complete depends on the protocol (§7.2):
//   Simple  the sender releases a tail counter after the whole slot;
//   LL      every 16-byte line carries the step number twice next to 8
//           bytes of data and is written with one 16-byte store;
//   LL128   every 128-byte line carries 120 data bytes and an 8-byte flag,
//           written with the data by one warp store (see the LL128
//           section below for what that rests on).
#pragma once

#include "device_common.cuh"

namespace vrccl {

enum SliceFlags : int {
  F_IN = 1,    // read this agent's input (pre-scaled) into the reduction
  F_OUT = 2,   // write the result to this agent's recv buffer
  F_POST = 4,  // apply the post-op (int32 avg)
  F_RECV = 8,    // receive on every in-edge
  F_SEND = 16,   // send on every out-edge
  F_DRECV = 32,  // direct: the slice was written into this agent's recv buffer by its predecessor
  F_DSEND = 64   // direct: write the result into the next rank's recv buffer
};

struct Agent {
  int rank, ch, proto;
  int nrecv, nsend;
  int re[2], se[2];
  unsigned long long rstep[2], sstep[2];
  int slices;     // FIFO steps done in this launch (fault injection clock)
  int rvDone;     // receiving steps done in this launch
  bool faulty;    // this agent is the injected fault
  unsigned long long headSeen[2];  // LL128: last value seen of each out-edge's head (per warp)
  int dre, dse;   // direct edges (ring, Simple): in and out, -1 if none
  unsigned long long drstep, dsstep;

  __device__ __forceinline__ void init(const DevComm& c, int proto_, int rank_, int ch_) {
    proto = proto_;
    rank = rank_;
    ch = ch_;
    nrecv = nsend = 0;
    slices = 0;
    rvDone = 0;
    headSeen[0] = headSeen[1] = 0;
    dre = dse = -1;
    drstep = dsstep = 0;
    faulty = (c.faultRank == rank_ && c.faultChannel == ch_);
  }
  __device__ __forceinline__ void addRecv(const DevComm& c, int e) {
    if (e < 0) return;
    re[nrecv] = e;
    rstep[nrecv] = ldRelaxed(&c.ctrl[proto][e].head);  // posted by this agent last launch
    ++nrecv;
  }
  __device__ __forceinline__ void addSend(const DevComm& c, int e) {
    if (e < 0) return;
    se[nsend] = e;
    sstep[nsend] = ldRelaxed(&c.ctrl[proto][e].tail);  // posted by this agent last launch
    ++nsend;
  }
  // The direct all-gather edges of a ring agent: recv from the previous
  // rank's edge, send on its own (the counters continue across launches).
  __device__ __forceinline__ void addDirect(const DevComm& c, int inEdge, int outEdge) {
    dre = inEdge;
    dse = outEdge;
    drstep = ldRelaxed(&c.dctrl[inEdge].head);
    dsstep = ldRelaxed(&c.dctrl[outEdge].tail);
  }
  __device__ __forceinline__ bool faultNow(const DevComm& c) const { return faulty && slices >= c.faultAfter; }
  __device__ __forceinline__ char* slot(const DevComm& c, int e, unsigned long long step) const {
    return c.fifo[proto] + (size_t(e) * kSteps + size_t(step % kSteps)) * slotBufferBytes(proto);
  }
  __device__ __forceinline__ void advance(int flags) {
    if (flags & F_RECV) {
      for (int i = 0; i < nrecv; ++i) ++rstep[i];
      ++rvDone;
    }
    if (flags & F_SEND)
      for (int i = 0; i < nsend; ++i) ++sstep[i];
    ++slices;
  }
  __device__ __forceinline__ void advanceDirect(int flags) {
    if (flags & F_DRECV) ++drstep;
    if (flags & F_DSEND) ++dsstep;
  }
  // LL / LL128 keep the sender's step only in registers during a launch;
  // store it so the next launch continues the flag sequence.
  __device__ __forceinline__ void finish(const DevComm& c) {
    if (proto != kSimple && threadIdx.x == 0)
      for (int i = 0; i < nsend; ++i) stRelaxed(&c.ctrl[proto][se[i]].tail, sstep[i]);
  }
};

// Wait (bounded) until *p >= need, acquiring it, with a cached last-seen
// value that spares the poll when it already covers `need`.
__device__ __forceinline__ bool flagAtLeast(const DevComm& c, const Agent& ag, const unsigned long long* p,
                                            unsigned long long need, unsigned long long& seen, int kind) {
  if (seen >= need) return true;
  Spin sp;
  unsigned long long v;
  while ((v = ldAcquire(p)) < need) {
    if (sp.tick(c, ag.rank, ag.ch, kind, need)) return false;
  }
  seen = v;
  return true;
}

// LL128: per FIFO slot, the warps of the agent that are done reading it;
// monotonic within a launch (zeroed at its start by llBegin).
__device__ __forceinline__ unsigned* llSlotDone() {
  __shared__ unsigned cnt[kSteps];
  return cnt;
}
__device__ __forceinline__ void llBegin() {
  if (threadIdx.x < kSteps) llSlotDone()[threadIdx.x] = 0;
  __syncthreads();
}

// LL / LL128, per warp: wait until every out-edge slot of this step is
// drained (lane 0 polls each head, caching the value it saw); false = give
// up (abort/timeout/fault).
__device__ __forceinline__ bool warpCredit(const DevComm& c, Agent& ag, int flags, int proto) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) {
    ok = !ag.faultNow(c);
    if (ok && (flags & F_SEND))
      for (int i = 0; i < ag.nsend && ok; ++i) {
        const unsigned long long need = ag.sstep[i] + 1;
        if (need > (unsigned long long)kSteps)
          ok = flagAtLeast(c, ag, &c.ctrl[proto][ag.se[i]].head, need - kSteps, ag.headSeen[i], 1);
      }
  }
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// LL / LL128, per warp, after its reads of a received slice: the last warp
// of the agent done with it returns the slot(s) to the sender. One
// shared-memory counter per slot position, growing within the launch,
// counts the warps done with each use; before counting itself for receiving
// step k a warp waits (bounded) until every warp has counted step k -
// VRCCL_STEPS, the counter's previous use. (A warp with no lines in a
// slice waits for no flag, so without that wait it could run a whole
// counter cycle ahead of a slower warp and the counts of two uses would
// mix: a grouped run of small tasks did that and never returned a slot.)
// The count is a relaxed shared-memory atomic: a warp counts itself only
// after it has used every value it loaded from the slot, so its loads are
// done (an acquire-release atomic here made every step wait for the warp's
// stores to complete). false = gave up (abort/timeout).
__device__ __forceinline__ bool warpDoneReading(const DevComm& c, Agent& ag, int proto, int lane) {
  __syncwarp();  // every lane's loads of the slot are done
  int ok = 1;
  if (lane == 0) {
    const unsigned k = unsigned(ag.rvDone);
    const unsigned W = blockDim.x >> 5;
    unsigned* cnt = &llSlotDone()[k % kSteps];
    Spin sp(15u);
    while (*reinterpret_cast<volatile unsigned*>(cnt) < (k / kSteps) * W)
      if (sp.tick(c, ag.rank, ag.ch, 4, ag.rstep[0] + 1)) {
        ok = 0;
        break;
      }
    if (ok) {
      const unsigned prev = atomicAdd(cnt, 1u);
      if (prev + 1 == (k / kSteps + 1) * W)
        for (int i = 0; i < ag.nrecv; ++i) stRelaxed(&c.ctrl[proto][ag.re[i]].head, ag.rstep[i] + 1);
    }
  }
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Reduction of one group of NW 32-bit words.
//   ring order: acc = op(received, own)       (recv first)
//   tree order: acc = op(op(own, recv0), recv1) (own first, children in order)
// Without F_IN the received value is copied; without F_RECV the own value is.
template <int DT, int OP, bool TREE, int NW>
__device__ __forceinline__ void reduceWords(uint32_t (&acc)[NW], const uint32_t (&x)[NW], const uint32_t (&r0)[NW],
                                            const uint32_t (&r1)[NW], int flags, int nrecv, float scale, int n) {
  const bool in = flags & F_IN;
  const bool rv = (flags & F_RECV) && nrecv > 0;
  if constexpr (sizeof(typename Ty<DT>::S) == 8) {
    // 8-byte elements: the same steps on word pairs
    uint32_t own[NW], v[NW];
#pragma unroll
    for (int w = 0; w < NW; ++w) own[w] = in ? x[w] : 0u;
    if (in) prescaleWords<DT, OP, NW>(own, scale, n);
#pragma unroll
    for (int w = 0; w < NW; ++w) v[w] = (TREE ? !in : rv) ? r0[w] : own[w];
    if constexpr (!TREE) {
      if (rv && in) combineWords<DT, OP, NW>(v, own);
    } else {
      if (in && rv) combineWords<DT, OP, NW>(v, r0);
      if (in && rv && nrecv > 1) combineWords<DT, OP, NW>(v, r1);
    }
    if (flags & F_POST) postopWords<DT, OP, NW>(v, n);
#pragma unroll
    for (int w = 0; w < NW; ++w) acc[w] = v[w];
  } else {
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      uint32_t own = in ? prescaleWord<DT, OP>(x[w], scale) : 0u;
      uint32_t v;
      if constexpr (!TREE) {
        v = rv ? (in ? combineWord<DT, OP>(r0[w], own) : r0[w]) : own;
      } else {
        if (in) {
          v = own;
          if (rv) v = combineWord<DT, OP>(v, r0[w]);
          if (rv && nrecv > 1) v = combineWord<DT, OP>(v, r1[w]);
        } else {
          v = r0[w];
        }
      }
      if (flags & F_POST) v = postopWord<DT, OP>(v, n);
      acc[w] = v;
    }
  }
}

// Same on single elements (the ragged end of a buffer).
template <int DT, int OP, bool TREE>
__device__ __forceinline__ typename Ty<DT>::S reduceElem(typename Ty<DT>::S x, typename Ty<DT>::S r0,
                                                         typename Ty<DT>::S r1, int flags, int nrecv, float scale,
                                                         int n) {
  using S = typename Ty<DT>::S;
  const bool in = flags & F_IN;
  const bool rv = (flags & F_RECV) && nrecv > 0;
  S own = in ? prescale<DT, OP>(x, scale, n) : S(0);
  S v;
  if constexpr (!TREE) {
    v = rv ? (in ? combine<DT, OP>(r0, own) : r0) : own;
  } else {
    if (in) {
      v = own;
      if (rv) v = combine<DT, OP>(v, r0);
      if (rv && nrecv > 1) v = combine<DT, OP>(v, r1);
    } else {
      v = r0;
    }
  }
  if (flags & F_POST) v = postop<DT, OP>(v, n);
  return v;
}

// ------------------------------------------------------- 8-byte user units
// LL and LL128 carry user data in 8-byte units. The last unit of a user
// buffer may be partial: read and write only its valid elements.
template <typename S>
__device__ __forceinline__ uint2 loadUnit(const char* p, int validBytes) {
  if (validBytes >= 8) return ldStream8(p);
  uint32_t w[2] = {0u, 0u};
  for (int b = 0; b < validBytes; ++b) w[b >> 2] |= uint32_t((unsigned char)p[b]) << (8 * (b & 3));
  return make_uint2(w[0], w[1]);
}
template <typename S>
__device__ __forceinline__ void storeUnit(char* p, uint2 v, int validBytes) {
  if (validBytes >= 8) {
    stStream8(p, v);
    return;
  }
  const uint32_t w[2] = {v.x, v.y};
  for (int b = 0; b < validBytes; ++b) p[b] = char((w[b >> 2] >> (8 * (b & 3))) & 0xffu);
}

// ---------------------------------------------------------------------- LL
// Line u of a slot carries user bytes [8u, 8u+8) of the slice as
// {data lo, flag, data hi, flag}, flag = (uint32)(step + 1). A reader spins
// on the line until both flags equal the expected step; the line's data is
// then complete (the two halves were written by one 16-byte store). Flags
// only grow, so slots are never cleared.
template <int DT, int OP, bool TREE, class Args>
__device__ bool llSlice(const Args& a, Agent& ag, const char* in, char* out, int nelem, int flags) {
  using S = typename Ty<DT>::S;
  const DevComm& c = a.comm;
  const int lane = threadIdx.x & 31;
  if (!warpCredit(c, ag, flags, kLL)) return false;

  const int nbytes = nelem * int(sizeof(S));
  const int nu = (nbytes + 7) / 8;
  const bool rv = (flags & F_RECV) && ag.nrecv > 0;
  const uint4* src[2] = {nullptr, nullptr};
  uint32_t rflag[2] = {0u, 0u};
  if (rv)
    for (int i = 0; i < ag.nrecv; ++i) {
      src[i] = reinterpret_cast<const uint4*>(ag.slot(c, ag.re[i], ag.rstep[i]));
      rflag[i] = uint32_t(ag.rstep[i] + 1);
    }
  uint4* dst[2] = {nullptr, nullptr};
  uint32_t sflag[2] = {0u, 0u};
  if (flags & F_SEND)
    for (int i = 0; i < ag.nsend; ++i) {
      dst[i] = reinterpret_cast<uint4*>(ag.slot(c, ag.se[i], ag.sstep[i]));
      sflag[i] = uint32_t(ag.sstep[i] + 1);
    }

  bool fail = false;
  for (int u = threadIdx.x; u < nu && !fail; u += blockDim.x) {
    const int valid = min(8, nbytes - 8 * u);
    uint2 xv = make_uint2(0, 0);
    if (flags & F_IN) xv = loadUnit<S>(in + 8 * u, valid);
    uint32_t r[2][2] = {{0u, 0u}, {0u, 0u}};
    if (rv) {
      for (int i = 0; i < ag.nrecv && !fail; ++i) {
        Spin sp;
        uint4 line;
        do {
          line = ldVolatile16(src[i] + u);
          if (line.y == rflag[i] && line.w == rflag[i]) break;
          if (sp.tick(c, ag.rank, ag.ch, 2, ag.rstep[i] + 1)) {
            fail = true;
            break;
          }
        } while (true);
        r[i][0] = line.x;
        r[i][1] = line.z;
      }
      if (fail) break;
    }
    uint32_t x[2] = {xv.x, xv.y}, acc[2];
    reduceWords<DT, OP, TREE, 2>(acc, x, r[0], r[1], flags, ag.nrecv, a.scale, a.nranks);
    if (flags & F_SEND)
      for (int i = 0; i < ag.nsend; ++i) stVolatile16(dst[i] + u, make_uint4(acc[0], sflag[i], acc[1], sflag[i]));
    if (flags & F_OUT) storeUnit<S>(out + 8 * u, make_uint2(acc[0], acc[1]), valid);
  }
  if (__any_sync(0xffffffffu, fail)) return false;
  if (rv && !warpDoneReading(c, ag, kLL, lane)) return false;
  ag.advance(flags);
  return true;
}

// ------------------------------------------------------------------- LL128
// A 128-byte line is eight 16-byte pieces held by eight lanes of a warp; a
// warp moves U groups of four lines per pass. Pieces 0..6 carry 16 user
// bytes, piece 7 carries 8 user bytes and, in its upper half, the 8-byte
// flag (step + 1); line L of a slice carries user bytes [120 L, 120 L + 120).
//
// As in NCCL ("NCCL architecture ...", §7.2, LL128), a line is written by
// one warp store (its eight lanes' pieces, the flag in the same store) and
// read by one warp load, with no fence on either side: a reader that sees
// the flag trusts the rest of the line. NCCL gets that from NVLink writing
// a 128-byte line at once; here it rests on one GPU's memory system
// handling a warp's aligned 128-byte line access as a whole, which the PTX
// memory model does not promise but which a probe on this GPU never saw
// violated (3.1e9 piece loads of lines being rewritten concurrently,
// volatile and L2-only accesses, writer and reader on the same and on
// different dies: no torn 16-byte piece, no torn 128-byte line); the GPU
// tests stress it.
// a ? x : y as one selp (no branch on a per-lane condition)
__device__ __forceinline__ uint32_t selectWord(bool a, uint32_t x, uint32_t y) {
  uint32_t r;
  asm("{\n.reg .pred q;\nsetp.ne.u32 q, %1, 0;\nselp.b32 %0, %2, %3, q;\n}" : "=r"(r) : "r"(uint32_t(a)), "r"(x), "r"(y));
  return r;
}

template <int U, int DT, int OP, bool TREE, class Args>
__device__ __forceinline__ bool ll128Passes(const Args& a, Agent& ag, const char* in, char* out, int nbytes,
                                            int nlines, int flags, const char* const* src, char* const* dst) {
  using S = typename Ty<DT>::S;
  constexpr int NR = TREE ? 2 : 1;    // in-edges
  const DevComm& c = a.comm;
  const bool rv = (flags & F_RECV) && ag.nrecv > 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int p = lane & 7;     // piece of the line this lane moves
  const int k = lane >> 3;    // line within a group of four
  bool fail = false;
  // A pass covers lines g0 + 4u + k (u < U); lane p of group k moves piece
  // p of each of them.
  for (int g0 = warp * 4 * U; g0 < nlines; g0 += nwarps * 4 * U) {
    int ub[U], valid0[U], valid1[U];
    uint32_t x[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int line = g0 + 4 * u + k;
      const bool active = line < nlines;
      ub[u] = line * kLL128DataBytes + p * 16;  // first user byte of this piece
      valid0[u] = active ? max(0, min(8, nbytes - ub[u])) : 0;
      valid1[u] = (active && p < 7) ? max(0, min(8, nbytes - ub[u] - 8)) : 0;
      x[u][0] = x[u][1] = x[u][2] = x[u][3] = 0u;
      if ((flags & F_IN) && valid0[u] > 0) {
        const uint2 u0 = loadUnit<S>(in + ub[u], valid0[u]);
        x[u][0] = u0.x;
        x[u][1] = u0.y;
        if (valid1[u] > 0) {
          const uint2 u1 = loadUnit<S>(in + ub[u] + 8, valid1[u]);
          x[u][2] = u1.x;
          x[u][3] = u1.y;
        }
      }
    }
    uint32_t r[U][NR][4];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int i = 0; i < NR; ++i) r[u][i][0] = r[u][i][1] = r[u][i][2] = r[u][i][3] = 0u;
    if (rv) {
      // one warp load per group of four lines (all of each line at once);
      // the line is complete when its flag (lane 7's upper half) is the
      // step's, else that line is loaded again
      for (int i = 0; i < ag.nrecv && i < NR && !fail; ++i) {
        const uint32_t wlo = uint32_t(ag.rstep[i] + 1), whi = uint32_t((ag.rstep[i] + 1) >> 32);
        bool have[U];
#pragma unroll
        for (int u = 0; u < U; ++u) have[u] = g0 + 4 * u + k >= nlines;  // no such line: nothing to wait for
        Spin sp;
        while (true) {
          bool all = true;
#pragma unroll
          for (int u = 0; u < U; ++u) {
            // the eight lanes of a line load it together, in one instruction
            __syncwarp();
            uint4 v = make_uint4(0, 0, 0, 0);
            if (!have[u]) v = ldVolatile16(reinterpret_cast<const uint4*>(src[i] + size_t(g0 + 4 * u + k) * 128 + p * 16));
            const bool flagOk = p == 7 && v.z == wlo && v.w == whi;
            const bool lineOk = __shfl_sync(0xffffffffu, flagOk, (lane & ~7) | 7);
            if (!have[u] && lineOk) {
              r[u][i][0] = v.x; r[u][i][1] = v.y;
              r[u][i][2] = p < 7 ? v.z : 0u; r[u][i][3] = p < 7 ? v.w : 0u;
              have[u] = true;
            }
            all &= have[u];
          }
          if (__all_sync(0xffffffffu, all)) break;
          if (sp.tick(c, ag.rank, ag.ch, 3, ag.rstep[i] + 1)) fail = true;
          if (__any_sync(0xffffffffu, fail)) {
            fail = true;
            break;
          }
        }
      }
      if (fail) break;
    }
    uint32_t acc[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u)
      reduceWords<DT, OP, TREE, 4>(acc[u], x[u], r[u][0], r[u][NR - 1], flags, ag.nrecv, a.scale, a.nranks);
    if (flags & F_SEND) {
      // One warp store per group of four lines, the flag in lane 7's piece.
      // A line must leave in one instruction of its eight lanes: the words
      // are chosen without a branch (a branch on the lane could let the
      // compiler issue the flag lane's store apart from the others'), and
      // the warp is brought together right before each store.
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const bool active = g0 + 4 * u + k < nlines;
        for (int i = 0; i < ag.nsend; ++i) {
          const unsigned long long f = ag.sstep[i] + 1;
          const uint32_t w2 = selectWord(p < 7, acc[u][2], uint32_t(f));
          const uint32_t w3 = selectWord(p < 7, acc[u][3], uint32_t(f >> 32));
          __syncwarp();
          if (active)
            stVolatile16(reinterpret_cast<uint4*>(dst[i] + size_t(g0 + 4 * u + k) * 128 + p * 16),
                         make_uint4(acc[u][0], acc[u][1], w2, w3));
        }
      }
    }
    if (flags & F_OUT) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (valid0[u] > 0) storeUnit<S>(out + ub[u], make_uint2(acc[u][0], acc[u][1]), valid0[u]);
        if (valid1[u] > 0) storeUnit<S>(out + ub[u] + 8, make_uint2(acc[u][2], acc[u][3]), valid1[u]);
      }
    }
  }
  return !fail;
}

// One LL128 slice. Every warp works on its own: it waits for the out-edges'
// credit itself (lane 0 polls the head, caching it), and the last warp
// done reading the slice returns the slot(s) to the sender; no CTA-wide
// barrier per slice. A warp can run ahead of another by fewer than
// VRCCL_STEPS slices (reading a slot's next use needs the sender to have
// seen the slot returned), so one counter per slot tells when a use is done.
template <int U, int DT, int OP, bool TREE, class Args>
__device__ bool llSlice128(const Args& a, Agent& ag, const char* in, char* out, int nelem, int flags) {
  using S = typename Ty<DT>::S;
  const DevComm& c = a.comm;
  const int lane = threadIdx.x & 31;
  if (!warpCredit(c, ag, flags, kLL128)) return false;
  const int nbytes = nelem * int(sizeof(S));
  const int nlines = (nbytes + kLL128DataBytes - 1) / kLL128DataBytes;
  const bool rv = (flags & F_RECV) && ag.nrecv > 0;
  const char* src[2] = {nullptr, nullptr};
  if (rv)
    for (int i = 0; i < ag.nrecv; ++i) src[i] = ag.slot(c, ag.re[i], ag.rstep[i]);
  char* dst[2] = {nullptr, nullptr};
  if (flags & F_SEND)
    for (int i = 0; i < ag.nsend; ++i) dst[i] = ag.slot(c, ag.se[i], ag.sstep[i]);
  // U = 4 (the wide kernels, for long slices): more loads and flags in
  // flight per warp; U = 1: the shortest chain per line. The two live in
  // different kernels: the four-group code in the same kernel measured
  // slower on short slices (ring LL128, bf16 16 KiB: 37 -> 49 us).
  if (!ll128Passes<U, DT, OP, TREE>(a, ag, in, out, nbytes, nlines, flags, src, dst)) return false;
  if (rv && !warpDoneReading(c, ag, kLL128, lane)) return false;
  ag.advance(flags);
  return true;
}

template <int PROTO, int DT, int OP, bool TREE, class Args>
__device__ __forceinline__ bool runSlice(const Args& a, Agent& ag, const char* in, char* out, int nelem,
                                         int flags) {
  if constexpr (PROTO == kLL) return llSlice<DT, OP, TREE>(a, ag, in, out, nelem, flags);
  if constexpr (PROTO == kLL128) return llSlice128<1, DT, OP, TREE>(a, ag, in, out, nelem, flags);
  if constexpr (PROTO == kLL128Wide) return llSlice128<4, DT, OP, TREE>(a, ag, in, out, nelem, flags);
}

}  // namespace vrccl
