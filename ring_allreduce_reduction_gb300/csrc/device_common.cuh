// Device-side building blocks: memory-model primitives, bounded waits and
// the element arithmetic of one reduction step.
//
// All parties of a FIFO are agents of one kernel on one GPU, so gpu-scope
// release/acquire is enough where NCCL uses system-scope fences between
// GPUs ("NCCL architecture: topology, channels, algorithms and protocols",
// §7.2, Simple: fence_acq_rel_sys then the tail store).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>
#include <type_traits>

#include "vrccl_internal.h"

namespace vrccl {

// ------------------------------------------------------------ memory model

__device__ __forceinline__ unsigned long long ldAcquire(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ldRelaxed(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void stRelaxed(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void stRelease(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void fenceAcqRelGpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ unsigned long long globalTimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// LL line access: one 16-byte volatile access carries data and flags
// together ("NCCL architecture ...", §7.2, LL).
__device__ __forceinline__ uint4 ldVolatile16(const uint4* p) {
  uint4 v;
  asm volatile("ld.volatile.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ void stVolatile16(uint4* p, uint4 v) {
  asm volatile("st.volatile.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Streaming user data (read once / written once) and L2-resident FIFO data.
__device__ __forceinline__ uint4 ldStream16(const void* p) { return __ldcs(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ void stStream16(void* p, uint4 v) { __stcs(reinterpret_cast<uint4*>(p), v); }
__device__ __forceinline__ uint4 ldFifo16(const void* p) { return __ldcg(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ void stFifo16(void* p, uint4 v) { __stcg(reinterpret_cast<uint4*>(p), v); }
// A FIFO store under an L2 policy (evictLastPolicy below): the slot stays in
// L2 until its receiver has read and dropped it.
__device__ __forceinline__ void stFifoHint16(void* p, uint4 v, unsigned long long policy) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w), "l"(policy)
               : "memory");
}
__device__ __forceinline__ uint2 ldStream8(const void* p) { return __ldcs(reinterpret_cast<const uint2*>(p)); }
__device__ __forceinline__ void stStream8(void* p, uint2 v) { __stcs(reinterpret_cast<uint2*>(p), v); }
__device__ __forceinline__ uint2 ldFifo8(const void* p) { return __ldcg(reinterpret_cast<const uint2*>(p)); }
__device__ __forceinline__ void stFifo8(void* p, uint2 v) { __stcg(reinterpret_cast<uint2*>(p), v); }

// ------------------------------------------------------------ mbarrier + bulk copy
// Shared-memory barriers with transaction counts and the non-tensor bulk
// copy engine (TMA): one thread moves a whole FIFO slot or input slice
// into shared memory and the barrier completes when the bytes have landed.

__device__ __forceinline__ uint32_t smemAddr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbarInit(unsigned long long* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smemAddr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbarExpectTx(unsigned long long* bar, unsigned bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smemAddr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbarArrive(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smemAddr(bar)) : "memory");
}
// true once the phase of the given parity has completed
__device__ __forceinline__ bool mbarTryWait(unsigned long long* bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(smemAddr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// global -> shared bulk copy; bytes and both addresses multiples of 16
__device__ __forceinline__ void bulkLoad(void* dstSmem, const void* srcGlobal, unsigned bytes,
                                         unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smemAddr(dstSmem)),
      "l"(srcGlobal), "r"(bytes), "r"(smemAddr(bar))
      : "memory");
}
// The same copy, tagged to be evicted from L2 first: for data read once
// (an agent's own input), so it does not push out FIFO lines that are still
// to be read.
__device__ __forceinline__ unsigned long long evictLastPolicy() {
  unsigned long long pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ unsigned long long evictFirstPolicy() {
  unsigned long long pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void bulkLoadOnce(void* dstSmem, const void* srcGlobal, unsigned bytes,
                                             unsigned long long* bar, unsigned long long policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smemAddr(dstSmem)),
      "l"(srcGlobal), "r"(bytes), "r"(smemAddr(bar)), "l"(policy)
      : "memory");
}
// Starts pulling a global range into L2 (no destination in this SM).
__device__ __forceinline__ void bulkPrefetchL2(const void* srcGlobal, unsigned bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(srcGlobal), "r"(bytes) : "memory");
}
// Orders this thread's earlier generic-proxy accesses (the flag acquire)
// before its later async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fenceProxyAsync() { asm volatile("fence.proxy.async;" ::: "memory"); }

__device__ __forceinline__ unsigned atomAddAcqRelCta(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(smemAddr(p)), "r"(v)
               : "memory");
  return old;
}
// Drops a 128-byte L2 line without writing it back: for a FIFO slot whose
// contents have been consumed and will be rewritten by its sender.
__device__ __forceinline__ void discardL2(const void* p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}
__device__ __forceinline__ void redMaxRelaxed(unsigned long long* p, unsigned long long v) {
  asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// ------------------------------------------------------------ bounded waits

// Records the first failure of the launch and raises the device abort word.
__device__ __forceinline__ void recordFailure(const DevComm& c, int code, int rank, int ch, int kind,
                                              unsigned long long step) {
  if (atomicCAS(&c.status->code, 0, code) == 0) {
    c.status->rank = rank;
    c.status->channel = ch;
    c.status->kind = kind;
    c.status->step = step;
  }
  __threadfence();
  atomicExch(c.devAbort, 1);
}

// One spinning thread's budget. Every `mask+1` polls it reads the clock;
// the abort words (one of them in host memory, a slow read) and the
// timeout are checked only when at least kCheckNs have passed since the last
// check, so a waiter is rarely stuck in a slow read when its flag arrives.
// Past the communicator's timeout it records vrcclTimeout.
struct Spin {
  static constexpr unsigned long long kCheckNs = 50000;
  unsigned long long t0, last;
  unsigned n;
  unsigned mask;
  __device__ __forceinline__ Spin(unsigned mask_ = 255u) : t0(0), last(0), n(0), mask(mask_) {}
  // true = give up
  __device__ __forceinline__ bool tick(const DevComm& c, int rank, int ch, int kind, unsigned long long step) {
    if ((++n & mask) != 0) return false;
    const unsigned long long now = globalTimer();
    if (t0 == 0) {
      t0 = last = now;
      return false;
    }
    if (now - last < kCheckNs) return false;
    last = now;
    if (*reinterpret_cast<volatile int*>(c.devAbort)) return true;
    if (*c.hostAbort) {
      recordFailure(c, vrcclAborted, rank, ch, kind, step);
      return true;
    }
    if (now - t0 > c.timeoutNs) {
      recordFailure(c, vrcclTimeout, rank, ch, kind, step);
      return true;
    }
    return false;
  }
};

// Wait until *p >= v (acquire). false = gave up.
__device__ __forceinline__ bool waitGE(const unsigned long long* p, unsigned long long v, const DevComm& c,
                                       int rank, int ch, int kind) {
  Spin s;
  while (ldAcquire(p) < v) {
    if (s.tick(c, rank, ch, kind, v)) return false;
  }
  return true;
}

__device__ __forceinline__ bool aborted(const DevComm& c) {
  return *reinterpret_cast<volatile int*>(c.devAbort) != 0 || *c.hostAbort != 0;
}

// ------------------------------------------------------------ element types

template <int DT> struct Ty;
template <> struct Ty<vrcclInt32> {
  using S = int32_t;
  static constexpr bool kFloat = false;
};
template <> struct Ty<vrcclInt8> {
  using S = int8_t;
  static constexpr bool kFloat = false;
};
template <> struct Ty<vrcclUint8> {
  using S = uint8_t;
  static constexpr bool kFloat = false;
};
template <> struct Ty<vrcclInt64> {
  using S = long long;
  static constexpr bool kFloat = false;
};
template <> struct Ty<vrcclFloat32> {
  using S = float;
  static constexpr bool kFloat = true;
  __device__ static __forceinline__ float toF(float x) { return x; }
  __device__ static __forceinline__ float fromF(float x) { return x; }
};
template <> struct Ty<vrcclBfloat16> {
  using S = unsigned short;
  static constexpr bool kFloat = true;
  __device__ static __forceinline__ float toF(unsigned short x) { return __bfloat162float(__ushort_as_bfloat16(x)); }
  __device__ static __forceinline__ unsigned short fromF(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  }
};
template <> struct Ty<vrcclFloat16> {
  using S = unsigned short;
  static constexpr bool kFloat = true;
  __device__ static __forceinline__ float toF(unsigned short x) { return __half2float(__ushort_as_half(x)); }
  __device__ static __forceinline__ unsigned short fromF(float x) { return __half_as_ushort(__float2half_rn(x)); }
};
// float64 computes in binary64 itself (no widening type).
template <> struct Ty<vrcclFloat64> {
  using S = double;
  static constexpr bool kFloat = true;
};

// One reduction step op(a, b); a is the running value. 2- and 4-byte
// floating types: the op in binary32 without contraction, then one rounding
// to the type; float64: the op in binary64. max and min keep `a` on a tie.
// Integer sum/prod wrap modulo 2^bits (computed in the unsigned type of the
// same width); max/min compare in the type (uint8 unsigned).
template <int DT, int OP>
__device__ __forceinline__ typename Ty<DT>::S combine(typename Ty<DT>::S a, typename Ty<DT>::S b) {
  using S = typename Ty<DT>::S;
  if constexpr (!Ty<DT>::kFloat) {
    using U = std::make_unsigned_t<S>;
    if constexpr (OP == vrcclSum || OP == vrcclAvg) return S(U(U(a) + U(b)));
    if constexpr (OP == vrcclProd) return S(U(U(a) * U(b)));
    if constexpr (OP == vrcclMax) return b > a ? b : a;
    if constexpr (OP == vrcclMin) return b < a ? b : a;
  } else if constexpr (DT == vrcclFloat64) {
    if constexpr (OP == vrcclSum || OP == vrcclAvg) return __dadd_rn(a, b);
    if constexpr (OP == vrcclProd) return __dmul_rn(a, b);
    if constexpr (OP == vrcclMax) return b > a ? b : a;
    if constexpr (OP == vrcclMin) return b < a ? b : a;
  } else {
    float fa = Ty<DT>::toF(a), fb = Ty<DT>::toF(b);
    if constexpr (OP == vrcclSum || OP == vrcclAvg) return Ty<DT>::fromF(__fadd_rn(fa, fb));
    if constexpr (OP == vrcclProd) return Ty<DT>::fromF(__fmul_rn(fa, fb));
    if constexpr (OP == vrcclMax) return fb > fa ? b : a;
    if constexpr (OP == vrcclMin) return fb < fa ? b : a;
  }
}

// What a rank feeds into the reduction for its own element (avg scale):
// the binary32 1/n for the 2- and 4-byte floating types, the binary64 1/n
// for float64.
template <int DT, int OP>
__device__ __forceinline__ typename Ty<DT>::S prescale(typename Ty<DT>::S x, float scale, int n) {
  if constexpr (OP == vrcclAvg && DT == vrcclFloat64) {
    return __dmul_rn(x, 1.0 / double(n));
  } else if constexpr (OP == vrcclAvg && Ty<DT>::kFloat) {
    return Ty<DT>::fromF(__fmul_rn(Ty<DT>::toF(x), scale));
  } else {
    return x;
  }
}

// Applied where a chunk becomes final: integer avg divides, truncating
// toward zero (C++ integer division).
template <int DT, int OP>
__device__ __forceinline__ typename Ty<DT>::S postop(typename Ty<DT>::S x, int n) {
  using S = typename Ty<DT>::S;
  if constexpr (OP == vrcclAvg && !Ty<DT>::kFloat) return S(x / n);
  return x;
}

// ------------------------------------------------------------ packed words
// Data moves as 32-bit words. A word holds one 4-byte element, two 2-byte
// elements or four 1-byte elements (element 0 in the low bits, as they sit
// in memory); an 8-byte element spans two consecutive words (low word
// first). The word-array forms below take NW words whose boundaries are
// element boundaries.

__device__ __forceinline__ int32_t fromWord(uint32_t w, int32_t*) { return int32_t(w); }
__device__ __forceinline__ float fromWord(uint32_t w, float*) { return __uint_as_float(w); }
__device__ __forceinline__ uint32_t toWord(int32_t x) { return uint32_t(x); }
__device__ __forceinline__ uint32_t toWord(float x) { return __float_as_uint(x); }

template <typename S>
__device__ __forceinline__ S fromPair(uint32_t lo, uint32_t hi) {
  const unsigned long long v = (unsigned long long)lo | ((unsigned long long)hi << 32);
  S x;
  memcpy(&x, &v, 8);
  return x;
}
template <typename S>
__device__ __forceinline__ void toPair(S x, uint32_t& lo, uint32_t& hi) {
  unsigned long long v;
  memcpy(&v, &x, 8);
  lo = uint32_t(v);
  hi = uint32_t(v >> 32);
}

// Two 2-byte sums in one instruction. For bf16 and fp16 the binary32 sum
// of two values of the type is either exact or differs from the exact sum
// by far less than half a unit of the type, so one correctly rounded
// (round-to-nearest-even) packed add gives the same bits as "binary32 add,
// then round to the type".
__device__ __forceinline__ uint32_t addBf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t addF16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// op on the elements of one word (not for 8-byte types).
template <int DT, int OP>
__device__ __forceinline__ uint32_t combineWord(uint32_t a, uint32_t b) {
  using S = typename Ty<DT>::S;
  static_assert(sizeof(S) <= 4, "8-byte elements span two words");
  if constexpr (sizeof(S) == 4) {
    return toWord(combine<DT, OP>(fromWord(a, (S*)nullptr), fromWord(b, (S*)nullptr)));
  } else if constexpr ((OP == vrcclSum || OP == vrcclAvg) && DT == vrcclBfloat16) {
    return addBf16x2(a, b);
  } else if constexpr ((OP == vrcclSum || OP == vrcclAvg) && DT == vrcclFloat16) {
    return addF16x2(a, b);
  } else if constexpr (sizeof(S) == 2) {
    uint32_t lo = combine<DT, OP>(S(a & 0xffffu), S(b & 0xffffu));
    uint32_t hi = combine<DT, OP>(S(a >> 16), S(b >> 16));
    return lo | (hi << 16);
  } else if constexpr (OP == vrcclSum || OP == vrcclAvg) {
    return __vadd4(a, b);  // four byte sums modulo 2^8, no carry between bytes
  } else if constexpr (OP == vrcclMax) {
    return DT == vrcclInt8 ? __vmaxs4(a, b) : __vmaxu4(a, b);
  } else if constexpr (OP == vrcclMin) {
    return DT == vrcclInt8 ? __vmins4(a, b) : __vminu4(a, b);
  } else {
    uint32_t d = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) d |= (((a >> (8 * i)) * (b >> (8 * i))) & 0xffu) << (8 * i);
    return d;
  }
}
template <int DT, int OP>
__device__ __forceinline__ uint32_t prescaleWord(uint32_t a, float scale) {
  using S = typename Ty<DT>::S;
  static_assert(sizeof(S) <= 4, "8-byte elements span two words");
  if constexpr (!(OP == vrcclAvg && Ty<DT>::kFloat)) {
    return a;
  } else if constexpr (sizeof(S) == 4) {
    return toWord(prescale<DT, OP>(fromWord(a, (S*)nullptr), scale, 1));
  } else {
    // binary32 products, then both rounded (to nearest even) by one packed
    // conversion; the high half of the word is the second element.
    const float lo = __fmul_rn(Ty<DT>::toF(S(a & 0xffffu)), scale);
    const float hi = __fmul_rn(Ty<DT>::toF(S(a >> 16)), scale);
    uint32_t d;
    if constexpr (DT == vrcclBfloat16)
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    else
      asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
  }
}
template <int DT, int OP>
__device__ __forceinline__ uint32_t postopWord(uint32_t a, int n) {
  using S = typename Ty<DT>::S;
  static_assert(sizeof(S) <= 4, "8-byte elements span two words");
  if constexpr (!(OP == vrcclAvg && !Ty<DT>::kFloat)) {
    return a;
  } else if constexpr (sizeof(S) == 4) {
    return uint32_t(int32_t(a) / n);
  } else {
    uint32_t d = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) d |= (uint32_t(uint8_t(postop<DT, OP>(S(a >> (8 * i)), n)))) << (8 * i);
    return d;
  }
}

// The same three steps on NW words (whole elements).
template <int DT, int OP, int NW>
__device__ __forceinline__ void combineWords(uint32_t (&a)[NW], const uint32_t (&b)[NW]) {
  using S = typename Ty<DT>::S;
  if constexpr (sizeof(S) == 8) {
#pragma unroll
    for (int w = 0; w < NW; w += 2)
      toPair(combine<DT, OP>(fromPair<S>(a[w], a[w + 1]), fromPair<S>(b[w], b[w + 1])), a[w], a[w + 1]);
  } else {
#pragma unroll
    for (int w = 0; w < NW; ++w) a[w] = combineWord<DT, OP>(a[w], b[w]);
  }
}
template <int DT, int OP, int NW>
__device__ __forceinline__ void prescaleWords(uint32_t (&a)[NW], float scale, int n) {
  using S = typename Ty<DT>::S;
  if constexpr (sizeof(S) == 8) {
#pragma unroll
    for (int w = 0; w < NW; w += 2) toPair(prescale<DT, OP>(fromPair<S>(a[w], a[w + 1]), scale, n), a[w], a[w + 1]);
  } else {
#pragma unroll
    for (int w = 0; w < NW; ++w) a[w] = prescaleWord<DT, OP>(a[w], scale);
  }
}
template <int DT, int OP, int NW>
__device__ __forceinline__ void postopWords(uint32_t (&a)[NW], int n) {
  using S = typename Ty<DT>::S;
  if constexpr (sizeof(S) == 8) {
#pragma unroll
    for (int w = 0; w < NW; w += 2) toPair(postop<DT, OP>(fromPair<S>(a[w], a[w + 1]), n), a[w], a[w + 1]);
  } else {
#pragma unroll
    for (int w = 0; w < NW; ++w) a[w] = postopWord<DT, OP>(a[w], n);
  }
}

}  // namespace vrccl
