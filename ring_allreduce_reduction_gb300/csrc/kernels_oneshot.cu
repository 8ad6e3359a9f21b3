// One-shot AllReduce: every output element is made in one pass from all n
// inputs and stored to all n recv buffers. No FIFO, no flags, no agent ever
// waits on another, so it moves exactly the essential bytes (n inputs read,
// n outputs written) and runs at the HBM roofline. It is the bound the ring
// is measured against.
//
// The association is the ring's: an element of ring chunk j (under the
// ring's channel partition and loop chunking for the same channel count C
// and chunk K, "NCCL Source Code Deep Dive", §2.2-§2.3) is folded as
//   op(...op(op(x[j+1], x[j+2]), x[j+3])..., x[j])     (ranks mod n)
// with the same avg pre-scale and int32 avg post-op, so for one (C, K) the
// two algorithms give identical bits.
#include "device_common.cuh"

namespace vrccl {

constexpr int kOneShotThreads = 512;
constexpr int kOneShotUnroll = 4;  // 16-byte vectors per thread per tile

struct ChunkPos {
  int j;                   // ring chunk (0..n-1) of the element
  unsigned long long end;  // first element past that chunk
};

// Ring chunk of element idx: channel parts of alignUp(ceil(count/C), A),
// loops of n*K, and a last loop of n chunks of alignUp(ceil(rem/n), A).
__device__ __forceinline__ ChunkPos ringChunkOf(unsigned long long idx, unsigned long long count, int n, int C,
                                                unsigned long long K, unsigned long long A) {
  const unsigned long long part = ((count + C - 1) / C + A - 1) / A * A;
  const unsigned long long chLo = idx / part * part;
  const unsigned long long chHi = min(count, chLo + part);
  const unsigned long long within = idx - chLo;
  const unsigned long long loop = (unsigned long long)n * K;
  const unsigned long long loopOff = within / loop * loop;
  const unsigned long long rem = chHi - chLo - loopOff;
  const unsigned long long k = rem >= loop ? K : ((rem + n - 1) / n + A - 1) / A * A;
  const unsigned long long j = (within - loopOff) / k;
  ChunkPos p;
  p.j = (int)j;
  p.end = min(chHi, chLo + loopOff + (j + 1) * k);
  return p;
}

template <int DT, int OP>
__global__ void __launch_bounds__(kOneShotThreads) oneShotKernel(const __grid_constant__ KArgs a) {
  using S = typename Ty<DT>::S;
  constexpr int E = sizeof(S);
  constexpr int V = 16 / E;
  constexpr int G = 8;  // loads issued together per fold group
  const int n = a.nranks;
  const unsigned long long count = a.count;
  const unsigned long long nvec = count / V;
  const unsigned long long K = (unsigned long long)a.chunkElems;
  const unsigned long long tile = (unsigned long long)blockDim.x * kOneShotUnroll;

  for (unsigned long long t0 = blockIdx.x * tile; t0 < nvec; t0 += (unsigned long long)gridDim.x * tile) {
    ChunkPos cp = ringChunkOf(t0 * V, count, n, a.nchannels, K, V);
#pragma unroll
    for (int u = 0; u < kOneShotUnroll; ++u) {
      const unsigned long long vi = t0 + (unsigned long long)u * blockDim.x + threadIdx.x;
      if (vi >= nvec) break;
      const unsigned long long e = vi * V;
      if (e >= cp.end) cp = ringChunkOf(e, count, n, a.nchannels, K, V);
      int rk = cp.j + 1 == n ? 0 : cp.j + 1;
      uint4 v0 = ldStream16(reinterpret_cast<const char*>(a.send[rk]) + e * E);
      uint32_t acc[4] = {v0.x, v0.y, v0.z, v0.w};
      prescaleWords<DT, OP, 4>(acc, a.scale, n);
      int left = n - 1;
      while (left > 0) {
        const int g = left < G ? left : G;
        uint4 v[G];
        int q = rk;
#pragma unroll
        for (int i = 0; i < G; ++i) {
          if (i < g) {
            q = q + 1 == n ? 0 : q + 1;
            v[i] = ldStream16(reinterpret_cast<const char*>(a.send[q]) + e * E);
          }
        }
#pragma unroll
        for (int i = 0; i < G; ++i) {
          if (i < g) {
            uint32_t b[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            prescaleWords<DT, OP, 4>(b, a.scale, n);
            combineWords<DT, OP, 4>(acc, b);
          }
        }
        rk = q;
        left -= g;
      }
      postopWords<DT, OP, 4>(acc, n);
      const uint4 out = make_uint4(acc[0], acc[1], acc[2], acc[3]);
      for (int r = 0; r < n; ++r) stStream16(reinterpret_cast<char*>(a.recv[r]) + e * E, out);
    }
  }

  // The ragged end (fewer than 16 bytes past the last whole vector).
  if (blockIdx.x == 0) {
    const unsigned long long idx = nvec * V + threadIdx.x;
    if (threadIdx.x < V && idx < count) {
      const int j = ringChunkOf(idx, count, n, a.nchannels, K, V).j;
      int rk = j + 1 == n ? 0 : j + 1;
      S acc = prescale<DT, OP>(reinterpret_cast<const S*>(a.send[rk])[idx], a.scale, n);
      for (int i = 1; i < n; ++i) {
        rk = rk + 1 == n ? 0 : rk + 1;
        acc = combine<DT, OP>(acc, prescale<DT, OP>(reinterpret_cast<const S*>(a.send[rk])[idx], a.scale, n));
      }
      acc = postop<DT, OP>(acc, n);
      for (int r = 0; r < n; ++r) reinterpret_cast<S*>(a.recv[r])[idx] = acc;
    }
  }
}

#define VRCCL_ONESHOT_ROW(DT)                                                                            \
  {(const void*)oneShotKernel<DT, 0>, (const void*)oneShotKernel<DT, 1>, (const void*)oneShotKernel<DT, 2>, \
   (const void*)oneShotKernel<DT, 3>, (const void*)oneShotKernel<DT, 4>}

extern const void* const kOneShot[vrcclNumTypes][5] = {
    VRCCL_ONESHOT_ROW(0), VRCCL_ONESHOT_ROW(1), VRCCL_ONESHOT_ROW(2), VRCCL_ONESHOT_ROW(3),
    VRCCL_ONESHOT_ROW(4), VRCCL_ONESHOT_ROW(5), VRCCL_ONESHOT_ROW(6), VRCCL_ONESHOT_ROW(7)};

}  // namespace vrccl
