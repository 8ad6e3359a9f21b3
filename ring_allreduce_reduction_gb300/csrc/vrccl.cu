// Host side of libvrccl: communicator lifecycle, argument checks, schedule
// choice and the single cooperative launch per AllReduce.
//
// Sources cited: "NCCL Source Code Deep Dive: A GPU Journey of One
// AllReduce" (Deep Dive) and "NCCL architecture: topology, channels,
// algorithms and protocols" (Architecture).
#include <cuda_runtime.h>
#include <unistd.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <sys/syscall.h>
#include <utility>
#include <vector>

#include "model.h"
#include "parse.h"
#include "tuner.h"
#include "vrccl_internal.h"

using namespace vrccl;

namespace vrccl {
// Types 0-3 and 4-7 of the two largest tables live in separate translation
// units (compile time).
extern const void* const kRingSimple[4][5];
extern const void* const kTreeSimple[4][5];
extern const void* const kRingSimpleX[4][5];
extern const void* const kTreeSimpleX[4][5];
extern const void* const kRingLL[vrcclNumTypes][5];
extern const void* const kTreeLL[vrcclNumTypes][5];
extern const void* const kRingLL128[vrcclNumTypes][5];
extern const void* const kTreeLL128[vrcclNumTypes][5];
extern const void* const kRingLL128W[4][5];
extern const void* const kTreeLL128W[4][5];
extern const void* const kRingLL128WX[4][5];
extern const void* const kTreeLL128WX[4][5];
extern const void* const kOneShot[vrcclNumTypes][5];
extern const void* const kGroupSimple[vrcclNumTypes][5];
extern const void* const kGroupLL[vrcclNumTypes][5];
extern const void* const kGroupLL128[vrcclNumTypes][5];

const void* groupKernelFor(int proto, int dtype, int op) {
  if (dtype < 0 || dtype >= vrcclNumTypes || op < 0 || op >= 5) return nullptr;
  switch (proto) {
    case kSimple: return kGroupSimple[dtype][op];
    case kLL: return kGroupLL[dtype][op];
    case kLL128: return kGroupLL128[dtype][op];
  }
  return nullptr;
}

int maxDynamicSmem(const void* fn, int device) {
  int optin = 0;
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return optin - int(fa.sharedSizeBytes);
}

const void* kernelFor(int algo, int proto, int dtype, int op) {
  if (dtype < 0 || dtype >= vrcclNumTypes || op < 0 || op >= 5) return nullptr;
  const bool x = dtype >= 4;  // the second half of a split table
  const int d = dtype & 3;
  switch (proto * 2 + algo) {
    case kSimple * 2 + kRing: return x ? kRingSimpleX[d][op] : kRingSimple[d][op];
    case kSimple * 2 + kTree: return x ? kTreeSimpleX[d][op] : kTreeSimple[d][op];
    case kLL * 2 + kRing: return kRingLL[dtype][op];
    case kLL * 2 + kTree: return kTreeLL[dtype][op];
    case kLL128 * 2 + kRing: return kRingLL128[dtype][op];
    case kLL128 * 2 + kTree: return kTreeLL128[dtype][op];
    case kLL128Wide * 2 + kRing: return x ? kRingLL128WX[d][op] : kRingLL128W[d][op];
    case kLL128Wide * 2 + kTree: return x ? kTreeLL128WX[d][op] : kTreeLL128W[d][op];
  }
  return nullptr;
}
}  // namespace vrccl

// Sentinels at both ends of the communicator, as ncclComm's startMagic /
// endMagic (Deep Dive §2.1): a stale or foreign handle fails the check.
static constexpr uint64_t kMagic = 0x5652434331474233ull;  // "VRCC1GB3"

// A validated collective call. AllReduce: count = elements per rank.
// ReduceScatter / AllGather: count = elements per block.
struct Call {
  int coll, dtype, op, algo, proto;
  size_t count;
  std::vector<const void*> send;
  std::vector<void*> recv;
  vrcclStream_t stream;
};

struct GroupSched {
  int algo, proto, channels;
  size_t chunk;
  int launch;  // order of the launch that ran the call within its group
};

struct vrcclComm {
  uint64_t startMagic;
  int device;
  int nranks;
  int maxChannels;
  int smCount;
  DevComm dc;
  void* fifoAlloc[kNumProtos];
  void* ctrlAlloc;
  void* statusAlloc;  // DevStatus + devAbort word
  int* hostAbortPinned;
  cudaStream_t internal;
  bool failed;
  bool aborted;
  // schedule
  int forceChannels;
  size_t forceChunkBytes;
  // VRCCL_ALGO / VRCCL_PROTO per collective (index CollId): algorithms
  // (bit kRing, bit kTree) and protocols (bits kSimple, kLL, kLL128) "auto"
  // may choose.
  unsigned envAlgoMask[3], envProtoMask[3];
  int envChannels;
  size_t envSliceBytes;
  int envWarps, envPrefetch;
  bool direct;  // Simple ring AllReduce: all-gather through the recv buffers
  bool debug;
  bool haveLast;
  int lastAlgo, lastProto, lastChannels;
  size_t lastChunk;
  int lastSlice, lastThreads, lastBlocks;
  // LL / LL128 flags are the low bits of a growing step count: an upper
  // bound of the steps issued so far decides when to clear the FIFOs.
  unsigned long long llStepBound[kNumProtos];
  Tuner tuner;
  std::vector<Call> pending;            // calls registered inside a group
  std::vector<GroupSched> groupSched;   // per call of the last group: what ran
  int groupLaunches;                    // launches made by the last group
  uint64_t endMagic;
};

static std::mutex gLiveMu;
static std::vector<vrcclComm*> gLive;  // communicators not yet destroyed

static bool validComm(const vrcclComm* c) {
  return c && c->startMagic == kMagic && c->endMagic == kMagic;
}

static int envInt(const char* name, int dflt) {
  const char* v = getenv(name);
  if (!v || !*v) return dflt;
  return atoi(v);
}

// VRCCL_ALGO / VRCCL_PROTO (NCCL's parseList syntax) -> per-collective
// masks in this library's ids; false for a string with an unknown name.
static bool envMasks(unsigned algoMask[3], unsigned protoMask[3]) {
  unsigned a[kNumParseFuncs], p[kNumParseFuncs];
  if (parseList(getenv("VRCCL_ALGO"), kParseAlgo, a) != 0) return false;
  if (parseList(getenv("VRCCL_PROTO"), kParseProto, p) != 0) return false;
  static const int kFn[3] = {kFnAllReduce, kFnReduceScatter, kFnAllGather};  // by CollId
  for (int c = 0; c < 3; ++c) {
    const unsigned am = a[kFn[c]], pm = p[kFn[c]];
    algoMask[c] = ((am >> 1) & 1u) << kRing | (am & 1u) << kTree;          // NCCL: Tree bit 0, Ring bit 1
    protoMask[c] = (pm & 1u) << kLL | ((pm >> 1) & 1u) << kLL128 | ((pm >> 2) & 1u) << kSimple;
  }
  return true;
}

static const char* kAlgoName[4] = {"Ring", "Tree", "Auto", "OneShot"};
static const char* kProtoName[3] = {"Simple", "LL", "LL128"};
static const size_t kElemSize[vrcclNumTypes] = {4, 4, 2, 2, 1, 1, 8, 8};

static size_t fifoBytes(int proto, int nranks, int maxCh) {
  return size_t(3) * maxCh * nranks * kSteps * slotBufferBytes(proto);
}

extern "C" const char* vrcclGetErrorString(vrcclResult_t r) {
  switch (r) {
    case vrcclSuccess: return "no error";
    case vrcclInvalidArgument: return "invalid argument";
    case vrcclInvalidUsage: return "invalid usage";
    case vrcclInternalError: return "internal error";
    case vrcclCudaError: return "CUDA error";
    case vrcclTimeout: return "device wait timed out";
    case vrcclAborted: return "communicator aborted";
    default: return "unknown result code";
  }
}

static void freeComm(vrcclComm* c) {
  {
    std::lock_guard<std::mutex> lk(gLiveMu);
    gLive.erase(std::remove(gLive.begin(), gLive.end(), c), gLive.end());
  }
  for (int p = 0; p < kNumProtos; ++p)
    if (c->fifoAlloc[p]) cudaFree(c->fifoAlloc[p]);
  if (c->ctrlAlloc) cudaFree(c->ctrlAlloc);
  if (c->statusAlloc) cudaFree(c->statusAlloc);
  if (c->hostAbortPinned) cudaFreeHost(c->hostAbortPinned);
  if (c->internal) cudaStreamDestroy(c->internal);
  c->startMagic = c->endMagic = 0;
  delete c;
}

extern "C" vrcclResult_t vrcclCommInit(vrcclComm_t* comm, int nranks, int nchannels) {
  if (!comm) return vrcclInvalidArgument;
  *comm = nullptr;
  if (nranks < 1 || nranks > kMaxRanks || nchannels < 1 || nchannels > VRCCL_MAX_CHANNELS)
    return vrcclInvalidArgument;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return vrcclCudaError;
  vrcclComm* c = new vrcclComm();
  memset(static_cast<void*>(c), 0, sizeof(*c));
  new (&c->tuner) Tuner();
  new (&c->pending) std::vector<Call>();
  new (&c->groupSched) std::vector<GroupSched>();
  c->startMagic = c->endMagic = kMagic;
  c->device = dev;
  c->nranks = nranks;
  c->maxChannels = nchannels;
  cudaDeviceGetAttribute(&c->smCount, cudaDevAttrMultiProcessorCount, dev);
  const size_t nEdges = size_t(3) * nchannels * nranks;
  bool ok = true;
  for (int p = 0; p < kNumProtos && ok; ++p) {
    ok = cudaMalloc(&c->fifoAlloc[p], fifoBytes(p, nranks, nchannels)) == cudaSuccess &&
         cudaMemset(c->fifoAlloc[p], 0, fifoBytes(p, nranks, nchannels)) == cudaSuccess;
  }
  // one control block per edge and protocol, then one per edge for the
  // direct all-gather counters
  ok = ok && cudaMalloc(&c->ctrlAlloc, nEdges * (kNumProtos + 1) * sizeof(EdgeCtrl)) == cudaSuccess &&
       cudaMemset(c->ctrlAlloc, 0, nEdges * (kNumProtos + 1) * sizeof(EdgeCtrl)) == cudaSuccess;
  ok = ok && cudaMalloc(&c->statusAlloc, 256) == cudaSuccess && cudaMemset(c->statusAlloc, 0, 256) == cudaSuccess;
  ok = ok && cudaHostAlloc((void**)&c->hostAbortPinned, 64, cudaHostAllocMapped) == cudaSuccess;
  ok = ok && cudaStreamCreateWithFlags(&c->internal, cudaStreamNonBlocking) == cudaSuccess;
  int* devAbortHostView = nullptr;
  if (ok) {
    *c->hostAbortPinned = 0;
    ok = cudaHostGetDevicePointer((void**)&devAbortHostView, c->hostAbortPinned, 0) == cudaSuccess;
  }
  ok = ok && cudaDeviceSynchronize() == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    freeComm(c);
    return vrcclCudaError;
  }
  for (int p = 0; p < kNumProtos; ++p) {
    c->dc.fifo[p] = static_cast<char*>(c->fifoAlloc[p]);
    c->dc.ctrl[p] = static_cast<EdgeCtrl*>(c->ctrlAlloc) + p * nEdges;
  }
  c->dc.dctrl = static_cast<EdgeCtrl*>(c->ctrlAlloc) + kNumProtos * nEdges;
  c->dc.status = static_cast<DevStatus*>(c->statusAlloc);
  c->dc.devAbort = reinterpret_cast<int*>(static_cast<char*>(c->statusAlloc) + 128);
  c->dc.hostAbort = devAbortHostView;
  c->dc.nranks = nranks;
  c->dc.maxChannels = nchannels;
  c->dc.faultRank = -1;
  c->dc.faultChannel = -1;
  c->dc.faultAfter = 0;
  long long tmo = envInt("VRCCL_TIMEOUT_MS", 2000);
  if (tmo < 1) tmo = 2000;
  c->dc.timeoutNs = (unsigned long long)tmo * 1000000ull;
  const char* dbg = getenv("VRCCL_DEBUG");
  c->debug = dbg && (strcasecmp(dbg, "INFO") == 0 || strcasecmp(dbg, "TRACE") == 0);
  if (!envMasks(c->envAlgoMask, c->envProtoMask)) {
    freeComm(c);
    return vrcclInvalidArgument;  // "Unrecognized element token"
  }
  c->envChannels = std::min(envInt("VRCCL_NCHANNELS", 0), nchannels);
  c->envSliceBytes = (size_t)std::max(0, envInt("VRCCL_SLICE_BYTES", 0)) / 16 * 16;
  c->envWarps = std::max(0, envInt("VRCCL_SIMPLE_WARPS", 0));
  c->envPrefetch = std::min(kMaxPrefetch, std::max(0, envInt("VRCCL_PREFETCH", 0)));
  c->direct = envInt("VRCCL_DIRECT", 1) != 0;
  c->tuner.loadEnvFile(nranks);
  {
    std::lock_guard<std::mutex> lk(gLiveMu);
    gLive.push_back(c);
  }
  *comm = c;
  return vrcclSuccess;
}

extern "C" vrcclResult_t vrcclCommDestroy(vrcclComm_t comm) {
  if (!comm) return vrcclSuccess;
  if (!validComm(comm)) return vrcclInvalidArgument;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(comm->device);
  cudaError_t e = cudaDeviceSynchronize();
  freeComm(comm);
  cudaSetDevice(prev);
  return e == cudaSuccess ? vrcclSuccess : vrcclCudaError;
}

extern "C" vrcclResult_t vrcclCommCount(vrcclComm_t comm, int* nranks) {
  if (!validComm(comm) || !nranks) return vrcclInvalidArgument;
  *nranks = comm->nranks;
  return vrcclSuccess;
}

extern "C" vrcclResult_t vrcclCommSetSchedule(vrcclComm_t comm, int nchannels, size_t chunkBytes) {
  if (!validComm(comm)) return vrcclInvalidArgument;
  if (nchannels < 0 || nchannels > comm->maxChannels) return vrcclInvalidArgument;
  if (chunkBytes % 16) return vrcclInvalidArgument;
  comm->forceChannels = nchannels;
  comm->forceChunkBytes = chunkBytes;
  return vrcclSuccess;
}

extern "C" vrcclResult_t vrcclCommSetDirect(vrcclComm_t comm, int enable) {
  if (!validComm(comm) || (enable != 0 && enable != 1)) return vrcclInvalidArgument;
  comm->direct = enable != 0;
  return vrcclSuccess;
}

extern "C" vrcclResult_t vrcclCommSetTimeout(vrcclComm_t comm, uint64_t timeoutMs) {
  if (!validComm(comm) || timeoutMs < 1 || timeoutMs > 3600000ull) return vrcclInvalidArgument;
  comm->dc.timeoutNs = timeoutMs * 1000000ull;
  return vrcclSuccess;
}

extern "C" vrcclResult_t vrcclCommInjectFault(vrcclComm_t comm, int rank, int channel, int afterSteps) {
  if (!validComm(comm)) return vrcclInvalidArgument;
  if (rank < 0) {
    comm->dc.faultRank = comm->dc.faultChannel = -1;
    return vrcclSuccess;
  }
  if (rank >= comm->nranks || channel < 0 || channel >= comm->maxChannels || afterSteps < 0)
    return vrcclInvalidArgument;
  comm->dc.faultRank = rank;
  comm->dc.faultChannel = channel;
  comm->dc.faultAfter = afterSteps;
  return vrcclSuccess;
}

extern "C" vrcclResult_t vrcclCommAbort(vrcclComm_t comm) {
  if (!validComm(comm)) return vrcclInvalidArgument;
  *reinterpret_cast<volatile int*>(comm->hostAbortPinned) = 1;
  comm->aborted = true;
  return vrcclSuccess;
}

static vrcclResult_t readStatus(vrcclComm_t comm, DevStatus* st) {
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(comm->device);
  cudaError_t e = cudaMemcpyAsync(st, comm->dc.status, sizeof(DevStatus), cudaMemcpyDeviceToHost, comm->internal);
  if (e == cudaSuccess) e = cudaStreamSynchronize(comm->internal);
  cudaSetDevice(prev);
  return e == cudaSuccess ? vrcclSuccess : vrcclCudaError;
}

extern "C" vrcclResult_t vrcclCommGetAsyncError(vrcclComm_t comm, vrcclResult_t* asyncErr) {
  if (!validComm(comm) || !asyncErr) return vrcclInvalidArgument;
  DevStatus st;
  vrcclResult_t r = readStatus(comm, &st);
  if (r != vrcclSuccess) return r;
  *asyncErr = st.code ? (vrcclResult_t)st.code : (comm->aborted ? vrcclAborted : vrcclSuccess);
  if (*asyncErr != vrcclSuccess) comm->failed = true;
  return vrcclSuccess;
}

extern "C" vrcclResult_t vrcclCommGetErrorInfo(vrcclComm_t comm, int* rank, int* channel, uint64_t* step) {
  if (!validComm(comm)) return vrcclInvalidArgument;
  DevStatus st;
  vrcclResult_t r = readStatus(comm, &st);
  if (r != vrcclSuccess) return r;
  if (rank) *rank = st.code ? st.rank : -1;
  if (channel) *channel = st.code ? st.channel : -1;
  if (step) *step = st.code ? st.step : 0;
  return vrcclSuccess;
}

extern "C" vrcclResult_t vrcclCommGetLastSchedule(vrcclComm_t comm, int* algo, int* proto, int* nchannels,
                                                  size_t* chunkElems) {
  if (!validComm(comm)) return vrcclInvalidArgument;
  if (!comm->haveLast) return vrcclInvalidUsage;
  if (algo) *algo = comm->lastAlgo;
  if (proto) *proto = comm->lastProto;
  if (nchannels) *nchannels = comm->lastChannels;
  if (chunkElems) *chunkElems = comm->lastChunk;
  return vrcclSuccess;
}

// ------------------------------------------------------------------ launch

// Blocks of `threads` threads of `fn` with `smem` bytes of dynamic shared
// memory that can be resident at once on the device.
static int residentCapacity(const vrcclComm* c, const void* fn, int threads, size_t smem) {
  struct Key {
    const void* fn;
    int threads;
    size_t smem;
    int per;
  };
  static std::mutex mu;
  static std::vector<Key> cache;
  std::lock_guard<std::mutex> lk(mu);
  for (auto& e : cache)
    if (e.fn == fn && e.threads == threads && e.smem == smem) return e.per * c->smCount;
  if (smem > 0) {
    static std::vector<const void*> raised;
    if (std::find(raised.begin(), raised.end(), fn) == raised.end()) {
      const int want = maxDynamicSmem(fn, c->device);
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, want) != cudaSuccess && c->debug)
        // the launch still runs, in the smaller shapes that fit the default
        fprintf(stderr, "vrccl: could not raise a kernel's dynamic shared memory to %d bytes\n", want);
      cudaGetLastError();
      raised.push_back(fn);
    }
  }
  int per = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, fn, threads, smem) != cudaSuccess) {
    cudaGetLastError();
    per = 0;
  }
  cache.push_back({fn, threads, smem, per});
  return per * c->smCount;
}

// Shape of one Simple agent: 2 producer warps, a publisher warp and W
// consumer warps, `stages`
// shared-memory stages of (own input + received slots) x slice bytes. The
// first shape (most consumer warps, deepest pipeline, largest slice) with
// which every agent of the launch is resident at once wins.
struct SimpleShape {
  int threads;
  int stages;
  size_t sliceBytes;
  size_t smem;
};
static bool pickSimpleShape(const vrcclComm* c, const void* fn, int agents, int nbuf, size_t maxSlice,
                            int maxWarps, SimpleShape* out) {
  static const int kWarps[] = {16, 8, 4, 2, 1};
  for (size_t slice = maxSlice; slice >= 2048; slice /= 2) {
    for (int st = kMaxStages; st >= 2; --st) {
      for (int w : kWarps) {
        if (w > maxWarps) continue;
        const size_t smem = size_t(st) * nbuf * slice;
        const int threads = 32 * (3 + w);
        if (residentCapacity(c, fn, threads, smem) >= agents) {
          *out = {threads, st, slice, smem};
          return true;
        }
      }
    }
  }
  return false;
}

static int agentsPerChannel(int algo, int n) { return algo == kRing ? n : 2 * n - 1; }

// The 2n buffers of a call, as byte ranges, must not overlap, except that a
// recv buffer may sit at its in-place position: the send buffer itself
// (AllReduce), block r of rank r's send buffer (ReduceScatter), or the
// range holding block r of rank r's recv buffer (AllGather).
static bool overlapFree(int coll, const void* const* s, void* const* r, int n, size_t sendBytes,
                        size_t recvBytes) {
  std::vector<std::pair<uintptr_t, uintptr_t>> iv;
  iv.reserve(2 * n);
  for (int i = 0; i < n; ++i) {
    const uintptr_t sb = (uintptr_t)s[i], rb = (uintptr_t)r[i];
    const bool inPlace = coll == kAllReduce      ? rb == sb
                       : coll == kReduceScatter ? rb == sb + size_t(i) * recvBytes
                                                : sb == rb + size_t(i) * sendBytes;
    if (inPlace) {
      iv.push_back(coll == kAllGather ? std::make_pair(rb, rb + recvBytes) : std::make_pair(sb, sb + sendBytes));
    } else {
      iv.push_back({sb, sb + sendBytes});
      iv.push_back({rb, rb + recvBytes});
    }
  }
  std::sort(iv.begin(), iv.end());
  for (size_t i = 1; i < iv.size(); ++i)
    if (iv[i].first < iv[i - 1].second) return false;
  return true;
}

static const char* kCollName[3] = {"AllReduce", "ReduceScatter", "AllGather"};

// ------------------------------------------------------------- one call

// Argument checks (ncclEnqueueCheck: CommCheck, then ArgsCheck, Deep Dive
// (Japanese edition) ch.6).
static vrcclResult_t checkCall(vrcclComm_t comm, int coll, const void* const* sendbufs, void* const* recvbufs,
                               size_t count, vrcclDataType_t dtype, vrcclRedOp_t op, vrcclAlgo_t algo,
                               vrcclProto_t proto) {
  if (!validComm(comm)) return vrcclInvalidArgument;
  if ((unsigned)dtype >= (unsigned)vrcclNumTypes || (unsigned)op >= (unsigned)vrcclNumOps ||
      (unsigned)algo > (unsigned)vrcclAlgoOneShot || (unsigned)proto > (unsigned)vrcclProtoAuto)
    return vrcclInvalidArgument;
  if (coll != kAllReduce && algo != vrcclAlgoRing) return vrcclInvalidArgument;
  if (comm->failed || comm->aborted) return vrcclInvalidUsage;
  if (count == 0) return vrcclSuccess;  // touches nothing: the pointers are not examined
  if (!sendbufs || !recvbufs) return vrcclInvalidArgument;
  const int n = comm->nranks;
  for (int r = 0; r < n; ++r) {
    if (!sendbufs[r] || !recvbufs[r]) return vrcclInvalidArgument;
    if (((uintptr_t)sendbufs[r] | (uintptr_t)recvbufs[r]) & 15u) return vrcclInvalidArgument;
  }
  const size_t E = kElemSize[dtype];
  const size_t blocks = coll == kAllReduce ? 1 : (size_t)n;
  if (count > (size_t(1) << 40) / E / blocks) return vrcclInvalidArgument;
  // Every block of the phases starts on a 16-byte boundary, like a buffer.
  if (coll != kAllReduce && n > 1 && (count * E) % 16) return vrcclInvalidArgument;
  const size_t blockBytes = count * E;
  const size_t sendBytes = coll == kReduceScatter ? blockBytes * n : blockBytes;
  const size_t recvBytes = coll == kAllGather ? blockBytes * n : blockBytes;
  if (!overlapFree(coll, sendbufs, recvbufs, n, sendBytes, recvBytes)) return vrcclInvalidArgument;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev != comm->device) return vrcclInvalidUsage;
  return vrcclSuccess;
}

// The launch shape of one ring/tree launch.
struct Shape {
  int A, P, C;
  int threads, stages;
  size_t smem, sliceBytes, chunkBytes;
  const void* fn;
  int per;  // agents per channel
  Choice tuned;  // what the tuning table (or the size rule) proposed
};

// Chooses algorithm, protocol and channels for `bytes` per rank (the tuning
// table, or what the caller / environment forced), then the largest agent
// shape with which every agent of the launch is resident at once (all
// agents wait on each other). grouped: the kernel is the grouped ring.
static vrcclResult_t chooseShape(vrcclComm_t comm, int coll, int algo, int proto, size_t bytes, int kdtype, int kop,
                                 size_t kE, bool grouped, Shape* out) {
  const int n = comm->nranks;
  const bool userAlgo = coll == kAllReduce && algo != vrcclAlgoAuto && !grouped;
  const bool userProto = proto != vrcclProtoAuto;
  // What "auto" may choose: the environment's lists, narrowed by the call
  // (an explicit algorithm or protocol is the only choice) and by what the
  // collective has (the phases, a group's runs and the one-shot's order
  // are the ring's). An empty choice is NCCL's "no algorithm/protocol
  // available".
  unsigned algoMask = comm->envAlgoMask[coll], protoMask = comm->envProtoMask[coll];
  if (userAlgo && algo != vrcclAlgoOneShot) algoMask = 1u << algo;
  if (coll != kAllReduce || grouped || algo == vrcclAlgoOneShot || n == 1) algoMask &= 1u << kRing;
  if (algo == vrcclAlgoOneShot || n == 1) algoMask = 1u << kRing;  // a single rank is a local copy
  if (userProto) protoMask = 1u << proto;
  if (algo == vrcclAlgoOneShot) protoMask = 1u << kSimple;
  if (!algoMask || !protoMask) return vrcclInvalidUsage;
  Choice ch = comm->tuner.choose(n, bytes, (int)kE, comm->maxChannels, algoMask, protoMask);
  const int A = ch.algo, P = ch.proto;
  int C = comm->forceChannels ? comm->forceChannels
        : comm->envChannels   ? comm->envChannels
        : (ch.channels > 0 ? std::min(ch.channels, comm->maxChannels)
                           : defaultChannels(P, bytes, n, comm->maxChannels));
  const bool userChannels = comm->forceChannels || comm->envChannels;
  // LL128 with at least two whole slices per agent takes the wide kernels.
  const size_t perAgent = bytes / std::max(C, 1) / (A == kRing ? n : 1);
  const int kp = P == kLL128 && !grouped && perAgent >= 2 * slotDataBytes(kLL128) ? kLL128Wide : P;
  const void* fn = grouped ? groupKernelFor(P, kdtype, kop) : kernelFor(A, kp, kdtype, kop);
  if (!fn) return vrcclInternalError;
  const int per = agentsPerChannel(A, n);
  if (!userChannels && ch.channels == 0 && per * C > comm->smCount) {
    // Every agent does the same work, so a launch runs at the pace of the
    // most crowded SM: use a whole number of agents per SM.
    const int k = per * C / comm->smCount;
    C = std::max(1, k * comm->smCount / per);
  }
  Shape s;
  s.tuned = ch;
  s.A = A;
  s.P = P;
  s.fn = fn;
  s.per = per;
  s.threads = 256;
  s.stages = 0;
  s.smem = 0;
  s.sliceBytes = slotDataBytes(P);
  const size_t wantSlice = std::min(comm->envSliceBytes ? comm->envSliceBytes
                                    : ch.sliceBytes     ? ch.sliceBytes
                                                        : kSimpleSlotBytes,
                                    kSimpleSlotBytes);
  if (algo == vrcclAlgoOneShot) {
    s.sliceBytes = wantSlice;  // no agents: only C and the chunk matter
  } else if (P == kSimple) {
    // Shrink the agent first, then (if the caller left it open) the channels.
    const int nbuf = A == kTree ? 3 : 2;
    SimpleShape sh;
    // 2-byte types do twice the element arithmetic per byte: with a large
    // share per agent they take twice the consumer warps (measured on the
    // bf16 avg bucket, 1 GiB per rank: 16 warps 3.40 ms, 8 warps 3.47 ms;
    // before the ring's consumer loop was compiled per slice kind 5.1 and
    // 6.2 ms; the bf16 sum at 256 MiB is 3 % faster with 8, fp32 2 %
    // slower with 16). Below 1 MiB per agent the larger block only adds
    // latency (bf16 1 KiB: 41 us with 8 warps, 49 us with 16).
    const bool wide = kE == 2 && bytes / std::max(C, 1) >= (size_t(1) << 20);
    const int maxWarps = comm->envWarps ? std::min(comm->envWarps, kMaxConsumerWarps) : (wide ? 16 : 8);
    while (!pickSimpleShape(comm, fn, per * C, nbuf, wantSlice, maxWarps, &sh)) {
      if (userChannels || C == 1) return userAlgo || userChannels ? vrcclInvalidUsage : vrcclInternalError;
      --C;
    }
    s.threads = sh.threads;
    s.stages = sh.stages;
    s.smem = sh.smem;
    s.sliceBytes = sh.sliceBytes;
  } else {
    int cap = residentCapacity(comm, fn, s.threads, 0);
    while (cap < per * C && s.threads > 64) {
      s.threads /= 2;
      cap = residentCapacity(comm, fn, s.threads, 0);
    }
    if (cap < per * C) {
      if (userChannels) return vrcclInvalidUsage;
      C = cap / per;
      if (C < 1) return userAlgo ? vrcclInvalidUsage : vrcclInternalError;
    }
    if (P == kLL128) s.sliceBytes = s.sliceBytes / 240 * 240;  // whole lines and 16-byte slice starts
  }
  s.C = C;
  s.sliceBytes = std::max<size_t>(s.sliceBytes / 16 * 16, 16);
  // Chunk: VRCCL_STEPS/2 slots (ALLREDUCE_CHUNKSTEPS = NCCL_STEPS/2, Deep
  // Dive (Japanese edition) ch.6). Fewer slots per chunk than the FIFO depth
  // is what keeps the credit ring deadlock-free.
  size_t chunkBytes = comm->forceChunkBytes ? comm->forceChunkBytes
                    : (ch.chunkBytes ? ch.chunkBytes : s.sliceBytes * (kSteps / 2));
  chunkBytes = std::min(chunkBytes, s.sliceBytes * (kSteps / 2));
  s.chunkBytes = std::max<size_t>(chunkBytes / 16 * 16, 16);
  *out = s;
  return vrcclSuccess;
}

// LL / LL128 flags are the low 32 bits of each edge's step count: before a
// launch that may take up to `steps` more steps per edge, clear the FIFO and
// its counters if a flag value could repeat one still sitting in a slot.
static vrcclResult_t llReserve(vrcclComm_t comm, int P, unsigned long long steps, vrcclStream_t stream) {
  if (P == kSimple) return vrcclSuccess;
  const int n = comm->nranks;
  if (comm->llStepBound[P] + steps > (1ull << 31)) {
    const size_t nEdges = size_t(3) * comm->maxChannels * n;
    if (cudaMemsetAsync(comm->fifoAlloc[P], 0, fifoBytes(P, n, comm->maxChannels), (cudaStream_t)stream) !=
            cudaSuccess ||
        cudaMemsetAsync(comm->dc.ctrl[P], 0, nEdges * sizeof(EdgeCtrl), (cudaStream_t)stream) != cudaSuccess)
      return vrcclCudaError;
    comm->llStepBound[P] = 0;
  }
  comm->llStepBound[P] += steps;
  return vrcclSuccess;
}

// Upper bound of the FIFO steps one edge takes for `elems` elements over C
// channels in slices of `sliceElems`.
static unsigned long long stepBound(int n, unsigned long long elems, int C, int sliceElems) {
  const unsigned long long perCh = (elems + C - 1) / C + 1;
  return 2ull * n * ((perCh + sliceElems - 1) / sliceElems + 2ull * n + 2);
}

static vrcclResult_t cooperativeLaunch(const void* fn, int blocks, int threads, size_t smem, void* arg,
                                       vrcclStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {arg};
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e == cudaErrorCooperativeLaunchTooLarge ? vrcclInvalidUsage : vrcclCudaError;
  }
  return vrcclSuccess;
}

static void recordLast(vrcclComm_t comm, int algo, const Shape& s, size_t E, int blocks) {
  comm->haveLast = true;
  comm->lastAlgo = algo;
  comm->lastProto = s.P;
  comm->lastChannels = s.C;
  comm->lastChunk = s.chunkBytes / E;
  comm->lastSlice = (int)(s.sliceBytes / E);
  comm->lastThreads = s.threads;
  comm->lastBlocks = blocks;
}

static void debugLine(vrcclComm_t comm, const char* what, size_t bytes, const char* algoName, const Shape& s,
                      int blocks) {
  if (!comm->debug) return;
  char host[64] = {0};
  gethostname(host, sizeof(host) - 1);
  char src[64];
  if (s.tuned.measured)
    snprintf(src, sizeof(src), "measured (%d-byte rows, 2^%d B)", s.tuned.esize, s.tuned.log2bytes);
  else
    snprintf(src, sizeof(src), "size rule");
  fprintf(stderr,
          "%s:%d:%ld [%d] VRCCL INFO %s: %zu Bytes -> Algo %s proto %s channel{Lo..Hi}={0..%d} "
          "chunk %zu slice %zu threads %d blocks %d nranks %d tuning %s\n",
          host, (int)getpid(), (long)syscall(SYS_gettid), comm->device, what, bytes, algoName, kProtoName[s.P],
          s.C - 1, s.chunkBytes, s.sliceBytes, s.threads, blocks, comm->nranks, src);
}

// The one-shot AllReduce: C and the chunk as the ring/Simple schedule has
// them (before any co-residency shrink, which the one-shot does not need),
// then one plain launch of a grid that fills every SM.
static vrcclResult_t launchOneShot(vrcclComm_t comm, const Call& k, const Shape& s) {
  const int n = comm->nranks;
  const size_t E = kElemSize[k.dtype];
  const void* fn = kOneShot[k.dtype][k.op];
  const int threads = 512;
  const int perSm = residentCapacity(comm, fn, threads, 0) / std::max(1, comm->smCount);
  if (perSm < 1) return vrcclInternalError;
  KArgs ka;
  memset(&ka, 0, sizeof(ka));
  ka.comm = comm->dc;
  ka.count = k.count;
  ka.coll = kAllReduce;
  ka.nranks = n;
  ka.nchannels = s.C;
  ka.chunkElems = (int)(s.chunkBytes / E);
  ka.sliceElems = (int)(s.sliceBytes / E);
  ka.scale = 1.0f / (float)n;
  for (int r = 0; r < n; ++r) {
    ka.send[r] = k.send[r];
    ka.recv[r] = k.recv[r];
  }
  const unsigned long long tiles = (k.count / (16 / E) + threads * 4 - 1) / (threads * 4);
  const unsigned grid = (unsigned)std::max<unsigned long long>(1, std::min<unsigned long long>(tiles,
                                                                   (unsigned long long)perSm * comm->smCount));
  void* args[] = {&ka};
  cudaError_t e = cudaLaunchKernel(fn, dim3(grid), dim3(threads), args, 0, (cudaStream_t)k.stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return vrcclCudaError;
  }
  Shape r = s;
  r.threads = threads;
  r.P = kSimple;
  recordLast(comm, vrcclAlgoOneShot, r, E, (int)grid);
  debugLine(comm, "AllReduce", k.count * E, "OneShot", r, (int)grid);
  return vrcclSuccess;
}

// Runs one validated call as one launch.
static vrcclResult_t runCall(vrcclComm_t comm, const Call& k) {
  const int n = comm->nranks;
  const size_t E = kElemSize[k.dtype];
  if (k.count == 0) return vrcclSuccess;  // taskAppend step 4: nothing to do
  // The all-gather phase only copies: it runs as 4-byte words, whatever
  // the type (the blocks are whole 16-byte units).
  int kdtype = k.dtype, kop = k.op;
  size_t kcount = k.count, kE = E;
  if (k.coll == kAllGather && n > 1) {
    kdtype = vrcclInt32;
    kop = vrcclSum;
    kcount = k.count * E / 4;
    kE = 4;
  }
  // bytes = one rank's send (AllReduce, ReduceScatter) or recv (AllGather)
  // buffer; the phases take the ring's entries of the table at that size.
  const size_t bytes = k.coll == kAllReduce ? k.count * E : k.count * E * n;
  Shape s;
  vrcclResult_t res = chooseShape(comm, k.coll, k.algo, k.proto, bytes, kdtype, kop, kE, false, &s);
  if (res != vrcclSuccess) return res;
  if (k.algo == vrcclAlgoOneShot) return launchOneShot(comm, k, s);
  const int sliceElems = (int)(s.sliceBytes / kE);
  res = llReserve(comm, s.P, stepBound(n, bytes / kE, s.C, sliceElems), k.stream);
  if (res != vrcclSuccess) return res;

  KArgs ka;
  memset(&ka, 0, sizeof(ka));
  ka.comm = comm->dc;
  ka.count = kcount;
  ka.coll = n == 1 ? kAllReduce : k.coll;  // one rank: every collective is the copy
  ka.nranks = n;
  ka.nchannels = s.C;
  ka.chunkElems = (int)(s.chunkBytes / kE);
  ka.sliceElems = sliceElems;
  ka.scale = 1.0f / (float)n;
  ka.stages = s.stages;
  ka.prefetch = s.P == kSimple ? comm->envPrefetch : 0;
  ka.direct = comm->direct && s.A == kRing && s.P == kSimple && (k.coll == kAllReduce || k.coll == kAllGather) &&
              n > 1;
  for (int r = 0; r < n; ++r) {
    ka.send[r] = k.send[r];
    ka.recv[r] = k.recv[r];
  }
  const int blocks = s.per * s.C;
  res = cooperativeLaunch(s.fn, blocks, s.threads, s.smem, &ka, k.stream);
  if (res != vrcclSuccess) return res;
  recordLast(comm, s.A, s, E, blocks);
  debugLine(comm, kCollName[k.coll], bytes, kAlgoName[s.A], s, blocks);
  return vrcclSuccess;
}

// ----------------------------------------------------------------- groups
//
// ncclGroupStart / ncclGroupEnd ("NCCL architecture ...", §9.2 and §9.6;
// Deep Dive (Japanese edition) ch.5 and ch.6): between the two, calls are
// checked and only registered; the outermost vrcclGroupEnd schedules what
// each communicator registered. The group depth is per thread.

static thread_local int tlGroupDepth = 0;
static thread_local std::vector<vrcclComm*> tlGroupComms;

static bool isLive(vrcclComm* c) {
  std::lock_guard<std::mutex> lk(gLiveMu);
  return std::find(gLive.begin(), gLive.end(), c) != gLive.end();
}

// Grouping: AllReduces of one (type, op, requested protocol) on the ring
// (algo ring or auto) are bucketed, sorted by size, largest first, and cut
// into runs whose sizes lie within 4x of the run's largest (ncclPrepareTasks,
// "NCCL architecture ...", §9.2). A run is scheduled as a whole: the
// protocol and channel budget come from the tuning table at the run's total
// size (its launch latency is paid once, which is what numPipeOps expresses
// in NCCL's model), each task takes the channel count a call of its own
// size would get, and tasks fill channel ranges round-robin. Every other
// call runs alone.
// A run with its launch shape and each task's channel count. A task whose
// part on a channel is shorter than one ring loop (n chunks) pays the loop's
// 2n-1 dependent steps with chunks too small to hide a hop's latency, so a
// grouped task takes just enough channels to give each a full loop, at most
// the launch's: the group's many tasks then run side by side on different
// channels (measured on the 224-tensor bucket: 8.96 ms with each task on the
// channels a call of its size would use, 13.2 ms with every task on all 19).
struct PlannedRun {
  Shape s;
  std::vector<int> idx;
  std::vector<int> nch;
};

static vrcclResult_t planRun(vrcclComm_t comm, const std::vector<Call>& calls, const std::vector<int>& run,
                             PlannedRun* out) {
  const int n = comm->nranks;
  const Call& k0 = calls[run[0]];
  const size_t E = kElemSize[k0.dtype];
  size_t total = 0;
  for (int i : run) total += calls[i].count * E;
  vrcclResult_t res = chooseShape(comm, kAllReduce, vrcclAlgoRing, k0.proto, total, k0.dtype, k0.op, E, true,
                                  &out->s);
  if (res != vrcclSuccess) return res;
  out->idx = run;
  out->nch.clear();
  const size_t loopBytes = size_t(n) * out->s.chunkBytes;
  for (int i : run) {
    const size_t b = calls[i].count * E;
    int nch = comm->forceChannels ? comm->forceChannels
            : comm->envChannels   ? comm->envChannels
                                  : (int)std::min<size_t>((b + loopBytes - 1) / loopBytes, (size_t)out->s.C);
    out->nch.push_back(std::max(1, std::min(nch, out->s.C)));
  }
  return vrcclSuccess;
}

static bool sameLaunch(const Shape& a, const Shape& b) {
  return a.fn == b.fn && a.C == b.C && a.threads == b.threads && a.stages == b.stages && a.smem == b.smem &&
         a.sliceBytes == b.sliceBytes && a.chunkBytes == b.chunkBytes;
}

// Enqueues planned runs. Consecutive runs with the same launch shape share
// launches (one plan holds a group's collectives, "NCCL architecture ...",
// §9.6); a launch takes tasks until its parameter block is full. Within a
// launch, each task (largest first) takes the window of channels whose most
// loaded channel carries the fewest bytes so far.
static vrcclResult_t launchRuns(vrcclComm_t comm, const std::vector<Call>& calls, const std::vector<PlannedRun>& runs) {
  const int n = comm->nranks;
  const int maxTasks = std::min(kMaxGroupTasks, kGroupPtrs / n);
  vrcclResult_t res = vrcclSuccess;
  GroupArgs* g = new GroupArgs;
  size_t r = 0, t0 = 0;  // next run, next task within it
  while (r < runs.size() && res == vrcclSuccess) {
    const Shape& s = runs[r].s;
    const Call& k0 = calls[runs[r].idx[0]];
    const size_t E = kElemSize[k0.dtype];
    const int sliceElems = (int)(s.sliceBytes / E);
    memset(static_cast<void*>(g), 0, sizeof(*g));
    g->comm = comm->dc;
    g->nranks = n;
    g->nchannels = s.C;
    g->chunkElems = (int)(s.chunkBytes / E);
    g->sliceElems = sliceElems;
    g->stages = s.stages;
    g->prefetch = s.P == kSimple ? comm->envPrefetch : 0;
    g->direct = comm->direct && s.P == kSimple && n > 1;
    g->scale = 1.0f / (float)n;
    std::vector<double> load(s.C, 0.0);
    unsigned long long steps = 0;
    size_t bytes = 0;
    int t = 0;
    while (t < maxTasks && r < runs.size() && sameLaunch(runs[r].s, s)) {
      const int ci = runs[r].idx[t0];
      const Call& k = calls[ci];
      const int nch = runs[r].nch[t0];
      int best = 0;
      double bestLoad = -1.0;
      for (int st = 0; st < s.C; ++st) {
        double m = 0.0;
        for (int j = 0; j < nch; ++j) m = std::max(m, load[(st + j) % s.C]);
        if (bestLoad < 0.0 || m < bestLoad) {
          bestLoad = m;
          best = st;
        }
      }
      for (int j = 0; j < nch; ++j) load[(best + j) % s.C] += double(k.count * E) / nch;
      g->task[t].count = k.count;
      g->task[t].chLo = best;
      g->task[t].nch = nch;
      for (int q = 0; q < n; ++q) {
        g->send[t * n + q] = k.send[q];
        g->recv[t * n + q] = k.recv[q];
      }
      steps += stepBound(n, k.count, nch, sliceElems);
      bytes += k.count * E;
      comm->groupSched[ci] = {kRing, s.P, nch, s.chunkBytes / E, comm->groupLaunches};
      ++t;
      if (++t0 == runs[r].idx.size()) {
        ++r;
        t0 = 0;
      }
    }
    g->ntasks = t;
    res = llReserve(comm, s.P, steps, k0.stream);
    if (res == vrcclSuccess) res = cooperativeLaunch(s.fn, s.per * s.C, s.threads, s.smem, g, k0.stream);
    if (res == vrcclSuccess) {
      ++comm->groupLaunches;
      recordLast(comm, kRing, s, E, s.per * s.C);
      debugLine(comm, "AllReduce(group)", bytes, "Ring", s, s.per * s.C);
    }
  }
  delete g;
  return res;
}

static vrcclResult_t runGroup(vrcclComm_t comm) {
  std::vector<Call> calls;
  calls.swap(comm->pending);
  comm->groupSched.assign(calls.size(), GroupSched{-1, -1, 0, 0, -1});
  comm->groupLaunches = 0;
  vrcclResult_t res = vrcclSuccess;
  // bucket -> call indices, in call order
  std::vector<std::pair<long long, std::vector<int>>> buckets;
  std::vector<int> alone;
  for (int i = 0; i < (int)calls.size(); ++i) {
    const Call& k = calls[i];
    const bool ringable = k.coll == kAllReduce && comm->nranks > 1 && k.count > 0 &&
                          (k.algo == vrcclAlgoRing ||
                           (k.algo == vrcclAlgoAuto && (comm->envAlgoMask[kAllReduce] & (1u << kRing))));
    if (!ringable) {
      alone.push_back(i);
      continue;
    }
    const long long key = ((long long)k.dtype * vrcclNumOps + k.op) * 8 + k.proto;
    auto it = std::find_if(buckets.begin(), buckets.end(), [&](const auto& b) { return b.first == key; });
    if (it == buckets.end()) {
      buckets.push_back({key, {}});
      it = buckets.end() - 1;
    }
    it->second.push_back(i);
  }
  std::vector<PlannedRun> planned;
  for (auto& b : buckets) {
    std::vector<int>& v = b.second;
    std::stable_sort(v.begin(), v.end(), [&](int a, int c) { return calls[a].count > calls[c].count; });
    size_t i = 0;
    while (i < v.size() && res == vrcclSuccess) {
      size_t j = i + 1;
      while (j < v.size() && calls[v[i]].count < 4 * calls[v[j]].count) ++j;
      planned.emplace_back();
      res = planRun(comm, calls, std::vector<int>(v.begin() + i, v.begin() + j), &planned.back());
      i = j;
    }
  }
  if (res == vrcclSuccess) res = launchRuns(comm, calls, planned);
  for (size_t a = 0; a < alone.size() && res == vrcclSuccess; ++a) {
    const Call& k = calls[alone[a]];
    res = runCall(comm, k);
    if (res == vrcclSuccess && k.count > 0)
      comm->groupSched[alone[a]] = {comm->lastAlgo, comm->lastProto, comm->lastChannels, comm->lastChunk,
                                    comm->groupLaunches++};
  }
  return res;
}

extern "C" vrcclResult_t vrcclGroupStart(void) {
  ++tlGroupDepth;
  return vrcclSuccess;
}

extern "C" vrcclResult_t vrcclGroupEnd(void) {
  if (tlGroupDepth <= 0) return vrcclInvalidUsage;
  if (--tlGroupDepth > 0) return vrcclSuccess;
  std::vector<vrcclComm*> comms;
  comms.swap(tlGroupComms);
  vrcclResult_t res = vrcclSuccess;
  for (vrcclComm* c : comms) {
    if (!isLive(c)) continue;
    if (res == vrcclSuccess) {
      res = runGroup(c);
    } else {
      c->pending.clear();  // an earlier launch failed: drop the rest of the group
    }
  }
  return res;
}

extern "C" vrcclResult_t vrcclCommGetGroupSchedule(vrcclComm_t comm, int index, int* algo, int* proto,
                                                   int* nchannels, size_t* chunkElems, int* launch) {
  if (!validComm(comm)) return vrcclInvalidArgument;
  if (index < 0 || index >= (int)comm->groupSched.size()) return vrcclInvalidArgument;
  const GroupSched& g = comm->groupSched[index];
  if (g.algo < 0) return vrcclInvalidUsage;  // nothing was launched for that call (count 0)
  if (algo) *algo = g.algo;
  if (proto) *proto = g.proto;
  if (nchannels) *nchannels = g.channels;
  if (chunkElems) *chunkElems = g.chunk;
  if (launch) *launch = g.launch;
  return vrcclSuccess;
}

// Checks a call, then runs it now or, inside a group, registers it.
static vrcclResult_t enqueue(int coll, const void* const* sendbufs, void* const* recvbufs, size_t count,
                             vrcclDataType_t dtype, vrcclRedOp_t op, vrcclAlgo_t algo, vrcclProto_t proto,
                             vrcclComm_t comm, vrcclStream_t stream) {
  vrcclResult_t res = checkCall(comm, coll, sendbufs, recvbufs, count, dtype, op, algo, proto);
  if (res != vrcclSuccess) return res;
  if (count == 0 && tlGroupDepth == 0) return vrcclSuccess;  // taskAppend step 4: nothing to do
  Call k;
  k.coll = coll;
  k.dtype = dtype;
  k.op = op;
  k.algo = algo;
  k.proto = proto;
  k.count = count;
  if (count > 0) {
    k.send.assign(sendbufs, sendbufs + comm->nranks);
    k.recv.assign(recvbufs, recvbufs + comm->nranks);
  }
  k.stream = stream;
  if (tlGroupDepth > 0) {
    // All of a group's calls on one communicator share one stream.
    if (!comm->pending.empty() && comm->pending[0].stream != stream) return vrcclInvalidUsage;
    if (comm->pending.empty() &&
        std::find(tlGroupComms.begin(), tlGroupComms.end(), comm) == tlGroupComms.end())
      tlGroupComms.push_back(comm);
    comm->pending.push_back(std::move(k));
    return vrcclSuccess;
  }
  return runCall(comm, k);
}

extern "C" vrcclResult_t vrcclAllReduce(const void* const* sendbufs, void* const* recvbufs, size_t count,
                                        vrcclDataType_t dtype, vrcclRedOp_t op, vrcclAlgo_t algo,
                                        vrcclProto_t proto, vrcclComm_t comm, vrcclStream_t stream) {
  return enqueue(kAllReduce, sendbufs, recvbufs, count, dtype, op, algo, proto, comm, stream);
}

extern "C" vrcclResult_t vrcclReduceScatter(const void* const* sendbufs, void* const* recvbufs, size_t recvcount,
                                            vrcclDataType_t dtype, vrcclRedOp_t op, vrcclProto_t proto,
                                            vrcclComm_t comm, vrcclStream_t stream) {
  return enqueue(kReduceScatter, sendbufs, recvbufs, recvcount, dtype, op, vrcclAlgoRing, proto, comm, stream);
}

extern "C" vrcclResult_t vrcclAllGather(const void* const* sendbufs, void* const* recvbufs, size_t sendcount,
                                        vrcclDataType_t dtype, vrcclProto_t proto, vrcclComm_t comm,
                                        vrcclStream_t stream) {
  return enqueue(kAllGather, sendbufs, recvbufs, sendcount, dtype, vrcclSum, vrcclAlgoRing, proto, comm, stream);
}

extern "C" vrcclResult_t vrcclCommGetLaunchShape(vrcclComm_t comm, int* blocks, int* threads, int* sliceElems) {
  if (!validComm(comm)) return vrcclInvalidArgument;
  if (!comm->haveLast) return vrcclInvalidUsage;
  if (blocks) *blocks = comm->lastBlocks;
  if (threads) *threads = comm->lastThreads;
  if (sliceElems) *sliceElems = comm->lastSlice;
  return vrcclSuccess;
}

extern "C" vrcclResult_t vrcclCommLoadTuning(vrcclComm_t comm, const char* path, int* loaded) {
  if (!validComm(comm) || !path) return vrcclInvalidArgument;
  Tuner t;
  int k = t.load(path, comm->nranks);
  if (k < 0) return vrcclInvalidArgument;
  comm->tuner = t;
  if (loaded) *loaded = k;
  return vrcclSuccess;
}

extern "C" vrcclResult_t vrcclParseList(const char* spec, int kind, unsigned* masks) {
  if (!masks || (kind != 0 && kind != 1)) return vrcclInvalidArgument;
  return parseList(spec, kind == 0 ? kParseAlgo : kParseProto, masks) == 0 ? vrcclSuccess : vrcclInvalidArgument;
}

extern "C" vrcclResult_t vrcclModelPredict(const vrcclModelGraph_t* graph, vrcclAlgo_t algo, vrcclProto_t proto,
                                           size_t bytes, int numPipeOps, float* latUs, float* algBwGBs,
                                           float* timeUs) {
  if (!graph || (algo != vrcclAlgoRing && algo != vrcclAlgoTree) || (unsigned)proto >= (unsigned)vrcclProtoAuto)
    return vrcclInvalidArgument;
  const vrcclModelGraph_t& g = *graph;
  if (g.nranks < 2 || g.nnodes < 1 || g.nranks % g.nnodes || g.nchannels < 1 || g.bwIntra <= 0 ||
      (g.nnodes > 2 && g.bwInter <= 0) || g.hwIntra < 0 || g.hwIntra > 1 || g.arch < 0 || g.arch > 3 ||
      numPipeOps < 1)
    return vrcclInvalidArgument;
  ModelGraph m{g.nranks, g.nnodes, g.nchannels, g.bwIntra, g.bwInter, g.latencyInter, g.hwIntra, g.arch};
  double lat[2][3], bw[2][3];
  modelTable(m, lat, bw);
  if (latUs) *latUs = (float)lat[algo][proto];
  if (algBwGBs) *algBwGBs = (float)bw[algo][proto];
  if (timeUs) *timeUs = (float)modelTime(m, algo, proto, bytes, numPipeOps);
  return vrcclSuccess;
}


// Element-range sharding of one virtual-rank problem over several GPUs.
// Channels own independent contiguous ranges and never synchronise with
// each other ("NCCL architecture ...", §6.3), so the rule that cuts a
// buffer into channel parts (parts of alignUp(ceil(count/C), 16 bytes)
// elements, "NCCL Source Code Deep Dive", §2.2) cuts it into GPU parts one
// level up; each GPU then runs the whole AllReduce on its part with the
// schedule it chooses for that part.
extern "C" vrcclResult_t vrcclShardRange(size_t count, vrcclDataType_t dtype, int nshards, int shard, size_t* offset,
                                         size_t* length) {
  if ((unsigned)dtype >= (unsigned)vrcclNumTypes || nshards < 1 || shard < 0 || shard >= nshards || !offset ||
      !length)
    return vrcclInvalidArgument;
  const size_t A = 16 / kElemSize[dtype];
  const size_t part = count ? ((count + nshards - 1) / nshards + A - 1) / A * A : 0;
  const size_t lo = std::min(count, part * (size_t)shard);
  *offset = lo;
  *length = std::min(count, lo + part) - lo;
  return vrcclSuccess;
}
