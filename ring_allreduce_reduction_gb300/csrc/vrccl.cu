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

#include "tuner.h"
#include "vrccl_internal.h"

using namespace vrccl;

namespace vrccl {
extern const void* const kRingSimple[4][5];
extern const void* const kTreeSimple[4][5];
extern const void* const kRingLL[4][5];
extern const void* const kTreeLL[4][5];
extern const void* const kRingLL128[4][5];
extern const void* const kTreeLL128[4][5];
extern const void* const kOneShot[4][5];

const void* kernelFor(int algo, int proto, int dtype, int op) {
  if (dtype < 0 || dtype >= 4 || op < 0 || op >= 5) return nullptr;
  switch (proto * 2 + algo) {
    case kSimple * 2 + kRing: return kRingSimple[dtype][op];
    case kSimple * 2 + kTree: return kTreeSimple[dtype][op];
    case kLL * 2 + kRing: return kRingLL[dtype][op];
    case kLL * 2 + kTree: return kTreeLL[dtype][op];
    case kLL128 * 2 + kRing: return kRingLL128[dtype][op];
    case kLL128 * 2 + kTree: return kTreeLL128[dtype][op];
  }
  return nullptr;
}
}  // namespace vrccl

// Sentinels at both ends of the communicator, as ncclComm's startMagic /
// endMagic (Deep Dive §2.1): a stale or foreign handle fails the check.
static constexpr uint64_t kMagic = 0x5652434331474233ull;  // "VRCC1GB3"

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
  int envProto, envAlgo, envChannels;
  size_t envSliceBytes;
  int envWarps, envPrefetch;
  bool debug;
  bool haveLast;
  int lastAlgo, lastProto, lastChannels;
  size_t lastChunk;
  int lastSlice, lastThreads, lastBlocks;
  // LL / LL128 flags are the low bits of a growing step count: an upper
  // bound of the steps issued so far decides when to clear the FIFOs.
  unsigned long long llStepBound[kNumProtos];
  Tuner tuner;
  uint64_t endMagic;
};

static bool validComm(const vrcclComm* c) {
  return c && c->startMagic == kMagic && c->endMagic == kMagic;
}

static int envInt(const char* name, int dflt) {
  const char* v = getenv(name);
  if (!v || !*v) return dflt;
  return atoi(v);
}

static int parseProto(const char* v) {
  if (!v) return -1;
  std::string s(v);
  for (auto& ch : s) ch = (char)tolower(ch);
  if (s == "simple") return kSimple;
  if (s == "ll") return kLL;
  if (s == "ll128") return kLL128;
  return -1;
}
static int parseAlgo(const char* v) {
  if (!v) return -1;
  std::string s(v);
  for (auto& ch : s) ch = (char)tolower(ch);
  if (s == "ring") return kRing;
  if (s == "tree") return kTree;
  return -1;
}

static const char* kAlgoName[4] = {"Ring", "Tree", "Auto", "OneShot"};
static const char* kProtoName[3] = {"Simple", "LL", "LL128"};
static const size_t kElemSize[4] = {4, 4, 2, 2};

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
  ok = ok && cudaMalloc(&c->ctrlAlloc, nEdges * kNumProtos * sizeof(EdgeCtrl)) == cudaSuccess &&
       cudaMemset(c->ctrlAlloc, 0, nEdges * kNumProtos * sizeof(EdgeCtrl)) == cudaSuccess;
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
  c->envProto = parseProto(getenv("VRCCL_PROTO"));
  c->envAlgo = parseAlgo(getenv("VRCCL_ALGO"));
  c->envChannels = std::min(envInt("VRCCL_NCHANNELS", 0), nchannels);
  c->envSliceBytes = (size_t)std::max(0, envInt("VRCCL_SLICE_BYTES", 0)) / 16 * 16;
  c->envWarps = std::max(0, envInt("VRCCL_SIMPLE_WARPS", 0));
  c->envPrefetch = std::min(kMaxPrefetch, std::max(0, envInt("VRCCL_PREFETCH", 0)));
  c->tuner.loadEnvFile(nranks);
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
      int optin = 0;
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, c->device);
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - 1024);
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

// The one-shot AllReduce: C and the chunk as the ring/Simple schedule has
// them (before any co-residency shrink, which the one-shot does not need),
// then one plain launch of a grid that fills every SM.
static vrcclResult_t launchOneShot(vrcclComm_t comm, const void* const* sendbufs, void* const* recvbufs,
                                   size_t count, int dtype, int op, int C, const Choice& ch, vrcclStream_t stream) {
  const int n = comm->nranks;
  const size_t E = kElemSize[dtype];
  const size_t slice = std::max<size_t>(std::min(comm->envSliceBytes ? comm->envSliceBytes
                                                 : ch.sliceBytes     ? ch.sliceBytes
                                                                     : kSimpleSlotBytes,
                                                 kSimpleSlotBytes) / 16 * 16, 16);
  size_t chunkBytes = comm->forceChunkBytes ? comm->forceChunkBytes
                    : (ch.chunkBytes ? ch.chunkBytes : slice * (kSteps / 2));
  chunkBytes = std::min(chunkBytes, slice * (kSteps / 2));
  chunkBytes = std::max<size_t>(chunkBytes / 16 * 16, 16);
  const void* fn = kOneShot[dtype][op];
  const int threads = 512;
  const int perSm = residentCapacity(comm, fn, threads, 0) / std::max(1, comm->smCount);
  if (perSm < 1) return vrcclInternalError;
  KArgs ka;
  memset(&ka, 0, sizeof(ka));
  ka.comm = comm->dc;
  ka.count = count;
  ka.coll = kAllReduce;
  ka.nranks = n;
  ka.nchannels = C;
  ka.chunkElems = (int)(chunkBytes / E);
  ka.sliceElems = (int)(slice / E);
  ka.scale = 1.0f / (float)n;
  for (int r = 0; r < n; ++r) {
    ka.send[r] = sendbufs[r];
    ka.recv[r] = recvbufs[r];
  }
  const unsigned long long tiles = (count / (16 / E) + threads * 4 - 1) / (threads * 4);
  const unsigned grid = (unsigned)std::max<unsigned long long>(1, std::min<unsigned long long>(tiles,
                                                                   (unsigned long long)perSm * comm->smCount));
  void* args[] = {&ka};
  cudaError_t e = cudaLaunchKernel(fn, dim3(grid), dim3(threads), args, 0, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return vrcclCudaError;
  }
  comm->haveLast = true;
  comm->lastAlgo = vrcclAlgoOneShot;
  comm->lastProto = kSimple;
  comm->lastChannels = C;
  comm->lastChunk = chunkBytes / E;
  comm->lastSlice = (int)(slice / E);
  comm->lastThreads = threads;
  comm->lastBlocks = (int)grid;
  if (comm->debug)
    fprintf(stderr, "[%d] VRCCL INFO AllReduce: %zu Bytes -> Algo OneShot (ring order channel{Lo..Hi}={0..%d} "
            "chunk %zu) grid %u threads %d nranks %d\n", comm->device, count * E, C - 1, chunkBytes, grid, threads, n);
  return vrcclSuccess;
}

// One collective call: validate, choose the schedule, launch once.
//   coll   AllReduce: count = elements per rank. ReduceScatter / AllGather:
//          count = elements per block (recvcount / sendcount).
static vrcclResult_t enqueue(int coll, const void* const* sendbufs, void* const* recvbufs, size_t count,
                             vrcclDataType_t dtype, vrcclRedOp_t op, vrcclAlgo_t algo, vrcclProto_t proto,
                             vrcclComm_t comm, vrcclStream_t stream) {
  // Argument checks first (ncclEnqueueCheck: CommCheck, then ArgsCheck,
  // Deep Dive (Japanese edition) ch.6).
  if (!validComm(comm)) return vrcclInvalidArgument;
  if ((unsigned)dtype >= (unsigned)vrcclNumTypes || (unsigned)op >= (unsigned)vrcclNumOps ||
      (unsigned)algo > (unsigned)vrcclAlgoOneShot || (unsigned)proto > (unsigned)vrcclProtoAuto)
    return vrcclInvalidArgument;
  if (!sendbufs || !recvbufs) return vrcclInvalidArgument;
  if (coll != kAllReduce && algo != vrcclAlgoRing) return vrcclInvalidArgument;
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
  if (comm->failed || comm->aborted) return vrcclInvalidUsage;
  if (count == 0) return vrcclSuccess;  // taskAppend step 4: nothing to do

  int dev = 0;
  cudaGetDevice(&dev);
  if (dev != comm->device) return vrcclInvalidUsage;

  // The all-gather phase only copies: it runs as 4-byte words, whatever
  // the type (the blocks are whole 16-byte units).
  int kdtype = dtype, kop = op;
  size_t kcount = count, kE = E;
  if (coll == kAllGather) {
    kdtype = vrcclInt32;
    kop = vrcclSum;
    kcount = n > 1 ? blockBytes / 4 : count;
    kE = n > 1 ? 4 : E;
    if (n == 1) kdtype = dtype;  // a single rank is a plain copy in the user's type
  }

  // ---- schedule: algo, proto, channels, chunk, slice, threads
  // bytes = one rank's send (AllReduce, ReduceScatter) or recv (AllGather)
  // buffer; the phases take the ring's entries of the table at that size.
  const size_t bytes = coll == kAllReduce ? blockBytes : blockBytes * n;
  // The one-shot takes the ring/Simple schedule's channel count and chunk,
  // which fix its association order.
  const bool oneShot = algo == vrcclAlgoOneShot;
  const bool userAlgo = coll == kAllReduce && algo != vrcclAlgoAuto, userProto = proto != vrcclProtoAuto;
  const int fixA = coll != kAllReduce || oneShot ? kRing : userAlgo ? (int)algo : comm->envAlgo;
  const int fixP = oneShot ? kSimple : userProto ? (int)proto : comm->envProto;
  Choice ch = comm->tuner.choose(n, bytes, comm->maxChannels, n == 1 ? kRing : fixA, fixP);
  int A = fixA >= 0 ? fixA : ch.algo;
  int P = fixP >= 0 ? fixP : ch.proto;
  if (n == 1) A = kRing;  // a single rank is a local copy (ncclLaunchOneRank)
  int C = comm->forceChannels ? comm->forceChannels
        : comm->envChannels   ? comm->envChannels
        : (ch.channels > 0 ? std::min(ch.channels, comm->maxChannels)
                           : defaultChannels(P, bytes, n, comm->maxChannels));
  const bool userChannels = comm->forceChannels || comm->envChannels;

  const void* fn = kernelFor(A, P, kdtype, kop);
  if (!fn) return vrcclInternalError;
  const int per = agentsPerChannel(A, n);
  if (!userChannels && ch.channels == 0 && per * C > comm->smCount) {
    // Every agent does the same work, so a launch runs at the pace of the
    // most crowded SM: use a whole number of agents per SM.
    const int k = per * C / comm->smCount;
    C = std::max(1, k * comm->smCount / per);
  }
  if (oneShot) return launchOneShot(comm, sendbufs, recvbufs, count, dtype, op, C, ch, stream);
  int threads = 256, stages = 0;
  size_t smem = 0;
  size_t sliceBytes = slotDataBytes(P);
  if (P == kSimple) {
    // All agents of a launch wait on each other: they must all be resident.
    // Shrink the agent first, then (if the caller left it open) the channels.
    const int nbuf = A == kTree ? 3 : 2;
    const size_t want = std::min(comm->envSliceBytes ? comm->envSliceBytes
                                 : ch.sliceBytes     ? ch.sliceBytes
                                                     : kSimpleSlotBytes,
                                 kSimpleSlotBytes);
    SimpleShape sh;
    const int maxWarps = comm->envWarps ? comm->envWarps : 8;
    while (!pickSimpleShape(comm, fn, per * C, nbuf, want, maxWarps, &sh)) {
      if (userChannels || C == 1) return userAlgo || userChannels ? vrcclInvalidUsage : vrcclInternalError;
      --C;
    }
    threads = sh.threads;
    stages = sh.stages;
    smem = sh.smem;
    sliceBytes = sh.sliceBytes;
  } else {
    int cap = residentCapacity(comm, fn, threads, 0);
    while (cap < per * C && threads > 64) {
      threads /= 2;
      cap = residentCapacity(comm, fn, threads, 0);
    }
    if (cap < per * C) {
      if (userChannels) return vrcclInvalidUsage;
      C = cap / per;
      if (C < 1) return userAlgo ? vrcclInvalidUsage : vrcclInternalError;
    }
    if (P == kLL128) sliceBytes = sliceBytes / 240 * 240;  // whole lines and 16-byte slice starts
  }
  sliceBytes = std::max<size_t>(sliceBytes / 16 * 16, 16);
  const int sliceElems = (int)(sliceBytes / kE);
  // Chunk: VRCCL_STEPS/2 slots (ALLREDUCE_CHUNKSTEPS = NCCL_STEPS/2, Deep
  // Dive (Japanese edition) ch.6). Fewer slots per chunk than the FIFO depth
  // is what keeps the credit ring deadlock-free.
  size_t chunkBytes = comm->forceChunkBytes ? comm->forceChunkBytes
                    : (ch.chunkBytes ? ch.chunkBytes : sliceBytes * (kSteps / 2));
  chunkBytes = std::min(chunkBytes, sliceBytes * (kSteps / 2));
  chunkBytes = std::max<size_t>(chunkBytes / 16 * 16, 16);
  const int chunkElems = (int)(chunkBytes / kE);

  // ---- LL/LL128 flag wrap: clear the FIFO and its counters well before a
  // 32-bit flag could repeat a value still sitting in a slot.
  if (P != kSimple) {
    const unsigned long long perCh = (bytes + C - 1) / C / kE + 1;
    const unsigned long long bound = 2ull * n * ((perCh + sliceElems - 1) / sliceElems + 2ull * n + 2);
    if (comm->llStepBound[P] + bound > (1ull << 31)) {
      const size_t nEdges = size_t(3) * comm->maxChannels * n;
      if (cudaMemsetAsync(comm->fifoAlloc[P], 0, fifoBytes(P, n, comm->maxChannels), (cudaStream_t)stream) !=
              cudaSuccess ||
          cudaMemsetAsync(comm->dc.ctrl[P], 0, nEdges * sizeof(EdgeCtrl), (cudaStream_t)stream) != cudaSuccess)
        return vrcclCudaError;
      comm->llStepBound[P] = 0;
    }
    comm->llStepBound[P] += bound;
  }

  KArgs ka;
  memset(&ka, 0, sizeof(ka));
  ka.comm = comm->dc;
  ka.count = kcount;
  ka.coll = n == 1 ? kAllReduce : coll;  // one rank: every collective is the copy
  ka.nranks = n;
  ka.nchannels = C;
  ka.chunkElems = chunkElems;
  ka.sliceElems = sliceElems;
  ka.scale = 1.0f / (float)n;
  ka.stages = stages;
  ka.prefetch = P == kSimple ? comm->envPrefetch : 0;
  for (int r = 0; r < n; ++r) {
    ka.send[r] = sendbufs[r];
    ka.recv[r] = recvbufs[r];
  }
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)(per * C));
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&ka};
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e == cudaErrorCooperativeLaunchTooLarge ? vrcclInvalidUsage : vrcclCudaError;
  }
  comm->haveLast = true;
  comm->lastAlgo = A;
  comm->lastProto = P;
  comm->lastChannels = C;
  comm->lastChunk = chunkBytes / E;
  comm->lastSlice = (int)(sliceBytes / E);
  comm->lastThreads = threads;
  comm->lastBlocks = per * C;
  if (comm->debug) {
    char host[64] = {0};
    gethostname(host, sizeof(host) - 1);
    fprintf(stderr,
            "%s:%d:%ld [%d] VRCCL INFO %s: %zu Bytes -> Algo %s proto %s channel{Lo..Hi}={0..%d} "
            "chunk %zu slice %d threads %d nranks %d\n",
            host, (int)getpid(), (long)syscall(SYS_gettid), comm->device, kCollName[coll], bytes, kAlgoName[A],
            kProtoName[P], C - 1, chunkBytes, (int)(sliceBytes / E), threads, n);
  }
  return vrcclSuccess;
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
