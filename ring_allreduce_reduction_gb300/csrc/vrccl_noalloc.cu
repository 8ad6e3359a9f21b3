// vrcclAllReduceNoAlloc: the ring / Simple AllReduce without a
// communicator and without any allocation at call time.
//
// Some callers cannot allocate device memory when they need the reduction:
// code that runs under a memory-pool manager owning all of the device's
// memory, or a latency-critical path that cannot afford cudaMalloc's
// implicit device synchronisation, and that has no place to keep a
// communicator between calls. This entry point serves them with scratch
// memory that exists for as long as the library is loaded: one file-scope
// device array holding the FIFO slots, their head/tail counters and the
// status words, shared by every call on a device.
//
// Limits: at most kNoAllocMaxEdges ring edges (nranks x channels), i.e. at
// most 32 virtual ranks; the array is kNoAllocScratchBytes (about 16 MiB)
// on every GPU that loads the library, held until the process exits.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <utility>
#include <vector>

#include "vrccl_internal.h"

using namespace vrccl;

namespace {

constexpr int kNoAllocMaxEdges = 32;
constexpr size_t kNoAllocFifoBytes = size_t(kNoAllocMaxEdges) * kSteps * kSimpleSlotBytes;  // 16 MiB
constexpr size_t kNoAllocCtrlBytes = size_t(kNoAllocMaxEdges) * sizeof(EdgeCtrl);          // 8 KiB
constexpr size_t kNoAllocStatusBytes = 256;  // DevStatus at 0, device abort word at 128, host-abort stand-in at 192
constexpr size_t kNoAllocScratchBytes = kNoAllocFifoBytes + kNoAllocCtrlBytes + kNoAllocStatusBytes;
constexpr int kNoAllocThreads = 32 * (3 + 8);  // 2 producer warps, publisher, 8 consumer warps
constexpr int kNoAllocStages = 3;
constexpr size_t kNoAllocSmem = size_t(kNoAllocStages) * 2 * kSimpleSlotBytes;  // input + received slot
constexpr int kMaxDevices = 64;

// The scratch. In host code this name is only a stand-in for the symbol,
// not a device address: the address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char gNoAllocScratch[kNoAllocScratchBytes];

struct DeviceSetup {
  bool done;
  unsigned char* scratch;  // device address of gNoAllocScratch on this device
  unsigned long long timeoutNs;
};
DeviceSetup gSetup[kMaxDevices];
std::mutex gSetupMu;

// Once per device, with that device current: find the scratch's device
// address, raise the shared-memory limit of the 40 ring/Simple kernels,
// check that the launch shape below is resident for the largest grid, and
// read the wait limit (VRCCL_TIMEOUT_MS, as vrcclCommInit does). Only a
// set-up that succeeded is kept: a failure that passes (a call made inside
// a stream capture, say) is retried by the next call.
vrcclResult_t setupDevice(int dev, unsigned char** scratch, unsigned long long* timeoutNs) {
  std::lock_guard<std::mutex> lk(gSetupMu);
  DeviceSetup& s = gSetup[dev];
  if (!s.done) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, gNoAllocScratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return vrcclCudaError;
    }
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    for (int dt = 0; dt < vrcclNumTypes; ++dt) {
      for (int op = 0; op < vrcclNumOps; ++op) {
        const void* fn = kernelFor(kRing, kSimple, dt, op);
        int per = 0;
        if (!fn ||
            // the same limit the communicator path sets for these kernels,
            // so neither path lowers it for the other
            cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, maxDynamicSmem(fn, dev)) !=
                cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, fn, kNoAllocThreads, kNoAllocSmem) !=
                cudaSuccess ||
            per * sms < kNoAllocMaxEdges) {
          cudaGetLastError();
          return vrcclInternalError;
        }
      }
    }
    const char* tv = getenv("VRCCL_TIMEOUT_MS");
    long long ms = tv && *tv ? atoll(tv) : 2000;
    if (ms < 1) ms = 2000;
    s.scratch = static_cast<unsigned char*>(p);
    s.timeoutNs = (unsigned long long)ms * 1000000ull;
    s.done = true;
  }
  *scratch = s.scratch;
  *timeoutNs = s.timeoutNs;
  return vrcclSuccess;
}

// The 2n buffers as byte ranges must not overlap, except that a rank's
// recv buffer may be its own send buffer (in place), the rule of
// vrcclAllReduce.
bool overlapFree(const void* const* send, void* const* recv, int n, size_t bytes) {
  std::vector<std::pair<uintptr_t, uintptr_t>> iv;
  iv.reserve(2 * n);
  for (int i = 0; i < n; ++i) {
    const uintptr_t sb = (uintptr_t)send[i], rb = (uintptr_t)recv[i];
    iv.push_back({sb, sb + bytes});
    if (rb != sb) iv.push_back({rb, rb + bytes});
  }
  std::sort(iv.begin(), iv.end());
  for (size_t i = 1; i < iv.size(); ++i)
    if (iv[i].first < iv[i - 1].second) return false;
  return true;
}

}  // namespace

extern "C" vrcclResult_t vrcclAllReduceNoAlloc(const void* const* sendbufs, void* const* recvbufs, size_t count,
                                               int nranks, vrcclDataType_t dtype, vrcclRedOp_t op,
                                               vrcclStream_t stream) {
  static const size_t kElem[vrcclNumTypes] = {4, 4, 2, 2, 1, 1, 8, 8};
  if (nranks < 1 || (unsigned)dtype >= (unsigned)vrcclNumTypes || (unsigned)op >= (unsigned)vrcclNumOps ||
      !sendbufs || !recvbufs)
    return vrcclInvalidArgument;
  if (nranks > kNoAllocMaxEdges) return vrcclInvalidUsage;  // beyond the fixed scratch: use a communicator
  for (int r = 0; r < nranks; ++r) {
    if (!sendbufs[r] || !recvbufs[r]) return vrcclInvalidArgument;
    if (((uintptr_t)sendbufs[r] | (uintptr_t)recvbufs[r]) & 15u) return vrcclInvalidArgument;
  }
  const size_t E = kElem[dtype];
  if (count > (size_t(1) << 40) / E) return vrcclInvalidArgument;
  if (count == 0) return vrcclSuccess;
  if (!overlapFree(sendbufs, recvbufs, nranks, count * E)) return vrcclInvalidArgument;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return vrcclCudaError;
  unsigned char* scratch = nullptr;
  unsigned long long timeoutNs = 0;
  vrcclResult_t r = setupDevice(dev, &scratch, &timeoutNs);
  if (r != vrcclSuccess) return r;

  // Every call starts from zeroed counters and status words (the FIFO slots
  // themselves need no clearing: Simple slots carry no flags).
  cudaStream_t s = (cudaStream_t)stream;
  unsigned char* ctrl = scratch + kNoAllocFifoBytes;
  if (cudaMemsetAsync(ctrl, 0, kNoAllocCtrlBytes + kNoAllocStatusBytes, s) != cudaSuccess) return vrcclCudaError;

  KArgs ka;
  memset(&ka, 0, sizeof(ka));
  ka.comm.fifo[kSimple] = reinterpret_cast<char*>(scratch);
  ka.comm.ctrl[kSimple] = reinterpret_cast<EdgeCtrl*>(ctrl);
  ka.comm.status = reinterpret_cast<DevStatus*>(ctrl + kNoAllocCtrlBytes);
  ka.comm.devAbort = reinterpret_cast<int*>(ctrl + kNoAllocCtrlBytes + 128);
  ka.comm.hostAbort = reinterpret_cast<volatile int*>(ctrl + kNoAllocCtrlBytes + 192);
  ka.comm.timeoutNs = timeoutNs;
  ka.comm.nranks = nranks;
  ka.comm.maxChannels = std::max(1, std::min(4, kNoAllocMaxEdges / nranks));
  ka.comm.faultRank = ka.comm.faultChannel = -1;
  ka.count = count;
  ka.nranks = nranks;
  ka.nchannels = ka.comm.maxChannels;
  ka.sliceElems = (int)(kSimpleSlotBytes / E);
  ka.chunkElems = (int)(kSimpleSlotBytes * (kSteps / 2) / E);
  ka.scale = 1.0f / (float)nranks;
  ka.stages = kNoAllocStages;
  ka.prefetch = 0;
  for (int i = 0; i < nranks; ++i) {
    ka.send[i] = sendbufs[i];
    ka.recv[i] = recvbufs[i];
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(nranks * ka.nchannels));
  cfg.blockDim = dim3((unsigned)kNoAllocThreads);
  cfg.dynamicSmemBytes = kNoAllocSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&ka};
  if (cudaLaunchKernelExC(&cfg, kernelFor(kRing, kSimple, dtype, op), args) != cudaSuccess) {
    cudaGetLastError();
    return vrcclCudaError;
  }
  return vrcclSuccess;
}
