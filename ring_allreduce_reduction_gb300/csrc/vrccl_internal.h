// Internal layout shared by the host library and the sm_103a kernels.
//
// Device memory of one communicator (all owned by it, zeroed at init):
//
//   fifo[proto]  3 * maxChannels * nranks edges, each VRCCL_STEPS slots of
//                slotBytes[proto]. Edge e of
//                  [0, C*n)        ring edge (ch, r):   rank r -> r+1 on ch
//                  [C*n, 2*C*n)    tree up edge (ch, c): child c -> parent
//                  [2*C*n, 3*C*n)  tree down edge (ch, c): parent -> child c
//                (C = maxChannels). A Simple slot holds raw elements; an LL
//                slot holds 16-byte lines {data lo, flag, data hi, flag}; an
//                LL128 slot holds 128-byte lines of 120 data bytes and an
//                8-byte flag in bytes 120..127.
//   ctrl[proto]  one EdgeCtrl per edge: `tail` is written only by the edge's
//                sender, `head` only by its receiver, on separate 128-byte
//                lines (ncclSendMem.head / ncclRecvMem.tail of
//                "NCCL Source Code Deep Dive", §2.4). tail = slots the sender
//                has filled, head = slots the receiver has drained; both
//                only grow, across launches.
//   dctrl        one EdgeCtrl per ring edge for the "direct" all-gather:
//                tail = slices the sender wrote straight into the
//                receiver's recv buffer, head = slices the receiver took.
//   status       first device-side failure (code, rank, channel, step).
//   devAbort     set by the first agent that fails; every wait polls it.
//   hostAbort    mapped pinned host word raised by vrcclCommAbort.
#pragma once

#include <cstddef>
#include <cstdint>

#include "vrccl.h"

#ifndef __CUDACC__
#define __host__
#define __device__
#endif

namespace vrccl {

constexpr int kSteps = VRCCL_STEPS;
constexpr int kMaxRanks = VRCCL_MAX_RANKS;
constexpr int kNumProtos = 3;

enum ProtoId { kSimple = 0, kLL = 1, kLL128 = 2 };
// Kernel variant, not a wire protocol: LL128 moving four groups of lines per
// warp and pass (long slices). Same lines, flags and FIFOs as kLL128.
constexpr int kLL128Wide = 3;
__host__ __device__ constexpr int wireProto(int kernelProto) { return kernelProto == kLL128Wide ? kLL128 : kernelProto; }
enum AlgoId { kRing = 0, kTree = 1 };
// What one launch computes: the AllReduce, or one of its two ring phases
// run alone (ReduceScatter, AllGather).
enum CollId { kAllReduce = 0, kReduceScatter = 1, kAllGather = 2 };

// FIFO geometry (buffer bytes per slot) and the data one slot carries.
constexpr size_t kSimpleSlotBytes = 32 * 1024;  // data bytes per Simple slot (max slice)
constexpr int kLLSlotLines = 1024;              // 16-byte lines: 8 data bytes each
constexpr int kLL128SlotLines = 256;            // 128-byte lines: 120 data bytes each
constexpr int kLL128DataBytes = 120;
constexpr int kMaxStages = 8;          // Simple pipeline depth in shared memory
constexpr int kMaxConsumerWarps = 16;  // Simple: 3 service warps + up to 16 consumer warps
// Thread bound a kernel is compiled for. A Simple agent has at most 3 + 16
// warps (608 threads); its bound of 736 threads caps registers at 65536 / 736
// = 89 per thread, so two 352-thread agents (8 consumer warps) still fit on
// one SM without spilling. LL / LL128 agents use at most 256 threads (the
// host starts there and halves to fit), which leaves LL128's unrolled passes
// their registers.
__host__ __device__ constexpr int maxAgentThreads(int proto) { return proto == kSimple ? 736 : 256; }
constexpr int kMaxPrefetch = 32;       // Simple: largest input L2 prefetch distance (slices)

__host__ __device__ constexpr size_t slotBufferBytes(int proto) {
  return proto == kSimple ? kSimpleSlotBytes
       : proto == kLL     ? size_t(kLLSlotLines) * 16
                          : size_t(kLL128SlotLines) * 128;
}
__host__ __device__ constexpr size_t slotDataBytes(int proto) {
  return proto == kSimple ? kSimpleSlotBytes
       : proto == kLL     ? size_t(kLLSlotLines) * 8
                          : size_t(kLL128SlotLines) * kLL128DataBytes;
}

struct alignas(128) EdgeCtrl {
  unsigned long long tail;
  unsigned long long pad0[15];
  unsigned long long head;
  unsigned long long pad1[15];
};
static_assert(sizeof(EdgeCtrl) == 256, "EdgeCtrl layout");

struct DevStatus {
  int code;  // vrcclResult_t of the first failure, 0 = none
  int rank;
  int channel;
  int kind;  // 0 = tail wait, 1 = head wait, 2 = LL line, 3 = LL128 flag, 4 = stage barrier
  unsigned long long step;
};

struct DevComm {
  char* fifo[kNumProtos];
  EdgeCtrl* ctrl[kNumProtos];
  EdgeCtrl* dctrl;  // direct ring edges: tail = slices written into the next rank's recv buffer
  DevStatus* status;
  int* devAbort;
  volatile int* hostAbort;
  unsigned long long timeoutNs;
  int nranks;
  int maxChannels;
  int faultRank;  // fault injection: agent (faultRank, faultChannel) stops
  int faultChannel;
  int faultAfter;  // ... once it reaches this FIFO step of the launch
};

struct KArgs {
  DevComm comm;
  unsigned long long count;  // AllReduce: elements per rank; phases: elements per block
  int coll;                  // CollId
  int nranks;
  int nchannels;
  int chunkElems;  // ring chunk K (elements, multiple of 16 bytes)
  int sliceElems;  // elements per FIFO step (one slot)
  float scale;     // avg pre-scale 1.0f / n (binary32)
  int stages;      // Simple: shared-memory stages of the slice pipeline
  int prefetch;    // Simple: input slices pulled into L2 ahead of their stage (0 = off)
  int direct;      // Simple ring AllReduce: all-gather through the peers' recv buffers
  const void* send[kMaxRanks];
  void* recv[kMaxRanks];
};

// A grouped launch: several AllReduces of one type and op, run one after
// another by every channel they use (ncclGroupStart / ncclGroupEnd put a
// group's collectives into one plan, one kernel launch, "NCCL architecture
// ...", §9.6). Task t covers channels chLo .. chLo + nch - 1 (mod
// nchannels); its rank-r buffers are send[t * nranks + r] and
// recv[t * nranks + r]. The whole block is a kernel parameter (<= 32 KB).
constexpr int kMaxGroupTasks = 128;
constexpr int kGroupPtrs = 1536;  // per side: tasks x ranks of one launch
struct GroupTask {
  unsigned long long count;  // elements
  int chLo, nch;
};
struct GroupArgs {
  DevComm comm;
  int nranks;
  int nchannels;   // channels of the launch
  int chunkElems;  // ring chunk K (elements, multiple of 16 bytes)
  int sliceElems;  // elements per FIFO step
  int stages;      // Simple: shared-memory stages
  int prefetch;    // Simple: input L2 prefetch distance (0 = off)
  int direct;      // Simple: all-gather through the recv buffers
  int ntasks;
  float scale;     // avg pre-scale 1.0f / n
  GroupTask task[kMaxGroupTasks];
  const void* send[kGroupPtrs];
  void* recv[kGroupPtrs];
};
static_assert(sizeof(GroupArgs) < 32000, "GroupArgs must fit the kernel parameter space");

__host__ __device__ inline int ringEdge(int ch, int r, int n) { return ch * n + r; }
__host__ __device__ inline int treeUpEdge(int ch, int c, int n, int maxCh) { return maxCh * n + ch * n + c; }
__host__ __device__ inline int treeDownEdge(int ch, int c, int n, int maxCh) { return 2 * maxCh * n + ch * n + c; }

// Kernel table (defined by the kernel translation units).
// Returns the __global__ function for (algo, proto, dtype, op) or nullptr.
const void* kernelFor(int algo, int proto, int dtype, int op);
// Largest dynamic shared memory a block of kernel `fn` may request on
// `device`: the opt-in per-block limit less the kernel's static shared
// memory, which counts against the same limit.
int maxDynamicSmem(const void* fn, int device);
// The grouped ring kernel for (proto, dtype, op), or nullptr.
const void* groupKernelFor(int proto, int dtype, int op);

}  // namespace vrccl
