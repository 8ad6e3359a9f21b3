/*
 * vrccl -- ring AllReduce over n virtual ranks resident in one GPU's memory.
 *
 * C ABI of libvrccl.so. Plain C: no CUDA, C++ or torch types appear here;
 * a CUDA stream is passed as an opaque pointer (a cudaStream_t cast to
 * void*, NULL = the legacy default stream), and every buffer is a raw
 * device address on the communicator's device.
 *
 * Sources cited:
 *   [Deep Dive]    "NCCL Source Code Deep Dive: A GPU Journey of One
 *                  AllReduce" (aireadcode.com; English edition, chapters
 *                  1-4; the Japanese edition adds ch.5 tuning and ch.6
 *                  enqueue).
 *   [Architecture] "NCCL architecture: topology, channels, algorithms and
 *                  protocols" (arganzheng.life, part 4 of the series
 *                  "Communication and interconnect: from NCCL to RDMA").
 *
 * What it computes. An AllReduce over n ranks: every rank r contributes
 * sendbufs[r][0..count) and every rank receives, in recvbufs[r][0..count),
 * the elementwise op over all n contributions [Deep Dive §1.3]. The ranks
 * are virtual: n buffers in one GPU's HBM. Each channel owns a contiguous
 * 16-byte-aligned part of the elements and runs the whole algorithm on it
 * independently [Deep Dive §2.2; Architecture §6.3]. On a channel the ring
 * algorithm is a reduce-scatter followed by an all-gather, n-1 steps each,
 * chunked as RingARAlgorithm::getNextSendAddr describes [Deep Dive §2.3;
 * Architecture §9.4, runRing]; rank r hands chunks to rank r+1 (mod n)
 * through staging FIFOs in global memory, synchronised by one of the three
 * wire protocols Simple, LL and LL128 [Architecture §7.2]; with Simple the
 * all-gather writes each finished chunk straight into the next rank's recv
 * buffer instead (runRing's direct primitives; vrcclCommSetDirect). The tree
 * algorithm reduces up and broadcasts down the double binary tree
 * [Architecture §5.4, §9.4; Deep Dive ch.4, ncclGetBtree/ncclGetDtree].
 *
 * Numerics. Eight element types (vrcclDataType_t). bf16, fp16 and fp32 ops
 * are computed in binary32 (no contraction) and rounded (to nearest even)
 * to the element type after every step; fp64 ops are computed in binary64.
 * Integer sum/prod (int8, uint8, int32, int64) wrap modulo 2^bits; max/min
 * compare signed, unsigned for uint8. For the ring, an element of chunk j
 * ends up as
 *   op(...op(op(x[j+1], x[j+2]), x[j+3])..., x[j])        (ranks mod n)
 * where the first operand is the value that arrived from the previous rank
 * and max/min keep the first operand on a tie. avg (not an NCCL op on the
 * pages): the floating types multiply every input once by 1/n before the
 * sum (the binary32 1.0f/n for bf16/fp16/fp32, the binary64 1.0/n for
 * fp64); the integer types divide the wrapped sum by n, truncating toward
 * zero, once per chunk.
 *
 * Ordering and concurrency. Every call is asynchronous on its stream and
 * returns once the work is enqueued [Deep Dive §1.3, "Step 2"]; results are
 * defined after the stream is synchronised. Calls on one communicator
 * share its FIFOs: they must be ordered (one stream, or streams ordered by
 * events); calls that overlap on the GPU are undefined. Different
 * communicators are independent. Calls may be captured in a CUDA graph:
 * the FIFO counters and flags live in device memory and continue from one
 * replay to the next, so a replayed call gives the same results as a
 * direct one, provided the communicator's launches (captured or not) stay
 * ordered. A replay does not run the host's LL flag-wrap accounting (the
 * FIFOs are cleared before a 32-bit LL flag could repeat); that takes
 * about 2^31 LL steps per ring edge, i.e. millions of replayed LL calls.
 *
 * Errors. Synchronous errors return a code and launch nothing. A device-
 * side failure (a wait that timed out, or an abort) is reported later by
 * vrcclCommGetAsyncError; after it the communicator accepts only
 * vrcclCommGetAsyncError, vrcclCommGetErrorInfo and vrcclCommDestroy
 * (as a revoked NCCL communicator fails fast, [Deep Dive (Japanese
 * edition) ch.6, ncclEnqueueCheck step 1]).
 */
#ifndef VRCCL_H_
#define VRCCL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define VRCCL_VERSION_MAJOR 0
#define VRCCL_VERSION_MINOR 1

/* Largest number of virtual ranks one communicator accepts. */
#define VRCCL_MAX_RANKS 128
/* Largest channel count (NCCL's MAXCHANNELS, [Architecture §5.2]). */
#define VRCCL_MAX_CHANNELS 64
/* FIFO depth per edge and protocol: slots a sender may fill ahead of its
 * receiver (NCCL_STEPS is 8, [Architecture §6.5]; one GPU's HBM hop costs a
 * few microseconds, so twice NCCL's depth keeps ~100 KB in flight per edge). */
#define VRCCL_STEPS 16

typedef struct vrcclComm* vrcclComm_t;
typedef void* vrcclStream_t; /* a cudaStream_t */

/* Result codes, after ncclResult_t [Deep Dive (Japanese edition) ch.5]. */
typedef enum {
  vrcclSuccess = 0,
  vrcclInvalidArgument = 1, /* a bad pointer, size, enum or handle */
  vrcclInvalidUsage = 2,    /* a valid request this communicator or GPU cannot serve */
  vrcclInternalError = 3,
  vrcclCudaError = 4,       /* a CUDA runtime call failed */
  vrcclTimeout = 5,         /* a device-side wait gave up (asynchronous) */
  vrcclAborted = 6,         /* vrcclCommAbort was called (asynchronous) */
  vrcclNumResults = 7
} vrcclResult_t;

/* Element types [Deep Dive §1.3, ncclDataType_t]. Integer sum and prod
 * wrap modulo 2^bits, max and min compare signed (unsigned for uint8), avg
 * is the wrapped sum divided by n, truncating toward zero. bf16 / fp16 /
 * fp32 combine in binary32 and round to the type at every hop; fp64
 * combines in binary64; avg pre-scales each input by 1/n (binary32 for
 * the 2- and 4-byte types, binary64 for fp64). */
typedef enum {
  vrcclInt32 = 0,
  vrcclFloat32 = 1,
  vrcclBfloat16 = 2,
  vrcclFloat16 = 3,
  vrcclInt8 = 4,
  vrcclUint8 = 5,
  vrcclInt64 = 6,
  vrcclFloat64 = 7,
  vrcclNumTypes = 8
} vrcclDataType_t;

typedef enum {
  vrcclSum = 0,
  vrcclProd = 1,
  vrcclMax = 2,
  vrcclMin = 3,
  vrcclAvg = 4,
  vrcclNumOps = 5
} vrcclRedOp_t;

/* Schedules [Architecture §7.1]. vrcclAlgoOneShot is not on the pages: an
 * AllReduce that reads all n inputs of an element at once and writes all n
 * outputs (no FIFO), in the ring's association order for the ring's channel
 * count and chunk. It moves only the essential bytes and serves as the HBM
 * bound the ring is measured against; "auto" never picks it. */
typedef enum {
  vrcclAlgoRing = 0,
  vrcclAlgoTree = 1,
  vrcclAlgoAuto = 2,
  vrcclAlgoOneShot = 3
} vrcclAlgo_t;

/* Wire protocols [Architecture §7.2; Deep Dive §2.4]. */
typedef enum {
  vrcclProtoSimple = 0, /* slot of raw data, then a released tail counter */
  vrcclProtoLL = 1,     /* 16-byte lines: 4 B data, 4 B flag, 4 B data, 4 B flag */
  vrcclProtoLL128 = 2,  /* 128-byte lines: 120 B data, 8 B flag */
  vrcclProtoAuto = 3
} vrcclProto_t;

/*
 * vrcclCommInit -- create a communicator of `nranks` virtual ranks on the
 * current CUDA device, able to run up to `nchannels` channels.
 * Model: ncclCommInitAll, one process driving every rank [Deep Dive §1.2].
 * Allocates, on that device, the FIFOs of every protocol for up to
 * nchannels channels, their control words and status words (about
 * 3 * nranks * nchannels * 1.1 MiB), and zeroes them.
 *   comm      out: the new handle; owned by the caller until
 *             vrcclCommDestroy.
 *   nranks    1..VRCCL_MAX_RANKS.
 *   nchannels 1..VRCCL_MAX_CHANNELS; an upper bound, calls may use fewer.
 * Errors: vrcclInvalidArgument (null comm, out-of-range sizes);
 *         vrcclCudaError (no device, allocation failed; nothing is leaked).
 * Environment, read once here: VRCCL_TIMEOUT_MS (device wait limit,
 * default 2000), VRCCL_DEBUG=INFO (prints each call's decision line),
 * VRCCL_ALGO / VRCCL_PROTO (NCCL_ALGO / NCCL_PROTO's list syntax, see
 * vrcclParseList: what "auto" may choose; an unknown name makes this call
 * return vrcclInvalidArgument), VRCCL_NCHANNELS (channel count "auto" uses),
 * VRCCL_SLICE_BYTES (largest Simple FIFO slot to use, bytes; default and
 * most 32768), VRCCL_SIMPLE_WARPS (most consumer warps per Simple agent, at
 * most 16; default 16 for 2-byte types, 8 for 4-byte ones), VRCCL_PREFETCH (input slices a Simple agent pulls into L2
 * ahead of use, default 0 = off, at most 32), VRCCL_DIRECT (default 1; 0
 * selects the FIFO all-gather, see vrcclCommSetDirect), VRCCL_TUNE_FILE (a measured
 * tuning table, see vrcclCommLoadTuning; without it the table shipped next
 * to the library, tuning/gb300_n<nranks>.txt, is used when present).
 */
vrcclResult_t vrcclCommInit(vrcclComm_t* comm, int nranks, int nchannels);

/*
 * vrcclAllReduce -- AllReduce of `count` elements over the communicator's
 * n virtual ranks, enqueued on `stream` as one kernel launch.
 * Model: ncclAllReduce(sendbuff, recvbuff, count, datatype, op, comm,
 * stream) [Deep Dive §1.3], with the n per-rank pointers of a
 * single-process clique passed together and the algorithm and protocol
 * selectable per call.
 *   sendbufs  host array of n device pointers; sendbufs[r] holds `count`
 *             elements of `dtype`. Read during the call only.
 *   recvbufs  host array of n device pointers; recvbufs[r] receives
 *             `count` elements. recvbufs[r] == sendbufs[r] (in place) is
 *             allowed; any other overlap between the 2n buffers is not.
 *   count     elements per rank. 0 -> success, nothing launched, and the
 *             buffer pointers are not examined (they may be NULL)
 *             [Deep Dive (Japanese edition) ch.6, taskAppend step 4].
 *   dtype, op as above.
 *   algo      ring, tree, auto (the tuning table's choice among ring and
 *             tree), or one-shot (same bits as the ring with the same
 *             channel count and chunk; `proto` is then ignored).
 *   proto     simple, ll, ll128, or auto (the tuning table's choice).
 *   comm      a live communicator.
 *   stream    cudaStream_t on the communicator's device.
 * Every pointer must be 16-byte aligned. With n == 1 the result is a
 * copy of the input (after the avg scale), launched as the same kernel.
 * Errors: vrcclInvalidArgument (null/misaligned/overlapping pointers, bad
 * enum, null comm); vrcclInvalidUsage (communicator already failed, or the
 * forced schedule cannot be made co-resident on this GPU); vrcclCudaError
 * (launch failure).
 */
vrcclResult_t vrcclAllReduce(const void* const* sendbufs, void* const* recvbufs, size_t count,
                             vrcclDataType_t dtype, vrcclRedOp_t op, vrcclAlgo_t algo,
                             vrcclProto_t proto, vrcclComm_t comm, vrcclStream_t stream);

/*
 * vrcclReduceScatter -- the reduce-scatter phase of the ring AllReduce run
 * alone [Deep Dive §2.3: the AllReduce is a reduce-scatter phase and an
 * all-gather phase of n-1 steps each]. Block r of every rank's send buffer
 * is reduced into rank r's recv buffer, one launch on `stream`. The pages
 * give the phase, not a buffer contract; NCCL's ncclReduceScatter contract
 * is followed.
 *   sendbufs  host array of n device pointers; sendbufs[r] holds n blocks
 *             of `recvcount` elements (block q = elements [q*recvcount,
 *             (q+1)*recvcount)). Read during the call only.
 *   recvbufs  host array of n device pointers; recvbufs[r] receives
 *             `recvcount` elements: element e = op over ranks of their
 *             block r, element e, associated in ring order
 *             op(...op(x[r+1], x[r+2])..., x[r]). In place:
 *             recvbufs[r] == sendbufs[r] + r*recvcount elements.
 *   recvcount elements per block; recvcount * element size must be a
 *             multiple of 16 bytes when n > 1, so that every block starts
 *             on a 16-byte boundary. 0 -> success, nothing launched, the
 *             pointers not examined.
 *   dtype, op as for vrcclAllReduce (avg: the same pre-scale / post-op).
 *   proto     simple, ll, ll128, or auto. The schedule is the ring.
 * Channels split each block; a loop takes one chunk of every block. Errors
 * as for vrcclAllReduce, plus vrcclInvalidArgument for a block that is not
 * a multiple of 16 bytes.
 */
vrcclResult_t vrcclReduceScatter(const void* const* sendbufs, void* const* recvbufs, size_t recvcount,
                                 vrcclDataType_t dtype, vrcclRedOp_t op, vrcclProto_t proto,
                                 vrcclComm_t comm, vrcclStream_t stream);

/*
 * vrcclAllGather -- the all-gather phase of the ring AllReduce run alone
 * [Deep Dive §2.3]: rank q's send buffer lands as block q of every rank's
 * recv buffer, bit for bit, one launch on `stream`. NCCL's ncclAllGather
 * contract is followed.
 *   sendbufs  host array of n device pointers; sendbufs[r] holds
 *             `sendcount` elements. Read during the call only.
 *   recvbufs  host array of n device pointers; recvbufs[r] receives n
 *             blocks of `sendcount` elements. In place:
 *             sendbufs[r] == recvbufs[r] + r*sendcount elements.
 *   sendcount elements per block, with the same 16-byte rule as
 *             vrcclReduceScatter. 0 -> success, nothing launched.
 *   dtype     any type; the data moves as 4-byte words (no arithmetic).
 *   proto     simple, ll, ll128, or auto. The schedule is the ring.
 * Errors as for vrcclReduceScatter.
 */
vrcclResult_t vrcclAllGather(const void* const* sendbufs, void* const* recvbufs, size_t sendcount,
                             vrcclDataType_t dtype, vrcclProto_t proto, vrcclComm_t comm,
                             vrcclStream_t stream);

/*
 * vrcclGroupStart / vrcclGroupEnd -- ncclGroupStart / ncclGroupEnd
 * [Architecture §9.2, §9.6; Deep Dive (Japanese edition) ch.5]. Between
 * the two, vrcclAllReduce / vrcclReduceScatter / vrcclAllGather check their
 * arguments (and return any error at once) but only register the call; the
 * outermost vrcclGroupEnd schedules every registered call of every
 * communicator and enqueues it. Groups nest; the depth is per thread.
 * Scheduling, per communicator: AllReduces of one type, op and requested
 * protocol whose algo is ring or auto are sorted by size, largest first,
 * and cut into runs of sizes within 4x of the run's largest
 * (ncclPrepareTasks). A run is scheduled as a whole, by the tuning table at
 * its total size, and enqueued as one launch of the grouped ring kernel
 * (more launches if its pointers exceed the kernel's parameter space);
 * each of its calls gets the channel count a call of its own size would
 * get. Every other call is enqueued alone. The calls of one group are not
 * ordered among themselves: none may touch a buffer another one writes.
 * All of a group's calls on one communicator must use one stream
 * (vrcclInvalidUsage otherwise, at the call). vrcclGroupEnd returns the
 * first error of a launch and drops the calls not yet enqueued; without a
 * matching vrcclGroupStart it returns vrcclInvalidUsage. Like every call
 * here, it only enqueues: synchronise the stream before reading results.
 * vrcclAllReduceNoAlloc is never grouped.
 */
vrcclResult_t vrcclGroupStart(void);
vrcclResult_t vrcclGroupEnd(void);

/*
 * vrcclCommGetGroupSchedule -- what ran for call `index` (0-based, in call
 * order) of the communicator's most recent group: algorithm, protocol,
 * channel count, chunk (elements; together with the channel count it
 * fixes the association order of every float result), and the launch
 * (0-based, in enqueue order within the group) that carried it. Calls that
 * shared a launch report the same launch.
 * Errors: vrcclInvalidArgument (bad handle, index out of range);
 * vrcclInvalidUsage (nothing ran for that call: count 0).
 */
vrcclResult_t vrcclCommGetGroupSchedule(vrcclComm_t comm, int index, int* algo, int* proto, int* nchannels,
                                        size_t* chunkElems, int* launch);

/*
 * vrcclParseList -- the list syntax of VRCCL_ALGO / VRCCL_PROTO, which is
 * NCCL_ALGO / NCCL_PROTO's (parseList, [Architecture §8.5]): elements are
 * comma separated; a leading '^' excludes the listed names instead; a
 * "function:" prefix restricts a list to one collective; ';' separates
 * lists, the first of which may have no prefix (it applies to every
 * collective). Names are case-insensitive and are NCCL's: functions
 * Broadcast, Reduce, AllGather, ReduceScatter, AllReduce; algorithms Tree,
 * Ring, CollNetDirect, CollNetChain, NVLS, NVLSTree, PAT; protocols LL,
 * LL128, Simple. Of those this library has Ring and Tree (AllReduce; the
 * others are ring-only) and all three protocols; "auto" chooses among the
 * allowed ones, and a call left with none returns vrcclInvalidUsage.
 *   spec   the string (NULL or empty: everything allowed).
 *   kind   0 = algorithms, 1 = protocols.
 *   masks  out: 5 masks, one per function in the order above; bit i is the
 *          i-th name of the kind in the order above.
 * Errors: vrcclInvalidArgument for an unknown name (then vrcclCommInit
 * refuses the same string in the environment).
 */
vrcclResult_t vrcclParseList(const char* spec, int kind, unsigned* masks);

/*
 * vrcclModelPredict -- the pages' analytic model of an AllReduce's time,
 * T = latency * numPipeOps(ring) + bytes / (1000 * algorithm bandwidth) us
 * (ncclTopoTuneModel / ncclTopoGetAlgoTime, [Architecture §8.1-§8.3]),
 * with the constants the pages print. It serves to set the measured tuning
 * table beside the pages' model; the library never schedules by it.
 *   graph      ranks, nodes, channels, per-channel link bandwidth (GB/s)
 *              inside a node and across nodes, extra latency per inter-node
 *              step (us), intra-node hardware (0 NVLink, 1 PCI), GPU
 *              architecture (0 Volta, 1 Ampere, 2 Hopper, 3 Blackwell).
 *   algo       ring or tree; proto: simple, ll or ll128.
 *   bytes      message size; numPipeOps: operations aggregated with it (>= 1).
 *   latUs, algBwGBs, timeUs  out (each may be NULL).
 * Errors: vrcclInvalidArgument for an inconsistent graph or a bad enum.
 */
typedef struct {
  int nranks;
  int nnodes;
  int nchannels;
  float bwIntra;
  float bwInter;
  float latencyInter;
  int hwIntra;
  int arch;
} vrcclModelGraph_t;
vrcclResult_t vrcclModelPredict(const vrcclModelGraph_t* graph, vrcclAlgo_t algo, vrcclProto_t proto, size_t bytes,
                                int numPipeOps, float* latUs, float* algBwGBs, float* timeUs);

/*
 * vrcclCommSetDirect -- 1 (the default): the communicator's later ring /
 * Simple AllReduces and AllGathers run the all-gather through the ranks'
 * recv buffers instead of the FIFOs (the directRecvCopyDirectSend primitives of runRing, which
 * read and write a peer's user buffer where the ranks can address each
 * other, [Architecture §9.4, §10]): the step that finishes chunk r writes
 * it to rank r's recv buffer and straight into rank r+1's, each later step
 * forwards it from the rank's own recv buffer into the next rank's, and a
 * counter per ring edge, released after the writes, tells the next rank it
 * is there. The reduce-scatter still moves through the FIFOs. Results are
 * bit-identical to the FIFO form, which moves (6n-4) S bytes through the
 * SMs against the direct form's (5n-4) S. A standalone AllGather moves
 * each block the same way: written into the next rank's recv buffer, then
 * forwarded from there; grouped AllReduces do the same task by task. 0 (or
 * VRCCL_DIRECT=0 at vrcclCommInit) selects the FIFO all-gather. LL, LL128,
 * the tree and ReduceScatter always use the FIFOs.
 * Errors: vrcclInvalidArgument (bad handle, enable not 0 or 1).
 */
vrcclResult_t vrcclCommSetDirect(vrcclComm_t comm, int enable);

/*
 * vrcclCommSetSchedule -- pin the channel count and chunk size used by
 * later calls (0 = choose automatically, the default).
 *   nchannels  0, or 1..the communicator's nchannels.
 *   chunkBytes 0, or the ring chunk size K*E in bytes: a multiple of 16
 *              and at most VRCCL_STEPS/2 FIFO slots of the protocol in use
 *              (ALLREDUCE_CHUNKSTEPS = NCCL_STEPS/2, [Deep Dive (Japanese
 *              edition) ch.6]); a larger value is clamped at call time.
 * Errors: vrcclInvalidArgument.
 */
vrcclResult_t vrcclCommSetSchedule(vrcclComm_t comm, int nchannels, size_t chunkBytes);

/*
 * vrcclCommGetLastSchedule -- the schedule the last successful
 * vrcclAllReduce on this communicator used: algo, proto, channel count
 * and ring chunk size in elements (K). Any output pointer may be NULL.
 * With this a checker can replay the exact association order.
 * Errors: vrcclInvalidArgument (null comm); vrcclInvalidUsage (no call yet).
 */
vrcclResult_t vrcclCommGetLastSchedule(vrcclComm_t comm, int* algo, int* proto, int* nchannels,
                                       size_t* chunkElems);

/*
 * vrcclCommGetAsyncError -- the communicator's device-side status:
 * vrcclSuccess, vrcclTimeout or vrcclAborted
 * [Deep Dive §1.4, ncclCommGetAsyncError]. Does not wait for running
 * work; reads the status word through an internal stream.
 * Errors: vrcclInvalidArgument; vrcclCudaError.
 */
vrcclResult_t vrcclCommGetAsyncError(vrcclComm_t comm, vrcclResult_t* asyncErr);

/*
 * vrcclCommGetErrorInfo -- where the first device-side failure happened:
 * the virtual rank, channel and FIFO step of the wait that gave up (all -1
 * / 0 when there was none). Any output pointer may be NULL.
 */
vrcclResult_t vrcclCommGetErrorInfo(vrcclComm_t comm, int* rank, int* channel, uint64_t* step);

/*
 * vrcclCommSetTimeout -- device wait limit in milliseconds for later
 * launches (1..3600000). Every device spin-wait gives up after this long,
 * records vrcclTimeout and makes every other agent of the launch return.
 */
vrcclResult_t vrcclCommSetTimeout(vrcclComm_t comm, uint64_t timeoutMs);

/*
 * vrcclCommAbort -- raise the communicator's abort word, which every
 * device wait polls; running and later launches return early and the
 * communicator reports vrcclAborted [Deep Dive §1.4; Architecture §9.5,
 * abortFlag]. The communicator must still be destroyed.
 */
vrcclResult_t vrcclCommAbort(vrcclComm_t comm);

/*
 * vrcclCommDestroy -- wait for the communicator's work to finish
 * (device-synchronising), free everything it allocated, and invalidate
 * the handle. NULL is accepted and ignored.
 */
vrcclResult_t vrcclCommDestroy(vrcclComm_t comm);

/* vrcclCommCount -- the number of virtual ranks [Deep Dive §1.2]. */
vrcclResult_t vrcclCommCount(vrcclComm_t comm, int* nranks);

/* vrcclGetErrorString -- a static, human-readable name of a result code. */
const char* vrcclGetErrorString(vrcclResult_t result);

/*
 * vrcclCommInjectFault -- testing aid: in every later launch, agent
 * (rank, channel) of the given algorithm returns without doing its work
 * once it reaches FIFO step `afterSteps` of the launch, so its peers' waits
 * run out (a flag that nothing sets). rank = -1 clears the fault. Nothing
 * faults or traps: the launch ends when the waits give up.
 */
vrcclResult_t vrcclCommInjectFault(vrcclComm_t comm, int rank, int channel, int afterSteps);

/*
 * vrcclCommGetLaunchShape -- the launch geometry of the last successful
 * vrcclAllReduce: CTAs (one per agent), threads per CTA and elements per
 * FIFO slot. Any output pointer may be NULL.
 * Errors: vrcclInvalidArgument; vrcclInvalidUsage (no call yet).
 */
vrcclResult_t vrcclCommGetLaunchShape(vrcclComm_t comm, int* blocks, int* threads, int* sliceElems);

/*
 * vrcclCommLoadTuning -- replace the communicator's tuning table with the
 * entries of a measured table file that match its rank count. NCCL fills
 * latency/bandwidth tables from constants and takes the smallest predicted
 * time T = lat + bytes/bw [Architecture §8.2]; this table holds measured
 * times instead, and algo/proto/channels "auto" take its minimum at the
 * nearest measured power-of-two size. File format, one entry per line:
 *   nranks algo proto channels log2bytes sliceBytes microseconds [elementBytes]
 * ('#' starts a comment; algo/proto use the enum values above). A line with
 * elementBytes (1, 2, 4 or 8) applies to calls whose element type has that
 * size; a line without it applies to every element type. A call takes the
 * rows of its own element size if the table has any, else the rows without
 * one, else those of the nearest element size (the larger on a tie).
 *   loaded  out (may be NULL): entries kept.
 * Errors: vrcclInvalidArgument (null comm/path, unreadable file).
 */
vrcclResult_t vrcclCommLoadTuning(vrcclComm_t comm, const char* path, int* loaded);

/*
 * vrcclShardRange -- the part of one virtual-rank problem that GPU `shard`
 * of `nshards` computes, when the problem's element range is split across
 * GPUs [Architecture §6.3: channels own independent contiguous ranges and
 * never synchronise, so the channel partition of Deep Dive §2.2 applies one
 * level up]. Parts are contiguous, in shard order, of alignUp(ceil(count /
 * nshards), 16 bytes) elements; trailing parts may be short or empty. Each
 * GPU holds the n virtual ranks' slices [offset, offset + length) of their
 * buffers and runs vrcclAllReduce on them with a communicator of its own
 * (no data moves between GPUs: the outputs are disjoint). Host only.
 *   count    elements per virtual rank of the whole problem.
 *   offset, length  out: the shard's first element and element count.
 * Errors: vrcclInvalidArgument (bad dtype, nshards < 1, shard outside
 * [0, nshards), null outputs).
 */
vrcclResult_t vrcclShardRange(size_t count, vrcclDataType_t dtype, int nshards, int shard, size_t* offset,
                              size_t* length);

/*
 * vrcclAllReduceNoAlloc -- the ring / Simple AllReduce of vrcclAllReduce,
 * for callers that cannot allocate device memory when they need it (code
 * running under a memory-pool manager that owns all of the device's
 * memory, or a latency-critical path that cannot take cudaMalloc's implicit
 * device synchronisation) and keep no communicator. The pages have no
 * counterpart: NCCL always reduces through a communicator's buffers.
 *   sendbufs, recvbufs, count, dtype, op, stream: as for vrcclAllReduce
 *             (caller-owned, 16-byte aligned device buffers; in place
 *             allowed).
 *   nranks    1..32 virtual ranks (the count of sendbufs / recvbufs).
 * Schedule: ring, Simple, min(4, 32 / nranks) channels, chunk 256 KiB
 * (= vrcclCommSetSchedule(comm, that many channels, 262144) on the
 * communicator path, with identical results).
 * Memory: allocates nothing. Its scratch (FIFO slots, counters, status;
 * about 16 MiB) is one static device array that every GPU loading the
 * library holds until the process exits. The first call on a device looks
 * up that array's address, prepares the kernels and reads VRCCL_TIMEOUT_MS;
 * make that first call before any stream capture (a set-up that fails is
 * not kept: the next call tries again). Every call then zeroes the
 * counters and status words on `stream` and launches one kernel; calls
 * share the array, so calls that overlap on the GPU (other streams, other
 * host threads) race and give undefined results -- order them.
 * Errors: vrcclInvalidArgument (null/misaligned pointers, bad enum,
 * nranks < 1, buffers that overlap other than in place); vrcclInvalidUsage
 * (nranks > 32: the scratch is too small -- use a communicator);
 * vrcclCudaError / vrcclInternalError (set-up or launch failed).
 * Device-side failures are not reported (there is no communicator to
 * ask): a wait still gives up after VRCCL_TIMEOUT_MS (default 2 s) and
 * the kernel returns, but the call has already returned vrcclSuccess and
 * the recv buffers are then undefined.
 */
vrcclResult_t vrcclAllReduceNoAlloc(const void* const* sendbufs, void* const* recvbufs, size_t count, int nranks,
                                    vrcclDataType_t dtype, vrcclRedOp_t op, vrcclStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* VRCCL_H_ */
