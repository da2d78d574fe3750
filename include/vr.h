/*
 * vr.h -- C ABI of the virtual-rank ring AllReduce library (libvr.so).
 *
 * N "virtual ranks" each own one send buffer and one receive buffer of `count`
 * elements, all on the same GPU. vrAllReduce leaves in every receive buffer
 * the elementwise reduction of the N send buffers, computed by the ring
 * schedule of NCCL's ring AllReduce: per channel, N-1 reduce-scatter stages
 * then N-1 all-gather stages, moving chunks from rank r to rank r+1 through
 * per-edge FIFO staging buffers in one of three protocol formats.
 *
 * The reduction order is fixed by the schedule ("NCCL 原始碼解讀：一個
 * AllReduce 的 GPU 旅程", ch.2 §2.3, RingARAlgorithm::getNextSendAddr): within
 * each loop of N*chunk elements of a channel, chunk c is first sent by rank
 * c+1 and accumulates ranks c+2, ..., c in ring order, op(incoming, own),
 * rounded to the element type after every op. Results are therefore bit-exact
 * reproducible for every dtype, including floating point, for a given
 * (nRanks, nChannels, chunkBytes, count).
 *
 * Conventions for every entry point:
 *  - Pointers named "device" must be device (or managed) memory of the GPU
 *    that was current when the communicator was created. Pointers named
 *    "host" are ordinary host memory read during the call only.
 *  - No call retains a caller pointer after it returns, except that device
 *    buffers passed to vrAllReduce are accessed by the enqueued kernel until
 *    it completes on `stream`.
 *  - A communicator is not thread-safe; calls on one communicator must be
 *    issued from one thread at a time and enqueued on one stream (the same
 *    stream for every vrAllReduce on that communicator), like an NCCL
 *    communicator ("NCCL 原始碼解讀", ch.2 §2.1).
 *  - Errors are returned, never raised; no entry point aborts the process.
 */
#ifndef VR_H_
#define VR_H_

#include <stddef.h>
#include <stdint.h>

/* Exported symbol marker: the library is built with hidden visibility and
 * exports exactly the entry points declared here. */
#if defined(__GNUC__)
#define VR_API __attribute__((visibility("default")))
#else
#define VR_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque communicator handle (analog of ncclComm_t, "NCCL 原始碼解讀", ch.2
 * §2.1): owns the FIFO arena, the control words, the status word and the
 * per-call step base. Checked against a registry of live handles, so a
 * destroyed handle is rejected with vrInvalidArgument. */
typedef struct vrComm* vrComm_t;

/* Result codes. Mirror the shape of ncclResult_t ("NCCL 原始碼解讀", ch.1
 * §1.2 and ch.3 §3.1: invalid argument / invalid usage / internal error, and
 * ch.2 §2.1 asyncResult for errors found after enqueue). */
typedef enum {
  vrSuccess = 0,
  vrInvalidArgument = 1, /* null pointer, bad rank/channel count, unknown enum,
                            misaligned pointer, chunkBytes not a multiple of 16,
                            or a handle that is not a live communicator */
  vrInvalidUsage = 2,    /* valid arguments the device cannot run: too many
                            ranks x channels to be co-resident, FIFO too large */
  vrCudaError = 3,       /* a CUDA runtime call failed */
  vrInternalError = 4,   /* a bug in this library */
  vrTimeout = 5,         /* a device-side wait gave up (sticky, see below) */
  vrNumResults = 6
} vrResult_t;

/* FIFO protocols ("NCCL 原始碼解讀", ch.2 §2.4; bandwidth factors ch.5 §三):
 *  Simple: whole slots, one tail counter per slot step (producer) and one head
 *          counter (consumer), each on its own 128-byte line.
 *  LL:     16-byte lines of two 8-byte words {32-bit payload, 32-bit flag};
 *          data and flag arrive together, 50 % payload.
 *  LL128:  128-byte lines of 120 payload bytes and an 8-byte flag, 120/128
 *          payload. */
typedef enum { vrProtoSimple = 0, vrProtoLL = 1, vrProtoLL128 = 2, vrNumProtos = 3 } vrProto_t;

/* Element types. float16 is IEEE binary16, bfloat16 the upper half of binary32.
 * vrFloat8e4m3 and vrFloat8e5m2 are the OCP 8-bit floating-point formats
 * (E4M3: bias 7, no infinities, 0x7F/0xFF NaN, largest finite 448; E5M2:
 * bias 15, IEEE-like infinities and NaNs, largest finite 57344), the FP8
 * types that NCCL reduces on sm90 and later ("NCCL 原始碼解讀", ch.6, the FP8
 * type check). Their sum and product are computed exactly and rounded to
 * nearest even, a result past the largest finite value (or infinite)
 * saturating to it with its sign. */
typedef enum {
  vrInt8 = 0, vrUint8 = 1, vrInt32 = 2, vrUint32 = 3, vrInt64 = 4, vrUint64 = 5,
  vrFloat16 = 6, vrBfloat16 = 7, vrFloat32 = 8, vrFloat64 = 9, vrFloat8e4m3 = 10,
  vrFloat8e5m2 = 11, vrNumTypes = 12
} vrDataType_t;

/* Reductions. Integer sum and prod wrap (two's complement); max/min are
 * a > b ? a : b and a < b ? a : b (NaN behaviour unspecified).
 * vrAvg is the sum divided by nRanks, computed as the device op the host op
 * turns into ("NCCL 原始碼解讀", ch.6, hostToDevRedOp): for floating types
 * every rank's element is first multiplied by 1/nRanks (the factor rounded to
 * the element type, each product rounded to it), then summed in the ring's
 * order; for integer types the wrapped sum is divided by nRanks afterwards,
 * truncating toward zero (C division). Values >= vrNumOps are pre-multiplied
 * sums made by vrRedOpCreatePreMulSum on one communicator. */
typedef enum {
  vrSum = 0, vrProd = 1, vrMax = 2, vrMin = 3, vrAvg = 4, vrNumOps = 5
} vrRedOp_t;

/* Largest supported nRanks. */
#define VR_MAX_RANKS 128
/* Largest supported nChannels. */
#define VR_MAX_CHANNELS 128

/* Create a communicator for nRanks virtual ranks on the current CUDA device.
 * ("NCCL 原始碼解讀", ch.1 §1.2 ncclCommInitAll; ch.3 §3.3 commAlloc.)
 *  comm       [out, host] receives the handle; unchanged on error.
 *  nRanks     1 .. VR_MAX_RANKS.
 *  nChannels  1 .. VR_MAX_CHANNELS: the buffer is split into nChannels
 *             contiguous ranges (each divUp(count, nChannels) rounded up to 16
 *             bytes of elements), reduced independently and concurrently
 *             ("NCCL 原始碼解讀", ch.2 §2.2).
 *  proto      FIFO protocol.
 *  chunkBytes payload bytes per ring chunk; a multiple of 16, >= 16. It fixes
 *             the loop size N*chunkBytes and so the reduction order.
 * Allocates (cudaMalloc) the FIFO arena and control words, and a pinned host
 * status mirror; zeroes them. Environment knobs that never change results:
 * VR_FIFO_SLOT_BYTES (multiple of 256, 1 KiB..1 MiB), VR_FIFO_DEPTH
 * (2..64), VR_TRANSPORT (auto|global|warp|warpcluster), VR_CLUSTER_CTAS
 * (warpcluster: CTAs C a ring spans, 2 <= C <= min(16, nRanks) with
 * ceil(nRanks / C) <= 16), VR_FIFO_IN_DEPTH, VR_LATENCY_KERNEL (0: calls that
 * fit one pass of their rings, and Simple calls on rings inside one CTA, stay
 * on the general kernel), VR_TIMEOUT_MS,
 * VR_DEBUG (print the plan). Test only: VR_DEBUG_SILENT_RANK=k
 * makes virtual rank k never signal its neighbours, so that the others' waits
 * run out (vrTimeout). */
VR_API vrResult_t vrCommCreate(vrComm_t* comm, int nRanks, int nChannels, vrProto_t proto,
                        size_t chunkBytes);

/* Enqueue one AllReduce on `stream` (a cudaStream_t; NULL = legacy default).
 * ("NCCL 原始碼解讀", ch.1 §1.3 ncclAllReduce.)
 *  sendbufs [host array of nRanks device pointers] rank r's input; read only.
 *  recvbufs [host array of nRanks device pointers] rank r's output. In place
 *           (sendbufs[r] == recvbufs[r]) is allowed; other overlaps are not.
 *  count    elements per rank. 0 returns vrSuccess and launches nothing; the
 *           buffer pointers are then not examined (they may be NULL).
 *  dtype, op  element type and reduction.
 * Every pointer must be aligned to the element size; 16-byte-aligned buffers
 * take the vectorised path. The two host arrays are read during the call only.
 * Asynchronous: returns once the work is enqueued; synchronise `stream` before
 * reading the outputs. nRanks == 1 is a device-to-device copy (a scaling
 * kernel for a floating vrAvg or a pre-multiplied sum).
 * vrAvg and pre-multiplied sums run on the warp transports (vrCommGetInfo
 * transport 2 or 3) only: vrInvalidUsage on the others.
 * Returns vrTimeout without enqueuing if an earlier call on this communicator
 * timed out (sticky, like NCCL's asyncResult): destroy the communicator. */
VR_API vrResult_t vrAllReduce(vrComm_t comm, const void* const* sendbufs, void* const* recvbufs,
                       size_t count, vrDataType_t dtype, vrRedOp_t op, void* stream);

/* ReduceScatter on the ring: the reduce-scatter half of the AllReduce
 * schedule ("NCCL 原始碼解讀", ch.2 §2.3, the first (N-1)·chunkSteps steps
 * of nStepsPerLoop; traffic factor nRanks, ch.6 §五). Block b is folded
 * from rank b+1 around the ring to rank b, op(incoming, own), rounded to
 * the element type after every op.
 *  sendbufs [host array of nRanks device pointers] rank r's input of
 *           nRanks * recvcount elements; block b = elements
 *           [b * recvcount, (b + 1) * recvcount).
 *  recvbufs [host array of nRanks device pointers] rank r's output of
 *           recvcount elements: the reduction of block r. In place:
 *           recvbufs[r] == sendbufs[r] + r * recvcount elements.
 * Same rules as vrAllReduce otherwise. Runs on the warp transports
 * (vrCommGetInfo transport 2 or 3); vrInvalidUsage on the others. */
VR_API vrResult_t vrReduceScatter(vrComm_t comm, const void* const* sendbufs,
                                  void* const* recvbufs, size_t recvcount, vrDataType_t dtype,
                                  vrRedOp_t op, void* stream);

/* AllGather on the ring: the all-gather half of the schedule. Rank r's
 * output of nRanks * sendcount elements holds rank b's input in block b. The
 * data moves as bytes (as NCCL converts AllGather to int8, "NCCL 原始碼解讀",
 * ch.6); dtype only sets the element size.
 *  sendbufs [host array of nRanks device pointers] sendcount elements each.
 *  recvbufs [host array of nRanks device pointers] nRanks * sendcount each.
 *           In place: sendbufs[r] == recvbufs[r] + r * sendcount elements.
 * Same rules and transport restriction as vrReduceScatter. */
VR_API vrResult_t vrAllGather(vrComm_t comm, const void* const* sendbufs, void* const* recvbufs,
                              size_t sendcount, vrDataType_t dtype, void* stream);

/* AllReduce by the double binary tree ("NCCL 原始碼解讀", ch.4 ncclGetBtree /
 * ncclGetDtree; "NCCL 初始化流程源码级剖析", NCCL Tree 拓扑, Double Binary
 * Tree): the first alignUp(divUp(count, 2), 16/e) elements are reduced up the
 * first tree and broadcast back down it, the rest on the second tree; a node
 * combines its own element, then its first child's value, then its second
 * child's, op rounded to the element type at every step. Tree 0: rank 0 the
 * root, its child the largest power of two below N; rank r with lowest set bit
 * b under (r with bit b cleared, bit 2b set), or r - b when that is out of
 * range; children r - b/2 and r + b/2 (the second halved down while out of
 * range). Tree 1: the mirror r -> N-1-r for even N, tree 0 on ranks shifted by
 * one for odd N. The result differs from vrAllReduce's in floating-point
 * rounding (another order), not in integer or max/min results.
 * Same arguments and rules as vrAllReduce (in place allowed, count 0 returns
 * vrSuccess, nRanks 1 is a copy, sticky vrTimeout). Every rank is two warps:
 * a tree of up to 16 ranks lies in one CTA, a larger one spans the C CTAs of
 * a thread-block cluster, ceil(nRanks / C) or floor(nRanks / C) ranks in each
 * (the smallest C <= 16 leaving at most 16 ranks in each, or VR_CLUSTER_CTAS;
 * vrInvalidUsage if none). The Simple protocol
 * is used whatever the communicator's; its FIFOs live in shared memory (the
 * communicator's arena is not used). vrAvg and pre-multiplied sums scale the
 * inputs as vrAllReduce does (the integer average divides at the root). */
VR_API vrResult_t vrAllReduceTree(vrComm_t comm, const void* const* sendbufs,
                                  void* const* recvbufs, size_t count, vrDataType_t dtype,
                                  vrRedOp_t op, void* stream);

/* Calibration: the AllReduce's result without the ring. For every chunk c of
 * the ring schedule of this communicator (channels, loops of nRanks chunks of
 * chunkBytes, the last loop's chunk alignUp(divUp(rem, N), 16/e):
 * "NCCL 原始碼解讀", ch.2 §2.2-2.3), one kernel loads the N ranks' elements,
 * folds them in ring order from rank (c + 1) mod N, op(incoming, own) rounded
 * to the element type at every hop, and writes the fold to every output. The
 * result is bit for bit vrAllReduce's; the HBM traffic is the least the
 * operation allows (every input read once, every output written once), with
 * no FIFO, flag or wait. It measures the attainable ceiling of the ring
 * kernels on this GPU; it is not the ring.
 * Same arguments and rules as vrAllReduce (in place allowed, count 0 returns
 * vrSuccess), on any transport; it touches none of the communicator's FIFOs
 * and ignores its sticky timeout. */
VR_API vrResult_t vrRingWalk(vrComm_t comm, const void* const* sendbufs, void* const* recvbufs,
                             size_t count, vrDataType_t dtype, vrRedOp_t op, void* stream);

/* Wait for this communicator's outstanding work, free its memory and
 * invalidate the handle. ("NCCL 原始碼解讀", ch.1 §1.4.) Using the handle
 * afterwards returns vrInvalidArgument. */
VR_API vrResult_t vrCommDestroy(vrComm_t comm);

/* Report a device-side error found after enqueue, without synchronising
 * ("NCCL 原始碼解讀", ch.1 §1.4 ncclCommGetAsyncError). *asyncErr [out, host]
 * is vrSuccess, or vrTimeout once any wait of any kernel of this communicator
 * has given up. */
VR_API vrResult_t vrCommGetAsyncError(vrComm_t comm, vrResult_t* asyncErr);

/* Set the limit, in milliseconds (>= 1), of every device-side wait of later
 * calls on this communicator. Default 10000, or VR_TIMEOUT_MS. */
VR_API vrResult_t vrCommSetTimeout(vrComm_t comm, uint64_t timeoutMs);

/* Describe the communicator's plan (host ints written when non-NULL):
 * transport 0 = FIFOs in global memory (L2, one CTA per rank and channel;
 * VR_TRANSPORT=global), 2 = every rank a warp and every FIFO in one SM's
 * shared memory (the default for rings of 2 to 16 ranks), 3 = every rank a
 * warp, a ring spread over the C CTAs of a cluster, ceil(nRanks / C) or
 * floor(nRanks / C) ranks in each, with distributed shared memory on the CTA
 * boundaries (the default for 17 to VR_MAX_RANKS ranks); 1 is not used;
 * FIFO slot bytes and depth; device bytes the communicator allocated. */
VR_API vrResult_t vrCommGetInfo(vrComm_t comm, int* transport, int* slotBytes, int* depth,
                         size_t* deviceBytes);

/* The plan of one AllReduce of `count` elements of `dtype` on this
 * communicator, computed on the host (nothing is enqueued): *parts [out,
 * host] = the independent ring passes the call makes (per channel, loops of
 * nRanks chunks, "NCCL 原始碼解讀", ch.2 §2.2-2.3, each chunk moved in parts
 * of half the FIFO, at the FIFO geometry the call uses: on the warp
 * transports a call that needs one pass takes the smallest FIFO slot that
 * keeps it one pass, and a call that would need two or three passes takes,
 * when that saves a pass, one own-data slot per rank and the larger FIFO slot
 * it frees; results do not depend on it); *rings [out, host] = rings that run
 * at once (warp
 * transports: CTAs or clusters x rings per CTA; global: channels). A
 * ring takes its parts one after another, so ceil(parts / rings) passes of
 * 2(nRanks - 1) + 1 stages follow each other. Either pointer may be NULL.
 * vrInvalidArgument for a bad handle or dtype. */
VR_API vrResult_t vrCommGetPlan(vrComm_t comm, size_t count, vrDataType_t dtype, size_t* parts,
                                int* rings);

/* AllReduce without any allocation, for callers that cannot allocate device
 * memory where they need the collective: code under a framework's caching
 * allocator that must account for every device byte (a cudaMalloc of its own
 * could fail once the pool holds the GPU's memory, or upset its books), or a
 * latency-critical path where cudaMalloc/cudaFree would stall the device.
 * The pages have no counterpart of this call; it is this library's addition.
 * It computes exactly what a communicator created with (nRanks, nChannels,
 * proto, chunkBytes) and the global-memory FIFO transport computes, bit for
 * bit: same arguments and rules as vrAllReduce, minus the communicator, and
 * op limited to vrSum..vrMin (vrAvg and pre-multiplied sums need a
 * communicator: vrInvalidArgument).
 * Scratch (FIFOs, control words, status word) lives in one 4 MiB array that
 * the library defines in device memory; every GPU that loads the library
 * holds it until the process exits. Limits: nChannels * nRanks * 8448 + 256
 * bytes must fit in those 4 MiB (nChannels * nRanks <= 496), else
 * vrInvalidUsage; the grid (nChannels * nRanks CTAs) must be co-resident.
 * Calls allocate nothing: no cudaMalloc, cudaFree or allocating library
 * routine. The first call on each device, and the first call of each element
 * type, op and protocol on it, sets that device up (with the device current):
 * it looks up the array's device address and touches the kernel it launches.
 * Under lazy module loading (CUDA_MODULE_LOADING=LAZY, CUDA's default) that
 * set-up loads the library's modules, which reserves the 4 MiB array and
 * may allocate device memory: make those first calls before a caching pool
 * takes the GPU's memory and before any stream capture. A call with count 0
 * does the set-up and nothing else, so it serves as the warm-up. Every call
 * on a device shares the array: the call clears the part it uses
 * (cudaMemsetAsync on `stream`), so calls that overlap on the GPU (on
 * different streams, without ordering between them) race and give undefined
 * results. A device-side wait gives up after VR_TIMEOUT_MS milliseconds of
 * the environment (default 10 s); the outputs of that call are then
 * undefined and vrAllReduceNoAllocGetStatus reports vrTimeout until the next
 * call on the device clears the status. */
VR_API vrResult_t vrAllReduceNoAlloc(const void* const* sendbufs, void* const* recvbufs,
                                     size_t count, int nRanks, int nChannels, vrProto_t proto,
                                     size_t chunkBytes, vrDataType_t dtype, vrRedOp_t op,
                                     void* stream);

/* Status of the last vrAllReduceNoAlloc call on the current device, for the
 * same callers (it allocates nothing either; the pages have no counterpart).
 *  status  [out, host] vrSuccess, or vrTimeout if a device-side wait of that
 *          call gave up.
 * A synchronous read (cudaMemcpy of one word): call it after the stream of
 * the last call has been synchronised and before the next call, which clears
 * the status. vrInvalidArgument for a NULL pointer, vrCudaError if the read
 * fails. */
VR_API vrResult_t vrAllReduceNoAllocGetStatus(vrResult_t* status);

/* Create a pre-multiplied sum on `comm`: a reduction that multiplies every
 * rank's element by `scalar` (the product rounded to `dtype`; integers wrap)
 * and then sums the products in the ring's order ("NCCL 原始碼解讀", ch.6,
 * hostToDevRedOp: the host op becomes a sum whose inputs are scaled).
 *  op      [out, host] the new op, a value >= vrNumOps; unchanged on error.
 *  scalar  [host] one element of `dtype`, read during the call only.
 *  dtype   the element type the op is for: a call with another dtype returns
 *          vrInvalidArgument.
 * Valid on `comm` only, with vrAllReduce and vrReduceScatter on the on-chip
 * transports (warp, warpcluster), vrAllReduceTree and vrRingWalk; the
 * global-FIFO transport returns vrInvalidUsage for it, as it does for
 * vrAvg. At most 16 live ops per communicator (vrInvalidUsage
 * past that). */
VR_API vrResult_t vrRedOpCreatePreMulSum(vrRedOp_t* op, const void* scalar, vrDataType_t dtype,
                                         vrComm_t comm);

/* Release an op made by vrRedOpCreatePreMulSum on `comm`. vrInvalidArgument
 * for anything else. Calls already enqueued keep the scalar they were given. */
VR_API vrResult_t vrRedOpDestroy(vrRedOp_t op, vrComm_t comm);

/* Static description of a result code. Never NULL. */
VR_API const char* vrGetErrorString(vrResult_t result);

#ifdef __cplusplus
}
#endif

#endif /* VR_H_ */
