// vr_internal.h -- definitions shared by the host launcher and the kernels.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "vr.h"

#ifdef __CUDACC__
#define VR_HD __host__ __device__
#else
#define VR_HD
#endif

// Device status codes (the status word and its host mirror).
enum { VR_STATUS_OK = 0, VR_STATUS_TIMEOUT = 1 };

// Scaling of a sum (the average and the pre-multiplied sum): every rank's
// element multiplied by a scalar as it enters the fold, or the finished sum
// divided by N (integer average).
enum { VR_SCALE_NONE = 0, VR_SCALE_PREMUL = 1, VR_SCALE_POSTDIV = 2 };

// Kernel stage kinds, in the order a rank meets them within one loop.
// Stage k of rank r handles chunk (r - 1 - k) mod N ("NCCL 原始碼解讀：一個
// AllReduce 的 GPU 旅程", ch.2 §2.3, getNextSendAddr):
//   k = 0          SEND     own chunk -> FIFO
//   1 .. N-2       RRS      FIFO + own -> op -> FIFO
//   N-1            RRCS     FIFO + own -> op -> recv and FIFO
//   N .. 2N-3      RCS      FIFO -> recv and FIFO
//   2N-2           RECV     FIFO -> recv
// ReduceScatter adds RRC (the last stage: FIFO + own -> op -> recv, no send)
// and AllGather adds SC (the first stage: own -> FIFO and recv).
enum { VR_SEND = 0, VR_RRS = 1, VR_RRCS = 2, VR_RCS = 3, VR_RECV = 4, VR_RRC = 5, VR_SC = 6 };

// Collectives on the ring. ReduceScatter and AllGather are the two halves of
// the AllReduce schedule ("NCCL 原始碼解讀", ch.2 §2.3: nStepsPerLoop =
// 2 (N - 1) chunkSteps, (N - 1) chunkSteps for each half).
enum { VR_COLL_ALLREDUCE = 0, VR_COLL_REDUCESCATTER = 1, VR_COLL_ALLGATHER = 2 };

// What a stage kind does: receive from rank r-1, send to rank r+1, read the
// rank's own input, write its output, reduce incoming with own.
VR_HD constexpr bool vrKindRecv(int k) { return k != VR_SEND && k != VR_SC; }
VR_HD constexpr bool vrKindSend(int k) { return k != VR_RECV && k != VR_RRC; }
VR_HD constexpr bool vrKindOwn(int k) { return k <= VR_RRCS || k == VR_RRC || k == VR_SC; }
VR_HD constexpr bool vrKindOut(int k) { return k >= VR_RRCS; }
VR_HD constexpr bool vrKindReduce(int k) { return k == VR_RRS || k == VR_RRCS || k == VR_RRC; }

// Threads per CTA of the global-FIFO kernel.
#define VR_GENERIC_THREADS 256
// Packs (16 B) per thread per batch in the Simple data loop.
#define VR_SIMPLE_UNROLL 4
// LL128: 8 lanes per 128-byte line; rows of lines per warp per step.
#define VR_LL128_ROWS 4
// Warp transport: at most this many warps (whole rings of one warp per rank)
// per CTA, so at most this many ranks per ring.
#define VR_WARP_MAX_RANKS 16
#define VR_WARP_MAX_THREADS (32 * VR_WARP_MAX_RANKS)

// Placement of a ring (or a tree) of N ranks over the C CTAs of a thread-block
// cluster: CTA j holds ranks start(j) .. start(j) + size(j) - 1, the first
// N mod C CTAs ceil(N / C) ranks and the others floor(N / C). Any 2 <= C <= N
// works, so every ring size up to 16 C ranks has a split.
struct vrSplit {
  int lo, extra;  // floor(N / C), N mod C
  VR_HD vrSplit(int n, int c) : lo(n / c), extra(n % c) {}
  VR_HD int size(int j) const { return lo + (j < extra ? 1 : 0); }
  VR_HD int start(int j) const { return j * lo + (j < extra ? j : extra); }
  VR_HD int cta_of(int x) const {
    const int b = extra * (lo + 1);  // ranks in the larger CTAs
    return x < b ? x / (lo + 1) : extra + (x - b) / lo;
  }
};

// Control words of one FIFO edge (ch, r -> r+1): tail (written by the sender)
// and head (written by the receiver), each alone on a 128-byte line, like
// ncclSendMem.head / ncclRecvMem.tail ("NCCL 原始碼解讀", ch.2 §2.4).
#define VR_CTRL_WORDS_PER_EDGE 32
#define VR_CTRL_TAIL 0
#define VR_CTRL_HEAD 16

// The walk of one warp-ring call (vr_cursor.cuh), the same for every CTA:
// computed once on the host and read from kernel parameter space.
struct vrChannelShape {
  uint64_t S, fullLoops, lastRem, lastCur, partsFullLoop, partsLastLoop, units;
};
struct vrStepPlan {
  uint64_t per, loopElems, chunkElems, partBytes, payload, E, nFullCh, nUnits, G, blockBytes;
  uint64_t walkPieceBytes, walkPieces;  // ring-walk fold: work unit size, units per chunk
  vrChannelShape full, last;
  int N, coll;
};

// Kernel arguments, passed by value (kernel parameter space): the pointer
// tables are copied at launch, so the caller's host arrays are free on return.
struct vrRingArgs {
  uint64_t count;        // elements per rank
  uint64_t chunkElems;   // chunkBytes / elemSize
  uint64_t stepBase;     // flags of this call are stepBase + local step + 1
  uint64_t timeoutNs;    // limit of every device wait
  char* fifo;            // FIFO arena (global transport)
  uint64_t* ctrl;        // control words (global transport)
  int* status;           // device status word
  int* statusHost;       // device alias of the pinned host status mirror
  int nRanks;
  int nChannels;
  int alignMask;         // OR of the low 4 bits of every buffer pointer
  int silentRank;        // test-only: this rank never posts (-1: none)
  uint32_t slotBytes;    // FIFO slot bytes (one step) per edge
  uint32_t depth;        // FIFO slots per edge
  uint32_t inDepth;      // warp kernels: own-data prefetch slots
  int ringsPerCta;       // warp kernel: rings (or, on a cluster, ring parts) per CTA
  int ringWarps;         // warp kernel on a cluster: ranks of a ring per CTA
  int scale;             // sum kernels: VR_SCALE_* (average, pre-multiplied sum)
  uint64_t scalar;       // VR_SCALE_PREMUL: the scalar's element-type bits
  int coll;              // warp kernel: VR_COLL_*; count is then per block
  vrStepPlan plan;       // warp kernel: the walk of this call
  const void* send[VR_MAX_RANKS];
  void* recv[VR_MAX_RANKS];
};

// Payload bytes one step carries, per protocol, for a slot of `slotBytes`.
VR_HD static inline uint64_t vrPayloadPerStep(int proto, uint64_t slotBytes) {
  if (proto == vrProtoLL) return slotBytes / 2;           // 8 B payload per 16 B line
  if (proto == vrProtoLL128) return slotBytes / 128 * 120; // 120 B per 128 B line
  return slotBytes;
}

// Warp transport: bytes of one own-data slot (a step's payload, rounded up
// to 128 bytes).
VR_HD static inline uint32_t vrOwnSlotBytes(int proto, uint32_t slotBytes) {
  return (uint32_t)((vrPayloadPerStep(proto, slotBytes) + 127) / 128 * 128);
}

// Kernel table, one entry point per element type (one translation unit each);
// each returns the kernel for (op, proto) as a function handle for
// cudaLaunchKernelEx, or NULL.
#define VR_DECLARE_GETTER(NAME) const void* NAME(int op, int proto);
VR_DECLARE_GETTER(vrGetGeneric_i8)
VR_DECLARE_GETTER(vrGetGeneric_u8)
VR_DECLARE_GETTER(vrGetGeneric_i32)
VR_DECLARE_GETTER(vrGetGeneric_u32)
VR_DECLARE_GETTER(vrGetGeneric_i64)
VR_DECLARE_GETTER(vrGetGeneric_u64)
VR_DECLARE_GETTER(vrGetGeneric_f16)
VR_DECLARE_GETTER(vrGetGeneric_bf16)
VR_DECLARE_GETTER(vrGetGeneric_e4m3)
VR_DECLARE_GETTER(vrGetGeneric_e5m2)
VR_DECLARE_GETTER(vrGetGeneric_f32)
VR_DECLARE_GETTER(vrGetGeneric_f64)

// Warp-ring kernels (every rank a warp, FIFOs in shared memory), per op,
// protocol, and whether a ring spans the CTAs of a cluster.
#define VR_DECLARE_WARP_GETTER(NAME) const void* NAME(int op, int proto, int cluster);
VR_DECLARE_WARP_GETTER(vrGetWarp_i8)
VR_DECLARE_WARP_GETTER(vrGetWarp_u8)
VR_DECLARE_WARP_GETTER(vrGetWarp_i32)
VR_DECLARE_WARP_GETTER(vrGetWarp_u32)
VR_DECLARE_WARP_GETTER(vrGetWarp_i64)
VR_DECLARE_WARP_GETTER(vrGetWarp_u64)
VR_DECLARE_WARP_GETTER(vrGetWarp_f16)
VR_DECLARE_WARP_GETTER(vrGetWarp_bf16)
VR_DECLARE_WARP_GETTER(vrGetWarp_e4m3)
VR_DECLARE_WARP_GETTER(vrGetWarp_e5m2)
VR_DECLARE_WARP_GETTER(vrGetWarp_f32)
VR_DECLARE_WARP_GETTER(vrGetWarp_f64)

// Latency kernels (vr_ring_lat.cuh): the warp rings for calls that fit one
// pass of their rings, Simple and LL protocols, per op and whether a ring
// spans the CTAs of a cluster. A step carries at most 32 * VR_LAT_PACKS
// 16-byte packs of payload (each lane at most VR_LAT_PACKS).
#define VR_LAT_PACKS 8
VR_DECLARE_WARP_GETTER(vrGetLat_i8)
VR_DECLARE_WARP_GETTER(vrGetLat_u8)
VR_DECLARE_WARP_GETTER(vrGetLat_i32)
VR_DECLARE_WARP_GETTER(vrGetLat_u32)
VR_DECLARE_WARP_GETTER(vrGetLat_i64)
VR_DECLARE_WARP_GETTER(vrGetLat_u64)
VR_DECLARE_WARP_GETTER(vrGetLat_f16)
VR_DECLARE_WARP_GETTER(vrGetLat_bf16)
VR_DECLARE_WARP_GETTER(vrGetLat_e4m3)
VR_DECLARE_WARP_GETTER(vrGetLat_e5m2)
VR_DECLARE_WARP_GETTER(vrGetLat_f32)
VR_DECLARE_WARP_GETTER(vrGetLat_f64)

// Ring-walk calibration kernels (the fold without FIFOs), per op.
#define VR_DECLARE_WALK_GETTER(NAME) const void* NAME(int op);
VR_DECLARE_WALK_GETTER(vrGetWalk_i8)
VR_DECLARE_WALK_GETTER(vrGetWalk_u8)
VR_DECLARE_WALK_GETTER(vrGetWalk_i32)
VR_DECLARE_WALK_GETTER(vrGetWalk_u32)
VR_DECLARE_WALK_GETTER(vrGetWalk_i64)
VR_DECLARE_WALK_GETTER(vrGetWalk_u64)
VR_DECLARE_WALK_GETTER(vrGetWalk_f16)
VR_DECLARE_WALK_GETTER(vrGetWalk_bf16)
VR_DECLARE_WALK_GETTER(vrGetWalk_e4m3)
VR_DECLARE_WALK_GETTER(vrGetWalk_e5m2)
VR_DECLARE_WALK_GETTER(vrGetWalk_f32)
VR_DECLARE_WALK_GETTER(vrGetWalk_f64)

// Double-binary-tree AllReduce kernels (every rank two warps, tree edges in
// shared memory), Simple protocol, per op and whether a tree spans the CTAs
// of a cluster.
#define VR_DECLARE_TREE_GETTER(NAME) const void* NAME(int op, int cluster);
VR_DECLARE_TREE_GETTER(vrGetTree_i8)
VR_DECLARE_TREE_GETTER(vrGetTree_u8)
VR_DECLARE_TREE_GETTER(vrGetTree_i32)
VR_DECLARE_TREE_GETTER(vrGetTree_u32)
VR_DECLARE_TREE_GETTER(vrGetTree_i64)
VR_DECLARE_TREE_GETTER(vrGetTree_u64)
VR_DECLARE_TREE_GETTER(vrGetTree_f16)
VR_DECLARE_TREE_GETTER(vrGetTree_bf16)
VR_DECLARE_TREE_GETTER(vrGetTree_e4m3)
VR_DECLARE_TREE_GETTER(vrGetTree_e5m2)
VR_DECLARE_TREE_GETTER(vrGetTree_f32)
VR_DECLARE_TREE_GETTER(vrGetTree_f64)
