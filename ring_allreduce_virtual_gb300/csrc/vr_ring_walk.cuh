// vr_ring_walk.cuh -- the ring-walk calibration kernel: the AllReduce's
// result without the ring. For every chunk c of the ring schedule ("NCCL
// 原始碼解讀：一個 AllReduce 的 GPU 旅程", ch.2 §2.2-2.3: channels, loops
// of N chunks, the last loop's chunk alignUp(divUp(rem, N), 16/e)), a thread
// loads the N ranks' 16-byte packs, folds them in ring order from rank
// (c + 1) mod N, op(incoming, own) rounded to the element type at every hop,
// and writes the fold to every rank's output (an average or pre-multiplied
// sum scales it as the ring does). Bit for bit the ring's result,
// with the least HBM traffic the operation allows (N*B read, N*B written) and
// no FIFO, flag or wait: the attainable ceiling the ring kernels are measured
// against. It is a measuring stick, not a ring.
#pragma once

#include "vr_cursor.cuh"

namespace vr {

constexpr int kWalkThreads = 256;
// Ranks whose packs are loaded together before folding (loads in flight).
constexpr int kWalkBatch = 8;

// Segments of a channel: one per chunk of every loop.
__host__ __device__ inline uint64_t walk_segments(const vrChannelShape& sh, int N) {
  return (sh.fullLoops + (sh.lastRem ? 1 : 0)) * (uint64_t)N;
}
// Largest chunk of a channel, in elements.
__host__ __device__ inline uint64_t walk_max_chunk(const vrChannelShape& sh, uint64_t chunkElems) {
  return sh.fullLoops ? chunkElems : sh.lastCur;
}

// Units of work: every segment cut into pieces of walkPieceBytes per rank,
// sized so that every SM has a few (4 KiB .. 64 KiB: one to sixteen 16-byte
// packs per thread).
inline void walk_plan(vrStepPlan& P, int nSMs) {
  const uint64_t bytes = P.nFullCh * P.full.S * P.E + P.last.S * P.E;
  uint64_t piece = align_up(div_up(bytes, 4 * (uint64_t)nSMs), 4096);
  piece = piece < 4096 ? 4096 : piece > 65536 ? 65536 : piece;
  uint64_t maxChunk = P.nFullCh ? walk_max_chunk(P.full, P.chunkElems) : 0;
  if (P.last.S && walk_max_chunk(P.last, P.chunkElems) > maxChunk)
    maxChunk = walk_max_chunk(P.last, P.chunkElems);
  P.walkPieceBytes = piece;
  P.walkPieces = maxChunk ? div_up(maxChunk * P.E, piece) : 1;
}
__host__ __device__ inline uint64_t walk_units(const vrStepPlan& P) {
  const uint64_t segs = P.nFullCh * walk_segments(P.full, P.N) +
                        (P.last.S ? walk_segments(P.last, P.N) : 0);
  return segs * P.walkPieces;
}

// Segment g: elements [lo, hi) of every rank's buffer, all in one chunk, and
// the rank the chunk's fold starts from.
struct WalkSegment {
  uint64_t lo, hi;
  int start;
};

__device__ __forceinline__ WalkSegment walk_segment(const vrStepPlan& P, uint64_t g) {
  const int N = P.N;
  const uint64_t segsFull = walk_segments(P.full, N);
  uint64_t ch, v;
  const vrChannelShape* sh;
  if (g < P.nFullCh * segsFull) {
    ch = g / segsFull;
    v = g - ch * segsFull;
    sh = &P.full;
  } else {
    ch = P.nFullCh;
    v = g - P.nFullCh * segsFull;
    sh = &P.last;
  }
  const uint64_t loop = v / (uint64_t)N;
  const int c = (int)(v - loop * (uint64_t)N);
  const uint64_t cur = loop < sh->fullLoops ? P.chunkElems : sh->lastCur;
  const uint64_t rem = sh->S - loop * P.loopElems;
  const uint64_t base = ch * P.per + loop * P.loopElems;
  const uint64_t lo = (uint64_t)c * cur;
  WalkSegment s;
  s.lo = base + min_u64(lo, rem);
  s.hi = base + min_u64(lo + cur, rem);
  s.start = c + 1 == N ? 0 : c + 1;
  return s;
}

template <typename T, int OP>
__global__ void __launch_bounds__(kWalkThreads)
vr_ring_walk(const __grid_constant__ vrRingArgs a) {
  const vrStepPlan& P = a.plan;
  const int N = P.N;
  constexpr uint64_t E = sizeof(T), PE = 16 / sizeof(T);
  const bool vec = (a.alignMask & 15) == 0;
  const uint4 sPack = scalar_pack<T>(a.scalar);
  const bool premul = OP == 0 && a.scale == VR_SCALE_PREMUL;
  const uint64_t pieces = P.walkPieces;
  const uint64_t pieceElems = P.walkPieceBytes / E;
  const uint64_t nUnits = walk_units(P);
  for (uint64_t u = blockIdx.x; u < nUnits; u += gridDim.x) {
    const uint64_t g = u / pieces, piece = u - g * pieces;
    const WalkSegment s = walk_segment(P, g);
    const uint64_t pLo = s.lo + piece * pieceElems;
    if (pLo >= s.hi) continue;
    const uint64_t pHi = min_u64(s.hi, pLo + pieceElems);
    const uint32_t nPacks = (uint32_t)div_up(pHi - pLo, PE);
    for (uint32_t j = threadIdx.x; j < nPacks; j += kWalkThreads) {
      const uint64_t e0 = pLo + (uint64_t)j * PE;
      const uint32_t valid = (uint32_t)min_u64(16, (pHi - e0) * E);
      const uint64_t off = e0 * E;
      uint4 acc = make_uint4(0, 0, 0, 0);
      int rk = s.start;
      for (int b = 0; b < N; b += kWalkBatch) {
        uint4 x[kWalkBatch];
        int rr = rk;
#pragma unroll
        for (int t = 0; t < kWalkBatch; ++t) {
          if (b + t < N) {
            x[t] = load_pack<T>(static_cast<const char*>(a.send[rr]) + off, valid, vec);
            rr = rr + 1 == N ? 0 : rr + 1;
          }
        }
        // Scale after the whole batch is in flight: a use between the loads
        // would hold the next load back until this one returned.
#pragma unroll
        for (int t = 0; t < kWalkBatch; ++t) {
          if (b + t < N) {
            const uint4 v = premul ? hop16<T, 1>(x[t], sPack) : x[t];
            acc = (b + t == 0) ? v : hop16<T, OP>(acc, v);
          }
        }
        rk = rr;
      }
      if (OP == 0 && a.scale == VR_SCALE_POSTDIV) acc = div_pack<T>(acc, N);
      for (int r = 0; r < N; ++r) store_pack<T>(static_cast<char*>(a.recv[r]) + off, acc, valid, vec);
    }
  }
}

}  // namespace vr

#define VR_INSTANTIATE_WALK(GETTER, T)                                                    \
  const void* GETTER(int op) {                                                           \
    static const void* table[4] = {(const void*)vr::vr_ring_walk<T, 0>,                  \
                                   (const void*)vr::vr_ring_walk<T, 1>,                  \
                                   (const void*)vr::vr_ring_walk<T, 2>,                  \
                                   (const void*)vr::vr_ring_walk<T, 3>};                 \
    return (op < 0 || op > 3) ? nullptr : table[op];                                     \
  }
