// vr_ring_warp.cuh -- ring AllReduce with every virtual rank a warp and every
// FIFO in the shared memory of one SM.
//
// A CTA holds R whole rings of N warps each: warp (rho, r) is virtual rank r
// of ring rho. Rank r walks the ring schedule of "NCCL 原始碼解讀：一個
// AllReduce 的 GPU 旅程", ch.2 §2.3 (stage k on chunk (r - 1 - k) mod N,
// reduce-scatter then all-gather, receiving from rank r-1 and sending to rank
// r+1) through its own FIFO edge: `depth` slots of `slotBytes` in shared
// memory, with the Simple protocol's two signals of ch.2 §2.4 as mbarriers --
// "full" (the sender filled a slot) and "empty" (the receiver drained it).
// Every signal is a CTA-local mbarrier, so a hop costs shared-memory latency,
// and the FIFO traffic (about twice the input) never reaches L2 or HBM: HBM
// sees each input byte read once (a bulk TMA copy per step, prefetched
// `inDepth` steps ahead of its use) and each output byte written once.
//
// The ring's parts are independent passes (see vr_cursor.cuh), spread round
// robin over every ring of the grid, so all SMs share the work whatever the
// channel count.
//
// Every wait is bounded by the communicator's timeout; a wait that gives up
// raises the status word and the warp stops, after waiting for its own bulk
// copies to land.
#pragma once

#include "vr_cursor.cuh"
#include "vr_ring_cluster.cuh"  // shared-memory and bulk-copy primitives

namespace vr {

__device__ __forceinline__ void mbar_arrive_cta(uint32_t addr) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cta(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(addr), "r"(parity) : "memory");
  return ok != 0;
}

// Bounded wait by one lane on a CTA-local barrier phase.
__device__ __forceinline__ bool lane_wait_cta(uint32_t addr, uint32_t parity, const vrRingArgs& a) {
  if (mbar_try_wait_cta(addr, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cta(addr, parity)) return true;
    if ((it & 15) == 0) {
      if (ld_volatile_int(a.status) != VR_STATUS_OK) return false;
      if (globaltimer() - t0 > a.timeoutNs) {
        raise_timeout(a);
        return false;
      }
    }
  }
}

// Shared memory of one warp: D FIFO slots (its incoming edge), DI own-data
// slots, then (after all warps' data) its barriers: full[D], empty[D],
// inFull[DI].
struct WarpSmem {
  uint32_t fifo, own, full, empty, inFull;
};

__device__ __forceinline__ WarpSmem warp_smem(uint32_t base, int w, int nWarps, uint32_t D,
                                              uint32_t DI, uint32_t SLOT) {
  WarpSmem m;
  m.fifo = base + (uint32_t)w * (D + DI) * SLOT;
  m.own = m.fifo + D * SLOT;
  const uint32_t bars = base + (uint32_t)nWarps * (D + DI) * SLOT + (uint32_t)w * 8 * (2 * D + DI);
  m.full = bars;
  m.empty = bars + 8 * D;
  m.inFull = bars + 16 * D;
  return m;
}

// Per-warp state of one rank of one ring. Slot indices and mbarrier phase
// bits advance incrementally (no division per step).
struct WarpRank {
  const vrRingArgs* a;
  WarpSmem me, nx;
  const char* own;
  char* out;
  uint32_t sIn, phIn;      // next incoming FIFO slot and its phase
  uint32_t sOut, phOut;    // next outgoing FIFO slot and its phase
  uint32_t iOwn, phOwn;    // next own-data slot and its phase
  uint32_t ownUsed, issued;
  uint32_t D, DI, SLOT;
  int lane;
  bool outWrapped;         // every outgoing slot has been used once
  bool vec16, silent;
};

// The data of one step of stage kind KIND. FULL: a whole slot of aligned
// 16-byte packs (the common case), with no tail checks.
template <typename T, int OP, int KIND, bool FULL>
__device__ __forceinline__ void step_data_body(const WarpRank& w, uint32_t inSlot, uint32_t ownSlot,
                                          uint32_t outSlot, uint64_t off, uint32_t len) {
  constexpr bool rcv = KIND != VR_SEND, snd = KIND != VR_RECV;
  constexpr bool hasOwn = KIND <= VR_RRCS, hasOut = KIND >= VR_RRCS;
  constexpr bool red = KIND == VR_RRS || KIND == VR_RRCS;
  constexpr uint32_t U = 1;  // packs per lane per iteration (16 warps hide the latency)
  const uint32_t nPacks = (len + 15) >> 4;
  const uint32_t ownBytes = w.vec16 ? (len & ~15u) : 0u;
  const char* ownG = w.own + off;
  char* outG = w.out + off;
  for (uint32_t p0 = w.lane; p0 < nPacks; p0 += 32 * U) {
    uint4 v[U], x[U];
#pragma unroll
    for (uint32_t u = 0; u < U; ++u) {
      const uint32_t p = p0 + 32 * u;
      if (FULL || p < nPacks) {
        if (hasOwn) {
          if (FULL || p * 16 + 16 <= ownBytes) v[u] = ld_shared_v4(ownSlot + p * 16);
          else v[u] = load_pack<T>(ownG + (uint64_t)p * 16, len - p * 16, false);
        }
        if (rcv) x[u] = ld_shared_v4(inSlot + p * 16);
      }
    }
#pragma unroll
    for (uint32_t u = 0; u < U; ++u) {
      const uint32_t p = p0 + 32 * u;
      if (FULL || p < nPacks) {
        uint4 res;
        if (KIND == VR_SEND) res = v[u];
        else if (red) res = hop16<T, OP>(x[u], v[u]);
        else res = x[u];
        if (snd) st_shared_v4(outSlot + p * 16, res);
        if (hasOut) {
          if (FULL) st_cs_v4(outG + (uint64_t)p * 16, res);
          else store_pack<T>(outG + (uint64_t)p * 16, res, len - p * 16, w.vec16);
        }
      }
    }
  }
}

template <typename T, int OP, int KIND>
__device__ __forceinline__ void step_data_full(const WarpRank& w, uint32_t inSlot,
                                               uint32_t ownSlot, uint32_t outSlot, uint64_t off,
                                               uint32_t len) {
  step_data_body<T, OP, KIND, true>(w, inSlot, ownSlot, outSlot, off, len);
}
// Partial or unaligned steps (rare): out of line, to keep the hot path small.
template <typename T, int OP, int KIND>
__device__ __noinline__ void step_data_partial(const WarpRank& w, uint32_t inSlot,
                                               uint32_t ownSlot, uint32_t outSlot, uint64_t off,
                                               uint32_t len) {
  step_data_body<T, OP, KIND, false>(w, inSlot, ownSlot, outSlot, off, len);
}

// Prefetch the rank's next own-data step into own slot `slot` (lane 0).
__device__ __forceinline__ void prefetch_own(WarpRank& w, StepCursor& pre, uint32_t slot) {
  int kind;
  uint64_t off;
  uint32_t len;
  if (!pre.next(kind, off, len)) return;
  const uint32_t bytes = w.vec16 ? (len & ~15u) : 0u;
  const uint32_t bar = w.me.inFull + 8 * slot;
  mbar_arrive_expect_tx(bar, bytes);
  if (bytes) tma_load_1d(w.me.own + slot * w.SLOT, w.own + off, bytes, bar);
  ++w.issued;
}

// All the steps of one stage of one part: wait, move the data, signal.
// Returns false if a wait gave up.
template <typename T, int OP, int KIND>
__device__ __forceinline__ bool run_stage(WarpRank& w, StepCursor& pre, uint64_t off0,
                                       uint64_t plen) {
  constexpr bool rcv = KIND != VR_SEND, snd = KIND != VR_RECV;
  constexpr bool hasOwn = KIND <= VR_RRCS;
  const vrRingArgs& a = *w.a;
  for (uint64_t s = 0; s < plen; s += w.SLOT) {
    const uint32_t len = (uint32_t)min_u64(w.SLOT, plen - s);
    const uint32_t sIn = w.sIn, sOut = w.sOut, iIn = w.iOwn;
    // Lane 0 waits for the incoming slot, the outgoing slot and the own
    // data; the warp barrier then orders every lane's reads after its
    // acquires.
    bool ok = true;
    if (w.lane == 0) {
      if (rcv) ok = lane_wait_cta(w.me.full + 8 * sIn, w.phIn, a);
      if (ok && snd && w.outWrapped) ok = lane_wait_cta(w.nx.empty + 8 * sOut, w.phOut ^ 1u, a);
      if (ok && hasOwn) ok = lane_wait_cta(w.me.inFull + 8 * iIn, w.phOwn, a);
    }
    if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) return false;
    __syncwarp();
    const uint32_t inSlot = w.me.fifo + sIn * w.SLOT, ownSlot = w.me.own + iIn * w.SLOT;
    const uint32_t outSlot = w.nx.fifo + sOut * w.SLOT;
    if (len == w.SLOT && w.vec16)
      step_data_full<T, OP, KIND>(w, inSlot, ownSlot, outSlot, off0 + s, len);
    else
      step_data_partial<T, OP, KIND>(w, inSlot, ownSlot, outSlot, off0 + s, len);
    __syncwarp();
    if (w.lane == 0) {
      if (snd && !w.silent) mbar_arrive_cta(w.nx.full + 8 * sOut);
      if (rcv && !w.silent) mbar_arrive_cta(w.me.empty + 8 * sIn);
      if (hasOwn) {
        // This warp has read own slot iIn: refill it (the reads above are
        // ordered before the bulk copy's writes).
        fence_proxy_async_shared();
        prefetch_own(w, pre, iIn);
      }
    }
    if (snd && ++w.sOut == w.D) {
      w.sOut = 0;
      w.phOut ^= 1u;
      w.outWrapped = true;
    }
    if (rcv && ++w.sIn == w.D) {
      w.sIn = 0;
      w.phIn ^= 1u;
    }
    if (hasOwn) {
      ++w.ownUsed;
      if (++w.iOwn == w.DI) {
        w.iOwn = 0;
        w.phOwn ^= 1u;
      }
    }
  }
  return true;
}

template <typename T, int OP>
__global__ void __launch_bounds__(VR_WARP_MAX_THREADS, 1)
vr_ring_warp(const __grid_constant__ vrRingArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr uint64_t E = sizeof(T);
  const int N = a.nRanks;
  const int R = a.ringsPerCta;
  const int nWarps = R * N;
  const int warp = threadIdx.x >> 5;
  const int rho = warp / N, r = warp % N;
  const uint32_t base = smem_addr(smem);

  WarpRank w;
  w.a = &a;
  w.D = a.depth;
  w.DI = a.inDepth;
  w.SLOT = a.slotBytes;
  w.lane = threadIdx.x & 31;
  w.me = warp_smem(base, warp, nWarps, w.D, w.DI, w.SLOT);
  w.nx = warp_smem(base, rho * N + (r + 1) % N, nWarps, w.D, w.DI, w.SLOT);
  w.own = static_cast<const char*>(a.send[r]);
  w.out = static_cast<char*>(a.recv[r]);
  w.vec16 = (a.alignMask & 15) == 0;
  w.silent = (r == a.silentRank);
  w.sIn = w.phIn = w.sOut = w.phOut = w.iOwn = w.phOwn = w.ownUsed = w.issued = 0;
  w.outWrapped = false;

  __shared__ StepPlan plan;
  if (threadIdx.x == 0) {
    plan.init(a, E, gridDim.x * R, (uint64_t)w.SLOT * (w.D / 2), w.SLOT);
    for (int i = 0; i < nWarps; ++i) {
      const WarpSmem m = warp_smem(base, i, nWarps, w.D, w.DI, w.SLOT);
      for (uint32_t j = 0; j < w.D; ++j) {
        mbar_init(m.full + 8 * j, 1);   // the sending warp's lane 0
        mbar_init(m.empty + 8 * j, 1);  // the receiving warp's lane 0
      }
      for (uint32_t j = 0; j < w.DI; ++j) mbar_init(m.inFull + 8 * j, 1);  // arm + tx
    }
  }
  __syncthreads();

  const int ring = blockIdx.x * R + rho;
  const int nRings = gridDim.x * R;
  // `cur` only locates parts; `pre` (in shared memory: only lane 0 uses it)
  // walks the own-data steps for prefetching.
  __shared__ StepCursor preCursors[VR_WARP_MAX_RANKS];
  StepCursor& pre = preCursors[warp];
  StepCursor cur;
  cur.init(&plan, r, ring, 2 * N - 2);
  if (w.lane == 0) pre.init(&plan, r, ring, N - 1);
  if (w.lane == 0)
    for (uint32_t i = 0; i < w.DI; ++i) prefetch_own(w, pre, i);

  bool ok = true;
  for (uint64_t unit = (uint64_t)ring; ok && unit < plan.nUnits; unit += (uint64_t)nRings) {
    cur.unit = unit;
    cur.enter_part();
    for (int k = 0; ok && k <= 2 * N - 2; ++k) {
      if (k) {
        cur.c = cur.c == 0 ? N - 1 : cur.c - 1;
        cur.enter_stage();
      }
      if (!cur.plen) continue;
      const uint64_t off0 = cur.partBase + cur.lo * E;
      if (k == 0) ok = run_stage<T, OP, VR_SEND>(w, pre, off0, cur.plen);
      else if (k < N - 1) ok = run_stage<T, OP, VR_RRS>(w, pre, off0, cur.plen);
      else if (k == N - 1) ok = run_stage<T, OP, VR_RRCS>(w, pre, off0, cur.plen);
      else if (k < 2 * N - 2) ok = run_stage<T, OP, VR_RCS>(w, pre, off0, cur.plen);
      else ok = run_stage<T, OP, VR_RECV>(w, pre, off0, cur.plen);
    }
  }
  // Bulk copies this warp issued must land before it exits.
  if (w.lane == 0) {
    for (uint32_t j = w.ownUsed; j < w.issued; ++j) {
      const uint32_t bar = w.me.inFull + 8 * (j % w.DI), par = (j / w.DI) & 1u;
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait_cta(bar, par) && globaltimer() - t0 < a.timeoutNs) {
      }
    }
  }
}

}  // namespace vr

#define VR_INSTANTIATE_WARP(GETTER, T)                                            \
  const void* GETTER(int op) {                                                    \
    static const void* table[4] = {(const void*)vr::vr_ring_warp<T, 0>,            \
                                   (const void*)vr::vr_ring_warp<T, 1>,            \
                                   (const void*)vr::vr_ring_warp<T, 2>,            \
                                   (const void*)vr::vr_ring_warp<T, 3>};           \
    return (op < 0 || op > 3) ? nullptr : table[op];                              \
  }
