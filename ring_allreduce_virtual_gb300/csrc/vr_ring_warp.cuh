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
// and the FIFO traffic (about twice the input) never reaches L2 or HBM.
//
// Lane 0 of each rank warp brings the rank's own input in ahead of use: a
// bulk TMA copy per step into one of `inDepth` own slots, issued as soon as
// the warp has read the slot's previous step. So HBM sees each input byte read
// once and each output byte written once.
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
#include "vr_smem.cuh"

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
// Shared-memory accesses of LL / LL128 lines. Each 8-byte element of a vector
// access is single-copy atomic, so a flag and the payload beside it in one
// 8-byte word are seen together.
__device__ __forceinline__ void ld_volatile_shared_v2u64(uint32_t addr, uint64_t& x, uint64_t& y) {
  asm volatile("ld.volatile.shared.v2.u64 {%0,%1}, [%2];" : "=l"(x), "=l"(y) : "r"(addr) : "memory");
}
__device__ __forceinline__ void st_volatile_shared_v2u64(uint32_t addr, uint64_t x, uint64_t y) {
  asm volatile("st.volatile.shared.v2.u64 [%0], {%1,%2};" ::"r"(addr), "l"(x), "l"(y) : "memory");
}
__device__ __forceinline__ void ld_shared_v2u64(uint32_t addr, uint64_t& x, uint64_t& y) {
  asm volatile("ld.shared.v2.u64 {%0,%1}, [%2];" : "=l"(x), "=l"(y) : "r"(addr) : "memory");
}
__device__ __forceinline__ void st_shared_v2u64(uint32_t addr, uint64_t x, uint64_t y) {
  asm volatile("st.shared.v2.u64 [%0], {%1,%2};" ::"r"(addr), "l"(x), "l"(y) : "memory");
}
__device__ __forceinline__ uint64_t ld_shared_u64(uint32_t addr) {
  uint64_t v;
  asm volatile("ld.shared.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_shared_u64(uint32_t addr, uint64_t v) {
  asm volatile("st.shared.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}
// Barrier initialisation visible to the other warps and to the bulk-copy
// unit (completed by the CTA barrier that follows).
__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Bounded spin by one lane until `ready()` holds. False if it gave up.
template <typename F>
__device__ __forceinline__ bool lane_poll(F&& ready, const vrRingArgs& a) {
  // Short waits end before the clock is read.
  for (int it = 0; it < 32; ++it)
    if (ready()) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (ready()) return true;
    if ((it & 63) == 0) {
      if (ld_volatile_int(a.status) != VR_STATUS_OK) return false;
      if (globaltimer() - t0 > a.timeoutNs) {
        raise_timeout(a);
        return false;
      }
    }
  }
}

// Bounded wait by one lane on a CTA-local barrier phase.
__device__ __forceinline__ bool lane_wait_cta(uint32_t addr, uint32_t parity, const vrRingArgs& a) {
  for (int it = 0; it < 4; ++it)
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

// A ring may span the CTAs of a thread-block cluster (CL): then the warp
// whose next rank is in another CTA (RN) writes that rank's FIFO slots with
// st.async stores counted on its full barrier (every protocol), the warp
// whose previous rank is in another CTA waits on that barrier and signals the
// sender's "empty" barrier with a cluster-scope arrival, and every wait on a
// warp's own barriers and flags acquires at cluster scope. Edges inside a CTA
// stay CTA-local.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

template <bool CL>
__device__ __forceinline__ void st_next_v4(uint32_t addr, uint4 v) {
  if (CL)
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
  else
    st_shared_v4(addr, v);
}
template <bool CL>
__device__ __forceinline__ void st_next_v2u64(uint32_t addr, uint64_t x, uint64_t y) {
  if (CL)
    asm volatile("st.shared::cluster.v2.u64 [%0], {%1,%2};" ::"r"(addr), "l"(x), "l"(y) : "memory");
  else
    st_shared_v2u64(addr, x, y);
}
template <bool CL>
__device__ __forceinline__ void st_next_u64(uint32_t addr, uint64_t x) {
  if (CL)
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(x) : "memory");
  else
    st_shared_u64(addr, x);
}
// An LL line: two {payload32, flag32} words, each single-copy atomic.
template <bool CL>
__device__ __forceinline__ void st_next_ll(uint32_t addr, uint64_t x, uint64_t y) {
  if (CL)
    asm volatile("st.relaxed.cluster.shared::cluster.v2.u64 [%0], {%1,%2};" ::"r"(addr), "l"(x),
                 "l"(y)
                 : "memory");
  else
    st_volatile_shared_v2u64(addr, x, y);
}
// The reader's poll of an LL line of its own FIFO (written by a neighbour,
// with CL possibly in another CTA).
template <bool CL>
__device__ __forceinline__ void ld_in_ll(uint32_t addr, uint64_t& x, uint64_t& y) {
  if (CL)
    asm volatile("ld.relaxed.cluster.shared::cta.v2.u64 {%0,%1}, [%2];"
                 : "=l"(x), "=l"(y) : "r"(addr) : "memory");
  else
    ld_volatile_shared_v2u64(addr, x, y);
}
// LL128 flags of a batch of lines. The writer's flag lane stores the first
// line's flag with release semantics after the batch's payload (its group's
// lanes ordered before it by a warp barrier) and the other lines' flags after
// it; the reader's flag lane polls the first line's flag with acquire
// semantics, which makes the whole batch's payload visible. At cluster scope
// when the neighbour may be in another CTA.
template <bool CL>
__device__ __forceinline__ uint32_t ld_flag_acquire(uint32_t addr) {
  uint32_t v;
  if (CL)
    asm volatile("ld.acquire.cluster.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  else
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
template <bool CL>
__device__ __forceinline__ void st_next_flag_release(uint32_t addr, uint32_t v) {
  if (CL)
    asm volatile("st.release.cluster.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
  else
    asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
template <bool CL>
__device__ __forceinline__ void st_next_flag_relaxed(uint32_t addr, uint32_t v) {
  if (CL)
    asm volatile("st.relaxed.cluster.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
  else
    asm volatile("st.relaxed.cta.shared::cta.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Signal that a slot has been drained (count 1, no ordering): the arriving
// warp's reads of the slot have all returned -- their values were consumed
// before the warp barrier that precedes the arrival -- so the writer's next
// stores into the slot cannot reach them, and no release (at cluster scope a
// wait for every earlier remote store) is needed.
template <bool CL>
__device__ __forceinline__ void arrive_drained(uint32_t addr) {
  if (CL)
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr)
                 : "memory");
  else
    asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(addr) : "memory");
}

// Signal a neighbour's barrier (count 1, release).
template <bool CL>
__device__ __forceinline__ void arrive_peer(uint32_t addr) {
  if (CL)
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr)
                 : "memory");
  else
    mbar_arrive_cta(addr);
}
// Bounded wait by one lane on a barrier of this warp that a neighbour
// signals (acquire at the neighbour's scope).
template <bool CL>
__device__ __forceinline__ bool lane_wait_peer(uint32_t addr, uint32_t parity, const vrRingArgs& a) {
  if (!CL) return lane_wait_cta(addr, parity, a);
  for (int it = 0; it < 4; ++it)
    if (mbar_try_wait(addr, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(addr, parity)) return true;
    if ((it & 15) == 0) {
      if (ld_volatile_int(a.status) != VR_STATUS_OK) return false;
      if (globaltimer() - t0 > a.timeoutNs) {
        raise_timeout(a);
        return false;
      }
    }
  }
}

// Shared memory of one rank warp: D FIFO slots (its incoming edge), DI
// own-data slots (a step's payload each), then (after all warps' data) its
// barriers: full[D] (its incoming slot s was filled: the previous rank
// signals, this warp waits), empty[D] (its outgoing slot s in the next rank's
// FIFO was drained: the next rank signals, this warp waits), inFull[DI] (the
// bulk copy of own data landed). Every wait is on a barrier of the waiting
// warp's own CTA.
struct WarpSmem {
  uint32_t fifo, own, full, empty, inFull;
};

__device__ __forceinline__ WarpSmem warp_smem(uint32_t base, int w, int nWarps, uint32_t D,
                                              uint32_t DI, uint32_t SLOT, uint32_t OWNSLOT) {
  WarpSmem m;
  const uint32_t per = D * SLOT + DI * OWNSLOT;
  m.fifo = base + (uint32_t)w * per;
  m.own = m.fifo + D * SLOT;
  const uint32_t bars = base + (uint32_t)nWarps * per + (uint32_t)w * 8 * (2 * D + DI);
  m.full = bars;
  m.empty = bars + 8 * D;
  m.inFull = bars + 16 * D;
  return m;
}

// Per-warp state of one rank of one ring. Slot indices and mbarrier phase
// bits advance incrementally (no division per step).
struct WarpRank {
  const vrRingArgs* a;
  WarpSmem me;
  uint32_t nxFifo, nxFull;  // the next rank's FIFO slots and full barriers
  uint32_t pvEmpty;         // the previous rank's empty barriers
  const char* own;
  char* out;
  uint32_t sIn, phIn;      // next incoming FIFO slot and its phase
  uint32_t sOut, phOut;    // next outgoing FIFO slot and its phase
  uint32_t iOwn, phOwn;    // next own-data slot and its phase
  uint32_t sendCnt, recvCnt;  // steps sent / received on this rank's edges (LL flags)
  uint32_t D, DI, SLOT, OWNSLOT;
  int lane;
  uint32_t issued, ownUsed;  // own-data copies issued / consumed
  uint32_t iPre, owed;     // lane 0: next own slot to fill; refills owed to the next part
  StepWalk pre;            // lane 0: the walk of the own-data steps
  bool outWrapped;         // every outgoing slot has been used once
  bool vec16, silent;
  bool remoteNext, remotePrev;  // the next / previous rank is in another CTA
  int scale;               // sum kernels: VR_SCALE_*
  uint4 sPack;             // VR_SCALE_PREMUL: the scalar over 16 bytes
};

// The data of one Simple step of stage kind KIND: `len` bytes as 16-byte
// packs, one per lane per iteration (the CTA's other warps hide the latency).
// Own data comes from the own slot, except bytes the bulk copy left out (an
// unaligned buffer, or a ragged tail under 16 bytes), which come from global
// memory; output bytes likewise go out as 16-byte stores where aligned.
// FULL: a whole payload of aligned packs (the common case), no checks.
// RN: the next rank is in another CTA; its slot is written with st.async,
// which counts the bytes on its full barrier `outBar` (simple_tx_bytes).
template <typename T, int OP, int KIND, bool FULL, bool CL, bool RN>
__device__ __forceinline__ void step_data(const WarpRank& w, uint32_t inSlot, uint32_t ownSlot,
                                          uint32_t outSlot, uint64_t ownOff, uint64_t outOff,
                                          uint32_t len, uint32_t outBar) {
  constexpr bool rcv = vrKindRecv(KIND), snd = vrKindSend(KIND);
  constexpr bool hasOwn = vrKindOwn(KIND), hasOut = vrKindOut(KIND);
  constexpr bool red = vrKindReduce(KIND);
  const uint32_t nPacks = (len + 15) >> 4;
  const uint32_t vecBytes = w.vec16 ? (len & ~15u) : 0u;
  const char* ownG = w.own + ownOff;
  char* outG = w.out + outOff;
  for (uint32_t p = w.lane; p < nPacks; p += 32) {
    const uint32_t b = p * 16;
    uint4 v, x;
    if (hasOwn) {
      if (FULL || b < vecBytes) v = ld_shared_v4(ownSlot + b);
      else v = load_pack<T>(ownG + b, len - b, false);
      if (OP == 0 && KIND != VR_SC && w.scale == VR_SCALE_PREMUL) v = hop16<T, 1>(v, w.sPack);
    }
    if (rcv) x = ld_shared_v4(inSlot + b);
    uint4 res;
    if (KIND == VR_SEND || KIND == VR_SC) res = v;
    else if (red) res = hop16<T, OP>(x, v);
    else res = x;
    if (OP == 0 && (KIND == VR_RRCS || KIND == VR_RRC) && w.scale == VR_SCALE_POSTDIV)
      res = div_pack<T>(res, w.a->nRanks);
    if (snd) {
      if (RN) {
        if (!w.silent) st_async_v4(outSlot + b, res, outBar);
      } else {
        st_shared_v4(outSlot + b, res);
      }
    }
    if (hasOut) {
      if (FULL || b < vecBytes) st_cs_v4(outG + b, res);
      else store_pack<T>(outG + b, res, len - b, false);
    }
  }
}

// Bytes a Simple step of `len` bytes writes into the next rank's slot (whole
// 16-byte packs): what the receiver of an edge between CTAs expects on its
// full barrier.
__device__ __forceinline__ uint32_t simple_tx_bytes(uint32_t len) { return ((len + 15) >> 4) * 16; }

// Bytes an LL step of `len` payload bytes writes into the next rank's slot
// (two 16-byte lines per 16-byte pack).
__device__ __forceinline__ uint32_t ll_tx_bytes(uint32_t len) { return ((len + 15) >> 4) * 32; }

// Bytes an LL128 step of `len` payload bytes writes into the next rank's slot
// (whole 128-byte lines of 15 payload words and a flag word).
__device__ __forceinline__ uint32_t ll128_tx_bytes(uint32_t len) {
  return ((((len + 7) >> 3) + 14) / 15) * 128;
}

// LL step: every 16-byte pack of payload travels as two 16-byte lines of two
// 8-byte words {payload32, flag32}; the reader polls its own lines. A slot of
// S bytes holds the packs' first lines in its first half and their second
// lines in its second half (pack p: bytes 16 p and S/2 + 16 p), so that the
// lanes of a warp touch consecutive 16-byte lines, free of bank conflicts.
// Into another CTA (RN) the lines go as st.async stores counted on the
// receiver's full barrier (outBar; ll_tx_bytes), which that receiver has
// waited on for the whole step (`waited`) before reading without polling.
// Returns false if a poll gave up (on every lane).
template <typename T, int OP, int KIND, bool FULL, bool CL, bool RN>
__device__ __forceinline__ bool ll_step(const WarpRank& w, uint32_t inSlot, uint32_t ownSlot,
                                        uint32_t outSlot, uint64_t ownOff, uint64_t outOff,
                                        uint32_t len, uint32_t flagIn, uint32_t flagOut,
                                        uint32_t outBar, bool waited) {
  constexpr bool rcv = vrKindRecv(KIND), snd = vrKindSend(KIND);
  constexpr bool hasOwn = vrKindOwn(KIND), hasOut = vrKindOut(KIND);
  constexpr bool red = vrKindReduce(KIND);
  const vrRingArgs& a = *w.a;
  const uint32_t nPacks = (len + 15) >> 4;
  const uint32_t vecBytes = w.vec16 ? (len & ~15u) : 0u;
  const char* ownG = w.own + ownOff;
  char* outG = w.out + outOff;
  bool dead = false;
  for (uint32_t p = w.lane; p < nPacks; p += 32) {
    const uint32_t b = p * 16;
    uint4 v = make_uint4(0, 0, 0, 0), x = v;
    // Own pack: before the poll in one CTA, after it on a cluster (each
    // measured faster there).
    auto own_pack = [&]() {
      if (FULL || b < vecBytes) v = ld_shared_v4(ownSlot + b);
      else v = load_pack<T>(ownG + b, len - b, false);
      if (OP == 0 && KIND != VR_SC && w.scale == VR_SCALE_PREMUL) v = hop16<T, 1>(v, w.sPack);
    };
    if (hasOwn && !CL) own_pack();
    if (rcv) {
      const uint32_t q = inSlot + p * 16, q2 = q + (w.SLOT >> 1);
      uint64_t a0, a1, b0, b1;
      auto ready = [&]() {
        ld_in_ll<CL>(q, a0, a1);
        ld_in_ll<CL>(q2, b0, b1);
        return (uint32_t)(a0 >> 32) == flagIn && (uint32_t)(a1 >> 32) == flagIn &&
               (uint32_t)(b0 >> 32) == flagIn && (uint32_t)(b1 >> 32) == flagIn;
      };
      if (waited) {
        ld_in_ll<CL>(q, a0, a1);
        ld_in_ll<CL>(q2, b0, b1);
      } else if (!lane_poll(ready, a)) {
        dead = true;
        break;
      }
      x = make_uint4((uint32_t)a0, (uint32_t)a1, (uint32_t)b0, (uint32_t)b1);
    }
    if (hasOwn && CL) own_pack();
    uint4 res;
    if (KIND == VR_SEND || KIND == VR_SC) res = v;
    else if (red) res = hop16<T, OP>(x, v);
    else res = x;
    if (OP == 0 && (KIND == VR_RRCS || KIND == VR_RRC) && w.scale == VR_SCALE_POSTDIV)
      res = div_pack<T>(res, w.a->nRanks);
    if (snd && !w.silent) {
      if (RN) {
        st_async_v4(outSlot + p * 16, make_uint4(res.x, flagOut, res.y, flagOut), outBar);
        st_async_v4(outSlot + (w.SLOT >> 1) + p * 16, make_uint4(res.z, flagOut, res.w, flagOut),
                    outBar);
      } else {
        const uint64_t f = (uint64_t)flagOut << 32;
        st_next_ll<RN>(outSlot + p * 16, f | res.x, f | res.y);
        st_next_ll<RN>(outSlot + (w.SLOT >> 1) + p * 16, f | res.z, f | res.w);
      }
    }
    if (hasOut) {
      if (FULL || b < vecBytes) st_cs_v4(outG + b, res);
      else store_pack<T>(outG + b, res, len - b, false);
    }
  }
  return !__any_sync(0xffffffffu, dead);
}

// LL128 step: 128-byte lines, 8-byte words 0..14 payload and word 15 the
// flag. Lane j of an 8-lane group owns words 2j, 2j+1 of its line (lane 7:
// word 14 and the flag); a warp covers 4 lines per row and handles RB rows
// per handshake. The writer's group stores the batch's payload (every lane a
// 16-byte store, the flag lane zeroing the flag word), then after a warp
// barrier its flag lane stores every line's flag, the first with release
// semantics; the reader's flag lane acquires that first flag before the group
// reads the batch, so lines are consumed as soon as their batch is written.
// Into another CTA (RN) the lines go as 16-byte st.async stores, flag words
// included, counted on the receiver's full barrier (outBar; ll128_tx_bytes):
// a cluster-scope release per batch would also wait for the warp's earlier
// output stores. Its receiver has then waited on that barrier for the whole
// step (`waited`) and reads without polling.
template <typename T, int OP, int KIND, bool FULL, bool CL, bool RN>
__device__ __forceinline__ bool ll128_step(const WarpRank& w, uint32_t inSlot, uint32_t ownSlot,
                                           uint32_t outSlot, uint64_t ownOff, uint64_t outOff,
                                           uint32_t len, uint32_t flagIn, uint32_t flagOut,
                                           uint32_t outBar, bool waited) {
  constexpr bool rcv = vrKindRecv(KIND), snd = vrKindSend(KIND);
  constexpr bool hasOwn = vrKindOwn(KIND), hasOut = vrKindOut(KIND);
  constexpr bool red = vrKindReduce(KIND);
  // Rows of 4 lines handled per flag handshake: the flags of the batch are
  // polled together and published together, one fence each way. Fewer
  // rows where registers run out: max/min (their element selection), 8-bit
  // types (their byte-wise arithmetic), and on cluster rings all but the
  // 16- and 32-bit sums and products (their extra addressing).
  constexpr uint32_t RB = CL ? ((OP <= 1 && (sizeof(T) == 2 || sizeof(T) == 4)) ? 4 : 1)
                              : (OP <= 1 && sizeof(T) >= 2) ? 4 : 2;
  const vrRingArgs& a = *w.a;
  const uint32_t nWords = (len + 7) >> 3;
  const uint32_t nLines = (nWords + 14) / 15;
  const uint32_t nRows = (nLines + 3) >> 2;
  const uint32_t vecBytes = w.vec16 ? (len & ~15u) : 0u;  // bytes the bulk copy brought
  const uint32_t grp = w.lane >> 3, j = w.lane & 7;
  const bool flagLane = j == 7;
  const char* ownG = w.own + ownOff;
  char* outG = w.out + outOff;
  bool dead = false;
  // A whole payload (FULL) is whole lines, so every word of a line that
  // exists does too.
  auto ownWord = [&](uint32_t wi) -> uint64_t {
    if (!FULL && wi >= nWords) return 0;
    if (FULL || wi * 8 + 8 <= vecBytes) return ld_shared_u64(ownSlot + wi * 8);
    return load_word<T>(ownG + (uint64_t)wi * 8, len - wi * 8, false);
  };
  auto outWord = [&](uint32_t wi, uint64_t v) {
    if (!FULL && wi >= nWords) return;
    if (FULL || wi * 8 + 8 <= vecBytes) st_cs_u64(outG + (uint64_t)wi * 8, v);
    else store_word<T>(outG + (uint64_t)wi * 8, v, len - wi * 8, false);
  };
  for (uint32_t row0 = 0; row0 < nRows; row0 += RB) {
    uint64_t r0[RB], r1[RB];
    uint64_t x0[RB], x1[RB];
#pragma unroll
    for (uint32_t k = 0; k < RB; ++k) x0[k] = x1[k] = 0;
    if (rcv) {
      const uint32_t first = row0 * 4 + grp;  // the group's first line of the batch
      if (!waited && flagLane && !dead && first < nLines) {
        const uint32_t fq = inSlot + first * 128 + 120;
        dead = !lane_poll([&]() { return ld_flag_acquire<CL>(fq) == flagIn; }, a);
      }
      __syncwarp();
      // Every lane reads 16 bytes of its line; the flag lane's second word is
      // the flag, not payload.
#pragma unroll
      for (uint32_t k = 0; k < RB; ++k) {
        const uint32_t line = (row0 + k) * 4 + grp;
        if (line < nLines) ld_shared_v2u64(inSlot + line * 128 + 16 * j, x0[k], x1[k]);
      }
    }
#pragma unroll
    for (uint32_t k = 0; k < RB; ++k) {
      const uint32_t line = (row0 + k) * 4 + grp;
      const uint32_t w0 = line * 15 + 2 * j;
      uint64_t v0 = 0, v1 = 0;
      if (hasOwn && line < nLines) {
        v0 = ownWord(w0);
        if (!flagLane) v1 = ownWord(w0 + 1);
        if (OP == 0 && KIND != VR_SC && w.scale == VR_SCALE_PREMUL) {
          const uint64_t sw = (uint64_t)w.sPack.x | ((uint64_t)w.sPack.y << 32);
          v0 = hop8<T, 1>(v0, sw);
          v1 = hop8<T, 1>(v1, sw);
        }
      }
      if (KIND == VR_SEND || KIND == VR_SC) { r0[k] = v0; r1[k] = v1; }
      else if (red) { r0[k] = hop8<T, OP>(x0[k], v0); r1[k] = hop8<T, OP>(x1[k], v1); }
      else { r0[k] = x0[k]; r1[k] = x1[k]; }
      if (OP == 0 && (KIND == VR_RRCS || KIND == VR_RRC) && w.scale == VR_SCALE_POSTDIV) {
        r0[k] = div_word<T>(r0[k], w.a->nRanks);
        r1[k] = div_word<T>(r1[k], w.a->nRanks);
      }
    }
    if (snd && !w.silent) {
      // Payload first, the flag lane's flag word zeroed (no count is 0, so a
      // reader never takes it for its flag) ...
#pragma unroll
      for (uint32_t k = 0; k < RB; ++k) {
        const uint32_t line = (row0 + k) * 4 + grp;
        if (line < nLines) {
          if (RN) {
            const uint64_t y = flagLane ? (uint64_t)flagOut : r1[k];
            st_async_v4(outSlot + line * 128 + 16 * j,
                        make_uint4((uint32_t)r0[k], (uint32_t)(r0[k] >> 32), (uint32_t)y,
                                   (uint32_t)(y >> 32)),
                        outBar);
          } else {
            st_next_v2u64<RN>(outSlot + line * 128 + 16 * j, r0[k], flagLane ? 0ull : r1[k]);
          }
        }
      }
      __syncwarp();
      // ... then, after the group's payload, the batch's flags: the first
      // line's with release semantics, which the reader acquires.
      if (!RN && flagLane) {
#pragma unroll
        for (uint32_t k = 0; k < RB; ++k) {
          const uint32_t line = (row0 + k) * 4 + grp;
          if (line < nLines) {
            if (k == 0) st_next_flag_release<RN>(outSlot + line * 128 + 120, flagOut);
            else st_next_flag_relaxed<RN>(outSlot + line * 128 + 120, flagOut);
          }
        }
      }
    }
    if (hasOut) {
#pragma unroll
      for (uint32_t k = 0; k < RB; ++k) {
        const uint32_t line = (row0 + k) * 4 + grp;
        const uint32_t w0 = line * 15 + 2 * j;
        if (line < nLines) {
          outWord(w0, r0[k]);
          if (!flagLane) outWord(w0 + 1, r1[k]);
        }
      }
    }
  }
  return !__any_sync(0xffffffffu, dead);
}

// Lane 0: bulk-copy own-data step (off, len) into the next own slot (slots
// fill in turn, as they are consumed).
__device__ __forceinline__ void issue_own(WarpRank& w, uint64_t off, uint32_t len) {
  const uint32_t bytes = w.vec16 ? (len & ~15u) : 0u;
  const uint32_t bar = w.me.inFull + 8 * w.iPre;
  mbar_arrive_expect_tx(bar, bytes);
  if (bytes) tma_load_1d(w.me.own + w.iPre * w.OWNSLOT, w.own + off, bytes, bar);
  if (++w.iPre == w.DI) w.iPre = 0;
  ++w.issued;
}

// Lane 0, after a step consumed its own slot: refill it with the part's next
// own-data step; when the part has none left, the refill is owed to the
// ring's next part (refill_owed), so that no stage carries the code that
// enters a part.
__device__ __forceinline__ void prefetch_own(WarpRank& w) {
  uint64_t off;
  uint32_t len;
  if (w.pre.next_in_part(w.a->plan, off, len)) issue_own(w, off, len);
  else ++w.owed;
}

// Lane 0, after a part's last own-data stage (and at the start): the owed
// refills, from the ring's next parts.
__device__ __forceinline__ void refill_owed(WarpRank& w) {
  const vrStepPlan& P = w.a->plan;
  while (w.owed) {
    uint64_t off;
    uint32_t len;
    if (w.pre.next_in_part(P, off, len)) {
      issue_own(w, off, len);
      --w.owed;
    } else if (!w.pre.next_part(P)) {
      w.owed = 0;
    }
  }
}

// All the steps of one stage of one part: wait, move the data, signal.
// Returns false if a wait gave up.
template <typename T, int OP, int KIND, int PROTO, bool CL, bool RN>
__device__ __forceinline__ bool run_stage(WarpRank& w, uint64_t own0, uint64_t out0,
                                          uint32_t plen) {
  constexpr bool rcv = vrKindRecv(KIND), snd = vrKindSend(KIND);
  constexpr bool hasOwn = vrKindOwn(KIND);
  const vrRingArgs& a = *w.a;
  const uint32_t payload = (uint32_t)vrPayloadPerStep(PROTO, w.SLOT);
  for (uint32_t s = 0; s < plen; s += payload) {
    const uint32_t len = min(payload, plen - s);
    const uint32_t sIn = w.sIn, sOut = w.sOut, iIn = w.iOwn;
    // Wait for the incoming slot (Simple; LL and LL128 readers poll their
    // lines instead), the outgoing slot and the own data. On a cluster lane 0
    // waits (cluster-scope acquires) and the warp barrier then orders every
    // lane's reads after its acquires; in one CTA every lane waits itself
    // (measured faster: no broadcast).
    bool ok = true;
    if (!CL) {
      if (rcv && PROTO == vrProtoSimple) ok = lane_wait_cta(w.me.full + 8 * sIn, w.phIn, a);
      if (ok && snd && w.outWrapped) ok = lane_wait_cta(w.me.empty + 8 * sOut, w.phOut ^ 1u, a);
      if (ok && hasOwn) ok = lane_wait_cta(w.me.inFull + 8 * iIn, w.phOwn, a);
      if (!__all_sync(0xffffffffu, ok)) return false;
    } else {
      if (w.lane == 0) {
        if (rcv && PROTO == vrProtoSimple) {
          // From another CTA the step arrives by st.async: arm the barrier
          // with its bytes (this warp's arrival completes the phase with them).
          if (CL && w.remotePrev) mbar_arrive_expect_tx(w.me.full + 8 * sIn, simple_tx_bytes(len));
          ok = lane_wait_peer<CL>(w.me.full + 8 * sIn, w.phIn, a);
        }
        // LL and LL128 from another CTA likewise (st.async lines, ll_step,
        // ll128_step).
        if (rcv && PROTO != vrProtoSimple && w.remotePrev) {
          mbar_arrive_expect_tx(w.me.full + 8 * sIn,
                                PROTO == vrProtoLL ? ll_tx_bytes(len) : ll128_tx_bytes(len));
          ok = lane_wait_peer<CL>(w.me.full + 8 * sIn, w.phIn, a);
        }
        if (ok && snd && w.outWrapped)
          ok = lane_wait_peer<CL>(w.me.empty + 8 * sOut, w.phOut ^ 1u, a);
        if (ok && hasOwn) ok = lane_wait_cta(w.me.inFull + 8 * iIn, w.phOwn, a);
      }
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) return false;
      __syncwarp();
    }
    const uint32_t inSlot = w.me.fifo + sIn * w.SLOT, ownSlot = w.me.own + iIn * w.OWNSLOT;
    const uint32_t outSlot = w.nxFifo + sOut * w.SLOT;
    // A whole payload of aligned bytes takes the unchecked copy of the body.
    const bool full = len == payload && w.vec16;
    if (PROTO == vrProtoSimple) {
      if (full)
        step_data<T, OP, KIND, true, CL, RN>(w, inSlot, ownSlot, outSlot, own0 + s, out0 + s, len,
                                             w.nxFull + 8 * sOut);
      else
        step_data<T, OP, KIND, false, CL, RN>(w, inSlot, ownSlot, outSlot, own0 + s, out0 + s, len,
                                              w.nxFull + 8 * sOut);
    } else {
      const uint32_t flagIn = w.recvCnt + 1, flagOut = w.sendCnt + 1;
      bool good;
      if (PROTO == vrProtoLL)
        good = full ? ll_step<T, OP, KIND, true, CL, RN>(w, inSlot, ownSlot, outSlot, own0 + s, out0 + s,
                                                 len, flagIn, flagOut, w.nxFull + 8 * sOut,
                                                 CL && w.remotePrev)
                    : ll_step<T, OP, KIND, false, CL, RN>(w, inSlot, ownSlot, outSlot, own0 + s,
                                                  out0 + s, len, flagIn, flagOut,
                                                  w.nxFull + 8 * sOut, CL && w.remotePrev);
      else
        good = full ? ll128_step<T, OP, KIND, true, CL, RN>(w, inSlot, ownSlot, outSlot, own0 + s,
                                                    out0 + s, len, flagIn, flagOut,
                                                    w.nxFull + 8 * sOut, CL && w.remotePrev)
                    : ll128_step<T, OP, KIND, false, CL, RN>(w, inSlot, ownSlot, outSlot, own0 + s,
                                                     out0 + s, len, flagIn, flagOut,
                                                     w.nxFull + 8 * sOut, CL && w.remotePrev);
      if (!good) return false;
    }
    // Every lane's reads of the slots are done (their values are in
    // registers and stored onwards) before lane 0 releases the FIFO slots
    // and refills the own slot: a bulk copy's writes cannot reach a read that
    // has already returned, so the refill needs no proxy fence.
    __syncwarp();
    if (w.lane == 0) {
      // (Into another CTA the st.async stores signalled the data.)
      if (snd && !w.silent && PROTO == vrProtoSimple && !RN) mbar_arrive_cta(w.nxFull + 8 * sOut);
      if (rcv && !w.silent) {
        if (CL && w.remotePrev) arrive_drained<true>(w.pvEmpty + 8 * sIn);
        else arrive_drained<false>(w.pvEmpty + 8 * sIn);
      }
      if (hasOwn) prefetch_own(w);
    }
    if (hasOwn) ++w.ownUsed;
    if (snd) ++w.sendCnt;
    if (rcv) ++w.recvCnt;
    if (snd && ++w.sOut == w.D) {
      w.sOut = 0;
      w.phOut ^= 1u;
      w.outWrapped = true;
    }
    if (rcv && ++w.sIn == w.D) {
      w.sIn = 0;
      w.phIn ^= 1u;
    }
    if (hasOwn && ++w.iOwn == w.DI) {
      w.iOwn = 0;
      w.phOwn ^= 1u;
    }
  }
  return true;
}

// Stage kind of stage k of collective `coll` on a ring of N: AllReduce SEND,
// RRS x (N-2), RRCS, RCS x (N-2), RECV; ReduceScatter SEND, RRS x (N-2), RRC;
// AllGather SC, RCS x (N-2), RECV.
__device__ __forceinline__ int stage_kind(int coll, int N, int k) {
  if (coll == VR_COLL_REDUCESCATTER) return k == 0 ? VR_SEND : k < N - 1 ? VR_RRS : VR_RRC;
  if (coll == VR_COLL_ALLGATHER) return k == 0 ? VR_SC : k < N - 1 ? VR_RCS : VR_RECV;
  return k == 0 ? VR_SEND : k < N - 1 ? VR_RRS : k == N - 1 ? VR_RRCS
       : k < 2 * N - 2 ? VR_RCS : VR_RECV;
}

// One stage; on a cluster, the warp that sends into another CTA takes the
// st.async stores (RN), every other warp the CTA-local ones.
template <typename T, int OP, int KIND, int PROTO, bool CL>
__device__ __forceinline__ bool stage(WarpRank& w, uint64_t own0, uint64_t out0, uint32_t plen) {
  if constexpr (CL) {
    if (w.remoteNext) return run_stage<T, OP, KIND, PROTO, true, true>(w, own0, out0, plen);
  }
  return run_stage<T, OP, KIND, PROTO, CL, false>(w, own0, out0, plen);
}

// One stage of a run of one kind: the next stage of the part (but for the
// first), skipped when its slice is empty.
template <typename T, int OP, int KIND, int PROTO, bool CL>
__device__ __forceinline__ bool walk_stage(WarpRank& w, PartWalk& pw, const vrStepPlan& P,
                                           bool first) {
  if (!first) pw.next_stage(P);
  if (!pw.plen) return true;
  return stage<T, OP, KIND, PROTO, CL>(w, pw.own_offset(), pw.out_offset(), pw.plen);
}

// The stages of one part. LL and LL128 in one CTA: as runs of one kind
// (AllReduce SEND, RRS x (N-2), RRCS, RCS x (N-2), RECV; ReduceScatter SEND,
// RRS x (N-2), RRC; AllGather SC, RCS x (N-2), RECV), measured faster there;
// otherwise stage by stage through one instance of each kind's code.
template <typename T, int OP, int PROTO, bool CL>
__device__ __forceinline__ bool walk_part(WarpRank& w, PartWalk& pw, const vrStepPlan& P,
                                          int lastStage) {
  if constexpr (!CL && PROTO != vrProtoSimple) {
    const int N = P.N;
    if (P.coll == VR_COLL_ALLGATHER) {
      bool ok = walk_stage<T, OP, VR_SC, PROTO, CL>(w, pw, P, true);
      if (w.lane == 0) refill_owed(w);
      for (int k = 1; ok && k < N - 1; ++k)
        ok = walk_stage<T, OP, VR_RCS, PROTO, CL>(w, pw, P, false);
      return ok && walk_stage<T, OP, VR_RECV, PROTO, CL>(w, pw, P, false);
    }
    bool ok = walk_stage<T, OP, VR_SEND, PROTO, CL>(w, pw, P, true);
    for (int k = 1; ok && k < N - 1; ++k) ok = walk_stage<T, OP, VR_RRS, PROTO, CL>(w, pw, P, false);
    if (!ok) return false;
    if (P.coll == VR_COLL_REDUCESCATTER) {
      ok = walk_stage<T, OP, VR_RRC, PROTO, CL>(w, pw, P, false);
      if (w.lane == 0) refill_owed(w);
      return ok;
    }
    ok = walk_stage<T, OP, VR_RRCS, PROTO, CL>(w, pw, P, false);
    if (w.lane == 0) refill_owed(w);
    for (int k = N; ok && k < 2 * N - 2; ++k) ok = walk_stage<T, OP, VR_RCS, PROTO, CL>(w, pw, P, false);
    return ok && walk_stage<T, OP, VR_RECV, PROTO, CL>(w, pw, P, false);
  }
  const int lastOwn = P.coll == VR_COLL_ALLGATHER ? 0 : P.N - 1;
  bool ok = true;
  for (int k = 0; ok && k <= lastStage; ++k) {
    if (k) pw.next_stage(P);
    if (k == lastOwn + 1 && w.lane == 0) refill_owed(w);
    if (!pw.plen) continue;
    const uint64_t own0 = pw.own_offset(), out0 = pw.out_offset();
    const uint32_t plen = pw.plen;
    switch (stage_kind(P.coll, P.N, k)) {
      case VR_SEND: ok = stage<T, OP, VR_SEND, PROTO, CL>(w, own0, out0, plen); break;
      case VR_RRS: ok = stage<T, OP, VR_RRS, PROTO, CL>(w, own0, out0, plen); break;
      case VR_RRCS: ok = stage<T, OP, VR_RRCS, PROTO, CL>(w, own0, out0, plen); break;
      case VR_RCS: ok = stage<T, OP, VR_RCS, PROTO, CL>(w, own0, out0, plen); break;
      case VR_RECV: ok = stage<T, OP, VR_RECV, PROTO, CL>(w, own0, out0, plen); break;
      case VR_RRC: ok = stage<T, OP, VR_RRC, PROTO, CL>(w, own0, out0, plen); break;
      default: ok = stage<T, OP, VR_SC, PROTO, CL>(w, own0, out0, plen); break;
    }
  }
  // ReduceScatter's last stage reads own data: its refills after it.
  if (lastOwn == lastStage && w.lane == 0) refill_owed(w);
  return ok;
}

// The kernel. Every ring of N ranks lies in one CTA (R rings per CTA), or,
// with CL, spans the C CTAs of a thread-block cluster: CTA j of the cluster
// holds ranks vrSplit::start(j) .. start(j) + size(j) - 1 (ceil(N / C) =
// a.ringWarps or one fewer) of each of its R rings, and the edges between
// CTAs run through distributed shared memory.
template <typename T, int OP, int PROTO, bool CL>
__global__ void __launch_bounds__(VR_WARP_MAX_THREADS, 1)
vr_ring_warp(const __grid_constant__ vrRingArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const vrStepPlan& P = a.plan;
  const int N = a.nRanks;
  const int W = CL ? a.ringWarps : N;
  const int C = CL ? (int)cluster_nctarank() : 1;
  const int cta = CL ? (int)cluster_ctarank() : 0;
  const int R = a.ringsPerCta;
  const int nWarps = R * W;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t base = smem_addr(smem);
  const uint32_t D = a.depth, DI = a.inDepth, SLOT = a.slotBytes;
  const uint32_t OWNSLOT = vrOwnSlotBytes(PROTO, SLOT);
  // Stages: AllReduce 0 .. 2N-2; the halves 0 .. N-1. Stages that read own
  // data: AllReduce and ReduceScatter 0 .. N-1; AllGather 0.
  const int lastStage = a.coll == VR_COLL_ALLREDUCE ? 2 * N - 2 : N - 1;
  const int lastOwnStage = a.coll == VR_COLL_ALLGATHER ? 0 : N - 1;

  if (warp < nWarps) {
    // Each warp sets up its own barriers and (LL, LL128) clears its
    // FIFO slots: line flags count steps from 1, so no leftover of an earlier
    // kernel may look like a flag.
    const WarpSmem m = warp_smem(base, warp, nWarps, D, DI, SLOT, OWNSLOT);
    for (uint32_t j = lane; j < 2 * D + DI; j += 32) mbar_init(m.full + 8 * j, 1);
    fence_mbarrier_init();
    if (PROTO != vrProtoSimple)
      for (uint32_t b = lane * 16; b < D * SLOT; b += 32 * 16)
        st_shared_v4(m.fifo + b, make_uint4(0, 0, 0, 0));
  }
  // Every CTA's barriers and cleared slots before any neighbour touches them.
  if (CL) cluster_sync_all();
  else __syncthreads();

  // CL: this CTA holds Wc ranks of each ring (vrSplit); W, the larger count,
  // sets the layout, so a CTA of the smaller count leaves one warp per ring idle.
  const vrSplit sp(N, C);
  const int Wc = CL ? sp.size(cta) : W;
  if (warp < nWarps && (!CL || warp % W < Wc)) {
    const int rho = warp / W, lw = warp % W;
    const int r = CL ? sp.start(cta) + lw : cta * W + lw;
    // Rank r+1: the next warp of this ring here, or the first of the next
    // CTA's part of the ring; rank r-1 likewise backwards.
    int nxCta = cta, nxWarp = warp + 1, pvCta = cta, pvWarp = warp - 1;
    if (lw + 1 == Wc) {
      nxCta = cta + 1 == C ? 0 : cta + 1;
      nxWarp = rho * W;
    }
    if (lw == 0) {
      pvCta = cta == 0 ? C - 1 : cta - 1;
      pvWarp = rho * W + (CL ? sp.size(pvCta) : W) - 1;
    }
    WarpRank w;
    w.a = &a;
    w.D = D;
    w.DI = DI;
    w.SLOT = SLOT;
    w.OWNSLOT = OWNSLOT;
    w.lane = lane;
    w.me = warp_smem(base, warp, nWarps, D, DI, SLOT, OWNSLOT);
    const WarpSmem nx = warp_smem(base, nxWarp, nWarps, D, DI, SLOT, OWNSLOT);
    const WarpSmem pv = warp_smem(base, pvWarp, nWarps, D, DI, SLOT, OWNSLOT);
    w.remoteNext = nxCta != cta;
    w.remotePrev = pvCta != cta;
    w.nxFifo = w.remoteNext ? mapa_cluster(nx.fifo, (uint32_t)nxCta) : nx.fifo;
    w.nxFull = w.remoteNext ? mapa_cluster(nx.full, (uint32_t)nxCta) : nx.full;
    w.pvEmpty = w.remotePrev ? mapa_cluster(pv.empty, (uint32_t)pvCta) : pv.empty;
    w.own = static_cast<const char*>(a.send[r]);
    w.out = static_cast<char*>(a.recv[r]);
    w.vec16 = (a.alignMask & 15) == 0;
    w.silent = (r == a.silentRank);
    w.sIn = w.phIn = w.sOut = w.phOut = w.iOwn = w.phOwn = 0;
    w.sendCnt = w.recvCnt = 0;
    w.outWrapped = false;
    w.issued = w.ownUsed = 0;
    w.iPre = 0;
    w.scale = a.scale;
    w.sPack = scalar_pack<T>(a.scalar);

    const int ring = (int)(CL ? cluster_index() : blockIdx.x) * R + rho;
    const uint64_t nRings = (uint64_t)(CL ? cluster_count() : gridDim.x) * (uint64_t)R;
    // `pre` walks the own-data steps (stages that read the input) ahead of
    // the stage loop below.
    if (lane == 0) {
      w.pre.init(r, ring, lastOwnStage);
      w.owed = DI;
      refill_owed(w);
    }
    PartWalk pw;
    bool ok = true;
    for (uint64_t unit = (uint64_t)ring; ok && unit < P.nUnits; unit += nRings) {
      pw.enter(P, r, unit);
      ok = walk_part<T, OP, PROTO, CL>(w, pw, P, lastStage);
    }
    // Bulk copies this warp issued must land before it exits (only a wait that
    // gave up leaves some unread).
    if (lane == 0) {
      for (uint32_t j = w.ownUsed; j < w.issued; ++j) {
        const uint32_t bar = w.me.inFull + 8 * (j % DI), par = (j / DI) & 1u;
        const uint64_t tw = globaltimer();
        while (!mbar_try_wait_cta(bar, par) && globaltimer() - tw < a.timeoutNs) {
        }
      }
    }
  }
  // No CTA of a cluster leaves while a neighbour may still write its FIFO
  // slots or signal its barriers (every wait above is bounded, so every
  // thread gets here).
  if (CL) cluster_sync_all();
}

}  // namespace vr

#define VR_WARP_ROW(T, CL, OP)                                                              \
  {(const void*)vr::vr_ring_warp<T, OP, 0, CL>, (const void*)vr::vr_ring_warp<T, OP, 1, CL>, \
   (const void*)vr::vr_ring_warp<T, OP, 2, CL>}
#define VR_INSTANTIATE_WARP(GETTER, T)                                                       \
  const void* GETTER(int op, int proto, int cluster) {                                      \
    static const void* table[2][4][3] = {                                                   \
        {VR_WARP_ROW(T, false, 0), VR_WARP_ROW(T, false, 1), VR_WARP_ROW(T, false, 2),      \
         VR_WARP_ROW(T, false, 3)},                                                         \
        {VR_WARP_ROW(T, true, 0), VR_WARP_ROW(T, true, 1), VR_WARP_ROW(T, true, 2),         \
         VR_WARP_ROW(T, true, 3)}};                                                         \
    return (op < 0 || op > 3 || proto < 0 || proto > 2) ? nullptr                           \
                                                        : table[cluster ? 1 : 0][op][proto]; \
  }
