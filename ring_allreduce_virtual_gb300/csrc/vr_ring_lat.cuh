// vr_ring_lat.cuh -- the warp-ring collectives whose every stage moves one
// FIFO step: the calls that fit one pass of their rings (every ring runs at
// most one part; the latency-bound calls, small messages or long rings, whose
// time is 2N - 1 stages of fixed cost rather than data), and the Simple calls
// of any size on rings inside one CTA, where a ring runs its parts one after
// another and the leaner stage below keeps each rank warp's period short.
//
// The schedule, the FIFOs and their signals are those of vr_ring_warp.cuh
// ("NCCL 原始碼解讀：一個 AllReduce 的 GPU 旅程", ch.2 §2.3: stage k on chunk
// (r - 1 - k) mod N; ch.2 §2.4: the Simple protocol's full / empty signals and
// the LL protocol's flag-per-8-byte-word lines), so results are bit-identical.
// What one pass allows, and this kernel does:
//  * the stages run as straight-line runs of one kind (SEND, RRS x (N-2),
//    RRCS, RCS x (N-2), RECV for the AllReduce), with no dispatch per stage;
//  * a part is entered once, and the own-data prefetch follows the part's
//    own walk a few stages ahead (no search over parts), then enters the
//    ring's next part (every nRings-th unit); every lane copies
//    the 16-byte packs it will read itself with cp.async (a ragged last pack
//    zero-filled), so no bulk copy queues on the SM's copy engine, no lane
//    waits for another's copies, and no element is read from global memory
//    in a stage;
//  * every lane waits on the barriers itself (no broadcast from one lane);
//  * an LL step reads a lane's lines in batches of five before checking
//    their flags, re-reading only the lines that were not there, and reads
//    the own data only once the lines are in.
#pragma once

#include "vr_ring_warp.cuh"

namespace vr {

// Per-warp state of one rank of one ring.
struct LatRank {
  const vrRingArgs* a;
  WarpSmem me;
  uint32_t nxFifo, nxFull;  // the next rank's FIFO slots and full barriers
  uint32_t pvEmpty;         // the previous rank's empty barriers
  const char* own;
  char* out;
  uint32_t SLOT, OWNSLOT, DI;
  uint32_t sendCnt, recvCnt;  // steps sent / received (slot = count & 1, D = 2)
  uint32_t iOwn, phOwn;       // next own-data slot to consume and its phase
  uint32_t iPre;              // next own slot to fill
  int lane;
  bool silent, remotePrev;
  int scale;
  uint4 sPack;
  PartWalk pre;  // the parts' walk, ahead of the stages, for prefetching
  int preLast;   // the last stage that reads own data
  int rank;
  uint64_t preUnit, nRings;  // the part `pre` walks; the ring's stride over parts
  uint32_t owed;             // own-slot refills waiting for the ring's next part
};

// Every lane: copy its packs (lane + 32 i) of the next own-data step of the
// part (the next stage up to preLast with a non-empty slice) into the next
// own slot, then arrive on that slot's barrier (32 arrivals) when its copies
// have landed. A lane reads only the packs it copied itself. When the part
// has no own-data step left, the refill is owed to the ring's next part
// (lat_refill_next). False if nothing was issued.
__device__ __forceinline__ bool lat_prefetch(LatRank& w, const vrStepPlan& P) {
  while (w.pre.k <= w.preLast) {
    const uint32_t len = w.pre.plen;
    const uint64_t off = w.pre.own_offset();
    w.pre.next_stage(P);
    if (!len) continue;
    const uint32_t slot = w.me.own + w.iPre * w.OWNSLOT;
    const char* src = w.own + off;
    for (uint32_t b = (uint32_t)w.lane * 16u; b < len; b += 32u * 16u)
      cp_async_16(slot + b, src + b, min(16u, len - b));
    cp_async_arrive(w.me.inFull + 8 * w.iPre);
    if (++w.iPre == w.DI) w.iPre = 0;
    return true;
  }
  ++w.owed;
  return false;
}

// After a part's last own-data stage: the refills the part could not make
// go to the own-data steps of the ring's next parts (parts g, g + nRings,
// ...), issued here, a whole half-ring of stages before they are read.
// Nothing for a one-pass call.
__device__ __forceinline__ void lat_refill_next(LatRank& w, const vrStepPlan& P) {
  while (w.owed) {
    if (w.pre.k > w.preLast) {
      w.preUnit += w.nRings;
      if (w.preUnit >= P.nUnits) {
        w.owed = 0;
        return;
      }
      w.pre.enter(P, w.rank, w.preUnit);
    }
    --w.owed;
    lat_prefetch(w, P);  // owes it again if this part's own steps are used up
  }
}

// Bounded LL poll of the lines of the packs in `pend` (bit i: pack
// p0 + 32 i; its lines at 16 p and half + 16 p of the slot at `inSlot`):
// re-reads each until its four flags equal `flag`. False if the wait gave up.
template <bool CL, int B>
__device__ __forceinline__ bool lat_ll_poll(uint32_t inSlot, uint32_t half, uint32_t p0,
                                            uint32_t flag, uint32_t pend, uint4 (&x)[B],
                                            const vrRingArgs& a) {
  uint64_t t0 = 0;
  for (uint32_t it = 1; pend; ++it) {
#pragma unroll
    for (int i = 0; i < B; ++i) {
      if (pend & (1u << i)) {
        const uint32_t q = inSlot + (p0 + 32u * i) * 16u;
        uint64_t a0, a1, b0, b1;
        ld_in_ll<CL>(q, a0, a1);
        ld_in_ll<CL>(q + half, b0, b1);
        if ((uint32_t)(a0 >> 32) == flag && (uint32_t)(a1 >> 32) == flag &&
            (uint32_t)(b0 >> 32) == flag && (uint32_t)(b1 >> 32) == flag) {
          x[i] = make_uint4((uint32_t)a0, (uint32_t)a1, (uint32_t)b0, (uint32_t)b1);
          pend &= ~(1u << i);
        }
      }
    }
    if (pend && (it & 63) == 0) {
      if (it == 64) t0 = globaltimer();
      if (ld_volatile_int(a.status) != VR_STATUS_OK) return false;
      if (globaltimer() - t0 > a.timeoutNs) {
        raise_timeout(a);
        return false;
      }
    }
  }
  return true;
}

// Packs i0 .. i0 + B - 1 of this lane (pack lane + 32 i) of one step: loads
// first (Simple: own data and incoming slot; LL: the lines, polled), then the
// hop and the stores (LL reads each own pack there, so that a batch holds
// only its lines in registers while it polls). False if an LL poll gave up.
template <typename T, int OP, int KIND, int PROTO, bool CL, bool RN, int B>
__device__ __forceinline__ bool lat_batch(const LatRank& w, int i0, uint32_t len, uint32_t inSlot,
                                          uint32_t ownSlot, uint32_t outSlot, uint32_t outBar,
                                          char* outG) {
  constexpr bool rcv = vrKindRecv(KIND), snd = vrKindSend(KIND);
  constexpr bool hasOwn = vrKindOwn(KIND), hasOut = vrKindOut(KIND);
  constexpr bool red = vrKindReduce(KIND);
  const vrRingArgs& a = *w.a;
  const uint32_t vecBytes = len & ~15u;  // whole packs
  const uint32_t lane = (uint32_t)w.lane;
  uint4 v[B], x[B];
#pragma unroll
  for (int i = 0; i < B; ++i) {
    const uint32_t b = (lane + 32u * (i0 + i)) * 16u;
    v[i] = x[i] = make_uint4(0, 0, 0, 0);
    if (b < len) {
      // a ragged last pack zero-filled
      if (hasOwn && PROTO == vrProtoSimple) v[i] = ld_shared_v4(ownSlot + b);
      if (rcv && PROTO == vrProtoSimple) x[i] = ld_shared_v4(inSlot + b);
    }
  }
  if (rcv && PROTO == vrProtoLL) {
    const uint32_t flag = w.recvCnt + 1;
    uint32_t pend = 0;
#pragma unroll
    for (int i = 0; i < B; ++i) {
      const uint32_t p = lane + 32u * (i0 + i);
      if (p * 16u < len) {
        const uint32_t q = inSlot + p * 16u;
        uint64_t a0, a1, b0, b1;
        ld_in_ll<CL>(q, a0, a1);
        ld_in_ll<CL>(q + (w.SLOT >> 1), b0, b1);
        x[i] = make_uint4((uint32_t)a0, (uint32_t)a1, (uint32_t)b0, (uint32_t)b1);
        if ((uint32_t)(a0 >> 32) != flag || (uint32_t)(a1 >> 32) != flag ||
            (uint32_t)(b0 >> 32) != flag || (uint32_t)(b1 >> 32) != flag)
          pend |= 1u << i;
      }
    }
    if (pend && !lat_ll_poll<CL, B>(inSlot, w.SLOT >> 1, lane + 32u * (uint32_t)i0, flag, pend,
                                    x, a))
      return false;
  }
  const uint64_t f = (uint64_t)(w.sendCnt + 1) << 32;
#pragma unroll
  for (int i = 0; i < B; ++i) {
    const uint32_t p = lane + 32u * (i0 + i), b = p * 16u;
    if (b < len) {
      uint4 vi = (hasOwn && PROTO != vrProtoSimple) ? ld_shared_v4(ownSlot + b) : v[i];
      if (OP == 0 && KIND != VR_SC && w.scale == VR_SCALE_PREMUL) vi = hop16<T, 1>(vi, w.sPack);
      uint4 res;
      if (KIND == VR_SEND || KIND == VR_SC) res = vi;
      else if (red) res = hop16<T, OP>(x[i], vi);
      else res = x[i];
      if (OP == 0 && (KIND == VR_RRCS || KIND == VR_RRC) && w.scale == VR_SCALE_POSTDIV)
        res = div_pack<T>(res, a.nRanks);
      if (snd && !w.silent) {
        if (PROTO == vrProtoSimple) {
          // Into another CTA by st.async, counted on its full barrier.
          if (RN) st_async_v4(outSlot + b, res, outBar);
          else st_shared_v4(outSlot + b, res);
        } else {
          // first lines in the slot's first half, second lines in its second
          st_next_ll<RN>(outSlot + p * 16u, f | res.x, f | res.y);
          st_next_ll<RN>(outSlot + (w.SLOT >> 1) + p * 16u, f | res.z, f | res.w);
        }
      }
      if (hasOut) {
        if (b < vecBytes) st_cs_v4(outG + b, res);
        else store_pack<T>(outG + b, res, len - b, false);
      }
    }
  }
  return true;
}

// One stage of kind KIND: one step of pw.plen bytes (nothing if the part's
// slice of this stage's chunk is empty, on both sides of every edge alike).
// RN: the next rank is in another CTA of the cluster. False if a wait gave up.
template <typename T, int OP, int KIND, int PROTO, bool CL, bool RN>
__device__ __forceinline__ bool lat_step(LatRank& w, const PartWalk& pw) {
  constexpr bool rcv = vrKindRecv(KIND), snd = vrKindSend(KIND);
  constexpr bool hasOwn = vrKindOwn(KIND);
  const uint32_t len = pw.plen;
  if (!len) return true;
  const vrRingArgs& a = *w.a;
  const uint32_t sIn = w.recvCnt & 1u, phIn = (w.recvCnt >> 1) & 1u;
  const uint32_t sOut = w.sendCnt & 1u, phOut = (w.sendCnt >> 1) & 1u;
  // Every lane waits: the incoming slot (Simple; LL lines carry their own
  // flags), the outgoing slot once it has been used, and the own data.
  bool ok = true;
  if (rcv && PROTO == vrProtoSimple) {
    // From another CTA the step arrives by st.async: lane 0 arms the barrier
    // with its bytes (its arrival completes the phase with them).
    if (CL && w.remotePrev && w.lane == 0)
      mbar_arrive_expect_tx(w.me.full + 8 * sIn, simple_tx_bytes(len));
    ok = lane_wait_peer<CL>(w.me.full + 8 * sIn, phIn, a);
  }
  if (ok && snd && w.sendCnt >= 2) ok = lane_wait_peer<CL>(w.me.empty + 8 * sOut, phOut ^ 1u, a);
  if (ok && hasOwn) ok = lane_wait_cta(w.me.inFull + 8 * w.iOwn, w.phOwn, a);
  if (!__all_sync(0xffffffffu, ok)) return false;

  const uint32_t inSlot = w.me.fifo + sIn * w.SLOT, ownSlot = w.me.own + w.iOwn * w.OWNSLOT;
  const uint32_t outSlot = w.nxFifo + sOut * w.SLOT;
  char* outG = w.out + pw.out_offset();
  // Simple: a lane's packs one at a time (measured fastest); LL: in batches
  // of 5, whose lines are all read before any flag is checked (a step of up
  // to 2.5 KiB, the 72-rank call's, in one batch: measured fastest).
  constexpr int B = PROTO == vrProtoSimple ? 1 : 5;
  bool dead = false;
#pragma unroll
  for (int i0 = 0; i0 < VR_LAT_PACKS; i0 += B) {
    if ((uint32_t)(w.lane + 32 * i0) * 16u < len)
      dead |= !lat_batch<T, OP, KIND, PROTO, CL, RN, B>(w, i0, len, inSlot, ownSlot, outSlot,
                                                        w.nxFull + 8 * sOut, outG);
  }
  if (PROTO == vrProtoLL && __any_sync(0xffffffffu, dead)) return false;
  // Every lane's reads of the slots have returned (their values are stored
  // onwards) before lane 0 frees the FIFO slots; each lane refills the own
  // slot's packs it has just read.
  __syncwarp();
  if (hasOwn) lat_prefetch(w, w.a->plan);
  if (w.lane == 0) {
    // (Into another CTA the st.async stores signalled the data.)
    if (snd && !w.silent && PROTO == vrProtoSimple && !RN) mbar_arrive_cta(w.nxFull + 8 * sOut);
    if (rcv && !w.silent) {
      if (CL && w.remotePrev) arrive_drained<true>(w.pvEmpty + 8 * sIn);
      else arrive_drained<false>(w.pvEmpty + 8 * sIn);
    }
  }
  if (hasOwn) {
    if (++w.iOwn == w.DI) {
      w.iOwn = 0;
      w.phOwn ^= 1u;
    }
  }
  if (snd) ++w.sendCnt;
  if (rcv) ++w.recvCnt;
  return true;
}

// A stage on a cluster: the warp that sends into another CTA takes the
// shared::cluster stores (st.async for Simple, relaxed cluster-scope stores of
// flagged LL lines).
template <typename T, int OP, int KIND, int PROTO, bool CL>
__device__ __forceinline__ bool lat_stage(LatRank& w, const PartWalk& pw, bool remoteNext) {
  if constexpr (CL) {
    if (remoteNext) return lat_step<T, OP, KIND, PROTO, true, true>(w, pw);
  }
  return lat_step<T, OP, KIND, PROTO, CL, false>(w, pw);
}

// The stages of the part, as runs of one kind: AllReduce SEND, RRS x (N-2),
// RRCS, RCS x (N-2), RECV; ReduceScatter SEND, RRS x (N-2), RRC; AllGather SC,
// RCS x (N-2), RECV.
template <typename T, int OP, int PROTO, bool CL, bool MULTI>
__device__ __forceinline__ bool lat_part(LatRank& w, PartWalk& pw, const vrStepPlan& P,
                                         bool rn) {
  const int N = P.N;
  const int coll = P.coll;
  bool ok = coll == VR_COLL_ALLGATHER ? lat_stage<T, OP, VR_SC, PROTO, CL>(w, pw, rn)
                                      : lat_stage<T, OP, VR_SEND, PROTO, CL>(w, pw, rn);
  if (coll == VR_COLL_ALLGATHER) {
    if (MULTI) lat_refill_next(w, P);
    for (int k = 1; ok && k < N - 1; ++k) {
      pw.next_stage(P);
      ok = lat_stage<T, OP, VR_RCS, PROTO, CL>(w, pw, rn);
    }
    if (!ok) return false;
    pw.next_stage(P);
    return lat_stage<T, OP, VR_RECV, PROTO, CL>(w, pw, rn);
  }
  for (int k = 1; ok && k < N - 1; ++k) {
    pw.next_stage(P);
    ok = lat_stage<T, OP, VR_RRS, PROTO, CL>(w, pw, rn);
  }
  if (!ok) return false;
  pw.next_stage(P);
  if (coll == VR_COLL_REDUCESCATTER) {
    ok = lat_stage<T, OP, VR_RRC, PROTO, CL>(w, pw, rn);
    if (MULTI) lat_refill_next(w, P);
    return ok;
  }
  if (!lat_stage<T, OP, VR_RRCS, PROTO, CL>(w, pw, rn)) return false;
  if (MULTI) lat_refill_next(w, P);
  for (int k = N; ok && k < 2 * N - 2; ++k) {
    pw.next_stage(P);
    ok = lat_stage<T, OP, VR_RCS, PROTO, CL>(w, pw, rn);
  }
  if (!ok) return false;
  pw.next_stage(P);
  return lat_stage<T, OP, VR_RECV, PROTO, CL>(w, pw, rn);
}

// The kernel: rings laid out as in vr_ring_warp (R whole rings per CTA, or
// with CL a ring over the C CTAs of a cluster), ring g running part g, or with
// MULTI parts g, g + nRings, ... one after another. The one-pass kernels keep
// no code for the parts after the first (their code size is their speed).
template <typename T, int OP, int PROTO, bool CL, bool MULTI>
__global__ void __launch_bounds__(VR_WARP_MAX_THREADS, 1)
vr_ring_lat(const __grid_constant__ vrRingArgs a) {
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
  const uint32_t D = 2, DI = a.inDepth, SLOT = a.slotBytes;
  const uint32_t OWNSLOT = vrOwnSlotBytes(PROTO, SLOT);

  if (warp < nWarps) {
    // Barriers, and (LL) cleared FIFO slots: line flags count steps from 1.
    const WarpSmem m = warp_smem(base, warp, nWarps, D, DI, SLOT, OWNSLOT);
    // full and empty: one arrival (a neighbour's); inFull: one per lane
    // (cp.async completion).
    for (uint32_t j = lane; j < 2 * D + DI; j += 32) mbar_init(m.full + 8 * j, j < 2 * D ? 1 : 32);
    fence_mbarrier_init();
    if (PROTO != vrProtoSimple)
      for (uint32_t b = lane * 16; b < D * SLOT; b += 32 * 16)
        st_shared_v4(m.fifo + b, make_uint4(0, 0, 0, 0));
  }
  if (CL) cluster_sync_all();
  else __syncthreads();

  const int rho = warp / (W > 0 ? W : 1);
  const int ring = (int)(CL ? cluster_index() : blockIdx.x) * R + rho;
  // CL: this CTA holds Wc ranks of each ring (vrSplit); W, the larger count,
  // sets the layout, so a CTA of the smaller count leaves one warp per ring idle.
  const vrSplit sp(N, C);
  const int Wc = CL ? sp.size(cta) : W;
  if (warp < nWarps && (uint64_t)ring < P.nUnits && (!CL || warp % W < Wc)) {
    const int lw = warp % W;
    const int r = CL ? sp.start(cta) + lw : cta * W + lw;
    int nxCta = cta, nxWarp = warp + 1, pvCta = cta, pvWarp = warp - 1;
    if (lw + 1 == Wc) {
      nxCta = cta + 1 == C ? 0 : cta + 1;
      nxWarp = rho * W;
    }
    if (lw == 0) {
      pvCta = cta == 0 ? C - 1 : cta - 1;
      pvWarp = rho * W + (CL ? sp.size(pvCta) : W) - 1;
    }
    LatRank w;
    w.a = &a;
    w.SLOT = SLOT;
    w.OWNSLOT = OWNSLOT;
    w.DI = DI;
    w.lane = lane;
    w.me = warp_smem(base, warp, nWarps, D, DI, SLOT, OWNSLOT);
    const WarpSmem nx = warp_smem(base, nxWarp, nWarps, D, DI, SLOT, OWNSLOT);
    const WarpSmem pv = warp_smem(base, pvWarp, nWarps, D, DI, SLOT, OWNSLOT);
    const bool remoteNext = nxCta != cta;
    w.remotePrev = pvCta != cta;
    w.nxFifo = remoteNext ? mapa_cluster(nx.fifo, (uint32_t)nxCta) : nx.fifo;
    w.nxFull = remoteNext ? mapa_cluster(nx.full, (uint32_t)nxCta) : nx.full;
    w.pvEmpty = w.remotePrev ? mapa_cluster(pv.empty, (uint32_t)pvCta) : pv.empty;
    w.own = static_cast<const char*>(a.send[r]);
    w.out = static_cast<char*>(a.recv[r]);
    w.silent = (r == a.silentRank);
    w.sendCnt = w.recvCnt = 0;
    w.iOwn = w.phOwn = 0;
    w.iPre = 0;
    w.scale = a.scale;
    w.sPack = scalar_pack<T>(a.scalar);

    PartWalk pw;
    pw.enter(P, r, (uint64_t)ring);
    w.pre = pw;
    w.preLast = a.coll == VR_COLL_ALLGATHER ? 0 : N - 1;
    w.rank = r;
    w.preUnit = (uint64_t)ring;
    w.nRings = (uint64_t)(CL ? cluster_count() : gridDim.x) * (uint64_t)R;
    w.owed = 0;
    for (uint32_t i = 0; i < DI; ++i) lat_prefetch(w, P);
    if (MULTI) {
      lat_refill_next(w, P);  // a part with fewer own-data steps than own slots
      for (uint64_t unit = (uint64_t)ring; unit < P.nUnits; unit += w.nRings) {
        if (unit != (uint64_t)ring) pw.enter(P, r, unit);
        if (!lat_part<T, OP, PROTO, CL, true>(w, pw, P, remoteNext)) break;
      }
    } else {
      lat_part<T, OP, PROTO, CL, false>(w, pw, P, remoteNext);
    }
    // Copies this lane issued land before it exits (only a wait that gave up
    // leaves some unread).
    cp_async_wait_all();
  }
  // No CTA of a cluster leaves while a neighbour may still write its FIFO
  // slots or signal its barriers (every wait above is bounded).
  if (CL) cluster_sync_all();
}

}  // namespace vr

#define VR_LAT_ROW(T, CL, OP)                                            \
  {(const void*)vr::vr_ring_lat<T, OP, 0, CL, false>,                  \
   (const void*)vr::vr_ring_lat<T, OP, 1, CL, false>}
#define VR_LAT_ROW_MULTI(T, OP) {(const void*)vr::vr_ring_lat<T, OP, 0, false, true>, nullptr}
// Getter: `cluster` 0 = one-pass rings in one CTA, 1 = one-pass rings over a
// cluster, 2 = rings in one CTA running several passes (Simple only).
#define VR_INSTANTIATE_LAT(GETTER, T)                                                       \
  const void* GETTER(int op, int proto, int cluster) {                                     \
    static const void* table[3][4][2] = {                                                  \
        {VR_LAT_ROW(T, false, 0), VR_LAT_ROW(T, false, 1), VR_LAT_ROW(T, false, 2),        \
         VR_LAT_ROW(T, false, 3)},                                                         \
        {VR_LAT_ROW(T, true, 0), VR_LAT_ROW(T, true, 1), VR_LAT_ROW(T, true, 2),           \
         VR_LAT_ROW(T, true, 3)},                                                          \
        {VR_LAT_ROW_MULTI(T, 0), VR_LAT_ROW_MULTI(T, 1), VR_LAT_ROW_MULTI(T, 2),           \
         VR_LAT_ROW_MULTI(T, 3)}};                                                         \
    return (op < 0 || op > 3 || proto < 0 || proto > 1 || cluster < 0 || cluster > 2)      \
               ? nullptr                                                                   \
               : table[cluster][op][proto];                                                \
  }
