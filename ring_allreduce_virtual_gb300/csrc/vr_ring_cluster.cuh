// vr_ring_cluster.cuh -- ring AllReduce whose FIFOs live in distributed shared
// memory: one thread-block cluster of N CTAs per ring, CTA r = virtual rank r.
//
// The schedule is the one of the global-memory kernel ("NCCL 原始碼解讀：一個
// AllReduce 的 GPU 旅程", ch.2 §2.3): stages k = 0 .. 2N-2 on chunk
// (r - 1 - k) mod N, received from rank r-1 and sent to rank r+1, chunks moved
// in parts of at most half the FIFO. What changes is where the FIFO is and how
// a step is signalled (the Simple protocol of ch.2 §2.4 -- whole slots with a
// producer-side "full" and a consumer-side "empty" signal -- in the form the
// Blackwell SM offers for SM-to-SM transfers):
//
//  * FIFO edge r-1 -> r = `depth` slots in CTA r's shared memory. Rank r-1
//    writes a slot with st.async, each 16-byte store counting its bytes on
//    CTA r's "full" mbarrier of that slot (complete_tx); rank r arms the
//    barrier with the step's byte count and waits for the phase. No flag, no
//    fence, no L2 traffic.
//  * Rank r frees a slot by a remote arrive on rank r-1's "empty" mbarrier
//    (one arrival per consumer warp).
//  * Rank r's own data is prefetched by a producer warp with bulk TMA copies
//    (global -> shared) `inDepth` steps ahead of its use; the consumer warps
//    read it from shared memory.
//  * Every (channel, loop, part) is an independent pass of the ring, so the
//    grid is a persistent set of clusters that share out the parts round
//    robin; which rank starts each element's fold depends only on the chunk
//    map, never on which cluster carries the part.
//
// Every wait is bounded by the communicator's timeout; a wait that gives up
// raises the status word, the CTA stops issuing work, waits for its own bulk
// copies, and meets the rest of its cluster at the final cluster barrier.
#pragma once

#include "vr_device.cuh"

namespace vr {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t mapa_cluster(uint32_t addr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(addr), "r"(rank));
  return d;
}
__device__ __forceinline__ void mbar_init(uint32_t addr, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(addr), "r"(count) : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t addr, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(addr), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_local(uint32_t addr) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(addr) : "memory");
}
// Remote "slot free" signal. The slot's bytes were loaded into registers and
// consumed (stored onwards) before this instruction issues.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t clusterAddr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(clusterAddr)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(addr), "r"(parity) : "memory");
  return ok != 0;
}
__device__ __forceinline__ void st_async_v4(uint32_t remoteAddr, uint4 v, uint32_t remoteBar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1,%2,%3,%4}, [%5];" ::"r"(
          remoteAddr),
      "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(remoteBar)
      : "memory");
}
__device__ __forceinline__ void tma_load_1d(uint32_t dst, const void* src, uint32_t bytes,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void bulk_copy_s2s(uint32_t dstCluster, uint32_t srcCta, uint32_t bytes,
                                              uint32_t dstBarCluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dstCluster),
      "r"(srcCta), "r"(bytes), "r"(dstBarCluster)
      : "memory");
}
__device__ __forceinline__ void bulk_store_s2g(void* dst, uint32_t srcCta, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(srcCta),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}

// Bounded wait on an mbarrier phase by one thread.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t addr, uint32_t parity,
                                                  const vrRingArgs& a) {
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

// Bounded wait by a whole warp: lane 0 spins, the others wait at the warp
// barrier, which orders their later shared-memory reads after lane 0's
// acquire. Returns the same verdict on every lane.
__device__ __forceinline__ bool warp_wait(uint32_t addr, uint32_t parity, const vrRingArgs& a) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait_bounded(addr, parity, a);
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  __syncwarp();
  return ok;
}

// The parts of the whole buffer, in a fixed order; part u belongs to cluster
// u mod G. For each of this cluster's parts, f(chBeg, loopOff, rem, cur, q).
template <typename F>
__device__ __forceinline__ void for_each_part(const vrRingArgs& a, uint64_t E, uint64_t partBytes,
                                              int group, int G, F&& f) {
  const int N = a.nRanks;
  const uint64_t align = 16 / E;
  const uint64_t per = align_up(div_up(a.count, (uint64_t)a.nChannels), align);
  const uint64_t loopElems = (uint64_t)N * a.chunkElems;
  int slot = 0;  // u mod G
  for (int ch = 0; ch < a.nChannels; ++ch) {
    const uint64_t chBeg = min_u64(a.count, (uint64_t)ch * per);
    const uint64_t S = min_u64(a.count, chBeg + per) - chBeg;
    for (uint64_t o = 0; o < S; o += loopElems) {
      const uint64_t rem = S - o;
      const uint64_t cur =
          rem < loopElems ? align_up(div_up(rem, (uint64_t)N), align) : a.chunkElems;
      for (uint64_t q = 0; q < cur * E; q += partBytes) {
        if (slot == group) {
          if (!f(chBeg, o, rem, cur, q)) return;
        }
        if (++slot == G) slot = 0;
      }
    }
  }
}

// The stages of one part for rank r: for each non-empty (stage, step),
// g(kind, byteOffset, len).
template <typename F>
__device__ __forceinline__ bool for_each_step(int N, int r, uint64_t E, uint64_t chBeg, uint64_t o,
                                              uint64_t rem, uint64_t cur, uint64_t q,
                                              uint64_t partBytes, uint64_t payload, int maxStage,
                                              F&& g) {
  for (int k = 0; k <= maxStage; ++k) {
    const int cid = (r + 2 * N - 1 - k) % N;
    const uint64_t lo = (uint64_t)cid * cur;
    if (lo >= rem) continue;
    const uint64_t nbytes = min_u64(rem - lo, cur) * E;
    if (q >= nbytes) continue;
    const uint64_t plen = min_u64(partBytes, nbytes - q);
    const int kind = k == 0 ? VR_SEND : k < N - 1 ? VR_RRS : k == N - 1 ? VR_RRCS
                   : k < 2 * N - 2 ? VR_RCS : VR_RECV;
    const uint64_t byteOff = (chBeg + o + lo) * E + q;
    for (uint64_t s = 0; s < plen; s += payload) {
      if (!g(kind, byteOff + s, (uint32_t)min_u64(payload, plen - s))) return false;
    }
  }
  return true;
}

template <typename T, int OP>
__global__ void __launch_bounds__(VR_CLUSTER_THREADS, 1)
vr_ring_cluster(const __grid_constant__ vrRingArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr uint64_t E = sizeof(T);
  constexpr int W = VR_CLUSTER_CONSUMER_WARPS;
  const int N = a.nRanks;
  const int r = blockIdx.x % N;  // == %cluster_ctarank: clusters are (N, 1, 1)
  const int group = blockIdx.x / N;
  const int G = gridDim.x / N;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t D = a.depth, DI = a.inDepth, SLOT = a.slotBytes;
  const uint32_t fifo = smem_addr(smem);         // D slots, filled by rank r-1's copies
  const uint32_t stage = fifo + D * SLOT;        // D slots: this rank's outgoing steps
  const uint32_t inbuf = stage + D * SLOT;       // DI slots of own data (TMA)
  const uint32_t bars = inbuf + DI * SLOT;
  auto full = [&](uint32_t i) { return bars + 8 * i; };
  auto empty = [&](uint32_t i) { return bars + 8 * (D + i); };
  auto staged = [&](uint32_t i) { return bars + 8 * (2 * D + i); };
  auto inFull = [&](uint32_t i) { return bars + 8 * (3 * D + i); };
  auto inEmpty = [&](uint32_t i) { return bars + 8 * (3 * D + DI + i); };

  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < D; ++i) {
      mbar_init(full(i), 1);       // the receiver's arm; bytes arrive as tx
      mbar_init(empty(i), W + 1);  // rank r+1's consumer warps + this rank's sender
      mbar_init(staged(i), W);     // this rank's consumer warps filled stage slot i
    }
    for (uint32_t i = 0; i < DI; ++i) {
      mbar_init(inFull(i), 1);     // the producer's arm; bytes arrive as tx
      mbar_init(inEmpty(i), W);    // one arrival per local consumer warp
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  cluster_sync_all();

  const int rNext = (r + 1) % N, rPrev = (r + N - 1) % N;
  const uint32_t nextFifo = mapa_cluster(fifo, rNext);
  const uint32_t nextFull0 = mapa_cluster(full(0), rNext);
  const uint32_t prevEmpty0 = mapa_cluster(empty(0), rPrev);
  const bool vec16 = (a.alignMask & 15) == 0;
  const uint64_t payload = SLOT;
  const uint64_t partBytes = payload * (D / 2);
  const char* own = static_cast<const char*>(a.send[r]);
  char* out = static_cast<char*>(a.recv[r]);
  const bool silent = (r == a.silentRank);

  if (warp == 0) {
    // ------------------------------------------------ producer: own data
    if (lane == 0) {
      uint64_t ownIdx = 0;
      for_each_part(a, E, partBytes, group, G,
                    [&](uint64_t chBeg, uint64_t o, uint64_t rem, uint64_t cur, uint64_t q) {
        return for_each_step(N, r, E, chBeg, o, rem, cur, q, partBytes, payload, N - 1,
                             [&](int kind, uint64_t off, uint32_t len) {
          (void)kind;
          const uint32_t i = (uint32_t)(ownIdx % DI);
          if (ownIdx >= DI && !mbar_wait_bounded(inEmpty(i), (uint32_t)((ownIdx / DI - 1) & 1), a))
            return false;
          const uint32_t bytes = vec16 ? (len & ~15u) : 0u;
          mbar_arrive_expect_tx(inFull(i), bytes);
          if (bytes) tma_load_1d(inbuf + i * SLOT, own + off, bytes, inFull(i));
          ++ownIdx;
          return true;
        });
      });
      // Every bulk copy issued must land before the CTA may exit, also after
      // an abort: wait for the last one of each slot, bounded by time only.
      const uint64_t first = ownIdx > DI ? ownIdx - DI : 0;
      for (uint64_t j = first; j < ownIdx; ++j) {
        const uint32_t bar = inFull((uint32_t)(j % DI)), par = (uint32_t)((j / DI) & 1);
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(bar, par) && globaltimer() - t0 < a.timeoutNs) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ sender: bulk copies
    if (lane == 0) {
      uint64_t sendIdx = 0, lastIssue = 0;
      bool ok = true;
      for_each_part(a, E, partBytes, group, G,
                    [&](uint64_t chBeg, uint64_t o, uint64_t rem, uint64_t cur, uint64_t q) {
        return ok = for_each_step(N, r, E, chBeg, o, rem, cur, q, partBytes, payload, 2 * N - 2,
                                  [&](int kind, uint64_t off, uint32_t len) {
          if (!kind_send(kind)) return true;  // the last stage only writes recv
          const uint32_t sOut = (uint32_t)(sendIdx % D);
          if (!mbar_wait_bounded(staged(sOut), (uint32_t)((sendIdx / D) & 1), a)) return false;
          const uint32_t src = stage + sOut * SLOT;
          if (!silent)
            bulk_copy_s2s(nextFifo + sOut * SLOT, src, ((len + 15) >> 4) * 16, nextFull0 + 8 * sOut);
          const uint32_t outBytes = vec16 ? (len & ~15u) : 0u;
          if (kind_out(kind) && outBytes) {
            bulk_store_s2g(out + off, src, outBytes);
            bulk_commit();
            bulk_wait_read_all();  // the stage slot may be refilled after this
          }
          mbar_arrive_local(empty(sOut));
          lastIssue = globaltimer();
          ++sendIdx;
          return true;
        });
      });
      bulk_wait_all();  // outputs written before the kernel ends
      if (!ok) {
        // Copies into a neighbour's shared memory complete there; after an
        // abort nobody waits for them, so give the last one time to read
        // this CTA's stage slot before the CTA may exit.
        while (globaltimer() - lastIssue < 100000ull) {
        }
      }
    }
  } else {
    // ------------------------------------------------ consumers
    const int cw = warp - 2;
    uint64_t sendIdx = 0, recvIdx = 0, ownIdx = 0;
    for_each_part(a, E, partBytes, group, G,
                  [&](uint64_t chBeg, uint64_t o, uint64_t rem, uint64_t cur, uint64_t q) {
      return for_each_step(N, r, E, chBeg, o, rem, cur, q, partBytes, payload, 2 * N - 2,
                           [&](int kind, uint64_t off, uint32_t len) {
        const bool rcv = kind_recv(kind), snd = kind_send(kind);
        const bool hasOwn = kind_own(kind), hasOut = kind_out(kind), red = kind_reduce(kind);
        const uint32_t nPacks = (len + 15) >> 4;
        const uint32_t sIn = (uint32_t)(recvIdx % D), sOut = (uint32_t)(sendIdx % D);
        const uint32_t iIn = (uint32_t)(ownIdx % DI);
        if (rcv) {
          if (cw == 0 && lane == 0) mbar_arrive_expect_tx(full(sIn), nPacks * 16);
          if (!warp_wait(full(sIn), (uint32_t)((recvIdx / D) & 1), a)) return false;
        }
        if (snd && sendIdx >= D &&
            !warp_wait(empty(sOut), (uint32_t)((sendIdx / D - 1) & 1), a))
          return false;
        if (hasOwn && !warp_wait(inFull(iIn), (uint32_t)((ownIdx / DI) & 1), a)) return false;
        const uint32_t ownBytes = vec16 ? (len & ~15u) : 0u;
        // Outputs the sender's bulk store does not cover: the last stage (no
        // stage slot), unaligned buffers, and a final partial 16 bytes.
        const uint32_t outDirectFrom = (snd && vec16) ? (len & ~15u) : 0u;
        const uint32_t inSlot = fifo + sIn * SLOT, ownSlot = inbuf + iIn * SLOT;
        const uint32_t outSlot = stage + sOut * SLOT;
        for (uint32_t p = cw * 32 + lane; p < nPacks; p += W * 32) {
          uint4 v = make_uint4(0, 0, 0, 0), x = v;
          if (hasOwn) {
            if (p * 16 + 16 <= ownBytes) v = ld_shared_v4(ownSlot + p * 16);
            else v = load_pack<T>(own + off + (uint64_t)p * 16, len - p * 16, false);
          }
          if (rcv) x = ld_shared_v4(inSlot + p * 16);
          const uint4 res = kind == VR_SEND ? v : (red ? hop16<T, OP>(x, v) : x);
          if (snd) st_shared_v4(outSlot + p * 16, res);
          if (hasOut && p * 16 >= outDirectFrom)
            store_pack<T>(out + off + (uint64_t)p * 16, res, len - p * 16, vec16);
        }
        if (snd) fence_proxy_async_shared();  // stage writes before the bulk copies read them
        __syncwarp();
        if (lane == 0) {
          if (snd) mbar_arrive_local(staged(sOut));
          if (rcv && !silent) mbar_arrive_remote(prevEmpty0 + 8 * sIn);
          if (hasOwn) mbar_arrive_local(inEmpty(iIn));
        }
        if (snd) ++sendIdx;
        if (rcv) ++recvIdx;
        if (hasOwn) ++ownIdx;
        return true;
      });
    });
  }
  __syncwarp();
  // No CTA of the cluster leaves while a neighbour may still signal or copy
  // into its shared memory.
  cluster_sync_all();
}

}  // namespace vr

#define VR_INSTANTIATE_CLUSTER(GETTER, T)                                         \
  const void* GETTER(int op) {                                                    \
    static const void* table[4] = {(const void*)vr::vr_ring_cluster<T, 0>,         \
                                   (const void*)vr::vr_ring_cluster<T, 1>,         \
                                   (const void*)vr::vr_ring_cluster<T, 2>,         \
                                   (const void*)vr::vr_ring_cluster<T, 3>};        \
    return (op < 0 || op > 3) ? nullptr : table[op];                              \
  }
