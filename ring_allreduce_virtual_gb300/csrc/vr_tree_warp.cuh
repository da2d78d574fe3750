// vr_tree_warp.cuh -- double-binary-tree AllReduce with every virtual rank a
// pair of warps and every tree edge a FIFO in the shared memory of one SM.
//
// The trees are those of "NCCL 原始碼解讀：一個 AllReduce 的 GPU 旅程", ch.4
// (ncclGetBtree: rank 0 the root with the largest power of two below N as its
// child; rank r with lowest set bit b under "r with bit b cleared and bit 2b
// set", or under r - b when that is out of range, with children r - b/2 and
// r + b/2, the second halved down while out of range; ncclGetDtree: the
// second tree is the mirror r -> N - 1 - r for even N and the first tree on
// ranks shifted by one for odd N). Each tree reduces half of the buffer
// ("NVIDIA GPU 集合通信库 NCCL 初始化流程源码级剖析", NCCL Tree 拓扑, Double
// Binary Tree): from the leaves to the root a node reduces the data its
// children send with its own (own first, then child 0, then child 1, rounded
// to the element type at every op), then the root's result is broadcast back
// down.
//
// A CTA (CL: a thread-block cluster, ceil(N / C) or floor(N / C) ranks in
// each of its C CTAs, placed by vrSplit)
// runs one tree over all N ranks, even ones the first tree and odd ones the
// second: warp 2i of a CTA moves its rank's reduction up the tree and warp
// 2i+1 moves the result down, so the two phases of different pieces overlap.
// Every rank owns three FIFOs of `depth` slots, each with a "full" barrier:
// one from each child on the way up and one from its parent on the way down
// (the root's up warp feeds its own down FIFO); the "empty" barriers live with
// the senders (its up output, its two down outputs), so every wait is on a
// barrier of the waiting warp's own CTA and edges between CTAs of a cluster
// are signalled at cluster scope. `inDepth` own-data slots per rank are
// filled by its up warp with bulk TMA copies ahead of use. The half of the
// buffer a tree reduces is cut into pieces of one slot per rank, spread round
// robin over the CTAs (clusters) of that tree; every warp takes the same
// pieces in the same order, so slot k mod depth carries piece k of every FIFO.
//
// Every wait is bounded by the communicator's timeout; a wait that gives up
// raises the status word and the warp stops.
#pragma once

#include "vr_ring_warp.cuh"  // barrier and shared-memory primitives

namespace vr {

// Parent and children of rank r in tree `tree` of N ranks (-1: none).
__device__ __forceinline__ void tree_btree(int N, int r, int& up, int& d0, int& d1) {
  if (r == 0) {
    int p = 1;
    while (p < N) p <<= 1;
    up = -1;
    d0 = -1;
    d1 = N > 1 ? p >> 1 : -1;
    return;
  }
  const int b = r & -r;  // lowest set bit
  int parent = (r - b) | (2 * b);
  if (parent >= N) parent = r - b;
  up = parent;
  int step = b >> 1;
  d0 = step ? r - step : -1;
  while (step && r + step >= N) step >>= 1;
  d1 = step ? r + step : -1;
}
__device__ __forceinline__ void tree_node(int N, int r, int tree, int& up, int& d0, int& d1) {
  if (tree == 0) {
    tree_btree(N, r, up, d0, d1);
    return;
  }
  const bool mirror = (N & 1) == 0;
  const int m = mirror ? N - 1 - r : (r + N - 1) % N;
  tree_btree(N, m, up, d0, d1);
  auto back = [&](int x) { return x < 0 ? -1 : mirror ? N - 1 - x : (x + 1) % N; };
  up = back(up);
  d0 = back(d0);
  d1 = back(d1);
}

// Shared memory of the i-th of the W ranks of a CTA: FIFOs up0, up1 (from its
// children), down (from its parent), `depth` slots each, and `inDepth`
// own-data slots; then, after every rank's slots, its barriers: full[3][D] of
// its FIFOs, upEmpty[D] (its up output drained), downEmpty[2][D] (its two
// down outputs drained), inFull[DI] (own data landed).
struct TreeSmem {
  uint32_t fifo[3];   // slot 0 of up0, up1, down
  uint32_t full[3];
  uint32_t upEmpty;
  uint32_t downEmpty[2];
  uint32_t own, inFull;
};
__device__ __forceinline__ TreeSmem tree_smem(uint32_t base, int i, int W, uint32_t D,
                                              uint32_t DI, uint32_t SLOT) {
  TreeSmem m;
  const uint32_t per = (3 * D + DI) * SLOT;
  const uint32_t bars = base + (uint32_t)W * per + (uint32_t)i * 8 * (6 * D + DI);
  for (int f = 0; f < 3; ++f) {
    m.fifo[f] = base + (uint32_t)i * per + (uint32_t)f * D * SLOT;
    m.full[f] = bars + (uint32_t)f * 8 * D;
  }
  m.upEmpty = bars + 24 * D;
  m.downEmpty[0] = bars + 32 * D;
  m.downEmpty[1] = bars + 40 * D;
  m.own = base + (uint32_t)i * per + 3 * D * SLOT;
  m.inFull = bars + 48 * D;
  return m;
}

// Rank x's shared memory as seen from this CTA: local, or (CL) the
// shared::cluster window of the CTA holding it (placed by `sp`; W, the
// largest count of ranks in a CTA, sets every CTA's layout).
template <bool CL>
__device__ __forceinline__ TreeSmem tree_smem_of(uint32_t base, int x, int W, const vrSplit& sp,
                                                 int myCta, uint32_t D, uint32_t DI,
                                                 uint32_t SLOT) {
  const int cx = CL ? sp.cta_of(x) : 0;
  TreeSmem m = tree_smem(base, CL ? x - sp.start(cx) : x, W, D, DI, SLOT);
  if (CL && cx != myCta) {
    const uint32_t c = (uint32_t)cx;
    for (int f = 0; f < 3; ++f) {
      m.fifo[f] = mapa_cluster(m.fifo[f], c);
      m.full[f] = mapa_cluster(m.full[f], c);
    }
    m.upEmpty = mapa_cluster(m.upEmpty, c);
    m.downEmpty[0] = mapa_cluster(m.downEmpty[0], c);
    m.downEmpty[1] = mapa_cluster(m.downEmpty[1], c);
  }
  return m;
}

// Signal a barrier of rank x (another CTA's at cluster scope).
template <bool CL>
__device__ __forceinline__ void tree_arrive(uint32_t bar, bool remote) {
  if (CL && remote) arrive_peer<true>(bar);
  else mbar_arrive_cta(bar);
}
// A drained slot (no ordering needed: see arrive_drained).
template <bool CL>
__device__ __forceinline__ void tree_drained(uint32_t bar, bool remote) {
  if (CL && remote) arrive_drained<true>(bar);
  else arrive_drained<false>(bar);
}

// The geometry of one call: the element range of the tree's half, the
// pieces of it, and this CTA's share.
struct TreeHalf {
  uint64_t lo, hi;       // elements of the half
  uint64_t pieceElems;
  uint64_t nPieces;
};

// A store of one pack into a tree FIFO slot: into another CTA by st.async,
// counted on the receiver's full barrier `bar` (nothing when the rank is
// silent), else a plain (shared::cluster with CL) store.
template <bool CL>
__device__ __forceinline__ void tree_put(uint32_t addr, uint4 v, bool async, uint32_t bar,
                                         bool silent) {
  if (CL && async) {
    if (!silent) st_async_v4(addr, v, bar);
  } else {
    st_next_v4<CL>(addr, v);
  }
}

// One piece's data on the way up: own, op child 0, op child 1 -> dst. The
// own data is in the own slot (bulk copy), except bytes the copy left out.
template <typename T, int OP, bool CL>
__device__ __forceinline__ void tree_up_data(int lane, uint32_t ownSlot, const char* own,
                                             uint32_t c0, uint32_t c1, bool h0, bool h1,
                                             uint32_t dst, bool dstAsync, uint32_t dstBar,
                                             bool silent, uint32_t len, bool vec, bool premul,
                                             uint4 sPack, int divN) {
  const uint32_t nPacks = (len + 15) >> 4;
  const uint32_t vecBytes = vec ? (len & ~15u) : 0u;
  for (uint32_t p = lane; p < nPacks; p += 32) {
    const uint32_t b = p * 16;
    uint4 v = b < vecBytes ? ld_shared_v4(ownSlot + b) : load_pack<T>(own + b, len - b, false);
    if (OP == 0 && premul) v = hop16<T, 1>(v, sPack);
    if (h0) v = hop16<T, OP>(v, ld_shared_v4(c0 + b));
    if (h1) v = hop16<T, OP>(v, ld_shared_v4(c1 + b));
    if (OP == 0 && divN) v = div_pack<T>(v, divN);
    tree_put<CL>(dst + b, v, dstAsync, dstBar, silent);
  }
}

// One piece's data on the way down: src -> output and the children's FIFOs.
template <typename T, bool CL>
__device__ __forceinline__ void tree_down_data(int lane, uint32_t src, char* out, uint32_t k0,
                                               uint32_t k1, bool h0, bool h1, bool a0, bool a1,
                                               uint32_t b0, uint32_t b1, bool silent, uint32_t len,
                                               bool vec) {
  const uint32_t nPacks = (len + 15) >> 4;
  const uint32_t vecBytes = vec ? (len & ~15u) : 0u;
  for (uint32_t p = lane; p < nPacks; p += 32) {
    const uint32_t b = p * 16;
    const uint4 x = ld_shared_v4(src + b);
    if (h0) tree_put<CL>(k0 + b, x, a0, b0, silent);
    if (h1) tree_put<CL>(k1 + b, x, a1, b1, silent);
    if (b < vecBytes) st_cs_v4(out + b, x);
    else store_pack<T>(out + b, x, len - b, false);
  }
}

template <typename T, int OP, bool CL>
__global__ void __launch_bounds__(2 * 32 * VR_WARP_MAX_RANKS, 1)
vr_tree_warp(const __grid_constant__ vrRingArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr uint64_t E = sizeof(T);
  const int N = a.nRanks;
  const int W = CL ? a.ringWarps : N;  // ranks per CTA (CL: the larger count)
  const int myCta = CL ? (int)cluster_ctarank() : 0;
  const vrSplit sp(N, CL ? (int)cluster_nctarank() : 1);
  const int Wc = CL ? sp.size(myCta) : N;  // ranks in this CTA
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t base = smem_addr(smem);
  const uint32_t D = a.depth, DI = a.inDepth, SLOT = a.slotBytes;
  const uint64_t group = CL ? cluster_index() : blockIdx.x;
  const uint64_t nGroups = CL ? cluster_count() : gridDim.x;
  const int tree = (int)(group & 1);
  const uint64_t G = (nGroups - tree + 1) / 2;  // CTAs (clusters) of this tree
  const uint64_t cta = group >> 1;

  if (warp < 2 * W && (warp & 1) == 0) {
    const TreeSmem m = tree_smem(base, warp >> 1, W, D, DI, SLOT);
    for (uint32_t j = lane; j < 6 * D + DI; j += 32) mbar_init(m.full[0] + 8 * j, 1);
    fence_mbarrier_init();
  }
  if (CL) cluster_sync_all();
  else __syncthreads();

  if (warp < 2 * Wc) {
    // This tree's half of the buffer, in pieces of one slot per rank.
    const uint64_t split = min_u64(align_up(div_up(a.count, 2), 16 / E), a.count);
    TreeHalf half;
    half.lo = tree == 0 ? 0 : split;
    half.hi = tree == 0 ? split : a.count;
    half.pieceElems = SLOT / E;
    half.nPieces = div_up(half.hi - half.lo, half.pieceElems);

    const int r = (CL ? sp.start(myCta) : 0) + (warp >> 1);
    const bool upWarp = (warp & 1) == 0;
    int up, d0, d1;
    tree_node(N, r, tree, up, d0, d1);
    const TreeSmem me = tree_smem(base, warp >> 1, W, D, DI, SLOT);
    const bool vec = (a.alignMask & 15) == 0;
    const bool silent = r == a.silentRank;
    const bool h0 = d0 >= 0, h1 = d1 >= 0;
    auto remote = [&](int x) { return CL && sp.cta_of(x) != myCta; };
    bool ok = true;
    uint32_t k = 0;  // pieces this warp has moved
    if (upWarp) {
      // Where this rank's partial goes: its parent's up FIFO (the slot of the
      // child it is) or, at the root, its own down FIFO.
      uint32_t dstFifo, dstFull;
      bool dstRemote = false;
      if (up >= 0) {
        int pu, p0, p1;
        tree_node(N, up, tree, pu, p0, p1);
        const TreeSmem pm = tree_smem_of<CL>(base, up, W, sp, myCta, D, DI, SLOT);
        const int f = p0 == r ? 0 : 1;
        dstFifo = pm.fifo[f];
        dstFull = pm.full[f];
        dstRemote = remote(up);
      } else {
        dstFifo = me.fifo[2];
        dstFull = me.full[2];
      }
      // The children's "up output drained" barriers.
      const uint32_t c0Empty = h0 ? tree_smem_of<CL>(base, d0, W, sp, myCta, D, DI, SLOT).upEmpty : 0;
      const uint32_t c1Empty = h1 ? tree_smem_of<CL>(base, d1, W, sp, myCta, D, DI, SLOT).upEmpty : 0;
      const char* own = static_cast<const char*>(a.send[r]);
      // Sum kernels: a pre-multiplied sum scales every own element as it
      // enters; the integer average divides at the root, once, before the
      // result goes down.
      const bool premul = OP == 0 && a.scale == VR_SCALE_PREMUL;
      const uint4 sPack = scalar_pack<T>(a.scalar);
      const int divN = OP == 0 && a.scale == VR_SCALE_POSTDIV && up < 0 ? N : 0;
      // Lane 0 copies the own data of this group's piece j into own slot j
      // mod DI, DI pieces ahead of use.
      uint32_t issued = 0;
      auto prefetch = [&](uint32_t j) {
        const uint64_t pc = cta + (uint64_t)j * G;
        if (pc >= half.nPieces) return;
        const uint64_t e0 = half.lo + pc * half.pieceElems;
        const uint32_t len = (uint32_t)(min_u64(half.pieceElems, half.hi - e0) * E);
        const uint32_t bytes = vec ? (len & ~15u) : 0u;
        const uint32_t bar = me.inFull + 8 * (j % DI);
        mbar_arrive_expect_tx(bar, bytes);
        if (bytes) tma_load_1d(me.own + (j % DI) * SLOT, own + e0 * E, bytes, bar);
        ++issued;
      };
      if (lane == 0)
        for (uint32_t j = 0; j < DI; ++j) prefetch(j);
      for (uint64_t pc = cta; ok && pc < half.nPieces; pc += G, ++k) {
        const uint64_t e0 = half.lo + pc * half.pieceElems;
        const uint32_t len = (uint32_t)(min_u64(half.pieceElems, half.hi - e0) * E);
        const uint32_t s = k % D, ph = (k / D) & 1u;
        const uint32_t io = k % DI, pho = (k / DI) & 1u;
        if (lane == 0) {
          // A child in another CTA sends by st.async: arm its full barrier
          // with the piece's bytes (this arrival completes the phase).
          if (CL && h0 && remote(d0)) mbar_arrive_expect_tx(me.full[0] + 8 * s, simple_tx_bytes(len));
          if (CL && h1 && remote(d1)) mbar_arrive_expect_tx(me.full[1] + 8 * s, simple_tx_bytes(len));
          if (h0) ok = lane_wait_peer<CL>(me.full[0] + 8 * s, ph, a);
          if (ok && h1) ok = lane_wait_peer<CL>(me.full[1] + 8 * s, ph, a);
          if (ok && k >= D) ok = lane_wait_peer<CL>(me.upEmpty + 8 * s, ph ^ 1u, a);
          if (ok) ok = lane_wait_cta(me.inFull + 8 * io, pho, a);
        }
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
        __syncwarp();
        tree_up_data<T, OP, CL>(lane, me.own + io * SLOT, own + e0 * E, me.fifo[0] + s * SLOT,
                                me.fifo[1] + s * SLOT, h0, h1, dstFifo + s * SLOT, dstRemote,
                                dstFull + 8 * s, silent, len, vec, premul, sPack, divN);
        // Every lane's reads of the slots have returned: release them, and
        // refill the own slot (no proxy fence needed for a read that returned).
        __syncwarp();
        if (lane == 0) {
          if (!silent) {
            if (!dstRemote) tree_arrive<CL>(dstFull + 8 * s, false);
            if (h0) tree_drained<CL>(c0Empty + 8 * s, remote(d0));
            if (h1) tree_drained<CL>(c1Empty + 8 * s, remote(d1));
          }
          prefetch(k + DI);
        }
      }
      // Bulk copies this warp issued must land before it exits (only a wait
      // that gave up leaves some unread).
      if (lane == 0) {
        for (uint32_t j = k; j < issued; ++j) {
          const uint32_t bar = me.inFull + 8 * (j % DI), par = (j / DI) & 1u;
          const uint64_t tw = globaltimer();
          while (!mbar_try_wait_cta(bar, par) && globaltimer() - tw < a.timeoutNs) {
          }
        }
      }
    } else {
      // The result arrives in this rank's down FIFO; it goes to the output and
      // to each child's down FIFO.
      uint32_t k0 = 0, k1 = 0, f0 = 0, f1 = 0;
      if (h0) {
        const TreeSmem cm = tree_smem_of<CL>(base, d0, W, sp, myCta, D, DI, SLOT);
        k0 = cm.fifo[2];
        f0 = cm.full[2];
      }
      if (h1) {
        const TreeSmem cm = tree_smem_of<CL>(base, d1, W, sp, myCta, D, DI, SLOT);
        k1 = cm.fifo[2];
        f1 = cm.full[2];
      }
      // Who drained this rank's down slot tells its sender: the parent (its
      // down output to this child) or, at the root, its own up warp.
      uint32_t srcEmpty;
      bool srcRemote = false;
      if (up >= 0) {
        int pu, p0, p1;
        tree_node(N, up, tree, pu, p0, p1);
        srcEmpty = tree_smem_of<CL>(base, up, W, sp, myCta, D, DI, SLOT).downEmpty[p0 == r ? 0 : 1];
        srcRemote = remote(up);
      } else {
        srcEmpty = me.upEmpty;
      }
      for (uint64_t pc = cta; ok && pc < half.nPieces; pc += G, ++k) {
        const uint64_t e0 = half.lo + pc * half.pieceElems;
        const uint32_t len = (uint32_t)(min_u64(half.pieceElems, half.hi - e0) * E);
        const uint32_t s = k % D, ph = (k / D) & 1u;
        if (lane == 0) {
          if (CL && srcRemote) mbar_arrive_expect_tx(me.full[2] + 8 * s, simple_tx_bytes(len));
          ok = lane_wait_peer<CL>(me.full[2] + 8 * s, ph, a);
          if (ok && h0 && k >= D) ok = lane_wait_peer<CL>(me.downEmpty[0] + 8 * s, ph ^ 1u, a);
          if (ok && h1 && k >= D) ok = lane_wait_peer<CL>(me.downEmpty[1] + 8 * s, ph ^ 1u, a);
        }
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
        __syncwarp();
        tree_down_data<T, CL>(lane, me.fifo[2] + s * SLOT,
                              static_cast<char*>(a.recv[r]) + e0 * E, k0 + s * SLOT,
                              k1 + s * SLOT, h0, h1, h0 && remote(d0), h1 && remote(d1),
                              f0 + 8 * s, f1 + 8 * s, silent, len, vec);
        __syncwarp();
        if (lane == 0 && !silent) {
          // (Into another CTA the st.async stores signalled the data.)
          if (h0 && !remote(d0)) tree_arrive<CL>(f0 + 8 * s, false);
          if (h1 && !remote(d1)) tree_arrive<CL>(f1 + 8 * s, false);
          tree_drained<CL>(srcEmpty + 8 * s, srcRemote);
        }
      }
    }
  }
  // No CTA of a cluster leaves while a neighbour may still write its FIFOs or
  // signal its barriers (every wait above is bounded).
  if (CL) cluster_sync_all();
}

}  // namespace vr

#define VR_INSTANTIATE_TREE(GETTER, T)                                                    \
  const void* GETTER(int op, int cluster) {                                              \
    static const void* table[2][4] = {                                                   \
        {(const void*)vr::vr_tree_warp<T, 0, false>, (const void*)vr::vr_tree_warp<T, 1, false>, \
         (const void*)vr::vr_tree_warp<T, 2, false>, (const void*)vr::vr_tree_warp<T, 3, false>}, \
        {(const void*)vr::vr_tree_warp<T, 0, true>, (const void*)vr::vr_tree_warp<T, 1, true>,   \
         (const void*)vr::vr_tree_warp<T, 2, true>, (const void*)vr::vr_tree_warp<T, 3, true>}};  \
    return (op < 0 || op > 3) ? nullptr : table[cluster ? 1 : 0][op];                    \
  }
