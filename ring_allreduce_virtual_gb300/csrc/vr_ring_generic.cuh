// vr_ring_generic.cuh -- ring AllReduce over FIFOs in global memory (L2).
//
// One CTA per (channel, virtual rank); the whole grid is launched
// cooperatively so that every rank of every channel is resident at once (the
// ranks wait on each other). Rank r of channel ch walks the ring schedule of
// "NCCL 原始碼解讀：一個 AllReduce 的 GPU 旅程", ch.2 §2.3: loops of
// N * chunkElems elements, and in each loop stages k = 0 .. 2N-2 on chunk
// (r - 1 - k) mod N, receiving from rank r-1 and sending to rank r+1 through
// the FIFO of edge (ch, r -> r+1). A chunk moves as a sequence of FIFO steps
// of at most one slot of payload each.
//
// Flow control per protocol (same book, ch.2 §2.4):
//  Simple  one thread waits for the incoming tail (data ready) and the
//          outgoing head (slot free), the CTA moves the slot, then one thread
//          publishes tail (release) and head.
//  LL      every 8-byte FIFO word carries 4 payload bytes and a 32-bit flag;
//          readers poll their own words, so data needs no separate signal.
//          Slot reuse still waits on the head counter.
//  LL128   every 128-byte line carries 120 payload bytes and a 64-bit flag
//          published with release after the warp wrote the payload; readers
//          acquire the flag, then read the payload. Slot reuse waits on head.
// Flags and counters hold stepBase + local step + 1, with stepBase growing
// from call to call, so the arena is never cleared between calls.
#pragma once

#include "vr_device.cuh"

namespace vr {

struct RankCtx {
  const vrRingArgs* a;
  const char* own;
  char* out;
  char* fifoOut;
  const char* fifoIn;
  uint64_t* ctrlOut;
  uint64_t* ctrlIn;
  uint64_t sendIdx;
  uint64_t recvIdx;
  int tid;
  bool silent;
  bool vec16;
  bool vec8;
};

// ----------------------------------------------------------------- Simple
template <typename T, int OP>
__device__ void simple_step(RankCtx& c, int kind, uint64_t byteOff, uint32_t len, int* sAbort) {
  constexpr int NT = VR_GENERIC_THREADS;
  constexpr int U = VR_SIMPLE_UNROLL;
  const vrRingArgs& a = *c.a;
  const bool rcv = kind_recv(kind), snd = kind_send(kind);
  const bool own = kind_own(kind), out = kind_out(kind), red = kind_reduce(kind);
  const uint64_t gOut = a.stepBase + c.sendIdx, gIn = a.stepBase + c.recvIdx;
  if (c.tid == 0) {
    bool ok = true;
    if (rcv) ok = wait_ge(c.ctrlIn + VR_CTRL_TAIL, gIn + 1, a);
    if (ok && snd && c.sendIdx >= a.depth)
      ok = wait_ge(c.ctrlOut + VR_CTRL_HEAD, gOut + 1 - a.depth, a);
    if (!ok) *sAbort = 1;
  }
  __syncthreads();
  if (*(volatile int*)sAbort) return;
  const char* src = c.own + byteOff;
  char* dst = c.out + byteOff;
  const char* in = c.fifoIn + (c.recvIdx % a.depth) * a.slotBytes;
  char* fo = c.fifoOut + (c.sendIdx % a.depth) * a.slotBytes;
  const uint32_t nPacks = (len + 15) / 16;
  for (uint32_t base = 0; base < nPacks; base += NT * U) {
    uint4 v[U], x[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t p = base + u * NT + c.tid;
      if (p < nPacks) {
        if (own) v[u] = load_pack<T>(src + (uint64_t)p * 16, len - p * 16, c.vec16);
        if (rcv) x[u] = ld_cg_v4(in + (uint64_t)p * 16);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t p = base + u * NT + c.tid;
      if (p < nPacks) {
        uint4 res = kind == VR_SEND ? v[u] : (red ? hop16<T, OP>(x[u], v[u]) : x[u]);
        if (snd) st_cg_v4(fo + (uint64_t)p * 16, res);
        if (out) store_pack<T>(dst + (uint64_t)p * 16, res, len - p * 16, c.vec16);
      }
    }
  }
  __syncthreads();
  if (c.tid == 0 && !c.silent) {
    if (snd) {
      fence_acq_rel_gpu();  // the CTA's slot writes (ordered by the barrier) before tail
      st_relaxed_gpu(c.ctrlOut + VR_CTRL_TAIL, gOut + 1);
    }
    if (rcv) st_relaxed_gpu(c.ctrlIn + VR_CTRL_HEAD, gIn + 1);
  }
  if (snd) ++c.sendIdx;
  if (rcv) ++c.recvIdx;
}

// --------------------------------------------------------------------- LL
// A 16-byte pack of payload travels as two 16-byte lines of two 8-byte words
// {payload32, flag32}.
__device__ __forceinline__ bool ll_read_pack(const char* q, uint32_t flag, uint4& x,
                                             const vrRingArgs& a) {
  uint64_t w0, w1, w2, w3;
  ld_volatile_v2u64(q, w0, w1);
  ld_volatile_v2u64(q + 16, w2, w3);
  auto ready = [&]() {
    return (uint32_t)(w0 >> 32) == flag && (uint32_t)(w1 >> 32) == flag &&
           (uint32_t)(w2 >> 32) == flag && (uint32_t)(w3 >> 32) == flag;
  };
  if (!ready()) {
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
      ld_volatile_v2u64(q, w0, w1);
      ld_volatile_v2u64(q + 16, w2, w3);
      if (ready()) break;
      if ((it & 63) == 0) {
        if (ld_volatile_int(a.status) != VR_STATUS_OK) return false;
        if (globaltimer() - t0 > a.timeoutNs) {
          raise_timeout(a);
          return false;
        }
      }
    }
  }
  x = make_uint4((uint32_t)w0, (uint32_t)w1, (uint32_t)w2, (uint32_t)w3);
  return true;
}

__device__ __forceinline__ void ll_write_pack(char* q, uint4 v, uint32_t flag) {
  const uint64_t f = (uint64_t)flag << 32;
  st_volatile_v2u64(q, f | v.x, f | v.y);
  st_volatile_v2u64(q + 16, f | v.z, f | v.w);
}

template <typename T, int OP>
__device__ void ll_step(RankCtx& c, int kind, uint64_t byteOff, uint32_t len, int* sAbort) {
  constexpr int NT = VR_GENERIC_THREADS;
  const vrRingArgs& a = *c.a;
  const bool rcv = kind_recv(kind), snd = kind_send(kind);
  const bool own = kind_own(kind), out = kind_out(kind), red = kind_reduce(kind);
  const uint64_t gOut = a.stepBase + c.sendIdx, gIn = a.stepBase + c.recvIdx;
  if (c.tid == 0 && snd && c.sendIdx >= a.depth) {
    if (!wait_ge(c.ctrlOut + VR_CTRL_HEAD, gOut + 1 - a.depth, a)) *sAbort = 1;
  }
  __syncthreads();
  if (*(volatile int*)sAbort) return;
  const uint32_t flagOut = (uint32_t)(gOut + 1), flagIn = (uint32_t)(gIn + 1);
  const char* src = c.own + byteOff;
  char* dst = c.out + byteOff;
  const char* in = c.fifoIn + (c.recvIdx % a.depth) * a.slotBytes;
  char* fo = c.fifoOut + (c.sendIdx % a.depth) * a.slotBytes;
  const uint32_t nPacks = (len + 15) / 16;
  bool dead = false;
  for (uint32_t p = c.tid; p < nPacks; p += NT) {
    uint4 v = make_uint4(0, 0, 0, 0), x = v;
    if (own) v = load_pack<T>(src + (uint64_t)p * 16, len - p * 16, c.vec16);
    if (rcv && !ll_read_pack(in + (uint64_t)p * 32, flagIn, x, a)) {
      dead = true;
      break;
    }
    uint4 res = kind == VR_SEND ? v : (red ? hop16<T, OP>(x, v) : x);
    if (snd && !c.silent) ll_write_pack(fo + (uint64_t)p * 32, res, flagOut);
    if (out) store_pack<T>(dst + (uint64_t)p * 16, res, len - p * 16, c.vec16);
  }
  if (dead) *(volatile int*)sAbort = 1;
  __syncthreads();
  if (*(volatile int*)sAbort) return;
  if (c.tid == 0 && rcv && !c.silent) st_relaxed_gpu(c.ctrlIn + VR_CTRL_HEAD, gIn + 1);
  if (snd) ++c.sendIdx;
  if (rcv) ++c.recvIdx;
}

// ------------------------------------------------------------------ LL128
// Line layout: 8-byte words 0..14 payload, word 15 the flag. Lane j of an
// 8-lane group owns words 2j and 2j+1 of its line; lane 7 owns word 14 and the
// flag. A warp covers 4 lines per row and VR_LL128_ROWS rows per batch, with
// one release fence per batch.
template <typename T, int OP>
__device__ void ll128_step(RankCtx& c, int kind, uint64_t byteOff, uint32_t len, int* sAbort) {
  constexpr int NT = VR_GENERIC_THREADS;
  constexpr int NW = NT / 32;
  constexpr int R = VR_LL128_ROWS;
  const vrRingArgs& a = *c.a;
  const bool rcv = kind_recv(kind), snd = kind_send(kind);
  const bool own = kind_own(kind), out = kind_out(kind), red = kind_reduce(kind);
  const uint64_t gOut = a.stepBase + c.sendIdx, gIn = a.stepBase + c.recvIdx;
  if (c.tid == 0 && snd && c.sendIdx >= a.depth) {
    if (!wait_ge(c.ctrlOut + VR_CTRL_HEAD, gOut + 1 - a.depth, a)) *sAbort = 1;
  }
  __syncthreads();
  if (*(volatile int*)sAbort) return;
  const char* src = c.own + byteOff;
  char* dst = c.out + byteOff;
  const char* in = c.fifoIn + (c.recvIdx % a.depth) * a.slotBytes;
  char* fo = c.fifoOut + (c.sendIdx % a.depth) * a.slotBytes;
  const int lane = c.tid & 31, warp = c.tid >> 5;
  const int grp = lane >> 3, j = lane & 7;
  const bool flagLane = j == 7;
  const uint32_t nWords = (len + 7) / 8;
  const uint32_t nLines = (nWords + 14) / 15;
  const uint32_t nRows = (nLines + 3) / 4;
  bool dead = false;
  for (uint32_t row0 = warp; row0 < nRows; row0 += NW * R) {
    uint64_t v0[R], v1[R], x0[R], x1[R];
    uint32_t line[R];
    bool has[R];
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
      line[rr] = (row0 + rr * NW) * 4 + grp;
      has[rr] = (row0 + rr * NW) < nRows && line[rr] < nLines;
      v0[rr] = v1[rr] = x0[rr] = x1[rr] = 0;
    }
    // own payload words (issued before the flag wait)
    if (own) {
#pragma unroll
      for (int rr = 0; rr < R; ++rr) {
        if (!has[rr]) continue;
        const uint32_t w = line[rr] * 15 + 2 * j;
        if (w < nWords) v0[rr] = load_word<T>(src + (uint64_t)w * 8, len - w * 8, c.vec8);
        if (!flagLane && w + 1 < nWords)
          v1[rr] = load_word<T>(src + (uint64_t)(w + 1) * 8, len - (w + 1) * 8, c.vec8);
      }
    }
    if (rcv) {
      if (flagLane) {
        const uint64_t flag = gIn + 1;
        bool any = false;
        for (int rr = 0; rr < R && !dead; ++rr) {
          if (!has[rr]) continue;
          any = true;
          const uint64_t* fp = reinterpret_cast<const uint64_t*>(in + (uint64_t)line[rr] * 128 + 120);
          if (ld_relaxed_gpu(fp) != flag) {
            const uint64_t t0 = globaltimer();
            for (uint32_t it = 1;; ++it) {
              if (ld_relaxed_gpu(fp) == flag) break;
              if ((it & 63) == 0) {
                if (ld_volatile_int(a.status) != VR_STATUS_OK) { dead = true; break; }
                if (globaltimer() - t0 > a.timeoutNs) { raise_timeout(a); dead = true; break; }
              }
            }
          }
        }
        if (any && !dead) fence_acq_rel_gpu();
      }
      __syncwarp();  // the flag lanes' acquire, before every lane's payload loads
      if (__any_sync(0xffffffffu, dead)) { dead = true; break; }
#pragma unroll
      for (int rr = 0; rr < R; ++rr) {
        if (!has[rr]) continue;
        const char* q = in + (uint64_t)line[rr] * 128 + 16 * j;
        if (flagLane) x0[rr] = ld_cg_u64(q);
        else ld_cg_v2u64(q, x0[rr], x1[rr]);
      }
    }
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
      if (kind == VR_SEND) { x0[rr] = v0[rr]; x1[rr] = v1[rr]; }
      else if (red) { x0[rr] = hop8<T, OP>(x0[rr], v0[rr]); x1[rr] = hop8<T, OP>(x1[rr], v1[rr]); }
    }
    if (snd && !c.silent) {
#pragma unroll
      for (int rr = 0; rr < R; ++rr) {
        if (!has[rr]) continue;
        char* q = fo + (uint64_t)line[rr] * 128 + 16 * j;
        if (flagLane) st_cg_u64(q, x0[rr]);
        else st_cg_v2u64(q, x0[rr], x1[rr]);
      }
      __syncwarp();
      if (flagLane) {
        bool any = false;
#pragma unroll
        for (int rr = 0; rr < R; ++rr) any |= has[rr];
        if (any) fence_acq_rel_gpu();  // the group's payload (ordered by the warp barrier)
#pragma unroll
        for (int rr = 0; rr < R; ++rr)
          if (has[rr])
            st_relaxed_gpu(reinterpret_cast<uint64_t*>(fo + (uint64_t)line[rr] * 128 + 120), gOut + 1);
      }
    }
    if (out) {
#pragma unroll
      for (int rr = 0; rr < R; ++rr) {
        if (!has[rr]) continue;
        const uint32_t w = line[rr] * 15 + 2 * j;
        if (w < nWords) store_word<T>(dst + (uint64_t)w * 8, x0[rr], len - w * 8, c.vec8);
        if (!flagLane && w + 1 < nWords)
          store_word<T>(dst + (uint64_t)(w + 1) * 8, x1[rr], len - (w + 1) * 8, c.vec8);
      }
    }
  }
  if (dead) *(volatile int*)sAbort = 1;
  __syncthreads();
  if (*(volatile int*)sAbort) return;
  if (c.tid == 0 && rcv && !c.silent) st_relaxed_gpu(c.ctrlIn + VR_CTRL_HEAD, gIn + 1);
  if (snd) ++c.sendIdx;
  if (rcv) ++c.recvIdx;
}

// ----------------------------------------------------------------- kernel
template <typename T, int OP, int PROTO>
__global__ void __launch_bounds__(VR_GENERIC_THREADS, 4)
vr_ring_generic(const __grid_constant__ vrRingArgs a) {
  __shared__ int sAbort;
  const int N = a.nRanks;
  const int r = blockIdx.x % N;
  const int ch = blockIdx.x / N;
  const int rPrev = (r + N - 1) % N;
  if (threadIdx.x == 0) sAbort = 0;
  __syncthreads();

  constexpr uint64_t E = sizeof(T);
  const uint64_t align = 16 / E;
  const uint64_t per = align_up(div_up(a.count, (uint64_t)a.nChannels), align);
  const uint64_t chBeg = min_u64(a.count, (uint64_t)ch * per);
  const uint64_t chEnd = min_u64(a.count, chBeg + per);
  const uint64_t S = chEnd - chBeg;

  RankCtx c;
  c.a = &a;
  c.own = static_cast<const char*>(a.send[r]);
  c.out = static_cast<char*>(a.recv[r]);
  c.fifoOut = a.fifo + (uint64_t)(ch * N + r) * a.depth * a.slotBytes;
  c.fifoIn = a.fifo + (uint64_t)(ch * N + rPrev) * a.depth * a.slotBytes;
  c.ctrlOut = a.ctrl + (uint64_t)(ch * N + r) * VR_CTRL_WORDS_PER_EDGE;
  c.ctrlIn = a.ctrl + (uint64_t)(ch * N + rPrev) * VR_CTRL_WORDS_PER_EDGE;
  c.sendIdx = 0;
  c.recvIdx = 0;
  c.tid = threadIdx.x;
  c.silent = (r == a.silentRank);
  c.vec16 = (a.alignMask & 15) == 0;
  c.vec8 = (a.alignMask & 7) == 0;

  // Chunks move in parts of at most half the FIFO, each part walking all
  // 2N-1 stages before the next part starts. Stage 0 sends without
  // receiving, so a part must fit in the FIFO with room to spare, or every
  // edge fills at once and no rank can receive. The order of the parts does
  // not change which rank starts each element's fold, so results do not
  // depend on it.
  const uint64_t payload = vrPayloadPerStep(PROTO, a.slotBytes);
  const uint64_t partBytes = payload * (a.depth / 2);
  const uint64_t loopElems = (uint64_t)N * a.chunkElems;
  for (uint64_t o = 0; o < S; o += loopElems) {
    const uint64_t rem = S - o;
    const uint64_t cur = rem < loopElems ? align_up(div_up(rem, (uint64_t)N), align) : a.chunkElems;
    for (uint64_t q = 0; q < cur * E; q += partBytes) {
      for (int k = 0; k <= 2 * N - 2; ++k) {
        const int cid = (r + 2 * N - 1 - k) % N;
        const uint64_t lo = (uint64_t)cid * cur;
        if (lo >= rem) continue;  // empty chunk: neither side moves a step
        const uint64_t nbytes = min_u64(rem - lo, cur) * E;
        if (q >= nbytes) continue;  // short last chunk: no such part
        const uint64_t plen = min_u64(partBytes, nbytes - q);
        const int kind = k == 0 ? VR_SEND : k < N - 1 ? VR_RRS : k == N - 1 ? VR_RRCS
                       : k < 2 * N - 2 ? VR_RCS : VR_RECV;
        const uint64_t byteOff = (chBeg + o + lo) * E + q;
        for (uint64_t s = 0; s < plen; s += payload) {
          const uint32_t len = (uint32_t)min_u64(payload, plen - s);
          if (PROTO == vrProtoSimple) simple_step<T, OP>(c, kind, byteOff + s, len, &sAbort);
          else if (PROTO == vrProtoLL) ll_step<T, OP>(c, kind, byteOff + s, len, &sAbort);
          else ll128_step<T, OP>(c, kind, byteOff + s, len, &sAbort);
          if (*(volatile int*)&sAbort) return;
        }
      }
    }
  }
}

}  // namespace vr

// Instantiate the 4 ops x 3 protocols of one element type and a getter.
#define VR_INSTANTIATE_GENERIC(GETTER, T)                                      \
  const void* GETTER(int op, int proto) {                                    \
    static const void* table[4][3] = {                                       \
        {(const void*)vr::vr_ring_generic<T, 0, 0>, (const void*)vr::vr_ring_generic<T, 0, 1>, \
         (const void*)vr::vr_ring_generic<T, 0, 2>},                         \
        {(const void*)vr::vr_ring_generic<T, 1, 0>, (const void*)vr::vr_ring_generic<T, 1, 1>, \
         (const void*)vr::vr_ring_generic<T, 1, 2>},                         \
        {(const void*)vr::vr_ring_generic<T, 2, 0>, (const void*)vr::vr_ring_generic<T, 2, 1>, \
         (const void*)vr::vr_ring_generic<T, 2, 2>},                         \
        {(const void*)vr::vr_ring_generic<T, 3, 0>, (const void*)vr::vr_ring_generic<T, 3, 1>, \
         (const void*)vr::vr_ring_generic<T, 3, 2>}};                        \
    if (op < 0 || op > 3 || proto < 0 || proto > 2) return nullptr;          \
    return table[op][proto];                                                 \
  }
