// vr_cursor.cuh -- a resumable walk over one rank's FIFO steps.
//
// The walk is the ring schedule of "NCCL 原始碼解讀：一個 AllReduce 的 GPU
// 旅程", ch.2 §2.2-2.3: channels of alignUp(divUp(count, nChannels), 16/e)
// elements; in each channel loops of N * chunkElems elements, the last loop's
// chunk alignUp(divUp(rem, N), 16/e); at stage k rank r handles chunk
// (r - 1 - k) mod N. Each chunk moves in parts of `partBytes` (half the FIFO,
// so that stage 0, which sends without receiving, never fills every edge at
// once), and a part moves as steps of at most `payload` bytes. Every
// (channel, loop, part) is an independent pass of the ring; the parts are
// numbered channel by channel, loop by loop, and part u belongs to ring
// u mod G.
//
// The plan (vrStepPlan) holds the constants of one call; the host computes
// it once and every thread reads it from kernel parameter space. next()
// yields the steps in order; a cursor limited to stages 0 .. N-1 walks
// exactly the steps that read the rank's own input (for prefetching it). The
// walk costs a few divisions per part and a few additions per step.
#pragma once

#include "vr_device.cuh"

namespace vr {

// Loop structure of a channel of S elements.
VR_HD inline vrChannelShape plan_shape(uint64_t S, uint64_t L, uint64_t chunkElems, uint64_t E,
                                       uint64_t align, uint64_t N, uint64_t partBytes) {
  vrChannelShape sh;
  sh.S = S;
  sh.fullLoops = S / L;
  sh.lastRem = S - sh.fullLoops * L;
  // AllReduce splits the last loop into N chunks; the halves (L equal to
  // the chunk) keep the remainder as one chunk.
  sh.lastCur =
      sh.lastRem ? (L == chunkElems ? sh.lastRem : align_up(div_up(sh.lastRem, N), align)) : 0;
  sh.partsFullLoop = div_up(chunkElems * E, partBytes);
  sh.partsLastLoop = sh.lastRem ? div_up(sh.lastCur * E, partBytes) : 0;
  sh.units = sh.fullLoops * sh.partsFullLoop + sh.partsLastLoop;
  return sh;
}

// The walk of one call.
//
// AllReduce walks the whole buffer: loops of N chunks, stage k on chunk
// (r - 1 - k) mod N. ReduceScatter and AllGather walk one block (`count` is
// then the per-rank block): loops of one chunk, and at stage k the same range
// of block (r - 1 - k) mod N (ReduceScatter, N stages ending at block r) or
// of block (r - k) mod N (AllGather, N stages starting at block r).
VR_HD inline void plan_init(vrStepPlan& P, const vrRingArgs& a, uint64_t elemSize,
                            uint64_t nGroups, uint64_t partB, uint64_t pay) {
  P.E = elemSize;
  const uint64_t align = 16 / P.E;
  P.N = a.nRanks;
  P.coll = a.coll;
  P.per = align_up(div_up(a.count, (uint64_t)a.nChannels), align);
  P.chunkElems = a.chunkElems;
  P.loopElems = P.coll == VR_COLL_ALLREDUCE ? (uint64_t)P.N * P.chunkElems : P.chunkElems;
  P.blockBytes = a.count * P.E;
  P.partBytes = partB;
  P.payload = pay;
  P.G = nGroups;
  P.nFullCh = P.per ? a.count / P.per : 0;  // no elements: no channels
  P.full = plan_shape(P.per, P.loopElems, P.chunkElems, P.E, align, (uint64_t)P.N, P.partBytes);
  P.last = plan_shape(a.count - P.nFullCh * P.per, P.loopElems, P.chunkElems, P.E, align,
                      (uint64_t)P.N, P.partBytes);
  P.nUnits = P.nFullCh * P.full.units + P.last.units;
}

struct StepCursor {
  int N, r, maxStage, coll;
  // the current part
  uint64_t unit, partBase, rem, cur, q;
  // the current stage
  int k, c;
  uint64_t lo, plen, s;
  bool inUnit;

  VR_HD void init(const vrStepPlan& P, int rank, int grp, int lastStage) {
    N = P.N;
    coll = P.coll;
    r = rank;
    maxStage = lastStage;
    unit = (uint64_t)grp;
    inUnit = false;
  }

  // Enter part `unit`: find its channel, loop and offset within the chunk.
  VR_HD void enter_part(const vrStepPlan& P) {
    uint64_t ch, v;
    const vrChannelShape* sh;
    const uint64_t fullUnits = P.nFullCh * P.full.units;
    if (unit < fullUnits) {
      ch = unit / P.full.units;
      v = unit - ch * P.full.units;
      sh = &P.full;
    } else {
      ch = P.nFullCh;
      v = unit - fullUnits;
      sh = &P.last;
    }
    const uint64_t ppl = sh->partsFullLoop;
    uint64_t loop = ppl ? v / ppl : 0;
    if (loop < sh->fullLoops) {
      cur = P.chunkElems;
    } else {
      loop = sh->fullLoops;
      cur = sh->lastCur;
    }
    q = (v - loop * ppl) * P.partBytes;
    const uint64_t o = loop * P.loopElems;
    rem = sh->S - o;
    partBase = (ch * P.per + o) * P.E + q;
    k = 0;
    c = coll == VR_COLL_ALLGATHER ? r : (r + N - 1) % N;
    enter_stage(P);
  }

  VR_HD void enter_stage(const vrStepPlan& P) {
    plen = 0;
    if (coll == VR_COLL_ALLREDUCE) {
      lo = (uint64_t)c * cur;
      if (lo < rem) {
        const uint64_t nbytes = min_u64(rem - lo, cur) * P.E;
        if (q < nbytes) plen = min_u64(P.partBytes, nbytes - q);
      }
    } else {
      lo = 0;  // the same range of every block
      const uint64_t nbytes = cur * P.E;
      if (q < nbytes) plen = min_u64(P.partBytes, nbytes - q);
    }
    s = 0;
  }

  // The next stage of the current part (chunk index one back on the ring).
  VR_HD void next_stage(const vrStepPlan& P) {
    c = c == 0 ? N - 1 : c - 1;
    enter_stage(P);
  }

  // Stage kind of stage k.
  VR_HD int kind_of(int kk) const {
    if (coll == VR_COLL_REDUCESCATTER) return kk == 0 ? VR_SEND : kk < N - 1 ? VR_RRS : VR_RRC;
    if (coll == VR_COLL_ALLGATHER) return kk == 0 ? VR_SC : kk < N - 1 ? VR_RCS : VR_RECV;
    return kk == 0 ? VR_SEND : kk < N - 1 ? VR_RRS : kk == N - 1 ? VR_RRCS
         : kk < 2 * N - 2 ? VR_RCS : VR_RECV;
  }
  // Byte offsets of the current stage in the rank's input and output.
  VR_HD uint64_t own_offset(const vrStepPlan& P) const {
    if (coll == VR_COLL_REDUCESCATTER) return (uint64_t)c * P.blockBytes + partBase;
    return partBase + lo * P.E;
  }
  VR_HD uint64_t out_offset(const vrStepPlan& P) const {
    if (coll == VR_COLL_ALLGATHER) return (uint64_t)c * P.blockBytes + partBase;
    return partBase + lo * P.E;
  }

  // The next step: kind (VR_SEND ...), byte offset into the rank's input,
  // and length. False when the walk is over.
  VR_HD bool next(const vrStepPlan& P, int& kind, uint64_t& off, uint32_t& len) {
    for (;;) {
      if (!inUnit) {
        if (unit >= P.nUnits) return false;
        enter_part(P);
        unit += P.G;
        inUnit = true;
      }
      if (s < plen) {
        kind = kind_of(k);
        off = own_offset(P) + s;
        len = (uint32_t)min_u64(P.payload, plen - s);
        s += P.payload;
        return true;
      }
      if (++k > maxStage) {
        inUnit = false;
        continue;
      }
      next_stage(P);
    }
  }
};

}  // namespace vr
