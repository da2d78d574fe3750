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
// it once and every thread reads it from kernel parameter space. PartWalk
// gives the stages of one part (up to three divisions to enter it; an add, a
// multiply and two compares per stage); StepWalk strings the parts of a ring
// together step by step.
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

// Quotient of two 64-bit counts, in 32-bit arithmetic when both fit.
VR_HD inline uint64_t div_u64(uint64_t a, uint64_t b) {
  if (((a | b) >> 32) == 0) return (uint64_t)((uint32_t)a / (uint32_t)b);
  return a / b;
}

// One part of the walk, stage by stage. At stage k the rank handles chunk
// (block) c, with c one back on the ring at every stage; the stage's bytes
// start at ownBase + c * ownStep in the input and outBase + c * outStep in the
// output, and number plen (0: the chunk has nothing in this part).
struct PartWalk {
  uint64_t ownBase, ownStep, outBase, outStep;
  uint64_t remB, curB, q;  // loop bytes left, chunk bytes, part offset in its chunk
  uint32_t plen, plenU;    // this stage's length; the length at every whole chunk
  uint32_t plenLast;       // the length at chunk fullC, the loop's partial chunk
  int N, k, c;
  int fullC;               // chunks 0 .. fullC - 1 of the loop are whole
  bool uniform;            // every chunk of the part's loop is whole

  // Enter part `unit` of rank r at stage 0: find its channel, loop and
  // offset within the chunk.
  VR_HD void enter(const vrStepPlan& P, int r, uint64_t unit) {
    uint64_t ch, v;
    const vrChannelShape* sh;
    const uint64_t fullUnits = P.nFullCh * P.full.units;
    if (unit < fullUnits) {
      ch = div_u64(unit, P.full.units);
      v = unit - ch * P.full.units;
      sh = &P.full;
    } else {
      ch = P.nFullCh;
      v = unit - fullUnits;
      sh = &P.last;
    }
    const uint64_t ppl = sh->partsFullLoop;
    uint64_t loop = ppl ? div_u64(v, ppl) : 0;
    uint64_t cur;
    if (loop < sh->fullLoops) {
      cur = P.chunkElems;
    } else {
      loop = sh->fullLoops;
      cur = sh->lastCur;
    }
    q = (v - loop * ppl) * P.partBytes;
    const uint64_t o = loop * P.loopElems;
    N = P.N;
    remB = (sh->S - o) * P.E;
    curB = cur * P.E;
    const uint64_t partBase = (ch * P.per + o) * P.E + q;
    ownBase = outBase = partBase;
    if (P.coll == VR_COLL_ALLREDUCE) {
      ownStep = outStep = curB;
      uniform = remB >= (uint64_t)N * curB;
    } else {
      // The halves: the same range of every block; own blocks (ReduceScatter)
      // or output blocks (AllGather) are blockBytes apart.
      ownStep = P.coll == VR_COLL_REDUCESCATTER ? P.blockBytes : 0;
      outStep = P.coll == VR_COLL_ALLGATHER ? P.blockBytes : 0;
      uniform = true;
    }
    plenU = (uint32_t)min_u64(P.partBytes, curB - q);
    // A loop shorter than N whole chunks (AllReduce's last): fullC whole
    // chunks, then one of lastB bytes (possibly none), then empty ones.
    fullC = N;
    plenLast = 0;
    if (!uniform) {
      fullC = (int)div_u64(remB, curB);
      const uint64_t lastB = remB - (uint64_t)fullC * curB;
      plenLast = q < lastB ? (uint32_t)min_u64(P.partBytes, lastB - q) : 0u;
    }
    k = 0;
    c = P.coll == VR_COLL_ALLGATHER ? r : (r + N - 1) % N;
    plen = stage_len(P);
  }

  // Length of the current stage: the part's slice of chunk c.
  VR_HD uint32_t stage_len(const vrStepPlan&) const {
    return c < fullC ? plenU : c == fullC ? plenLast : 0u;
  }

  VR_HD void next_stage(const vrStepPlan& P) {
    c = c == 0 ? N - 1 : c - 1;
    ++k;
    plen = stage_len(P);
  }

  VR_HD uint64_t own_offset() const { return ownBase + (uint64_t)c * ownStep; }
  VR_HD uint64_t out_offset() const { return outBase + (uint64_t)c * outStep; }
};

// The steps of stages 0 .. maxStage of every part of ring `grp`, in order:
// with maxStage the last stage that reads the input, exactly the steps that
// read the rank's own data (for prefetching it).
struct StepWalk {
  PartWalk pw;
  uint64_t unit;
  uint32_t s;
  int r, maxStage;
  bool inPart;

  VR_HD void init(int rank, int grp, int lastStage) {
    r = rank;
    maxStage = lastStage;
    unit = (uint64_t)grp;
    inPart = false;
  }

  // The next own-data step of the current part: byte offset into the rank's
  // input and length. False when the part has none left (or none is entered).
  VR_HD bool next_in_part(const vrStepPlan& P, uint64_t& off, uint32_t& len) {
    if (!inPart) return false;
    for (;;) {
      if (s < pw.plen) {
        off = pw.own_offset() + s;
        len = (uint32_t)min_u64(P.payload, pw.plen - s);
        s += (uint32_t)P.payload;
        return true;
      }
      if (pw.k >= maxStage) {
        inPart = false;
        return false;
      }
      pw.next_stage(P);
      s = 0;
    }
  }

  // Enter the ring's next part. False when the walk is over.
  VR_HD bool next_part(const vrStepPlan& P) {
    if (unit >= P.nUnits) return false;
    pw.enter(P, r, unit);
    unit += P.G;
    s = 0;
    inPart = true;
    return true;
  }

  // The next step over all the ring's parts. False when the walk is over.
  VR_HD bool next(const vrStepPlan& P, uint64_t& off, uint32_t& len) {
    for (;;) {
      if (next_in_part(P, off, len)) return true;
      if (!next_part(P)) return false;
    }
  }
};

}  // namespace vr
