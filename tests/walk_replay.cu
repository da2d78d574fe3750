// walk_replay.cu -- replays the warp rings' walk (the plan and the part/step
// walkers the kernels use, from vr_cursor.cuh) on the host for random calls,
// and checks, rank by rank:
//  * every step lies inside the rank's buffers and, unless the halves' block
//    stride is off 16 bytes (the library then takes the element-wise path),
//    starts on a 16-byte boundary (bulk copies and vector accesses);
//  * the stages that read the input read every input byte exactly once and
//    the stages that write the output write every output byte exactly once
//    (AllReduce: the whole buffer both ways; ReduceScatter: all N blocks in,
//    block r out; AllGather: the block in, all N blocks out);
//  * the own-data prefetch walk (StepWalk) yields exactly the input steps of
//    the stage walk, in the same order.
// Exit status 0 when every check holds; prints the first failure otherwise.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "vr_cursor.cuh"

using namespace vr;

namespace {

uint64_t rng_state = 0x9E3779B97F4A7C15ull;
uint64_t next_rand() {  // splitmix64
  uint64_t z = (rng_state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
uint64_t pick(uint64_t lo, uint64_t hi) { return lo + next_rand() % (hi - lo + 1); }

// Stage kinds of stage k, as the kernels assign them.
int kind_of(int coll, int N, int k) {
  if (coll == VR_COLL_REDUCESCATTER) return k == 0 ? VR_SEND : k < N - 1 ? VR_RRS : VR_RRC;
  if (coll == VR_COLL_ALLGATHER) return k == 0 ? VR_SC : k < N - 1 ? VR_RCS : VR_RECV;
  return k == 0 ? VR_SEND : k < N - 1 ? VR_RRS : k == N - 1 ? VR_RRCS
       : k < 2 * N - 2 ? VR_RCS : VR_RECV;
}

struct Step { uint64_t off; uint32_t len; };

int fail(const char* what, int trial) {
  fprintf(stderr, "trial %d: %s\n", trial, what);
  return 1;
}

}  // namespace

int main(int argc, char** argv) {
  const int trials = argc > 1 ? atoi(argv[1]) : 2000;
  for (int t = 0; t < trials; ++t) {
    const int coll = (int)pick(0, 2);
    const int N = (int)pick(2, 16);
    const uint64_t E = 1ull << pick(0, 3);
    const int nCh = (int)pick(1, 8);
    const uint64_t chunkBytes = 16 * pick(1, 4096);
    const uint64_t count = pick(1, (uint64_t)(1 << 16) / E);  // per rank, or per block
    const uint64_t payload = 256 * pick(2, 16);               // a slot's payload
    const uint64_t G = pick(1, 40);                            // rings running at once
    vrRingArgs a;
    memset(&a, 0, sizeof(a));
    a.count = count;
    a.chunkElems = chunkBytes / E;
    a.nRanks = N;
    a.nChannels = nCh;
    a.coll = coll;
    vrStepPlan P;
    plan_init(P, a, E, G, payload, payload);
    const bool ar = coll == VR_COLL_ALLREDUCE;
    const uint64_t inBytes = (coll == VR_COLL_REDUCESCATTER ? (uint64_t)N : 1) * count * E;
    const uint64_t outBytes = (coll == VR_COLL_ALLGATHER ? (uint64_t)N : 1) * count * E;
    const int lastStage = ar ? 2 * N - 2 : N - 1;
    const int lastOwnStage = coll == VR_COLL_ALLGATHER ? 0 : N - 1;
    // The halves' blocks are `count` elements apart: when that stride is not
    // a multiple of 16 bytes the library takes the element-wise path, so only
    // the other calls must start every step on a 16-byte boundary.
    const bool aligned = ar || (count * E) % 16 == 0;
    for (int r = 0; r < N; ++r) {
      std::vector<uint8_t> inCov(inBytes, 0), outCov(outBytes, 0);
      for (uint64_t ring = 0; ring < G; ++ring) {
        std::vector<Step> ownSteps;
        for (uint64_t unit = ring; unit < P.nUnits; unit += G) {
          PartWalk pw;
          pw.enter(P, r, unit);
          for (int k = 0; k <= lastStage; ++k) {
            if (k) pw.next_stage(P);
            if (!pw.plen) continue;
            const int kind = kind_of(coll, N, k);
            for (uint32_t s = 0; s < pw.plen; s += (uint32_t)P.payload) {
              const uint32_t len = (uint32_t)min_u64(P.payload, pw.plen - s);
              if (vrKindOwn(kind)) {
                const uint64_t o = pw.own_offset() + s;
                if (o + len > inBytes) return fail("input step out of bounds", t);
                if (aligned && o % 16) return fail("input step not 16-byte aligned", t);
                for (uint64_t b = o; b < o + len; ++b) ++inCov[b];
                ownSteps.push_back(Step{o, len});
              }
              if (vrKindOut(kind)) {
                const uint64_t o = pw.out_offset() + s;
                if (o + len > outBytes) return fail("output step out of bounds", t);
                if (aligned && o % 16) return fail("output step not 16-byte aligned", t);
                for (uint64_t b = o; b < o + len; ++b) ++outCov[b];
              }
            }
          }
        }
        // The prefetch walk of this ring yields the same input steps.
        StepWalk sw;
        sw.init(r, (int)ring, lastOwnStage);
        size_t i = 0;
        uint64_t off;
        uint32_t len;
        while (sw.next(P, off, len)) {
          if (i >= ownSteps.size() || ownSteps[i].off != off || ownSteps[i].len != len)
            return fail("prefetch walk differs from the stage walk", t);
          ++i;
        }
        if (i != ownSteps.size()) return fail("prefetch walk ends early", t);
      }
      for (uint64_t b = 0; b < inBytes; ++b)
        if (inCov[b] != 1) return fail("an input byte not read exactly once", t);
      for (uint64_t b = 0; b < outBytes; ++b) {
        // ReduceScatter writes block r only, into an output of one block.
        if (outCov[b] != 1) return fail("an output byte not written exactly once", t);
      }
    }
  }
  printf("ok %d\n", trials);
  return 0;
}
