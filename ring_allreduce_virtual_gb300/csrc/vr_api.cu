// vr_api.cu -- the C ABI: communicator lifetime, argument checks, the
// per-call plan (step base, FIFO reset) and the kernel launch.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <string>

#include "vr_cursor.cuh"
#include "vr_ring_walk.cuh"
#include "vr_internal.h"

namespace {

// Sentinels at both ends of the handle, like the start/end magic of ncclComm
// ("NCCL 原始碼解讀：一個 AllReduce 的 GPU 旅程", ch.2 §2.1).
constexpr uint64_t kMagic = 0x7672436f6d6d3031ull;  // "vrComm01"
// Flags in LL lines are 32 bits: the FIFO is cleared before the step counter
// could reach this value, so a stale flag never equals a live one.
constexpr uint64_t kStepWrap = 1ull << 31;

struct Comm {
  uint64_t magicStart;
  int nRanks;
  int nChannels;
  vrProto_t proto;
  size_t chunkBytes;
  int device;
  int nSMs;
  int transport;  // 0: global-memory FIFOs, 2: warp rings (one SM's shared
                  // memory), 3: warp rings over the CTAs of a cluster (1, FIFOs
                  // in distributed shared memory, is retired)
  int ringsPerCta;      // warp: rings (3: ring parts) per CTA
  int clusterCtas;      // 3: CTAs a ring spans
  int ringWarps;        // 3: ranks of a ring per CTA (the larger count, vrSplit)
  uint32_t slotBytes;
  uint32_t depth;
  uint32_t inDepth;     // warp: own-data prefetch slots
  size_t smemBytes;     // warp: dynamic shared memory per CTA
  int maxGroups;        // warp: CTAs (3: clusters) resident at once
  // Warp transports: a second FIFO geometry with one own-data slot per rank,
  // which frees room for a larger FIFO slot (so fewer, larger parts). Used for
  // a call whose parts would need more passes than rings at the default
  // geometry while it runs only a few passes (latency-bound). 0: none.
  uint32_t altSlotBytes = 0;
  size_t altSmemBytes = 0;
  int altMaxGroups = 0;
  // Warp transports: the FIFO geometry was chosen here (not set by hand), so
  // a call may also take a smaller slot (see warpGeom).
  bool autoSlot = false;
  // Warp transports: calls that fit one pass of their rings run the latency
  // kernel (vr_ring_lat.cuh); VR_LATENCY_KERNEL=0 keeps them on the general
  // kernel.
  bool latency = true;
  char* fifo;
  size_t fifoBytes;
  uint64_t* ctrl;
  size_t ctrlBytes;
  int* statusDev;
  int* statusHost;     // pinned, mapped
  int* statusHostDev;  // device alias of statusHost
  cudaEvent_t done;    // recorded after each launch
  bool pending;
  uint64_t stepBase;
  uint64_t stepWrap;  // clear the FIFO before stepBase + steps reaches this
  uint64_t timeoutNs;
  int silentRank;
  bool debug;
  // Pre-multiplied sums created on this communicator: op vrNumOps + i.
  bool preMulUsed[16];
  vrDataType_t preMulType[16];
  uint64_t preMulBits[16];
  uint64_t magicEnd;
};

std::mutex& registryMutex() {
  static std::mutex* m = new std::mutex;
  return *m;
}
std::set<Comm*>& registry() {
  static std::set<Comm*>* s = new std::set<Comm*>;
  return *s;
}

Comm* lookup(vrComm_t h) {
  Comm* c = reinterpret_cast<Comm*>(h);
  std::lock_guard<std::mutex> g(registryMutex());
  if (!c || !registry().count(c)) return nullptr;
  if (c->magicStart != kMagic || c->magicEnd != kMagic) return nullptr;
  return c;
}

int elemSize(vrDataType_t t) {
  switch (t) {
    case vrInt8: case vrUint8: return 1;
    case vrFloat16: case vrBfloat16: return 2;
    case vrFloat8e4m3: case vrFloat8e5m2: return 1;
    case vrInt32: case vrUint32: case vrFloat32: return 4;
    case vrInt64: case vrUint64: case vrFloat64: return 8;
    default: return 0;
  }
}

constexpr int kMaxPreMulOps = 16;

// A reduction as the kernels see it: the kernel's op and a sum's scaling.
struct KernelOp {
  int op;
  int scale;
  uint64_t scalar;
};

bool isFloatType(vrDataType_t t) {
  return t == vrFloat16 || t == vrBfloat16 || t == vrFloat32 || t == vrFloat64 ||
         t == vrFloat8e4m3 || t == vrFloat8e5m2;
}

// `x` rounded to the element type `t` (round to nearest even), as its bits.
uint64_t floatBits(vrDataType_t t, double x) {
  uint64_t b = 0;
  if (t == vrFloat32) {
    const float f = (float)x;
    memcpy(&b, &f, sizeof(f));
  } else if (t == vrFloat64) {
    memcpy(&b, &x, sizeof(x));
  } else if (t == vrFloat16) {
    const __half h = __double2half(x);
    memcpy(&b, &h, sizeof(h));
  } else if (t == vrFloat8e4m3 || t == vrFloat8e5m2) {  // saturating, as the ops
    b = __nv_cvt_double_to_fp8(x, __NV_SATFINITE, t == vrFloat8e4m3 ? __NV_E4M3 : __NV_E5M2);
  } else {
    const __nv_bfloat16 h = __double2bfloat16(x);
    memcpy(&b, &h, sizeof(h));
  }
  return b;
}

// Plain ops pass through; the average is the sum with 1/N pre-multiplied
// (floating types) or the sum divided by N (integer types); a pre-multiplied
// sum is the sum with its scalar ("NCCL 原始碼解讀", ch.6: hostToDevRedOp
// turns the host op into the device op). False for an unknown op or a
// pre-multiplied sum made for another type.
bool resolveOp(const Comm* c, vrRedOp_t op, vrDataType_t dtype, KernelOp* k) {
  k->op = 0;
  k->scale = VR_SCALE_NONE;
  k->scalar = 0;
  if (op >= vrSum && op <= vrMin) {
    k->op = (int)op;
    return true;
  }
  if (op == vrAvg) {
    if (isFloatType(dtype)) {
      k->scale = VR_SCALE_PREMUL;
      k->scalar = floatBits(dtype, 1.0 / (double)c->nRanks);
    } else {
      k->scale = VR_SCALE_POSTDIV;
    }
    return true;
  }
  const int i = (int)op - (int)vrNumOps;
  if (i < 0 || i >= kMaxPreMulOps || !c->preMulUsed[i] || c->preMulType[i] != dtype) return false;
  k->scale = VR_SCALE_PREMUL;
  k->scalar = c->preMulBits[i];
  return true;
}

const void* genericKernel(vrDataType_t t, int op, int proto) {
  switch (t) {
    case vrInt8: return vrGetGeneric_i8(op, proto);
    case vrUint8: return vrGetGeneric_u8(op, proto);
    case vrInt32: return vrGetGeneric_i32(op, proto);
    case vrUint32: return vrGetGeneric_u32(op, proto);
    case vrInt64: return vrGetGeneric_i64(op, proto);
    case vrUint64: return vrGetGeneric_u64(op, proto);
    case vrFloat16: return vrGetGeneric_f16(op, proto);
    case vrBfloat16: return vrGetGeneric_bf16(op, proto);
    case vrFloat8e4m3: return vrGetGeneric_e4m3(op, proto);
    case vrFloat8e5m2: return vrGetGeneric_e5m2(op, proto);
    case vrFloat32: return vrGetGeneric_f32(op, proto);
    case vrFloat64: return vrGetGeneric_f64(op, proto);
    default: return nullptr;
  }
}

const void* warpKernel(vrDataType_t t, int op, int proto, bool cluster) {
  const int cl = cluster ? 1 : 0;
  switch (t) {
    case vrInt8: return vrGetWarp_i8(op, proto, cl);
    case vrUint8: return vrGetWarp_u8(op, proto, cl);
    case vrInt32: return vrGetWarp_i32(op, proto, cl);
    case vrUint32: return vrGetWarp_u32(op, proto, cl);
    case vrInt64: return vrGetWarp_i64(op, proto, cl);
    case vrUint64: return vrGetWarp_u64(op, proto, cl);
    case vrFloat16: return vrGetWarp_f16(op, proto, cl);
    case vrBfloat16: return vrGetWarp_bf16(op, proto, cl);
    case vrFloat8e4m3: return vrGetWarp_e4m3(op, proto, cl);
    case vrFloat8e5m2: return vrGetWarp_e5m2(op, proto, cl);
    case vrFloat32: return vrGetWarp_f32(op, proto, cl);
    case vrFloat64: return vrGetWarp_f64(op, proto, cl);
    default: return nullptr;
  }
}

// The latency kernel: one-pass rings in one CTA or over a cluster, or
// (several) rings in one CTA running several passes.
const void* latKernel(vrDataType_t t, int op, int proto, bool cluster, bool multi) {
  const int cl = cluster ? 1 : multi ? 2 : 0;
  switch (t) {
    case vrInt8: return vrGetLat_i8(op, proto, cl);
    case vrUint8: return vrGetLat_u8(op, proto, cl);
    case vrInt32: return vrGetLat_i32(op, proto, cl);
    case vrUint32: return vrGetLat_u32(op, proto, cl);
    case vrInt64: return vrGetLat_i64(op, proto, cl);
    case vrUint64: return vrGetLat_u64(op, proto, cl);
    case vrFloat16: return vrGetLat_f16(op, proto, cl);
    case vrBfloat16: return vrGetLat_bf16(op, proto, cl);
    case vrFloat8e4m3: return vrGetLat_e4m3(op, proto, cl);
    case vrFloat8e5m2: return vrGetLat_e5m2(op, proto, cl);
    case vrFloat32: return vrGetLat_f32(op, proto, cl);
    case vrFloat64: return vrGetLat_f64(op, proto, cl);
    default: return nullptr;
  }
}

// Launch configuration of the warp-ring kernels: `groups` CTAs (transport
// 2) or clusters of clusterCtas CTAs (transport 3), ringsPerCta * ringWarps
// warps each.
void warpLaunchConfig(const Comm* c, cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr,
                      int groups, cudaStream_t st, size_t smem = 0, int rings = 0) {
  memset(cfg, 0, sizeof(*cfg));
  const int C = c->transport == 3 ? c->clusterCtas : 1;
  cfg->gridDim = dim3((unsigned)(groups * C));
  cfg->blockDim = dim3((unsigned)(32 * (rings ? rings : c->ringsPerCta) * c->ringWarps));
  cfg->dynamicSmemBytes = smem ? smem : c->smemBytes;
  cfg->stream = st;
  if (C > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg->attrs = attr;
    cfg->numAttrs = 1;
  }
}

const void* walkKernel(vrDataType_t t, int op) {
  switch (t) {
    case vrInt8: return vrGetWalk_i8(op);
    case vrUint8: return vrGetWalk_u8(op);
    case vrInt32: return vrGetWalk_i32(op);
    case vrUint32: return vrGetWalk_u32(op);
    case vrInt64: return vrGetWalk_i64(op);
    case vrUint64: return vrGetWalk_u64(op);
    case vrFloat16: return vrGetWalk_f16(op);
    case vrBfloat16: return vrGetWalk_bf16(op);
    case vrFloat8e4m3: return vrGetWalk_e4m3(op);
    case vrFloat8e5m2: return vrGetWalk_e5m2(op);
    case vrFloat32: return vrGetWalk_f32(op);
    case vrFloat64: return vrGetWalk_f64(op);
    default: return nullptr;
  }
}

const void* treeKernel(vrDataType_t t, int op, bool cluster) {
  const int cl = cluster ? 1 : 0;
  switch (t) {
    case vrInt8: return vrGetTree_i8(op, cl);
    case vrUint8: return vrGetTree_u8(op, cl);
    case vrInt32: return vrGetTree_i32(op, cl);
    case vrUint32: return vrGetTree_u32(op, cl);
    case vrInt64: return vrGetTree_i64(op, cl);
    case vrUint64: return vrGetTree_u64(op, cl);
    case vrFloat16: return vrGetTree_f16(op, cl);
    case vrBfloat16: return vrGetTree_bf16(op, cl);
    case vrFloat8e4m3: return vrGetTree_e4m3(op, cl);
    case vrFloat8e5m2: return vrGetTree_e5m2(op, cl);
    case vrFloat32: return vrGetTree_f32(op, cl);
    case vrFloat64: return vrGetTree_f64(op, cl);
    default: return nullptr;
  }
}

// Dynamic shared memory and cluster-size attributes of the cluster kernels,
// raised once per kernel to the largest any communicator asked for.
bool prepareClusterKernel(const void* k, size_t smem, int nRanks) {
  static std::mutex* m = new std::mutex;
  static std::map<const void*, size_t>* done = new std::map<const void*, size_t>;
  std::lock_guard<std::mutex> g(*m);
  auto it = done->find(k);
  if (it != done->end() && it->second >= smem) return true;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  (void)nRanks;
  (*done)[k] = smem;
  return true;
}

// An NVTX range around each collective entry point, like the markers at
// NCCL's API entry points ("NCCL 原始碼解讀", ch.3 §3.1 and ch.6): a profiler
// shows each call's host-side span; with no tool attached it costs a branch.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

long envLong(const char* name, long dflt) {
  const char* s = getenv(name);
  if (!s || !*s) return dflt;
  char* end = nullptr;
  long v = strtol(s, &end, 0);
  return (end && *end == 0) ? v : dflt;
}

uint64_t divUp(uint64_t a, uint64_t b) { return (a + b - 1) / b; }
uint64_t alignUp(uint64_t a, uint64_t b) { return divUp(a, b) * b; }

// Upper bound on the FIFO steps any edge of any channel makes in one call
// (channel 0 is the largest): per loop, 2(N-1) chunk transfers of at most
// ceil(chunk bytes / payload per step) steps each.
uint64_t stepsBound(const Comm* c, uint64_t count, int es) {
  const uint64_t align = 16 / (uint64_t)es;
  const uint64_t per = alignUp(divUp(count, (uint64_t)c->nChannels), align);
  const uint64_t S = per < count ? per : count;
  const uint64_t chunkElems = c->chunkBytes / (uint64_t)es;
  const uint64_t L = (uint64_t)c->nRanks * chunkElems;
  const uint64_t payload = vrPayloadPerStep(c->proto, c->slotBytes);
  const uint64_t fullLoops = S / L;
  const uint64_t rem = S - fullLoops * L;
  const uint64_t partBytes = payload * (c->depth / 2);
  // Steps of one chunk transfer: whole parts, then the steps of the last part.
  auto stepsOf = [&](uint64_t bytes) {
    return bytes / partBytes * divUp(partBytes, payload) + divUp(bytes % partBytes, payload);
  };
  uint64_t bound = fullLoops * 2 * (uint64_t)(c->nRanks - 1) * stepsOf(chunkElems * (uint64_t)es);
  if (rem) {
    const uint64_t cur = alignUp(divUp(rem, (uint64_t)c->nRanks), align);
    bound += 2 * (uint64_t)(c->nRanks - 1) * stepsOf(cur * (uint64_t)es);
  }
  return bound;
}

// Number of parts (independent ring passes) in one call: per channel, whole
// loops of chunkBytes plus the last loop's shorter chunk, cut into parts of
// half the FIFO.
uint64_t partsOf(const Comm* c, uint64_t count, int es, int coll = VR_COLL_ALLREDUCE,
                 uint32_t slotBytes = 0) {
  if (!slotBytes) slotBytes = c->slotBytes;
  const uint64_t align = 16 / (uint64_t)es;
  const uint64_t per = alignUp(divUp(count, (uint64_t)c->nChannels), align);
  const uint64_t chunkElems = c->chunkBytes / (uint64_t)es;
  const bool ar = coll == VR_COLL_ALLREDUCE;
  const uint64_t L = ar ? (uint64_t)c->nRanks * chunkElems : chunkElems;
  const uint64_t partBytes = vrPayloadPerStep(c->proto, slotBytes) * (c->depth / 2);
  auto ofChannel = [&](uint64_t S) {
    const uint64_t full = S / L, rem = S - full * L;
    uint64_t n = full * divUp(chunkElems * (uint64_t)es, partBytes);
    const uint64_t lastCur = ar ? alignUp(divUp(rem, (uint64_t)c->nRanks), align) : rem;
    if (rem) n += divUp(lastCur * (uint64_t)es, partBytes);
    return n;
  };
  const uint64_t nFull = count / per, last = count - nFull * per;
  return nFull * ofChannel(per) + (last ? ofChannel(last) : 0);
}

// A cluster of C CTAs can hold a ring (or a tree) of N ranks: 2 <= C <= 16,
// C <= N, at most 16 ranks (warps, or warp pairs for the tree) in a CTA.
bool clusterSplitOk(int N, int C) {
  return C >= 2 && C <= 16 && C <= N && divUp((uint64_t)N, (uint64_t)C) <= VR_WARP_MAX_RANKS;
}

// The CTAs of the cluster that a ring (tree) of N > 16 ranks spans: the
// smallest C that leaves at most 16 ranks in a CTA (CTAs of ceil(N / C) and
// floor(N / C) ranks), so that each SM holds as many rank warps, and each
// ring crosses as few CTA boundaries, as a split allows; 0 if none (N > 256).
int clusterCtas(int N) {
  for (int C = 2; C <= 16; ++C)
    if (clusterSplitOk(N, C)) return C;
  return 0;
}

void freeComm(Comm* c) {
  if (c->fifo) cudaFree(c->fifo);
  if (c->ctrl) cudaFree(c->ctrl);
  if (c->statusDev) cudaFree(c->statusDev);
  if (c->statusHost) cudaFreeHost(c->statusHost);
  if (c->done) cudaEventDestroy(c->done);
  c->magicStart = c->magicEnd = 0;
  delete c;
}

struct DeviceGuard {
  int prev = -1;
  bool changed = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) {
      changed = cudaSetDevice(dev) == cudaSuccess;
    }
  }
  ~DeviceGuard() {
    if (changed) cudaSetDevice(prev);
  }
};

// CTAs (transport 2) or clusters (transport 3) of one warp-ring launch:
// enough for every part to have its own ring, at most what is resident.
int warpGroups(const Comm* c, uint64_t parts, int maxGroups = 0) {
  if (!maxGroups) maxGroups = c->maxGroups;
  const uint64_t g = divUp(parts ? parts : 1, (uint64_t)c->ringsPerCta);
  return (int)(g < (uint64_t)maxGroups ? g : maxGroups);
}

// The FIFO geometry of one warp-ring call: the default; for a call that needs
// one pass, the smallest slot that still needs one; or the one-own-slot
// geometry when that takes a latency-bound call (2 or 3 passes of its rings
// one after another) to fewer passes. Results do not depend on it.
struct WarpGeom {
  uint32_t slot, inDepth;
  size_t smem;
  uint64_t parts;
  int groups;
};
WarpGeom warpGeom(const Comm* c, uint64_t count, int es, int coll) {
  WarpGeom g{c->slotBytes, c->inDepth, c->smemBytes, partsOf(c, count, es, coll), 0};
  g.groups = warpGroups(c, g.parts);
  const uint64_t rings = (uint64_t)g.groups * (uint64_t)c->ringsPerCta;
  const uint64_t passes = divUp(g.parts, rings);
  // A call that needs one pass takes the smallest slot (a multiple of 512
  // bytes) with which it still does: its bytes spread over as many rings as
  // run at once, each stage moving a shorter step.
  if (passes <= 1 && c->autoSlot) {
    const uint64_t maxRings = (uint64_t)c->maxGroups * (uint64_t)c->ringsPerCta;
    for (uint32_t s = 512; s < c->slotBytes; s += 512) {
      const uint64_t parts = partsOf(c, count, es, coll, s);
      if (parts > maxRings) continue;
      const size_t perWarp = (size_t)c->depth * s + (size_t)c->inDepth * vrOwnSlotBytes(c->proto, s) +
                             8 * (2 * (size_t)c->depth + (size_t)c->inDepth);
      return WarpGeom{s, c->inDepth, (size_t)c->ringsPerCta * (size_t)c->ringWarps * perWarp, parts,
                      warpGroups(c, parts)};
    }
    return g;
  }
  if (!c->altSlotBytes) return g;
  if (passes < 2 || passes > 3) return g;
  const uint64_t altParts = partsOf(c, count, es, coll, c->altSlotBytes);
  const int altGroups = warpGroups(c, altParts, c->altMaxGroups);
  const uint64_t altPasses = divUp(altParts, (uint64_t)altGroups * (uint64_t)c->ringsPerCta);
  if (altPasses >= passes) return g;
  return WarpGeom{c->altSlotBytes, 1, c->altSmemBytes, altParts, altGroups};
}

// One warp-ring launch of `coll` over `count` elements (per block for the
// halves) of `es` bytes, kernel for (dtype, op).
vrResult_t launchWarpRing(Comm* c, int coll, const void* const* sendbufs, void* const* recvbufs,
                          size_t count, vrDataType_t dtype, KernelOp op, int alignMask,
                          cudaStream_t st) {
  const int es = elemSize(dtype);
  vrRingArgs a;
  memset(&a, 0, sizeof(a));
  a.count = count;
  a.chunkElems = c->chunkBytes / (size_t)es;
  a.timeoutNs = c->timeoutNs;
  a.status = c->statusDev;
  a.statusHost = c->statusHostDev;
  a.nRanks = c->nRanks;
  a.nChannels = c->nChannels;
  a.alignMask = alignMask;
  a.silentRank = c->silentRank;
  const WarpGeom geom = warpGeom(c, count, es, coll);
  a.slotBytes = geom.slot;
  a.depth = c->depth;
  a.inDepth = geom.inDepth;
  a.ringsPerCta = c->ringsPerCta;
  a.ringWarps = c->ringWarps;
  a.coll = coll;
  a.scale = op.scale;
  a.scalar = op.scalar;
  for (int r = 0; r < c->nRanks; ++r) {
    a.send[r] = sendbufs[r];
    a.recv[r] = recvbufs[r];
  }
  const uint64_t parts = geom.parts;
  int groups = geom.groups;
  int rings = c->ringsPerCta;
  // A call whose parts all run at once (one part per ring, one step per
  // stage: depth 2), on 16-byte aligned buffers, with steps of at most
  // VR_LAT_PACKS packs per lane, takes the latency kernel, Simple and LL. It
  // keeps as many own-data steps in flight as the shared memory of the
  // default geometry holds, up to all of the part's own-data stages. A Simple
  // call of several passes on rings inside one CTA (transport 2) takes it too,
  // in the default geometry: there its shorter stage gives each rank warp a
  // shorter period than the general kernel's (16 x 1 GiB fp32: 0.975 against
  // 0.948 of the measured copy peak). On a cluster, and for LL, the general
  // kernel measured faster at several passes.
  const uint64_t stepPayload = vrPayloadPerStep(c->proto, geom.slot);
  const bool onePass = parts <= (uint64_t)groups * (uint64_t)c->ringsPerCta;
  const bool lat = c->latency && c->proto != vrProtoLL128 && c->depth == 2 &&
                   (alignMask & 15) == 0 && stepPayload <= 32u * 16u * VR_LAT_PACKS &&
                   (onePass || (c->proto == vrProtoSimple && c->transport == 2));
  size_t smem = geom.smem;
  if (lat && onePass) {
    // As few rings per CTA (cluster) as keep every part in its own ring: the
    // rank warps of a CTA share its four schedulers, so a CTA with fewer of
    // them runs each stage sooner. The geometry's own groups are resident at
    // once, so these (at most as many CTAs of fewer warps) are too.
    const int avail = geom.inDepth == 1 && c->altMaxGroups ? c->altMaxGroups : c->maxGroups;
    rings = (int)((parts + (uint64_t)avail - 1) / (uint64_t)avail);
    if (rings < 1) rings = 1;
    if (rings > c->ringsPerCta) rings = c->ringsPerCta;
    groups = (int)((parts + (uint64_t)rings - 1) / (uint64_t)rings);
    a.ringsPerCta = rings;
    const size_t warps = (size_t)rings * (size_t)c->ringWarps;
    const size_t fixed = (size_t)c->depth * geom.slot + 8 * 2 * (size_t)c->depth;
    const size_t perOwn = (size_t)vrOwnSlotBytes(c->proto, geom.slot) + 8;
    const size_t budget = c->smemBytes > smem ? c->smemBytes : smem;
    const uint32_t ownStages = coll == VR_COLL_ALLGATHER ? 1u : (uint32_t)c->nRanks;
    uint32_t di = (uint32_t)((budget / warps - fixed) / perOwn);
    if (di > ownStages) di = ownStages;
    if (di < 1) di = 1;
    a.inDepth = di;
    smem = warps * (fixed + di * perOwn);
  }
  const void* kernel = lat ? latKernel(dtype, op.op, (int)c->proto, c->transport == 3, !onePass)
                           : warpKernel(dtype, op.op, (int)c->proto, c->transport == 3);
  if (!kernel) return vrInternalError;
  if (!prepareClusterKernel(kernel, smem, c->nRanks)) return vrCudaError;
  // The walk every CTA follows: computed here once, read from parameter space.
  const uint64_t payload = vrPayloadPerStep(c->proto, geom.slot);
  vr::plan_init(a.plan, a, (uint64_t)es, (uint64_t)groups * (uint64_t)rings,
                payload * (c->depth / 2), payload);
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  warpLaunchConfig(c, &cfg, attr, groups, st, smem, rings);
  void* args[] = {&a};
  if (cudaLaunchKernelExC(&cfg, kernel, args) != cudaSuccess) {
    cudaGetLastError();
    return vrCudaError;
  }
  if (cudaEventRecord(c->done, st) != cudaSuccess) return vrCudaError;
  c->pending = true;
  if (c->debug)
    fprintf(stderr,
            "[vr] warp ring%s: coll %d count %zu dtype %d op %d: %d groups, %llu parts, slot %u, "
            "inDepth %u\n",
            lat ? " (latency kernel)" : "", coll, count, (int)dtype, op.op, groups,
            (unsigned long long)parts, geom.slot, a.inDepth);
  return vrSuccess;
}

// Checks shared by ReduceScatter and AllGather: a live communicator on the
// warp transport, known type and op, no sticky timeout, and rank buffers of
// `sendElems` / `recvElems` elements aligned to the element size.
vrResult_t checkHalf(Comm* c, const void* const* sendbufs, void* const* recvbufs, int es,
                     int* alignMask) {
  *alignMask = 0;
  for (int r = 0; r < c->nRanks; ++r) {
    const uintptr_t s = (uintptr_t)sendbufs[r], d = (uintptr_t)recvbufs[r];
    if (!s || !d || s % es || d % es) return vrInvalidArgument;
    *alignMask |= (int)((s | d) & 15);
  }
  return vrSuccess;
}

}  // namespace

// One ring-walk fold launch (the calibration kernel; also a one-rank
// pre-multiplied sum).
vrResult_t launchWalk(Comm* c, const void* const* sendbufs, void* const* recvbufs, size_t count,
                      vrDataType_t dtype, KernelOp kop, int alignMask, cudaStream_t st) {
  const int es = elemSize(dtype);
  vrRingArgs a;
  memset(&a, 0, sizeof(a));
  a.count = count;
  a.chunkElems = c->chunkBytes / (size_t)es;
  a.nRanks = c->nRanks;
  a.nChannels = c->nChannels;
  a.alignMask = alignMask;
  a.coll = VR_COLL_ALLREDUCE;
  a.scale = kop.scale;
  a.scalar = kop.scalar;
  for (int r = 0; r < c->nRanks; ++r) {
    a.send[r] = sendbufs[r];
    a.recv[r] = recvbufs[r];
  }
  // The chunk map of the AllReduce (parts play no role here).
  vr::plan_init(a.plan, a, (uint64_t)es, 1, c->chunkBytes, c->chunkBytes);
  vr::walk_plan(a.plan, c->nSMs);
  const void* kernel = walkKernel(dtype, kop.op);
  if (!kernel) return vrInternalError;
  const uint64_t units = vr::walk_units(a.plan);
  const uint64_t maxCtas = (uint64_t)c->nSMs * 8;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)(units < maxCtas ? (units ? units : 1) : maxCtas));
  cfg.blockDim = dim3(vr::kWalkThreads);
  cfg.stream = st;
  void* args[] = {&a};
  if (cudaLaunchKernelExC(&cfg, kernel, args) != cudaSuccess) {
    cudaGetLastError();
    return vrCudaError;
  }
  return vrSuccess;
}

extern "C" {

const char* vrGetErrorString(vrResult_t r) {
  switch (r) {
    case vrSuccess: return "no error";
    case vrInvalidArgument: return "invalid argument";
    case vrInvalidUsage: return "invalid usage";
    case vrCudaError: return "CUDA error";
    case vrInternalError: return "internal error";
    case vrTimeout: return "a device-side wait timed out";
    default: return "unknown result code";
  }
}

vrResult_t vrCommCreate(vrComm_t* comm, int nRanks, int nChannels, vrProto_t proto,
                        size_t chunkBytes) {
  if (!comm || nRanks < 1 || nRanks > VR_MAX_RANKS || nChannels < 1 ||
      nChannels > VR_MAX_CHANNELS || proto < vrProtoSimple || proto >= vrNumProtos ||
      chunkBytes < 16 || chunkBytes % 16 != 0)
    return vrInvalidArgument;

  Comm* c = new Comm();
  c->magicStart = c->magicEnd = kMagic;
  c->nRanks = nRanks;
  c->nChannels = nChannels;
  c->proto = proto;
  c->chunkBytes = chunkBytes;
  c->debug = envLong("VR_DEBUG", 0) != 0;
  c->silentRank = (int)envLong("VR_DEBUG_SILENT_RANK", -1);
  c->latency = envLong("VR_LATENCY_KERNEL", 1) != 0;
  c->timeoutNs = (uint64_t)envLong("VR_TIMEOUT_MS", 10000) * 1000000ull;
  // Test only: a lower wrap point exercises the FIFO reset without 2^31 steps.
  c->stepWrap = (uint64_t)envLong("VR_DEBUG_STEP_WRAP", (long)kStepWrap);
  if (c->stepWrap < 1 || c->stepWrap > kStepWrap) c->stepWrap = kStepWrap;
  if (cudaGetDevice(&c->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->nSMs, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess) {
    delete c;
    return vrCudaError;
  }
  c->transport = 0;
  c->slotBytes = (uint32_t)envLong("VR_FIFO_SLOT_BYTES", 16384);
  c->depth = (uint32_t)envLong("VR_FIFO_DEPTH", 4);
  c->inDepth = (uint32_t)envLong("VR_FIFO_IN_DEPTH", 4);
  // Slots are whole pairs of 128-byte lines, so every protocol's payload per
  // step (LL128: 120 bytes a line) is a multiple of 16 bytes.
  if (c->slotBytes < 1024 || c->slotBytes > (1u << 20) || c->slotBytes % 256 != 0 ||
      c->depth < 2 || c->depth > 64 || c->inDepth < 1 || c->inDepth > 64) {
    delete c;
    return vrInvalidArgument;
  }

  // Transport: warp rings in one SM's shared memory (2..16 ranks) or over the
  // CTAs of a cluster (more ranks); FIFOs in global memory when asked for
  // (VR_TRANSPORT=global) or when no warp ring fits the device.
  const char* tenv = getenv("VR_TRANSPORT");
  const std::string tsel = tenv && *tenv ? tenv : "auto";
  const bool warpOk = nRanks >= 2 && nRanks <= VR_WARP_MAX_RANKS;
  const bool warpClusterOk = nRanks >= 2 && (tsel == "warpcluster" || !warpOk);
  if (tsel != "auto" && tsel != "global" && tsel != "warp" && tsel != "warpcluster") {
    delete c;
    return vrInvalidArgument;
  }
  if ((tsel == "warp" && !warpOk) || (tsel == "warpcluster" && nRanks < 2)) {
    delete c;
    return vrInvalidUsage;
  }
  int optinSmem = 0;
  if (cudaDeviceGetAttribute(&optinSmem, cudaDevAttrMaxSharedMemoryPerBlockOptin, c->device) !=
      cudaSuccess) {
    delete c;
    return vrCudaError;
  }
  // Rings of warps: a whole ring in one CTA for 2..16 ranks; else a ring over
  // the C CTAs of a cluster (clusterCtas), ceil(N / C) or floor(N / C) ranks
  // per CTA (vrSplit), with C from VR_CLUSTER_CTAS or clusterCtas().
  int C = 1;
  if (warpClusterOk) {
    const long want = envLong("VR_CLUSTER_CTAS", 0);
    C = want ? (clusterSplitOk(nRanks, (int)want) ? (int)want : 0) : clusterCtas(nRanks);
    if (!C && tsel == "warpcluster") {
      delete c;
      return vrInvalidUsage;
    }
  }
  const bool useWarp = warpOk && (tsel == "auto" || tsel == "warp");
  const bool useWarpCluster = C >= 2 && (tsel == "warpcluster" || (tsel == "auto" && !warpOk));
  if (useWarp || useWarpCluster) {
    // W warps of each of R rings per CTA, 16 warps at most. Unless set, the
    // depths are 2 and 2 (parts of one slot) and the slot is the largest
    // multiple of 512 bytes that fits them in the shared memory of one SM.
    if (!getenv("VR_FIFO_DEPTH")) c->depth = 2;
    if (!getenv("VR_FIFO_IN_DEPTH")) c->inDepth = 2;
    const int W = useWarpCluster ? (int)divUp((uint64_t)nRanks, (uint64_t)C) : nRanks;
    int R = VR_WARP_MAX_RANKS / W;
    const size_t barsPerWarp = 8 * (2 * (size_t)c->depth + (size_t)c->inDepth);
    // Per warp: depth FIFO slots, inDepth own-data slots of one step's
    // payload, and the barriers; the kernel's static shared memory comes on
    // top.
    auto perWarp = [&](uint32_t slot) {
      return (size_t)c->depth * slot + (size_t)c->inDepth * vrOwnSlotBytes(proto, slot) +
             barsPerWarp;
    };
    const void* k = warpKernel(vrFloat32, 0, (int)proto, useWarpCluster);
    cudaFuncAttributes fa;
    size_t staticSmem = 4096;
    if (cudaFuncGetAttributes(&fa, k) == cudaSuccess)
      staticSmem = fa.sharedSizeBytes;
    else
      cudaGetLastError();
    if (!getenv("VR_FIFO_SLOT_BYTES")) {
      const size_t warps = (size_t)R * (size_t)W;
      uint32_t slot = 512;
      while (slot < 16384 && warps * perWarp(slot + 512) + staticSmem <= (size_t)optinSmem)
        slot += 512;
      c->slotBytes = slot;
    } else {
      // A slot set by hand: as many rings per CTA as its FIFOs leave room for.
      while (R > 1 &&
             (size_t)R * W * perWarp(c->slotBytes) + staticSmem > (size_t)optinSmem)
        --R;
    }
    c->smemBytes = (size_t)R * W * perWarp(c->slotBytes);
    c->transport = useWarpCluster ? 3 : 2;
    c->ringsPerCta = R;
    c->ringWarps = W;
    c->clusterCtas = useWarpCluster ? C : 1;
    int groups = 0;
    if (c->slotBytes >= 512 && c->smemBytes + staticSmem <= (size_t)optinSmem &&
        prepareClusterKernel(k, c->smemBytes, nRanks)) {
      if (useWarpCluster) {
        cudaLaunchConfig_t cfg;
        cudaLaunchAttribute attr[1];
        warpLaunchConfig(c, &cfg, attr, c->nSMs, 0);
        if (cudaOccupancyMaxActiveClusters(&groups, k, &cfg) != cudaSuccess) {
          cudaGetLastError();
          groups = 0;
        }
      } else {
        groups = c->nSMs;
      }
    }
    if (groups > 0) {
      c->maxGroups = groups;
      c->autoSlot = !getenv("VR_FIFO_SLOT_BYTES") && !getenv("VR_FIFO_IN_DEPTH") &&
                    !getenv("VR_FIFO_DEPTH");
      // The one-own-slot geometry (Comm::altSlotBytes): the largest slot that
      // fits with one own-data slot per rank, unless the FIFO geometry was
      // set by hand.
      if (!getenv("VR_FIFO_SLOT_BYTES") && !getenv("VR_FIFO_IN_DEPTH") &&
          !getenv("VR_FIFO_DEPTH")) {
        const size_t warps = (size_t)R * (size_t)W;
        const size_t bars1 = 8 * (2 * (size_t)c->depth + 1);
        auto perWarp1 = [&](uint32_t slot) {
          return (size_t)c->depth * slot + vrOwnSlotBytes(proto, slot) + bars1;
        };
        uint32_t slot = c->slotBytes;
        while (slot < 16384 && warps * perWarp1(slot + 256) + staticSmem <= (size_t)optinSmem)
          slot += 256;
        if (slot > c->slotBytes) {
          const size_t smem = warps * perWarp1(slot);
          int g = 0;
          if (prepareClusterKernel(k, smem, nRanks)) {
            if (useWarpCluster) {
              cudaLaunchConfig_t cfg;
              cudaLaunchAttribute attr[1];
              warpLaunchConfig(c, &cfg, attr, c->nSMs, 0, smem);
              if (cudaOccupancyMaxActiveClusters(&g, k, &cfg) != cudaSuccess) {
                cudaGetLastError();
                g = 0;
              }
            } else {
              g = c->nSMs;
            }
          }
          if (g > 0) {
            c->altSlotBytes = slot;
            c->altSmemBytes = smem;
            c->altMaxGroups = g;
          }
        }
      }
    } else if (tsel == "warp" || tsel == "warpcluster") {
      delete c;
      return vrInvalidUsage;
    } else {
      c->transport = 0;
      c->slotBytes = (uint32_t)envLong("VR_FIFO_SLOT_BYTES", 16384);
      c->depth = (uint32_t)envLong("VR_FIFO_DEPTH", 4);
      c->inDepth = (uint32_t)envLong("VR_FIFO_IN_DEPTH", 4);
    }
  }
  // Global FIFOs: every rank of every channel must be resident at once.
  if (nRanks > 1 && c->transport == 0) {
    int perSM = 0;
    const void* k = genericKernel(vrFloat32, 0, proto);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&perSM, k, VR_GENERIC_THREADS, 0) !=
        cudaSuccess) {
      delete c;
      return vrCudaError;
    }
    if ((long)perSM * c->nSMs < (long)nRanks * nChannels) {
      delete c;
      return vrInvalidUsage;
    }
  }

  const size_t edges = c->transport == 0 ? (size_t)nChannels * (size_t)nRanks : 1;
  c->fifoBytes = edges * c->depth * c->slotBytes;
  c->ctrlBytes = edges * VR_CTRL_WORDS_PER_EDGE * sizeof(uint64_t);
  bool ok = cudaMalloc(&c->fifo, c->fifoBytes) == cudaSuccess &&
            cudaMalloc(&c->ctrl, c->ctrlBytes) == cudaSuccess &&
            cudaMalloc(&c->statusDev, sizeof(int)) == cudaSuccess &&
            cudaHostAlloc(&c->statusHost, sizeof(int), cudaHostAllocMapped) == cudaSuccess &&
            cudaHostGetDevicePointer(&c->statusHostDev, c->statusHost, 0) == cudaSuccess &&
            cudaEventCreateWithFlags(&c->done, cudaEventDisableTiming) == cudaSuccess &&
            cudaMemset(c->fifo, 0, c->fifoBytes) == cudaSuccess &&
            cudaMemset(c->ctrl, 0, c->ctrlBytes) == cudaSuccess &&
            cudaMemset(c->statusDev, 0, sizeof(int)) == cudaSuccess &&
            cudaDeviceSynchronize() == cudaSuccess;
  if (!ok) {
    freeComm(c);
    return vrCudaError;
  }
  *c->statusHost = VR_STATUS_OK;
  if (c->debug)
    fprintf(stderr,
            "[vr] comm %p: nRanks %d nChannels %d proto %d chunkBytes %zu transport %d slot %u "
            "depth %u inDepth %u fifo %zu B ctrl %zu B smem %zu B groups %d rings/CTA %d "
            "CTAs/ring %d; one-own-slot slot %u smem %zu B groups %d\n",
            (void*)c, nRanks, nChannels, (int)proto, chunkBytes, c->transport, c->slotBytes,
            c->depth, c->inDepth, c->fifoBytes, c->ctrlBytes, c->smemBytes, c->maxGroups,
            c->ringsPerCta, c->clusterCtas, c->altSlotBytes, c->altSmemBytes, c->altMaxGroups);
  {
    std::lock_guard<std::mutex> g(registryMutex());
    registry().insert(c);
  }
  *comm = reinterpret_cast<vrComm_t>(c);
  return vrSuccess;
}

vrResult_t vrAllReduce(vrComm_t comm, const void* const* sendbufs, void* const* recvbufs,
                       size_t count, vrDataType_t dtype, vrRedOp_t op, void* stream) {
  NvtxRange range("vrAllReduce");
  Comm* c = lookup(comm);
  if (!c) return vrInvalidArgument;
  const int es = elemSize(dtype);
  KernelOp kop;
  if (!es || !resolveOp(c, op, dtype, &kop)) return vrInvalidArgument;
  if (*(volatile int*)c->statusHost != VR_STATUS_OK) return vrTimeout;
  // Zero elements: nothing to reduce; the buffers may be empty (NULL) ones
  // ("NCCL 原始碼解讀", ch.6: count 0 returns success before any work).
  if (count == 0) return vrSuccess;
  if (!sendbufs || !recvbufs) return vrInvalidArgument;
  int alignMask = 0;
  for (int r = 0; r < c->nRanks; ++r) {
    const uintptr_t s = (uintptr_t)sendbufs[r], d = (uintptr_t)recvbufs[r];
    if (!s || !d || s % es || d % es) return vrInvalidArgument;
    alignMask |= (int)((s | d) & 15);
  }
  DeviceGuard guard(c->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  if (c->nRanks == 1) {  // one rank: the result is its own buffer (scaled)
    if (kop.scale == VR_SCALE_PREMUL)
      return launchWalk(c, sendbufs, recvbufs, count, dtype, kop, alignMask, st);
    if (sendbufs[0] != recvbufs[0] &&
        cudaMemcpyAsync(recvbufs[0], sendbufs[0], count * (size_t)es, cudaMemcpyDeviceToDevice,
                        st) != cudaSuccess)
      return vrCudaError;
    return vrSuccess;
  }

  if (c->transport == 2 || c->transport == 3)
    return launchWarpRing(c, VR_COLL_ALLREDUCE, sendbufs, recvbufs, count, dtype, kop, alignMask,
                          st);
  // The average and pre-multiplied sums run on the warp rings only.
  if (kop.scale != VR_SCALE_NONE) return vrInvalidUsage;
  const uint64_t bound = stepsBound(c, count, es);
  if (c->stepBase + bound >= c->stepWrap) {
    if (bound >= kStepWrap) return vrInvalidUsage;
    if (cudaMemsetAsync(c->fifo, 0, c->fifoBytes, st) != cudaSuccess ||
        cudaMemsetAsync(c->ctrl, 0, c->ctrlBytes, st) != cudaSuccess)
      return vrCudaError;
    c->stepBase = 0;
  }

  vrRingArgs a;
  memset(&a, 0, sizeof(a));
  a.count = count;
  a.chunkElems = c->chunkBytes / (size_t)es;
  a.stepBase = c->stepBase;
  a.timeoutNs = c->timeoutNs;
  a.fifo = c->fifo;
  a.ctrl = c->ctrl;
  a.status = c->statusDev;
  a.statusHost = c->statusHostDev;
  a.nRanks = c->nRanks;
  a.nChannels = c->nChannels;
  a.alignMask = alignMask;
  a.silentRank = c->silentRank;
  a.slotBytes = c->slotBytes;
  a.depth = c->depth;
  for (int r = 0; r < c->nRanks; ++r) {
    a.send[r] = sendbufs[r];
    a.recv[r] = recvbufs[r];
  }

  const void* kernel = genericKernel(dtype, kop.op, (int)c->proto);
  if (!kernel) return vrInternalError;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)(c->nChannels * c->nRanks));
  cfg.blockDim = dim3(VR_GENERIC_THREADS);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&a};
  cudaError_t e = cudaLaunchKernelExC(&cfg, kernel, args);
  if (e == cudaErrorCooperativeLaunchTooLarge) {
    cudaGetLastError();
    return vrInvalidUsage;
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return vrCudaError;
  }
  if (cudaEventRecord(c->done, st) != cudaSuccess) return vrCudaError;
  c->pending = true;
  if (c->debug)
    fprintf(stderr, "[vr] allreduce count %zu dtype %d op %d: grid %d stepBase %llu bound %llu\n",
            count, (int)dtype, (int)op, c->nChannels * c->nRanks,
            (unsigned long long)c->stepBase, (unsigned long long)bound);
  c->stepBase += bound;
  return vrSuccess;
}

vrResult_t vrReduceScatter(vrComm_t comm, const void* const* sendbufs, void* const* recvbufs,
                           size_t recvcount, vrDataType_t dtype, vrRedOp_t op, void* stream) {
  NvtxRange range("vrReduceScatter");
  Comm* c = lookup(comm);
  if (!c) return vrInvalidArgument;
  const int es = elemSize(dtype);
  KernelOp kop;
  if (!es || !resolveOp(c, op, dtype, &kop)) return vrInvalidArgument;
  if (*(volatile int*)c->statusHost != VR_STATUS_OK) return vrTimeout;
  if (recvcount == 0) return vrSuccess;
  if (!sendbufs || !recvbufs) return vrInvalidArgument;
  int alignMask = 0;
  vrResult_t res = checkHalf(c, sendbufs, recvbufs, es, &alignMask);
  if (res != vrSuccess) return res;
  DeviceGuard guard(c->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (c->nRanks == 1) {  // one rank: its own block (scaled)
    if (kop.scale == VR_SCALE_PREMUL)
      return launchWalk(c, sendbufs, recvbufs, recvcount, dtype, kop, alignMask, st);
    if (sendbufs[0] != recvbufs[0] &&
        cudaMemcpyAsync(recvbufs[0], sendbufs[0], recvcount * (size_t)es, cudaMemcpyDeviceToDevice,
                        st) != cudaSuccess)
      return vrCudaError;
    return vrSuccess;
  }
  if (c->transport != 2 && c->transport != 3) return vrInvalidUsage;
  // Block b of an input starts b * recvcount elements in: the vector paths
  // (bulk copies, 16-byte accesses) need that stride 16-byte aligned too.
  alignMask |= (int)((recvcount * (size_t)es) & 15);
  return launchWarpRing(c, VR_COLL_REDUCESCATTER, sendbufs, recvbufs, recvcount, dtype, kop,
                        alignMask, st);
}

vrResult_t vrAllGather(vrComm_t comm, const void* const* sendbufs, void* const* recvbufs,
                       size_t sendcount, vrDataType_t dtype, void* stream) {
  NvtxRange range("vrAllGather");
  Comm* c = lookup(comm);
  if (!c) return vrInvalidArgument;
  const int es = elemSize(dtype);
  if (!es) return vrInvalidArgument;
  if (*(volatile int*)c->statusHost != VR_STATUS_OK) return vrTimeout;
  if (sendcount == 0) return vrSuccess;
  if (!sendbufs || !recvbufs) return vrInvalidArgument;
  int alignMask = 0;
  vrResult_t res = checkHalf(c, sendbufs, recvbufs, es, &alignMask);
  if (res != vrSuccess) return res;
  DeviceGuard guard(c->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (c->nRanks == 1) {
    if (sendbufs[0] != recvbufs[0] &&
        cudaMemcpyAsync(recvbufs[0], sendbufs[0], sendcount * (size_t)es, cudaMemcpyDeviceToDevice,
                        st) != cudaSuccess)
      return vrCudaError;
    return vrSuccess;
  }
  if (c->transport != 2 && c->transport != 3) return vrInvalidUsage;
  // Block b of an output starts b * sendcount elements in: the vector paths
  // need that stride 16-byte aligned too. A copy: moved as bytes whatever the
  // element type.
  alignMask |= (int)((sendcount * (size_t)es) & 15);
  return launchWarpRing(c, VR_COLL_ALLGATHER, sendbufs, recvbufs, sendcount * (size_t)es, vrUint8,
                        KernelOp{0, VR_SCALE_NONE, 0}, alignMask, st);
}

vrResult_t vrAllReduceTree(vrComm_t comm, const void* const* sendbufs, void* const* recvbufs,
                           size_t count, vrDataType_t dtype, vrRedOp_t op, void* stream) {
  NvtxRange range("vrAllReduceTree");
  Comm* c = lookup(comm);
  if (!c) return vrInvalidArgument;
  const int es = elemSize(dtype);
  KernelOp kop;
  if (!es || !resolveOp(c, op, dtype, &kop)) return vrInvalidArgument;
  if (*(volatile int*)c->statusHost != VR_STATUS_OK) return vrTimeout;
  if (count == 0) return vrSuccess;
  if (!sendbufs || !recvbufs) return vrInvalidArgument;
  int alignMask = 0;
  for (int r = 0; r < c->nRanks; ++r) {
    const uintptr_t s = (uintptr_t)sendbufs[r], d = (uintptr_t)recvbufs[r];
    if (!s || !d || s % es || d % es) return vrInvalidArgument;
    alignMask |= (int)((s | d) & 15);
  }
  DeviceGuard guard(c->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int N = c->nRanks;
  if (N == 1) {  // one rank: the result is its own buffer (scaled)
    if (kop.scale == VR_SCALE_PREMUL)
      return launchWalk(c, sendbufs, recvbufs, count, dtype, kop, alignMask, st);
    if (sendbufs[0] != recvbufs[0] &&
        cudaMemcpyAsync(recvbufs[0], sendbufs[0], count * (size_t)es, cudaMemcpyDeviceToDevice,
                        st) != cudaSuccess)
      return vrCudaError;
    return vrSuccess;
  }
  // Two warps per rank: a tree of up to 16 ranks in one CTA; a larger one over
  // the C CTAs of a cluster, ceil(N / C) or floor(N / C) ranks each (vrSplit;
  // C from clusterCtas(), or VR_CLUSTER_CTAS, which also splits a small tree
  // for testing).
  int C = 1;
  const long want = envLong("VR_CLUSTER_CTAS", 0);
  if (want) {
    if (want == 1 ? N > VR_WARP_MAX_RANKS : !clusterSplitOk(N, (int)want)) return vrInvalidUsage;
    C = (int)want;
  } else if (N > VR_WARP_MAX_RANKS) {
    C = clusterCtas(N);
    if (!C) return vrInvalidUsage;
  }
  const bool cl = C > 1;
  const int W = (int)divUp((uint64_t)N, (uint64_t)C);  // the larger count
  int optin = 0;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, c->device) !=
      cudaSuccess)
    return vrCudaError;
  // Three FIFOs of depth 2 and two own-data slots per rank; the slot is the
  // largest multiple of 256 bytes (at most 16 KiB) that fits them and their
  // barriers in one SM.
  const uint32_t D = 2, DI = 2;
  auto smemOf = [&](uint32_t slot) {
    return (size_t)W * ((3 * D + DI) * slot + 8 * (6 * D + DI));
  };
  uint32_t slot = 256;
  while (slot < 16384 && smemOf(slot + 256) <= (size_t)optin) slot += 256;
  const size_t smem = smemOf(slot);
  const void* kernel = treeKernel(dtype, kop.op, cl);
  if (!kernel) return vrInternalError;
  if (!prepareClusterKernel(kernel, smem, N)) return vrCudaError;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  memset(&cfg, 0, sizeof(cfg));
  cfg.blockDim = dim3((unsigned)(64 * W));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  int groups = c->nSMs;  // CTAs (clusters) resident at once
  if (cl) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3((unsigned)(c->nSMs / C * C));
    if (cudaOccupancyMaxActiveClusters(&groups, kernel, &cfg) != cudaSuccess) {
      cudaGetLastError();
      return vrCudaError;
    }
    if (groups < 2) return vrInvalidUsage;
  }
  // Pieces of one slot per rank in each tree's half; as many CTAs (clusters)
  // per tree as the larger half has pieces, at most half of those resident.
  const uint64_t pieceElems = slot / (uint32_t)es;
  const uint64_t split = alignUp(divUp(count, 2), 16 / (uint64_t)es) < count
                             ? alignUp(divUp(count, 2), 16 / (uint64_t)es) : count;
  const uint64_t pieces = divUp(split, pieceElems);
  const uint64_t perTree = pieces < (uint64_t)(groups / 2) ? pieces : (uint64_t)(groups / 2);
  vrRingArgs a;
  memset(&a, 0, sizeof(a));
  a.count = count;
  a.timeoutNs = c->timeoutNs;
  a.status = c->statusDev;
  a.statusHost = c->statusHostDev;
  a.nRanks = N;
  a.ringWarps = W;
  a.alignMask = alignMask;
  a.silentRank = c->silentRank;
  a.slotBytes = slot;
  a.depth = D;
  a.inDepth = DI;
  a.scale = kop.scale;
  a.scalar = kop.scalar;
  for (int r = 0; r < N; ++r) {
    a.send[r] = sendbufs[r];
    a.recv[r] = recvbufs[r];
  }
  cfg.gridDim = dim3((unsigned)(2 * (perTree ? perTree : 1) * C));
  void* args[] = {&a};
  if (cudaLaunchKernelExC(&cfg, kernel, args) != cudaSuccess) {
    cudaGetLastError();
    return vrCudaError;
  }
  if (cudaEventRecord(c->done, st) != cudaSuccess) return vrCudaError;
  c->pending = true;
  return vrSuccess;
}

vrResult_t vrRingWalk(vrComm_t comm, const void* const* sendbufs, void* const* recvbufs,
                      size_t count, vrDataType_t dtype, vrRedOp_t op, void* stream) {
  Comm* c = lookup(comm);
  if (!c) return vrInvalidArgument;
  const int es = elemSize(dtype);
  KernelOp kop;
  if (!es || !resolveOp(c, op, dtype, &kop)) return vrInvalidArgument;
  if (count == 0) return vrSuccess;
  if (!sendbufs || !recvbufs) return vrInvalidArgument;
  int alignMask = 0;
  for (int r = 0; r < c->nRanks; ++r) {
    const uintptr_t s = (uintptr_t)sendbufs[r], d = (uintptr_t)recvbufs[r];
    if (!s || !d || s % es || d % es) return vrInvalidArgument;
    alignMask |= (int)((s | d) & 15);
  }
  DeviceGuard guard(c->device);
  return launchWalk(c, sendbufs, recvbufs, count, dtype, kop, alignMask,
                    static_cast<cudaStream_t>(stream));
}

vrResult_t vrRedOpCreatePreMulSum(vrRedOp_t* op, const void* scalar, vrDataType_t dtype,
                                  vrComm_t comm) {
  Comm* c = lookup(comm);
  const int es = elemSize(dtype);
  if (!c || !op || !scalar || !es) return vrInvalidArgument;
  for (int i = 0; i < kMaxPreMulOps; ++i) {
    if (c->preMulUsed[i]) continue;
    c->preMulUsed[i] = true;
    c->preMulType[i] = dtype;
    c->preMulBits[i] = 0;
    memcpy(&c->preMulBits[i], scalar, (size_t)es);
    *op = (vrRedOp_t)((int)vrNumOps + i);
    return vrSuccess;
  }
  return vrInvalidUsage;
}

vrResult_t vrRedOpDestroy(vrRedOp_t op, vrComm_t comm) {
  Comm* c = lookup(comm);
  const int i = (int)op - (int)vrNumOps;
  if (!c || i < 0 || i >= kMaxPreMulOps || !c->preMulUsed[i]) return vrInvalidArgument;
  c->preMulUsed[i] = false;
  return vrSuccess;
}

vrResult_t vrCommDestroy(vrComm_t comm) {
  Comm* c = lookup(comm);
  if (!c) return vrInvalidArgument;
  {
    std::lock_guard<std::mutex> g(registryMutex());
    registry().erase(c);
  }
  vrResult_t res = vrSuccess;
  {
    DeviceGuard guard(c->device);
    if (c->pending && cudaEventSynchronize(c->done) != cudaSuccess) res = vrCudaError;
    freeComm(c);
  }
  return res;
}

vrResult_t vrCommGetAsyncError(vrComm_t comm, vrResult_t* asyncErr) {
  Comm* c = lookup(comm);
  if (!c || !asyncErr) return vrInvalidArgument;
  *asyncErr = *(volatile int*)c->statusHost == VR_STATUS_OK ? vrSuccess : vrTimeout;
  return vrSuccess;
}

vrResult_t vrCommSetTimeout(vrComm_t comm, uint64_t timeoutMs) {
  Comm* c = lookup(comm);
  if (!c || timeoutMs < 1 || timeoutMs > 3600ull * 1000ull) return vrInvalidArgument;
  c->timeoutNs = timeoutMs * 1000000ull;
  return vrSuccess;
}

vrResult_t vrCommGetInfo(vrComm_t comm, int* transport, int* slotBytes, int* depth,
                         size_t* deviceBytes) {
  Comm* c = lookup(comm);
  if (!c) return vrInvalidArgument;
  if (transport) *transport = c->transport;
  if (slotBytes) *slotBytes = (int)c->slotBytes;
  if (depth) *depth = (int)c->depth;
  if (deviceBytes) *deviceBytes = c->fifoBytes + c->ctrlBytes + sizeof(int);
  return vrSuccess;
}

vrResult_t vrCommGetPlan(vrComm_t comm, size_t count, vrDataType_t dtype, size_t* parts,
                         int* rings) {
  Comm* c = lookup(comm);
  if (!c) return vrInvalidArgument;
  const int es = elemSize(dtype);
  if (!es) return vrInvalidArgument;
  uint64_t p = count ? partsOf(c, count, es) : 0;
  int g = 0;
  if (c->nRanks == 1 || count == 0) {
    g = 0;
  } else if (c->transport == 2 || c->transport == 3) {
    const WarpGeom geom = warpGeom(c, count, es, VR_COLL_ALLREDUCE);
    p = geom.parts;
    g = geom.groups * c->ringsPerCta;
  } else {
    g = c->nChannels;
  }
  if (parts) *parts = (size_t)p;
  if (rings) *rings = g;
  return vrSuccess;
}

}  // extern "C"
