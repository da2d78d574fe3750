// vr_noalloc.cu -- vrAllReduceNoAlloc: the global-memory FIFO AllReduce with
// its scratch (FIFO slots, control words, status word) in a fixed array that
// the library itself owns, so that a call allocates nothing.
//
// Some callers cannot allocate device memory at the point where they need an
// AllReduce: code running under a framework's caching allocator that must
// account for every device byte (a stray cudaMalloc can fail once the pool
// has reserved the GPU's memory, or break its bookkeeping), and code on a
// latency-critical path where cudaMalloc/cudaFree would stall the device. For
// them this entry point takes only the caller's input and output buffers.
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "vr_internal.h"

// Scratch of every vrAllReduceNoAlloc call on a device: the status words
// (the first 256 bytes, at a fixed place so that vrAllReduceNoAllocGetStatus
// finds them whatever the last call's geometry), then the FIFO slots, then the
// control words. Every GPU that runs a call holds this array until the
// process exits.
#define VR_NOALLOC_SCRATCH_BYTES (4u << 20)
#define VR_NOALLOC_SLOT_BYTES 4096u
#define VR_NOALLOC_DEPTH 2u
#define VR_NOALLOC_STATUS_BYTES 256u
static __device__ __align__(256) unsigned char vrNoAllocScratch[VR_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex gMutex;
void* gScratch[kMaxDevices];  // device address of vrNoAllocScratch, per device

// Once per device, with that device current: the array's device address (in
// host code its name is only a host-side stand-in).
void* scratchAddress(int dev) {
  std::lock_guard<std::mutex> g(gMutex);
  if (!gScratch[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, vrNoAllocScratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    gScratch[dev] = p;
  }
  return gScratch[dev];
}

int elemSizeOf(vrDataType_t t) {
  switch (t) {
    case vrInt8: case vrUint8: return 1;
    case vrFloat16: case vrBfloat16: return 2;
    case vrFloat8e4m3: case vrFloat8e5m2: return 1;
    case vrInt32: case vrUint32: case vrFloat32: return 4;
    case vrInt64: case vrUint64: case vrFloat64: return 8;
    default: return 0;
  }
}

const void* genericKernelFor(vrDataType_t t, int op, int proto) {
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

// The kernel a call will launch, touched once per device and kernel: with
// lazy module loading (CUDA_MODULE_LOADING=LAZY, the default) a kernel's
// module is loaded at its first use, which may allocate device memory, so
// the first call of each kind on a device does it here -- also for a call
// with count 0, which therefore serves as a warm-up.
bool touchKernel(int dev, const void* kernel) {
  static std::mutex m;
  static const void* seen[kMaxDevices][64];
  static int nSeen[kMaxDevices];
  std::lock_guard<std::mutex> g(m);
  for (int i = 0; i < nSeen[dev]; ++i)
    if (seen[dev][i] == kernel) return true;
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (nSeen[dev] < 64) seen[dev][nSeen[dev]++] = kernel;
  return true;
}

long envLong(const char* name, long dflt) {
  const char* s = getenv(name);
  if (!s || !*s) return dflt;
  char* end = nullptr;
  const long v = strtol(s, &end, 0);
  return (end && *end == 0) ? v : dflt;
}

}  // namespace

extern "C" VR_API vrResult_t vrAllReduceNoAlloc(const void* const* sendbufs, void* const* recvbufs,
                                                size_t count, int nRanks, int nChannels,
                                                vrProto_t proto, size_t chunkBytes,
                                                vrDataType_t dtype, vrRedOp_t op, void* stream) {
  const int es = elemSizeOf(dtype);
  if (nRanks < 1 || nRanks > VR_MAX_RANKS || nChannels < 1 || nChannels > VR_MAX_CHANNELS ||
      proto < vrProtoSimple || proto >= vrNumProtos || chunkBytes < 16 || chunkBytes % 16 != 0 ||
      !es || op < vrSum || op > vrMin)
    return vrInvalidArgument;
  // The FIFOs of every (channel, rank) edge, their control words and the
  // status word must fit in the fixed scratch array.
  const size_t edges = (size_t)nChannels * (size_t)nRanks;
  const size_t fifoBytes = edges * VR_NOALLOC_DEPTH * VR_NOALLOC_SLOT_BYTES;
  const size_t ctrlBytes = edges * VR_CTRL_WORDS_PER_EDGE * sizeof(uint64_t);
  if (VR_NOALLOC_STATUS_BYTES + fifoBytes + ctrlBytes > VR_NOALLOC_SCRATCH_BYTES)
    return vrInvalidUsage;
  const void* kernel = genericKernelFor(dtype, (int)op, (int)proto);
  if (!kernel) return vrInternalError;
  // Set-up of this device (the array's address, the kernel's module) before
  // anything else, so that a call with count 0 is a warm-up.
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return vrCudaError;
  char* scratch = static_cast<char*>(scratchAddress(dev));
  if (!scratch || !touchKernel(dev, kernel)) return vrCudaError;
  if (count == 0) return vrSuccess;
  if (!sendbufs || !recvbufs) return vrInvalidArgument;
  int alignMask = 0;
  for (int r = 0; r < nRanks; ++r) {
    const uintptr_t s = (uintptr_t)sendbufs[r], d = (uintptr_t)recvbufs[r];
    if (!s || !d || s % es || d % es) return vrInvalidArgument;
    alignMask |= (int)((s | d) & 15);
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (nRanks == 1) {
    if (sendbufs[0] != recvbufs[0] &&
        cudaMemcpyAsync(recvbufs[0], sendbufs[0], count * (size_t)es, cudaMemcpyDeviceToDevice,
                        st) != cudaSuccess)
      return vrCudaError;
    return vrSuccess;
  }
  // The array keeps the previous call's flags and status: clear the part
  // this call uses (its step counters start again at zero).
  const size_t used = VR_NOALLOC_STATUS_BYTES + fifoBytes + ctrlBytes;
  if (cudaMemsetAsync(scratch, 0, used, st) != cudaSuccess) return vrCudaError;

  vrRingArgs a;
  memset(&a, 0, sizeof(a));
  a.count = count;
  a.chunkElems = chunkBytes / (size_t)es;
  a.stepBase = 0;
  // Device waits give up after VR_TIMEOUT_MS milliseconds (default 10 s);
  // VR_DEBUG_SILENT_RANK names a rank that never signals (fault tests).
  long ms = envLong("VR_TIMEOUT_MS", 10000);
  if (ms < 1 || ms > 3600L * 1000L) ms = 10000;
  a.timeoutNs = (uint64_t)ms * 1000000ull;
  a.status = reinterpret_cast<int*>(scratch);
  a.statusHost = a.status + 1;  // no host mirror: a second device word
  a.fifo = scratch + VR_NOALLOC_STATUS_BYTES;
  a.ctrl = reinterpret_cast<uint64_t*>(scratch + VR_NOALLOC_STATUS_BYTES + fifoBytes);
  a.nRanks = nRanks;
  a.nChannels = nChannels;
  a.alignMask = alignMask;
  a.silentRank = (int)envLong("VR_DEBUG_SILENT_RANK", -1);
  a.slotBytes = VR_NOALLOC_SLOT_BYTES;
  a.depth = VR_NOALLOC_DEPTH;
  for (int r = 0; r < nRanks; ++r) {
    a.send[r] = sendbufs[r];
    a.recv[r] = recvbufs[r];
  }
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)edges);
  cfg.blockDim = dim3(VR_GENERIC_THREADS);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&a};
  const cudaError_t e = cudaLaunchKernelExC(&cfg, kernel, args);
  if (e == cudaErrorCooperativeLaunchTooLarge) {
    cudaGetLastError();
    return vrInvalidUsage;
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return vrCudaError;
  }
  return vrSuccess;
}

extern "C" VR_API vrResult_t vrAllReduceNoAllocGetStatus(vrResult_t* status) {
  if (!status) return vrInvalidArgument;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return vrCudaError;
  const char* scratch = static_cast<const char*>(scratchAddress(dev));
  if (!scratch) return vrCudaError;
  // A plain synchronous copy into a host int: it allocates nothing.
  int v = 0;
  if (cudaMemcpy(&v, scratch, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return vrCudaError;
  }
  *status = v == VR_STATUS_OK ? vrSuccess : vrTimeout;
  return vrSuccess;
}
