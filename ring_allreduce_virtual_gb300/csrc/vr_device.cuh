// vr_device.cuh -- device primitives: memory-model operations in inline PTX,
// bounded waits, 16-byte pack I/O and the per-type reduction of one hop.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>
#include <string.h>

#include <type_traits>

#include "vr_internal.h"

namespace vr {

// ---------------------------------------------------------------------------
// Memory-model operations (PTX ISA memory consistency model, sm_70+).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t ld_relaxed_gpu(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_gpu(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ int ld_volatile_int(const int* p) {
  int v;
  asm volatile("ld.volatile.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// FIFO payload: cached in L2 only (never a stale L1 line).
__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_cg_v4(void* p, uint4 v) {
  asm volatile("st.global.cg.v4.u32 [%0], {%1,%2,%3,%4};"
               ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ uint64_t ld_cg_u64(const void* p) {
  uint64_t v;
  asm volatile("ld.global.cg.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_cg_u64(void* p, uint64_t v) {
  asm volatile("st.global.cg.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void ld_cg_v2u64(const void* p, uint64_t& a, uint64_t& b) {
  asm volatile("ld.global.cg.v2.u64 {%0,%1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ void st_cg_v2u64(void* p, uint64_t a, uint64_t b) {
  asm volatile("st.global.cg.v2.u64 [%0], {%1,%2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}

// LL lines: each 8-byte element is one single-copy-atomic access, so a flag
// and the payload beside it in the same word are seen together.
__device__ __forceinline__ void ld_volatile_v2u64(const void* p, uint64_t& a, uint64_t& b) {
  asm volatile("ld.volatile.global.v2.u64 {%0,%1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ void st_volatile_v2u64(void* p, uint64_t a, uint64_t b) {
  asm volatile("st.volatile.global.v2.u64 [%0], {%1,%2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}

// Own data and outputs: streamed once, so marked evict-first to leave L2 to
// the FIFO lines.
__device__ __forceinline__ uint4 ld_cs_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ void st_cs_v4(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
               ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ uint64_t ld_cs_u64(const void* p) {
  uint64_t v;
  asm volatile("ld.global.cs.u64 %0, [%1];" : "=l"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ void st_cs_u64(void* p, uint64_t v) {
  asm volatile("st.global.cs.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// ---------------------------------------------------------------------------
// Bounded waits. Every spin ends: on success, when the communicator's status
// word turns non-zero (another wait gave up), or after timeoutNs, in which
// case the status word and its host mirror are set to VR_STATUS_TIMEOUT.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void raise_timeout(const vrRingArgs& a) {
  if (atomicCAS(a.status, VR_STATUS_OK, VR_STATUS_TIMEOUT) == VR_STATUS_OK) {
    *(volatile int*)a.statusHost = VR_STATUS_TIMEOUT;
    __threadfence_system();
  }
}

// Wait until *p >= target (acquire). Returns false if the wait gave up.
static __device__ __noinline__ bool wait_ge(const uint64_t* p, uint64_t target, const vrRingArgs& a) {
  if (ld_relaxed_gpu(p) >= target) {
    fence_acq_rel_gpu();
    return true;
  }
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (ld_relaxed_gpu(p) >= target) {
      fence_acq_rel_gpu();
      return true;
    }
    if ((it & 63) == 0) {
      if (ld_volatile_int(a.status) != VR_STATUS_OK) return false;
      if (globaltimer() - t0 > a.timeoutNs) {
        raise_timeout(a);
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// One hop of the reduction, on raw 32- or 64-bit words holding whole elements.
// op(incoming, own), rounded to the element type: integer sum/prod wrap;
// float16 / bfloat16 / float32 / float64 use the IEEE round-to-nearest-even
// instructions of their own width, in the forms that the compiler may not
// fuse into a multiply-add (a pre-multiplied sum's product and the next sum
// are two roundings); max/min select the original bits with
// a > b ? a : b and a < b ? a : b.
// ---------------------------------------------------------------------------
enum { OP_SUM = 0, OP_PROD = 1, OP_MAX = 2, OP_MIN = 3 };

template <typename T, int OP> struct Hop;

template <int OP> struct Hop<int8_t, OP> {
  using Word = uint32_t;
  static __device__ __forceinline__ uint32_t apply(uint32_t a, uint32_t b) {
    if (OP == OP_SUM) return __vadd4(a, b);
    if (OP == OP_MAX) return __vmaxs4(a, b);
    if (OP == OP_MIN) return __vmins4(a, b);
    uint32_t r = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) r |= ((((a >> (8 * i)) & 0xffu) * ((b >> (8 * i)) & 0xffu)) & 0xffu) << (8 * i);
    return r;
  }
};
template <int OP> struct Hop<uint8_t, OP> {
  using Word = uint32_t;
  static __device__ __forceinline__ uint32_t apply(uint32_t a, uint32_t b) {
    if (OP == OP_SUM) return __vadd4(a, b);
    if (OP == OP_MAX) return __vmaxu4(a, b);
    if (OP == OP_MIN) return __vminu4(a, b);
    return Hop<int8_t, OP_PROD>::apply(a, b);
  }
};
template <int OP> struct Hop<int32_t, OP> {
  using Word = uint32_t;
  static __device__ __forceinline__ uint32_t apply(uint32_t a, uint32_t b) {
    if (OP == OP_SUM) return a + b;
    if (OP == OP_PROD) return a * b;
    int32_t x = (int32_t)a, y = (int32_t)b;
    if (OP == OP_MAX) return (uint32_t)(x > y ? x : y);
    return (uint32_t)(x < y ? x : y);
  }
};
template <int OP> struct Hop<uint32_t, OP> {
  using Word = uint32_t;
  static __device__ __forceinline__ uint32_t apply(uint32_t a, uint32_t b) {
    if (OP == OP_SUM) return a + b;
    if (OP == OP_PROD) return a * b;
    if (OP == OP_MAX) return a > b ? a : b;
    return a < b ? a : b;
  }
};
template <int OP> struct Hop<int64_t, OP> {
  using Word = uint64_t;
  static __device__ __forceinline__ uint64_t apply(uint64_t a, uint64_t b) {
    if (OP == OP_SUM) return a + b;
    if (OP == OP_PROD) return a * b;
    int64_t x = (int64_t)a, y = (int64_t)b;
    if (OP == OP_MAX) return (uint64_t)(x > y ? x : y);
    return (uint64_t)(x < y ? x : y);
  }
};
template <int OP> struct Hop<uint64_t, OP> {
  using Word = uint64_t;
  static __device__ __forceinline__ uint64_t apply(uint64_t a, uint64_t b) {
    if (OP == OP_SUM) return a + b;
    if (OP == OP_PROD) return a * b;
    if (OP == OP_MAX) return a > b ? a : b;
    return a < b ? a : b;
  }
};
template <int OP> struct Hop<float, OP> {
  using Word = uint32_t;
  static __device__ __forceinline__ uint32_t apply(uint32_t a, uint32_t b) {
    float x = __uint_as_float(a), y = __uint_as_float(b);
    if (OP == OP_SUM) return __float_as_uint(__fadd_rn(x, y));
    if (OP == OP_PROD) return __float_as_uint(__fmul_rn(x, y));
    if (OP == OP_MAX) return x > y ? a : b;
    return x < y ? a : b;
  }
};
template <int OP> struct Hop<double, OP> {
  using Word = uint64_t;
  static __device__ __forceinline__ uint64_t apply(uint64_t a, uint64_t b) {
    double x = __longlong_as_double((long long)a), y = __longlong_as_double((long long)b);
    if (OP == OP_SUM) return (uint64_t)__double_as_longlong(__dadd_rn(x, y));
    if (OP == OP_PROD) return (uint64_t)__double_as_longlong(__dmul_rn(x, y));
    if (OP == OP_MAX) return x > y ? a : b;
    return x < y ? a : b;
  }
};
template <int OP> struct Hop<__half, OP> {
  using Word = uint32_t;
  static __device__ __forceinline__ uint32_t apply(uint32_t a, uint32_t b) {
    __half2 x = *reinterpret_cast<__half2*>(&a), y = *reinterpret_cast<__half2*>(&b);
    if (OP == OP_SUM) { __half2 r = __hadd2_rn(x, y); return *reinterpret_cast<uint32_t*>(&r); }
    if (OP == OP_PROD) { __half2 r = __hmul2_rn(x, y); return *reinterpret_cast<uint32_t*>(&r); }
    float2 fx = __half22float2(x), fy = __half22float2(y);
    bool lo = OP == OP_MAX ? fx.x > fy.x : fx.x < fy.x;
    bool hi = OP == OP_MAX ? fx.y > fy.y : fx.y < fy.y;
    return ((lo ? a : b) & 0xffffu) | ((hi ? a : b) & 0xffff0000u);
  }
};
template <int OP> struct Hop<__nv_bfloat16, OP> {
  using Word = uint32_t;
  static __device__ __forceinline__ uint32_t apply(uint32_t a, uint32_t b) {
    __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&a);
    __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162*>(&b);
    if (OP == OP_SUM) { __nv_bfloat162 r = __hadd2_rn(x, y); return *reinterpret_cast<uint32_t*>(&r); }
    if (OP == OP_PROD) { __nv_bfloat162 r = __hmul2_rn(x, y); return *reinterpret_cast<uint32_t*>(&r); }
    float2 fx = __bfloat1622float2(x), fy = __bfloat1622float2(y);
    bool lo = OP == OP_MAX ? fx.x > fy.x : fx.x < fy.x;
    bool hi = OP == OP_MAX ? fx.y > fy.y : fx.y < fy.y;
    return ((lo ? a : b) & 0xffffu) | ((hi ? a : b) & 0xffff0000u);
  }
};

// The 8-bit floating types (E4M3: 4 exponent bits, no infinities, largest
// finite 448; E5M2: 5 exponent bits, largest finite 57344) as one-byte tag
// types. A sum or product converts both operands exactly to float (through
// half, which holds every 8-bit value), computes with the non-contracting
// round-to-nearest float instruction, and rounds to the format to nearest
// even, saturating at the largest finite value. The float result is exact
// for E4M3 and for every product; an E5M2 sum may round in float first,
// which cannot change the final rounding (float's 24-bit significand is more
// than twice E5M2's 3 bits plus two: innocuous double rounding). max/min
// compare the codes as sign-magnitude integers, which order like the values.
struct vr_fp8_e4m3 { uint8_t bits; };
struct vr_fp8_e5m2 { uint8_t bits; };

__device__ __forceinline__ int fp8_key(uint32_t code) {
  return (code & 0x80u) ? -(int)(code & 0x7Fu) : (int)(code & 0x7Fu);
}

template <__nv_fp8_interpretation_t K, int OP>
__device__ __forceinline__ uint32_t hop_fp8x4(uint32_t a, uint32_t b) {
  uint32_t r = 0;
  if (OP == OP_SUM || OP == OP_PROD) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float2 x = __half22float2(
          __half2(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(a >> (16 * h)), K)));
      const float2 y = __half22float2(
          __half2(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(b >> (16 * h)), K)));
      const float2 z = OP == OP_SUM ? make_float2(__fadd_rn(x.x, y.x), __fadd_rn(x.y, y.y))
                                    : make_float2(__fmul_rn(x.x, y.x), __fmul_rn(x.y, y.y));
      r |= (uint32_t)__nv_cvt_float2_to_fp8x2(z, __NV_SATFINITE, K) << (16 * h);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t ca = (a >> (8 * i)) & 0xFFu, cb = (b >> (8 * i)) & 0xFFu;
      const bool takeA = OP == OP_MAX ? fp8_key(ca) > fp8_key(cb) : fp8_key(ca) < fp8_key(cb);
      r |= (takeA ? ca : cb) << (8 * i);
    }
  }
  return r;
}
template <int OP> struct Hop<vr_fp8_e4m3, OP> {
  using Word = uint32_t;
  static __device__ __forceinline__ uint32_t apply(uint32_t a, uint32_t b) {
    return hop_fp8x4<__NV_E4M3, OP>(a, b);
  }
};
template <int OP> struct Hop<vr_fp8_e5m2, OP> {
  using Word = uint32_t;
  static __device__ __forceinline__ uint32_t apply(uint32_t a, uint32_t b) {
    return hop_fp8x4<__NV_E5M2, OP>(a, b);
  }
};

// Apply one hop to 8 and 16 bytes of whole elements.
template <typename T, int OP>
__device__ __forceinline__ uint64_t hop8(uint64_t a, uint64_t b) {
  using H = Hop<T, OP>;
  if constexpr (sizeof(typename H::Word) == 8) {
    return H::apply(a, b);
  } else {
    uint32_t lo = H::apply((uint32_t)a, (uint32_t)b);
    uint32_t hi = H::apply((uint32_t)(a >> 32), (uint32_t)(b >> 32));
    return (uint64_t)lo | ((uint64_t)hi << 32);
  }
}
template <typename T, int OP>
__device__ __forceinline__ uint4 hop16(uint4 a, uint4 b) {
  using H = Hop<T, OP>;
  if constexpr (sizeof(typename H::Word) == 4) {
    return make_uint4(H::apply(a.x, b.x), H::apply(a.y, b.y), H::apply(a.z, b.z),
                      H::apply(a.w, b.w));
  } else {
    const uint64_t lo = H::apply((uint64_t)a.x | ((uint64_t)a.y << 32),
                                 (uint64_t)b.x | ((uint64_t)b.y << 32));
    const uint64_t hi = H::apply((uint64_t)a.z | ((uint64_t)a.w << 32),
                                 (uint64_t)b.z | ((uint64_t)b.w << 32));
    return make_uint4((uint32_t)lo, (uint32_t)(lo >> 32), (uint32_t)hi, (uint32_t)(hi >> 32));
  }
}

// The scalar of a pre-multiplied sum replicated over 16 bytes of elements.
template <typename T>
__device__ __forceinline__ uint4 scalar_pack(uint64_t bits) {
  uint4 v;
  T* e = reinterpret_cast<T*>(&v);
  T s;
  memcpy(&s, &bits, sizeof(T));
  for (int i = 0; i < (int)(16 / sizeof(T)); ++i) e[i] = s;
  return v;
}

// Integer average: every element of a pack divided by n, truncating toward
// zero as C does (a no-op for floating types, whose average is a
// pre-multiplied sum).
template <typename T>
__device__ __forceinline__ uint4 div_pack(uint4 v, int n) {
  if constexpr (std::is_integral<T>::value) {
    T* e = reinterpret_cast<T*>(&v);
    for (int i = 0; i < (int)(16 / sizeof(T)); ++i) {
      if constexpr (std::is_signed<T>::value)
        e[i] = (T)((long long)e[i] / (long long)n);
      else
        e[i] = (T)((unsigned long long)e[i] / (unsigned long long)n);
    }
  }
  return v;
}
template <typename T>
__device__ __forceinline__ uint64_t div_word(uint64_t v, int n) {
  if constexpr (std::is_integral<T>::value) {
    T* e = reinterpret_cast<T*>(&v);
    for (int i = 0; i < (int)(8 / sizeof(T)); ++i) {
      if constexpr (std::is_signed<T>::value)
        e[i] = (T)((long long)e[i] / (long long)n);
      else
        e[i] = (T)((unsigned long long)e[i] / (unsigned long long)n);
    }
  }
  return v;
}

// ---------------------------------------------------------------------------
// User-buffer I/O of up to 16 (or 8) bytes of whole elements. `valid` is the
// number of bytes inside the buffer; `vec` says the address is aligned for the
// full-width access. Partial or unaligned pieces go element by element.
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ uint4 load_pack(const char* p, uint32_t valid, bool vec) {
  if (vec && valid >= 16) return ld_cs_v4(p);
  uint4 v = make_uint4(0, 0, 0, 0);
  T* e = reinterpret_cast<T*>(&v);
  for (uint32_t i = 0; i * sizeof(T) < valid && i * sizeof(T) < 16; ++i)
    e[i] = reinterpret_cast<const T*>(p)[i];
  return v;
}
template <typename T>
__device__ __forceinline__ void store_pack(char* p, uint4 v, uint32_t valid, bool vec) {
  if (vec && valid >= 16) { st_cs_v4(p, v); return; }
  const T* e = reinterpret_cast<const T*>(&v);
  for (uint32_t i = 0; i * sizeof(T) < valid && i * sizeof(T) < 16; ++i)
    reinterpret_cast<T*>(p)[i] = e[i];
}
template <typename T>
__device__ __forceinline__ uint64_t load_word(const char* p, uint32_t valid, bool vec) {
  if (vec && valid >= 8) return ld_cs_u64(p);
  uint64_t v = 0;
  T* e = reinterpret_cast<T*>(&v);
  for (uint32_t i = 0; i * sizeof(T) < valid && i * sizeof(T) < 8; ++i)
    e[i] = reinterpret_cast<const T*>(p)[i];
  return v;
}
template <typename T>
__device__ __forceinline__ void store_word(char* p, uint64_t v, uint32_t valid, bool vec) {
  if (vec && valid >= 8) { st_cs_u64(p, v); return; }
  const T* e = reinterpret_cast<const T*>(&v);
  for (uint32_t i = 0; i * sizeof(T) < valid && i * sizeof(T) < 8; ++i)
    reinterpret_cast<T*>(p)[i] = e[i];
}

// What a stage kind does: receive from rank r-1, send to rank r+1, read the
// rank's own input, write its output, reduce incoming with own.
__device__ __forceinline__ bool kind_recv(int k) { return vrKindRecv(k); }
__device__ __forceinline__ bool kind_send(int k) { return vrKindSend(k); }
__device__ __forceinline__ bool kind_own(int k) { return vrKindOwn(k); }
__device__ __forceinline__ bool kind_out(int k) { return vrKindOut(k); }
__device__ __forceinline__ bool kind_reduce(int k) { return vrKindReduce(k); }

__host__ __device__ __forceinline__ uint64_t div_up(uint64_t a, uint64_t b) { return (a + b - 1) / b; }
__host__ __device__ __forceinline__ uint64_t align_up(uint64_t a, uint64_t b) { return div_up(a, b) * b; }
__host__ __device__ __forceinline__ uint64_t min_u64(uint64_t a, uint64_t b) { return a < b ? a : b; }

}  // namespace vr
