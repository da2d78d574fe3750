/*
 * vr_oracle.c -- plain CPU oracle for the virtual-rank ring AllReduce (and
 * its halves and the double-binary-tree AllReduce, at the end).
 *
 * TEST INFRASTRUCTURE ONLY. The tests, the package smoke check and the
 * benchmark's CPU-baseline / reference arm load this file's shared library.
 * The CUDA library never links, includes or calls it, and this file includes
 * nothing from the CUDA library: the two implement the chunk map and the
 * arithmetic independently.
 *
 * What is computed. N ranks each hold `count` elements; every rank ends with
 * the elementwise reduction of the N buffers. The reduction ORDER is the one
 * the ring schedule fixes, so floating-point results are defined bit for bit:
 *
 *  1. Channels. "Each channel handles count/nChannels elements" as one
 *     contiguous range (NCCL 原始碼解讀：一個 AllReduce 的 GPU 旅程, ch.2 §2.2,
 *     channel walkthrough, step 3). Reading taken: the per-channel size is
 *     divUp(count, nChannels) rounded up to 16 bytes of elements; trailing
 *     channels may be short or empty.
 *  2. Loops and chunks. Inside a channel the data is walked in loops of
 *     N * chunkElems elements; in a loop whose remainder `rem` is smaller than
 *     that, the chunk is alignUp(divUp(rem, N), 16/elemSize) elements; chunk c
 *     of a loop covers [c*cur, min(rem, (c+1)*cur)) and may be empty
 *     (same book, ch.2 §2.3, RingARAlgorithm::getNextSendAddr).
 *  3. Order. The chunk a rank sends at stage s is (ringIndex + N - 1 - s) mod N
 *     (same passage), and each rank receives from its ring predecessor and sends
 *     to its successor. So at stage 0 chunk c leaves rank c+1, and its partial
 *     sum then visits ranks c+2, ..., c in ring order:
 *         acc = x[c+1]; acc = op(acc, x[c+2]); ... ; acc = op(acc, x[c])
 *     with op(incoming partial, own value), rounded to the element type after
 *     every op because the partial travels between ranks in that type.
 *  4. Every rank's output is that acc (the all-gather half only copies).
 *
 * Arithmetic. Integers wrap (two's complement) for sum and prod; max/min use
 * a > b ? a : b (and a < b ? a : b). float32 and float64 use C arithmetic
 * (build with -ffp-contract=off, no fast-math). float16 and bfloat16 are held
 * as raw 16-bit codes: both operands are decoded exactly to double, the op is
 * done in double, and the result is rounded to the 16-bit format by
 * round_to_format() below, written from the IEEE 754 definition of
 * round-to-nearest-even with gradual underflow and overflow to infinity. For
 * + and * the double result is either exact or, by Figueroa's condition for
 * innocuous double rounding (p >= 2q + 2, "When is double rounding
 * innocuous?", SIGNUM 1995), rounds to the same 16-bit value as the exact
 * result would.
 *
 * NaN inputs: parity unpinned (the pages say nothing; the generated inputs
 * contain none).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Element type codes of this oracle (its own numbering). */
enum {
  OR_INT8 = 0, OR_UINT8 = 1, OR_INT32 = 2, OR_UINT32 = 3, OR_INT64 = 4,
  OR_UINT64 = 5, OR_FLOAT16 = 6, OR_BFLOAT16 = 7, OR_FLOAT32 = 8, OR_FLOAT64 = 9,
  OR_FP8E4M3 = 10, OR_FP8E5M2 = 11
};
/* Reduction codes of this oracle. */
enum { OR_SUM = 0, OR_PROD = 1, OR_MAX = 2, OR_MIN = 3 };

static int elem_size(int dtype) {
  switch (dtype) {
    case OR_INT8: case OR_UINT8: case OR_FP8E4M3: case OR_FP8E5M2: return 1;
    case OR_FLOAT16: case OR_BFLOAT16: return 2;
    case OR_INT32: case OR_UINT32: case OR_FLOAT32: return 4;
    case OR_INT64: case OR_UINT64: case OR_FLOAT64: return 8;
    default: return 0;
  }
}

static uint64_t div_up(uint64_t a, uint64_t b) { return (a + b - 1) / b; }
static uint64_t align_up(uint64_t a, uint64_t b) { return div_up(a, b) * b; }

/* ------------------------------------------------------------------------ */
/* 16-bit floating-point formats, from the IEEE 754 definitions.             */
/* p = significand bits including the implicit bit; emin = exponent of the   */
/* smallest normal; emax = exponent of the largest finite.                   */
/* ------------------------------------------------------------------------ */
typedef struct { int p, emin, emax, ebits; } fmt16;
static const fmt16 FMT_F16 = {11, -14, 15, 5};
static const fmt16 FMT_BF16 = {8, -126, 127, 8};

/* Round a double to the nearest value of format f, ties to even, with
 * subnormals and overflow to +-inf. Returns the rounded value as a double
 * (exactly representable in f). */
double oracle_round_to_format(double x, int p, int emin, int emax) {
  if (isnan(x) || isinf(x) || x == 0.0) return x;
  int e2;
  frexp(x, &e2);          /* |x| = m * 2^e2, 0.5 <= m < 1: leading bit 2^(e2-1) */
  int E = e2 - 1;
  if (E < emin) E = emin; /* below the normal range the quantum stays fixed */
  double quantum = ldexp(1.0, E - (p - 1));
  double n = x / quantum;              /* exact: division by a power of two */
  double r = nearbyint(n);             /* default rounding mode: ties to even */
  double y = r * quantum;
  double maxf = ldexp(2.0 - ldexp(1.0, 1 - p), emax);
  if (fabs(y) > maxf) return copysign(INFINITY, x);
  return y;
}

static double round_fmt(double x, fmt16 f) {
  return oracle_round_to_format(x, f.p, f.emin, f.emax);
}

/* Decode a 16-bit code of format f to double (exact). */
static double decode16(uint16_t h, fmt16 f) {
  int mbits = f.p - 1;
  int sign = (h >> 15) & 1;
  int ef = (h >> mbits) & ((1 << f.ebits) - 1);
  int mf = h & ((1 << mbits) - 1);
  int bias = f.emax;
  double v;
  if (ef == (1 << f.ebits) - 1) {
    v = mf ? NAN : INFINITY;
  } else if (ef == 0) {
    v = ldexp((double)mf, f.emin - mbits);           /* subnormal or zero */
  } else {
    v = ldexp((double)(mf | (1 << mbits)), ef - bias - mbits);
  }
  return sign ? -v : v;
}

/* Encode a double that is exactly representable in f (as returned by
 * round_fmt) to its 16-bit code. NaN maps to the quiet NaN with an empty
 * payload. */
static uint16_t encode16(double y, fmt16 f) {
  int mbits = f.p - 1;
  int bias = f.emax;
  uint16_t sign = signbit(y) ? 0x8000u : 0u;
  uint16_t expmask = (uint16_t)(((1 << f.ebits) - 1) << mbits);
  if (isnan(y)) return (uint16_t)(expmask | (1u << (mbits - 1)));
  if (isinf(y)) return (uint16_t)(sign | expmask);
  double a = fabs(y);
  if (a == 0.0) return sign;
  int e2;
  frexp(a, &e2);
  int E = e2 - 1;
  if (E < f.emin) {                                   /* subnormal */
    uint64_t m = (uint64_t)ldexp(a, mbits - f.emin);
    return (uint16_t)(sign | m);
  }
  uint64_t m = (uint64_t)ldexp(a, mbits - E);         /* in [2^mbits, 2^(mbits+1)) */
  m -= (uint64_t)1 << mbits;
  return (uint16_t)(sign | ((uint16_t)(E + bias) << mbits) | m);
}

double oracle_f16_decode(uint16_t h) { return decode16(h, FMT_F16); }
double oracle_bf16_decode(uint16_t h) { return decode16(h, FMT_BF16); }
uint16_t oracle_f16_from_double(double x) { return encode16(round_fmt(x, FMT_F16), FMT_F16); }
uint16_t oracle_bf16_from_double(double x) { return encode16(round_fmt(x, FMT_BF16), FMT_BF16); }

/* ------------------------------------------------------------------------ */
/* 8-bit floating-point formats (the OCP 8-bit floating point formats: E4M3  */
/* with 4 exponent bits, bias 7, no infinities, S.1111.111 the only NaN,     */
/* largest finite 448; E5M2 with 5 exponent bits, bias 15, IEEE-like         */
/* infinities and NaNs, largest finite 57344). The pages say only that an    */
/* FP8 reduction needs sm90 or later ("NCCL 原始碼解讀", ch.6, the FP8 type  */
/* check); reading taken: an op is computed exactly and rounded to nearest   */
/* even, and a result beyond the largest finite value (or an infinity)       */
/* saturates to it, keeping its sign (the GPU's conversion to these formats  */
/* exists only in that saturating form).                                     */
/* ------------------------------------------------------------------------ */
typedef struct { int p, emin, bias, ebits, has_inf; double maxf; } fmt8;
static const fmt8 FMT_E4M3 = {4, -6, 7, 4, 0, 448.0};
static const fmt8 FMT_E5M2 = {3, -14, 15, 5, 1, 57344.0};

static double decode8(uint8_t h, fmt8 f) {
  int mbits = f.p - 1;
  int sign = (h >> 7) & 1;
  int ef = (h >> mbits) & ((1 << f.ebits) - 1);
  int mf = h & ((1 << mbits) - 1);
  int eall = (1 << f.ebits) - 1, mall = (1 << mbits) - 1;
  double v;
  if (f.has_inf && ef == eall) {
    v = mf ? NAN : INFINITY;
  } else if (!f.has_inf && ef == eall && mf == mall) {
    v = NAN;
  } else if (ef == 0) {
    v = ldexp((double)mf, f.emin - mbits);           /* subnormal or zero */
  } else {
    v = ldexp((double)(mf | (1 << mbits)), ef - f.bias - mbits);
  }
  return sign ? -v : v;
}

/* Round to nearest even with an unbounded exponent range above, then
 * saturate to +-maxf; NaN stays NaN. */
static double round8(double x, fmt8 f) {
  if (isnan(x)) return x;
  if (isinf(x)) return copysign(f.maxf, x);
  double y = oracle_round_to_format(x, f.p, f.emin, 1000);
  if (fabs(y) > f.maxf) y = copysign(f.maxf, x);
  return y;
}

/* Encode a finite value exactly representable in f, or a NaN (as the NaN
 * with every exponent and significand bit set). */
static uint8_t encode8(double y, fmt8 f) {
  int mbits = f.p - 1;
  uint8_t sign = signbit(y) ? 0x80u : 0u;
  if (isnan(y)) return 0x7Fu;
  double a = fabs(y);
  if (a == 0.0) return sign;
  int e2;
  frexp(a, &e2);
  int E = e2 - 1;
  if (E < f.emin) return (uint8_t)(sign | (uint64_t)ldexp(a, mbits - f.emin));
  uint64_t m = (uint64_t)ldexp(a, mbits - E) - ((uint64_t)1 << mbits);
  return (uint8_t)(sign | ((E + f.bias) << mbits) | m);
}

double oracle_fp8e4m3_decode(uint8_t h) { return decode8(h, FMT_E4M3); }
double oracle_fp8e5m2_decode(uint8_t h) { return decode8(h, FMT_E5M2); }
uint8_t oracle_fp8e4m3_from_double(double x) { return encode8(round8(x, FMT_E4M3), FMT_E4M3); }
uint8_t oracle_fp8e5m2_from_double(double x) { return encode8(round8(x, FMT_E5M2), FMT_E5M2); }

/* ------------------------------------------------------------------------ */
/* One reduction op, in the element type.                                    */
/* ------------------------------------------------------------------------ */
static double combine_double(int op, double a, double b) {
  switch (op) {
    case OR_SUM: return a + b;
    case OR_PROD: return a * b;
    case OR_MAX: return a > b ? a : b;
    default: return a < b ? a : b;
  }
}

static float combine_float(int op, float a, float b) {
  switch (op) {
    case OR_SUM: return a + b;
    case OR_PROD: return a * b;
    case OR_MAX: return a > b ? a : b;
    default: return a < b ? a : b;
  }
}

static uint16_t combine_fmt16(int op, uint16_t a, uint16_t b, fmt16 f) {
  double x = decode16(a, f), y = decode16(b, f);
  return encode16(round_fmt(combine_double(op, x, y), f), f);
}

/* Integers: sum/prod wrap modulo 2^bits (computed in uint64_t, truncated by
 * the caller's cast); max/min compare as signed or unsigned. */
#define COMBINE_INT(NAME, T, UT)                                              \
  static T NAME(int op, T a, T b) {                                          \
    switch (op) {                                                            \
      case OR_SUM: return (T)(UT)((uint64_t)(UT)a + (uint64_t)(UT)b);        \
      case OR_PROD: return (T)(UT)((uint64_t)(UT)a * (uint64_t)(UT)b);       \
      case OR_MAX: return a > b ? a : b;                                     \
      default: return a < b ? a : b;                                         \
    }                                                                        \
  }
COMBINE_INT(combine_i8, int8_t, uint8_t)
COMBINE_INT(combine_u8, uint8_t, uint8_t)
COMBINE_INT(combine_i32, int32_t, uint32_t)
COMBINE_INT(combine_u32, uint32_t, uint32_t)
COMBINE_INT(combine_i64, int64_t, uint64_t)
COMBINE_INT(combine_u64, uint64_t, uint64_t)

static uint16_t combine_f16(int op, uint16_t a, uint16_t b) { return combine_fmt16(op, a, b, FMT_F16); }
static uint16_t combine_bf16(int op, uint16_t a, uint16_t b) { return combine_fmt16(op, a, b, FMT_BF16); }
/* Sums and products of two 8-bit values are exact in double: one rounding. */
static uint8_t combine_fmt8(int op, uint8_t a, uint8_t b, fmt8 f) {
  double x = decode8(a, f), y = decode8(b, f);
  return encode8(round8(combine_double(op, x, y), f), f);
}
static uint8_t combine_e4m3(int op, uint8_t a, uint8_t b) { return combine_fmt8(op, a, b, FMT_E4M3); }
static uint8_t combine_e5m2(int op, uint8_t a, uint8_t b) { return combine_fmt8(op, a, b, FMT_E5M2); }
static float combine_f32(int op, float a, float b) { return combine_float(op, a, b); }
static double combine_f64(int op, double a, double b) { return combine_double(op, a, b); }

/* The fold of one chunk c over elements [b, e): start at rank c+1, then visit
 * ranks c+2, ..., c in ring order. */
#define DEFINE_FOLD(NAME, T, COMBINE)                                         \
  static void NAME(int op, int N, const void* const* xs, void* outv,          \
                   uint64_t b, uint64_t e, int c) {                           \
    T* out = (T*)outv;                                                        \
    for (uint64_t i = b; i < e; ++i) {                                        \
      T acc = ((const T*)xs[(c + 1) % N])[i];                                 \
      for (int k = 2; k <= N; ++k)                                            \
        acc = COMBINE(op, acc, ((const T*)xs[(c + k) % N])[i]);               \
      out[i] = acc;                                                           \
    }                                                                         \
  }
DEFINE_FOLD(fold_i8, int8_t, combine_i8)
DEFINE_FOLD(fold_u8, uint8_t, combine_u8)
DEFINE_FOLD(fold_i32, int32_t, combine_i32)
DEFINE_FOLD(fold_u32, uint32_t, combine_u32)
DEFINE_FOLD(fold_i64, int64_t, combine_i64)
DEFINE_FOLD(fold_u64, uint64_t, combine_u64)
DEFINE_FOLD(fold_f16, uint16_t, combine_f16)
DEFINE_FOLD(fold_bf16, uint16_t, combine_bf16)
DEFINE_FOLD(fold_f32, float, combine_f32)
DEFINE_FOLD(fold_f64, double, combine_f64)
DEFINE_FOLD(fold_e4m3, uint8_t, combine_e4m3)
DEFINE_FOLD(fold_e5m2, uint8_t, combine_e5m2)

typedef void (*fold_fn)(int, int, const void* const*, void*, uint64_t, uint64_t, int);

static fold_fn fold_for(int dtype) {
  switch (dtype) {
    case OR_INT8: return fold_i8;
    case OR_UINT8: return fold_u8;
    case OR_INT32: return fold_i32;
    case OR_UINT32: return fold_u32;
    case OR_INT64: return fold_i64;
    case OR_UINT64: return fold_u64;
    case OR_FLOAT16: return fold_f16;
    case OR_BFLOAT16: return fold_bf16;
    case OR_FLOAT32: return fold_f32;
    case OR_FLOAT64: return fold_f64;
    case OR_FP8E4M3: return fold_e4m3;
    case OR_FP8E5M2: return fold_e5m2;
    default: return 0;
  }
}

/* ------------------------------------------------------------------------ */
/* The chunk map (steps 1 and 2 above).                                      */
/* ------------------------------------------------------------------------ */

/* Channel ch covers [*beg, *end) of the buffer. */
void oracle_channel_range(uint64_t count, int nChannels, int elemSize, int ch,
                          uint64_t* beg, uint64_t* end) {
  uint64_t align = 16 / (uint64_t)elemSize;
  uint64_t per = align_up(div_up(count, (uint64_t)nChannels), align);
  uint64_t b = (uint64_t)ch * per;
  uint64_t e = b + per;
  if (b > count) b = count;
  if (e > count) e = count;
  *beg = b;
  *end = e;
}

/* Visit every non-empty chunk of every loop of every channel in schedule
 * order. For each: channel, loop index, chunk id c, absolute [b, e). */
typedef void (*chunk_visitor)(void* ctx, int ch, uint64_t loop, int c,
                              uint64_t b, uint64_t e);

static void walk_chunks(uint64_t count, int N, int nChannels, int elemSize,
                        uint64_t chunkBytes, chunk_visitor visit, void* ctx) {
  uint64_t align = 16 / (uint64_t)elemSize;
  uint64_t chunkElems = chunkBytes / (uint64_t)elemSize;
  uint64_t loopElems = (uint64_t)N * chunkElems;
  for (int ch = 0; ch < nChannels; ++ch) {
    uint64_t cb, ce;
    oracle_channel_range(count, nChannels, elemSize, ch, &cb, &ce);
    uint64_t size = ce - cb;
    uint64_t loop = 0;
    for (uint64_t off = 0; off < size; off += loopElems, ++loop) {
      uint64_t rem = size - off;
      uint64_t cur = rem < loopElems ? align_up(div_up(rem, (uint64_t)N), align)
                                     : chunkElems;
      for (int c = 0; c < N; ++c) {
        uint64_t lo = (uint64_t)c * cur;
        if (lo >= rem) continue;               /* empty chunk */
        uint64_t hi = lo + cur < rem ? lo + cur : rem;
        visit(ctx, ch, loop, c, cb + off + lo, cb + off + hi);
      }
    }
  }
}

typedef struct {
  uint64_t n, cap;
  int32_t* ch;
  int64_t* loop;
  int32_t* chunk;
  uint64_t* beg;
  uint64_t* end;
} range_list;

static void count_visit(void* ctx, int ch, uint64_t loop, int c, uint64_t b,
                        uint64_t e) {
  (void)ch; (void)loop; (void)c; (void)b; (void)e;
  ((range_list*)ctx)->n++;
}

static void store_visit(void* ctx, int ch, uint64_t loop, int c, uint64_t b,
                        uint64_t e) {
  range_list* L = (range_list*)ctx;
  if (L->n < L->cap) {
    L->ch[L->n] = ch;
    L->loop[L->n] = (int64_t)loop;
    L->chunk[L->n] = c;
    L->beg[L->n] = b;
    L->end[L->n] = e;
  }
  L->n++;
}

/* Number of non-empty chunk ranges (for sizing the arrays below). */
uint64_t oracle_num_chunk_ranges(uint64_t count, int N, int nChannels,
                                 int elemSize, uint64_t chunkBytes) {
  range_list L = {0};
  walk_chunks(count, N, nChannels, elemSize, chunkBytes, count_visit, &L);
  return L.n;
}

/* Fill up to `cap` chunk ranges; returns the total number. */
uint64_t oracle_chunk_ranges(uint64_t count, int N, int nChannels, int elemSize,
                             uint64_t chunkBytes, uint64_t cap, int32_t* ch,
                             int64_t* loop, int32_t* chunk, uint64_t* beg,
                             uint64_t* end) {
  range_list L = {0, cap, ch, loop, chunk, beg, end};
  walk_chunks(count, N, nChannels, elemSize, chunkBytes, store_visit, &L);
  return L.n;
}

/* ------------------------------------------------------------------------ */
/* The AllReduce result (steps 3 and 4 above).                               */
/* ------------------------------------------------------------------------ */
typedef struct {
  fold_fn fold;
  int op, N;
  const void* const* xs;
  void* out;
  uint64_t lo, hi;     /* this worker's element range */
} fold_ctx;

static void fold_visit(void* ctxv, int ch, uint64_t loop, int c, uint64_t b,
                       uint64_t e) {
  (void)ch; (void)loop;
  fold_ctx* f = (fold_ctx*)ctxv;
  if (b < f->lo) b = f->lo;
  if (e > f->hi) e = f->hi;
  if (b < e) f->fold(f->op, f->N, f->xs, f->out, b, e, c);
}

typedef struct {
  fold_ctx f;
  uint64_t count;
  int nChannels, elemSize;
  uint64_t chunkBytes;
} worker_arg;

static void* worker(void* p) {
  worker_arg* w = (worker_arg*)p;
  walk_chunks(w->count, w->f.N, w->nChannels, w->elemSize, w->chunkBytes,
              fold_visit, &w->f);
  return 0;
}

/* out[i] = the ring-order reduction of xs[0..N-1][i] for every i < count.
 * The work is split over nThreads contiguous element ranges; each element is
 * still folded by exactly the steps above, so the result does not depend on
 * nThreads. Returns 0 on success, -1 on a bad argument. */
int oracle_allreduce(int dtype, int op, int N, uint64_t count, int nChannels,
                     uint64_t chunkBytes, const void* const* xs, void* out,
                     int nThreads) {
  int es = elem_size(dtype);
  fold_fn fold = fold_for(dtype);
  if (!es || !fold || op < OR_SUM || op > OR_MIN || N < 1 || nChannels < 1 ||
      chunkBytes < 16 || chunkBytes % 16 != 0)
    return -1;
  if (count == 0) return 0;
  if (nThreads < 1) nThreads = 1;
  if ((uint64_t)nThreads > count) nThreads = (int)count;
  worker_arg* args = (worker_arg*)calloc((size_t)nThreads, sizeof(worker_arg));
  pthread_t* tids = (pthread_t*)calloc((size_t)nThreads, sizeof(pthread_t));
  if (!args || !tids) { free(args); free(tids); return -1; }
  for (int t = 0; t < nThreads; ++t) {
    worker_arg* w = &args[t];
    w->f.fold = fold;
    w->f.op = op;
    w->f.N = N;
    w->f.xs = xs;
    w->f.out = out;
    w->f.lo = count / (uint64_t)nThreads * (uint64_t)t;
    w->f.hi = t == nThreads - 1 ? count : count / (uint64_t)nThreads * (uint64_t)(t + 1);
    w->count = count;
    w->nChannels = nChannels;
    w->elemSize = es;
    w->chunkBytes = chunkBytes;
  }
  int started = 0;
  for (int t = 1; t < nThreads; ++t) {
    if (pthread_create(&tids[t], 0, worker, &args[t]) != 0) break;
    started = t;
  }
  worker(&args[0]);
  for (int t = 1; t <= started; ++t) pthread_join(tids[t], 0);
  int rc = 0;
  for (int t = started + 1; t < nThreads; ++t) {  /* threads that failed to start */
    worker(&args[t]);
  }
  free(args);
  free(tids);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* The same result for selected elements only.                               */
/* ------------------------------------------------------------------------ */

/* Chunk id of element i: the channel holding i, the loop holding i inside it,
 * that loop's chunk size, and the chunk of the loop holding i (steps 1-2). */
static int chunk_of(uint64_t i, uint64_t count, int N, int nChannels, int elemSize,
                    uint64_t chunkBytes) {
  uint64_t align = 16 / (uint64_t)elemSize;
  uint64_t per = align_up(div_up(count, (uint64_t)nChannels), align);
  uint64_t ch = i / per;
  uint64_t cb = ch * per;
  uint64_t ce = cb + per < count ? cb + per : count;
  uint64_t size = ce - cb;
  uint64_t loopElems = (uint64_t)N * (chunkBytes / (uint64_t)elemSize);
  uint64_t loop = (i - cb) / loopElems;
  uint64_t off = loop * loopElems;
  uint64_t rem = size - off;
  uint64_t cur = rem < loopElems ? align_up(div_up(rem, (uint64_t)N), align)
                                 : chunkBytes / (uint64_t)elemSize;
  return (int)((i - cb - off) / cur);
}

/* For m selected element indices idx[0..m) of buffers of `count` elements:
 * vals holds the N ranks' values at those indices, rank-major (vals[r*m + j]
 * is rank r's element idx[j]); out[j] receives the reduced value of element
 * idx[j]. Returns 0, or -1 on a bad argument. */
int oracle_allreduce_at(int dtype, int op, int N, uint64_t count, int nChannels,
                        uint64_t chunkBytes, const void* vals, const uint64_t* idx,
                        uint64_t m, void* out) {
  int es = elem_size(dtype);
  fold_fn fold = fold_for(dtype);
  if (!es || !fold || op < OR_SUM || op > OR_MIN || N < 1 || nChannels < 1 ||
      chunkBytes < 16 || chunkBytes % 16 != 0)
    return -1;
  const void** xs = (const void**)calloc((size_t)N, sizeof(void*));
  if (!xs) return -1;
  for (int r = 0; r < N; ++r) xs[r] = (const char*)vals + (size_t)r * m * (size_t)es;
  int rc = 0;
  for (uint64_t j = 0; j < m; ++j) {
    if (idx[j] >= count) { rc = -1; break; }
    int c = chunk_of(idx[j], count, N, nChannels, es, chunkBytes);
    fold(op, N, xs, out, j, j + 1, c);
  }
  free(xs);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* ReduceScatter and AllGather, the two halves of the ring.                  */
/* ------------------------------------------------------------------------ */

/* ReduceScatter: rank k's send buffer holds N blocks of recvcount elements;
 * rank b receives the reduction of block b over all ranks. The ring
 * reduce-scatter of "NCCL 原始碼解讀：一個 AllReduce 的 GPU 旅程", ch.2 §2.3
 * (the first (N-1)·chunkSteps steps of nStepsPerLoop, the rank sending at
 * stage s the block (ringIndex + N - 1 - s) mod N) starts block b at rank
 * b+1 and completes it at rank b, so its fold is
 *     acc = x[b+1]; acc = op(acc, x[b+2]); ... ; acc = op(acc, x[b])
 * over block b, whatever the channel and chunk split. outs[b] receives it. */
int oracle_reduce_scatter(int dtype, int op, int N, uint64_t recvcount, const void* const* xs,
                          void* const* outs) {
  int es = elem_size(dtype);
  fold_fn fold = fold_for(dtype);
  if (!es || !fold || op < OR_SUM || op > OR_MIN || N < 1) return -1;
  const void** blk = (const void**)calloc((size_t)N, sizeof(void*));
  if (!blk) return -1;
  for (int b = 0; b < N; ++b) {
    for (int k = 0; k < N; ++k)
      blk[k] = (const char*)xs[k] + (size_t)b * recvcount * (size_t)es;
    /* the fold of "chunk" b over the N views of block b */
    fold(op, N, blk, outs[b], 0, recvcount, b);
  }
  free(blk);
  return 0;
}

/* AllGather: rank b's receive buffer holds the N send buffers of sendcount
 * elements, block k = rank k's buffer (a copy; the type only sets the size). */
int oracle_all_gather(int elemSize, int N, uint64_t sendcount, const void* const* xs,
                      void* const* outs) {
  if (elemSize < 1 || N < 1) return -1;
  const size_t bytes = (size_t)sendcount * (size_t)elemSize;
  for (int b = 0; b < N; ++b)
    for (int k = 0; k < N; ++k)
      memcpy((char*)outs[b] + (size_t)k * bytes, xs[k], bytes);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Double binary tree AllReduce.                                             */
/* ------------------------------------------------------------------------ */
/* The tree of "NCCL 原始碼解讀：一個 AllReduce 的 GPU 旅程", ch.4
 * (ncclGetBtree), as a rule on rank numbers: rank 0 is the root and its one
 * child is the largest power of two below N; any other rank r, with b its
 * lowest set bit, has the parent "r with bit b cleared and bit 2b set", or
 * r - b when that is out of range, and the children r - b/2 and r + b/2 (the
 * second one, while out of
 * range, moved to r + b/4, r + b/8, ...; none once the step reaches 0). The
 * second tree (ncclGetDtree) is the mirror image r -> N - 1 - r of the first
 * for even N and, for odd N, the first tree on ranks shifted by one
 * (r -> r - 1 mod N; reading taken for the elided part of the listing: the
 * ranks the first tree gives are shifted back by + 1 mod N). Each tree
 * reduces half of the buffer ("NCCL 初始化流程源码级剖析", NCCL Tree 拓扑,
 * Double Binary Tree: the first half of the elements on tree 1, the rest on
 * tree 2): reduce from the leaves to the root -- a node reduces the data its
 * children send with its own -- then broadcast from the root. */
static void btree_node(int N, int r, int* up, int* d0, int* d1) {
  if (r == 0) {
    int p = 1;
    while (p < N) p <<= 1;
    *up = -1;
    *d0 = -1;
    *d1 = N > 1 ? p >> 1 : -1;
    return;
  }
  int b = 1;
  while (!(r & b)) b <<= 1;
  int parent = (r - b) | (2 * b);
  if (parent >= N) parent = r - b;
  *up = parent;
  int step = b >> 1;
  *d0 = step ? r - step : -1;
  while (step && r + step >= N) step >>= 1;
  *d1 = step ? r + step : -1;
}

/* Parent and children of rank r in tree `tree` (0 or 1); -1 where none. */
void oracle_tree_node(int N, int r, int tree, int* up, int* d0, int* d1) {
  if (tree == 0) {
    btree_node(N, r, up, d0, d1);
    return;
  }
  int u, a, b;
  if (N % 2 == 0) {
    btree_node(N, N - 1 - r, &u, &a, &b);
    *up = u < 0 ? -1 : N - 1 - u;
    *d0 = a < 0 ? -1 : N - 1 - a;
    *d1 = b < 0 ? -1 : N - 1 - b;
  } else {
    btree_node(N, (r - 1 + N) % N, &u, &a, &b);
    *up = u < 0 ? -1 : (u + 1) % N;
    *d0 = a < 0 ? -1 : (a + 1) % N;
    *d1 = b < 0 ? -1 : (b + 1) % N;
  }
}

/* First element of the second tree's half: half the buffer rounded up to
 * 16 bytes of elements (the same rounding as the ring's channel split). */
uint64_t oracle_tree_split(uint64_t count, int elemSize) {
  uint64_t h = align_up(div_up(count, 2), 16 / (uint64_t)elemSize);
  return h < count ? h : count;
}

/* The reduction of one element by tree `tree`: a node's value is its own
 * element, then op(value, value of child d0), then op(value, value of child
 * d1) for the children it has (reading taken: own first, then the children
 * in the order the tree names them), rounded to the element type at every op
 * because values travel between ranks in that type. Nodes are visited so
 * that every child comes before its parent (`order`, children-first). */
#define DEFINE_TREE_FOLD(NAME, T, COMBINE)                                                 \
  static void NAME(int op, int N, const void* const* xs, void* outv, uint64_t b,          \
                   uint64_t e, const int* order, const int* d0, const int* d1, T* val) {  \
    T* out = (T*)outv;                                                                     \
    for (uint64_t i = b; i < e; ++i) {                                                     \
      for (int k = 0; k < N; ++k) {                                                        \
        int r = order[k];                                                                  \
        T acc = ((const T*)xs[r])[i];                                                      \
        if (d0[r] >= 0) acc = COMBINE(op, acc, val[d0[r]]);                                \
        if (d1[r] >= 0) acc = COMBINE(op, acc, val[d1[r]]);                                \
        val[r] = acc;                                                                      \
      }                                                                                    \
      out[i] = val[order[N - 1]];                                                          \
    }                                                                                      \
  }
DEFINE_TREE_FOLD(tfold_i8, int8_t, combine_i8)
DEFINE_TREE_FOLD(tfold_u8, uint8_t, combine_u8)
DEFINE_TREE_FOLD(tfold_i32, int32_t, combine_i32)
DEFINE_TREE_FOLD(tfold_u32, uint32_t, combine_u32)
DEFINE_TREE_FOLD(tfold_i64, int64_t, combine_i64)
DEFINE_TREE_FOLD(tfold_u64, uint64_t, combine_u64)
DEFINE_TREE_FOLD(tfold_f16, uint16_t, combine_f16)
DEFINE_TREE_FOLD(tfold_bf16, uint16_t, combine_bf16)
DEFINE_TREE_FOLD(tfold_f32, float, combine_f32)
DEFINE_TREE_FOLD(tfold_f64, double, combine_f64)
DEFINE_TREE_FOLD(tfold_e4m3, uint8_t, combine_e4m3)
DEFINE_TREE_FOLD(tfold_e5m2, uint8_t, combine_e5m2)

/* Children-first order of tree `tree`: a node after all its descendants,
 * the root last. Returns 0, or -1 if the rule does not give one tree. */
static int tree_order(int N, int tree, int* order, int* d0, int* d1) {
  int* up = (int*)malloc((size_t)N * sizeof(int));
  int* stack = (int*)malloc((size_t)N * 2 * sizeof(int));
  int root = -1, n = 0, top = 0, rc = 0;
  if (!up || !stack) {
    free(up);
    free(stack);
    return -1;
  }
  for (int r = 0; r < N; ++r) {
    oracle_tree_node(N, r, tree, &up[r], &d0[r], &d1[r]);
    if (up[r] < 0) root = r;
  }
  /* iterative post-order from the root */
  if (root >= 0) {
    stack[top++] = root;
    stack[top++] = 0;
  }
  while (top > 0) {
    int state = stack[--top], r = stack[--top];
    if (state == 0) {
      stack[top++] = r;
      stack[top++] = 1;
      if (d1[r] >= 0) { stack[top++] = d1[r]; stack[top++] = 0; }
      if (d0[r] >= 0) { stack[top++] = d0[r]; stack[top++] = 0; }
      if (top > 2 * N) { rc = -1; break; }
    } else {
      if (n >= N) { rc = -1; break; }
      order[n++] = r;
    }
  }
  if (n != N) rc = -1;
  free(up);
  free(stack);
  return rc;
}

int oracle_tree_allreduce(int dtype, int op, int N, uint64_t count, const void* const* xs,
                          void* out) {
  int es = elem_size(dtype);
  if (!es || op < OR_SUM || op > OR_MIN || N < 1) return -1;
  int* order = (int*)malloc((size_t)N * 3 * sizeof(int));
  void* val = malloc((size_t)N * 8);
  if (!order || !val) {
    free(order);
    free(val);
    return -1;
  }
  int* d0 = order + N;
  int* d1 = order + 2 * N;
  const uint64_t h = oracle_tree_split(count, es);
  int rc = 0;
  for (int tree = 0; tree < 2 && rc == 0; ++tree) {
    const uint64_t b = tree == 0 ? 0 : h, e = tree == 0 ? h : count;
    if (tree_order(N, tree, order, d0, d1) != 0) {
      rc = -1;
      break;
    }
    switch (dtype) {
      case OR_INT8: tfold_i8(op, N, xs, out, b, e, order, d0, d1, (int8_t*)val); break;
      case OR_UINT8: tfold_u8(op, N, xs, out, b, e, order, d0, d1, (uint8_t*)val); break;
      case OR_INT32: tfold_i32(op, N, xs, out, b, e, order, d0, d1, (int32_t*)val); break;
      case OR_UINT32: tfold_u32(op, N, xs, out, b, e, order, d0, d1, (uint32_t*)val); break;
      case OR_INT64: tfold_i64(op, N, xs, out, b, e, order, d0, d1, (int64_t*)val); break;
      case OR_UINT64: tfold_u64(op, N, xs, out, b, e, order, d0, d1, (uint64_t*)val); break;
      case OR_FLOAT16: tfold_f16(op, N, xs, out, b, e, order, d0, d1, (uint16_t*)val); break;
      case OR_BFLOAT16: tfold_bf16(op, N, xs, out, b, e, order, d0, d1, (uint16_t*)val); break;
      case OR_FLOAT32: tfold_f32(op, N, xs, out, b, e, order, d0, d1, (float*)val); break;
      case OR_FP8E4M3: tfold_e4m3(op, N, xs, out, b, e, order, d0, d1, (uint8_t*)val); break;
      case OR_FP8E5M2: tfold_e5m2(op, N, xs, out, b, e, order, d0, d1, (uint8_t*)val); break;
      default: tfold_f64(op, N, xs, out, b, e, order, d0, d1, (double*)val); break;
    }
  }
  free(order);
  free(val);
  return rc;
}


/* ------------------------------------------------------------------------ */
/* Average and pre-multiplied sum.                                           */
/* ------------------------------------------------------------------------ */
/* NCCL's host-to-device op conversion ("NCCL 原始碼解讀", ch.6, hostToDevRedOp)
 * turns the average and the user's pre-multiplied sum into sums. Readings
 * taken (the pages name the step, not the rules): a pre-multiplied sum with
 * scalar s multiplies every rank's element by s (s and the product rounded to
 * the element type; integers wrap) as it enters the ring's fold, which is then
 * the sum's; the average is that with s = 1/N for floating types, and for
 * integer types the sum's result divided by N (C division, truncating toward
 * zero). kind 0: pre-multiplied sum by `scalar` (floating types) or
 * `iscalar` (integer types); kind 1: average. ReduceScatter likewise
 * (coll 1: xs hold N blocks of `count` / N elements). */
static int scaled_inputs(int dtype, double scalar, int64_t iscalar, int N, uint64_t count,
                         const void* const* xs, void** ys) {
  const int es = elem_size(dtype);
  for (int r = 0; r < N; ++r) {
    ys[r] = malloc((size_t)(count ? count : 1) * (size_t)es);
    if (!ys[r]) return -1;
  }
  for (int r = 0; r < N; ++r) {
    for (uint64_t i = 0; i < count; ++i) {
      switch (dtype) {
#define PREMUL_INT(CODE, T, FN)                                                      \
        case CODE: ((T*)ys[r])[i] = FN(OR_PROD, ((const T*)xs[r])[i], (T)iscalar); break;
        PREMUL_INT(OR_INT8, int8_t, combine_i8)
        PREMUL_INT(OR_UINT8, uint8_t, combine_u8)
        PREMUL_INT(OR_INT32, int32_t, combine_i32)
        PREMUL_INT(OR_UINT32, uint32_t, combine_u32)
        PREMUL_INT(OR_INT64, int64_t, combine_i64)
        PREMUL_INT(OR_UINT64, uint64_t, combine_u64)
#undef PREMUL_INT
        case OR_FLOAT16:
          ((uint16_t*)ys[r])[i] = combine_f16(OR_PROD, ((const uint16_t*)xs[r])[i],
                                              oracle_f16_from_double(scalar));
          break;
        case OR_BFLOAT16:
          ((uint16_t*)ys[r])[i] = combine_bf16(OR_PROD, ((const uint16_t*)xs[r])[i],
                                               oracle_bf16_from_double(scalar));
          break;
        case OR_FLOAT32:
          ((float*)ys[r])[i] = combine_f32(OR_PROD, ((const float*)xs[r])[i], (float)scalar);
          break;
        case OR_FP8E4M3:
          ((uint8_t*)ys[r])[i] = combine_e4m3(OR_PROD, ((const uint8_t*)xs[r])[i],
                                              oracle_fp8e4m3_from_double(scalar));
          break;
        case OR_FP8E5M2:
          ((uint8_t*)ys[r])[i] = combine_e5m2(OR_PROD, ((const uint8_t*)xs[r])[i],
                                              oracle_fp8e5m2_from_double(scalar));
          break;
        default:
          ((double*)ys[r])[i] = combine_f64(OR_PROD, ((const double*)xs[r])[i], scalar);
          break;
      }
    }
  }
  return 0;
}

static int is_float_type(int dtype) {
  return dtype == OR_FLOAT16 || dtype == OR_BFLOAT16 || dtype == OR_FLOAT32 ||
         dtype == OR_FLOAT64 || dtype == OR_FP8E4M3 || dtype == OR_FP8E5M2;
}

/* Divide every element of the outputs' first `count` elements by N
 * (integer types only). */
static void divide_by_n(int dtype, int N, uint64_t count, void* const* outs, int nOut) {
  if (is_float_type(dtype)) return;
  for (int o = 0; o < nOut; ++o) {
    for (uint64_t i = 0; i < count; ++i) {
      switch (dtype) {
        case OR_INT8: ((int8_t*)outs[o])[i] = (int8_t)(((int8_t*)outs[o])[i] / N); break;
        case OR_UINT8: ((uint8_t*)outs[o])[i] = (uint8_t)(((uint8_t*)outs[o])[i] / (unsigned)N); break;
        case OR_INT32: ((int32_t*)outs[o])[i] = ((int32_t*)outs[o])[i] / N; break;
        case OR_UINT32: ((uint32_t*)outs[o])[i] = ((uint32_t*)outs[o])[i] / (uint32_t)N; break;
        case OR_INT64: ((int64_t*)outs[o])[i] = ((int64_t*)outs[o])[i] / N; break;
        default: ((uint64_t*)outs[o])[i] = ((uint64_t*)outs[o])[i] / (uint64_t)N; break;
      }
    }
  }
}

int oracle_allreduce_scaled(int dtype, int kind, double scalar, int64_t iscalar, int coll, int N,
                            uint64_t count, int nChannels, uint64_t chunkBytes,
                            const void* const* xs, void* const* outs, int nThreads) {
  const int es = elem_size(dtype);
  if (!es || N < 1 || (kind != 0 && kind != 1) || (coll != 0 && coll != 1)) return -1;
  const int premul = kind == 0 || is_float_type(dtype);
  const double s = kind == 0 ? scalar : 1.0 / (double)N;
  const int64_t is = kind == 0 ? iscalar : 1;
  void** ys = (void**)calloc((size_t)N, sizeof(void*));
  if (!ys) return -1;
  int rc = 0;
  if (premul) rc = scaled_inputs(dtype, s, is, N, count, xs, ys);
  const void* const* in = premul ? (const void* const*)ys : xs;
  if (rc == 0) {
    if (coll == 0)
      rc = oracle_allreduce(dtype, OR_SUM, N, count, nChannels, chunkBytes, in, outs[0],
                            nThreads);
    else
      rc = oracle_reduce_scatter(dtype, OR_SUM, N, N ? count / (uint64_t)N : 0, in, outs);
  }
  if (rc == 0 && !premul)
    divide_by_n(dtype, N, coll == 0 ? count : count / (uint64_t)N, outs, coll == 0 ? 1 : N);
  for (int r = 0; r < N; ++r) free(ys[r]);
  free(ys);
  return rc;
}

/* The double-binary-tree AllReduce with the average or a pre-multiplied sum:
 * the same reading of the host-to-device op conversion as above (every
 * rank's element times s before the tree's fold, which is then the sum's; the
 * integer average divides the tree's wrapped sum by N, toward zero). */
int oracle_tree_allreduce_scaled(int dtype, int kind, double scalar, int64_t iscalar, int N,
                                 uint64_t count, const void* const* xs, void* out) {
  const int es = elem_size(dtype);
  if (!es || N < 1 || (kind != 0 && kind != 1)) return -1;
  const int premul = kind == 0 || is_float_type(dtype);
  const double s = kind == 0 ? scalar : 1.0 / (double)N;
  const int64_t is = kind == 0 ? iscalar : 1;
  void** ys = (void**)calloc((size_t)N, sizeof(void*));
  if (!ys) return -1;
  int rc = 0;
  if (premul) rc = scaled_inputs(dtype, s, is, N, count, xs, ys);
  if (rc == 0)
    rc = oracle_tree_allreduce(dtype, OR_SUM, N, count,
                               premul ? (const void* const*)ys : xs, out);
  if (rc == 0 && !premul) {
    void* outs[1] = {out};
    divide_by_n(dtype, N, count, outs, 1);
  }
  for (int r = 0; r < N; ++r) free(ys[r]);
  free(ys);
  return rc;
}
