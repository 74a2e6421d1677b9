// Device helpers shared by the verification kernels: workspace layout,
// element unpacking, the online softmax / argmax accumulators, and thin
// inline-PTX wrappers for mbarriers and bulk (TMA) copies on sm_103a.
#pragma once

#include <cuda_runtime.h>
#include <float.h>
#include <stdint.h>

#include "spec_verify.h"

namespace specv {

// ---------------------------------------------------------------------------
// Constants
// ---------------------------------------------------------------------------

constexpr float kLog2e = 1.4426950408889634f;  // log2(e): exp(x) = 2^(x log2 e)
constexpr float kLn2f = 0.693147180559945309f;  // ln 2

// Sweep kernel geometry.
constexpr int kSweepConsumerWarps = 8;
// + one producer warp (lane 0 issues the bulk copies) + one bookkeeping warp
// (unit partials, completion counters, accept decisions).
constexpr int kSweepThreads = (kSweepConsumerWarps + 2) * 32;
constexpr int kStageBytes = 16384;
constexpr int kStages = 4;
constexpr int kSweepMinBlocks = 3;  // CTAs per SM the register budget is sized for
constexpr int kRedDepth = 8;  // unit-end reduction slots in flight

// Final-pass kernel geometry.
constexpr int kFinalThreads = 256;
constexpr int kSegElems = 256;  // one warp x 8 elements
constexpr int kMaxSegs = SPEC_MAX_V / kSegElems;
constexpr int kMaxSlices = 64;  // CTAs that share one request's final row(s)

// Bounded waits: give up after this many nanoseconds of spinning.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// ---------------------------------------------------------------------------
// Workspace layout (all offsets 256-byte aligned).  The header is written by
// the plan kernel and read back by spec_verify_report().
// ---------------------------------------------------------------------------

struct WsHeader {
  int32_t status;
  int32_t bad_requests;
  int32_t first_bad;
  int32_t rows_planned;
  int32_t units_total;
  int32_t work_next;
  int32_t chunks_per_row;
  int32_t chunk_elems;
  unsigned long long chunks_swept;
  unsigned long long final_rows;
  int32_t residual_zero;
  int32_t pad0;
  unsigned long long sweep_bytes;
  unsigned long long final_bytes;
  int32_t sweep_exited;     // sweep CTAs that have finished
  int32_t final_ctas_done;  // final-pass CTAs that have finished
  int32_t row_kinds;        // rows in the sweep's list: 1 greedy, 2 sampling (bits)
  int32_t pad[43];
};
static_assert(sizeof(WsHeader) == 256, "header is one 256-byte block");

// Per-unit partial result of the sweep: softmax (m, s) or argmax (m, arg).
// One 8-byte word, written and read in a single access, so that a reader on
// another SM sees either the whole partial or the empty marker.
struct __align__(8) Partial {
  float m;       // largest logit of the chunk
  uint32_t aux;  // sampling rows: bits of s = sum 2^(z*sc - fl(m*sc)); greedy rows: lowest index of m
};
// What a partial slot holds from the plan kernel until its unit is stored: m
// is a NaN, which no chunk max can be (max-reductions skip NaN logits).
constexpr unsigned long long kPartialEmpty = 0x7FC0DEAD7FC0DEADull;

struct WsLayout {
  size_t header, rowdesc, flags, first_reject, state, bad_bits, done, pos_c, pos_arg,
      partials, seg_mass, slice_out, final_done, rowbase, warm, total;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Vocabulary chunks per row: at least two (so that the last units of a round
// are short and a rejection found while a row streams spares its second
// half), more only for the smallest batches (about 256 units when all rows
// are active: 8 chunks for one request of 16 positions), chunks of at least
// 2048 elements.  Larger units cost more at the end of a round and in bytes
// read past a rejection; smaller ones cost per-unit claims and bookkeeping,
// which is what set the small-batch rounds (measured on GB300 with 1 to 256
// requests of 151936 logits: 2048 units made the 1-request round 41.5 us,
// 256 make it 28 us).
__host__ __device__ inline int chunks_per_row(long long rows_max, int V) {
  long long want = (256 + rows_max - 1) / rows_max;
  if (want < 2) want = 2;
  long long maxc = (V + 2047) / 2048;
  if (maxc < 1) maxc = 1;
  if (want > maxc) want = maxc;
  if (want < 1) want = 1;
  return (int)want;
}

// Elements per chunk: a multiple of 8 so chunk starts keep 16-byte alignment.
__host__ __device__ inline int chunk_elems_for(int V, int C) {
  int e = (V + C - 1) / C;
  return (e + 7) & ~7;
}

__host__ __device__ inline int segments_of(int V) { return (V + kSegElems - 1) / kSegElems; }

__host__ __device__ inline WsLayout ws_layout(int B, int k, int C, int V) {
  WsLayout l;
  size_t o = 0;
  size_t slots = (size_t)B * (size_t)k * 2;
  l.header = o;       o = align256(o + sizeof(WsHeader));
  l.rowdesc = o;      o = align256(o + slots * sizeof(int4));
  l.flags = o;        o = align256(o + (size_t)B * sizeof(int32_t));
  l.first_reject = o; o = align256(o + (size_t)B * sizeof(int32_t));
  l.state = o;        o = align256(o + (size_t)B * sizeof(unsigned long long));
  l.bad_bits = o;     o = align256(o + (size_t)B * sizeof(uint32_t));
  l.done = o;         o = align256(o + (size_t)B * k * sizeof(int32_t));
  l.pos_c = o;        o = align256(o + (size_t)B * k * sizeof(float4));
  l.pos_arg = o;      o = align256(o + (size_t)B * k * sizeof(int32_t));
  l.partials = o;     o = align256(o + slots * (size_t)C * sizeof(Partial));
  l.seg_mass = o;     o = align256(o + (size_t)B * segments_of(V) * sizeof(float2));
  l.slice_out = o;    o = align256(o + (size_t)B * kMaxSlices * sizeof(float2));
  l.final_done = o;   o = align256(o + (size_t)B * sizeof(int32_t));
  l.rowbase = o;      o = align256(o + (size_t)B * sizeof(int2));
  l.warm = o;         o = align256(o + 2 * (size_t)C * sizeof(Partial));
  l.total = o;
  return l;
}

// Request flags written by the plan kernel.
constexpr int kReqValid = 1;
constexpr int kReqGreedy = 2;

// ---------------------------------------------------------------------------
// Elements
// ---------------------------------------------------------------------------

__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

template <typename TIn>
struct ElemTraits;
template <>
struct ElemTraits<float> {
  static constexpr int kSize = 4;
  static constexpr int kPerVec = 4;  // elements per 16-byte vector
  static __device__ __forceinline__ float load(const float* p, long long i) { return __ldg(p + i); }
  static __device__ __forceinline__ float to_float(float x) { return x; }
  static __device__ __forceinline__ void unpack(const uint4& v, float* x) {
    x[0] = __uint_as_float(v.x);
    x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z);
    x[3] = __uint_as_float(v.w);
  }
};
template <>
struct ElemTraits<uint16_t> {
  static constexpr int kSize = 2;
  static constexpr int kPerVec = 8;
  static __device__ __forceinline__ float load(const uint16_t* p, long long i) {
    return bf16_to_f32(__ldg(p + i));
  }
  static __device__ __forceinline__ float to_float(uint16_t x) { return bf16_to_f32(x); }
  static __device__ __forceinline__ void unpack(const uint4& v, float* x) {
    x[0] = __uint_as_float(v.x << 16);
    x[1] = __uint_as_float(v.x & 0xffff0000u);
    x[2] = __uint_as_float(v.y << 16);
    x[3] = __uint_as_float(v.y & 0xffff0000u);
    x[4] = __uint_as_float(v.z << 16);
    x[5] = __uint_as_float(v.z & 0xffff0000u);
    x[6] = __uint_as_float(v.w << 16);
    x[7] = __uint_as_float(v.w & 0xffff0000u);
  }
};

// ---------------------------------------------------------------------------
// Scalar math
// ---------------------------------------------------------------------------

// 2^x on the special-function unit (relative error about 2^-22; subnormal
// results flush to zero, which only drops terms below 2^-126 of the max).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Scale that turns a logit into base-2 log-probability units: log2(e) / T.
// Every kernel derives it with this one function so that all of them work
// with bit-identical values.
__device__ __forceinline__ float softmax_scale(float T) { return __fdiv_rn(kLog2e, T); }

// A temperature the kernels accept: 0 (greedy) or a finite normal float.
__device__ __forceinline__ bool temperature_ok(float T) {
  return T == 0.0f || (T >= FLT_MIN && T <= FLT_MAX);
}

// ---------------------------------------------------------------------------
// Accumulators.  SoftAcc holds a running max m, ms = fl(m*sc) and
// s = sum 2^(z*sc - ms); merges rescale by 2^(ms_old - ms_new).  ArgAcc
// keeps the largest value and its lowest index.
// ---------------------------------------------------------------------------

struct SoftAcc {
  float m, ms, s;
};

__device__ __forceinline__ void soft_init(SoftAcc& a) {
  a.m = -FLT_MAX;
  a.ms = -FLT_MAX;
  a.s = 0.0f;
}

template <int N>
__device__ __forceinline__ void soft_add(SoftAcc& a, const float* x, float sc) {
  float gm = x[0];
#pragma unroll
  for (int e = 1; e < N; ++e) gm = fmaxf(gm, x[e]);
  if (gm > a.m) {
    float nms = __fmul_rn(gm, sc);
    a.s = __fmul_rn(a.s, ex2(__fsub_rn(a.ms, nms)));
    a.m = gm;
    a.ms = nms;
  }
  float t = 0.0f;
#pragma unroll
  for (int e = 0; e < N; ++e) t = __fadd_rn(t, ex2(fmaf(x[e], sc, -a.ms)));
  a.s = __fadd_rn(a.s, t);
}

__device__ __forceinline__ void soft_add1(SoftAcc& a, float x, float sc) { soft_add<1>(a, &x, sc); }

// Packed two-lane arithmetic (bf16x2 max; f32x2 FMA / add, sm_100 and later):
// one instruction does the work of two.
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ float2 f32x2_fma(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float2 f32x2_add(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float2 f32x2_mul(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float2 ex2x2(float2 y) { return make_float2(ex2(y.x), ex2(y.y)); }

// Fold one 16-byte vector of logits into a softmax accumulator: packed max
// to find a new running max, packed FMA for z*sc - ms, one ex2 per element,
// packed pairwise sums.
template <typename TIn>
__device__ __forceinline__ void soft_add_vec(SoftAcc& a, const uint4& v, float sc);

template <>
__device__ __forceinline__ void soft_add_vec<uint16_t>(SoftAcc& a, const uint4& v, float sc) {
  const uint32_t mx = bf16x2_max(bf16x2_max(v.x, v.y), bf16x2_max(v.z, v.w));
  const float gm = fmaxf(__uint_as_float(mx << 16), __uint_as_float(mx & 0xffff0000u));
  if (gm > a.m) {
    const float nms = __fmul_rn(gm, sc);
    a.s = __fmul_rn(a.s, ex2(__fsub_rn(a.ms, nms)));
    a.m = gm;
    a.ms = nms;
  }
  const float2 s2 = make_float2(sc, sc), c2 = make_float2(-a.ms, -a.ms);
  const float2 e0 = ex2x2(f32x2_fma(
      make_float2(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u)), s2, c2));
  const float2 e1 = ex2x2(f32x2_fma(
      make_float2(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u)), s2, c2));
  const float2 e2 = ex2x2(f32x2_fma(
      make_float2(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xffff0000u)), s2, c2));
  const float2 e3 = ex2x2(f32x2_fma(
      make_float2(__uint_as_float(v.w << 16), __uint_as_float(v.w & 0xffff0000u)), s2, c2));
  const float2 t = f32x2_add(f32x2_add(e0, e1), f32x2_add(e2, e3));
  a.s = __fadd_rn(a.s, __fadd_rn(t.x, t.y));
}

template <>
__device__ __forceinline__ void soft_add_vec<float>(SoftAcc& a, const uint4& v, float sc) {
  const float x0 = __uint_as_float(v.x), x1 = __uint_as_float(v.y);
  const float x2 = __uint_as_float(v.z), x3 = __uint_as_float(v.w);
  const float gm = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
  if (gm > a.m) {
    const float nms = __fmul_rn(gm, sc);
    a.s = __fmul_rn(a.s, ex2(__fsub_rn(a.ms, nms)));
    a.m = gm;
    a.ms = nms;
  }
  const float2 s2 = make_float2(sc, sc), c2 = make_float2(-a.ms, -a.ms);
  const float2 e0 = ex2x2(f32x2_fma(make_float2(x0, x1), s2, c2));
  const float2 e1 = ex2x2(f32x2_fma(make_float2(x2, x3), s2, c2));
  const float2 t = f32x2_add(e0, e1);
  a.s = __fadd_rn(a.s, __fadd_rn(t.x, t.y));
}

__device__ __forceinline__ void soft_merge(SoftAcc& a, const SoftAcc& b) {
  if (b.m > a.m) {
    a.s = __fadd_rn(__fmul_rn(a.s, ex2(__fsub_rn(a.ms, b.ms))), b.s);
    a.m = b.m;
    a.ms = b.ms;
  } else {
    a.s = __fadd_rn(a.s, __fmul_rn(b.s, ex2(__fsub_rn(b.ms, a.ms))));
  }
}

__device__ __forceinline__ SoftAcc soft_shfl_xor(const SoftAcc& a, int mask) {
  SoftAcc b;
  b.m = __shfl_xor_sync(0xffffffffu, a.m, mask);
  b.ms = __shfl_xor_sync(0xffffffffu, a.ms, mask);
  b.s = __shfl_xor_sync(0xffffffffu, a.s, mask);
  return b;
}

__device__ __forceinline__ void soft_warp_reduce(SoftAcc& a) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    SoftAcc b = soft_shfl_xor(a, off);
    // Merge in a fixed lane order so that every lane ends with the same bits.
    int lane = threadIdx.x & 31;
    if (lane & off) {
      SoftAcc t = b;
      soft_merge(t, a);
      a = t;
    } else {
      soft_merge(a, b);
    }
  }
}

struct ArgAcc {
  float v;
  int i;
};

__device__ __forceinline__ void arg_init(ArgAcc& a) {
  a.v = -INFINITY;
  a.i = INT32_MAX;
}

// ---------------------------------------------------------------------------
// One consumer thread's batch of a stage: N 16-byte vectors of one row held
// in registers.  Vectors past the stage's end are -inf in every element, so
// they change neither a max nor a sum of exponentials.
// ---------------------------------------------------------------------------
template <typename TIn>
__device__ __forceinline__ uint4 neg_inf_vec() {
  const uint32_t w = sizeof(TIn) == 2 ? 0xFF80FF80u : 0xFF800000u;
  return make_uint4(w, w, w, w);
}

// Largest element of the batch.
template <typename TIn, int N>
__device__ __forceinline__ float batch_max(const uint4 (&v)[N]) {
  static_assert((N & (N - 1)) == 0, "batch_max reduces a power-of-two batch");
  if constexpr (sizeof(TIn) == 2) {
    uint32_t m[N];
#pragma unroll
    for (int t = 0; t < N; ++t)
      m[t] = bf16x2_max(bf16x2_max(v[t].x, v[t].y), bf16x2_max(v[t].z, v[t].w));
#pragma unroll
    for (int w = N / 2; w > 0; w >>= 1)
#pragma unroll
      for (int t = 0; t < w; ++t) m[t] = bf16x2_max(m[t], m[t + w]);
    return fmaxf(__uint_as_float(m[0] << 16), __uint_as_float(m[0] & 0xffff0000u));
  } else {
    float m[N];
#pragma unroll
    for (int t = 0; t < N; ++t)
      m[t] = fmaxf(fmaxf(__uint_as_float(v[t].x), __uint_as_float(v[t].y)),
                   fmaxf(__uint_as_float(v[t].z), __uint_as_float(v[t].w)));
#pragma unroll
    for (int w = N / 2; w > 0; w >>= 1)
#pragma unroll
      for (int t = 0; t < w; ++t) m[t] = fmaxf(m[t], m[t + w]);
    return m[0];
  }
}

// Element e (in index order) of one vector.
template <typename TIn>
__device__ __forceinline__ float vec_elem(const uint4& v, int e) {
  const uint32_t w = e < ElemTraits<TIn>::kPerVec / 2
                         ? (e < ElemTraits<TIn>::kPerVec / 4 ? v.x : v.y)
                         : (e < 3 * ElemTraits<TIn>::kPerVec / 4 ? v.z : v.w);
  if (ElemTraits<TIn>::kPerVec == 4) return __uint_as_float(w);
  return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
}

// Softmax accumulation of a batch: one max, at most one rescale, then
// independent packed FMAs, one ex2 per element and four packed accumulators.
template <typename TIn, int N>
__device__ __forceinline__ void soft_stage(SoftAcc& a, const uint4 (&v)[N], float sc,
                                           float gm) {
  if (gm > a.m) {
    const float nms = __fmul_rn(gm, sc);
    a.s = __fmul_rn(a.s, ex2(__fsub_rn(a.ms, nms)));
    a.m = gm;
    a.ms = nms;
  }
  const float2 s2 = make_float2(sc, sc), c2 = make_float2(-a.ms, -a.ms);
  float2 acc[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) acc[q] = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int t = 0; t < N; ++t) {
    const uint32_t w[4] = {v[t].x, v[t].y, v[t].z, v[t].w};
    if (ElemTraits<TIn>::kPerVec == 8) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 z = make_float2(__uint_as_float(w[q] << 16), __uint_as_float(w[q] & 0xffff0000u));
        acc[q] = f32x2_add(acc[q], ex2x2(f32x2_fma(z, s2, c2)));
      }
    } else {
      const int q0 = (t & 1) * 2;
      acc[q0] = f32x2_add(acc[q0], ex2x2(f32x2_fma(make_float2(__uint_as_float(w[0]), __uint_as_float(w[1])), s2, c2)));
      acc[q0 + 1] = f32x2_add(acc[q0 + 1], ex2x2(f32x2_fma(make_float2(__uint_as_float(w[2]), __uint_as_float(w[3])), s2, c2)));
    }
  }
  const float2 t2 = f32x2_add(f32x2_add(acc[0], acc[1]), f32x2_add(acc[2], acc[3]));
  a.s = __fadd_rn(a.s, __fadd_rn(t2.x, t2.y));
}

// The same with the batch's max computed here.
template <typename TIn, int N>
__device__ __forceinline__ void soft_stage(SoftAcc& a, const uint4 (&v)[N], float sc) {
  soft_stage<TIn>(a, v, sc, batch_max<TIn>(v));
}

// Argmax of a batch: one max; only when it beats the running best, a scan in
// index order for its first occurrence.  `first` is the element index of
// vector 0, vectors are `stride` elements apart.
template <typename TIn, int N>
__device__ __forceinline__ void arg_stage(ArgAcc& a, const uint4 (&v)[N], int first, int stride,
                                          float gm) {
  constexpr int EPV = ElemTraits<TIn>::kPerVec;
  if (!(gm > a.v)) return;
  // The first vector whose max is gm (its elements come before the next
  // vector's), then its first element equal to gm: the lowest index.
  int t_hit = -1;
#pragma unroll
  for (int t = N - 1; t >= 0; --t) {
    const uint4 one[1] = {v[t]};
    if (batch_max<TIn>(one) == gm) t_hit = t;
  }
  uint4 w = v[0];
#pragma unroll
  for (int t = 1; t < N; ++t)
    if (t == t_hit) w = v[t];
  int e_hit = 0;
#pragma unroll
  for (int e = EPV - 1; e >= 0; --e)
    if (vec_elem<TIn>(w, e) == gm) e_hit = e;
  a.v = gm;
  a.i = t_hit >= 0 ? first + t_hit * stride + e_hit : INT32_MAX;
}

template <typename TIn, int N>
__device__ __forceinline__ void arg_stage(ArgAcc& a, const uint4 (&v)[N], int first, int stride) {
  arg_stage<TIn>(a, v, first, stride, batch_max<TIn>(v));
}

// Elements must be offered in increasing index order within one accumulator.
__device__ __forceinline__ void arg_add(ArgAcc& a, float x, int idx) {
  if (x > a.v) {
    a.v = x;
    a.i = idx;
  }
}

__device__ __forceinline__ void arg_merge(ArgAcc& a, const ArgAcc& b) {
  if (b.v > a.v || (b.v == a.v && b.i < a.i)) a = b;
}

__device__ __forceinline__ void arg_warp_reduce(ArgAcc& a) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    ArgAcc b;
    b.v = __shfl_xor_sync(0xffffffffu, a.v, off);
    b.i = __shfl_xor_sync(0xffffffffu, a.i, off);
    arg_merge(a, b);
  }
}

// ---------------------------------------------------------------------------
// Float-float arithmetic: a value carried as an unevaluated sum hi + lo of
// two floats (about 48 significant bits).  GB300 executes double precision
// at a small fraction of its single-precision rate (a dependent double FMA
// costs about 64 cycles, a float-double-float round trip about 190), so the
// kernels keep their extra precision this way instead.  Built from the
// error-free transformations TwoSum (Knuth), FastTwoSum (Dekker) and
// TwoProduct with a fused multiply-add; every operation is an explicitly
// rounded intrinsic so that the compiler cannot contract or reorder them.
// ---------------------------------------------------------------------------
struct FF {
  float hi, lo;
};

// a + b = s + e exactly.
__device__ __forceinline__ FF two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}

// a + b = s + e exactly, given |a| >= |b| (or a == 0).
__device__ __forceinline__ FF fast_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

// a * b = p + e exactly.
__device__ __forceinline__ FF two_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return {p, __fmaf_rn(a, b, -p)};
}

__device__ __forceinline__ FF ff_add(FF a, FF b) {
  FF s = two_sum(a.hi, b.hi);
  const FF t = two_sum(a.lo, b.lo);
  s.lo = __fadd_rn(s.lo, t.hi);
  s = fast_two_sum(s.hi, s.lo);
  s.lo = __fadd_rn(s.lo, t.lo);
  return fast_two_sum(s.hi, s.lo);
}

__device__ __forceinline__ FF ff_neg(FF a) { return {-a.hi, -a.lo}; }
__device__ __forceinline__ FF ff_sub(FF a, FF b) { return ff_add(a, ff_neg(b)); }

__device__ __forceinline__ FF ff_add_f(FF a, float b) {
  FF s = two_sum(a.hi, b);
  s.lo = __fadd_rn(s.lo, a.lo);
  return fast_two_sum(s.hi, s.lo);
}

__device__ __forceinline__ FF ff_mul_f(FF a, float b) {
  FF p = two_prod(a.hi, b);
  p.lo = __fmaf_rn(a.lo, b, p.lo);
  return fast_two_sum(p.hi, p.lo);
}

// Comparisons of normalised values (|lo| at most half an ulp of hi).
__device__ __forceinline__ bool ff_le(FF a, FF b) {
  return a.hi < b.hi || (a.hi == b.hi && a.lo <= b.lo);
}
__device__ __forceinline__ float ff_to_float(FF a) { return __fadd_rn(a.hi, a.lo); }

__device__ __forceinline__ FF ff_shfl_xor(FF a, int off) {
  return {__shfl_xor_sync(0xffffffffu, a.hi, off), __shfl_xor_sync(0xffffffffu, a.lo, off)};
}

// Sum over the aligned groups of 2^levels lanes, in a fixed butterfly order
// (every lane of a group gets the same bits).
// One butterfly level: both partners add (lower lane's value, upper lane's
// value) in that order, so they compute the same bits.  The operands are
// selected first, so that the warp runs one addition, not one per branch.
__device__ __forceinline__ FF ff_level_add(FF x, int off) {
  const FF y = ff_shfl_xor(x, off);
  const bool upper = (threadIdx.x & off) != 0;
  const FF a = {upper ? y.hi : x.hi, upper ? y.lo : x.lo};
  const FF b = {upper ? x.hi : y.hi, upper ? x.lo : y.lo};
  return ff_add(a, b);
}

__device__ __forceinline__ FF group_sum_ff(FF x, int levels) {
#pragma unroll
  for (int l = 0; l < 5; ++l)
    if (l < levels) x = ff_level_add(x, 1 << l);
  return x;
}

// Two independent sums over the same lanes, level by level (their chains
// interleave).
__device__ __forceinline__ void group_sum_ff2(FF& x, FF& z, int levels) {
#pragma unroll
  for (int l = 0; l < 5; ++l) {
    if (l < levels) {
      x = ff_level_add(x, 1 << l);
      z = ff_level_add(z, 1 << l);
    }
  }
}

__device__ __forceinline__ float group_max(float x, int levels) {
  for (int l = 0; l < levels; ++l) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1 << l));
  return x;
}

__device__ __forceinline__ FF warp_sum_ff(FF x) { return group_sum_ff(x, 5); }

// Shuffle levels that cover lanes 0 .. n-1 (n <= 32).
__device__ __forceinline__ int levels_for(int n) { return n <= 1 ? 0 : 32 - __clz(n - 1); }

// ---------------------------------------------------------------------------
// Inline PTX: mbarrier, bulk async copy, programmatic dependent launch.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe: has the phase with this parity completed?
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase with the given parity to complete.  Gives up after
// kWaitLimitNs or when *abort becomes non-zero; returns false then.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  unsigned long long t0 = global_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63) == 63) {
      if (*abort) return false;
      if (global_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// 1-D bulk copy global -> shared, completing `bytes` of transaction on `bar`,
// with an L2 cache policy.  dst and src 16-byte aligned, bytes a positive
// multiple of 16.  The row streams read each byte once and take evict_first,
// so lines that will be read again (the OPD pass-2 re-read, the caller's
// other data) are not the ones replaced.
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Release: this thread's earlier writes are visible to whoever acquires the
// value this atomic leaves (or a later one in the word's modification order).
__device__ __forceinline__ void atom_or_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("{\n\t.reg .b64 t;\n\tatom.release.gpu.global.or.b64 t, [%0], %1;\n\t}" ::"l"(p),
               "l"(v)
               : "memory");
}

// A request's decision word: bit i of the low half = position i decided,
// bit i of the high half = position i accepted.  One atomic sets both, so a
// reader never sees one without the other.
__device__ __forceinline__ unsigned long long decision_bits(int i, bool accept) {
  const unsigned long long bit = 1ull << i;
  return accept ? (bit | (bit << 32)) : bit;
}

__device__ __forceinline__ void record_status(WsHeader* h, int code) {
  atomicCAS(&h->status, 0, code);
}

// ---------------------------------------------------------------------------
// Range checks of a SPEC_DEBUG build.  Each checked index into a buffer (a
// row, a descriptor, a partial slot, a segment, an output element) is
// compared with the buffer's extent; one that falls outside is counted in a
// device-wide counter, with the site of the first such check (read and reset
// through spec_debug_checks), and replaced by 0, a valid index at every
// site, so that the access stays inside the buffer.  Release builds compile
// the checks away.
// ---------------------------------------------------------------------------
enum SpecDebugSite {
  kSitePlanRowdesc = 1,   // plan: descriptor slot < 2 B k
  kSiteSweepRowdesc = 2,  // sweep: descriptor index < rows planned
  kSiteSweepRow = 3,      // sweep: logit row < rows of its buffer
  kSiteSweepPartial = 4,  // sweep: partial slot < rows x chunks
  kSiteSweepCount = 5,    // sweep: (request, position) counter < B k
  kSiteDecide = 6,        // sweep: decided (request, position) < B k
  kSiteFinalRow = 7,      // final pass: residual / bonus row < rows of its buffer
  kSiteFinalSegment = 8,  // final pass: chosen segment < segments of the row
  kSiteFinalToken = 9,    // final pass: sampled token < V
  kSiteOpdRow = 10,       // OPD statistics: logit row < rows of its buffer
  kSiteOpdOut = 11,       // OPD statistics: output element < B k
  kSiteD3d = 12,          // D3D selection: branch slot < branches
};

__device__ int g_debug_failures;  // checks that failed since the last reset
__device__ int g_debug_site;      // site of the first of them

__device__ __forceinline__ long long spec_debug_index(long long i, long long n, int site) {
  if (i >= 0 && i < n) return i;
  if (atomicAdd(&g_debug_failures, 1) == 0) atomicExch(&g_debug_site, site);
  return 0;
}

#ifdef SPEC_DEBUG
#define SPEC_CHECKED(i, n, site) spec_debug_index((long long)(i), (long long)(n), (site))
#else
#define SPEC_CHECKED(i, n, site) ((void)(n), (i))
#endif

// ---------------------------------------------------------------------------
// Partials: single 8-byte atomic exchanges and relaxed loads.
// ---------------------------------------------------------------------------

// The partial goes out as an atomic exchange: atomics are performed at L2,
// so the value is visible to other SMs at once (a plain store may linger in
// the SM until something drains it, and a deciding CTA would wait for it).
// Nothing waits for the old value.
__device__ __forceinline__ void store_partial(Partial* p, float m, uint32_t aux) {
  const unsigned long long v = ((unsigned long long)aux << 32) | __float_as_uint(m);
  asm volatile("{\n\t.reg .b64 t;\n\tatom.relaxed.gpu.global.exch.b64 t, [%0], %1;\n\t}" ::"l"(p),
               "l"(v)
               : "memory");
}

__device__ __forceinline__ unsigned long long load_u64_relaxed(const void* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Read a partial, waiting (bounded) while its slot still holds the empty
// marker: its unit has been counted, so its store is already on its way.
// Returns false if the wait ran out.
__device__ __forceinline__ bool load_partial(const Partial* p, float* m, uint32_t* aux) {
  unsigned long long v = load_u64_relaxed(p);
  if (v == kPartialEmpty) {
    const unsigned long long t0 = global_ns();
    for (;;) {
      __nanosleep(64);
      v = load_u64_relaxed(p);
      if (v != kPartialEmpty) break;
      if (global_ns() - t0 > kWaitLimitNs) return false;
    }
  }
  *m = __uint_as_float((uint32_t)v);
  *aux = (uint32_t)(v >> 32);
  return true;
}

// ---------------------------------------------------------------------------
// Combine the chunk partials of one row into its base-2 log normaliser
// c = fl(M*sc) + log2(S) (float-float), where M is the row max and
// S = sum_v 2^(z_v*sc - fl(M*sc)); log2 p(v) = z_v*sc - c.  Warp-cooperative:
// every lane returns the same value.  Returns false if the row has no finite
// mass (all -inf, or a NaN / +inf logit made S non-finite) or if a partial
// never arrived (*timed_out).
// ---------------------------------------------------------------------------

// log2 of a positive float as an exact exponent plus the single-precision
// log2 of the mantissa in [0.5, 1) (absolute error below 1e-7), summed in
// float-float.  Non-positive or non-finite input gives a non-finite result.
__device__ __forceinline__ FF log2_pos(float S) {
  if (!(S > 0.0f) || !(S <= FLT_MAX)) return {log2f(S), 0.0f};
  int e;
  const float mant = frexpf(S, &e);
  return two_sum((float)e, log2f(mant));
}

// One chunk's sum rescaled to the row reference ms_ref = fl(M*sc):
// s_c * 2^(fl(m_c*sc) - ms_ref) (the dominant chunk gets exactly 1; the
// difference is rounded once, which only touches terms far below the max).
__device__ __forceinline__ float chunk_term(float m_c, uint32_t s_bits, float sc, float ms_ref) {
  const float s_c = __uint_as_float(s_bits);
  if (s_c > 0.0f) return __fmul_rn(s_c, exp2f(__fsub_rn(__fmul_rn(m_c, sc), ms_ref)));
  return s_c == 0.0f ? 0.0f : __int_as_float(0x7fc00000);  // NaN stays NaN
}

// c = ms + log2(S) in float-float; ok iff S is a finite positive number.
__device__ __forceinline__ bool row_normaliser_from(float ms, float S, FF* c) {
  *c = ff_add(log2_pos(S), FF{ms, 0.0f});
  return S > 0.0f && S <= FLT_MAX;
}

__device__ __forceinline__ bool row_log2_normaliser(const Partial* parts, int nch, float sc,
                                                    FF* c_out, float* max_out,
                                                    bool* timed_out) {
  const int lane = threadIdx.x & 31;
  bool late = false;
  float m = -FLT_MAX;
  for (int c = lane; c < nch; c += 32) {
    float mc;
    uint32_t aux;
    if (load_partial(&parts[c], &mc, &aux)) m = fmaxf(m, mc);
    else late = true;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  const float msM = __fmul_rn(m, sc);
  FF S = {0.0f, 0.0f};
  for (int c = lane; c < nch; c += 32) {
    float mc;
    uint32_t aux;
    if (!load_partial(&parts[c], &mc, &aux)) {
      late = true;
      continue;
    }
    S = ff_add_f(S, chunk_term(mc, aux, sc, msM));
  }
  S = warp_sum_ff(S);
  late = __any_sync(0xffffffffu, late);
  *timed_out = late;
  *max_out = m;
  return row_normaliser_from(msM, ff_to_float(S), c_out) && !late;
}

// Both rows of a sampling position at once: parts[0, nch) are the target
// row's chunk partials and parts[nch, 2 nch) the draft row's (they are
// adjacent in the workspace).  Every partial is loaded in one round and kept
// in registers while 2 nch <= 32 * kMaxPartsPerLane.
constexpr int kMaxPartsPerLane = 8;

__device__ __forceinline__ void pair_log2_normalisers(const Partial* parts, int nch, float sc,
                                                      FF* ct, FF* cd, bool* ok_t,
                                                      bool* ok_d, bool* timed_out) {
  const int lane = threadIdx.x & 31;
  const int n2 = 2 * nch;
  if (n2 > 32 * kMaxPartsPerLane) {
    float mt, md;
    bool lt, ld;
    *ok_t = row_log2_normaliser(parts, nch, sc, ct, &mt, &lt);
    *ok_d = row_log2_normaliser(parts + nch, nch, sc, cd, &md, &ld);
    *timed_out = lt || ld;
    return;
  }
  if (n2 <= 32) {
    // One partial per lane (target chunks on lanes 0 .. nch-1, draft chunks
    // after them): reductions over just the lanes that hold data.
    const int lv = levels_for(n2);
    float mc = -FLT_MAX;
    uint32_t ac = 0u;
    bool late1 = false;
    if (lane < n2 && !load_partial(&parts[lane], &mc, &ac)) {
      late1 = true;
      mc = -FLT_MAX;
      ac = 0u;
    }
    const bool is_t = lane < nch, is_d = lane >= nch && lane < n2;
    // Lanes 0 .. 2^lv - 1 form the group that holds every partial; lane 0's
    // results go to the whole warp.
    const float mt = __shfl_sync(0xffffffffu, group_max(is_t ? mc : -FLT_MAX, lv), 0);
    const float md = __shfl_sync(0xffffffffu, group_max(is_d ? mc : -FLT_MAX, lv), 0);
    const float msT = __fmul_rn(mt, sc), msD = __fmul_rn(md, sc);
    const float term = (is_t || is_d) ? chunk_term(mc, ac, sc, is_t ? msT : msD) : 0.0f;
    FF St = {is_t ? term : 0.0f, 0.0f}, Sd = {is_d ? term : 0.0f, 0.0f};
    group_sum_ff2(St, Sd, lv);
    St = FF{__shfl_sync(0xffffffffu, St.hi, 0), __shfl_sync(0xffffffffu, St.lo, 0)};
    Sd = FF{__shfl_sync(0xffffffffu, Sd.hi, 0), __shfl_sync(0xffffffffu, Sd.lo, 0)};
    const bool late = __any_sync(0xffffffffu, late1);
    *timed_out = late;
    *ok_t = row_normaliser_from(msT, ff_to_float(St), ct) && !late;
    *ok_d = row_normaliser_from(msD, ff_to_float(Sd), cd) && !late;
    return;
  }
  float m[kMaxPartsPerLane];
  uint32_t a[kMaxPartsPerLane];
  bool late = false;
  float mt = -FLT_MAX, md = -FLT_MAX;
#pragma unroll
  for (int j = 0; j < kMaxPartsPerLane; ++j) {
    const int e = lane + 32 * j;
    m[j] = -FLT_MAX;
    a[j] = 0u;
    if (e < n2) {
      if (!load_partial(&parts[e], &m[j], &a[j])) {
        late = true;
        m[j] = -FLT_MAX;
        a[j] = 0u;
      }
      if (e < nch) mt = fmaxf(mt, m[j]);
      else md = fmaxf(md, m[j]);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
    md = fmaxf(md, __shfl_xor_sync(0xffffffffu, md, off));
  }
  const float msT = __fmul_rn(mt, sc), msD = __fmul_rn(md, sc);
  FF St = {0.0f, 0.0f}, Sd = {0.0f, 0.0f};
#pragma unroll
  for (int j = 0; j < kMaxPartsPerLane; ++j) {
    const int e = lane + 32 * j;
    if (e < nch) St = ff_add_f(St, chunk_term(m[j], a[j], sc, msT));
    else if (e < n2) Sd = ff_add_f(Sd, chunk_term(m[j], a[j], sc, msD));
  }
  group_sum_ff2(St, Sd, 5);
  late = __any_sync(0xffffffffu, late);
  *timed_out = late;
  *ok_t = row_normaliser_from(msT, ff_to_float(St), ct) && !late;
  *ok_d = row_normaliser_from(msD, ff_to_float(Sd), cd) && !late;
}

// Max and lowest index of a greedy row from its chunk partials.
__device__ __forceinline__ void row_argmax_from_parts(const Partial* parts, int nch, float* v_out,
                                                      int* i_out, bool* timed_out) {
  const int lane = threadIdx.x & 31;
  bool late = false;
  ArgAcc a;
  arg_init(a);
  for (int c = lane; c < nch; c += 32) {
    ArgAcc b;
    uint32_t aux;
    if (!load_partial(&parts[c], &b.v, &aux)) {
      late = true;
      continue;
    }
    b.i = (int)aux;
    arg_merge(a, b);
  }
  arg_warp_reduce(a);
  late = __any_sync(0xffffffffu, late);
  *timed_out = late;
  *v_out = a.v;
  *i_out = late ? INT32_MAX : a.i;
}

}  // namespace specv
