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
constexpr double kLn2 = 0.69314718055994530942;

// Sweep kernel geometry.
constexpr int kSweepConsumerWarps = 8;
constexpr int kSweepThreads = (kSweepConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kStageBytes = 16384;
constexpr int kStages = 6;
constexpr int kRedDepth = kStages + 2;  // unit-end reduction slots in flight

// Final-pass kernel geometry.
constexpr int kFinalThreads = 1024;
constexpr int kSegElems = 256;  // one warp x 8 elements
constexpr int kMaxSegs = SPEC_MAX_V / kSegElems;

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
  int32_t pad[46];
};
static_assert(sizeof(WsHeader) == 256, "header is one 256-byte block");

// Per-unit partial result of the sweep: softmax (m, s) or argmax (m, arg).
struct __align__(16) Partial {
  float m;    // largest logit of the chunk
  float s;    // sum of 2^(z*sc - fl(m*sc)) over the chunk (sampling rows)
  int arg;    // lowest index attaining m (greedy rows)
  int pad;
};

struct WsLayout {
  size_t header, rowlist, flags, first_reject, acc_bits, dec_bits, bad_bits, done, pos_c, pos_arg,
      partials, total;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Vocabulary chunks per row: enough units to keep every SM busy when all
// rows are active, chunks of at least 2048 elements.
__host__ __device__ inline int chunks_per_row(long long rows_max, int V) {
  long long want = (16384 + rows_max - 1) / rows_max;
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

__host__ __device__ inline WsLayout ws_layout(int B, int k, int C) {
  WsLayout l;
  size_t o = 0;
  size_t slots = (size_t)B * (size_t)k * 2;
  l.header = o;       o = align256(o + sizeof(WsHeader));
  l.rowlist = o;      o = align256(o + slots * sizeof(int32_t));
  l.flags = o;        o = align256(o + (size_t)B * sizeof(int32_t));
  l.first_reject = o; o = align256(o + (size_t)B * sizeof(int32_t));
  l.acc_bits = o;     o = align256(o + (size_t)B * sizeof(uint32_t));
  l.dec_bits = o;     o = align256(o + (size_t)B * sizeof(uint32_t));
  l.bad_bits = o;     o = align256(o + (size_t)B * sizeof(uint32_t));
  l.done = o;         o = align256(o + (size_t)B * k * sizeof(int32_t));
  l.pos_c = o;        o = align256(o + slots * sizeof(double));
  l.pos_arg = o;      o = align256(o + (size_t)B * k * sizeof(int32_t));
  l.partials = o;     o = align256(o + slots * (size_t)C * sizeof(Partial));
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

// Double-precision warp sum (fixed butterfly order: all lanes get the same bits).
__device__ __forceinline__ double warp_sum_f64(double x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// ---------------------------------------------------------------------------
// Combine the chunk partials of one row into its base-2 log normaliser
// c = fl(M*sc) + log2(S), where M is the row max and
// S = sum_v 2^(z_v*sc - fl(M*sc)); log2 p(v) = z_v*sc - c.  Warp-cooperative:
// every lane returns the same value.  Returns false if the row has no finite
// mass (all -inf, or a NaN / +inf logit made S non-finite).
// ---------------------------------------------------------------------------

__device__ __forceinline__ bool row_log2_normaliser(const Partial* parts, int nch, float sc,
                                                    double* c_out, float* max_out) {
  const int lane = threadIdx.x & 31;
  float m = -FLT_MAX;
  for (int c = lane; c < nch; c += 32) m = fmaxf(m, __ldcg(&parts[c].m));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  const float msM = __fmul_rn(m, sc);
  double S = 0.0;
  for (int c = lane; c < nch; c += 32) {
    float mc = __ldcg(&parts[c].m);
    float sc_c = __ldcg(&parts[c].s);
    if (sc_c > 0.0f) S += (double)sc_c * exp2((double)__fmul_rn(mc, sc) - (double)msM);
    else if (!(sc_c == 0.0f)) S = __longlong_as_double(0x7ff8000000000000ll);  // NaN
  }
  S = warp_sum_f64(S);
  *c_out = (double)msM + log2(S);
  *max_out = m;
  return S > 0.0 && S <= 1.79e308;
}

__device__ __forceinline__ void row_argmax_from_parts(const Partial* parts, int nch, float* v_out,
                                                      int* i_out) {
  const int lane = threadIdx.x & 31;
  ArgAcc a;
  arg_init(a);
  for (int c = lane; c < nch; c += 32) {
    ArgAcc b;
    b.v = __ldcg(&parts[c].m);
    b.i = __ldcg(&parts[c].arg);
    arg_merge(a, b);
  }
  arg_warp_reduce(a);
  *v_out = a.v;
  *i_out = a.i;
}

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

// 1-D bulk copy global -> shared, completing `bytes` of transaction on `bar`.
// dst and src 16-byte aligned, bytes a positive multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void record_status(WsHeader* h, int code) {
  atomicCAS(&h->status, 0, code);
}

}  // namespace specv
