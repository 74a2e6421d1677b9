// Final pass: P slice CTAs per request.
//
// Each request's decisions (recorded by the sweep) give n, the first rejected
// position, or L if none; the round emits n + 1 tokens (DFlash notes,
// section 3.1, steps 6-7):
//   - sampling, n < L: one token from normalize(max(0, p_n - q_n)) (AdaFlash
//     Section 2.1; AdaFlash reading notes, basic idea, step 4);
//   - sampling, n == L: one token from p_L (target row L, read only now);
//   - greedy, n < L: the target argmax at n, already known from the sweep;
//   - greedy, n == L: the argmax of target row L.
// Sampling is by inverse CDF in ascending vocabulary index with u_L.  The
// row(s) are split into P slices of 256-entry segments; slice CTA p streams
// its slice once and writes one record per segment, then bumps the
// request's counter.  The last slice CTA to finish forms the segment prefix
// sums in float-float, picks the segment holding u_L * total, and re-reads that
// segment to place the token exactly.
//
// Records: a residual segment stores sum max(0, p - q) and the q mass where
// p > q, with p and q normalised by the row normalisers from the sweep; the
// slices also sum D = sum (p - q) over the pair, from which the combine
// corrects for the normalisers' residual error (see MassSpec).  A bonus segment
// stores its own max m and s = sum 2^(z*sc - fl(m*sc)); the last CTA weighs
// it by 2^(fl(m*sc) - REF), REF the largest segment reference, so the row is
// read once and the common normaliser cancels in the CDF.
#pragma once

#include "common.cuh"

namespace specv {

struct FinalParams {
  const void* target;
  const void* draft;
  const int32_t* tokens;
  const int32_t* lengths;
  const float* uniforms;
  const float* temperature;
  int B, k, V;
  int P;           // slice CTAs per request; CTA x is slice x % P of request x / P
  int sweep_grid;  // CTAs of the sweep grid this pass follows
  int test_late;   // testing aid: slices other than the first give up waiting (see below)
  long long rows_t, rows_d;  // rows of the target and draft buffers (range checks)
  int direct;      // rows in pinned host memory: slices load them, no bulk copies
  int32_t* out_tokens;
  int32_t* num_accepted;
  unsigned char* ws;
  WsLayout lay;
};

constexpr int kFinalWarps = kFinalThreads / 32;
constexpr int kJobNone = 0, kJobResidual = 1, kJobBonus = 2, kJobGreedyRowL = 3, kJobInvalid = 4,
              kJobTargetOnly = 5;

struct FinalShared {
  long long dwarp[kFinalWarps];   // a slice's share of D, per warp (fixed point)
  float warp_f[kFinalWarps];
  int warp_i[kFinalWarps];
  float4 pos_c[32];               // float-float log2 normalisers (target, draft) per position (k <= 31)
  int32_t pos_arg[32];
  int32_t tok[32];                // draft tokens x_0 .. x_{k-1}
  long long dsx[2];               // combine: D shares summed per warp (fixed point)
  long long wsum[kFinalWarps];    // combine: per warp, its sum of weights (fixed point),
  long long wexcl[kFinalWarps];   //          its last candidate segment's prefix
  int wcand[kFinalWarps];         //          and that segment (-1: none)
  float warp_w[kFinalWarps];      //          and its largest weight bound
  float uL;
  int job, n, token, last, late, any_late, bad_in, warm;
};

// Is a request's outcome known from its decision word?  n = the first
// rejected position among the L verified ones (or L); known when every
// position before n is decided (and so accepted).
__device__ __forceinline__ bool outcome_known_word(unsigned long long st, int L) {
  const uint32_t dec = (uint32_t)st, acc = (uint32_t)(st >> 32);
  const uint32_t lmask = (L >= 32) ? 0xffffffffu : ((1u << L) - 1u);
  const uint32_t rej = dec & ~acc & lmask;
  const int n = rej ? (__ffs((int)rej) - 1) : L;
  const uint32_t pre = (n >= 32) ? 0xffffffffu : ((1u << n) - 1u);
  return (dec & acc & pre) == pre;
}

// A slice CTA that gave up (its wait for the request's outcome, or for its
// own copies, ran out) still counts itself in final_done, with this mark
// added; the last slice to arrive then writes -1 outputs for the request
// instead of combining records that were never written.
constexpr int kLateMark = 1 << 16;
constexpr int kArriveMask = kLateMark - 1;  // slices arrived (P <= kMaxSlices)
static_assert(kMaxSlices < kLateMark, "the arrival count stays below the late mark");
static_assert(kMaxSlices <= 64 && kFinalThreads >= 64, "slice results reduce over two warps");
// The testing aid's wait: slices other than the first wait this long for an
// event that never happens, as if their request's outcome never arrived.
constexpr unsigned long long kTestLateLimitNs = 1000000ull;

// ---------------------------------------------------------------------------
// Segment loads: lane l holds entries 8l .. 8l+7 of a segment as raw bits
// (one 16-byte vector for bf16, two for fp32).  Entries >= V hold -inf.
// ---------------------------------------------------------------------------

template <typename TIn>
struct Seg8 {
  uint4 v[sizeof(TIn) == 2 ? 1 : 2];
};

template <typename TIn>
__device__ __forceinline__ void seg_load(Seg8<TIn>& s, const TIn* row, int e0, int V, bool vec_ok) {
  const uint4* src = reinterpret_cast<const uint4*>(row + e0);
  if (vec_ok && e0 + 8 <= V) {
#pragma unroll
    for (int w = 0; w < (int)(sizeof(s.v) / 16); ++w) s.v[w] = __ldg(src + w);
    return;
  }
  uint32_t* words = reinterpret_cast<uint32_t*>(s.v);
  if (sizeof(TIn) == 2) {
    const uint16_t* r = reinterpret_cast<const uint16_t*>(row);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const uint32_t lo = e0 + e < V ? __ldg(r + e0 + e) : 0xFF80u;
      const uint32_t hi = e0 + e + 1 < V ? __ldg(r + e0 + e + 1) : 0xFF80u;
      words[e / 2] = lo | (hi << 16);
    }
  } else {
    const uint32_t* r = reinterpret_cast<const uint32_t*>(row);
#pragma unroll
    for (int e = 0; e < 8; ++e) words[e] = e0 + e < V ? __ldg(r + e0 + e) : 0xFF800000u;
  }
}

// Entries 2j and 2j+1 of a lane's segment piece as a float pair.
template <typename TIn>
__device__ __forceinline__ float2 seg_pair(const Seg8<TIn>& s, int j);
template <>
__device__ __forceinline__ float2 seg_pair<uint16_t>(const Seg8<uint16_t>& s, int j) {
  const uint32_t w = j == 0 ? s.v[0].x : j == 1 ? s.v[0].y : j == 2 ? s.v[0].z : s.v[0].w;
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
template <>
__device__ __forceinline__ float2 seg_pair<float>(const Seg8<float>& s, int j) {
  const uint4& v = s.v[j >> 1];
  return (j & 1) ? make_float2(__uint_as_float(v.z), __uint_as_float(v.w))
                 : make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
}

__device__ __forceinline__ float2 f32x2_sub(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// How the entries of one request's final row(s) are weighed.
//
// Target-only entries (the bonus fallback of a zero residual): p = 2^(zt*sc - a).
//
// Residual entries max(0, p - q).  Two things make a plain p - q in single
// precision too coarse when q is close to p, where the residual's total mass
// (the total variation of p and q) is small and every error is magnified by
// its inverse in the normalised CDF:
//   - the difference of two nearly equal numbers, each rounded relative to
//     itself: the entries are formed as p - q = (p + q) * (-tanh(delta*ln2/2))
//     with delta = log2 q - log2 p = (zd - zt)*sc - (c_d - a) taken from the
//     logits directly, so that the error is relative to |p - q|;
//   - the row normalisers a and c_d come from the sweep's single-precision
//     sums and their ratio is off by up to a few 1e-7, which shifts every
//     entry by the same fraction of q.  The slice pass therefore also sums
//     D = sum_v (p_v - q_v) over the whole row pair (each slice its share, in
//     float-float), with p and q normalised by those normalisers; exactly
//     normalised, the residual is max(0, p - (1 + mu) q) with
//     mu = D / (1 - D), and each segment's weight is corrected by
//     -mu * (its q mass where p > q) in the combine.
// a and dc = c_d - a are carried as hi + lo single-precision pairs
// (float-float) so that they keep their accuracy.
struct MassSpec {
  float sc;
  float a_hi, a_lo;
  float dc_hi, dc_lo;
  bool has_q;
};

// -tanh(k * delta) / delta with k = ln(2) / 2, as a polynomial in w = delta^2:
// the Maclaurin series of tanh, tanh z = z - z^3/3 + 2z^5/15 - 17z^7/315 +
// 62z^9/2835 - 1382z^11/155925 + ..., truncated after z^11.  For |delta| <= 1
// (|z| <= 0.347) the first omitted term is below 1.1e-8 of the sum.  The
// coefficients are the series' own, scaled by powers of k by the compiler.
constexpr double kTanhK = 0.34657359027997265471;  // ln(2) / 2
constexpr float kTh0 = (float)(-kTanhK);
constexpr float kTh1 = (float)(kTanhK * kTanhK * kTanhK / 3.0);
constexpr float kTh2 = (float)(-2.0 * kTanhK * kTanhK * kTanhK * kTanhK * kTanhK / 15.0);
constexpr float kTh3 = (float)(17.0 * kTanhK * kTanhK * kTanhK * kTanhK * kTanhK * kTanhK * kTanhK /
                               315.0);
constexpr float kTh4 = (float)(-62.0 * kTanhK * kTanhK * kTanhK * kTanhK * kTanhK * kTanhK * kTanhK *
                               kTanhK * kTanhK / 2835.0);
constexpr float kTh5 = (float)(1382.0 * kTanhK * kTanhK * kTanhK * kTanhK * kTanhK * kTanhK * kTanhK *
                               kTanhK * kTanhK * kTanhK * kTanhK / 155925.0);
// Beyond |delta| = 1 the plain difference p - q loses at most a factor
// (1 + 2^-1) / (1 - 2^-1) = 3 of relative precision.
constexpr float kTanhRange = 1.0f;

// Signed residual entries rh = p - q and the draft probabilities qb of a lane's
// 8 entries (residual job).  Packed two-lane arithmetic gives each entry
// exactly the bits of the scalar formula, so the slice pass and the re-scan
// agree.
template <typename TIn>
__device__ __forceinline__ void residual_entries(const Seg8<TIn>& t, const Seg8<TIn>& d,
                                                 const MassSpec& ms, float (&rh)[8],
                                                 float (&qb)[8]) {
  const float2 sc2 = make_float2(ms.sc, ms.sc);
  const float2 na2 = make_float2(-ms.a_hi, -ms.a_hi);
  const float2 nd2 = make_float2(-ms.dc_hi, -ms.dc_hi), dh2 = make_float2(ms.dc_hi, ms.dc_hi);
  const float2 h1 = make_float2(kTh1, kTh1), h2 = make_float2(kTh2, kTh2);
  const float2 h3 = make_float2(kTh3, kTh3), h4 = make_float2(kTh4, kTh4);
  const float2 h5 = make_float2(kTh5, kTh5), h0 = make_float2(kTh0, kTh0);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 zt = seg_pair(t, j), zd = seg_pair(d, j);
    // p and q relative to the high parts of the normalisers only: the low
    // parts would scale every p, or every q, by the same factor 1 + O(1e-7),
    // which the mu correction absorbs like any other normaliser error.  q is
    // formed with the same two high parts that delta subtracts, so that
    // q / p = 2^delta holds to rounding.  zd - zt is exact for bf16 logits
    // (rounded once for fp32); the fused multiply-add rounds delta once more,
    // relative to delta itself.
    const float2 a = ex2x2(f32x2_fma(zt, sc2, na2));
    const float2 b = ex2x2(f32x2_sub(f32x2_fma(zd, sc2, na2), dh2));
    const float2 dl = f32x2_fma(f32x2_sub(zd, zt), sc2, nd2);
    const float2 w = f32x2_mul(dl, dl);
    float2 poly = f32x2_fma(h5, w, h4);
    poly = f32x2_fma(poly, w, h3);
    poly = f32x2_fma(poly, w, h2);
    poly = f32x2_fma(poly, w, h1);
    poly = f32x2_fma(poly, w, h0);
    const float2 small = f32x2_mul(f32x2_add(a, b), f32x2_mul(dl, poly));
    const float2 plain = f32x2_sub(a, b);
    // A NaN delta (both logits -inf) or an infinite one takes the plain
    // difference: 0, -q or p.
    rh[2 * j] = fabsf(dl.x) <= kTanhRange ? small.x : plain.x;
    rh[2 * j + 1] = fabsf(dl.y) <= kTanhRange ? small.y : plain.y;
    qb[2 * j] = b.x;
    qb[2 * j + 1] = b.y;
  }
}

// Target-only entries p = 2^(zt*sc - a) of a lane's 8 entries.
template <typename TIn>
__device__ __forceinline__ void target_entries(const Seg8<TIn>& t, const MassSpec& ms,
                                               float (&r)[8]) {
  const float2 sc2 = make_float2(ms.sc, ms.sc);
  const float2 na2 = make_float2(-ms.a_hi, -ms.a_hi), al2 = make_float2(ms.a_lo, ms.a_lo);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 pt = ex2x2(f32x2_sub(f32x2_fma(seg_pair(t, j), sc2, na2), al2));
    r[2 * j] = pt.x;
    r[2 * j + 1] = pt.y;
  }
}

// Weight of one residual entry once mu is known: max(0, (p - q) - mu q).
__device__ __forceinline__ float residual_weight(float rh, float qb, float mu) {
  return fmaxf(__fmaf_rn(-mu, qb, rh), 0.0f);
}

// Bonus entries relative to the segment reference msr = fl(m*sc), m the
// segment max (an all -inf segment has no mass).
template <typename TIn>
__device__ __forceinline__ void bonus_masses(const Seg8<TIn>& t, float sc, float msr,
                                             float (&r)[8]) {
  const float2 sc2 = make_float2(sc, sc), nm2 = make_float2(-msr, -msr);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 e = ex2x2(f32x2_fma(seg_pair(t, j), sc2, nm2));
    r[2 * j] = msr == -INFINITY ? 0.0f : e.x;
    r[2 * j + 1] = msr == -INFINITY ? 0.0f : e.y;
  }
}

template <typename TIn>
__device__ __forceinline__ float seg8_max(const Seg8<TIn>& t) {
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 z = seg_pair(t, j);
    m = fmaxf(m, fmaxf(z.x, z.y));
  }
  return m;
}

// Sum of 8 entries in a fixed order (pairs first).
__device__ __forceinline__ float sum8(const float (&r)[8]) {
  const float2 a = f32x2_add(make_float2(r[0], r[1]), make_float2(r[2], r[3]));
  const float2 b = f32x2_add(make_float2(r[4], r[5]), make_float2(r[6], r[7]));
  const float2 c = f32x2_add(a, b);
  return __fadd_rn(c.x, c.y);
}

__device__ __forceinline__ float warp_sum_f32(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, off));
  return x;
}

__device__ __forceinline__ float warp_max_f32(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
  return x;
}

// 2^(a - b) for a <= b: the difference rounded once (it is exact while a
// and b are within a factor of two), so the relative error stays near 1e-7
// wherever the power is not negligible.
__device__ __forceinline__ float exp2_diff(float a, float b) { return exp2f(__fsub_rn(a, b)); }

// One segment's record (warp-cooperative: every lane gets the same value):
//   residual:    (sum max(0, p - q), sum of q where p > q)
//   target only: (sum p, 0)
//   bonus:       (segment max m, sum 2^(z*sc - fl(m*sc)))
// For a residual, *dlane gets this lane's sum of p - q over its 8 entries
// (the share of D, see MassSpec).
template <typename TIn>
__device__ __forceinline__ float2 seg_record(const Seg8<TIn>& t, const Seg8<TIn>& d,
                                             const MassSpec& ms, bool bonus, float* dlane) {
  float r[8];
  if (bonus) {
    const float m = warp_max_f32(seg8_max(t));
    bonus_masses(t, ms.sc, __fmul_rn(m, ms.sc), r);
    return make_float2(m, warp_sum_f32(sum8(r)));
  }
  if (!ms.has_q) {
    target_entries(t, ms, r);
    return make_float2(warp_sum_f32(sum8(r)), 0.0f);
  }
  float qb[8];
  residual_entries(t, d, ms, r, qb);
  float rp = 0.0f, qp = 0.0f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    if (r[e] > 0.0f) {
      rp = __fadd_rn(rp, r[e]);
      qp = __fadd_rn(qp, qb[e]);
    }
  }
  *dlane = sum8(r);
  // Both sums in one butterfly: two shuffles, one packed add per level.
  float2 v = make_float2(rp, qp);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    v = f32x2_add(v, make_float2(__shfl_xor_sync(0xffffffffu, v.x, off),
                                 __shfl_xor_sync(0xffffffffu, v.y, off)));
  return v;
}

// CDF weight of a segment record: the residual mass corrected by mu (0 for
// target-only records), or for the bonus its sum rescaled from its own
// reference to REF.
__device__ __forceinline__ float seg_weight(float2 r, bool bonus, float sc, float REF, float mu) {
  if (!bonus) return fmaxf(__fmaf_rn(-mu, r.y, r.x), 0.0f);
  if (r.y == 0.0f) return 0.0f;
  return __fmul_rn(r.y, exp2_diff(__fmul_rn(r.x, sc), REF));
}

// Fixed-point sums.  The combine adds weights as 64-bit integers, each
// weight scaled by a power of two chosen from the largest one: integer sums
// are exact and independent of their order, so a prefix sum costs one
// integer add per step instead of a float-float addition, and the chain of
// dependent steps after the last slice arrives stays short.  Quantising a
// weight to 2^-50 of the largest changes the CDF by less than 2^-37 of its
// total even over 2^13 segments.  The slices' shares of D are summed the
// same way, on a fixed scale of 2^58 (|D| <= 2).
constexpr float kDScale = 288230376151711744.0f;       // 2^58
constexpr float kDUnscale = 3.4694469519536142e-18f;   // 2^-58

// 2^e as a float (e in [-126, 127]).
__device__ __forceinline__ float exp2_int(int e) { return __int_as_float((e + 127) << 23); }

__device__ __forceinline__ long long warp_sum_i64(long long x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

__device__ __forceinline__ long long warp_incl_scan_i64(long long x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  return x;
}

// ---------------------------------------------------------------------------
// Slice passes.  Warp w takes segments s_lo + w, s_lo + w + 8, ... in
// batches of U; the next batch is loaded before the current one is
// computed, so that every warp always has loads in flight.
// ---------------------------------------------------------------------------

template <typename TIn>
__host__ __device__ constexpr int slice_batch() {
  return sizeof(TIn) == 2 ? 2 : 1;
}

// Records of segments [s_lo, s_hi) (see seg_record); *dsum accumulates this
// thread's share of D in float-float.
template <typename TIn>
__device__ void slice_records(const TIn* rt, const TIn* rd, int V, const MassSpec& ms, bool bonus,
                              int s_lo, int s_hi, float2* rec, bool vec_ok,
                              long long* dsum) {
  constexpr int U = slice_batch<TIn>();
  constexpr int STEP = kFinalWarps * U;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool has_q = !bonus && ms.has_q;
  Seg8<TIn> ta[U], da[U], tb[U], db[U];
  auto load = [&](Seg8<TIn>(&t)[U], Seg8<TIn>(&d)[U], int s0) {
#pragma unroll
    for (int q = 0; q < U; ++q) {
      const int seg = s0 + q * kFinalWarps;
      if (seg < s_hi) {
        seg_load(t[q], rt, seg * kSegElems + lane * 8, V, vec_ok);
        if (has_q) seg_load(d[q], rd, seg * kSegElems + lane * 8, V, vec_ok);
      }
    }
  };
  auto process = [&](const Seg8<TIn>(&t)[U], const Seg8<TIn>(&d)[U], int s0) {
#pragma unroll
    for (int q = 0; q < U; ++q) {
      const int seg = s0 + q * kFinalWarps;
      if (seg >= s_hi) break;
      float dl = 0.0f;
      const float2 out = seg_record(t[q], d[q], ms, bonus, &dl);
      *dsum += __float2ll_rn(__fmul_rn(dl, kDScale));
      if (lane == 0) __stcg(&rec[seg], out);
    }
  };
  int s0 = s_lo + warp;
  if (s0 >= s_hi) return;
  load(ta, da, s0);
  for (;;) {
    if (s0 + STEP < s_hi) load(tb, db, s0 + STEP);
    process(ta, da, s0);
    s0 += STEP;
    if (s0 >= s_hi) break;
    if (s0 + STEP < s_hi) load(ta, da, s0 + STEP);
    process(tb, db, s0);
    s0 += STEP;
    if (s0 >= s_hi) break;
  }
}

// The same records, with the slice streamed through shared memory by bulk
// copies (rows 16-byte aligned): a ring of kFinalStages pieces, each S
// segments of the target row and, for a residual, the same S segments of the
// draft row after them.  Every warp takes the piece's segments w, w + 8, ...
// and computes exactly what slice_records computes; the last warp to be done
// with a slot refills it, so warps are not held together at every piece.  Far more bytes in flight per CTA than register
// loads allow, which is what a request finishing alone, at the end of a
// round, needs.  Returns false if a wait ran out.
constexpr int kFinalStages = 3;
constexpr int kFinalStageBytes = 16384;

struct FinalRing {
  uint64_t full[kFinalStages];
  int freed[kFinalStages];  // warps done with the slot's current piece
  int issued;               // pieces issued so far (in order)
  int abort_flag;
};

template <typename TIn>
__device__ bool slice_records_staged(const TIn* rt, const TIn* rd, int V, const MassSpec& ms,
                                     bool bonus, int s_lo, int s_hi, float2* rec,
                                     unsigned char* ring, FinalRing& fr, long long* dsum) {
  constexpr int SB = kSegElems * (int)sizeof(TIn);  // bytes of one segment of one row
  constexpr int NV = SB / 512;                      // 16-byte vectors per lane per segment
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool has_q = !bonus && ms.has_q;
  const int R = has_q ? 2 : 1;
  const int S = kFinalStageBytes / (R * SB);
  const int npieces = (s_hi - s_lo + S - 1) / S;
  if (threadIdx.x == 0) {
    for (int j = 0; j < kFinalStages; ++j) {
      mbar_init(&fr.full[j], 1);
      fr.freed[j] = 0;
    }
    fr.issued = 0;
    fr.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Bytes of segments [g0, g1) of one row (the row's last segment may be
  // short; V * size is a multiple of 16, so every size is).
  auto piece_bytes = [&](int j) {
    const int g0 = s_lo + j * S, g1 = min(s_hi, g0 + S);
    return (uint32_t)((min((long long)V, (long long)g1 * kSegElems) - (long long)g0 * kSegElems) *
                      (long long)sizeof(TIn));
  };
  auto issue = [&](int j) {
    const int slot = j % kFinalStages;
    const int g0 = s_lo + j * S;
    const uint32_t nb = piece_bytes(j);
    unsigned char* dst = ring + slot * kFinalStageBytes;
    mbar_arrive_expect_tx(&fr.full[slot], nb * R);
    const uint64_t pol = l2_policy_evict_first();
    bulk_g2s_hint(dst, rt + (size_t)g0 * kSegElems, nb, &fr.full[slot], pol);
    if (has_q) bulk_g2s_hint(dst + S * SB, rd + (size_t)g0 * kSegElems, nb, &fr.full[slot], pol);
    atomicMax(&fr.issued, j + 1);
  };
  if (threadIdx.x == 0)
    for (int j = 0; j < kFinalStages && j < npieces; ++j) issue(j);
  bool ok = true;
  for (int j = 0; j < npieces; ++j) {
    const int slot = j % kFinalStages;
    if (ok && !mbar_wait_bounded(&fr.full[slot], (uint32_t)(j / kFinalStages) & 1u, &fr.abort_flag)) {
      ok = false;
      *(volatile int*)&fr.abort_flag = 1;
    }
    const int g0 = s_lo + j * S, nseg = min(s_hi - g0, S);
    const uint4* buf = reinterpret_cast<const uint4*>(ring + slot * kFinalStageBytes);
    if (ok) {
      for (int ls = warp; ls < nseg; ls += kFinalWarps) {
        const int seg = g0 + ls;
        const int e0 = seg * kSegElems + lane * 8;
        Seg8<TIn> t, d;
#pragma unroll
        for (int w = 0; w < NV; ++w) t.v[w] = buf[ls * SB / 16 + lane * NV + w];
        if (has_q) {
#pragma unroll
          for (int w = 0; w < NV; ++w) d.v[w] = buf[(S + ls) * SB / 16 + lane * NV + w];
        }
        // Entries past the end of the row are not in the stage.
        if (e0 + 8 > V) {
          uint32_t* tw = reinterpret_cast<uint32_t*>(t.v);
          uint32_t* dw = reinterpret_cast<uint32_t*>(d.v);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            if (e0 + e < V) continue;
            if (sizeof(TIn) == 2) {
              const uint32_t hi = (e & 1) ? 0xFF800000u : 0u, keep = (e & 1) ? 0x0000FFFFu : 0xFFFF0000u;
              const uint32_t lo = (e & 1) ? 0u : 0x0000FF80u;
              tw[e / 2] = (tw[e / 2] & keep) | hi | lo;
              dw[e / 2] = (dw[e / 2] & keep) | hi | lo;
            } else {
              tw[e] = 0xFF800000u;
              dw[e] = 0xFF800000u;
            }
          }
        }
        float dl = 0.0f;
        const float2 out = seg_record(t, d, ms, bonus, &dl);
        *dsum += __float2ll_rn(__fmul_rn(dl, kDScale));
        if (lane == 0) __stcg(&rec[seg], out);
      }
    }
    // This warp is done with the slot (its reads are in registers); the last
    // of the warps to be done refills it with piece j + stages.
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      if (atomicAdd(&fr.freed[slot], 1) == kFinalWarps - 1) {
        fr.freed[slot] = 0;
        if (ok && !*(volatile int*)&fr.abort_flag && j + kFinalStages < npieces)
          issue(j + kFinalStages);
      }
    }
  }
  ok = __syncthreads_and(ok);
  if (!ok && threadIdx.x == 0) {
    // A wait ran out: let the copies still in flight land (bounded) before
    // the shared memory is given back.  Pieces go out in order, one slot at a
    // time, so only the last piece issued into each slot can be in flight.
    int dummy = 0;
    const int issued = fr.issued;
    for (int j = max(0, issued - kFinalStages); j < issued; ++j)
      mbar_wait_bounded(&fr.full[j % kFinalStages], (uint32_t)(j / kFinalStages) & 1u,
                        (volatile int*)&dummy);
  }
  __syncthreads();
  return ok;
}

// Largest entry of segments [s_lo, s_hi) and its lowest index (block-wide).
template <typename TIn>
__device__ ArgAcc slice_argmax(const TIn* row, int V, int s_lo, int s_hi, bool vec_ok,
                               FinalShared& sh) {
  constexpr int U = 2 * slice_batch<TIn>();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  ArgAcc a;
  arg_init(a);
  for (int s0 = s_lo + warp; s0 < s_hi; s0 += kFinalWarps * U) {
    Seg8<TIn> t[U];
#pragma unroll
    for (int q = 0; q < U; ++q) {
      const int seg = s0 + q * kFinalWarps;
      if (seg < s_hi) seg_load(t[q], row, seg * kSegElems + lane * 8, V, vec_ok);
    }
#pragma unroll
    for (int q = 0; q < U; ++q) {
      const int seg = s0 + q * kFinalWarps;
      if (seg >= s_hi) break;
      const int e0 = seg * kSegElems + lane * 8;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 z = seg_pair(t[q], j);
        arg_add(a, z.x, e0 + 2 * j);
        arg_add(a, z.y, e0 + 2 * j + 1);
      }
    }
  }
  arg_warp_reduce(a);
  if (lane == 0) {
    sh.warp_f[warp] = a.v;
    sh.warp_i[warp] = a.i;
  }
  __syncthreads();
  ArgAcc r;
  arg_init(r);
#pragma unroll
  for (int w = 0; w < kFinalWarps; ++w) {
    ArgAcc o;
    o.v = sh.warp_f[w];
    o.i = sh.warp_i[w];
    arg_merge(r, o);
  }
  __syncthreads();
  return r;
}

// Inverse CDF over the request's segment records (global, nseg entries):
// the first entry whose cumulative weight exceeds u * total.  Block-wide.
// Returns -1 on every thread if the weights have no mass or one of them is
// not a finite number; otherwise warp 0 gets the token and the other warps
// kPicked.  dshares: the P slices' shares of D (fixed point, 2^-58) for a
// residual, from which mu = D / (1 - D) is formed here (their loads go out
// with the record loads), or null (mu = 0).  rec_sm: nseg float2 of shared
// memory.  dry: made-up records and shares instead of rec and dshares (see
// final_body); nothing global is read from them or written either way.
constexpr int kPicked = INT32_MAX - 1;

template <typename TIn>
__device__ __noinline__ int cdf_pick(const TIn* rt, const TIn* rd, int V, MassSpec ms, bool bonus,
                                     float u, const float2* rec, int nseg, bool vec_ok,
                                     FinalShared& sh, float2* rec_sm, const long long* dshares,
                                     int P, bool dry) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool residual = !bonus && ms.has_q;
  // One round of loads: the D shares (threads < P) and the records, with
  // the largest weight bound (record.x, or a bonus record's sum) and the
  // bonus reference.
  long long dfx = 0;
  if (dshares != nullptr && (int)threadIdx.x < P) dfx = dry ? 0ll : __ldcg(&dshares[threadIdx.x]);
  float refm = -FLT_MAX, wmx = 0.0f;
  auto take = [&](int s, float2 r) {
    rec_sm[s] = r;
    if (bonus) {
      if (r.y > 0.0f) refm = fmaxf(refm, __fmul_rn(r.x, ms.sc));
      wmx = fmaxf(wmx, r.y);
    } else {
      wmx = fmaxf(wmx, r.x);
    }
  };
  // The first kRecRound records of each thread are all loaded before any is
  // stored, so that their loads overlap (the shared-memory stores would
  // otherwise hold each load behind the previous one).
  constexpr int kRecRound = 4;
  float2 rr[kRecRound];
#pragma unroll
  for (int q = 0; q < kRecRound; ++q) {
    const int s = threadIdx.x + q * kFinalThreads;
    rr[q] = s < nseg ? (dry ? make_float2(1.0f, 0.5f) : __ldcg(&rec[s])) : make_float2(0.0f, 0.0f);
  }
#pragma unroll
  for (int q = 0; q < kRecRound; ++q) {
    const int s = threadIdx.x + q * kFinalThreads;
    if (s < nseg) take(s, rr[q]);
  }
  for (int s = threadIdx.x + kRecRound * kFinalThreads; s < nseg; s += kFinalThreads)
    take(s, dry ? make_float2(1.0f, 0.5f) : __ldcg(&rec[s]));
  if (dshares != nullptr && warp < 2) {  // P <= 64 shares over two warps
    dfx = warp_sum_i64(dfx);
    if (lane == 0) sh.dsx[warp] = dfx;
  }
  refm = warp_max_f32(refm);
  wmx = warp_max_f32(wmx);
  if (lane == 0) {
    sh.warp_f[warp] = refm;
    sh.warp_w[warp] = wmx;
  }
  __syncthreads();
  // mu, REF and the weight bound: every thread forms them from the same
  // values in the same order.
  float mu = 0.0f;
  if (dshares != nullptr) {
    const float Df = __fmul_rn(__ll2float_rn(sh.dsx[0] + sh.dsx[1]), kDUnscale);
    mu = (Df > -1.0f && Df < 1.0f) ? __fdiv_rn(Df, __fsub_rn(1.0f, Df)) : 0.0f;
  }
  float REF = -FLT_MAX, WMX = 0.0f;
#pragma unroll
  for (int w = 0; w < kFinalWarps; ++w) {
    REF = fmaxf(REF, sh.warp_f[w]);
    WMX = fmaxf(WMX, sh.warp_w[w]);
  }
  if (!bonus) REF = 0.0f;
  // A residual weight R - mu Q+ exceeds R by at most about |mu| (Q+ is at
  // most the q mass, about 1); a bonus weight s * 2^(m*sc - REF) is at most
  // s.  Weights are clamped to the bound, which only ever trims rounding.
  const float bound = residual ? __fadd_ru(WMX, __fmul_ru(2.0f, fabsf(mu))) : WMX;
  if (!(bound > 0.0f && bound <= FLT_MAX)) return -1;  // uniform across the block
  // bound < 2^(eb+1); weights scaled by 2^S stay below 2^50, their sum below 2^63.
  const int eb = ((__float_as_int(bound) >> 23) & 0xff) - 127;
  const float fsc = exp2_int(min(126, 49 - eb));
  auto fixed = [&](float w) { return __float2ll_rn(__fmul_rn(fminf(w, bound), fsc)); };

  // Thread t owns segments [sa, sb).
  const int per = (nseg + kFinalThreads - 1) / kFinalThreads;
  const int sa = min(nseg, (int)threadIdx.x * per), sb = min(nseg, sa + per);
  long long loc = 0;
  bool finite = true;
  for (int s = sa; s < sb; ++s) {
    const float w = seg_weight(rec_sm[s], bonus, ms.sc, REF, mu);
    finite = finite && (w >= 0.0f && w <= FLT_MAX);
    loc += fixed(w);
  }
  const long long incl = warp_incl_scan_i64(loc);
  if (lane == 31) sh.wsum[warp] = incl;
  if (__syncthreads_or(!finite)) return -1;
  long long wv[kFinalWarps];
#pragma unroll
  for (int w = 0; w < kFinalWarps; ++w) wv[w] = sh.wsum[w];
  long long total = 0, run = 0;
#pragma unroll
  for (int w = 0; w < kFinalWarps; ++w) {
    if (w == warp) run = total;
    total += wv[w];
  }
  if (total <= 0) return -1;
  run += incl - loc;  // exclusive prefix of this thread's first segment
  // target = floor(total * u), u in [0, 1) scaled exactly to 64 bits.
  const long long target = (long long)__umul64hi((unsigned long long)total,
                                                 __float2ull_rz(__fmul_rn(u, 18446744073709551616.0f)));

  // The last segment with weight that starts at or before target: within a
  // thread the last one found, within a warp the highest lane that has one,
  // within the block the highest warp.
  int cand = -1;
  long long cand_excl = 0;
  for (int s = sa; s < sb; ++s) {
    const long long w = fixed(seg_weight(rec_sm[s], bonus, ms.sc, REF, mu));
    if (w > 0 && run <= target) {
      cand = s;
      cand_excl = run;
    }
    run += w;
  }
  const unsigned has = __ballot_sync(0xffffffffu, cand >= 0);
  if (has == 0u) {
    if (lane == 0) sh.wcand[warp] = -1;
  } else if (lane == 31 - __clz(has)) {
    sh.wcand[warp] = cand;
    sh.wexcl[warp] = cand_excl;
  }
  __syncthreads();
  if (warp != 0) return kPicked;
  // A positive total always has a candidate (the first segment with weight
  // starts at 0); j stays inside the row regardless.
  int j = 0;
  long long jexcl = 0;
#pragma unroll
  for (int w = kFinalWarps - 1; w >= 0; --w) {
    const int c = sh.wcand[w];
    if (c >= 0) {
      j = c;
      jexcl = sh.wexcl[w];
      break;
    }
  }
  if (!dry) j = (int)SPEC_CHECKED(j, nseg, kSiteFinalSegment);

  // Re-read segment j: the first entry whose cumulative weight exceeds the
  // target, or the segment's last entry with weight when the target lies
  // past the segment's own sum of entries (its record is that sum up to
  // rounding).
  Seg8<TIn> t, d;
  seg_load(t, rt, j * kSegElems + lane * 8, V, vec_ok);
  if (ms.has_q && !bonus) seg_load(d, rd, j * kSegElems + lane * 8, V, vec_ok);
  float r[8];
  if (bonus) {
    const float msr = __fmul_rn(rec_sm[j].x, ms.sc);
    bonus_masses(t, ms.sc, msr, r);
    const float scale = exp2_diff(msr, REF);
#pragma unroll
    for (int e = 0; e < 8; ++e) r[e] = __fmul_rn(r[e], scale);
  } else if (residual) {
    float qb[8];
    residual_entries(t, d, ms, r, qb);
#pragma unroll
    for (int e = 0; e < 8; ++e) r[e] = residual_weight(r[e], qb[e], mu);
  } else {
    target_entries(t, ms, r);
  }
  long long fe[8], lsum = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    fe[e] = fixed(fmaxf(r[e], 0.0f));  // a NaN entry counts as no weight
    lsum += fe[e];
  }
  long long cum = warp_incl_scan_i64(lsum) - lsum;
  const long long tseg = target - jexcl;
  int first_e = 8, last_pos = -1;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    cum += fe[e];
    if (first_e == 8 && fe[e] > 0 && cum > tseg) first_e = e;
    if (fe[e] > 0) last_pos = e;
  }
  const unsigned hit = __ballot_sync(0xffffffffu, first_e < 8);
  if (hit) {
    const int l = __ffs(hit) - 1;
    return j * kSegElems + l * 8 + __shfl_sync(0xffffffffu, first_e, l);
  }
  const unsigned hasm = __ballot_sync(0xffffffffu, last_pos >= 0);
  const int l = hasm ? 31 - __clz(hasm) : 0;
  return j * kSegElems + l * 8 + max(0, __shfl_sync(0xffffffffu, last_pos, l));
}

// Slice bounds in segments.
__device__ __forceinline__ int slice_lo(int part, int nseg, int P) {
  return (int)(((long long)part * nseg) / P);
}

// One slice CTA's work.  The CTA may start while the sweep is still running
// (it takes SMs the sweep has left): it first waits, bounded, until its
// request's outcome is known -- every position up to the first rejection
// (or all L) decided -- acquiring the deciders' writes with the mask.
template <typename TIn>
__device__ __forceinline__ void final_body(const FinalParams& p, FinalShared& sh, float2* rec_sm,
                                           FinalRing& fr) {
  const int nseg = segments_of(p.V);
  // A one-dimensional grid of B * P CTAs (a grid's y extent stops at 65535,
  // below the largest supported batch): slice `part` of request `b`.
  const int P = p.P;
  const int b = (int)(blockIdx.x / (unsigned)P), part = (int)(blockIdx.x - (unsigned)b * P);
  WsHeader* h = reinterpret_cast<WsHeader*>(p.ws + p.lay.header);
  float2* rec = reinterpret_cast<float2*>(p.ws + p.lay.seg_mass) + (size_t)b * nseg;
  // Per slice: (max, bits of its lowest index) of a greedy row L, or for a
  // residual the slice's share of D as a 64-bit fixed-point integer (2^-58).
  float2* slice_out = reinterpret_cast<float2*>(p.ws + p.lay.slice_out) + (size_t)b * kMaxSlices;
  int32_t* final_done = reinterpret_cast<int32_t*>(p.ws + p.lay.final_done);
  const int L = __ldg(&p.lengths[b]);
  const float T = __ldg(&p.temperature[b]);
  // The request's first rows, written by the plan kernel: loaded now, off
  // the path that follows the outcome.
  const int2 rb = __ldcg(reinterpret_cast<const int2*>(p.ws + p.lay.rowbase) + b);

  // A slice that starts before its request's outcome is known (small
  // batches: the pass launches behind the sweep and waits) first runs the
  // combine once on made-up records, writing nothing global, so that its
  // code is in the caches when the real combine runs: otherwise the one CTA
  // per request that combines fetches that code from memory, on the round's
  // critical path, and after an L2 flush that took 17 of a single request's
  // 44 us.
  if (threadIdx.x == 0) {
    const unsigned long long st0 =
        ld_acquire_u64(reinterpret_cast<const unsigned long long*>(p.ws + p.lay.state) + b);
    const int f0 = __ldcg(reinterpret_cast<const int32_t*>(p.ws + p.lay.flags) + b);
    sh.warm = (f0 & kReqValid) && part == 0 && !outcome_known_word(st0, L);
  }
  __syncthreads();
  if (sh.warm) {
    MassSpec wm = {};
    wm.sc = 1.0f;
    wm.has_q = true;
    const TIn* wr = reinterpret_cast<const TIn*>(p.ws);  // any 1 KB the call owns
    (void)cdf_pick<TIn>(wr, wr, kSegElems, wm, false, 0.5f, nullptr, 1, true, sh, rec_sm,
                        reinterpret_cast<const long long*>(slice_out), P, true);
  }

  // Warp 0: wait for the outcome (flags and masks, every lane the same),
  // then one round of loads of every position's normalisers, argmax and
  // draft token (lane t for position t); n: the first rejected position, or L.
  if (threadIdx.x < 32) {
    const int t = threadIdx.x;
    const uint32_t lmask = (L >= 32) ? 0xffffffffu : ((1u << L) - 1u);
    // The per-position inputs the plan does not check (lane t: position t):
    // tokens x_t in [0, V) for t < L and, when sampling, uniforms u_t in
    // [0, 1) for t <= L.  Any one out of range makes the request invalid.
    const int x_t = t < p.k ? __ldg(&p.tokens[(size_t)b * p.k + t]) : 0;
    const float u_t = (T != 0.0f && t <= L && t <= p.k)
                          ? __ldg(&p.uniforms[(size_t)b * (p.k + 1) + t])
                          : 0.0f;
    // The request's flags are the plan's (fixed for the round).  The first
    // look at the decision word goes out with the input loads above (its
    // acquire holds back only the loads after it); the wait then polls the
    // word alone.  A row without mass is recorded in bad_bits before the
    // decision that releases it, so bad_bits is read once, after the acquire
    // that ends the wait.
    int f = __ldcg(reinterpret_cast<const int32_t*>(p.ws + p.lay.flags) + b);
    unsigned long long st =
        ld_acquire_u64(reinterpret_cast<const unsigned long long*>(p.ws + p.lay.state) + b);
    if (t == L) sh.uL = u_t;  // the final token's uniform (0 at T = 0)
    const bool in_ok = (t >= L || (x_t >= 0 && x_t < p.V)) &&
                       (T == 0.0f || t > L || (u_t >= 0.0f && u_t < 1.0f));  // NaN fails
    const bool inputs_ok = __all_sync(0xffffffffu, in_ok);
    uint32_t dec = 0, acc = 0, bad = 0;
    bool late = false;
    // Testing aid: this slice never sees its outcome and gives up after a
    // short wait, exercising the path a real timeout takes.
    const bool never = p.test_late && part != 0;
    const unsigned long long limit = never ? kTestLateLimitNs : kWaitLimitNs;
    const unsigned long long t0 = global_ns();
    while (inputs_ok && (f & kReqValid)) {  // otherwise no outcome to wait for
      dec = (uint32_t)st;
      acc = (uint32_t)(st >> 32);
      if (outcome_known_word(st, L) && !never) break;
      if (global_ns() - t0 > limit) {
        late = true;
        break;
      }
      __nanosleep(128);
      st = ld_acquire_u64(reinterpret_cast<const unsigned long long*>(p.ws + p.lay.state) + b);
    }
    bad = __ldcg(reinterpret_cast<const uint32_t*>(p.ws + p.lay.bad_bits) + b);
    const float4* pos_c = reinterpret_cast<const float4*>(p.ws + p.lay.pos_c);
    const int32_t* pos_arg = reinterpret_cast<const int32_t*>(p.ws + p.lay.pos_arg);
    float4 c4 = make_float4(0.f, 0.f, 0.f, 0.f);
    int g = -1;
    if (t < p.k) {
      const size_t bi = (size_t)b * p.k + t;
      c4 = __ldcg(&pos_c[bi]);
      g = __ldcg(&pos_arg[bi]);
    }
    const int x = t < p.k ? x_t : -1;
    // A request the plan admitted whose tokens or uniforms are out of range:
    // recorded once, by the slice that writes its outputs.
    const bool bad_in = (f & kReqValid) && !inputs_ok;
    if (bad_in) f = 0;
    if (late) {
      if (t == 0) record_status(h, SPEC_ERR_TIMEOUT);
      f = 0;  // no outcome: the request reports -1
    }
    sh.pos_c[t] = c4;
    sh.pos_arg[t] = g;
    sh.tok[t] = x;
    __syncwarp();
    if (t == 0) {
      int job = kJobInvalid, n = -1, token = -1;
      if (f & kReqValid) {
        const uint32_t rej = dec & ~acc & lmask;
        n = rej ? (__ffs((int)rej) - 1) : L;
        const uint32_t prefix = (n >= 32) ? 0xffffffffu : ((1u << n) - 1u);
        if ((dec & acc & prefix) != prefix) {
          if (part == 0) record_status(h, SPEC_ERR_INTERNAL);
          n = -1;
        } else if (bad & (n < L ? ((prefix << 1) | 1u) : lmask)) {
          if (part == 0) {
            atomicAdd(&h->bad_requests, 1);
            atomicMin(&h->first_bad, b);
            record_status(h, SPEC_ERR_BAD_INPUT);
          }
          n = -1;
        } else if (f & kReqGreedy) {
          if (n < L) {
            job = kJobNone;
            token = sh.pos_arg[n];
          } else {
            job = kJobGreedyRowL;
          }
        } else {
          job = (n < L) ? kJobResidual : kJobBonus;
        }
      }
      sh.job = job;
      sh.n = n;
      sh.token = token;
      sh.late = late ? 1 : 0;
      sh.bad_in = bad_in ? 1 : 0;
    }
  }
  __syncthreads();
  const int job = sh.job;
  const int n = sh.n;
  int token = sh.token;
  bool gave_up = sh.late != 0;

  // At most 32 outputs per request: warp 0 writes them all (after cdf_pick,
  // only warp 0 holds the token).
  static_assert(SPEC_MAX_K + 1 <= 32, "one warp writes a request's outputs");
  auto write_outputs = [&](bool invalid, int final_token) {
    for (int j = threadIdx.x; j <= p.k; j += kFinalThreads) {
      int v = -1;
      if (!invalid) {
        if (j < n) v = sh.tok[j];
        else if (j == n) v = final_token;
      }
      p.out_tokens[(size_t)b * (p.k + 1) + j] = v;
    }
    if (threadIdx.x == 0) p.num_accepted[b] = invalid ? -1 : n;
  };
  // ---- this slice's share of the row(s) (none for kJobNone / kJobInvalid) ----
  const bool rows_job = (job == kJobResidual || job == kJobBonus || job == kJobGreedyRowL);
  const TIn* trow = nullptr;
  const TIn* drow = nullptr;
  bool vec_ok = false;
  MassSpec ms = {};
  const bool bonus = (job == kJobBonus);
  if (rows_job) {
    // Row n of the request in either buffer: its first rows (rb) come from
    // the plan kernel (padded or packed layout).
    trow = static_cast<const TIn*>(p.target) +
           (size_t)SPEC_CHECKED((long long)rb.x + n, p.rows_t, kSiteFinalRow) * (size_t)p.V;
    drow = job == kJobResidual
               ? static_cast<const TIn*>(p.draft) +
                     (size_t)SPEC_CHECKED((long long)rb.y + n, p.rows_d, kSiteFinalRow) *
                         (size_t)p.V
               : trow;
    vec_ok = ((reinterpret_cast<uintptr_t>(trow) | reinterpret_cast<uintptr_t>(drow)) & 15u) == 0;
    const int s_lo = slice_lo(part, nseg, P), s_hi = slice_lo(part + 1, nseg, P);
    ms.sc = job == kJobGreedyRowL ? 0.0f : softmax_scale(T);
    if (job == kJobResidual) {
      const float4 c4 = sh.pos_c[n];
      ms.a_hi = c4.x;
      ms.a_lo = c4.y;
      const FF dc = ff_sub(FF{c4.z, c4.w}, FF{c4.x, c4.y});
      ms.dc_hi = dc.hi;
      ms.dc_lo = dc.lo;
      ms.has_q = true;
    }
    if (job == kJobGreedyRowL) {
      const ArgAcc a = slice_argmax(trow, p.V, s_lo, s_hi, vec_ok, sh);
      if (threadIdx.x == 0) __stcg(&slice_out[part], make_float2(a.v, __int_as_float(a.i)));
    } else {
      long long dsum = 0;
      // Aligned rows in device memory stream through shared memory; others
      // (and rows in host memory) are loaded directly.
      if (vec_ok && ((size_t)p.V * sizeof(TIn)) % 16 == 0 && !p.direct) {
        if (!slice_records_staged(trow, drow, p.V, ms, bonus, s_lo, s_hi, rec,
                                  reinterpret_cast<unsigned char*>(rec_sm), fr, &dsum)) {
          gave_up = true;  // block-uniform: the staged pass ends in a block-wide vote
          if (threadIdx.x == 0) record_status(h, SPEC_ERR_TIMEOUT);
        }
      } else {
        slice_records(trow, drow, p.V, ms, bonus, s_lo, s_hi, rec, vec_ok, &dsum);
      }
      if (job == kJobResidual) {
        // The slice's share of D (fixed point, 2^-58), summed over the block.
        const long long wsum = warp_sum_i64(dsum);
        if ((threadIdx.x & 31) == 0) sh.dwarp[threadIdx.x >> 5] = wsum;
        __syncthreads();
        if (threadIdx.x == 0) {
          long long total = 0;
#pragma unroll
          for (int w = 0; w < kFinalWarps; ++w) total += sh.dwarp[w];
          __stcg(reinterpret_cast<long long*>(slice_out) + part, total);
        }
      }
    }
  }
  // ---- the last slice CTA of the request writes the outputs ----
  // Every slice counts itself in, also one without rows to stream or one
  // that gave up, so that the count always completes.
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int inc = 1 + (gave_up ? kLateMark : 0);
    const int old = atomicAdd(&final_done[b], inc);
    sh.last = (old & kArriveMask) == P - 1;
    sh.any_late = (old + inc) >= kLateMark;
  }
  __syncthreads();
  if (!sh.last) return;
  __threadfence();
  if (sh.any_late) {  // some slice has no outcome or no records: no token
    write_outputs(true, -1);
    return;
  }
  if (!rows_job) {
    if (sh.bad_in && threadIdx.x == 0) {
      atomicAdd(&h->bad_requests, 1);
      atomicMin(&h->first_bad, b);
      record_status(h, SPEC_ERR_BAD_INPUT);
    }
    write_outputs(job == kJobInvalid, token);
    return;
  }

  bool bad = false;
  if (job == kJobGreedyRowL) {
    // The P <= 64 slice maxima, one per lane of the first two warps.
    if (threadIdx.x < 64) {
      ArgAcc r;
      arg_init(r);
      if ((int)threadIdx.x < P) {
        const float2 so = __ldcg(&slice_out[threadIdx.x]);
        r.v = so.x;
        r.i = __float_as_int(so.y);
      }
      arg_warp_reduce(r);
      if ((threadIdx.x & 31) == 0) {
        sh.warp_f[threadIdx.x >> 5] = r.v;
        sh.warp_i[threadIdx.x >> 5] = r.i;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      ArgAcc r = {sh.warp_f[0], sh.warp_i[0]};
      const ArgAcc o = {sh.warp_f[1], sh.warp_i[1]};
      arg_merge(r, o);
      sh.token = r.i;
    }
    __syncthreads();
    token = sh.token;
    bad = (token == INT32_MAX);
  } else {
    const float u = sh.uL;
    // A residual's D = sum (p - q) over the row pair comes from the slices'
    // shares; cdf_pick turns it into mu = D / (1 - D), the correction for
    // the normalisers' ratio.
    token = cdf_pick(trow, drow, p.V, ms, bonus, u, rec, nseg, vec_ok, sh, rec_sm,
                     job == kJobResidual ? reinterpret_cast<const long long*>(slice_out) : nullptr,
                     P, false);
    if (token < 0 && job == kJobResidual) {
      // Residual mass zero (p_n == q_n up to rounding): draw from p_n.
      if (threadIdx.x == 0) atomicAdd(&h->residual_zero, 1);
      MassSpec pm = ms;
      pm.has_q = false;
      long long unused = 0;
      slice_records(trow, trow, p.V, pm, false, 0, nseg, rec, vec_ok, &unused);
      __threadfence_block();
      __syncthreads();
      token = cdf_pick(trow, trow, p.V, pm, false, u, rec, nseg, vec_ok, sh, rec_sm, nullptr, P,
                       false);
    }
    bad = (token < 0);
  }
  if (!bad && threadIdx.x < 32) token = (int)SPEC_CHECKED(token, p.V, kSiteFinalToken);
  if (threadIdx.x == 0) {
    const unsigned long long rows = job == kJobResidual ? 2ull : 1ull;
    atomicAdd(&h->final_rows, rows);
    atomicAdd(&h->final_bytes, rows * (unsigned long long)p.V * sizeof(TIn));
    if (bad) {
      atomicAdd(&h->bad_requests, 1);
      atomicMin(&h->first_bad, b);
      record_status(h, SPEC_ERR_BAD_INPUT);
    }
  }
  write_outputs(bad, token);
}

template <typename TIn>
__global__ void __launch_bounds__(kFinalThreads, 3) final_kernel(FinalParams p) {
  extern __shared__ __align__(128) unsigned char fsm_raw[];
  __shared__ FinalShared sh;
  __shared__ FinalRing fr;
  // The next call's plan kernel may launch now; it waits for this grid to
  // finish before it touches the workspace.
  pdl_launch_dependents();
  // fsm_raw holds the slice ring first and the combine's segment records
  // after it.
  final_body<TIn>(p, sh, reinterpret_cast<float2*>(fsm_raw), fr);
  // The grid must not finish before the sweep grid has (the next call's plan
  // waits only for this one): the last CTA out waits, bounded, for every
  // sweep CTA to have counted itself out.
  __syncthreads();
  if (threadIdx.x == 0) {
    WsHeader* h = reinterpret_cast<WsHeader*>(p.ws + p.lay.header);
    __threadfence();
    const int total = (int)gridDim.x;
    if (atomicAdd(&h->final_ctas_done, 1) == total - 1) {
      const unsigned long long t0 = global_ns();
      while (*(volatile int32_t*)&h->sweep_exited < p.sweep_grid) {
        if (global_ns() - t0 > kWaitLimitNs) {
          record_status(h, SPEC_ERR_TIMEOUT);
          break;
        }
        __nanosleep(256);
      }
    }
  }
}

}  // namespace specv
