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
  int32_t* out_tokens;
  int32_t* num_accepted;
  unsigned char* ws;
  WsLayout lay;
};

constexpr int kFinalWarps = kFinalThreads / 32;
constexpr int kJobNone = 0, kJobResidual = 1, kJobBonus = 2, kJobGreedyRowL = 3, kJobInvalid = 4,
              kJobTargetOnly = 5;

struct FinalShared {
  FF warp_ff[kFinalWarps + 1];
  float warp_f[kFinalWarps];
  int warp_i[kFinalWarps];
  float4 pos_c[32];               // float-float log2 normalisers (target, draft) per position (k <= 31)
  int32_t pos_arg[32];
  int32_t tok[32];                // draft tokens x_0 .. x_{k-1}
  FF cand_excl;
  float REF, mu;
  int job, n, cand, token, last, late, any_late, bad_in;
};

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
                              int s_lo, int s_hi, float2* rec, bool vec_ok, FF* dsum) {
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
      *dsum = ff_add_f(*dsum, dl);
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
                                     unsigned char* ring, FinalRing& fr, FF* dsum) {
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
        *dsum = ff_add_f(*dsum, dl);
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

__device__ __forceinline__ FF ff_shfl_up(FF a, int off) {
  return {__shfl_up_sync(0xffffffffu, a.hi, off), __shfl_up_sync(0xffffffffu, a.lo, off)};
}

// Inclusive warp scan in float-float (lane order).
__device__ __forceinline__ FF warp_incl_scan_ff(FF x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const FF y = ff_shfl_up(x, off);
    if (lane >= off) x = ff_add(y, x);
  }
  return x;
}

// Block-wide exclusive scan of one float-float per thread; all threads get
// the total.
__device__ __forceinline__ FF block_exclusive_scan_ff(FF x, FinalShared& sh, FF* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const FF incl = warp_incl_scan_ff(x);
  if (lane == 31) sh.warp_ff[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const FF w = lane < kFinalWarps ? sh.warp_ff[lane] : FF{0.0f, 0.0f};
    const FF wi = warp_incl_scan_ff(w);
    FF wx = ff_shfl_up(wi, 1);
    if (lane == 0) wx = FF{0.0f, 0.0f};
    __syncwarp();
    if (lane < kFinalWarps) sh.warp_ff[lane] = wx;
    if (lane == kFinalWarps - 1) sh.warp_ff[kFinalWarps] = wi;
  }
  __syncthreads();
  // Exclusive prefix within the warp, then the warp's offset.
  FF ex = ff_shfl_up(incl, 1);
  if (lane == 0) ex = FF{0.0f, 0.0f};
  ex = ff_add(sh.warp_ff[warp], ex);
  *total = sh.warp_ff[kFinalWarps];
  __syncthreads();
  return ex;
}

// Inverse CDF over the request's segment records (global, nseg entries):
// the first entry whose cumulative weight exceeds u * total.  Block-wide;
// returns the token, or -1 if the total weight is not a finite positive
// number.  rec_sm: nseg float2 of shared memory.  mu: the residual's
// normaliser correction (0 otherwise).
template <typename TIn>
__device__ int cdf_pick(const TIn* rt, const TIn* rd, int V, const MassSpec& ms, bool bonus,
                        float u, const float2* rec, int nseg, bool vec_ok, FinalShared& sh,
                        float2* rec_sm, float mu) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool residual = !bonus && ms.has_q;
  float refm = -FLT_MAX;
  for (int s = threadIdx.x; s < nseg; s += kFinalThreads) {
    const float2 r = __ldcg(&rec[s]);
    rec_sm[s] = r;
    if (bonus && r.y > 0.0f) refm = fmaxf(refm, __fmul_rn(r.x, ms.sc));
  }
  float REF = 0.0f;
  if (bonus) {
    refm = warp_max_f32(refm);
    if (lane == 0) sh.warp_f[warp] = refm;
  }
  __syncthreads();
  if (bonus) {
    REF = -FLT_MAX;
#pragma unroll
    for (int w = 0; w < kFinalWarps; ++w) REF = fmaxf(REF, sh.warp_f[w]);
  }
  // Thread t owns segments [sa, sb).
  const int per = (nseg + kFinalThreads - 1) / kFinalThreads;
  const int sa = min(nseg, (int)threadIdx.x * per), sb = min(nseg, sa + per);
  // Exclusive prefix of the weights, in float-float.
  FF loc = {0.0f, 0.0f};
  for (int s = sa; s < sb; ++s) loc = ff_add_f(loc, seg_weight(rec_sm[s], bonus, ms.sc, REF, mu));
  FF total;
  FF run = block_exclusive_scan_ff(loc, sh, &total);
  if (!(total.hi > 0.0f && total.hi <= FLT_MAX)) return -1;  // uniform across the block
  const FF target = ff_mul_f(total, u);

  // The last segment with positive weight that starts at or before target.
  if (threadIdx.x == 0) sh.cand = -1;
  __syncthreads();
  int cand = -1;
  FF cand_excl = {0.0f, 0.0f};
  for (int s = sa; s < sb; ++s) {
    const float w = seg_weight(rec_sm[s], bonus, ms.sc, REF, mu);
    if (w > 0.0f && ff_le(run, target)) {
      cand = s;
      cand_excl = run;
    }
    run = ff_add_f(run, w);
  }
  if (cand >= 0) atomicMax(&sh.cand, cand);
  __syncthreads();
  const int j = sh.cand;
  if (cand >= 0 && cand == j) sh.cand_excl = cand_excl;
  __syncthreads();

  // Re-read segment j: the first entry whose cumulative weight exceeds the
  // target, or the segment's last entry with mass when rounding left the
  // target just past the segment's own sum.
  if (warp == 0) {
    Seg8<TIn> t, d;
    seg_load(t, rt, j * kSegElems + lane * 8, V, vec_ok);
    if (ms.has_q && !bonus) seg_load(d, rd, j * kSegElems + lane * 8, V, vec_ok);
    float r[8];
    float scale = 1.0f;
    if (bonus) {
      const float msr = __fmul_rn(rec_sm[j].x, ms.sc);
      bonus_masses(t, ms.sc, msr, r);
      scale = exp2_diff(msr, REF);
    } else if (residual) {
      float qb[8];
      residual_entries(t, d, ms, r, qb);
#pragma unroll
      for (int e = 0; e < 8; ++e) r[e] = residual_weight(r[e], qb[e], mu);
    } else {
      target_entries(t, ms, r);
    }
    // Cumulative weight within the segment, in float-float: lane sums, then
    // an exclusive scan over the lanes, then entry by entry.
    FF lsum = {0.0f, 0.0f};
#pragma unroll
    for (int e = 0; e < 8; ++e) lsum = ff_add_f(lsum, r[e]);
    const FF lincl = warp_incl_scan_ff(lsum);
    FF cum = ff_shfl_up(lincl, 1);
    if (lane == 0) cum = FF{0.0f, 0.0f};
    const FF tseg = ff_sub(target, sh.cand_excl);
    int first_e = 8, last_pos = -1;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      cum = ff_add_f(cum, r[e]);
      if (first_e == 8 && r[e] > 0.0f && !ff_le(ff_mul_f(cum, scale), tseg)) first_e = e;
      if (r[e] > 0.0f) last_pos = e;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, first_e < 8);
    int token;
    if (hit) {
      const int l = __ffs(hit) - 1;
      token = j * kSegElems + l * 8 + __shfl_sync(0xffffffffu, first_e, l);
    } else {
      const unsigned has = __ballot_sync(0xffffffffu, last_pos >= 0);
      const int l = has ? 31 - __clz(has) : 0;
      token = j * kSegElems + l * 8 + max(0, __shfl_sync(0xffffffffu, last_pos, l));
    }
    if (lane == 0) sh.token = token;
  }
  __syncthreads();
  const int tk = sh.token;
  __syncthreads();
  return tk;
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
  // Per slice: (max, bits of its lowest index) of a greedy row L, or the
  // slice's share of D (hi, lo) for a residual.
  float2* slice_out = reinterpret_cast<float2*>(p.ws + p.lay.slice_out) + (size_t)b * kMaxSlices;
  int32_t* final_done = reinterpret_cast<int32_t*>(p.ws + p.lay.final_done);
  const int L = __ldg(&p.lengths[b]);
  const float T = __ldg(&p.temperature[b]);

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
    const bool in_ok = (t >= L || (x_t >= 0 && x_t < p.V)) &&
                       (T == 0.0f || t > L || (u_t >= 0.0f && u_t < 1.0f));  // NaN fails
    const bool inputs_ok = __all_sync(0xffffffffu, in_ok);
    int f = 0;
    uint32_t dec = 0, acc = 0, bad = 0;
    bool late = false;
    // Testing aid: this slice never sees its outcome and gives up after a
    // short wait, exercising the path a real timeout takes.
    const bool never = p.test_late && part != 0;
    const unsigned long long limit = never ? kTestLateLimitNs : kWaitLimitNs;
    const unsigned long long t0 = global_ns();
    for (;;) {
      f = __ldcg(reinterpret_cast<const int32_t*>(p.ws + p.lay.flags) + b);
      if (!inputs_ok) break;  // invalid: no outcome to wait for
      const unsigned long long st =
          ld_acquire_u64(reinterpret_cast<const unsigned long long*>(p.ws + p.lay.state) + b);
      dec = (uint32_t)st;
      acc = (uint32_t)(st >> 32);
      bad = __ldcg(reinterpret_cast<const uint32_t*>(p.ws + p.lay.bad_bits) + b);
      if (!(f & kReqValid)) break;
      const uint32_t rej = dec & ~acc & lmask;
      const int nn = rej ? (__ffs((int)rej) - 1) : L;
      const uint32_t pre = (nn >= 32) ? 0xffffffffu : ((1u << nn) - 1u);
      if ((dec & acc & pre) == pre && !never) break;
      if (global_ns() - t0 > limit) {
        late = true;
        break;
      }
      __nanosleep(256);
    }
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
    // Row n of the request in either buffer: its first rows come from the
    // plan kernel (padded or packed layout).
    const int2 rb = __ldcg(reinterpret_cast<const int2*>(p.ws + p.lay.rowbase) + b);
    trow = static_cast<const TIn*>(p.target) + ((size_t)rb.x + n) * (size_t)p.V;
    drow = job == kJobResidual
               ? static_cast<const TIn*>(p.draft) + ((size_t)rb.y + n) * (size_t)p.V
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
      FF dsum = {0.0f, 0.0f};
      // Aligned rows stream through shared memory; others load directly.
      if (vec_ok && ((size_t)p.V * sizeof(TIn)) % 16 == 0) {
        if (!slice_records_staged(trow, drow, p.V, ms, bonus, s_lo, s_hi, rec,
                                  reinterpret_cast<unsigned char*>(rec_sm), fr, &dsum)) {
          gave_up = true;  // block-uniform: the staged pass ends in a block-wide vote
          if (threadIdx.x == 0) record_status(h, SPEC_ERR_TIMEOUT);
        }
      } else {
        slice_records(trow, drow, p.V, ms, bonus, s_lo, s_hi, rec, vec_ok, &dsum);
      }
      if (job == kJobResidual) {
        // The slice's share of D, summed over the block in float-float.
        FF total;
        (void)block_exclusive_scan_ff(dsum, sh, &total);
        if (threadIdx.x == 0) __stcg(&slice_out[part], make_float2(total.hi, total.lo));
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
    const float u = __ldg(&p.uniforms[(size_t)b * (p.k + 1) + L]);
    // Residual: D = sum (p - q) over the row pair from the slices' shares,
    // then mu = D / (1 - D), the correction for the normalisers' ratio.
    float mu = 0.0f;
    if (job == kJobResidual) {
      // The P <= 64 shares, one per lane of the first two warps.
      if (threadIdx.x < 64) {
        FF D = {0.0f, 0.0f};
        if ((int)threadIdx.x < P) {
          const float2 so = __ldcg(&slice_out[threadIdx.x]);
          D = FF{so.x, so.y};
        }
        D = warp_sum_ff(D);
        if ((threadIdx.x & 31) == 0) sh.warp_ff[threadIdx.x >> 5] = D;
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        const float Df = ff_to_float(ff_add(sh.warp_ff[0], sh.warp_ff[1]));
        sh.mu = (Df > -1.0f && Df < 1.0f) ? __fdiv_rn(Df, __fsub_rn(1.0f, Df)) : 0.0f;
      }
      __syncthreads();
      mu = sh.mu;
    }
    token = cdf_pick(trow, drow, p.V, ms, bonus, u, rec, nseg, vec_ok, sh, rec_sm, mu);
    if (token < 0 && job == kJobResidual) {
      // Residual mass zero (p_n == q_n up to rounding): draw from p_n.
      if (threadIdx.x == 0) atomicAdd(&h->residual_zero, 1);
      MassSpec pm = ms;
      pm.has_q = false;
      FF unused = {0.0f, 0.0f};
      slice_records(trow, trow, p.V, pm, false, 0, nseg, rec, vec_ok, &unused);
      __threadfence_block();
      __syncthreads();
      token = cdf_pick(trow, trow, p.V, pm, false, u, rec, nseg, vec_ok, sh, rec_sm, 0.0f);
    }
    bad = (token < 0);
  }
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
