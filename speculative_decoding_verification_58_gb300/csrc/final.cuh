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
// its slice once and writes one mass per segment, then bumps the request's
// counter.  The last slice CTA to finish forms the segment prefix sums in
// double, picks the segment holding u_L * total, and re-reads that segment
// to place the token exactly.
//
// Masses: residual entries max(0, p - q) use the row normalisers from the
// sweep.  Bonus entries use each slice's own max as reference,
// 2^(z*sc - ref_p), and the last CTA rescales the slices by 2^(ref_p - ref);
// the common normaliser cancels in the CDF.
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
  int P;  // slice CTAs per request (gridDim.x)
  int32_t* out_tokens;
  int32_t* num_accepted;
  unsigned char* ws;
  WsLayout lay;
};

constexpr int kFinalWarps = kFinalThreads / 32;
constexpr int kJobNone = 0, kJobResidual = 1, kJobBonus = 2, kJobGreedyRowL = 3, kJobInvalid = 4;

struct FinalShared {
  double warp_d[kFinalWarps + 1];
  float4 warp_f[kFinalWarps];
  float scale[kMaxSlices];  // bonus: 2^(ref_p - ref) per slice
  int job, n, token, cand, last;
};

// Eight consecutive elements e0..e0+7 of a row (entries >= V read as -inf).
template <typename TIn>
__device__ __forceinline__ void load8(const TIn* row, int e0, int V, bool vec_ok, float* x) {
  using Tr = ElemTraits<TIn>;
  if (vec_ok && e0 + 8 <= V) {
    const uint4* v = reinterpret_cast<const uint4*>(row + e0);
    if (Tr::kPerVec == 8) {
      Tr::unpack(__ldg(v), x);
    } else {
      Tr::unpack(__ldg(v), x);
      Tr::unpack(__ldg(v + 1), x + 4);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = (e0 + e < V) ? Tr::load(row, e0 + e) : -INFINITY;
  }
}

// One lane's 8 entries of a segment as raw bits (one 16-byte vector for bf16,
// two for fp32), so that several segments can be in flight before any
// arithmetic.  Entries >= V hold -inf.
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

template <typename TIn>
__device__ __forceinline__ void seg_unpack(const Seg8<TIn>& s, float* x) {
#pragma unroll
  for (int w = 0; w < (int)(sizeof(s.v) / 16); ++w)
    ElemTraits<TIn>::unpack(s.v[w], x + w * ElemTraits<TIn>::kPerVec);
}

// Segments a warp keeps in flight per row.
template <typename TIn>
__host__ __device__ constexpr int seg_batch() {
  return sizeof(TIn) == 2 ? 4 : 2;
}

// Mass of one entry: 2^(zt*sc - a) for p (a = its log2 normaliser, or a
// slice reference for the bonus), minus 2^(zd*sc - c_d) for q when there is
// a draft row, clamped at 0.  a and c_d come as hi + lo single-precision
// pairs so that the normaliser keeps double accuracy.  The slice pass and
// the re-scan call this with identical arguments, so both see the same bits.
__device__ __forceinline__ float entry_mass(float zt, float zd, float sc, float a_hi, float a_lo,
                                            float cd_hi, float cd_lo, bool has_q) {
  const float p = ex2(__fsub_rn(fmaf(zt, sc, -a_hi), a_lo));
  if (!has_q) return p;
  const float q = ex2(__fsub_rn(fmaf(zd, sc, -cd_hi), cd_lo));
  return fmaxf(__fsub_rn(p, q), 0.0f);
}

// Block-wide exclusive scan of one double per thread; all threads get the total.
__device__ __forceinline__ double block_exclusive_scan_f64(double x, FinalShared& sh,
                                                           double* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double incl = x;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) sh.warp_d[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const double w = lane < kFinalWarps ? sh.warp_d[lane] : 0.0;
    double wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += y;
    }
    if (lane < kFinalWarps) sh.warp_d[lane] = wi - w;
    if (lane == kFinalWarps - 1) sh.warp_d[kFinalWarps] = wi;
  }
  __syncthreads();
  const double ex = (incl - x) + sh.warp_d[warp];
  *total = sh.warp_d[kFinalWarps];
  __syncthreads();
  return ex;
}

// Slice bounds in segments.
__device__ __forceinline__ int slice_lo(int part, int nseg, int P) {
  return (int)(((long long)part * nseg) / P);
}
__device__ __forceinline__ int slice_of(int seg, int nseg, int P) {
  int p = (int)(((long long)seg * P) / nseg);
  while (p + 1 < P && slice_lo(p + 1, nseg, P) <= seg) ++p;
  while (p > 0 && slice_lo(p, nseg, P) > seg) --p;
  return p;
}

// Segment masses of segments [s_lo, s_hi) into seg_mass (global): warp w
// takes segments s_lo + w, s_lo + w + 8, ... (a few at a time, loads first);
// lane l holds entries 8l..8l+7 of a segment.  rd == nullptr: no draft row.
template <typename TIn>
__device__ void slice_masses(const TIn* rt, const TIn* rd, int V, float sc, float a_hi, float a_lo,
                             float cd_hi, float cd_lo, int s_lo, int s_hi, float* seg_mass,
                             bool vec_ok) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool has_q = (rd != nullptr);
  constexpr int U = seg_batch<TIn>();
  for (int s0 = s_lo + warp; s0 < s_hi; s0 += kFinalWarps * U) {
    Seg8<TIn> t[U], d[U];
#pragma unroll
    for (int q = 0; q < U; ++q) {
      const int seg = s0 + q * kFinalWarps;
      if (seg < s_hi) {
        seg_load(t[q], rt, seg * kSegElems + lane * 8, V, vec_ok);
        if (has_q) seg_load(d[q], rd, seg * kSegElems + lane * 8, V, vec_ok);
      }
    }
#pragma unroll
    for (int q = 0; q < U; ++q) {
      const int seg = s0 + q * kFinalWarps;
      if (seg >= s_hi) break;
      float zt[8], zd[8];
      seg_unpack(t[q], zt);
      if (has_q) seg_unpack(d[q], zd);
      float m = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e)
        m = __fadd_rn(m, entry_mass(zt[e], has_q ? zd[e] : 0.f, sc, a_hi, a_lo, cd_hi, cd_lo,
                                    has_q));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = __fadd_rn(m, __shfl_xor_sync(0xffffffffu, m, off));
      if (lane == 0) __stcg(&seg_mass[seg], m);
    }
  }
}

// Largest entry of segments [s_lo, s_hi) (block-wide; all threads get it).
template <typename TIn>
__device__ float slice_max(const TIn* row, int V, int s_lo, int s_hi, bool vec_ok, FinalShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int U = 2 * seg_batch<TIn>();
  float m = -INFINITY;
  for (int s0 = s_lo + warp; s0 < s_hi; s0 += kFinalWarps * U) {
    Seg8<TIn> t[U];
#pragma unroll
    for (int q = 0; q < U; ++q) {
      const int seg = s0 + q * kFinalWarps;
      if (seg < s_hi) seg_load(t[q], row, seg * kSegElems + lane * 8, V, vec_ok);
    }
#pragma unroll
    for (int q = 0; q < U; ++q) {
      if (s0 + q * kFinalWarps >= s_hi) break;
      float z[8];
      seg_unpack(t[q], z);
#pragma unroll
      for (int e = 0; e < 8; ++e) m = fmaxf(m, z[e]);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (lane == 0) sh.warp_f[warp].x = m;
  __syncthreads();
  float r = -INFINITY;
#pragma unroll
  for (int w = 0; w < kFinalWarps; ++w) r = fmaxf(r, sh.warp_f[w].x);
  __syncthreads();
  return r;
}

// Largest entry of segments [s_lo, s_hi) and its lowest index (block-wide).
template <typename TIn>
__device__ ArgAcc slice_argmax(const TIn* row, int V, int s_lo, int s_hi, bool vec_ok,
                               FinalShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int U = 2 * seg_batch<TIn>();
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
      float z[8];
      seg_unpack(t[q], z);
      const int e0 = seg * kSegElems + lane * 8;
#pragma unroll
      for (int e = 0; e < 8; ++e) arg_add(a, z[e], e0 + e);
    }
  }
  arg_warp_reduce(a);
  if (lane == 0) sh.warp_f[warp] = make_float4(a.v, __int_as_float(a.i), 0.f, 0.f);
  __syncthreads();
  ArgAcc r;
  arg_init(r);
#pragma unroll
  for (int w = 0; w < kFinalWarps; ++w) {
    ArgAcc o;
    o.v = sh.warp_f[w].x;
    o.i = __float_as_int(sh.warp_f[w].y);
    arg_merge(r, o);
  }
  __syncthreads();
  return r;
}

// How the masses of one request were formed, for the re-scan.
struct MassSpec {
  float sc;
  float a_hi, a_lo;      // p's normaliser (residual, or p alone)
  float cd_hi, cd_lo;    // q's normaliser (residual)
  bool has_q;
  bool slice_ref;        // bonus: p's reference is the segment's slice reference
};

// Inverse CDF over the request's segment masses (global, nseg entries, each
// scaled by sh.scale[slice]): the first entry whose cumulative mass exceeds
// u * total.  Block-wide; returns the token, or -1 if the total mass is not
// a finite positive number.
template <typename TIn>
__device__ int cdf_pick(const TIn* rt, const TIn* rd, int V, const MassSpec& ms,
                        const float* slice_ref, int P, double u, const float* seg_mass, int nseg,
                        bool vec_ok, FinalShared& sh, double* seg_excl, float* seg_val) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int s = threadIdx.x; s < nseg; s += kFinalThreads) seg_val[s] = __ldcg(&seg_mass[s]);
  __syncthreads();
  // Exclusive prefix of the scaled segment masses, in double.
  const int per = (nseg + kFinalThreads - 1) / kFinalThreads;
  const int sa = min(nseg, (int)threadIdx.x * per), sb = min(nseg, sa + per);
  double loc = 0.0;
  for (int s = sa; s < sb; ++s) loc += (double)seg_val[s] * (double)sh.scale[slice_of(s, nseg, P)];
  double total;
  double run = block_exclusive_scan_f64(loc, sh, &total);
  for (int s = sa; s < sb; ++s) {
    seg_excl[s] = run;
    run += (double)seg_val[s] * (double)sh.scale[slice_of(s, nseg, P)];
  }
  if (!(total > 0.0 && total <= 1.79e308)) return -1;  // uniform across the block
  const double target = u * total;

  // The last segment with positive mass that starts at or before target.
  if (threadIdx.x == 0) sh.cand = -1;
  __syncthreads();
  int cand = -1;
  for (int s = sa; s < sb; ++s)
    if (seg_val[s] > 0.0f && sh.scale[slice_of(s, nseg, P)] > 0.0f && seg_excl[s] <= target) cand = s;
  if (cand >= 0) atomicMax(&sh.cand, cand);
  __syncthreads();
  const int j = sh.cand;

  // Re-read segment j: the first entry whose cumulative mass exceeds the
  // target, or the segment's last entry with mass when rounding left the
  // target just past the segment's own sum.
  if (warp == 0) {
    const int pj = slice_of(j, nseg, P);
    const double scale = (double)sh.scale[pj];
    const float a_hi = ms.slice_ref ? __ldcg(&slice_ref[pj]) : ms.a_hi;
    const float a_lo = ms.slice_ref ? 0.0f : ms.a_lo;
    const int e0 = j * kSegElems + lane * 8;
    float zt[8], zd[8];
    load8(rt, e0, V, vec_ok, zt);
    if (ms.has_q) load8(rd, e0, V, vec_ok, zd);
    float r[8], c[8];
    float run_f = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      r[e] = entry_mass(zt[e], ms.has_q ? zd[e] : 0.f, ms.sc, a_hi, a_lo, ms.cd_hi, ms.cd_lo,
                        ms.has_q);
      run_f = __fadd_rn(run_f, r[e]);
      c[e] = run_f;
    }
    float incl = run_f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl = __fadd_rn(incl, y);
    }
    float lex = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) lex = 0.0f;
    const double tprime = target - seg_excl[j];
    int first_e = 8, last_pos = -1;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float cum = __fadd_rn(lex, c[e]);
      if (first_e == 8 && r[e] > 0.0f && (double)cum * scale > tprime) first_e = e;
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
  const int t = sh.token;
  __syncthreads();
  return t;
}

template <typename TIn>
__global__ void __launch_bounds__(kFinalThreads, 4) final_kernel(FinalParams p) {
  extern __shared__ __align__(16) unsigned char fsm_raw[];
  __shared__ FinalShared sh;
  const int nseg = segments_of(p.V);
  double* seg_excl = reinterpret_cast<double*>(fsm_raw);
  float* seg_val = reinterpret_cast<float*>(fsm_raw + (size_t)nseg * sizeof(double));

  pdl_wait();
  const int part = blockIdx.x, b = blockIdx.y, P = gridDim.x;
  WsHeader* h = reinterpret_cast<WsHeader*>(p.ws + p.lay.header);
  const int32_t* flags = reinterpret_cast<const int32_t*>(p.ws + p.lay.flags);
  const uint32_t* acc_bits = reinterpret_cast<const uint32_t*>(p.ws + p.lay.acc_bits);
  const uint32_t* dec_bits = reinterpret_cast<const uint32_t*>(p.ws + p.lay.dec_bits);
  const uint32_t* bad_bits = reinterpret_cast<const uint32_t*>(p.ws + p.lay.bad_bits);
  const double* pos_c = reinterpret_cast<const double*>(p.ws + p.lay.pos_c);
  const int32_t* pos_arg = reinterpret_cast<const int32_t*>(p.ws + p.lay.pos_arg);
  float* seg_mass = reinterpret_cast<float*>(p.ws + p.lay.seg_mass) + (size_t)b * nseg;
  float* slice_ref = reinterpret_cast<float*>(p.ws + p.lay.slice_ref) + (size_t)b * kMaxSlices;
  int32_t* slice_arg = reinterpret_cast<int32_t*>(p.ws + p.lay.slice_arg) + (size_t)b * kMaxSlices;
  int32_t* final_done = reinterpret_cast<int32_t*>(p.ws + p.lay.final_done);
  const int L = p.lengths[b];
  const float T = p.temperature[b];

  // n from the decision masks: the first rejected position, or L.
  if (threadIdx.x == 0) {
    const int f = __ldcg(&flags[b]);
    int job = kJobInvalid, n = -1, token = -1;
    if (f & kReqValid) {
      const uint32_t dec = __ldcg(&dec_bits[b]), acc = __ldcg(&acc_bits[b]);
      const uint32_t bad = __ldcg(&bad_bits[b]);
      const uint32_t lmask = (L >= 32) ? 0xffffffffu : ((1u << L) - 1u);
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
          token = __ldcg(&pos_arg[(size_t)b * p.k + n]);
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
  }
  __syncthreads();
  const int job = sh.job;
  const int n = sh.n;
  int token = sh.token;
  __syncthreads();

  auto write_outputs = [&](bool invalid, int final_token) {
    for (int j = threadIdx.x; j <= p.k; j += kFinalThreads) {
      int v = -1;
      if (!invalid) {
        if (j < n) v = p.tokens[(size_t)b * p.k + j];
        else if (j == n) v = final_token;
      }
      p.out_tokens[(size_t)b * (p.k + 1) + j] = v;
    }
    if (threadIdx.x == 0) p.num_accepted[b] = invalid ? -1 : n;
  };
  if (job == kJobNone || job == kJobInvalid) {
    if (part == 0) write_outputs(job == kJobInvalid, token);
    return;
  }

  // ---- this slice's share of the row(s) ----
  const TIn* trow = static_cast<const TIn*>(p.target) + ((size_t)b * (p.k + 1) + n) * (size_t)p.V;
  const TIn* drow = job == kJobResidual
                        ? static_cast<const TIn*>(p.draft) + ((size_t)b * p.k + n) * (size_t)p.V
                        : nullptr;
  const bool vec_ok =
      ((reinterpret_cast<uintptr_t>(trow) | reinterpret_cast<uintptr_t>(drow)) & 15u) == 0;
  const int s_lo = slice_lo(part, nseg, P), s_hi = slice_lo(part + 1, nseg, P);
  const float sc = job == kJobGreedyRowL ? 0.0f : softmax_scale(T);
  MassSpec ms = {};
  ms.sc = sc;
  if (job == kJobResidual) {
    const double ct = __ldcg(&pos_c[((size_t)b * p.k + n) * 2]);
    const double cd = __ldcg(&pos_c[((size_t)b * p.k + n) * 2 + 1]);
    ms.a_hi = (float)ct;
    ms.a_lo = (float)(ct - (double)ms.a_hi);
    ms.cd_hi = (float)cd;
    ms.cd_lo = (float)(cd - (double)ms.cd_hi);
    ms.has_q = true;
    slice_masses(trow, drow, p.V, sc, ms.a_hi, ms.a_lo, ms.cd_hi, ms.cd_lo, s_lo, s_hi, seg_mass,
                 vec_ok);
  } else if (job == kJobBonus) {
    // Reference: this slice's max (an all -inf slice keeps -FLT_MAX and zero mass).
    const float m = slice_max(trow, p.V, s_lo, s_hi, vec_ok, sh);
    const float ref = (m == -INFINITY) ? -FLT_MAX : __fmul_rn(m, sc);
    ms.slice_ref = true;
    slice_masses(trow, static_cast<const TIn*>(nullptr), p.V, sc, ref, 0.0f, 0.0f, 0.0f, s_lo,
                 s_hi, seg_mass, vec_ok);
    if (threadIdx.x == 0) __stcg(&slice_ref[part], ref);
  } else {
    const ArgAcc a = slice_argmax(trow, p.V, s_lo, s_hi, vec_ok, sh);
    if (threadIdx.x == 0) {
      __stcg(&slice_ref[part], a.v);
      __stcg(&slice_arg[part], a.i);
    }
  }

  // ---- the last slice CTA of the request combines ----
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    sh.last = atomicAdd(&final_done[b], 1) == P - 1;
  }
  __syncthreads();
  if (!sh.last) return;
  __threadfence();

  bool bad = false;
  if (job == kJobGreedyRowL) {
    if (threadIdx.x == 0) {
      ArgAcc r;
      arg_init(r);
      for (int q = 0; q < P; ++q) {
        ArgAcc o;
        o.v = __ldcg(&slice_ref[q]);
        o.i = __ldcg(&slice_arg[q]);
        arg_merge(r, o);
      }
      sh.token = r.i;
    }
    __syncthreads();
    token = sh.token;
    bad = (token == INT32_MAX);
  } else {
    // Per-slice scale: 2^(ref_p - max ref) for the bonus, 1 for a residual.
    if (threadIdx.x < 32) {
      const int q = threadIdx.x;
      float r = (job == kJobBonus && q < P) ? __ldcg(&slice_ref[q]) : -FLT_MAX;
      float rm = r;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) rm = fmaxf(rm, __shfl_xor_sync(0xffffffffu, rm, off));
      if (q < P && q < kMaxSlices) {
        sh.scale[q] = job == kJobBonus
                          ? (r > -FLT_MAX ? exp2f((float)((double)r - (double)rm)) : 0.0f)
                          : 1.0f;
      }
    }
    __syncthreads();
    const double u = (double)p.uniforms[(size_t)b * (p.k + 1) + L];
    token = cdf_pick(trow, drow, p.V, ms, slice_ref, P, u, seg_mass, nseg, vec_ok, sh, seg_excl,
                     seg_val);
    if (token < 0 && job == kJobResidual) {
      // Residual mass zero (p_n == q_n up to rounding): draw from p_n.
      if (threadIdx.x == 0) atomicAdd(&h->residual_zero, 1);
      MassSpec pm = ms;
      pm.has_q = false;
      slice_masses(trow, static_cast<const TIn*>(nullptr), p.V, sc, pm.a_hi, pm.a_lo, 0.0f, 0.0f,
                   0, nseg, seg_mass, vec_ok);
      __syncthreads();
      token = cdf_pick(trow, static_cast<const TIn*>(nullptr), p.V, pm, slice_ref, P, u, seg_mass,
                       nseg, vec_ok, sh, seg_excl, seg_val);
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

}  // namespace specv
