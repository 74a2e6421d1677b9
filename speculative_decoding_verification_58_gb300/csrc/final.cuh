// Final pass: one CTA per request.
//
// Reads the per-position decisions the sweep recorded, finds n (the first
// rejected position, or L if none), and emits the round's n + 1 tokens
// (DFlash notes, section 3.1, steps 6-7):
//   - sampling, n < L: one token from normalize(max(0, p_n - q_n)) (AdaFlash
//     Section 2.1; AdaFlash reading notes, basic idea, step 4);
//   - sampling, n == L: one token from p_L (target row L, read only now);
//   - greedy, n < L: the target argmax at n, already known from the sweep;
//   - greedy, n == L: the argmax of target row L.
// Sampling is by inverse CDF in ascending vocabulary index with u_L: the row
// is streamed once to get per-segment masses (256 entries per segment), the
// segment prefix sums are formed in double, and one segment is re-read to
// place u_L * total exactly.
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
  int32_t* out_tokens;
  int32_t* num_accepted;
  unsigned char* ws;
  WsLayout lay;
};

constexpr int kFinalWarps = kFinalThreads / 32;
constexpr int kJobNone = 0, kJobResidual = 1, kJobBonus = 2, kJobGreedyRowL = 3, kJobInvalid = 4;

// Shared scratch of the final kernel; seg arrays are dynamic (sized by V).
struct FinalShared {
  double warp_d[kFinalWarps + 1];
  float4 warp_f[kFinalWarps];
  int job, n, token, cand, bad;
  double c;
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

// Probability mass of one entry in the distribution being sampled:
// max(0, p - q) for a residual, p for the bonus (no draft row).  The same
// instruction sequence is used in the segment pass and the re-scan so both
// see bit-identical values.
__device__ __forceinline__ float entry_mass(float zt, float zd, float sc, float ct_hi, float ct_lo,
                                            float cd_hi, float cd_lo, bool has_q) {
  const float p = ex2(__fsub_rn(fmaf(zt, sc, -ct_hi), ct_lo));
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
    double y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) sh.warp_d[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    double w = sh.warp_d[lane];
    double wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      double y = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += y;
    }
    sh.warp_d[lane] = wi - w;
    if (lane == 31) sh.warp_d[kFinalWarps] = wi;
  }
  __syncthreads();
  const double ex = (incl - x) + sh.warp_d[warp];
  *total = sh.warp_d[kFinalWarps];
  __syncthreads();
  return ex;
}

// Whole-row online softmax statistics (CTA-wide), as in the sweep.  Returns
// false if the row has no finite mass.  c = fl(M*sc) + log2(S).
template <typename TIn>
__device__ bool row_normaliser_cta(const TIn* row, int V, float sc, FinalShared& sh, double* c) {
  using Tr = ElemTraits<TIn>;
  constexpr int EPV = Tr::kPerVec;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  SoftAcc a;
  soft_init(a);
  const bool vec_ok = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  int done = 0;
  if (vec_ok) {
    const int nvec = (int)(((long long)V * Tr::kSize) >> 4);
    const uint4* v = reinterpret_cast<const uint4*>(row);
#pragma unroll 4
    for (int j = threadIdx.x; j < nvec; j += kFinalThreads) {
      float x[EPV];
      Tr::unpack(__ldg(v + j), x);
      soft_add<EPV>(a, x, sc);
    }
    done = nvec * EPV;
  }
  for (int e = done + threadIdx.x; e < V; e += kFinalThreads) soft_add1(a, Tr::load(row, e), sc);
  soft_warp_reduce(a);
  if (lane == 0) sh.warp_f[warp] = make_float4(a.m, a.ms, a.s, 0.f);
  __syncthreads();
  if (warp == 0) {
    SoftAcc r;
    r.m = sh.warp_f[lane].x;
    r.ms = sh.warp_f[lane].y;
    r.s = sh.warp_f[lane].z;
    soft_warp_reduce(r);
    if (lane == 0) {
      const double S = (double)r.s;
      sh.c = (double)r.ms + log2_pos(S);
      sh.bad = !(S > 0.0 && S <= 3.4e38);
    }
  }
  __syncthreads();
  *c = sh.c;
  const bool ok = !sh.bad;
  __syncthreads();
  return ok;
}

// Whole-row argmax (lowest index on ties), CTA-wide.
template <typename TIn>
__device__ int row_argmax_cta(const TIn* row, int V, FinalShared& sh) {
  using Tr = ElemTraits<TIn>;
  constexpr int EPV = Tr::kPerVec;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  ArgAcc a;
  arg_init(a);
  const bool vec_ok = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  int done = 0;
  if (vec_ok) {
    const int nvec = (int)(((long long)V * Tr::kSize) >> 4);
    const uint4* v = reinterpret_cast<const uint4*>(row);
#pragma unroll 4
    for (int j = threadIdx.x; j < nvec; j += kFinalThreads) {
      float x[EPV];
      Tr::unpack(__ldg(v + j), x);
#pragma unroll
      for (int e = 0; e < EPV; ++e) arg_add(a, x[e], j * EPV + e);
    }
    done = nvec * EPV;
  }
  for (int e = done + threadIdx.x; e < V; e += kFinalThreads) arg_add(a, Tr::load(row, e), e);
  arg_warp_reduce(a);
  if (lane == 0) sh.warp_f[warp] = make_float4(a.v, __int_as_float(a.i), 0.f, 0.f);
  __syncthreads();
  if (warp == 0) {
    ArgAcc r;
    r.v = sh.warp_f[lane].x;
    r.i = __float_as_int(sh.warp_f[lane].y);
    arg_warp_reduce(r);
    if (lane == 0) sh.token = r.i;
  }
  __syncthreads();
  const int t = sh.token;
  __syncthreads();
  return t;
}

// Inverse-CDF sample of the distribution with entry masses entry_mass(...)
// at uniform u.  Returns the token, or -1 if the total mass is zero.
template <typename TIn>
__device__ int sample_row(const TIn* rt, const TIn* rd, int V, float sc, double ct, double cd,
                          double u, FinalShared& sh, float* seg_sum, double* seg_excl) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool has_q = (rd != nullptr);
  const float ct_hi = (float)ct, ct_lo = (float)(ct - (double)ct_hi);
  const float cd_hi = (float)cd, cd_lo = (float)(cd - (double)cd_hi);
  const bool vec_ok = ((reinterpret_cast<uintptr_t>(rt) | reinterpret_cast<uintptr_t>(rd)) & 15u) == 0;
  const int nseg = (V + kSegElems - 1) / kSegElems;

  // 1) Segment masses: warp w takes segments w, w + 32, ...; lane l holds
  //    entries 8l..8l+7 of the segment.
  constexpr int U = 2;
  for (int s0 = warp; s0 < nseg; s0 += kFinalWarps * U) {
    float zt[U][8], zd[U][8];
#pragma unroll
    for (int q = 0; q < U; ++q) {
      const int seg = s0 + q * kFinalWarps;
      const int e0 = seg * kSegElems + lane * 8;
      if (seg < nseg) {
        load8(rt, e0, V, vec_ok, zt[q]);
        if (has_q) load8(rd, e0, V, vec_ok, zd[q]);
      }
    }
#pragma unroll
    for (int q = 0; q < U; ++q) {
      const int seg = s0 + q * kFinalWarps;
      if (seg >= nseg) break;
      float m = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e)
        m = __fadd_rn(m, entry_mass(zt[q][e], has_q ? zd[q][e] : 0.f, sc, ct_hi, ct_lo, cd_hi,
                                    cd_lo, has_q));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = __fadd_rn(m, __shfl_xor_sync(0xffffffffu, m, off));
      if (lane == 0) seg_sum[seg] = m;
    }
  }
  __syncthreads();

  // 2) Exclusive prefix sums over segments in double.
  const int per = (nseg + kFinalThreads - 1) / kFinalThreads;
  const int sa = min(nseg, (int)threadIdx.x * per), sb = min(nseg, sa + per);
  double loc = 0.0;
  for (int s = sa; s < sb; ++s) loc += (double)seg_sum[s];
  double total;
  double run = block_exclusive_scan_f64(loc, sh, &total);
  for (int s = sa; s < sb; ++s) {
    seg_excl[s] = run;
    run += (double)seg_sum[s];
  }
  if (!(total > 0.0)) return -1;  // uniform across the block
  const double target = u * total;

  // 3) The last segment with positive mass that starts at or before target.
  if (threadIdx.x == 0) sh.cand = -1;
  __syncthreads();
  int cand = -1;
  for (int s = sa; s < sb; ++s)
    if (seg_sum[s] > 0.0f && seg_excl[s] <= target) cand = s;
  if (cand >= 0) atomicMax(&sh.cand, cand);
  __syncthreads();
  const int j = sh.cand;

  // 4) Re-read that segment and find the first entry whose cumulative mass
  //    exceeds the target (or the segment's last entry with mass, when
  //    rounding left the target just past the segment's own sum).
  if (warp == 0) {
    const int e0 = j * kSegElems + lane * 8;
    float zt[8], zd[8];
    load8(rt, e0, V, vec_ok, zt);
    if (has_q) load8(rd, e0, V, vec_ok, zd);
    float r[8], c[8];
    float run_f = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      r[e] = entry_mass(zt[e], has_q ? zd[e] : 0.f, sc, ct_hi, ct_lo, cd_hi, cd_lo, has_q);
      run_f = __fadd_rn(run_f, r[e]);
      c[e] = run_f;
    }
    // Exclusive prefix of the lane totals.
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
      if (first_e == 8 && r[e] > 0.0f && (double)cum > tprime) first_e = e;
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
__global__ void __launch_bounds__(kFinalThreads, 1) final_kernel(FinalParams p) {
  extern __shared__ __align__(16) unsigned char fsm_raw[];
  __shared__ FinalShared sh;
  const int nseg = (p.V + kSegElems - 1) / kSegElems;
  double* seg_excl = reinterpret_cast<double*>(fsm_raw);
  float* seg_sum = reinterpret_cast<float*>(fsm_raw + (size_t)nseg * sizeof(double));

  pdl_wait();
  const int b = blockIdx.x;
  WsHeader* h = reinterpret_cast<WsHeader*>(p.ws + p.lay.header);
  const int32_t* flags = reinterpret_cast<const int32_t*>(p.ws + p.lay.flags);
  const uint32_t* acc_bits = reinterpret_cast<const uint32_t*>(p.ws + p.lay.acc_bits);
  const uint32_t* dec_bits = reinterpret_cast<const uint32_t*>(p.ws + p.lay.dec_bits);
  const uint32_t* bad_bits = reinterpret_cast<const uint32_t*>(p.ws + p.lay.bad_bits);
  const double* pos_c = reinterpret_cast<const double*>(p.ws + p.lay.pos_c);
  const int32_t* pos_arg = reinterpret_cast<const int32_t*>(p.ws + p.lay.pos_arg);
  const int L = p.lengths[b];
  const float T = p.temperature[b];

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
        record_status(h, SPEC_ERR_INTERNAL);
        n = -1;
      } else if (bad & (n < L ? ((prefix << 1) | 1u) : lmask)) {
        atomicAdd(&h->bad_requests, 1);
        atomicMin(&h->first_bad, b);
        record_status(h, SPEC_ERR_BAD_INPUT);
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

  const TIn* trow_n = static_cast<const TIn*>(p.target) + ((size_t)b * (p.k + 1) + (n < 0 ? 0 : n)) * (size_t)p.V;
  bool bad = false;
  if (job == kJobGreedyRowL) {
    token = row_argmax_cta<TIn>(trow_n, p.V, sh);
    bad = (token == INT32_MAX);
    if (threadIdx.x == 0) {
      atomicAdd(&h->final_rows, 1ull);
      atomicAdd(&h->final_bytes, (unsigned long long)p.V * sizeof(TIn));
    }
  } else if (job == kJobResidual || job == kJobBonus) {
    const float sc = softmax_scale(T);
    const double u = (double)p.uniforms[(size_t)b * (p.k + 1) + L];
    double ct, cd = 0.0;
    const TIn* drow = nullptr;
    if (job == kJobResidual) {
      ct = __ldcg(&pos_c[((size_t)b * p.k + n) * 2]);
      cd = __ldcg(&pos_c[((size_t)b * p.k + n) * 2 + 1]);
      drow = static_cast<const TIn*>(p.draft) + ((size_t)b * p.k + n) * (size_t)p.V;
    } else {
      bad = !row_normaliser_cta<TIn>(trow_n, p.V, sc, sh, &ct);
    }
    if (!bad) {
      token = sample_row<TIn>(trow_n, drow, p.V, sc, ct, cd, u, sh, seg_sum, seg_excl);
      if (token < 0 && drow != nullptr) {
        // Residual mass zero (p_n == q_n up to rounding): draw from p_n.
        if (threadIdx.x == 0) atomicAdd(&h->residual_zero, 1);
        token = sample_row<TIn>(trow_n, nullptr, p.V, sc, ct, 0.0, u, sh, seg_sum, seg_excl);
      }
      bad = (token < 0);
    }
    if (threadIdx.x == 0) {
      atomicAdd(&h->final_rows, drow ? 2ull : 1ull);
      atomicAdd(&h->final_bytes, (drow ? 2ull : 1ull) * p.V * sizeof(TIn));
    }
  }
  if (bad && threadIdx.x == 0) {
    atomicAdd(&h->bad_requests, 1);
    atomicMin(&h->first_bad, b);
    record_status(h, SPEC_ERR_BAD_INPUT);
  }
  const bool invalid = (job == kJobInvalid) || bad;

  // Outputs: x_0..x_{n-1}, the final token, then -1.
  for (int j = threadIdx.x; j <= p.k; j += kFinalThreads) {
    int v = -1;
    if (!invalid) {
      if (j < n) v = p.tokens[(size_t)b * p.k + j];
      else if (j == n) v = token;
    }
    p.out_tokens[(size_t)b * (p.k + 1) + j] = v;
  }
  if (threadIdx.x == 0) p.num_accepted[b] = invalid ? -1 : n;
}

}  // namespace specv
