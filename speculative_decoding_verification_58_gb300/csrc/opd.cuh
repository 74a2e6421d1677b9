// On-policy distillation (OPD) supervision statistics, AdaFlash Section 3.1.
//
// For request b and every verified position i < L_b, with p = softmax of
// target row i and q = softmax of draft row i (temperature 1):
//   x*        = argmax_y p(y)                       (lowest index on ties)
//   hard      = -log q(x*)                          (hard-label term)
//   rkl       = sum_y q(y) log(q(y) / p(y))         (reverse KL)
//   rkl_clip  = sum_y min{ q(y) log(q(y) / p(y)), delta }   (entry-wise clipping)
// and per request loss = alpha * mean_i hard + (1 - alpha) * mean_i rkl_clip
// (the mixture OPD loss; the mean runs over the L_b verified positions).
//
// The clipped sum needs both normalisers before its first term, so every
// logit is used twice: pass 1 folds it into softmax and argmax partials, pass
// 2 into the sums.  A cluster of CS CTAs (4 for large vocabularies) owns one
// position at a time, each CTA one CS-th of the vocabulary of both rows.  A
// producer warp streams its part through a shared-memory ring with bulk
// copies; eight consumer warps compute; a bookkeeping warp merges the
// consumers' partials, sends them to the other CTAs of the cluster through
// distributed shared memory (remote store + remote mbarrier arrive), and
// every CTA combines all parts in rank order into the same normalisers.  Pass
// 2 of a position is streamed one position after its pass 1, so the
// exchange is off the consumers' path, and the second read of each part (a
// CTA's last few hundred kilobytes) is served by L2: pass 1 loads carry an
// evict-last hint, pass 2 loads evict-first.  Two CTAs per SM.  Clusters
// that would hold whole rows in shared memory need 8 or 16 CTAs, which leave
// a fifth of GB300's SMs idle.
//
// Verification in the same pass (spec_verify_opd): the statistics read every
// verified row pair anyway, so the same kernel also decides each position of
// a valid request at T = 1 (the statistics' own normalisers: accept iff
// u_i < min(1, p(x_i) / q(x_i)), AdaFlash Section 2.1) or T = 0 (accept iff
// x_i is the target argmax) and publishes the decision, the row normalisers
// and the argmax exactly as the row sweep does, so that the final pass
// samples the residual or bonus token unchanged.  Requests at any other
// temperature are left to the row sweep, which runs after this kernel.
#pragma once

#include "common.cuh"

namespace specv {

constexpr int kOpdConsumerWarps = 8;
constexpr int kOpdMaxCluster = 4;
constexpr int kOpdBookWarp = 0, kOpdProducerWarp = 1, kOpdFirstConsumerWarp = 2;
constexpr int kOpdThreads = (kOpdConsumerWarps + 2) * 32;
constexpr int kOpdNC = kOpdConsumerWarps * 32;      // consumer threads
constexpr int kOpdStages = 3;
constexpr int kOpdMinBlocks = 2;  // CTAs per SM the register budget is sized for
constexpr int kOpdPieceBytes = 16384;               // one row's part of a stage
constexpr int kOpdStageBytes = 2 * kOpdPieceBytes;  // target piece, then draft piece
constexpr int kOpdVecPerThread = kOpdPieceBytes / 16 / kOpdNC;  // 16-byte vectors per row
static_assert(kOpdVecPerThread * 16 * kOpdNC == kOpdPieceBytes, "a piece splits evenly");

struct OpdParams {
  const void* target;      // [B, k+1, V]
  const void* draft;       // [B, k, V]
  const int32_t* lengths;  // [B]
  // Verification in the same pass (verify != 0): inputs, and the workspace the
  // plan kernel prepared and the final pass reads.
  int verify;
  const int32_t* tokens;     // [B, k]
  const float* uniforms;     // [B, k+1]
  const float* temperature;  // [B]
  unsigned char* ws;
  WsLayout lay;
  int B, k, V;
  int slice;     // elements of each row per CTA of a cluster (multiple of 8)
  int vec_ok;    // rows 16-byte aligned: bulk copies; else ordinary loads
  float delta;
  int32_t* x_star;  // [B, k]
  float* hard;      // [B, k]
  float* rkl;       // [B, k]
  float* rkl_clip;  // [B, k]
};

struct OpdStageInfo {
  int j;     // index of the position in this cluster's list
  int pass;  // 1 or 2
  int e0;    // first element of the stage within this CTA's part of the rows
  int ne;    // elements of each row in the stage
  int last;  // last stage of the pass over this CTA's part
};

// Pass-1 partial of a CTA (or a consumer warp): both rows' softmax partials
// and the target's argmax.  32 bytes, moved as two float4.
struct __align__(16) OpdP1 {
  float mt, mst, st;
  float md, msd, sd;
  float argv;
  int argi;
};
// Pass-2 partial: unclipped and clipped sums (float-float) and whether some
// unclipped term was +inf.
struct __align__(16) OpdP2 {
  float kl_hi, kl_lo, kc_hi, kc_lo;
  int inf;
  int pad[3];
};

struct OpdSmem {
  unsigned char ring[kOpdStages][kOpdStageBytes];
  OpdStageInfo info[kOpdStages];
  uint64_t full[kOpdStages], empty[kOpdStages];
  // Per position slot (j & 1): consumer warps done with pass 1 / pass 2,
  // normalisers published, the other CTA's partials arrived.
  uint64_t p1_done[2], p2_done[2], norm_ready[2], peer1[2], peer2[2];
  OpdP1 p1w[2][kOpdConsumerWarps];
  OpdP2 p2w[2][kOpdConsumerWarps];
  OpdP1 p1_peer[2][kOpdMaxCluster];  // [slot][sender rank], written by the other CTAs
  OpdP2 p2_peer[2][kOpdMaxCluster];
  float4 norms[2];   // c = lse_d - lse_t, -lse_d log2 e, lse_d, valid
  int nx[2];         // x*
  int abort_flag;
};

// ---------------------------------------------------------------------------
// Cluster and cache-policy helpers (inline PTX).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_map(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void dsmem_st4(uint32_t a, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}
// Arrive on an mbarrier of another CTA of the cluster, releasing this
// thread's earlier writes (the DSMEM stores before it) at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                   bar_cluster_addr)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for a phase the other CTA completes (acquire at cluster scope).
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, uint32_t parity,
                                                          volatile int* abort) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 63) == 63) {
      if (*abort) return false;
      if (global_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}
// Per-element pass-2 term q log(q/p) = q (dz - c) with dz = z_d - z_t,
// c = lse_d - lse_t and q = 2^(z_d log2 e + nl2d), nl2d = -lse_d log2 e.
// Only infinite logits make it non-finite; then 0 log 0 = 0 (z_d = -inf)
// and q > 0 where p = 0 gives +inf.
struct OpdSums {
  float kl, kc;
  int inf;
};

__device__ __forceinline__ void opd_add(OpdSums& s, float zt, float zd, float c, float nl2d,
                                        float delta) {
  const float q = ex2(fmaf(zd, kLog2e, nl2d));
  const float dz = __fsub_rn(zd, zt);
  float t = __fmul_rn(q, __fsub_rn(dz, c));
  if (!(fabsf(t) <= FLT_MAX)) {
    t = (zd == -INFINITY) ? 0.0f : INFINITY;
    if (t == INFINITY) {
      s.inf = 1;
      t = 0.0f;
      s.kc = __fadd_rn(s.kc, delta);
    }
  } else {
    s.kc = __fadd_rn(s.kc, fminf(t, delta));
  }
  s.kl = __fadd_rn(s.kl, t);
}

// The next position of this cluster, q, q + ncl, ... that has a verified row
// pair (i < L_b, L_b valid); -1 when there is none.
__device__ __forceinline__ int opd_next_active(const OpdParams& p, int q, int ncl) {
  const int npos = p.B * p.k;
  for (; q < npos; q += ncl) {
    const int b = q / p.k, i = q - b * p.k;
    const int L = __ldg(&p.lengths[b]);
    if (L >= 1 && L <= p.k && i < L) return q;
  }
  return -1;
}

// Every role walks the same unit sequence over this cluster's active
// positions: P1(0), P1(1), P2(0), P1(2), P2(1), ..., P2(m-1).  Pass 2 of a
// position comes one position after its pass 1, so the cluster's exchange of
// normalisers never holds the consumers up.
template <typename F>
__device__ __forceinline__ void opd_walk(const OpdParams& p, int cid, int ncl, F&& unit) {
  int q_prev = -1;
  int q = opd_next_active(p, cid, ncl);
  for (int j = 0;; ++j) {
    if (q >= 0 && !unit(q, j, 1)) return;
    if (j >= 1 && !unit(q_prev, j - 1, 2)) return;
    if (q < 0) return;
    q_prev = q;
    q = opd_next_active(p, q + ncl, ncl);
  }
}

__device__ __forceinline__ void opd_abort(OpdSmem& sm) {
  *(volatile int*)&sm.abort_flag = 1;
}

// ---------------------------------------------------------------------------
// Producer warp: this CTA's part of both rows, chunk by chunk, into the ring.
// ---------------------------------------------------------------------------
template <typename TIn>
__device__ void opd_producer(const OpdParams& p, OpdSmem& sm, int cid, int ncl, int s0) {
  const int lane = threadIdx.x & 31;
  constexpr int CH = kOpdPieceBytes / (int)sizeof(TIn);  // elements of a row per stage
  const int n = max(0, min(p.slice, p.V - s0));
  const uint64_t pol_keep = l2_policy_evict_last(), pol_drop = l2_policy_evict_first();
  int it = 0;
  opd_walk(p, cid, ncl, [&](int q, int j, int pass) -> bool {
    q = (int)SPEC_CHECKED(q, (long long)p.B * p.k, kSiteOpdRow);
    const int b = q / p.k, i = q - b * p.k;
    const TIn* t = static_cast<const TIn*>(p.target) + ((size_t)b * (p.k + 1) + i) * (size_t)p.V + s0;
    const TIn* d = static_cast<const TIn*>(p.draft) + ((size_t)b * p.k + i) * (size_t)p.V + s0;
    const int nch = n > 0 ? (n + CH - 1) / CH : 1;
    for (int c = 0; c < nch; ++c, ++it) {
      const int s = it % kOpdStages, round = it / kOpdStages;
      if (round > 0 && !mbar_wait_bounded(&sm.empty[s], (round - 1) & 1, &sm.abort_flag)) {
        opd_abort(sm);
        return false;
      }
      const int e0 = c * CH;
      const int ne = max(0, min(CH, n - e0));
      const int core = p.vec_ok ? ((ne * (int)sizeof(TIn)) & ~15) / (int)sizeof(TIn) : 0;
      TIn* dt = reinterpret_cast<TIn*>(sm.ring[s]);
      TIn* dd = reinterpret_cast<TIn*>(sm.ring[s] + kOpdPieceBytes);
      // What the bulk copies cannot take (a ragged end, or every element of
      // rows that are not 16-byte aligned) goes through ordinary loads.
      for (int e = core + lane; e < ne; e += 32) {
        dt[e] = __ldg(t + e0 + e);
        dd[e] = __ldg(d + e0 + e);
      }
      __syncwarp();
      if (lane == 0) {
        sm.info[s] = OpdStageInfo{j, pass, e0, ne, c == nch - 1 ? 1 : 0};
        // The stage was last read with ordinary loads: order those before
        // the copy engine's writes.
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        const uint32_t bytes = (uint32_t)core * sizeof(TIn);
        mbar_arrive_expect_tx(&sm.full[s], 2 * bytes);
        if (bytes > 0) {
          const uint64_t pol = pass == 1 ? pol_keep : pol_drop;
          bulk_g2s_hint(dt, t + e0, bytes, &sm.full[s], pol);
          bulk_g2s_hint(dd, d + e0, bytes, &sm.full[s], pol);
        }
      }
      __syncwarp();
    }
    return true;
  });
}

// ---------------------------------------------------------------------------
// Consumer warps: pass 1 folds a stage into softmax / argmax partials, pass 2
// into the sums; at the end of a pass each warp leaves its partial for the
// bookkeeping warp.
// ---------------------------------------------------------------------------
template <typename TIn>
__device__ void opd_consumers(const OpdParams& p, OpdSmem& sm, int cid, int ncl, int s0) {
  using Tr = ElemTraits<TIn>;
  constexpr int EPV = Tr::kPerVec;
  const int lane = threadIdx.x & 31;
  const int warp = (threadIdx.x >> 5) - kOpdFirstConsumerWarp;
  const int ctid = threadIdx.x - kOpdFirstConsumerWarp * 32;
  const float delta = p.delta;
  int it = 0;
  opd_walk(p, cid, ncl, [&](int q, int j, int pass) -> bool {
    const int slot = j & 1;
    const uint32_t par = (j >> 1) & 1;
    float c = 0.0f, nl2d = 0.0f;
    if (pass == 2) {
      if (!mbar_wait_bounded(&sm.norm_ready[slot], par, &sm.abort_flag)) {
        opd_abort(sm);
        return false;
      }
      const float4 nr = sm.norms[slot];
      c = nr.x;
      nl2d = nr.y;
    }
    SoftAcc at, ad;
    soft_init(at);
    soft_init(ad);
    ArgAcc ag;
    arg_init(ag);
    OpdSums sums = {0.0f, 0.0f, 0};
    for (;;) {
      const int s = it % kOpdStages;
      if (!mbar_wait_bounded(&sm.full[s], (it / kOpdStages) & 1, &sm.abort_flag)) {
        opd_abort(sm);
        return false;
      }
      const OpdStageInfo I = sm.info[s];
      const uint4* rt = reinterpret_cast<const uint4*>(sm.ring[s]);
      const uint4* rd = reinterpret_cast<const uint4*>(sm.ring[s] + kOpdPieceBytes);
      const int nvec = I.ne / EPV;
      uint4 vt[kOpdVecPerThread], vd[kOpdVecPerThread];
#pragma unroll
      for (int u = 0; u < kOpdVecPerThread; ++u) {
        const int v = ctid + u * kOpdNC;
        if (v < nvec) {
          vt[u] = rt[v];
          vd[u] = rd[v];
        }
      }
      // Elements past the last whole vector (a ragged end): one per thread.
      const int rem = I.ne - nvec * EPV;
      float xt = 0.0f, xd = 0.0f;
      if (ctid < rem) {
        xt = Tr::to_float(reinterpret_cast<const TIn*>(sm.ring[s])[nvec * EPV + ctid]);
        xd = Tr::to_float(
            reinterpret_cast<const TIn*>(sm.ring[s] + kOpdPieceBytes)[nvec * EPV + ctid]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[s]);
      ++it;
      if (pass == 1) {
        // The whole batch at once, as in the row sweep: one max and at most one
        // rescale per row, then independent exponentials; vectors past the
        // stage's end are -inf.
        const int base = s0 + I.e0;
        // Only a stage that ends a part is short: the others skip the padding.
        if (nvec < kOpdVecPerThread * kOpdNC) {
#pragma unroll
          for (int u = 0; u < kOpdVecPerThread; ++u) {
            if (ctid + u * kOpdNC >= nvec) {
              vt[u] = neg_inf_vec<TIn>();
              vd[u] = neg_inf_vec<TIn>();
            }
          }
        }
        // One max of the target batch serves its argmax and its softmax.
        const float gmt = batch_max<TIn>(vt);
        arg_stage<TIn>(ag, vt, base + ctid * EPV, kOpdNC * EPV, gmt);
        soft_stage<TIn>(at, vt, kLog2e, gmt);
        soft_stage<TIn>(ad, vd, kLog2e);
        if (ctid < rem) {
          soft_add1(at, xt, kLog2e);
          soft_add1(ad, xd, kLog2e);
          arg_add(ag, xt, base + nvec * EPV + ctid);
        }
      } else {
        // Fast path in packed pairs; only infinite logits make a term
        // non-finite, and then the stage is summed again term by term.
        const float2 m1 = make_float2(-1.0f, -1.0f), l2e = make_float2(kLog2e, kLog2e);
        const float2 n2 = make_float2(nl2d, nl2d), mc = make_float2(-c, -c);
        float2 kl2 = make_float2(0.0f, 0.0f), kc2 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int u = 0; u < kOpdVecPerThread; ++u) {
          const int v = ctid + u * kOpdNC;
          if (v < nvec) {
            float a[EPV], b[EPV];
            Tr::unpack(vt[u], a);
            Tr::unpack(vd[u], b);
#pragma unroll
            for (int e = 0; e < EPV; e += 2) {
              const float2 zt2 = make_float2(a[e], a[e + 1]), zd2 = make_float2(b[e], b[e + 1]);
              const float2 dz = f32x2_fma(zt2, m1, zd2);
              const float2 q = ex2x2(f32x2_fma(zd2, l2e, n2));
              const float2 t = f32x2_mul(q, f32x2_add(dz, mc));
              kl2 = f32x2_add(kl2, t);
              kc2 = f32x2_add(kc2, make_float2(fminf(t.x, delta), fminf(t.y, delta)));
            }
          }
        }
        if (ctid < rem) {
          const float t = __fmul_rn(ex2(fmaf(xd, kLog2e, nl2d)), __fsub_rn(__fsub_rn(xd, xt), c));
          kl2.x = __fadd_rn(kl2.x, t);
          kc2.x = __fadd_rn(kc2.x, fminf(t, delta));
        }
        const float kls = __fadd_rn(kl2.x, kl2.y);
        if (fabsf(kls) <= FLT_MAX) {
          sums.kl = __fadd_rn(sums.kl, kls);
          sums.kc = __fadd_rn(sums.kc, __fadd_rn(kc2.x, kc2.y));
        } else {
#pragma unroll
          for (int u = 0; u < kOpdVecPerThread; ++u) {
            const int v = ctid + u * kOpdNC;
            if (v < nvec) {
              float a[EPV], b[EPV];
              Tr::unpack(vt[u], a);
              Tr::unpack(vd[u], b);
              for (int e = 0; e < EPV; ++e) opd_add(sums, a[e], b[e], c, nl2d, delta);
            }
          }
          if (ctid < rem) opd_add(sums, xt, xd, c, nl2d, delta);
        }
      }
      if (I.last) break;
    }
    // End of the pass over this CTA's part: one partial per warp.
    if (pass == 1) {
      soft_warp_reduce(at);
      soft_warp_reduce(ad);
      arg_warp_reduce(ag);
      if (lane == 0) {
        sm.p1w[slot][warp] = OpdP1{at.m, at.ms, at.s, ad.m, ad.ms, ad.s, ag.v, ag.i};
        mbar_arrive(&sm.p1_done[slot]);
      }
    } else {
      const FF kl = warp_sum_ff({sums.kl, 0.0f}), kc = warp_sum_ff({sums.kc, 0.0f});
      const int inf = __any_sync(0xffffffffu, sums.inf) ? 1 : 0;
      if (lane == 0) {
        sm.p2w[slot][warp] = OpdP2{kl.hi, kl.lo, kc.hi, kc.lo, inf, {0, 0, 0}};
        mbar_arrive(&sm.p2_done[slot]);
      }
    }
    return true;
  });
}

// Softmax / argmax partial of one OpdP1 as accumulators (lanes without one
// hold the identity).
__device__ __forceinline__ void opd_p1_unpack(const OpdP1& a, bool have, SoftAcc& t, SoftAcc& d,
                                              ArgAcc& g) {
  soft_init(t);
  soft_init(d);
  arg_init(g);
  if (have) {
    t = SoftAcc{a.mt, a.mst, a.st};
    d = SoftAcc{a.md, a.msd, a.sd};
    g = ArgAcc{a.argv, a.argi};
  }
}

// Both rows' base-2 log normalisers L2 = ref + log2(S) (float-float) from the
// parts the lanes hold (lane r: rank r's part; lanes without one hold the
// identity).  Reference exponents: the largest fl(max * scale) of each row;
// the parts' sums are brought to it and added in float-float.  Warp-wide;
// every lane gets the same values.  Returns whether both rows have finite,
// positive mass.
__device__ __forceinline__ bool opd_pair_norms(const SoftAcc& t, const SoftAcc& d, bool have,
                                               FF* l2t, FF* l2d) {
  const float rt = group_max(t.ms, 5), rd = group_max(d.ms, 5);
  FF st = {0.0f, 0.0f}, sd = {0.0f, 0.0f};
  if (have) {
    if (t.s != 0.0f) st = two_prod(t.s, ex2(__fsub_rn(t.ms, rt)));
    if (d.s != 0.0f) sd = two_prod(d.s, ex2(__fsub_rn(d.ms, rd)));
  }
  st = warp_sum_ff(st);
  sd = warp_sum_ff(sd);
  const float St = ff_to_float(st), Sd = ff_to_float(sd);
  *l2t = ff_add_f(two_sum(rt, log2f(st.hi)), __fdiv_rn(st.lo, st.hi) * kLog2e);
  *l2d = ff_add_f(two_sum(rd, log2f(sd.hi)), __fdiv_rn(sd.lo, sd.hi) * kLog2e);
  return St > 0.0f && St <= FLT_MAX && Sd > 0.0f && Sd <= FLT_MAX;
}

// The accept decision of position i of request b (verification mode; one
// thread), published as the row sweep publishes it: normalisers or argmax,
// bad-row bit, first rejection and the decision bits (a rejection releases
// the writes before it).  T is 0 or 1; l2t / l2d: log2 normalisers at
// temperature 1.
template <typename TIn>
__device__ __noinline__ void opd_decide(const OpdParams& p, int b, int i, int x, float T, float u,
                                        float zt_x, float zd_x, ArgAcc g, FF l2t, FF l2d,
                                        bool sums_ok) {
  const size_t bi = (size_t)b * p.k + i;
  bool accept, row_ok;
  if (T == 0.0f) {
    row_ok = (g.i != INT32_MAX);
    accept = (g.i == x);
    __stcg(reinterpret_cast<int32_t*>(p.ws + p.lay.pos_arg) + bi, g.i);
  } else {
    row_ok = sums_ok;
    const float sc = kLog2e;
    // As in the row sweep's decision: a token the target gives probability
    // zero is never accepted, one the drafter gives zero always is;
    // otherwise d = log2 p(x) - log2 q(x) in float-float and 2^d.
    float ratio;
    if (zt_x == -INFINITY) {
      ratio = 0.0f;
    } else if (zd_x == -INFINITY) {
      ratio = 1.0f;
    } else {
      const FF dd = ff_sub(ff_sub(two_prod(zt_x, sc), l2t), ff_sub(two_prod(zd_x, sc), l2d));
      const float df = ff_to_float(dd);
      ratio = df >= 0.0f ? 1.0f : exp2f(df);
    }
    accept = u < ratio;
    __stcg(reinterpret_cast<float4*>(p.ws + p.lay.pos_c) + bi,
           make_float4(l2t.hi, l2t.lo, l2d.hi, l2d.lo));
  }
  if (!row_ok) {
    accept = false;
    atomicOr(reinterpret_cast<uint32_t*>(p.ws + p.lay.bad_bits) + b, 1u << i);
  }
  unsigned long long* state = reinterpret_cast<unsigned long long*>(p.ws + p.lay.state) + b;
  if (!accept) atomicMin(reinterpret_cast<int32_t*>(p.ws + p.lay.first_reject) + b, i);
  if (accept) atomicOr(state, decision_bits(i, true));
  else atom_or_release_u64(state, decision_bits(i, false));
}

// ---------------------------------------------------------------------------
// Bookkeeping warp: merges the consumer warps' partials, exchanges them with
// the other CTA of the cluster, publishes the normalisers (pass 1) or writes
// the position's results (pass 2, rank 0).
// ---------------------------------------------------------------------------
template <typename TIn, bool kVerify>
__device__ void opd_bookkeeper(const OpdParams& p, OpdSmem& sm, int cid, int ncl, uint32_t CS,
                               uint32_t rank) {
  const int lane = threadIdx.x & 31;
  float zstar[2] = {0.0f, 0.0f};  // z_d[x*] per slot, loaded when x* becomes known
  // Every position of this cluster starts as x* = -1 / NaN: positions past
  // L_b keep it, verified ones are overwritten with their results, and a
  // wait that runs out leaves the rest visibly unset.
  if (rank == 0) {
    for (int q = cid + ncl * lane; q < p.B * p.k; q += 32 * ncl) {
      p.x_star[q] = -1;
      p.hard[q] = p.rkl[q] = p.rkl_clip[q] = __int_as_float(0x7fc00000);
    }
    __syncwarp();
  }
  opd_walk(p, cid, ncl, [&](int q, int j, int pass) -> bool {
    const int slot = j & 1;
    const uint32_t par = (j >> 1) & 1;
    const int b = q / p.k, i = q - b * p.k;
    if (pass == 1) {
      // Verification (rank 0, lane 0) of a valid request at T = 0 or 1: what
      // the decision needs, loaded before the wait so that the loads overlap
      // it.  The plan kernel has checked the request's inputs (tokens in
      // range for a valid request).
      int vflags = 0, x = 0;
      float T = 0.0f, u = 0.0f, zt_x = 0.0f, zd_x = 0.0f;
      if (kVerify && rank == 0 && lane == 0) {
        vflags = __ldcg(reinterpret_cast<const int32_t*>(p.ws + p.lay.flags) + b);
        T = __ldg(&p.temperature[b]);
        if (!(T == 0.0f || T == 1.0f)) vflags = 0;  // left to the row sweep
        if (vflags & kReqValid) {
          x = __ldg(&p.tokens[(size_t)b * p.k + i]);
          // A token out of range (the final pass turns its request into -1)
          // reads element 0 instead.
          if ((unsigned)x >= (unsigned)p.V) x = 0;
          if (T != 0.0f) {
            u = __ldg(&p.uniforms[(size_t)b * (p.k + 1) + i]);
            zt_x = ElemTraits<TIn>::load(
                static_cast<const TIn*>(p.target) + ((size_t)b * (p.k + 1) + i) * (size_t)p.V, x);
            zd_x = ElemTraits<TIn>::load(
                static_cast<const TIn*>(p.draft) + ((size_t)b * p.k + i) * (size_t)p.V, x);
          }
        }
      }
      if (!mbar_wait_bounded(&sm.p1_done[slot], par, &sm.abort_flag)) {
        opd_abort(sm);
        return false;
      }
      SoftAcc t, d;
      ArgAcc g;
      opd_p1_unpack(sm.p1w[slot][lane < kOpdConsumerWarps ? lane : 0], lane < kOpdConsumerWarps,
                    t, d, g);
      soft_warp_reduce(t);
      soft_warp_reduce(d);
      arg_warp_reduce(g);
      const OpdP1 mine = {t.m, t.ms, t.s, d.m, d.ms, d.s, g.v, g.i};
      const bool other_rank = lane < (int)CS && lane != (int)rank;
      if (CS > 1) {
        // Lane r sends this CTA's part to CTA r of the cluster.
        if (other_rank) {
          const uint32_t dst = dsmem_map(&sm.p1_peer[slot][rank], (uint32_t)lane);
          dsmem_st4(dst, make_float4(mine.mt, mine.mst, mine.st, mine.md));
          dsmem_st4(dst + 16, make_float4(mine.msd, mine.sd, mine.argv, __int_as_float(mine.argi)));
          mbar_arrive_remote(dsmem_map(&sm.peer1[slot], (uint32_t)lane));
        }
        if (!mbar_wait_cluster_bounded(&sm.peer1[slot], par, &sm.abort_flag)) {
          opd_abort(sm);
          return false;
        }
      }
      // Lane r holds rank r's part; every CTA combines them in rank order.
      opd_p1_unpack(other_rank ? sm.p1_peer[slot][lane] : mine, lane < (int)CS, t, d, g);
      arg_warp_reduce(g);
      FF l2t, l2d;
      const bool valid = opd_pair_norms(t, d, lane < (int)CS, &l2t, &l2d);
      if (lane == 0) {
        // c = (L2_d - L2_t) ln 2, -L2_d and lse_d = L2_d ln 2.
        sm.norms[slot] = make_float4(ff_to_float(ff_mul_f(ff_sub(l2d, l2t), kLn2f)),
                                     -ff_to_float(l2d), ff_to_float(ff_mul_f(l2d, kLn2f)),
                                     valid ? 1.0f : 0.0f);
        sm.nx[slot] = g.i;
        // Rank 0 will need z_d[x*] for the hard-label term: load it now.
        if (rank == 0 && valid) {
          const TIn* drow = static_cast<const TIn*>(p.draft) + ((size_t)b * p.k + i) * (size_t)p.V;
          zstar[slot] = ElemTraits<TIn>::load(drow, SPEC_CHECKED(g.i, p.V, kSiteOpdRow));
        }
        mbar_arrive(&sm.norm_ready[slot]);
        if (kVerify && rank == 0 && (vflags & kReqValid) && i < __ldg(&p.lengths[b]))
          opd_decide<TIn>(p, b, i, x, T, u, zt_x, zd_x, g, l2t, l2d, valid);
      }
      __syncwarp();
      return true;
    }
    // pass 2
    if (!mbar_wait_bounded(&sm.p2_done[slot], par, &sm.abort_flag)) {
      opd_abort(sm);
      return false;
    }
    const bool have = lane < kOpdConsumerWarps;
    const OpdP2 w = sm.p2w[slot][have ? lane : 0];
    FF kl = have ? FF{w.kl_hi, w.kl_lo} : FF{0.0f, 0.0f};
    FF kc = have ? FF{w.kc_hi, w.kc_lo} : FF{0.0f, 0.0f};
    kl = warp_sum_ff(kl);
    kc = warp_sum_ff(kc);
    int inf = __any_sync(0xffffffffu, have && w.inf) ? 1 : 0;
    if (CS > 1) {
      // Every CTA sends its sums to every other one, so that no CTA leaves
      // while a message to it is still on its way.
      if (lane < (int)CS && lane != (int)rank) {
        const uint32_t dst = dsmem_map(&sm.p2_peer[slot][rank], (uint32_t)lane);
        dsmem_st4(dst, make_float4(kl.hi, kl.lo, kc.hi, kc.lo));
        dsmem_st4(dst + 16, make_float4(__int_as_float(inf), 0.0f, 0.0f, 0.0f));
        mbar_arrive_remote(dsmem_map(&sm.peer2[slot], (uint32_t)lane));
      }
      if (!mbar_wait_cluster_bounded(&sm.peer2[slot], par, &sm.abort_flag)) {
        opd_abort(sm);
        return false;
      }
      if (rank == 0) {
        // Rank order: this CTA's part first, then ranks 1, 2, ...
        for (uint32_t r = 1; r < CS; ++r) {
          const OpdP2 o = sm.p2_peer[slot][r];
          kl = ff_add(kl, FF{o.kl_hi, o.kl_lo});
          kc = ff_add(kc, FF{o.kc_hi, o.kc_lo});
          inf |= o.inf;
        }
      }
    }
    if (rank == 0 && lane == 0) {
      const float4 nr = sm.norms[slot];
      if (nr.w != 0.0f) {
        const long long qo = SPEC_CHECKED(q, (long long)p.B * p.k, kSiteOpdOut);
        p.x_star[qo] = sm.nx[slot];
        p.hard[qo] = __fsub_rn(nr.z, zstar[slot]);
        p.rkl[qo] = inf ? INFINITY : ff_to_float(kl);
        p.rkl_clip[qo] = ff_to_float(kc);
      } else {
        p.x_star[q] = -1;
        p.hard[q] = p.rkl[q] = p.rkl_clip[q] = __int_as_float(0x7fc00000);
      }
    }
    __syncwarp();
    return true;
  });
}

// kVerify: also decide the verified positions (spec_verify_opd); the
// statistics-only instance compiles without any of that code.
template <typename TIn, bool kVerify>
__global__ void __launch_bounds__(kOpdThreads, kOpdMinBlocks) opd_kernel(OpdParams p) {
  extern __shared__ __align__(128) unsigned char opd_dyn[];
  OpdSmem& sm = *reinterpret_cast<OpdSmem*>(opd_dyn);
  const uint32_t CS = cluster_size(), rank = cluster_rank();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kOpdStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kOpdConsumerWarps);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.p1_done[s], kOpdConsumerWarps);
      mbar_init(&sm.p2_done[s], kOpdConsumerWarps);
      mbar_init(&sm.norm_ready[s], 1);
      mbar_init(&sm.peer1[s], CS > 1 ? CS - 1 : 1);
      mbar_init(&sm.peer2[s], CS > 1 ? CS - 1 : 1);
    }
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  // Both CTAs' barriers exist before either arrives on the other's.
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
  // Verification mode reads what the plan kernel wrote.
  if (kVerify) pdl_wait();
  const int cid = blockIdx.x / CS, ncl = gridDim.x / CS;
  const int s0 = (int)rank * p.slice;
  const int warp = threadIdx.x >> 5;
  if (warp >= kOpdFirstConsumerWarp) opd_consumers<TIn>(p, sm, cid, ncl, s0);
  else if (warp == kOpdProducerWarp) opd_producer<TIn>(p, sm, cid, ncl, s0);
  else opd_bookkeeper<TIn, kVerify>(p, sm, cid, ncl, CS, rank);
  // Verification mode: count the CTA out, as the row sweep does, so that the
  // final pass can hold its completion until every CTA of this grid is done.
  if constexpr (kVerify) {
    __syncthreads();
    if (threadIdx.x == 0) {
      WsHeader* h = reinterpret_cast<WsHeader*>(p.ws + p.lay.header);
      if (*(volatile int*)&sm.abort_flag) record_status(h, SPEC_ERR_TIMEOUT);
      __threadfence();
      atomicAdd(&h->sweep_exited, 1);
    }
  }
}
// Per-request mixture loss, one warp per request, after the statistics.
__global__ void opd_loss_kernel(const int32_t* lengths, const float* hard, const float* rkl_clip,
                                int B, int k, float alpha, float* loss) {
  pdl_wait();
  const int b = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= B) return;
  const int L = __ldg(&lengths[b]);
  const bool ok = L >= 1 && L <= k;
  FF h = {0.0f, 0.0f}, c = {0.0f, 0.0f};
  if (ok && lane < L) {
    h.hi = hard[(size_t)b * k + lane];
    c.hi = rkl_clip[(size_t)b * k + lane];
  }
  h = warp_sum_ff(h);
  c = warp_sum_ff(c);
  if (lane == 0) {
    if (!ok) {
      loss[b] = __int_as_float(0x7fc00000);
    } else {
      const float mh = __fdiv_rn(ff_to_float(h), (float)L);
      const float mc = __fdiv_rn(ff_to_float(c), (float)L);
      loss[b] = __fadd_rn(__fmul_rn(alpha, mh), __fmul_rn(__fsub_rn(1.0f, alpha), mc));
    }
  }
}

}  // namespace specv
