// Row sweep: one streaming pass over every logit row verification needs.
//
// For a sampling row (T > 0) it computes the row's online max and sum of
// 2^((z - max) * log2(e) / T) (p and q must be normalised over the whole
// vocabulary: AdaFlash Section 2.1); for a greedy row (T == 0) the max and
// its lowest index (DFlash notes, section 5.2, worked example #4).
//
// Persistent, warp-specialised CTAs.  Lane 0 of the producer warp claims
// work units (one vocabulary chunk of one row) from a global counter and
// streams each chunk into a ring of shared-memory stages with 1-D bulk async
// copies (cp.async.bulk, completion on an mbarrier).  Eight consumer warps
// read the stages with 16-byte shared loads, fold them into per-thread
// accumulators, and at the end of a unit reduce them with warp shuffles and
// one mbarrier-guarded exchange; warp 0 writes the unit's partial.
//
// Verification mode also decides: the CTA that completes the last chunk of
// (request b, position i) combines the partials, gathers p(x_i) and q(x_i),
// and applies the accept test u_i < min(1, p(x_i)/q(x_i)) (or argmax == x_i at
// T == 0) in double precision.  A rejection is published in first_reject[b];
// the producer skips chunks of positions behind a known rejection, since
// only tokens before the first rejection are kept (AdaFlash Section 2.1).
#pragma once

#include "common.cuh"

namespace specv {

struct SweepParams {
  const void* target;        // verify: [B, k+1, V]; stats: [rows, V]
  const void* draft;         // verify: [B, k, V]
  const int32_t* tokens;     // [B, k]
  const float* uniforms;     // [B, k+1]
  const float* temperature;  // verify: [B]; stats: [rows]
  int B, k, V, nch, chunk_elems;
  int early_exit;
  unsigned char* ws;
  WsLayout lay;
};

constexpr int kFlagFirst = 1, kFlagLast = 2, kFlagGreedy = 4, kFlagEnd = 8;

struct StageInfo {
  const void* row;  // row base (element 0)
  int part;         // Partial index: slot * nch + chunk
  int flags;
  int elem0;        // element index of the stage buffer's first byte
  int nbytes;       // bulk bytes in the stage (multiple of 16, may be 0)
  int head0, headn; // elements before the 16-byte aligned range (first stage)
  int tail0, tailn; // elements after it (last stage)
  float sc;         // log2(e) / T
  int slot;         // row slot ((b*k+i)<<1 | tensor) or row index
};

constexpr int kNC = kSweepConsumerWarps;
constexpr int kNCT = kNC * 32;

struct SweepSmem {
  alignas(128) unsigned char stage[kStages][kStageBytes];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t red_bar[kRedDepth];
  StageInfo info[kStages];
  float4 red[kRedDepth][kNC];
  int abort_flag;
};

__device__ __forceinline__ void sweep_abort(WsHeader* h, SweepSmem& sm) {
  record_status(h, SPEC_ERR_TIMEOUT);
  *(volatile int*)&sm.abort_flag = 1;
}

// ---------------------------------------------------------------------------
// Producer: one thread.
// ---------------------------------------------------------------------------
template <typename TIn, bool kVerify>
__device__ void sweep_producer(const SweepParams& p, SweepSmem& sm, WsHeader* h) {
  using Tr = ElemTraits<TIn>;
  const int32_t* rowlist = reinterpret_cast<const int32_t*>(p.ws + p.lay.rowlist);
  const int32_t* first_reject = reinterpret_cast<const int32_t*>(p.ws + p.lay.first_reject);
  const int units_total = __ldcg(&h->units_total);
  volatile int* abort_flag = &sm.abort_flag;
  int it = 0;
  bool ok = true;

  auto acquire = [&](int& s) -> bool {
    s = it % kStages;
    const int round = it / kStages;
    if (round > 0 && !mbar_wait_bounded(&sm.empty[s], (round - 1) & 1, abort_flag)) {
      sweep_abort(h, sm);
      return false;
    }
    return true;
  };

  for (;;) {
    const int u = atomicAdd(&h->work_next, 1);
    if (u >= units_total) break;
    const int row = u / p.nch;
    const int chunk = u - row * p.nch;
    const int slot = kVerify ? __ldcg(&rowlist[row]) : row;
    const TIn* rowp;
    float T;
    if (kVerify) {
      const int bi = slot >> 1;
      const int b = bi / p.k;
      const int i = bi - b * p.k;
      if (p.early_exit && *(volatile const int32_t*)&first_reject[b] < i) continue;
      T = __ldg(&p.temperature[b]);
      rowp = (slot & 1)
                 ? static_cast<const TIn*>(p.draft) + ((size_t)b * p.k + i) * (size_t)p.V
                 : static_cast<const TIn*>(p.target) + ((size_t)b * (p.k + 1) + i) * (size_t)p.V;
    } else {
      T = __ldg(&p.temperature[slot]);
      rowp = static_cast<const TIn*>(p.target) + (size_t)slot * (size_t)p.V;
    }
    const bool greedy = (T == 0.0f);
    const float sc = greedy ? 0.0f : softmax_scale(T);

    // Element range of the chunk and its 16-byte aligned core.
    const int e0 = chunk * p.chunk_elems;
    const int e1 = min(p.V, e0 + p.chunk_elems);
    const uintptr_t addr0 = reinterpret_cast<uintptr_t>(rowp + e0);
    int a0 = e0 + (int)(((16u - (unsigned)(addr0 & 15u)) & 15u) / Tr::kSize);
    if (a0 > e1) a0 = e1;
    const int core_bytes = (((e1 - a0) * Tr::kSize) & ~15);
    const int a1 = a0 + core_bytes / Tr::kSize;
    const int nstage = core_bytes > 0 ? (core_bytes + kStageBytes - 1) / kStageBytes : 1;
    const char* src0 = reinterpret_cast<const char*>(rowp + a0);
    atomicAdd(&h->chunks_swept, 1ull);
    atomicAdd(&h->sweep_bytes, (unsigned long long)(e1 - e0) * Tr::kSize);

    for (int j = 0; j < nstage; ++j) {
      int s;
      if (!acquire(s)) {
        ok = false;
        break;
      }
      const int off = j * kStageBytes;
      const int nb = core_bytes > 0 ? min(kStageBytes, core_bytes - off) : 0;
      StageInfo& I = sm.info[s];
      I.row = rowp;
      I.part = slot * p.nch + chunk;
      I.flags = (j == 0 ? kFlagFirst : 0) | (j == nstage - 1 ? kFlagLast : 0) |
                (greedy ? kFlagGreedy : 0);
      I.elem0 = a0 + off / Tr::kSize;
      I.nbytes = nb;
      I.head0 = e0;
      I.headn = a0 - e0;
      I.tail0 = a1;
      I.tailn = e1 - a1;
      I.sc = sc;
      I.slot = slot;
      if (nb > 0) {
        mbar_arrive_expect_tx(&sm.full[s], (uint32_t)nb);
        bulk_g2s(sm.stage[s], src0 + off, (uint32_t)nb, &sm.full[s]);
      } else {
        mbar_arrive(&sm.full[s]);
      }
      ++it;
    }
    if (!ok) break;
  }

  if (ok) {
    int s;
    if (acquire(s)) {
      sm.info[s].flags = kFlagEnd;
      mbar_arrive(&sm.full[s]);
      ++it;
      return;
    }
  }
  // Aborted: wait (bounded) for the copies still in flight into this CTA's
  // shared memory before the CTA may exit.
  for (int back = 1; back <= kStages && back <= it; ++back) {
    const int jt = it - back;
    int dummy = 0;
    mbar_wait_bounded(&sm.full[jt % kStages], (jt / kStages) & 1, (volatile int*)&dummy);
  }
}

// ---------------------------------------------------------------------------
// Decision for (b, i) once all of its chunks are in (warp-cooperative).
// ---------------------------------------------------------------------------
template <typename TIn>
__device__ void decide_position(const SweepParams& p, WsHeader* h, int bi, bool greedy, float sc) {
  const int lane = threadIdx.x & 31;
  const int b = bi / p.k;
  const int i = bi - b * p.k;
  const Partial* parts = reinterpret_cast<const Partial*>(p.ws + p.lay.partials);
  const Partial* pt = parts + (size_t)(bi << 1) * p.nch;
  double* pos_c = reinterpret_cast<double*>(p.ws + p.lay.pos_c);
  int32_t* pos_arg = reinterpret_cast<int32_t*>(p.ws + p.lay.pos_arg);
  uint32_t* bad_bits = reinterpret_cast<uint32_t*>(p.ws + p.lay.bad_bits);
  uint32_t* acc_bits = reinterpret_cast<uint32_t*>(p.ws + p.lay.acc_bits);
  uint32_t* dec_bits = reinterpret_cast<uint32_t*>(p.ws + p.lay.dec_bits);
  int32_t* first_reject = reinterpret_cast<int32_t*>(p.ws + p.lay.first_reject);
  const int x = __ldg(&p.tokens[(size_t)b * p.k + i]);

  bool accept, row_ok;
  if (greedy) {
    float v;
    int g;
    row_argmax_from_parts(pt, p.nch, &v, &g);
    row_ok = (g != INT32_MAX);
    accept = (g == x);
    if (lane == 0) __stcg(&pos_arg[bi], g);
  } else {
    const Partial* pd = parts + (size_t)((bi << 1) | 1) * p.nch;
    double ct, cd;
    float mt, md;
    const bool okt = row_log2_normaliser(pt, p.nch, sc, &ct, &mt);
    const bool okd = row_log2_normaliser(pd, p.nch, sc, &cd, &md);
    row_ok = okt && okd;
    const float zt = ElemTraits<TIn>::load(
        static_cast<const TIn*>(p.target) + ((size_t)b * (p.k + 1) + i) * (size_t)p.V, x);
    const float zd = ElemTraits<TIn>::load(
        static_cast<const TIn*>(p.draft) + ((size_t)b * p.k + i) * (size_t)p.V, x);
    // log2 p(x) and log2 q(x) in double: z*sc is exact in double.
    const double lp = (double)zt * (double)sc - ct;
    const double lq = (double)zd * (double)sc - cd;
    const double u = (double)__ldg(&p.uniforms[(size_t)b * (p.k + 1) + i]);
    // A token the target gives probability zero is never accepted; a token
    // the drafter gives probability zero (and the target not) always is.
    const double ratio = (lp == -INFINITY) ? 0.0 : exp2(lp - lq);
    accept = u < fmin(1.0, ratio);
    if (lane == 0) {
      __stcg(&pos_c[(size_t)bi * 2], ct);
      __stcg(&pos_c[(size_t)bi * 2 + 1], cd);
    }
  }
  // A row without finite mass makes the request invalid if the round reaches
  // it; it also ends the round there so no later row is read for nothing.
  if (!row_ok) accept = false;
  if (lane == 0) {
    if (!row_ok) atomicOr(&bad_bits[b], 1u << i);
    if (accept) atomicOr(&acc_bits[b], 1u << i);
    atomicOr(&dec_bits[b], 1u << i);
    if (!accept) atomicMin(&first_reject[b], i);
  }
}

// ---------------------------------------------------------------------------
// Consumers: warps 0..kNC-1.
// ---------------------------------------------------------------------------
template <typename TIn, bool kVerify>
__device__ void sweep_consumers(const SweepParams& p, SweepSmem& sm, WsHeader* h) {
  using Tr = ElemTraits<TIn>;
  constexpr int EPV = Tr::kPerVec;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ctid = threadIdx.x;
  volatile int* abort_flag = &sm.abort_flag;
  Partial* parts = reinterpret_cast<Partial*>(p.ws + p.lay.partials);
  int32_t* done = reinterpret_cast<int32_t*>(p.ws + p.lay.done);

  SoftAcc sa;
  ArgAcc aa;
  soft_init(sa);
  arg_init(aa);
  int it = 0, units = 0;
  for (;;) {
    const int s = it % kStages;
    if (!mbar_wait_bounded(&sm.full[s], (it / kStages) & 1, abort_flag)) {
      sweep_abort(h, sm);
      return;
    }
    const StageInfo I = sm.info[s];
    if (I.flags & kFlagEnd) return;
    const bool greedy = (I.flags & kFlagGreedy) != 0;
    const TIn* row = static_cast<const TIn*>(I.row);
    if (I.flags & kFlagFirst) {
      soft_init(sa);
      arg_init(aa);
      if (warp == 0 && lane < I.headn) {
        const float x = Tr::load(row, I.head0 + lane);
        if (greedy) arg_add(aa, x, I.head0 + lane);
        else soft_add1(sa, x, I.sc);
      }
    }
    const uint4* buf = reinterpret_cast<const uint4*>(sm.stage[s]);
    const int nvec = I.nbytes >> 4;
    if (greedy) {
#pragma unroll 4
      for (int j = ctid; j < nvec; j += kNCT) {
        float x[EPV];
        Tr::unpack(buf[j], x);
        const int base = I.elem0 + j * EPV;
#pragma unroll
        for (int e = 0; e < EPV; ++e) arg_add(aa, x[e], base + e);
      }
    } else {
#pragma unroll 4
      for (int j = ctid; j < nvec; j += kNCT) {
        float x[EPV];
        Tr::unpack(buf[j], x);
        soft_add<EPV>(sa, x, I.sc);
      }
    }
    if ((I.flags & kFlagLast) && warp == 0 && lane < I.tailn) {
      const float x = Tr::load(row, I.tail0 + lane);
      if (greedy) arg_add(aa, x, I.tail0 + lane);
      else soft_add1(sa, x, I.sc);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[s]);
    ++it;
    if (!(I.flags & kFlagLast)) continue;

    // ---- end of a unit: reduce the consumer warps' accumulators ----
    const int rs = units % kRedDepth;
    const uint32_t rpar = (uint32_t)(units / kRedDepth) & 1u;
    ++units;
    if (greedy) {
      arg_warp_reduce(aa);
      if (lane == 0) sm.red[rs][warp] = make_float4(aa.v, __int_as_float(aa.i), 0.f, 0.f);
    } else {
      soft_warp_reduce(sa);
      if (lane == 0) sm.red[rs][warp] = make_float4(sa.m, sa.ms, sa.s, 0.f);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.red_bar[rs]);
    if (warp != 0) continue;
    if (!mbar_wait_bounded(&sm.red_bar[rs], rpar, abort_flag)) {
      sweep_abort(h, sm);
      return;
    }
    Partial out;
    if (greedy) {
      ArgAcc a;
      arg_init(a);
      if (lane < kNC) {
        const float4 r = sm.red[rs][lane];
        a.v = r.x;
        a.i = __float_as_int(r.y);
      }
      arg_warp_reduce(a);
      out.m = a.v;
      out.s = 0.0f;
      out.arg = a.i;
    } else {
      SoftAcc a;
      soft_init(a);
      if (lane < kNC) {
        const float4 r = sm.red[rs][lane];
        a.m = r.x;
        a.ms = r.y;
        a.s = r.z;
      }
      soft_warp_reduce(a);
      out.m = a.m;
      out.s = a.s;
      out.arg = 0;
    }
    out.pad = 0;
    if (lane == 0) __stcg(reinterpret_cast<int4*>(&parts[I.part]), *reinterpret_cast<int4*>(&out));

    if (kVerify) {
      const int bi = I.slot >> 1;
      const int need = greedy ? p.nch : 2 * p.nch;
      int old = 0;
      if (lane == 0) {
        __threadfence();
        old = atomicAdd(&done[bi], 1);
      }
      old = __shfl_sync(0xffffffffu, old, 0);
      if (old == need - 1) {
        __threadfence();
        decide_position<TIn>(p, h, bi, greedy, I.sc);
      }
    }
  }
}

template <typename TIn, bool kVerify>
__global__ void __launch_bounds__(kSweepThreads, 2) sweep_kernel(SweepParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SweepSmem& sm = *reinterpret_cast<SweepSmem*>(smem_raw);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kNC);
    }
    for (int r = 0; r < kRedDepth; ++r) mbar_init(&sm.red_bar[r], kNC);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Everything below reads what the plan kernel wrote.
  pdl_wait();
  WsHeader* h = reinterpret_cast<WsHeader*>(p.ws + p.lay.header);
  if ((threadIdx.x >> 5) == kNC) {
    if ((threadIdx.x & 31) == 0) sweep_producer<TIn, kVerify>(p, sm, h);
    return;
  }
  sweep_consumers<TIn, kVerify>(p, sm, h);
}

}  // namespace specv
