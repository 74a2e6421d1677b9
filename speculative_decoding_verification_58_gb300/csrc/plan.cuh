// Plan kernel: validates the per-request device inputs, resets the per-call
// workspace state and lays out the descriptors of the logit rows the sweep
// reads, position-major (all requests' position 0, then position 1, ...), so
// that a rejection found at an early position can spare the rows behind it.
//
// One CTA, two flat-parallel passes: (1) every request's scalars are
// checked and its state reset (invalid requests land in a shared bitmask, or,
// for a batch of at most one request per thread, every request's row facts
// in a shared table); (2) every (position, request) item is counted and one
// block-wide scan places the row descriptors.
//
// Row addressing: request b's target rows are rows t0_b + 0..L_b of the
// target buffer and its draft rows d0_b + 0..L_b-1 of the draft buffer.  The
// padded layout [B, k+1, V] / [B, k, V] has t0_b = b(k+1), d0_b = bk; the
// packed layout (AdaFlash Section 3.3, a verification batch of total length
// sum_b k_b) takes t0_b, d0_b from the caller and checks them against the
// buffers' row counts.  Each descriptor carries its absolute row.
#pragma once

#include "common.cuh"

namespace specv {

struct PlanParams {
  const int32_t* tokens;      // [B, k]
  const int32_t* lengths;     // [B]
  const float* uniforms;      // [B, k+1]
  const float* temperature;   // [B]
  const int32_t* t_start;     // [B] packed layout: first target row of b (null: padded)
  const int32_t* d_start;     // [B] packed layout: first draft row of b
  long long rows_t, rows_d;   // packed layout: rows in the target / draft buffers
  int skip_t01;               // leave requests at T = 0 or 1 out of the row list
                              // (another kernel decides them: spec_verify_opd)
  int B, k, V, C, chunk_elems, nch;
  unsigned char* ws;
  WsLayout lay;
};

constexpr int kPlanThreads = 1024;

// Block-wide exclusive scan of one int per thread; returns the block total.
__device__ __forceinline__ int block_exclusive_scan(int x, int* excl, int* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (kPlanThreads / 32) ? warp_tot[lane] : 0;
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += y;
    }
    warp_tot[lane] = wi - w;  // exclusive prefix of warp totals
    if (lane == 31) warp_tot[32] = wi;
  }
  __syncthreads();
  *excl = incl - x + warp_tot[warp];
  int total = warp_tot[32];
  __syncthreads();
  return total;
}

// Fill n 8-byte words at dst with v (dst 16-byte aligned): 16-byte stores,
// consecutive threads on consecutive addresses.
__device__ __forceinline__ void fill_u64(unsigned long long* dst, size_t n, unsigned long long v) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  const uint4 v4 = make_uint4((uint32_t)v, (uint32_t)(v >> 32), (uint32_t)v, (uint32_t)(v >> 32));
  for (size_t j = threadIdx.x; j < n / 2; j += kPlanThreads) d4[j] = v4;
  if ((n & 1) && threadIdx.x == 0) dst[n - 1] = v;
}

__device__ __forceinline__ void fill_u32(uint32_t* dst, size_t n, uint32_t v) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  for (size_t j = threadIdx.x; j < n / 4; j += kPlanThreads) d4[j] = make_uint4(v, v, v, v);
  for (size_t j = (n & ~size_t(3)) + threadIdx.x; j < n; j += kPlanThreads) dst[j] = v;
}

// One request's row facts, kept in shared memory for the row pass when the
// batch has at most one request per thread.
struct PlanReq {
  int L;       // positions to verify
  int rows;    // rows per position in the row list: 0 (none), 1 (greedy) or 2
  float sc;    // log2(e) / T, 0 at T = 0
  int t0, d0;  // first target and draft rows
};
static_assert(kPlanThreads * sizeof(PlanReq) <= (SPEC_MAX_B / 32) * sizeof(uint32_t),
              "the request table fits in the bad-mask words it shares");

__global__ void __launch_bounds__(kPlanThreads, 1) plan_kernel(PlanParams p) {
  // This kernel may itself be launched early, behind the previous kernel on
  // the stream: nothing is read or written before that kernel has finished.
  pdl_wait();
  // Dependents may launch now; they wait for this grid's completion before
  // reading anything it writes.
  pdl_launch_dependents();
  // Either the bad-request bitmask (large batches) or the request table
  // (at most one request per thread).
  __shared__ __align__(16) uint32_t words[SPEC_MAX_B / 32];
  __shared__ int warp_tot[33];
  __shared__ int row_kinds;
  const int tid = threadIdx.x;
  const bool small = p.B <= kPlanThreads;
  uint32_t* bad_mask = words;
  PlanReq* req = reinterpret_cast<PlanReq*>(words);
  WsHeader* h = reinterpret_cast<WsHeader*>(p.ws + p.lay.header);
  int4* rowdesc = reinterpret_cast<int4*>(p.ws + p.lay.rowdesc);
  int2* rowbase = reinterpret_cast<int2*>(p.ws + p.lay.rowbase);
  int32_t* flags = reinterpret_cast<int32_t*>(p.ws + p.lay.flags);
  int32_t* first_reject = reinterpret_cast<int32_t*>(p.ws + p.lay.first_reject);

  // A small batch's request scalars are loaded first, so that their round
  // trip overlaps the workspace fills below.
  auto load_req = [&](int b, int& L, float& T, int2& rb) {
    L = __ldg(&p.lengths[b]);
    T = __ldg(&p.temperature[b]);
    rb = p.t_start != nullptr ? make_int2(__ldg(&p.t_start[b]), __ldg(&p.d_start[b]))
                              : make_int2(b * (p.k + 1), b * p.k);
  };
  int L0 = 0;
  float T0 = 0.0f;
  int2 rb0 = make_int2(0, 0);
  if (small && tid < p.B) load_req(tid, L0, T0, rb0);

  if (tid == 0) {
    h->status = SPEC_OK;
    h->bad_requests = 0;
    h->first_bad = INT32_MAX;
    h->work_next = 0;
    h->chunks_per_row = p.nch;
    h->chunk_elems = p.chunk_elems;
    h->chunks_swept = 0;
    h->final_rows = 0;
    h->residual_zero = 0;
    h->sweep_bytes = 0;
    h->final_bytes = 0;
    h->sweep_exited = 0;
    h->final_ctas_done = 0;
  }
  if (!small)
    for (int w = tid; w < ((p.B + 31) >> 5); w += kPlanThreads) bad_mask[w] = 0u;
  if (tid == 0) row_kinds = 0;

  // Per-call state that does not depend on the inputs, with coalesced
  // stores: decision masks, chunk and final-pass counters to zero, every
  // partial slot to the empty marker (the deciding CTA waits for its slots
  // to leave it).
  fill_u64(reinterpret_cast<unsigned long long*>(p.ws + p.lay.state), p.B, 0ull);
  fill_u32(reinterpret_cast<uint32_t*>(p.ws + p.lay.bad_bits), p.B, 0u);
  fill_u32(reinterpret_cast<uint32_t*>(p.ws + p.lay.final_done), p.B, 0u);
  fill_u32(reinterpret_cast<uint32_t*>(p.ws + p.lay.done), (size_t)p.B * p.k, 0u);
  fill_u64(reinterpret_cast<unsigned long long*>(p.ws + p.lay.partials),
           (size_t)p.B * p.k * 2 * p.C, kPartialEmpty);
  // Partials of a made-up position that the sweep's bookkeeping warps decide
  // once, without effect, to bring the decision code into their instruction
  // caches: m = 0, s = 1 (or index 0).
  fill_u64(reinterpret_cast<unsigned long long*>(p.ws + p.lay.warm), 2 * (size_t)p.C,
           ((unsigned long long)__float_as_uint(1.0f) << 32) | __float_as_uint(0.0f));
  __syncthreads();

  // Requests: the scalars the row list depends on (1 <= L <= k from the
  // length head's clamp, T is 0 or a finite normal float, packed rows inside
  // their buffers), request state, first rows.  The per-position inputs
  // (tokens in [0, V), uniforms in [0, 1)) are checked by the final pass,
  // which loads them anyway; until then every use guards its index.
  for (int b = tid; b < p.B; b += kPlanThreads) {
    int L = L0;
    float T = T0;
    int2 rb = rb0;
    if (!small) load_req(b, L, T, rb);
    bool bad = !(L >= 1 && L <= p.k && temperature_ok(T));
    // Packed rows: target rows t0 .. t0+L exist, and draft rows d0 .. d0+L-1
    // unless the request is greedy (its draft rows are never read).
    bad = bad || (p.t_start != nullptr &&
                  !(rb.x >= 0 && (long long)rb.x + L + 1 <= p.rows_t &&
                    (T == 0.0f || (rb.y >= 0 && (long long)rb.y + L <= p.rows_d))));
    flags[b] = bad ? 0 : (kReqValid | (T == 0.0f ? kReqGreedy : 0));
    first_reject[b] = p.k;
    rowbase[b] = rb;
    if (bad) {
      atomicAdd(&h->bad_requests, 1);
      atomicMin(&h->first_bad, b);
      atomicCAS(&h->status, SPEC_OK, SPEC_ERR_BAD_INPUT);
    }
    const bool listed = !bad && !(p.skip_t01 && (T == 0.0f || T == 1.0f));
    if (listed) atomicOr(&row_kinds, T == 0.0f ? 1 : 2);
    if (small) {
      req[b] = PlanReq{L, listed ? (T == 0.0f ? 1 : 2) : 0, T == 0.0f ? 0.0f : softmax_scale(T),
                       rb.x, rb.y};
    } else if (bad) {
      atomicOr(&bad_mask[b >> 5], 1u << (b & 31));
    }
  }
  __syncthreads();

  // Row pass, item it = i*B + b: the rows of (b, i) in position-major order;
  // one block-wide scan places their descriptors.
  auto item = [&](int b, int i, int& rows, float& sc, int& trow, int& drow) {
    if (small) {
      const PlanReq r = req[b];
      rows = i < r.L ? r.rows : 0;
      sc = r.sc;
      trow = r.t0 + i;
      drow = r.d0 + i;
      return;
    }
    const bool ok = !((bad_mask[b >> 5] >> (b & 31)) & 1u);
    const float T = __ldg(&p.temperature[b]);
    rows = (ok && i < __ldg(&p.lengths[b]) && !(p.skip_t01 && (T == 0.0f || T == 1.0f)))
               ? (T == 0.0f ? 1 : 2)
               : 0;
    sc = T == 0.0f ? 0.0f : softmax_scale(T);
    trow = (p.t_start != nullptr ? __ldg(&p.t_start[b]) : b * (p.k + 1)) + i;
    drow = (p.t_start != nullptr ? __ldg(&p.d_start[b]) : b * p.k) + i;
  };
  const int items = p.k * p.B;
  const int per = (items + kPlanThreads - 1) / kPlanThreads;
  const int lo = min(items, tid * per), hi = min(items, lo + per);
  int cnt = 0;
  for (int it = lo; it < hi; ++it) {
    const int i = it / p.B, b = it - i * p.B;
    int rows, trow, drow;
    float sc;
    item(b, i, rows, sc, trow, drow);
    cnt += rows;
  }
  int pos;
  const int total = block_exclusive_scan(cnt, &pos, warp_tot);
  for (int it = lo; it < hi; ++it) {
    const int i = it / p.B, b = it - i * p.B;
    int rows, trow, drow;
    float sc;
    item(b, i, rows, sc, trow, drow);
    if (rows == 0) continue;
    const int slot = (b * p.k + i) << 1;
    const long long slots = 2LL * p.B * p.k;
    rowdesc[SPEC_CHECKED(pos, slots, kSitePlanRowdesc)] = make_int4(slot, __float_as_int(sc), trow, 0);
    ++pos;
    if (rows == 2) {
      rowdesc[SPEC_CHECKED(pos, slots, kSitePlanRowdesc)] =
          make_int4(slot | 1, __float_as_int(sc), drow, 0);
      ++pos;
    }
  }
  if (tid == 0) {
    h->row_kinds = row_kinds;
    h->rows_planned = total;
    h->units_total = total * p.nch;
  }
}

}  // namespace specv
