// Plan kernel: validates the per-request device inputs, resets the per-call
// workspace state and lays out the descriptors of the logit rows the sweep
// reads, position-major (all requests' position 0, then position 1, ...), so
// that a rejection found at an early position can spare the rows behind it.
//
// One CTA, two flat-parallel passes: (1) every (request, position) item is
// checked with independent loads, invalid requests land in a shared bitmask;
// (2) every (position, request) item is counted, its request's state reset,
// and one block-wide scan places the row descriptors.
#pragma once

#include "common.cuh"

namespace specv {

struct PlanParams {
  const int32_t* tokens;      // [B, k]
  const int32_t* lengths;     // [B]
  const float* uniforms;      // [B, k+1]
  const float* temperature;   // [B]
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

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanParams p) {
  // Dependents may launch now; they wait for this grid's completion before
  // reading anything it writes.
  pdl_launch_dependents();
  __shared__ uint32_t bad_mask[SPEC_MAX_B / 32];
  __shared__ int warp_tot[33];
  const int tid = threadIdx.x;
  WsHeader* h = reinterpret_cast<WsHeader*>(p.ws + p.lay.header);
  int2* rowdesc = reinterpret_cast<int2*>(p.ws + p.lay.rowdesc);
  int32_t* flags = reinterpret_cast<int32_t*>(p.ws + p.lay.flags);
  int32_t* first_reject = reinterpret_cast<int32_t*>(p.ws + p.lay.first_reject);
  uint32_t* acc_bits = reinterpret_cast<uint32_t*>(p.ws + p.lay.acc_bits);
  uint32_t* dec_bits = reinterpret_cast<uint32_t*>(p.ws + p.lay.dec_bits);
  uint32_t* bad_bits = reinterpret_cast<uint32_t*>(p.ws + p.lay.bad_bits);
  int32_t* done = reinterpret_cast<int32_t*>(p.ws + p.lay.done);
  Partial* parts = reinterpret_cast<Partial*>(p.ws + p.lay.partials);
  int32_t* final_done = reinterpret_cast<int32_t*>(p.ws + p.lay.final_done);

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
  }
  const int words = (p.B + 31) >> 5;
  for (int w = tid; w < words; w += kPlanThreads) bad_mask[w] = 0u;
  __syncthreads();

  // Pass 1, item j = b*(k+1) + i: the request's scalars (at i = 0: 1 <= L <= k
  // from the length head's clamp, T is 0 or a finite normal float), token x_i
  // in [0, V) for i < L, uniform u_i in [0, 1) for i <= L when T > 0.
  const int k1 = p.k + 1;
  for (int j = tid; j < p.B * k1; j += kPlanThreads) {
    const int b = j / k1;
    const int i = j - b * k1;
    const int L = __ldg(&p.lengths[b]);
    const float T = __ldg(&p.temperature[b]);
    const int x = i < p.k ? __ldg(&p.tokens[(size_t)b * p.k + i]) : 0;
    const float u = __ldg(&p.uniforms[j]);
    bool bad = (i == 0) && !(L >= 1 && L <= p.k && temperature_ok(T));
    bad = bad || (i < L && i < p.k && (x < 0 || x >= p.V));
    bad = bad || (T > 0.0f && i <= L && !(u >= 0.0f && u < 1.0f));  // NaN fails
    if (bad) atomicOr(&bad_mask[b >> 5], 1u << (b & 31));
  }
  __syncthreads();

  // Pass 2, item it = i*B + b: rows of (b, i), state resets (one item per
  // request does the request-level ones), then the position-major layout.
  const int items = p.k * p.B;
  const int per = (items + kPlanThreads - 1) / kPlanThreads;
  const int lo = min(items, tid * per), hi = min(items, lo + per);
  int cnt = 0;
  for (int it = lo; it < hi; ++it) {
    const int i = it / p.B, b = it - i * p.B;
    const bool ok = !((bad_mask[b >> 5] >> (b & 31)) & 1u);
    const int L = __ldg(&p.lengths[b]);
    const bool greedy = __ldg(&p.temperature[b]) == 0.0f;
    done[(size_t)b * p.k + i] = 0;
    if (i == 0) {
      flags[b] = ok ? (kReqValid | (greedy ? kReqGreedy : 0)) : 0;
      first_reject[b] = p.k;
      acc_bits[b] = 0u;
      dec_bits[b] = 0u;
      bad_bits[b] = 0u;
      final_done[b] = 0;
      if (!ok) {
        atomicAdd(&h->bad_requests, 1);
        atomicMin(&h->first_bad, b);
        atomicCAS(&h->status, SPEC_OK, SPEC_ERR_BAD_INPUT);
      }
    }
    if (ok && i < L) cnt += greedy ? 1 : 2;
  }
  int pos;
  const int total = block_exclusive_scan(cnt, &pos, warp_tot);
  for (int it = lo; it < hi; ++it) {
    const int i = it / p.B, b = it - i * p.B;
    const bool ok = !((bad_mask[b >> 5] >> (b & 31)) & 1u);
    const int L = __ldg(&p.lengths[b]);
    if (!ok || i >= L) continue;
    const float T = __ldg(&p.temperature[b]);
    const float sc = T == 0.0f ? 0.0f : softmax_scale(T);
    const int slot = (b * p.k + i) << 1;
    rowdesc[pos++] = make_int2(slot, __float_as_int(sc));
    if (T != 0.0f) rowdesc[pos++] = make_int2(slot | 1, __float_as_int(sc));
    // The deciding CTA waits for these slots to leave the empty marker.
    const int ntensor = T != 0.0f ? 2 : 1;
    unsigned long long* slots = reinterpret_cast<unsigned long long*>(parts + (size_t)slot * p.nch);
    for (int c = 0; c < ntensor * p.nch; ++c) slots[c] = kPartialEmpty;
  }
  if (tid == 0) {
    h->rows_planned = total;
    h->units_total = total * p.nch;
  }
}

}  // namespace specv
