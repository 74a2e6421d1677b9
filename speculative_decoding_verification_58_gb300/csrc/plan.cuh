// Plan kernel: validates the per-request device inputs, resets the per-call
// workspace state and lays out the work list of logit rows the sweep reads,
// position-major (all requests' position 0, then position 1, ...), so that a
// rejection found at an early position can spare the rows behind it.
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
  __shared__ int warp_tot[33];
  WsHeader* h = reinterpret_cast<WsHeader*>(p.ws + p.lay.header);
  int32_t* rowlist = reinterpret_cast<int32_t*>(p.ws + p.lay.rowlist);
  int32_t* flags = reinterpret_cast<int32_t*>(p.ws + p.lay.flags);
  int32_t* first_reject = reinterpret_cast<int32_t*>(p.ws + p.lay.first_reject);
  uint32_t* acc_bits = reinterpret_cast<uint32_t*>(p.ws + p.lay.acc_bits);
  uint32_t* dec_bits = reinterpret_cast<uint32_t*>(p.ws + p.lay.dec_bits);
  uint32_t* bad_bits = reinterpret_cast<uint32_t*>(p.ws + p.lay.bad_bits);
  int32_t* done = reinterpret_cast<int32_t*>(p.ws + p.lay.done);

  if (threadIdx.x == 0) {
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
  __syncthreads();

  // Validate every request and reset its decision state.
  for (int b = threadIdx.x; b < p.B; b += kPlanThreads) {
    const int L = p.lengths[b];
    const float T = p.temperature[b];
    bool ok = L >= 1 && L <= p.k && temperature_ok(T);
    if (ok) {
      for (int i = 0; i < L; ++i) {
        int x = p.tokens[(size_t)b * p.k + i];
        ok = ok && x >= 0 && x < p.V;
      }
      if (T > 0.0f) {
        for (int i = 0; i <= L; ++i) {
          float u = p.uniforms[(size_t)b * (p.k + 1) + i];
          ok = ok && u >= 0.0f && u < 1.0f;  // false for NaN
        }
      }
    }
    flags[b] = ok ? (kReqValid | (T == 0.0f ? kReqGreedy : 0)) : 0;
    first_reject[b] = p.k;
    acc_bits[b] = 0u;
    dec_bits[b] = 0u;
    bad_bits[b] = 0u;
    for (int i = 0; i < p.k; ++i) done[(size_t)b * p.k + i] = 0;
    if (!ok) {
      atomicAdd(&h->bad_requests, 1);
      atomicMin(&h->first_bad, b);
      atomicCAS(&h->status, SPEC_OK, SPEC_ERR_BAD_INPUT);
    }
  }
  __syncthreads();

  // Position-major work list.  Entry = slot of the row: ((b*k + i) << 1) | tensor,
  // tensor 0 = target row i, 1 = draft row i (sampling requests only).
  int base = 0;
  for (int i = 0; i < p.k; ++i) {
    for (int b0 = 0; b0 < p.B; b0 += kPlanThreads) {
      const int b = b0 + threadIdx.x;
      int n = 0;
      if (b < p.B) {
        const int f = flags[b];
        if ((f & kReqValid) && i < p.lengths[b]) n = (f & kReqGreedy) ? 1 : 2;
      }
      int off;
      const int tot = block_exclusive_scan(n, &off, warp_tot);
      if (n > 0) {
        const int slot = (b * p.k + i) << 1;
        rowlist[base + off] = slot;
        if (n == 2) rowlist[base + off + 1] = slot | 1;
      }
      base += tot;
    }
  }
  if (threadIdx.x == 0) {
    h->rows_planned = base;
    h->units_total = base * p.nch;
  }
}

}  // namespace specv
