// D3D branch selection ("D3D: Decoupled Diffusion Drafting for Asynchronous
// Speculative Decoding", Methodology, asynchronous inference).  While the
// target verifies a block, the drafter prepares successor blocks for selected
// rejection positions and for full acceptance; once the round's outcome is
// known, a branch whose assumed verified prefix matches is a cache hit and its
// block becomes the next draft, and a miss calls for a synchronous draft.
//
// Branch j of request b assumes that the round emits token branch_tok[b][j]
// at position branch_pos[b][j] (a rejection there, or the bonus token when the
// position is L_b); with n = num_accepted[b] it matches when branch_pos == n
// and branch_tok == out_tokens[b][n].  The lowest matching slot wins.
//
// One warp per request: the lanes compare 32 branches at a time and a ballot
// picks the first match; the warp then copies the branch's block.  The data
// per request is a few hundred bytes, so the kernel is latency-bound; it is
// launched behind the final pass with programmatic dependent launch.
#pragma once

#include "common.cuh"

namespace specv {

constexpr int kD3dWarps = 8;  // requests per CTA
constexpr int kD3dCountThreads = 1024;

__global__ void __launch_bounds__(kD3dWarps * 32) d3d_select_kernel(
    const int32_t* num_accepted, const int32_t* out_tokens, const int32_t* branch_pos,
    const int32_t* branch_tok, const int32_t* branch_block, int B, int k, int NB, int blk,
    int32_t* hit, int32_t* next_block) {
  // The outcome may come from the kernel just before this one on the stream.
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * kD3dWarps + (threadIdx.x >> 5);
  if (b >= B) return;
  const int n = __ldg(&num_accepted[b]);
  int found = -1;
  if (n >= 0 && n <= k) {
    const int token = __ldg(&out_tokens[(size_t)b * (k + 1) + n]);
    const int32_t* pos = branch_pos + (size_t)b * NB;
    const int32_t* tok = branch_tok + (size_t)b * NB;
    for (int j0 = 0; j0 < NB; j0 += 32) {
      const int j = j0 + lane;
      bool match = false;
      if (j < NB) {
        const int ps = __ldg(&pos[j]);
        match = ps >= 0 && ps == n && __ldg(&tok[j]) == token;
      }
      const unsigned m = __ballot_sync(0xffffffffu, match);
      if (m != 0u) {
        found = j0 + __ffs((int)m) - 1;
        break;
      }
    }
  }
  if (lane == 0) hit[b] = found;
  const int32_t* src =
      branch_block + ((size_t)b * NB + SPEC_CHECKED(found >= 0 ? found : 0, NB, kSiteD3d)) * blk;
  for (int t = lane; t < blk; t += 32)
    next_block[(size_t)b * blk + t] = found >= 0 ? __ldg(&src[t]) : -1;
}

// Number of requests that hit (one CTA; deterministic integer sum).
__global__ void __launch_bounds__(kD3dCountThreads) d3d_count_kernel(const int32_t* hit, int B,
                                                                     int32_t* hits) {
  pdl_wait();
  __shared__ int warp_sum[kD3dCountThreads / 32];
  int c = 0;
  for (int b = threadIdx.x; b < B; b += kD3dCountThreads) c += hit[b] >= 0 ? 1 : 0;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
  if ((threadIdx.x & 31) == 0) warp_sum[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x < 32) {
    c = warp_sum[threadIdx.x];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
    if (threadIdx.x == 0) *hits = c;
  }
}

}  // namespace specv
