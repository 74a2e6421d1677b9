/*
 * spec_verify.h - C ABI of the GB300 (sm_103a) batched speculative-decoding
 * verification library (libspecverify.so).
 *
 * The operation follows AdaFlash: Adaptive Speculative Decoding via
 * On-Policy Distilled Diffusion Drafters (arXiv 2607.19223), Section 2.1
 * "Speculative Decoding": for each request b and draft position i < L_b, the
 * draft token x_i is accepted with probability min{1, p_i(x_i) / q_i(x_i)},
 * where p_i = softmax(target_logits[b,i,:] / T_b) and
 * q_i = softmax(draft_logits[b,i,:] / T_b); every token before the first
 * rejected one is kept and a corrected token is drawn at the rejection point
 * from normalize(max(0, p_i - q_i)) (the residual distribution; restated in
 * the AdaFlash reading notes, "Speculative decoding: the basic idea", step 4,
 * and in the DFlash notes, section 5.2).  When all L_b drafts are accepted,
 * one more token is drawn from p_{L_b} (DFlash notes, section 3.1, steps 6-7:
 * m accepted + 1 emitted).  At T_b == 0 the rule is greedy matching: accept
 * while x_i equals the target argmax, emit the target argmax at the first
 * mismatch (DFlash notes, section 5.2, worked example #4; AdaFlash Appendix
 * B.1).  L_b is the per-request verification length chosen by an adaptive
 * length head, 1 <= L_b <= k (AdaFlash Section 3.2, the clamp of k-hat).
 *
 * Readings where the pages are silent:
 *   - the accept test for position i uses uniforms[b][i] and is the strict
 *     comparison u < min(1, ratio);
 *   - the final (residual or bonus) token uses uniforms[b][L_b];
 *   - sampling is by inverse CDF in ascending vocabulary index: the first
 *     index whose cumulative mass exceeds u * total mass, so a token of zero
 *     probability is never emitted;
 *   - argmax ties go to the lowest index;
 *   - if the residual mass is zero, the token is drawn from p instead.
 *
 * Conventions for every entry point:
 *   - Device pointers are CUDA device (or managed) memory owned by the caller;
 *     the library allocates nothing, keeps no state between calls and never
 *     synchronises the stream except where stated.
 *   - The two logits buffers of the verification entry points (spec_verify,
 *     spec_verify_ex, spec_verify_timed, spec_verify_packed,
 *     spec_verify_static), and the logits of spec_row_stats, may instead be
 *     pinned host memory that the GPU maps (cudaHostAlloc,
 *     cudaHostRegister): the kernels then read the rows they need over the
 *     CPU-GPU link with plain loads, without a copy (early exit also spares
 *     the link the rows it skips); results are those of the same call on
 *     device-resident logits.  One buffer in host memory and the other not,
 *     or host memory the GPU does not map, is SPEC_ERR_INVALID_ARG.  The OPD
 *     entry points (spec_opd_stats, spec_verify_opd) stream every row twice
 *     and take device-resident logits only (host memory:
 *     SPEC_ERR_INVALID_ARG).  Every other buffer is device memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously on it.
 *   - Host-detectable argument errors return immediately and launch nothing.
 *   - Errors in values that live on the device (tokens, lengths, temperature,
 *     uniforms, non-finite logits) cannot be seen by the host call: the
 *     affected request gets num_accepted = -1 and out_tokens all -1, and the
 *     workspace records SPEC_ERR_BAD_INPUT, readable with
 *     spec_verify_device_status() or spec_verify_report().  No kernel traps.
 *   - Every device-side wait is bounded; a wait that runs out records
 *     SPEC_ERR_TIMEOUT in the workspace and the kernel returns.  A request
 *     whose outcome or final token a timed-out wait left unknown reports
 *     num_accepted = -1 and out_tokens all -1, like an invalid request.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPEC_VERIFY_ABI_VERSION 1

/* Largest supported sizes. */
#define SPEC_MAX_B (1 << 18)   /* requests per call */
#define SPEC_MAX_K 31          /* draft positions per request (decisions are 32-bit masks) */
#define SPEC_MAX_V (1 << 21)   /* vocabulary size */

typedef enum {
  SPEC_OK = 0,
  SPEC_ERR_INVALID_ARG = 1,  /* bad size, null pointer or misaligned pointer */
  SPEC_ERR_UNSUPPORTED = 2,  /* valid request the library does not support (e.g. k > SPEC_MAX_K) */
  SPEC_ERR_WORKSPACE = 3,    /* workspace too small or not 256-byte aligned */
  SPEC_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  SPEC_ERR_BAD_INPUT = 5,    /* device-detected invalid value in some request */
  SPEC_ERR_TIMEOUT = 6,      /* a bounded device-side wait ran out */
  SPEC_ERR_INTERNAL = 7      /* internal consistency check failed */
} spec_status_t;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype_t;

/* Flags for spec_verify_ex. */
#define SPEC_FLAG_FULL_SWEEP 1u  /* sweep every row i < L_b even past a known rejection */
/*
 * Testing aid, never for production: in the final pass, every slice CTA of a
 * request except the first waits (bounded, 1 ms) for an event that never
 * happens, as if the request's outcome never arrived.  It exercises the path
 * a real device-side timeout takes: every request with more than one slice
 * then reports num_accepted = -1 and out_tokens all -1, and the workspace
 * records SPEC_ERR_TIMEOUT; nothing faults and the stream stays usable.
 */
#define SPEC_FLAG_TEST_LATE_SLICES 2u

/*
 * Bytes of device workspace spec_verify needs for a batch of B requests with
 * k draft positions over a vocabulary of V.  Depends only on (B, k, V).
 * Returns 0 for sizes outside the supported range.
 */
size_t spec_verify_workspace_bytes(int B, int k, int V);

/*
 * Batched verification (asynchronous on `stream`).
 *
 *   target_logits [B, k+1, V]  dtype, row-major contiguous; row i (i <= k) is
 *                              the target's next-token logits after x_0..x_{i-1}
 *   draft_logits  [B, k, V]    dtype, row-major contiguous; row i is the
 *                              drafter's distribution for position i (it may be a
 *                              marginal, as for one-pass diffusion drafters)
 *   dtype                      SPEC_F32 (float) or SPEC_BF16 (bfloat16 bits)
 *   draft_tokens  [B, k]       int32 in [0, V) for i < L_b
 *   lengths       [B]          int32 in [1, k]
 *   uniforms      [B, k+1]     float in [0, 1): u_i for the test at position i,
 *                              u_{L_b} for the final sample (unused at T = 0)
 *   temperature   [B]          float: 0 = greedy; otherwise a normal float
 *                              (>= 2^-126) and finite
 *   B, k, V                    B, k or V below 1 (an empty batch) is
 *                              SPEC_ERR_INVALID_ARG; B > SPEC_MAX_B,
 *                              k > SPEC_MAX_K or V > SPEC_MAX_V is
 *                              SPEC_ERR_UNSUPPORTED
 *   out_tokens    [B, k+1]     int32 out: x_0..x_{n-1}, the final token, then -1
 *   num_accepted  [B]          int32 out: n in [0, L_b], or -1 for a request
 *                              whose inputs were invalid
 *   workspace                  device scratch of >= spec_verify_workspace_bytes
 *                              bytes, 256-byte aligned; holds the status until the
 *                              next call on it.  Concurrent calls need separate
 *                              workspaces.
 *
 * Logit pointers must be aligned to their element size; 16-byte aligned rows
 * (V * element size a multiple of 16 and 16-byte aligned bases) take the fast
 * path.  Logits may contain -inf.  A sampling request (T > 0) needs finite,
 * positive mass in every row it reads: a NaN or +inf logit in such a row, or
 * a row of only -inf, makes the request invalid.  A greedy request (T = 0)
 * only takes argmaxes: a NaN entry is never the maximum, +inf is a maximum
 * like any other value (the lowest index among equal maxima wins), and a row
 * with no entry above -inf makes the request invalid.
 *
 * Returns SPEC_OK once the work is enqueued, or an error code (nothing
 * enqueued).
 */
spec_status_t spec_verify(const void* target_logits, const void* draft_logits,
                          spec_dtype_t dtype, const int32_t* draft_tokens,
                          const int32_t* lengths, const float* uniforms,
                          const float* temperature, int B, int k, int V,
                          int32_t* out_tokens, int32_t* num_accepted, void* workspace,
                          size_t workspace_bytes, void* stream);

/* spec_verify with flags (SPEC_FLAG_*).  flags = 0 is spec_verify. */
spec_status_t spec_verify_ex(const void* target_logits, const void* draft_logits,
                             spec_dtype_t dtype, const int32_t* draft_tokens,
                             const int32_t* lengths, const float* uniforms,
                             const float* temperature, int B, int k, int V,
                             int32_t* out_tokens, int32_t* num_accepted, void* workspace,
                             size_t workspace_bytes, void* stream, unsigned flags);

/*
 * Measurement only: spec_verify_ex that also records up to four caller-owned
 * CUDA events (cudaEvent_t as void*, any may be NULL) on `stream`: before the
 * plan kernel, before the row sweep, before the final pass, and after it.
 * Recording events between the kernels removes the launch overlap they
 * otherwise get from programmatic dependent launch, so use this to time the
 * kernels one by one and spec_verify for end-to-end numbers.
 */
spec_status_t spec_verify_timed(const void* target_logits, const void* draft_logits,
                                spec_dtype_t dtype, const int32_t* draft_tokens,
                                const int32_t* lengths, const float* uniforms,
                                const float* temperature, int B, int k, int V,
                                int32_t* out_tokens, int32_t* num_accepted, void* workspace,
                                size_t workspace_bytes, void* stream, unsigned flags,
                                void* ev_plan, void* ev_sweep, void* ev_final, void* ev_end);

/*
 * Verification over a packed (ragged) batch.  AdaFlash Section 3.3,
 * "Adaptive Request Scheduling": with per-request verification lengths
 * k_b, the serving engine packs the candidates into one verification batch
 * of total length sum_b k_b rather than padding every request to k.  The
 * logits then come as flat row buffers:
 *
 *   target_rows   [rows_t, V]  dtype; request b's target rows are
 *                              target_row_start[b] + 0 .. L_b (L_b + 1 rows:
 *                              one per draft position and one for the bonus)
 *   draft_rows    [rows_d, V]  dtype; request b's draft rows are
 *                              draft_row_start[b] + 0 .. L_b - 1.  May be NULL
 *                              when rows_d == 0 (all requests greedy).
 *   target_row_start, draft_row_start
 *                 [B]          int32 (device).  Any placement is allowed
 *                              (order, gaps, shared rows); the rows named must lie
 *                              inside their buffer.  A greedy request's draft
 *                              rows are never read and its draft_row_start is
 *                              not checked.
 *   rows_t, rows_d             row counts of the two buffers: 1 <= rows_t and
 *                              0 <= rows_d, both <= INT32_MAX.
 *
 * Everything else (tokens [B, k], uniforms [B, k+1], outputs, workspace,
 * flags) is as for spec_verify_ex; the results are identical to spec_verify
 * on the same rows laid out padded.  A request whose rows fall outside a
 * buffer is invalid (num_accepted = -1, SPEC_ERR_BAD_INPUT recorded).
 */
spec_status_t spec_verify_packed(const void* target_rows, long long rows_t,
                                 const void* draft_rows, long long rows_d, spec_dtype_t dtype,
                                 const int32_t* target_row_start,
                                 const int32_t* draft_row_start, const int32_t* draft_tokens,
                                 const int32_t* lengths, const float* uniforms,
                                 const float* temperature, int B, int k, int V,
                                 int32_t* out_tokens, int32_t* num_accepted, void* workspace,
                                 size_t workspace_bytes, void* stream, unsigned flags);

/*
 * spec_verify for callers that cannot allocate device memory.  (The paper
 * has no counterpart: this is a deployment convenience.)  Some callers are
 * handed only their input and output buffers -- for example an operator
 * plugged into a runtime that owns all device memory and offers no scratch,
 * or code on a serving hot path where an allocation would stall or is
 * forbidden -- so they cannot supply spec_verify's workspace.
 *
 * Instead of a workspace, this entry uses a fixed scratch array of
 * SPEC_STATIC_SCRATCH_BYTES that lives inside the library: every GPU that
 * loads the library holds that memory until the process exits.  The call
 * itself allocates nothing (no cudaMalloc, no allocating library routine).
 *   - Batches whose spec_verify_workspace_bytes(B, k, V) exceeds
 *     SPEC_STATIC_SCRATCH_BYTES are rejected with SPEC_ERR_UNSUPPORTED and
 *     nothing is launched.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture.
 *   - All calls on a GPU share the one array, which keeps the last call's
 *     contents; each call resets what it needs.  Calls that overlap on the
 *     GPU (other streams, other host threads) race and must be serialised
 *     by the caller.
 *   - Invalid device-side inputs, and a request whose result a device-side
 *     wait that ran out (2 s) left unknown, show as num_accepted[b] == -1
 *     and out_tokens all -1; the status word stays in the library's scratch
 *     and is not reported separately.
 * Arguments are those of spec_verify without the workspace.
 */
#define SPEC_STATIC_SCRATCH_BYTES (8u << 20)
spec_status_t spec_verify_static(const void* target_logits, const void* draft_logits,
                                 spec_dtype_t dtype, const int32_t* draft_tokens,
                                 const int32_t* lengths, const float* uniforms,
                                 const float* temperature, int B, int k, int V,
                                 int32_t* out_tokens, int32_t* num_accepted, void* stream);

/* What the last call on a workspace recorded. */
typedef struct {
  int32_t status;             /* spec_status_t recorded on the device */
  int32_t bad_requests;       /* requests with invalid inputs */
  int32_t first_bad_request;  /* lowest such request index, or -1 */
  int32_t rows_planned;       /* logit rows the plan admitted (sum over valid b of L_b or 2 L_b) */
  int64_t chunks_swept;       /* row chunks the sweep actually read */
  int32_t chunks_per_row;     /* vocabulary chunks per row used by the sweep */
  int32_t chunk_elems;        /* elements per chunk (last chunk may be shorter) */
  int64_t final_rows;         /* logit rows the final pass read (residual 2, bonus 1) */
  int32_t residual_zero;      /* requests whose residual mass was zero (fell back to p) */
  int32_t reserved;
  int64_t sweep_bytes;        /* logit bytes the sweep streamed from memory */
  int64_t final_bytes;        /* logit bytes the final pass streamed (first pass over its rows) */
} spec_verify_report_t;

/*
 * Wait for `stream`, then copy the report of the last spec_verify call on
 * `workspace` into *report (host memory).  Returns SPEC_OK or SPEC_ERR_CUDA.
 */
spec_status_t spec_verify_report(const void* workspace, void* stream,
                                 spec_verify_report_t* report);

/*
 * Wait for `stream` and return the device-recorded status of the last
 * spec_verify call on `workspace` (SPEC_OK, SPEC_ERR_BAD_INPUT,
 * SPEC_ERR_TIMEOUT or SPEC_ERR_INTERNAL), or SPEC_ERR_CUDA if reading it failed.
 */
spec_status_t spec_verify_device_status(const void* workspace, void* stream);

/*
 * The row sweep on its own: per-row statistics of `rows` rows of V logits
 * (step 1 of verification; AdaFlash Section 2.1 needs p and q normalised
 * over the full vocabulary).
 *   logits       [rows, V] dtype, row-major contiguous (device)
 *   temperature  [rows] float (device): 0 = argmax only
 *   row_max      [rows] float out: max_v z
 *   row_lse      [rows] float out: log sum_v exp(z_v / T) (natural log; NaN when T = 0)
 *   row_arg      [rows] int32 out: lowest index attaining the max for T = 0
 *                rows; -1 for T > 0 rows (their sweep keeps no index)
 * Uses the same kernels and arithmetic as spec_verify.  Temperatures are
 * not validated here: pass 0 or a finite normal float.
 */
size_t spec_row_stats_workspace_bytes(int rows, int V);
spec_status_t spec_row_stats(const void* logits, spec_dtype_t dtype, int rows, int V,
                             const float* temperature, float* row_max, float* row_lse,
                             int32_t* row_arg, void* workspace, size_t workspace_bytes,
                             void* stream);

/*
 * On-policy distillation (OPD) supervision statistics over the same batch
 * buffers as spec_verify (AdaFlash Section 3.1, "Mixture OPD Loss with
 * Reverse-KL" and "Entry-wise Divergence Clipping"; the AdaFlash reading
 * notes work one toy position through).  For every request b and verified
 * position i < L_b, with p = softmax(target row i) and q = softmax(draft row
 * i) at temperature 1 (the models' own distributions):
 *
 *   x_star   [B, k] int32 out: argmax_y p(y), lowest index on ties
 *   hard     [B, k] float out: -log q(x_star)                (hard-label term)
 *   rkl      [B, k] float out: sum_y q(y) log(q(y)/p(y))     (reverse KL)
 *   rkl_clip [B, k] float out: sum_y min{q(y) log(q(y)/p(y)), delta}
 *   loss     [B]    float out: alpha * mean_{i<L_b} hard + (1 - alpha) * mean_{i<L_b} rkl_clip
 *
 * target_logits [B, k+1, V] and draft_logits [B, k, V] (dtype) and lengths
 * [B] (int32 in [1, k]) are device buffers as for spec_verify.  An entry
 * with q = 0 adds nothing (0 log 0 = 0); one with q > 0 where p = 0 adds
 * +inf to rkl and delta to rkl_clip.  Positions i >= L_b get x_star = -1 and
 * NaN; an invalid L_b makes the whole request -1 / NaN (loss NaN); a row
 * without finite mass (NaN, +inf, all -inf) makes its position NaN.
 * delta must be finite and > 0 (the paper uses 0.01), alpha in [0, 1] (0.8).
 * Needs no workspace and so records no device status: every position starts
 * as -1 / NaN and is overwritten when its results are known, so a
 * device-side wait that runs out (2 s) leaves NaN behind.  Every logit is
 * used twice (normalisers first, then the sums); the second read is arranged
 * to come from L2.  Asynchronous on `stream`; returns SPEC_OK once enqueued.
 */
spec_status_t spec_opd_stats(const void* target_logits, const void* draft_logits,
                             spec_dtype_t dtype, const int32_t* lengths, int B, int k, int V,
                             float delta, float alpha, int32_t* x_star, float* hard, float* rkl,
                             float* rkl_clip, float* loss, void* stream);

/*
 * Verification and OPD statistics in one pass over the batch (AdaFlash
 * Section 3.1: the supervision comes from the rows verification reads;
 * Section 2.1 for the rule).  Arguments are spec_verify's (inputs, outputs,
 * workspace) followed by spec_opd_stats's (delta, alpha and the five
 * statistics outputs), with the same meaning, layouts and ranges; the
 * results equal those of the two calls, up to the near-ties of the
 * verification rule.
 *
 * Every verified row pair (i < L_b) is read once from memory for both: the
 * statistics need all L_b positions, so there is no early exit.  At T_b = 1
 * the statistics' normalisers decide position i; at T_b = 0 the target
 * argmax does; any other T_b adds a second pair of softmax sums.  The final
 * token then comes from the same final pass as spec_verify (residual row
 * pair, or bonus row L_b).  Device-detected errors and the status word
 * behave as for spec_verify (read them with spec_verify_device_status on
 * `workspace`); the statistics of a request whose L_b is valid are computed
 * even when another of its inputs is invalid.  Padded layout only.
 */
spec_status_t spec_verify_opd(const void* target_logits, const void* draft_logits,
                              spec_dtype_t dtype, const int32_t* draft_tokens,
                              const int32_t* lengths, const float* uniforms,
                              const float* temperature, int B, int k, int V, float delta,
                              float alpha, int32_t* out_tokens, int32_t* num_accepted,
                              int32_t* x_star, float* hard, float* rkl, float* rkl_clip,
                              float* loss, void* workspace, size_t workspace_bytes, void* stream);

/*
 * D3D branch selection after a verification round ("D3D: Decoupled
 * Diffusion Drafting for Asynchronous Speculative Decoding", Methodology,
 * asynchronous inference).  While the target verifies a block, a packed
 * drafter pass prepares successor blocks for selected rejection positions and
 * the full-acceptance case (position coverage C, token fan-out F: a budget of
 * block * [(C - 1) F + 2] tokens).  A prepared branch whose assumed verified
 * prefix matches the actual one is a cache hit and its block is reused;
 * otherwise the next block must be drafted synchronously.
 *
 *   num_accepted  [B]          int32: n from spec_verify (-1: invalid, never a hit)
 *   out_tokens    [B, k+1]     int32: from spec_verify; out_tokens[b][n] is the
 *                              token the round emitted after its accepted drafts
 *   branch_pos    [B, NB]      int32: position at which branch j assumes that token
 *                              (a rejection there, or L_b for full acceptance);
 *                              < 0 marks an unused slot
 *   branch_tok    [B, NB]      int32: the token branch j assumes at that position
 *   branch_block  [B, NB, blk] int32: the successor block prepared for branch j
 *   hit           [B]          int32 out: lowest j whose (pos, tok) equals
 *                              (n, out_tokens[b][n]), or -1 on a miss
 *   next_block    [B, blk]     int32 out: branch_block[b][hit], or all -1 on a miss
 *   hits          [1]          int32 out (may be NULL): number of requests that hit
 *
 * All device buffers; nothing is allocated.  Launched with programmatic
 * dependent launch, so it may directly follow spec_verify on `stream`.
 * Host-detectable errors return before anything is enqueued.
 */
spec_status_t spec_d3d_select(const int32_t* num_accepted, const int32_t* out_tokens,
                              const int32_t* branch_pos, const int32_t* branch_tok,
                              const int32_t* branch_block, int B, int k, int NB, int blk,
                              int32_t* hit, int32_t* next_block, int32_t* hits, void* stream);

/* Static description of a status code. */
const char* spec_status_string(spec_status_t status);

/* SPEC_VERIFY_ABI_VERSION of the loaded library. */
int spec_abi_version(void);

/*
 * Range-checking builds.  The library built with -DSPEC_DEBUG
 * (libspecverify_debug.so, same entry points and results) checks, on the
 * device, every index its kernels form into a buffer whose extent is known:
 * row descriptors, logit rows of both buffers, partial slots, completion
 * counters, segments, sampled tokens, OPD outputs and D3D branch slots.  An
 * index outside its range is counted, the site of the first failing check
 * kept, and the access redirected to element 0 of the same buffer, so that a
 * fault of the library's own indexing shows as a count instead of a stray
 * access.  Site codes:
 *    1 plan: descriptor slot        7 final pass: residual / bonus row
 *    2 sweep: descriptor index      8 final pass: chosen segment
 *    3 sweep: logit row             9 final pass: sampled token < V
 *    4 sweep: partial slot         10 OPD: logit row, argmax element
 *    5 sweep: completion counter   11 OPD: output element
 *    6 sweep: decided position     12 D3D: branch slot
 */

/* 1 if the loaded library is the range-checking build, else 0. */
int spec_debug_build(void);

/*
 * Wait for `stream`, then copy the range checks that failed on the current
 * device since the last reset into *failures and the site of the first of
 * them into *first_site (0 when none; both host pointers, either may be
 * null), and reset both when `reset` is non-zero.  The counters are
 * device-wide (every call on the device adds to them).  A release build
 * reports 0 and SPEC_OK.  Returns SPEC_OK or SPEC_ERR_CUDA.
 */
spec_status_t spec_debug_checks(int32_t* failures, int32_t* first_site, int reset, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
