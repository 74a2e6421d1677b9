/*
 * Plain, slow CPU oracle for batched speculative-decoding verification.
 *
 * TEST INFRASTRUCTURE ONLY.  This library exists to check the CUDA path.
 * Only the test suite, the package smoke check and the benchmark's CPU
 * baseline leg load it.  The product library never links, loads or calls it,
 * and it shares no code, header, table or helper with the CUDA sources.
 *
 * What it computes, per request b (independently), follows
 *   AdaFlash: Adaptive Speculative Decoding via On-Policy Distilled Diffusion
 *   Drafters (arXiv 2607.19223), Section 2.1 "Speculative Decoding":
 *   draft token x_i is accepted with probability min{1, p(x_i)/q(x_i)}, every
 *   token before the first rejected one is kept, and a corrected token is
 *   drawn from the residual distribution at the rejection point;
 * the residual distribution normalize(max(0, p - q)) is as restated in the
 *   AdaFlash reading notes (Zhongzhu Zhou), "Speculative decoding: the basic
 *   idea", step 4, and in the DFlash notes ("DFlash: Block Diffusion for Flash
 *   Speculative Decoding"), section 5.2;
 * the extra target token when every draft is accepted (m accepted + 1 emitted)
 *   is DFlash notes section 3.1, steps 6-7;
 * greedy verification at temperature 0 (accept iff the draft equals the target
 *   argmax, emit the target argmax at the first mismatch) is DFlash notes
 *   section 5.2, worked example #4, and AdaFlash Appendix B.1 (greedy is the
 *   default decoding mode);
 * the per-request verification length 1 <= L_b <= k comes from the adaptive
 *   length head's clamp, AdaFlash Section 3.2, Eq. for k-hat.
 *
 * All arithmetic is IEEE double, in vocabulary-index order, with no blocking
 * or reordering.  Build with -ffp-contract=off so that no fused multiply-add
 * changes the rounding between machines.
 *
 * Readings taken where the pages are silent:
 *  - decision i uses uniforms[b][i] with the strict test u < min(1, ratio);
 *  - the final (residual or bonus) sample uses uniforms[b][L_b];
 *  - inverse CDF in ascending vocabulary index: the first index j whose
 *    cumulative mass exceeds u * total;
 *  - argmax ties go to the lowest index;
 *  - if the residual mass is exactly zero, the sample is drawn from p;
 *  - temperature == 0 exactly selects the greedy rule; any T > 0 samples;
 *  - input domain (the pages state none): T is 0 or a finite normal float;
 *    a token the target gives probability zero is never accepted; a logit row
 *    the round reads that has no finite mass (NaN, +inf, or all -inf) makes
 *    the request invalid.
 */
#ifndef SPEC_VERIFY_ORACLE_H
#define SPEC_VERIFY_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* dtype codes for the logits buffers. */
#define ORACLE_F32 0
#define ORACLE_BF16 1

/*
 * Verify B requests.
 *   target_logits  [B, k+1, V]  (dtype; bf16 given as raw uint16 bits)
 *   draft_logits   [B, k,   V]
 *   draft_tokens   [B, k]  int32
 *   lengths        [B]     int32, valid range 1..k
 *   uniforms       [B, k+1] double (oracle_verify_f64u) or float (oracle_verify)
 *   temperature    [B]     float; 0 = greedy, > 0 finite = sampling
 * Outputs:
 *   out_tokens     [B, k+1] int32: n+1 tokens then -1
 *   num_accepted   [B]      int32: n, or -1 if the request's inputs are invalid
 * Optional diagnostics (each may be NULL), one value per request:
 *   margin         distance from every decision the outcome depended on to its
 *                  threshold: min over tested positions of |u_i - min(1,ratio_i)|
 *                  and, for the final sample, the distance from u to the edges
 *                  of the chosen cell of the normalised CDF.  0 when the
 *                  residual mass was zero.  +inf for greedy requests.
 *   final_mass     total unnormalised mass of the distribution the final token
 *                  was drawn from (residual: sum max(0,p-q); bonus: sum p).
 *                  NaN for greedy requests.
 *   residual_zero  1 if the residual mass was exactly zero (fallback to p).
 * Returns the number of invalid requests (0 when all were valid).
 */
int oracle_verify(const void* target_logits, const void* draft_logits, int dtype,
                  const int32_t* draft_tokens, const int32_t* lengths,
                  const float* uniforms, const float* temperature,
                  int B, int k, int V,
                  int32_t* out_tokens, int32_t* num_accepted,
                  double* margin, double* final_mass, int32_t* residual_zero);

int oracle_verify_f64u(const void* target_logits, const void* draft_logits, int dtype,
                       const int32_t* draft_tokens, const int32_t* lengths,
                       const double* uniforms, const float* temperature,
                       int B, int k, int V,
                       int32_t* out_tokens, int32_t* num_accepted,
                       double* margin, double* final_mass, int32_t* residual_zero);

/*
 * Per-row statistics of `rows` rows of V logits:
 *   row_max[r]  = max_v z[r][v]
 *   row_lse[r]  = log sum_v exp(z[r][v] / T_r)   (natural log, logits divided by T_r)
 *                 NaN when T_r == 0
 *   row_arg[r]  = lowest index attaining the maximum
 */
void oracle_row_stats(const void* logits, int dtype, int64_t rows, int V,
                      const float* temperature_per_row,
                      double* row_max, double* row_lse, int32_t* row_arg);

/*
 * On-policy distillation (OPD) supervision statistics, AdaFlash Section 3.1
 * ("Mixture OPD Loss with Reverse-KL" and "Entry-wise Divergence Clipping"),
 * worked through in the AdaFlash reading notes' numerical example for one
 * toy position.  For request b and every verified position i < L_b, with
 * p = softmax(target row i) and q = softmax(draft row i) (the models' own
 * distributions, temperature 1):
 *   x_star[b][i]   = argmax_y p(y)              (lowest index on ties)
 *   hard[b][i]     = -log q(x_star)             (hard-label cross-entropy term)
 *   rkl[b][i]      = sum_y q(y) log(q(y)/p(y))  (reverse KL, unclipped)
 *   rkl_clip[b][i] = sum_y min{ q(y) log(q(y)/p(y)), delta }
 *   loss[b]        = alpha * mean_{i<L_b} hard + (1 - alpha) * mean_{i<L_b} rkl_clip
 * Readings: 0 log 0 = 0 (an entry with q = 0 adds nothing); an entry with
 * q > 0 and p = 0 adds +inf (so delta after clipping); the pages average over
 * the k positions of a block, and with per-request lengths the average runs
 * over the L_b positions that were verified.  Positions i >= L_b get
 * x_star = -1 and NaN.  An invalid length makes the whole request NaN / -1;
 * a row without finite mass makes its position (and the loss) NaN.
 * Returns the number of requests with an invalid length.
 */
int oracle_opd_stats(const void* target_logits, const void* draft_logits, int dtype,
                     const int32_t* lengths, int B, int k, int V, double delta, double alpha,
                     int32_t* x_star, double* hard, double* rkl, double* rkl_clip,
                     double* loss);

/*
 * D3D branch selection after verification ("D3D: Decoupled Diffusion
 * Drafting for Asynchronous Speculative Decoding", Methodology, asynchronous
 * inference): while the target verifies a block, a packed drafter pass
 * prepares successor blocks for selected rejection positions and the
 * full-acceptance case; a branch whose assumed verified prefix matches the
 * actual one is a cache hit and its block is reused, otherwise the next
 * block must be drafted synchronously.
 *
 * Branch j of request b assumes that the round emits token branch_tok[b][j]
 * at position branch_pos[b][j] after accepting the drafts before it (a
 * rejection at that position, or the bonus token when the position is L_b).
 * The verified outcome of request b is n = num_accepted[b] and the token
 * out_tokens[b][n].  Branch j matches when branch_pos == n and branch_tok ==
 * out_tokens[b][n]; the lowest matching index is the hit.  A request with
 * n < 0 (invalid) never hits; branch_pos < 0 marks an unused slot.
 * Outputs: hit[b] = index or -1; next_block[b][0..blk) = the hit branch's
 * block, or -1s; returns the number of hits.
 */
int oracle_d3d_select(const int32_t* num_accepted, const int32_t* out_tokens,
                      const int32_t* branch_pos, const int32_t* branch_tok,
                      const int32_t* branch_block, int B, int k, int NB, int blk, int32_t* hit,
                      int32_t* next_block);

#ifdef __cplusplus
}
#endif

#endif
