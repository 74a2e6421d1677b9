// Plain fp64 CPU oracle for batched speculative-decoding verification.
//
// TEST INFRASTRUCTURE ONLY: see oracle.h for who may use it, what it follows
// and which readings of the pages it takes.  Single-threaded, double
// precision, every loop in vocabulary-index order.

#include "oracle.h"

#include <cfloat>
#include <cmath>
#include <cstring>
#include <limits>
#include <vector>

namespace {

const double kInf = std::numeric_limits<double>::infinity();
const double kNaN = std::numeric_limits<double>::quiet_NaN();

// One logit, widened exactly to double (bf16 -> fp32 -> fp64 is exact).
double logit_at(const void* base, int dtype, size_t idx) {
  if (dtype == ORACLE_F32) return (double)((const float*)base)[idx];
  uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
  float f;
  std::memcpy(&f, &bits, sizeof f);
  return (double)f;
}

// A row of V logits inside a [rows, V] buffer.
struct Row {
  const void* base;
  int dtype;
  size_t offset;
  int V;
  double z(int v) const { return logit_at(base, dtype, offset + (size_t)v); }
};

// Largest logit and the lowest index that attains it (greedy tie rule).
void row_argmax(const Row& r, double* max_out, int* arg_out) {
  double m = -kInf;
  int arg = -1;
  for (int v = 0; v < r.V; ++v) {
    double z = r.z(v);
    if (z > m) {
      m = z;
      arg = v;
    }
  }
  *max_out = m;
  *arg_out = arg;
}

// Softmax at temperature T written as log p(v) = (z_v - M)/T - log S with
// M = max_v z_v and S = sum_v exp((z_v - M)/T), summed in index order.
struct Softmax {
  double M;
  double logS;
  bool ok;  // the row has finite, positive mass (no NaN / +inf, not all -inf)
};

Softmax row_softmax(const Row& r, double T) {
  double M;
  int arg;
  row_argmax(r, &M, &arg);
  double S = 0.0;
  for (int v = 0; v < r.V; ++v) S += std::exp((r.z(v) - M) / T);
  return Softmax{M, std::log(S), S > 0.0 && std::isfinite(S)};
}

double log_prob(const Row& r, const Softmax& sm, double T, int v) {
  return (r.z(v) - sm.M) / T - sm.logS;
}

double prob(const Row& r, const Softmax& sm, double T, int v) {
  return std::exp(log_prob(r, sm, T, v));
}

// Inverse CDF in ascending index order: the first j whose running sum of
// mass exceeds u * total.  Entries of zero mass are never chosen.  Returns
// the chosen index and the normalised CDF at both edges of its cell.
int inverse_cdf(const std::vector<double>& mass, double total, double u, double* f_lo,
                double* f_hi) {
  const double target = u * total;
  double cum = 0.0;
  for (size_t j = 0; j < mass.size(); ++j) {
    double before = cum;
    cum += mass[j];
    if (cum > target) {
      *f_lo = before / total;
      *f_hi = cum / total;
      return (int)j;
    }
  }
  // Reached only if u * total rounded up to the full sum: take the last
  // entry with positive mass.
  for (size_t j = mass.size(); j-- > 0;) {
    if (mass[j] > 0.0) {
      *f_lo = (total - mass[j]) / total;
      *f_hi = 1.0;
      return (int)j;
    }
  }
  *f_lo = 0.0;
  *f_hi = 1.0;
  return 0;
}

bool valid_uniform(double u) { return u >= 0.0 && u < 1.0; }  // false for NaN

// One request.  Returns 0 if valid, 1 if its inputs were rejected.
int verify_one(const void* tl, const void* dl, int dtype, const int32_t* tok, int L, double T,
               const double* u, int k, int V, size_t t_off, size_t d_off, int32_t* out,
               int32_t* n_out, double* margin, double* final_mass, int32_t* residual_zero) {
  for (int j = 0; j <= k; ++j) out[j] = -1;
  *n_out = -1;
  *margin = kNaN;
  *final_mass = kNaN;
  *residual_zero = 0;

  // Input checks: the length head's clamp gives 1 <= L <= k; temperature is
  // 0 (greedy) or a finite normal float (>= 2^-126, so log2(e)/T stays finite
  // in single precision); tokens index the vocabulary; the uniforms a
  // sampling request uses lie in [0, 1).  Rows are checked as they are read:
  // a row without finite mass makes the request invalid.
  if (L < 1 || L > k) return 1;
  if (!(T >= 0.0) || std::isinf(T)) return 1;
  if (T > 0.0 && T < (double)FLT_MIN) return 1;
  for (int i = 0; i < L; ++i)
    if (tok[i] < 0 || tok[i] >= V) return 1;
  if (T > 0.0)
    for (int i = 0; i <= L; ++i)
      if (!valid_uniform(u[i])) return 1;

  auto target_row = [&](int i) { return Row{tl, dtype, t_off + (size_t)i * V, V}; };
  auto draft_row = [&](int i) { return Row{dl, dtype, d_off + (size_t)i * V, V}; };

  int n = L;
  if (T == 0.0) {
    // Greedy: accept while the draft equals the target argmax; at the first
    // mismatch emit the target argmax; if all L match, emit the argmax of
    // target row L.
    int final_token = -1;
    for (int i = 0; i < L; ++i) {
      double m;
      int g;
      row_argmax(target_row(i), &m, &g);
      if (g < 0) return 1;
      if (tok[i] != g) {
        n = i;
        final_token = g;
        break;
      }
    }
    if (n == L) {
      double m;
      row_argmax(target_row(L), &m, &final_token);
      if (final_token < 0) return 1;
    }
    for (int i = 0; i < n; ++i) out[i] = tok[i];
    out[n] = final_token;
    *n_out = n;
    *margin = kInf;
    return 0;
  }

  // Sampling: accept x_i iff u_i < min(1, p_i(x_i) / q_i(x_i)); stop at the
  // first rejection.
  double marg = kInf;
  for (int i = 0; i < L; ++i) {
    Row tr = target_row(i), dr = draft_row(i);
    Softmax ps = row_softmax(tr, T), qs = row_softmax(dr, T);
    if (!ps.ok || !qs.ok) return 1;
    // A token the target gives probability zero is never accepted; one the
    // drafter gives probability zero (and the target not) always is.
    double lp = log_prob(tr, ps, T, tok[i]);
    double ratio = lp == -kInf ? 0.0 : std::exp(lp - log_prob(dr, qs, T, tok[i]));
    double accept_prob = ratio < 1.0 ? ratio : 1.0;
    marg = std::fmin(marg, std::fabs(u[i] - accept_prob));
    if (!(u[i] < accept_prob)) {
      n = i;
      break;
    }
  }

  // Final token from uniforms[L]: the residual normalize(max(0, p_n - q_n))
  // at a rejection, or the target distribution of row L when all L drafts
  // were accepted.
  std::vector<double> mass(V);
  double total = 0.0;
  if (n < L) {
    Row tr = target_row(n), dr = draft_row(n);
    Softmax ps = row_softmax(tr, T), qs = row_softmax(dr, T);
    for (int v = 0; v < V; ++v) {
      double r = prob(tr, ps, T, v) - prob(dr, qs, T, v);
      mass[v] = r > 0.0 ? r : 0.0;
      total += mass[v];
    }
    if (total == 0.0) {
      // p_n == q_n, where a rejection has probability zero: draw from p_n.
      *residual_zero = 1;
      marg = 0.0;
      total = 0.0;
      for (int v = 0; v < V; ++v) {
        mass[v] = prob(tr, ps, T, v);
        total += mass[v];
      }
    }
  } else {
    Row tr = target_row(L);
    Softmax ps = row_softmax(tr, T);
    if (!ps.ok) return 1;
    for (int v = 0; v < V; ++v) {
      mass[v] = prob(tr, ps, T, v);
      total += mass[v];
    }
  }
  double f_lo, f_hi;
  int final_token = inverse_cdf(mass, total, u[L], &f_lo, &f_hi);
  marg = std::fmin(marg, std::fmin(u[L] - f_lo, f_hi - u[L]));

  for (int i = 0; i < n; ++i) out[i] = tok[i];
  out[n] = final_token;
  *n_out = n;
  *margin = marg;
  *final_mass = total;
  return 0;
}

int verify_all(const void* tl, const void* dl, int dtype, const int32_t* tokens,
               const int32_t* lengths, const double* uniforms, const float* temperature, int B,
               int k, int V, int32_t* out_tokens, int32_t* num_accepted, double* margin,
               double* final_mass, int32_t* residual_zero) {
  int bad = 0;
  for (int b = 0; b < B; ++b) {
    double m, fm;
    int32_t rz;
    size_t t_off = (size_t)b * (size_t)(k + 1) * (size_t)V;
    size_t d_off = (size_t)b * (size_t)k * (size_t)V;
    bad += verify_one(tl, dl, dtype, tokens + (size_t)b * k, lengths[b], (double)temperature[b],
                      uniforms + (size_t)b * (k + 1), k, V, t_off, d_off,
                      out_tokens + (size_t)b * (k + 1), num_accepted + b, &m, &fm, &rz);
    if (margin) margin[b] = m;
    if (final_mass) final_mass[b] = fm;
    if (residual_zero) residual_zero[b] = rz;
  }
  return bad;
}

}  // namespace

extern "C" int oracle_verify_f64u(const void* target_logits, const void* draft_logits, int dtype,
                                  const int32_t* draft_tokens, const int32_t* lengths,
                                  const double* uniforms, const float* temperature, int B, int k,
                                  int V, int32_t* out_tokens, int32_t* num_accepted,
                                  double* margin, double* final_mass, int32_t* residual_zero) {
  return verify_all(target_logits, draft_logits, dtype, draft_tokens, lengths, uniforms,
                    temperature, B, k, V, out_tokens, num_accepted, margin, final_mass,
                    residual_zero);
}

extern "C" int oracle_verify(const void* target_logits, const void* draft_logits, int dtype,
                             const int32_t* draft_tokens, const int32_t* lengths,
                             const float* uniforms, const float* temperature, int B, int k, int V,
                             int32_t* out_tokens, int32_t* num_accepted, double* margin,
                             double* final_mass, int32_t* residual_zero) {
  std::vector<double> u((size_t)B * (size_t)(k + 1));
  for (size_t j = 0; j < u.size(); ++j) u[j] = (double)uniforms[j];
  return verify_all(target_logits, draft_logits, dtype, draft_tokens, lengths, u.data(),
                    temperature, B, k, V, out_tokens, num_accepted, margin, final_mass,
                    residual_zero);
}

extern "C" void oracle_row_stats(const void* logits, int dtype, int64_t rows, int V,
                                 const float* temperature_per_row, double* row_max,
                                 double* row_lse, int32_t* row_arg) {
  for (int64_t r = 0; r < rows; ++r) {
    Row row{logits, dtype, (size_t)r * (size_t)V, V};
    double m;
    int arg;
    row_argmax(row, &m, &arg);
    row_max[r] = m;
    row_arg[r] = arg;
    double T = (double)temperature_per_row[r];
    if (T == 0.0) {
      row_lse[r] = kNaN;
    } else {
      Softmax sm = row_softmax(row, T);
      row_lse[r] = sm.M / T + sm.logS;
    }
  }
}

// ---------------------------------------------------------------------------
// OPD supervision statistics (AdaFlash Section 3.1), one position at a time:
// both softmaxes at temperature 1 in double, then the three sums in index
// order exactly as the formulas are written.
// ---------------------------------------------------------------------------
extern "C" int oracle_opd_stats(const void* target_logits, const void* draft_logits, int dtype,
                                const int32_t* lengths, int B, int k, int V, double delta,
                                double alpha, int32_t* x_star, double* hard, double* rkl,
                                double* rkl_clip, double* loss) {
  int bad = 0;
  for (int b = 0; b < B; ++b) {
    const int L = lengths[b];
    const bool ok_len = L >= 1 && L <= k;
    if (!ok_len) ++bad;
    double sum_hard = 0.0, sum_clip = 0.0;
    for (int i = 0; i < k; ++i) {
      const size_t o = (size_t)b * k + i;
      x_star[o] = -1;
      hard[o] = rkl[o] = rkl_clip[o] = kNaN;
      if (!ok_len || i >= L) continue;
      Row t{target_logits, dtype, ((size_t)b * (k + 1) + i) * (size_t)V, V};
      Row d{draft_logits, dtype, ((size_t)b * k + i) * (size_t)V, V};
      Softmax sp = row_softmax(t, 1.0), sq = row_softmax(d, 1.0);
      double mt;
      int arg;
      row_argmax(t, &mt, &arg);
      if (!sp.ok || !sq.ok) {
        sum_hard = sum_clip = kNaN;
        continue;
      }
      x_star[o] = arg;
      hard[o] = -log_prob(d, sq, 1.0, arg);
      double kl = 0.0, kl_clip = 0.0;
      for (int y = 0; y < V; ++y) {
        const double q = prob(d, sq, 1.0, y);
        const double p = prob(t, sp, 1.0, y);
        double term;
        if (q == 0.0) term = 0.0;          // 0 log 0 = 0
        else if (p == 0.0) term = kInf;    // mass where the target has none
        else term = q * std::log(q / p);
        kl += term;
        kl_clip += std::fmin(term, delta);
      }
      rkl[o] = kl;
      rkl_clip[o] = kl_clip;
      sum_hard += hard[o];
      sum_clip += kl_clip;
    }
    loss[b] = ok_len ? alpha * (sum_hard / L) + (1.0 - alpha) * (sum_clip / L) : kNaN;
  }
  return bad;
}

// ---------------------------------------------------------------------------
// D3D branch selection: compare every branch's assumption with the verified
// outcome, first match wins.
// ---------------------------------------------------------------------------
extern "C" int oracle_d3d_select(const int32_t* num_accepted, const int32_t* out_tokens,
                                 const int32_t* branch_pos, const int32_t* branch_tok,
                                 const int32_t* branch_block, int B, int k, int NB, int blk,
                                 int32_t* hit, int32_t* next_block) {
  int hits = 0;
  for (int b = 0; b < B; ++b) {
    const int n = num_accepted[b];
    int found = -1;
    if (n >= 0 && n <= k) {
      const int token = out_tokens[(size_t)b * (k + 1) + n];
      for (int j = 0; j < NB; ++j) {
        const size_t o = (size_t)b * NB + j;
        if (branch_pos[o] >= 0 && branch_pos[o] == n && branch_tok[o] == token) {
          found = j;
          break;
        }
      }
    }
    hit[b] = found;
    for (int t = 0; t < blk; ++t)
      next_block[(size_t)b * blk + t] =
          found >= 0 ? branch_block[((size_t)b * NB + found) * blk + t] : -1;
    if (found >= 0) ++hits;
  }
  return hits;
}
