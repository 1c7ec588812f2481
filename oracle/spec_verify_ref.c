/*
 * spec_verify_ref.c -- float64 CPU oracle of the batched speculative-sampling
 * verify step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg load this library.  The CUDA path shares no code, header,
 * table or helper with it, and it imports nothing from the CUDA path.
 *
 * Every step follows the pages in the order they state it, with no blocking,
 * fusion or reordering:
 *
 *  - Temperature softmax of each target row and each draft row:
 *    p = softmax(z / T), q likewise, with the same T for both.
 *    ("Fast Inference from Transformers via Speculative Decoding" explainer,
 *    PyTorch sketch, Step 1 and Step 2: softmax(logits / temperature);
 *    toolsku "LLM speculative decoding optimisation", verify sketch.)
 *  - Acceptance of draft token x_i with probability min(1, p_i(x_i)/q_i(x_i)),
 *    decided by u_i < p_i(x_i)/q_i(x_i).
 *    (disassemble-channel "Speculative Decoding theory", Step 3 acceptance
 *    formula and the simulation's `random() < acceptance_prob`.)
 *  - The first rejected position k truncates the draft: x_0..x_{k-1} are kept.
 *    (same page, Step 3: everything after the first rejection is discarded.)
 *  - At k, one token is drawn from the residual
 *    p'(x) = max(0, p(x) - q(x)) / sum_x' max(0, p(x') - q(x')),
 *    falling back to p when that sum is zero.
 *    (same page, "modified distribution" definition, and the simulation's
 *    fallback branch.)
 *  - When every draft is accepted, a bonus token is drawn from the target row
 *    at position gamma_b + 1.  (same page, Step 3 last paragraph; toolsku verify
 *    sketch, bonus branch.)
 *  - Greedy mode: with temperature -> 0 acceptance reduces to argmax matching.
 *    (explainer, "Implementation points", greedy paragraph; zvxbase
 *    "draft length by load", K=3 worked example.)  In a sampling call, a
 *    request whose temperature is exactly 0 takes these greedy steps.
 *
 * Readings where the pages are silent:
 *  - accept is strict: u < ratio; q(x) == 0 accepts.
 *  - no epsilons are added to q or to the residual sum.
 *  - the resample/bonus draws use their own uniform u[b][G]; the inverse CDF
 *    runs over ascending token id and returns the smallest j with C_j > u*S.
 *    If rounding leaves no such j, the largest j with r_j > 0 is returned:
 *    the token the exact inequality u*S < S selects.  (C_{V-1} is the same
 *    ascending sum as S, and u*S < S for u < 1 whenever S is a normal double,
 *    so this happens only when S is subnormal.)
 *  - "the residual sum is zero" is tested on the float64 sum; the mass itself
 *    is reported (resid_mass) so that a caller can tell a residual that
 *    cancelled to within rounding from a clear one.
 *  - num_accepted counts accepted drafts only (emitted = num_accepted + 1).
 *  - greedy argmax ties go to the lowest token id.
 *
 * Inputs are widened exactly (bf16 -> float32 -> double; float32 -> double).
 * Temperature is widened from float32.  Uniforms are passed as double so that
 * tests can probe decision boundaries finer than float32 allows; the public
 * float32 uniforms widen to double exactly.
 *
 * Layout: target logits [B][G+1][V], draft logits [B][G][V], draft tokens
 * [B][G], gamma [B], uniforms [B][G+1] (column i < gamma_b is the acceptance
 * draw of position i, column G is the resample/bonus draw), temperature [B],
 * out_tokens [B][G+1] (-1 after the emitted tokens), num_accepted [B].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define REF_F32 0
#define REF_BF16 1

/* Exact widening of one logit to double. */
static double logit_at(const void *base, int dtype, size_t idx) {
  if (dtype == REF_F32) return (double)((const float *)base)[idx];
  uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static size_t target_row(int b, int i, int G, int V) {
  return ((size_t)b * (size_t)(G + 1) + (size_t)i) * (size_t)V;
}

static size_t draft_row(int b, int i, int G, int V) {
  return ((size_t)b * (size_t)G + (size_t)i) * (size_t)V;
}

/*
 * Temperature softmax of one row in float64: m = max z, then
 * p[v] = exp((z[v] - m) / T) / sum_v' exp((z[v'] - m) / T), summed in plain
 * ascending order.  Writes p when p_out is non-NULL; returns the sum s and m.
 */
static void softmax_row(const void *base, int dtype, size_t off, int V, double T,
                        double *p_out, double *m_out, double *s_out) {
  double m = -INFINITY;
  for (int v = 0; v < V; ++v) {
    double z = logit_at(base, dtype, off + (size_t)v);
    if (z > m) m = z;
  }
  double s = 0.0;
  for (int v = 0; v < V; ++v) {
    double e = exp((logit_at(base, dtype, off + (size_t)v) - m) / T);
    if (p_out) p_out[v] = e;
    s += e;
  }
  if (p_out)
    for (int v = 0; v < V; ++v) p_out[v] /= s;
  *m_out = m;
  *s_out = s;
}

/* Probability of token x in a row whose max and sum are already known. */
static double prob_of(const void *base, int dtype, size_t off, int x, double T,
                      double m, double s) {
  return exp((logit_at(base, dtype, off + (size_t)x) - m) / T) / s;
}

/*
 * Inverse-CDF draw over weights r[0..V-1] with total S, driven by u in [0,1):
 * the smallest j whose inclusive prefix C_j exceeds u*S.  If rounding leaves
 * none (only for a subnormal S, where u*S can round up to S), the largest j
 * with r[j] > 0, which is the token the exact u*S < S selects.  *margin gets
 * the distance of u*S to the nearer edge of j's interval, divided by S.
 */
static int inverse_cdf(const double *r, int V, double S, double u, double *margin) {
  double target = u * S;
  double c_prev = 0.0, c = 0.0;
  for (int j = 0; j < V; ++j) {
    c_prev = c;
    c += r[j];
    if (c > target) {
      double lo = target - c_prev, hi = c - target;
      *margin = (lo < hi ? lo : hi) / S;
      return j;
    }
  }
  for (int j = V - 1; j >= 0; --j) {
    if (r[j] > 0.0) {
      *margin = 0.0;
      return j;
    }
  }
  *margin = 0.0;
  return 0;
}

/* Greedy steps for request b: g_i = argmax_v t[b][i][v] (lowest id on ties),
 * k = first i < gamma_b with x_i != g_i (else gamma_b), out = x_0..x_{k-1},
 * g_k.  tie[i] (optional) flags target rows whose maximum occurs twice.
 * Returns k. */
static int greedy_one(const void *target, int dtype, int b, int G, int V,
                      const int32_t *tokens, int gb, int32_t *out, int32_t *tie) {
  for (int i = 0; i <= G; ++i) {
    out[i] = -1;
    if (tie) tie[i] = 0;
  }
  int k = gb;
  for (int i = 0; i <= gb; ++i) {
    const size_t off = target_row(b, i, G, V);
    int best = 0, ties = 0;
    double zbest = logit_at(target, dtype, off);
    for (int v = 1; v < V; ++v) {
      const double z = logit_at(target, dtype, off + (size_t)v);
      if (z > zbest) {
        zbest = z;
        best = v;
        ties = 0;
      } else if (z == zbest) {
        ties = 1;
      }
    }
    if (tie) tie[i] = ties;
    if (i == gb || tokens[(size_t)b * G + i] != best) {
      k = i;
      out[i] = best;
      break;
    }
    out[i] = best; /* equals the accepted draft token */
  }
  return k;
}

typedef struct {
  const void *target;
  const void *draft;
  int dtype, B, G, V;
  const int32_t *tokens;
  const int32_t *gamma;
  const double *u;
  const float *temperature;
  int32_t *out_tokens;
  int32_t *num_accepted;
  double *p_tok, *q_tok, *margin_accept, *margin_cdf, *resid_mass;
  /* optional row statistics computed beforehand (rows-first mode): max and
   * sum of target row i at stats_t[b*(G+1)+i], draft row i at stats_d[b*G+i] */
  const double *stats_t_m, *stats_t_s, *stats_d_m, *stats_d_s;
} sample_args;

/* One request of the sampling verify step; returns 0, or -3 on malloc failure. */
static int sample_one(const sample_args *a, int b) {
  const int G = a->G, V = a->V, gb = a->gamma[b];
  const double T = (double)a->temperature[b];
  const double *u = a->u + (size_t)b * (size_t)(G + 1);
  int32_t *out = a->out_tokens + (size_t)b * (size_t)(G + 1);
  for (int i = 0; i <= G; ++i) out[i] = -1;
  if (a->margin_accept)
    for (int i = 0; i < G; ++i) a->margin_accept[(size_t)b * G + i] = NAN;
  if (a->p_tok)
    for (int i = 0; i < G; ++i) a->p_tok[(size_t)b * G + i] = NAN;
  if (a->q_tok)
    for (int i = 0; i < G; ++i) a->q_tok[(size_t)b * G + i] = NAN;
  if (a->resid_mass) a->resid_mass[b] = NAN;

  if (T == 0.0) {
    /* Temperature 0: the greedy steps.  There is no ratio and no CDF draw; an
     * exact argmax tie counts as a near-tie (margin 0), a decided row as far
     * from any tie (margin +inf). */
    int32_t tie[64];
    const int k = greedy_one(a->target, a->dtype, b, G, V, a->tokens, gb, out, tie);
    if (a->margin_accept)
      for (int i = 0; i < k && i < G; ++i)
        a->margin_accept[(size_t)b * G + i] = tie[i] ? 0.0 : INFINITY;
    if (a->margin_accept && k < gb) a->margin_accept[(size_t)b * G + k] = tie[k] ? 0.0 : INFINITY;
    if (a->margin_cdf) a->margin_cdf[b] = tie[k] ? 0.0 : INFINITY;
    a->num_accepted[b] = k;
    return 0;
  }

  /* Steps 1-2: per position, softmax both rows, gather at x_i, accept/reject. */
  int k = gb;
  for (int i = 0; i < gb; ++i) {
    const int x = a->tokens[(size_t)b * G + i];
    double mt, st, md, sd;
    if (a->stats_t_m) { /* the same softmax_row results, computed beforehand */
      mt = a->stats_t_m[(size_t)b * (G + 1) + i];
      st = a->stats_t_s[(size_t)b * (G + 1) + i];
      md = a->stats_d_m[(size_t)b * G + i];
      sd = a->stats_d_s[(size_t)b * G + i];
    } else {
      softmax_row(a->target, a->dtype, target_row(b, i, G, V), V, T, NULL, &mt, &st);
      softmax_row(a->draft, a->dtype, draft_row(b, i, G, V), V, T, NULL, &md, &sd);
    }
    const double p = prob_of(a->target, a->dtype, target_row(b, i, G, V), x, T, mt, st);
    const double q = prob_of(a->draft, a->dtype, draft_row(b, i, G, V), x, T, md, sd);
    if (a->p_tok) a->p_tok[(size_t)b * G + i] = p;
    if (a->q_tok) a->q_tok[(size_t)b * G + i] = q;
    const double ratio = (q == 0.0) ? INFINITY : p / q;
    if (a->margin_accept) a->margin_accept[(size_t)b * G + i] = fabs(u[i] - ratio);
    const int accept = (q == 0.0) || (u[i] < ratio);
    if (!accept) {
      k = i;
      break;
    }
    out[i] = x;
  }

  /* Step 3: residual at k, or the bonus row when every draft was accepted. */
  double *p = (double *)malloc(sizeof(double) * (size_t)V);
  double *r = (double *)malloc(sizeof(double) * (size_t)V);
  if (!p || !r) {
    free(p);
    free(r);
    return -3;
  }
  double m, s, S = 0.0;
  softmax_row(a->target, a->dtype, target_row(b, k, G, V), V, T, p, &m, &s);
  if (k < gb) {
    double *q = (double *)malloc(sizeof(double) * (size_t)V);
    if (!q) {
      free(p);
      free(r);
      return -3;
    }
    softmax_row(a->draft, a->dtype, draft_row(b, k, G, V), V, T, q, &m, &s);
    for (int v = 0; v < V; ++v) {
      const double d = p[v] - q[v];
      r[v] = d > 0.0 ? d : 0.0;
      S += r[v];
    }
    free(q);
    if (a->resid_mass) a->resid_mass[b] = S;
    if (S == 0.0) { /* residual vanished: fall back to p */
      for (int v = 0; v < V; ++v) {
        r[v] = p[v];
        S += r[v];
      }
    }
  } else {
    for (int v = 0; v < V; ++v) {
      r[v] = p[v];
      S += r[v];
    }
  }
  double margin = 0.0;
  out[k] = inverse_cdf(r, V, S, u[G], &margin);
  if (a->margin_cdf) a->margin_cdf[b] = margin;
  a->num_accepted[b] = k;
  free(p);
  free(r);
  return 0;
}

static int check_common(int B, int G, int V, int dtype, const int32_t *tokens,
                        const int32_t *gamma) {
  if (B < 0 || G < 0 || V < 1 || (dtype != REF_F32 && dtype != REF_BF16)) return -1;
  for (int b = 0; b < B; ++b) {
    if (gamma[b] < 0 || gamma[b] > G) return -1;
    for (int i = 0; i < gamma[b]; ++i) {
      const int32_t x = tokens[(size_t)b * G + i];
      if (x < 0 || x >= V) return -1;
    }
  }
  return 0;
}

/*
 * Sampling verify step for B requests.  p_tok, q_tok, margin_accept ([B][G]),
 * margin_cdf and resid_mass ([B]) are optional (NULL).  margin_accept[b][i] is
 * |u - ratio| for every evaluated position, NaN elsewhere; resid_mass[b] is
 * the float64 sum of max(0, p_k - q_k) after a rejection at k, NaN when every
 * draft was accepted.  Returns 0, -1 on invalid input, -3 on allocation
 * failure.  nthreads <= 0 uses the OpenMP default.
 *
 * rows_first != 0 changes only how the work is spread over threads: the
 * maximum and sum of every row that the acceptance tests may need (target
 * rows 0..gamma_b, draft rows 0..gamma_b-1) are computed first, one row per
 * OpenMP iteration, by the same softmax_row; the requests then run as before
 * on those values.  The results are identical; it serves batches with fewer
 * requests than threads.
 */
int sv_ref_sample(const void *target_logits, const void *draft_logits, int dtype, int B,
                  int G, int V, const int32_t *draft_tokens, const int32_t *gamma,
                  const double *uniforms, const float *temperature, int32_t *out_tokens,
                  int32_t *num_accepted, double *p_tok, double *q_tok,
                  double *margin_accept, double *margin_cdf, double *resid_mass,
                  int rows_first, int nthreads) {
  if (check_common(B, G, V, dtype, draft_tokens, gamma)) return -1;
  if (G > 63) return -1;
  for (int b = 0; b < B; ++b) {
    if (!(temperature[b] >= 0.0f) || isinf(temperature[b])) return -1;
    for (int i = 0; i <= G; ++i) {
      const double u = uniforms[(size_t)b * (G + 1) + i];
      if (!(u >= 0.0 && u < 1.0)) return -1;
    }
  }
  sample_args a = {target_logits, draft_logits, dtype, B, G, V, draft_tokens, gamma,
                   uniforms, temperature, out_tokens, num_accepted, p_tok, q_tok,
                   margin_accept, margin_cdf, resid_mass, NULL, NULL, NULL, NULL};
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#endif
  double *stats = NULL;
  if (rows_first && B > 0) {
    /* rows (b, i): target rows i = 0..G, then draft rows i = 0..G-1 */
    const size_t nt = (size_t)B * (size_t)(G + 1), nd = (size_t)B * (size_t)G;
    stats = (double *)malloc(sizeof(double) * 2 * (nt + nd));
    if (!stats) return -3;
    double *tm = stats, *ts = stats + nt, *dm = stats + 2 * nt, *ds = stats + 2 * nt + nd;
    const long nrows = (long)(nt + nd);
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (long r = 0; r < nrows; ++r) {
      if ((size_t)r < nt) {
        const int b = (int)(r / (G + 1)), i = (int)(r % (G + 1));
        if (i <= gamma[b] && temperature[b] != 0.0f)
          softmax_row(target_logits, dtype, target_row(b, i, G, V), V,
                      (double)temperature[b], NULL, &tm[r], &ts[r]);
      } else {
        const size_t rd = (size_t)r - nt;
        const int b = (int)(rd / (size_t)G), i = (int)(rd % (size_t)G);
        if (i < gamma[b] && temperature[b] != 0.0f)
          softmax_row(draft_logits, dtype, draft_row(b, i, G, V), V,
                      (double)temperature[b], NULL, &dm[rd], &ds[rd]);
      }
    }
    a.stats_t_m = tm;
    a.stats_t_s = ts;
    a.stats_d_m = dm;
    a.stats_d_s = ds;
  }
  int err = 0;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(min : err)
#endif
  for (int b = 0; b < B; ++b) {
    const int e = sample_one(&a, b);
    if (e < err) err = e;
  }
  (void)nthreads;
  free(stats);
  return err;
}

/*
 * Greedy verify step: g_i = argmax_v t[b][i][v] (lowest id on ties),
 * k = first i < gamma_b with x_i != g_i (else gamma_b),
 * out = x_0..x_{k-1}, g_k.  exact_tie ([B][G+1], optional) flags rows whose
 * maximum occurs more than once.  Returns 0 or -1 on invalid input.
 */
int sv_ref_greedy(const void *target_logits, int dtype, int B, int G, int V,
                  const int32_t *draft_tokens, const int32_t *gamma, int32_t *out_tokens,
                  int32_t *num_accepted, int32_t *exact_tie, int nthreads) {
  if (check_common(B, G, V, dtype, draft_tokens, gamma)) return -1;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (int b = 0; b < B; ++b) {
    int32_t *out = out_tokens + (size_t)b * (size_t)(G + 1);
    const int k = greedy_one(target_logits, dtype, b, G, V, draft_tokens, gamma[b], out,
                             exact_tie ? exact_tie + (size_t)b * (G + 1) : NULL);
    num_accepted[b] = k;
  }
  (void)nthreads;
  return 0;
}

/* Temperature softmax of one row (for the oracle's own tests). */
int sv_ref_softmax_row(const void *row, int dtype, int V, double T, double *p_out) {
  if (V < 1 || !(T > 0.0)) return -1;
  double m, s;
  softmax_row(row, dtype, 0, V, T, p_out, &m, &s);
  return 0;
}
