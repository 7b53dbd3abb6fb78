/*
 * spec_oracle.c -- fp64 CPU oracle for speculative-sampling verification.
 *
 * TEST INFRASTRUCTURE ONLY.  Plain sequential C, double precision, no
 * blocking, no fusion, no reordering beyond what each definition states.
 * Shares nothing with the CUDA library.  See spec_oracle.h for the sources.
 *
 * Notation: p = target law, q = draft law (as in the proof of
 * "CS3602_FINAL_SpeDec", section "2. 困惑度测试(PPL)"); gamma = number of
 * draft tokens per verify step (K in the OpenVINO notebook).
 */
#include "spec_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  double z;
  int32_t idx;
} zi_pair;

/* Logit value as a double.  bf16 is the upper half of an IEEE binary32. */
static double logit_at(const void *base, int32_t dtype, int64_t off) {
  if (dtype == ORACLE_F32) return (double)((const float *)base)[off];
  uint32_t bits = (uint32_t)((const uint16_t *)base)[off] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* Copy one row into z[] and report NaN / +inf (BAD_LOGIT) and a row whose
 * every logit is -inf or NaN (NO_FINITE).  -inf is a legal logit
 * (probability 0). */
static int32_t load_row(const void *base, int32_t dtype, int64_t off, int32_t V,
                        double *z) {
  int32_t st = 0;
  int any_above = 0;
  for (int32_t v = 0; v < V; ++v) {
    z[v] = logit_at(base, dtype, off + v);
    if (isnan(z[v]) || z[v] == INFINITY) st |= ORACLE_BAD_LOGIT;
    if (!isnan(z[v]) && z[v] > -INFINITY) any_above = 1;
  }
  if (!any_above) st |= ORACLE_NO_FINITE;
  return st;
}

static int32_t bad_uniform(float u) { return !(u >= 0.0f && u < 1.0f); }

/* Greedy decoding picks the most likely token, the first one on ties (the
 * argmax calls of "Prepare autoregressive sampling" and of the draft loop in
 * "Prepare speculative sampling").  Softmax is monotone, so the argmax of
 * the logits is the argmax of p. */
static int32_t argmax_first(const double *z, int32_t V) {
  int32_t best = 0;
  for (int32_t v = 1; v < V; ++v)
    if (z[v] > z[best]) best = v;
  return best;
}

static int cmp_desc(const void *a, const void *b) {
  const zi_pair *x = (const zi_pair *)a, *y = (const zi_pair *)b;
  if (x->z > y->z) return -1;
  if (x->z < y->z) return 1;
  return (x->idx > y->idx) - (x->idx < y->idx);
}

/*
 * Tempered softmax with top-k then top-p filtering ("CS3602_FINAL_SpeDec",
 * "项目结构": utils.py holds the top-k / top-p filtering and the logits
 * normalisation; "问题分析与讨论" item 2: sampling with temperature, top-k and
 * top-p).  The pages print no code for it; this is the plainest reading:
 *   t_v = z_v / T
 *   top-k: keep z_v >= (k-th largest z, counted with multiplicity)
 *   pi_v = exp(t_v - max t) / sum over the kept set
 *   top-p: walk the kept values from the largest down, one group of equal
 *          logits at a time; stop at the first group where the cumulative
 *          mass reaches top_p; keep every token whose logit is >= that group's
 *   renormalise over what is kept.
 * Ties are kept by both filters, so each is a threshold on the raw logit.
 * The row must hold a finite logit (checked by the caller).
 */
static void filtered_law(const double *z, int32_t V, double T, int32_t top_k,
                         double top_p, double *prob, double *e, zi_pair *srt,
                         double *topp_margin) {
  const int k_on = top_k > 0 && top_k < V;
  const int p_on = top_p < 1.0;
  double tau = -INFINITY; /* keep z_v >= tau */
  *topp_margin = INFINITY;

  if (k_on || p_on) {
    for (int32_t v = 0; v < V; ++v) {
      srt[v].z = z[v];
      srt[v].idx = v;
    }
    qsort(srt, (size_t)V, sizeof(zi_pair), cmp_desc);
  }
  if (k_on) tau = srt[top_k - 1].z;

  double zmax = -INFINITY;
  for (int32_t v = 0; v < V; ++v)
    if (z[v] > zmax) zmax = z[v];
  const double tmax = zmax / T;

  double Zk = 0.0;
  for (int32_t v = 0; v < V; ++v) {
    e[v] = (z[v] >= tau) ? exp(z[v] / T - tmax) : 0.0;
    Zk += e[v];
  }

  if (p_on) {
    double M = 0.0, M_prev = 0.0;
    int found = 0;
    int32_t j = 0;
    while (j < V && srt[j].z >= tau) {
      const double zj = srt[j].z;
      double group = 0.0;
      int32_t g = j;
      while (g < V && srt[g].z == zj) {
        group += e[srt[g].idx];
        ++g;
      }
      M_prev = M;
      M += group;
      if (M / Zk >= top_p) {
        tau = zj;
        const double hi = M / Zk - top_p, lo = top_p - M_prev / Zk;
        *topp_margin = hi < lo ? hi : lo;
        found = 1;
        break;
      }
      j = g;
    }
    if (!found) *topp_margin = fabs(M / Zk - top_p);
  }

  double Z = 0.0;
  for (int32_t v = 0; v < V; ++v) {
    if (!(z[v] >= tau)) e[v] = 0.0;
    Z += e[v];
  }
  for (int32_t v = 0; v < V; ++v) prob[v] = e[v] / Z;
}

/*
 * Inverse-CDF draw in vocabulary order: the smallest v with u*W < C_v, where
 * C_v = w_0 + ... + w_v and W = C_{V-1}.  If rounding leaves no such v, the
 * last v with w_v > 0.  *margin = distance of u from the chosen interval's
 * ends, in units of W.  Returns -1 if W == 0.
 */
static int32_t draw_icdf(const double *w, int32_t V, double u, double *margin) {
  double W = 0.0;
  for (int32_t v = 0; v < V; ++v) W += w[v];
  if (!(W > 0.0)) {
    *margin = 0.0;
    return -1;
  }
  const double target = u * W;
  double C = 0.0;
  int32_t last = -1;
  for (int32_t v = 0; v < V; ++v) {
    if (w[v] > 0.0) last = v;
    const double C_prev = C;
    C += w[v];
    if (target < C) {
      const double a = (target - C_prev) / W, b = (C - target) / W;
      *margin = a < b ? a : b;
      return v;
    }
  }
  *margin = 0.0;
  return last;
}

typedef struct {
  double *zt, *zd, *p, *q, *w, *e;
  zi_pair *srt;
} scratch_t;

static int scratch_alloc(scratch_t *s, int32_t V) {
  s->zt = (double *)malloc(sizeof(double) * (size_t)V);
  s->zd = (double *)malloc(sizeof(double) * (size_t)V);
  s->p = (double *)malloc(sizeof(double) * (size_t)V);
  s->q = (double *)malloc(sizeof(double) * (size_t)V);
  s->w = (double *)malloc(sizeof(double) * (size_t)V);
  s->e = (double *)malloc(sizeof(double) * (size_t)V);
  s->srt = (zi_pair *)malloc(sizeof(zi_pair) * (size_t)V);
  return s->zt && s->zd && s->p && s->q && s->w && s->e && s->srt;
}

static void scratch_free(scratch_t *s) {
  free(s->zt);
  free(s->zd);
  free(s->p);
  free(s->q);
  free(s->w);
  free(s->e);
  free(s->srt);
}

int32_t oracle_distribution(const void *z, int32_t dtype, int32_t V, double T,
                            int32_t top_k, double top_p, double *prob,
                            double *topp_margin) {
  scratch_t s;
  if (!scratch_alloc(&s, V)) {
    scratch_free(&s);
    return -1;
  }
  int32_t st = load_row(z, dtype, 0, V, s.zt);
  if (!(st & ORACLE_ERROR_MASK))
    filtered_law(s.zt, V, T, top_k, top_p, prob, s.e, s.srt, topp_margin);
  scratch_free(&s);
  return st;
}

/*
 * One verify step for row b (steps 3 and 4 of "Prepare speculative
 * sampling"; acceptance rule and residual law as in the proof of
 * "CS3602_FINAL_SpeDec", "2. 困惑度测试(PPL)"):
 *   for i = 0 .. gamma_b - 1, with x = draft token i and u = uniforms[b,i,0]:
 *     accept iff u < p_i(x) / q_i(x)   (u in [0,1), so a ratio >= 1 accepts;
 *                                       if q_i(x) == 0: accept iff p_i(x) > 0)
 *     on the first rejection: draw from norm(max(0, p_i - q_i)) with
 *     uniforms[b,i,1] (from p_i if that residual is empty) and stop;
 *   if every draft is accepted: draw from p_{gamma_b} with
 *   uniforms[b,gamma_b,1].
 * Target row i scores draft slot i; target row gamma_b is the bonus row.
 * Greedy (T == 0): accept while argmax(target row i) == x_i; the next token
 * is the argmax of the first mismatching (or the bonus) target row.
 */
static void verify_one_row(const void *target, const void *draft,
                           const int32_t *tokens, const float *uniforms,
                           const int32_t *gamma_per_row, const oracle_params *P,
                           int32_t b, scratch_t *s, int32_t *acc_out,
                           int32_t *next_out, int32_t *st_out, float *p_draft,
                           float *q_draft, oracle_row_diag *dg) {
  const int32_t V = P->V, gm = P->gamma_max;
  const int greedy = P->temperature == 0.0;
  int32_t st = 0;
  dg->accept_margin = INFINITY;
  dg->cdf_margin = INFINITY;
  dg->topp_margin = INFINITY;
  dg->residual_mass = 0.0;
  dg->n_tests = 0;
  dg->n_draws = 0;
  dg->fallback_p = 0;
  if (p_draft)
    for (int32_t i = 0; i < gm; ++i) p_draft[(int64_t)b * gm + i] = NAN;
  if (q_draft)
    for (int32_t i = 0; i < gm; ++i) q_draft[(int64_t)b * gm + i] = NAN;

  const int32_t gb = gamma_per_row ? gamma_per_row[b] : gm;
  if (gb < 0 || gb > gm) {
    *acc_out = 0;
    *next_out = -1;
    *st_out = ORACLE_BAD_GAMMA;
    return;
  }

  for (int32_t i = 0; i <= gb; ++i) {
    const int bonus = (i == gb);
    int32_t x = -1;
    if (!bonus) {
      x = tokens[(int64_t)b * gm + i];
      if (x < 0 || x >= V) st |= ORACLE_BAD_TOKEN;
    }
    st |= load_row(target, P->dtype,
                   (int64_t)b * P->t_row_stride + (int64_t)i * P->t_pos_stride, V,
                   s->zt);

    if (greedy) {
      if (st & ORACLE_ERROR_MASK) break;
      const int32_t a = argmax_first(s->zt, V);
      if (!bonus && a == x) continue;
      *acc_out = i;
      *next_out = a;
      *st_out = st;
      return;
    }

    const float *u_i = uniforms + ((int64_t)b * (gm + 1) + i) * 2;
    if (!bonus) {
      st |= load_row(draft, P->dtype,
                     (int64_t)b * P->d_row_stride + (int64_t)i * P->d_pos_stride,
                     V, s->zd);
      if (bad_uniform(u_i[0])) st |= ORACLE_BAD_UNIFORM;
    }
    if (st & ORACLE_ERROR_MASK) break;

    double mg;
    filtered_law(s->zt, V, P->temperature, P->top_k, P->top_p, s->p, s->e,
                 s->srt, &mg);
    if (mg < dg->topp_margin) dg->topp_margin = mg;

    if (bonus) {
      if (bad_uniform(u_i[1])) {
        st |= ORACLE_BAD_UNIFORM;
        break;
      }
      const int32_t tok = draw_icdf(s->p, V, (double)u_i[1], &dg->cdf_margin);
      dg->n_draws = 1;
      *acc_out = gb;
      *next_out = tok;
      *st_out = st;
      return;
    }

    filtered_law(s->zd, V, P->temperature, P->top_k, P->top_p, s->q, s->e,
                 s->srt, &mg);
    if (mg < dg->topp_margin) dg->topp_margin = mg;

    const double px = s->p[x], qx = s->q[x];
    if (p_draft) p_draft[(int64_t)b * gm + i] = (float)px;
    if (q_draft) q_draft[(int64_t)b * gm + i] = (float)qx;
    dg->n_tests += 1;
    int accept;
    const double u0 = (double)u_i[0];
    if (qx > 0.0) {
      const double ratio = px / qx;
      accept = u0 < ratio;
      const double m = fabs(u0 - (ratio < 1.0 ? ratio : 1.0));
      if (m < dg->accept_margin) dg->accept_margin = m;
    } else {
      st |= ORACLE_Q_ZERO;
      accept = px > 0.0;
    }
    if (accept) continue;

    if (bad_uniform(u_i[1])) {
      st |= ORACLE_BAD_UNIFORM;
      break;
    }
    /* norm(max(0, p - q)): max_fn of "Prepare autoregressive sampling",
     * sampled rather than arg-maxed, as the proof requires. */
    double W = 0.0;
    for (int32_t v = 0; v < V; ++v) {
      const double d = s->p[v] - s->q[v];
      s->w[v] = d > 0.0 ? d : 0.0;
      W += s->w[v];
    }
    dg->residual_mass = W;
    int32_t tok = draw_icdf(s->w, V, (double)u_i[1], &dg->cdf_margin);
    if (tok < 0) {
      dg->fallback_p = 1;
      tok = draw_icdf(s->p, V, (double)u_i[1], &dg->cdf_margin);
    }
    dg->n_draws = 1;
    *acc_out = i;
    *next_out = tok;
    *st_out = st;
    return;
  }
  /* error exit */
  *acc_out = 0;
  *next_out = -1;
  *st_out = st;
}

void oracle_verify_rows(const void *target, const void *draft,
                        const int32_t *draft_tokens, const float *uniforms,
                        const int32_t *gamma_per_row, const oracle_params *prm,
                        int32_t row_begin, int32_t row_end,
                        int32_t *accepted_len, int32_t *next_token,
                        int32_t *row_status, float *p_draft, float *q_draft,
                        oracle_row_diag *diag) {
  scratch_t s;
  if (!scratch_alloc(&s, prm->V)) {
    scratch_free(&s);
    for (int32_t b = row_begin; b < row_end; ++b) {
      accepted_len[b] = 0;
      next_token[b] = -1;
      row_status[b] = -1;
    }
    return;
  }
  for (int32_t b = row_begin; b < row_end; ++b) {
    oracle_row_diag dg;
    verify_one_row(target, draft, draft_tokens, uniforms, gamma_per_row, prm, b,
                   &s, &accepted_len[b], &next_token[b], &row_status[b], p_draft,
                   q_draft, &dg);
    if (diag) diag[b] = dg;
  }
  scratch_free(&s);
}

void oracle_sample_rows(const void *logits, int32_t dtype, int64_t row_stride,
                        int32_t n_rows, int32_t V, double T, int32_t top_k,
                        double top_p, const float *u, int32_t *tokens,
                        double *cdf_margin, double *topp_margin) {
  scratch_t s;
  for (int32_t n = 0; n < n_rows; ++n) {
    if (cdf_margin) cdf_margin[n] = INFINITY;
    if (topp_margin) topp_margin[n] = INFINITY;
  }
  if (!scratch_alloc(&s, V)) {
    scratch_free(&s);
    for (int32_t n = 0; n < n_rows; ++n) tokens[n] = -1;
    return;
  }
  for (int32_t n = 0; n < n_rows; ++n) {
    const int32_t st = load_row(logits, dtype, (int64_t)n * row_stride, V, s.zt);
    if (st & ORACLE_ERROR_MASK) {
      tokens[n] = -1;
      continue;
    }
    if (T == 0.0) {
      tokens[n] = argmax_first(s.zt, V);
      continue;
    }
    double mg, cm;
    filtered_law(s.zt, V, T, top_k, top_p, s.p, s.e, s.srt, &mg);
    tokens[n] = draw_icdf(s.p, V, (double)u[n], &cm);
    if (cdf_margin) cdf_margin[n] = cm;
    if (topp_margin) topp_margin[n] = mg;
  }
  scratch_free(&s);
}
