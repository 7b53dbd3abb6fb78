/*
 * spec_oracle.h -- plain, slow, fp64 CPU oracle for speculative-sampling
 * verification.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * CPU-baseline leg of the benchmark call it; the product path never does.
 * It shares no source, header, table or helper with the CUDA library.
 *
 * What it computes, and where each step comes from:
 *   - acceptance of draft token x with probability min(1, p(x)/q(x)), stop at
 *     the first rejection, resample that position from norm(max(0, p - q)),
 *     and draw one more token from p when every draft is accepted:
 *     "Text Generation via Speculative Sampling, KV Caching, and OpenVINO",
 *     section "Prepare speculative sampling" (steps 3 and 4), and the proof
 *     in "CS3602_FINAL_SpeDec", section "2. 困惑度测试(PPL)".
 *   - p and q are tempered softmaxes with top-k then top-p filtering:
 *     "CS3602_FINAL_SpeDec", sections "项目结构" (utils.py) and
 *     "问题分析与讨论" item 2.
 *
 * Parity status: greedy mode, the filters, the output law and the residual
 * identities are pinned by the CPU test-suite; intermediate probability
 * values beyond those identities are pinned only through them (the pages
 * print no worked numeric example).
 */
#ifndef SPEC_ORACLE_H
#define SPEC_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

/* Row status bits (identical meaning to the library's, written separately). */
enum {
  ORACLE_BAD_TOKEN   = 1 << 0, /* draft token outside [0, V) */
  ORACLE_BAD_LOGIT   = 1 << 1, /* NaN or +inf logit in an evaluated row */
  ORACLE_NO_FINITE   = 1 << 2, /* evaluated row: every logit is -inf or NaN */
  ORACLE_Q_ZERO      = 1 << 3, /* q(x) == 0 for an evaluated draft token (warning) */
  ORACLE_BAD_GAMMA   = 1 << 4, /* gamma_per_row[b] outside [0, gamma_max] */
  ORACLE_BAD_UNIFORM = 1 << 5  /* a used uniform is NaN or outside [0, 1) */
};
#define ORACLE_ERROR_MASK (ORACLE_BAD_TOKEN | ORACLE_BAD_LOGIT | ORACLE_NO_FINITE | \
                           ORACLE_BAD_GAMMA | ORACLE_BAD_UNIFORM)

typedef struct {
  int32_t B, gamma_max, V;
  int32_t dtype;          /* ORACLE_F32 or ORACLE_BF16 (raw uint16 bit patterns) */
  double temperature;     /* 0 => greedy */
  int32_t top_k;          /* <= 0 or >= V => off */
  double top_p;           /* >= 1 => off */
  int64_t t_pos_stride, t_row_stride;  /* elements */
  int64_t d_pos_stride, d_row_stride;
} oracle_params;

/* Per-row diagnostics used by the parity tests to classify disagreements. */
typedef struct {
  double accept_margin; /* min over evaluated tests of |u - min(1, p/q)|; +inf if none */
  double cdf_margin;    /* final draw: min(u - C_{k-1}/W, C_k/W - u); +inf if none */
  double topp_margin;   /* min over evaluated filtered rows of |M/Z - top_p| at j*, j*-1 */
  double residual_mass; /* W = sum max(0, p - q) at the rejected position, else 0 */
  int32_t n_tests;      /* acceptance tests evaluated */
  int32_t n_draws;      /* inverse-CDF draws made (0 or 1) */
  int32_t fallback_p;   /* 1 if the residual was empty and p was drawn instead */
  int32_t pad;
} oracle_row_diag;

/* Filtered tempered softmax of one row (T > 0).  prob[V] receives the law;
 * returns the status bits of the row; *topp_margin receives the top-p margin
 * (+inf when top-p is off).  Scratch is allocated internally. */
int32_t oracle_distribution(const void *z, int32_t dtype, int32_t V, double T,
                            int32_t top_k, double top_p, double *prob,
                            double *topp_margin);

/* Verify rows [row_begin, row_end).  Outputs are indexed by absolute row.
 * p_draft/q_draft ([B, gamma_max], may be NULL) receive p(x_i), q(x_i) for
 * evaluated positions and NaN elsewhere.  diag may be NULL. */
void oracle_verify_rows(const void *target, const void *draft,
                        const int32_t *draft_tokens, const float *uniforms,
                        const int32_t *gamma_per_row, const oracle_params *prm,
                        int32_t row_begin, int32_t row_end,
                        int32_t *accepted_len, int32_t *next_token,
                        int32_t *row_status, float *p_draft, float *q_draft,
                        oracle_row_diag *diag);

/* Draw one token per row from the filtered law of logits[n, :] (row stride
 * in elements) with uniform u[n]: the inverse CDF in vocabulary order, or the
 * argmax when T == 0.  Writes -1 for rows with an error.  Used to sample draft
 * tokens from q, as the speculative loop's first step does.  cdf_margin and
 * topp_margin (each [n], may be NULL) receive the distance of u from the
 * chosen CDF interval's ends (in units of the total weight) and the top-p
 * margin of the row's law; +inf where there is none (greedy, error rows,
 * top-p off), so that parity tests can tell draws that lie next to a
 * boundary from the rest. */
void oracle_sample_rows(const void *logits, int32_t dtype, int64_t row_stride,
                        int32_t n_rows, int32_t V, double T, int32_t top_k,
                        double top_p, const float *u, int32_t *tokens,
                        double *cdf_margin, double *topp_margin);

#ifdef __cplusplus
}
#endif
#endif
