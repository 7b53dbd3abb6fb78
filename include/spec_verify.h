/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) speculative-sampling
 * verification library (libspecverify.so).
 *
 * The operation is the verify step of speculative sampling: given the target
 * model's logits for gamma+1 positions and the draft model's logits and
 * tokens for gamma positions, decide how many draft tokens to accept and
 * which token to emit next, so that the emitted tokens follow the target
 * law exactly.  Sources:
 *   - "Text Generation via Speculative Sampling, KV Caching, and OpenVINO",
 *     section "Prepare speculative sampling": step 3 (accept draft tokens by
 *     comparing a uniform with the target/draft probability ratio, resample
 *     the first rejected position) and step 4 (one extra token when every
 *     draft is accepted);
 *   - "CS3602_FINAL_SpeDec", section "2. 困惑度测试(PPL)": acceptance
 *     probability min(1, p(x)/q(x)), residual law norm(max(0, p - q)) with
 *     normaliser 1 - beta, and the proof that the output law is p;
 *   - "CS3602_FINAL_SpeDec", sections "项目结构" and "问题分析与讨论" item 2:
 *     p and q are tempered softmaxes with top-k / top-p filtering.
 *
 * Conventions.  p = target law, q = draft law.  All tensor pointers are
 * device pointers owned by the caller; the library never allocates or frees
 * device memory on the call path.  Calls are asynchronous on the given CUDA
 * stream (a cudaStream_t passed as void*; NULL = legacy default stream);
 * only argument validation is synchronous, through the return code.
 * Per-row input errors never fault the device: they set row status bits and
 * give the row accepted_len = 0, next_token = -1.  The same inputs always
 * give bitwise identical outputs.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SPEC_OK = 0,
  SPEC_ERR_INVALID_ARG = 1, /* a parameter or pointer is invalid (nothing launched) */
  SPEC_ERR_UNSUPPORTED = 2, /* valid but not supported by this build/device */
  SPEC_ERR_WORKSPACE = 3,   /* workspace too small or misaligned */
  SPEC_ERR_CUDA = 4         /* a CUDA runtime call failed (launch or attribute) */
} spec_status;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

/* Row status bits (spec_debug.row_status). */
#define SPEC_ROW_BAD_TOKEN   (1 << 0) /* draft token outside [0, V) */
#define SPEC_ROW_BAD_LOGIT   (1 << 1) /* NaN or +inf logit in an evaluated row */
#define SPEC_ROW_NO_FINITE   (1 << 2) /* an evaluated row: every logit is -inf or NaN */
#define SPEC_ROW_Q_ZERO      (1 << 3) /* q(x) == 0 for a draft token (warning only:
                                         accepted iff p(x) > 0, the limit of min(1,p/q)) */
#define SPEC_ROW_BAD_GAMMA   (1 << 4) /* gamma_per_row[b] outside [0, gamma_max] */
#define SPEC_ROW_BAD_UNIFORM (1 << 5) /* a used uniform is NaN or outside [0, 1) */
#define SPEC_ROW_WAIT_TIMEOUT (1 << 6) /* a device-side wait for staged data gave up
                                          (hardware fault); the row's results are invalid */
#define SPEC_ROW_ERROR_MASK  (SPEC_ROW_BAD_TOKEN | SPEC_ROW_BAD_LOGIT | SPEC_ROW_NO_FINITE | \
                              SPEC_ROW_BAD_GAMMA | SPEC_ROW_BAD_UNIFORM | SPEC_ROW_WAIT_TIMEOUT)

/* spec_params.flags: always use the cluster-per-row kernel, even where the
   strip-parallel or the warp-per-row kernel would run (for comparisons and
   tests; the results are the same). */
#define SPEC_FLAG_CLUSTER_KERNEL 1

typedef struct {
  int32_t B;         /* rows (sequences); 0 => no-op */
  int32_t gamma_max; /* draft positions per row (>= 0) */
  int32_t V;         /* vocabulary size (>= 1, <= 2^24) */
  int32_t dtype;     /* spec_dtype of both logit tensors (bf16 = raw bfloat16) */
  float temperature; /* 0 => greedy (accept iff argmax p == draft token; the
                        next token is the argmax; draft logits are not read).
                        > 0 => sampling; must be >= 1e-30 and finite */
  float top_p;       /* nucleus mass in (0, 1]; >= 1 => off */
  int32_t top_k;     /* keep the top_k largest logits (ties kept); <= 0 or >= V => off */
  int32_t flags;     /* SPEC_FLAG_* bits; other bits must be 0 */
  /* Strides in elements.  Element (b, i, v) of the target logits is at
     target_logits[b*target_row_stride + i*target_pos_stride + v], of the draft
     logits at draft_logits[b*draft_row_stride + i*draft_pos_stride + v]. */
  int64_t target_pos_stride, target_row_stride;
  int64_t draft_pos_stride, draft_row_stride;
  /* Optional device array [B] of per-row draft lengths gamma_b in
     [0, gamma_max]; NULL => every row uses gamma_max.  Row b reads target
     positions 0..gamma_b and draft positions 0..gamma_b-1 only. */
  const int32_t *gamma_per_row;
  /* Tuning (0 = automatic): CTAs per row cluster (1, 2, 4 or 8) and the
     capacity of the on-chip candidate list used by top-k / top-p. */
  int32_t cluster_size;
  int32_t list_capacity;     /* 0..8192 */
} spec_params;

/* Optional device outputs (any member may be NULL). */
typedef struct {
  float *p_draft;       /* [B, gamma_max]: p(x_i) after filtering, for evaluated
                           positions; NaN elsewhere.  fp32. */
  float *q_draft;       /* [B, gamma_max]: q(x_i), same convention. */
  float *residual_mass; /* [B]: sum_v max(0, p - q) at the rejected position, else 0 */
  int32_t *row_status;  /* [B]: SPEC_ROW_* bits */
} spec_debug;

/*
 * Bytes of workspace a call with these parameters can use: the diagnostics
 * block that spec_verify accumulates into (counters of slow paths taken; see
 * spec_read_diagnostics), plus, where it applies (greedy, top-k and top-p
 * problems beyond the warp-per-row kernel's small vocabularies), the
 * strip-parallel kernel's per-position exchange area.  With less, or none
 * (0 bytes is valid), the call still runs, on the cluster-per-row kernel.
 */
size_t spec_verify_workspace_size(const spec_params *params);

/*
 * The verify step.
 *   target_logits  device, [B, gamma_max+1, V] with the strides above
 *                  (float32 or bfloat16).  Target position i scores draft
 *                  slot i; position gamma_b is the bonus position.
 *   draft_logits   device, [B, gamma_max, V] (same dtype).  Not read when
 *                  temperature == 0.  May be NULL when gamma_max == 0.
 *   draft_tokens   device int32 [B, gamma_max], contiguous.
 *   uniforms       device float32 [B, gamma_max+1, 2], contiguous:
 *                  [b,i,0] is the acceptance uniform of slot i, [b,i,1] the
 *                  uniform of a draw at position i (residual or bonus).
 *                  Values must lie in [0, 1).  Not read when greedy.
 *   accepted_len   device int32 [B]: number of accepted draft tokens.
 *   next_token     device int32 [B]: the resampled token at the first
 *                  rejection, or the bonus token when all were accepted.
 *   debug          optional (NULL) host struct of optional device outputs.
 *   workspace      optional device block of workspace_bytes (>= the size
 *                  above, 16-byte aligned) for diagnostics counters; NULL ok.
 * Returns SPEC_OK after enqueueing; errors are reported before any launch.
 * Positions after the first rejection are not read (early exit).
 */
spec_status spec_verify(const void *target_logits, const void *draft_logits,
                        const int32_t *draft_tokens, const float *uniforms,
                        const spec_params *params, int32_t *accepted_len,
                        int32_t *next_token, const spec_debug *debug,
                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * Draw one token per row of logits[n, V] (row stride in elements) from its
 * filtered tempered law (the argmax when temperature == 0), with uniform
 * u[n] in [0, 1): the inverse CDF in vocabulary order.  This is the draft
 * model's per-step sampler of "Prepare speculative sampling" step 1, with
 * the same filtering as spec_verify.  params->B is n, params->gamma_max must
 * be 0, params->target_row_stride is the row stride; the draft and
 * gamma_per_row fields are ignored.  tokens[n] (device int32) receives the
 * draws, -1 for rows with an error (row_status, optional, the bits).
 */
spec_status spec_sample(const void *logits, const float *u, const spec_params *params,
                        int32_t *tokens, int32_t *row_status, void *stream);

/*
 * spec_sample with a workspace (16-byte aligned, at least
 * spec_sample_workspace_size(params) bytes for the fastest kernels): filtered
 * (and greedy) draws then run on the strip-parallel kernel of spec_verify,
 * and vocabularies up to 1024 on its CTA-per-row kernel, exactly as
 * spec_verify draws a bonus token (a row is a sequence with no drafts).
 * Arguments, results and errors are those of spec_sample; with less
 * workspace, or none, the call runs as spec_sample.
 */
size_t spec_sample_workspace_size(const spec_params *params);

spec_status spec_sample_ws(const void *logits, const float *u, const spec_params *params,
                           int32_t *tokens, int32_t *row_status, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * spec_verify without a caller workspace and without any allocation: the
 * library's own fixed 64 MiB device block (a static device array) serves as
 * the workspace.  The pages describe no counterpart; it is a convenience of
 * this library for callers that cannot provide device memory.  Arguments
 * and results are those of spec_verify.  A problem whose workspace
 * (spec_verify_workspace_size) exceeds the block is rejected with
 * SPEC_ERR_WORKSPACE before any launch.
 *
 * The block is part of the library's device code: every device on which
 * the library's module is loaded holds the 64 MiB until the process exits
 * (or the context is destroyed), whether or not this entry point is called.
 * The first call on a device looks up the block's address with
 * cudaGetSymbolAddress (with that device current) and caches it for the
 * process; make that first call before any stream capture.  The cached
 * address is not valid after cudaDeviceReset or another teardown of the
 * device's primary context: do not call this entry point again in such a
 * process.  The block is shared by every call in the process on that
 * device and keeps the last call's contents (the call clears what must
 * start at zero): calls must not overlap in time (issue them on one stream,
 * or order the streams); overlapping calls race on it.
 */
spec_status spec_verify_noalloc(const void *target_logits, const void *draft_logits,
                                const int32_t *draft_tokens, const float *uniforms,
                                const spec_params *params, int32_t *accepted_len,
                                int32_t *next_token, const spec_debug *debug, void *stream);

/*
 * The step after spec_verify: append each row's accepted draft tokens and
 * its next token to the row's token sequence, give the key/value cache
 * length both models keep, and adapt the row's draft length.  The pages
 * ("Prepare speculative sampling", steps 3-4: the accepted tokens and the
 * resampled or bonus token are concatenated to the sequence;
 * "CS3602_FINAL_SpeDec", 更多实现: a dynamic gamma, additive increase /
 * multiplicative decrease as in TCP's AIMD, shrinking fast after poor
 * acceptance) leave the controller's constants open; they are parameters.
 *
 * Per row b with L = seq_len[b] on entry, a = accepted_len[b],
 * t = next_token[b], g = gamma_per_row[b] (gamma_max when NULL):
 *   - a valid row (0 <= g <= gamma_max, 0 <= a <= g, t >= 0, L >= 0) writes
 *     draft_tokens[b, 0..a) and then t at seq[b * seq_row_stride + L ...],
 *     dropping what would pass seq_capacity:
 *     seq_len[b] = L + min(a + 1, max(0, seq_capacity - L));
 *     kv_len[b] = min(L + a, seq_len[b]): the context plus the accepted
 *     drafts (the new token's entry comes with the next forward pass);
 *   - an invalid row (an error row of spec_verify: next_token -1) appends
 *     nothing: seq_len[b] = L, kv_len[b] = L;
 *   - gamma_next[b] = g + aimd->increase when the row accepted every draft
 *     (a == g), else floor(g * aimd->decrease) (the product in single
 *     precision), clamped to [aimd->gamma_min, aimd->gamma_max]; an invalid
 *     row counts as a rejection, with g clamped to [0, gamma_max].
 * accepted_len, next_token [B] and draft_tokens [B, gamma_max] (contiguous)
 * are device int32 (spec_verify's outputs and inputs); seq, seq_len (in/out)
 * and the optional kv_len, gamma_next [B] are device int32.  aimd is a host
 * struct, required when gamma_next is given: 0 <= gamma_min <= gamma_max,
 * increase >= 0, 0 <= decrease <= 1.  Asynchronous on stream; argument
 * errors are returned before any launch; B == 0 is a no-op.
 */
typedef struct {
  int32_t gamma_min, gamma_max;
  int32_t increase;
  float decrease;
} spec_aimd;

spec_status spec_commit(int32_t B, int32_t gamma_max, const int32_t *accepted_len,
                        const int32_t *next_token, const int32_t *draft_tokens,
                        const int32_t *gamma_per_row, int32_t *seq, int64_t seq_row_stride,
                        int32_t seq_capacity, int32_t *seq_len, int32_t *kv_len,
                        int32_t *gamma_next, const spec_aimd *aimd, void *stream);

/*
 * The law of the token the speculative sampler emits, for scoring (e.g.
 * perplexity): "CS3602_FINAL_SpeDec", section 2 困惑度测试 (PPL).  For row
 * r (one position: target logits target_logits[r * target_row_stride + v],
 * draft logits draft_logits[r * draft_row_stride + v], v < V) with the
 * tempered laws p and q, the acceptance rate beta = sum_v min(p(v), q(v))
 * and R = sum_v max(0, p(v) - q(v)), the emitted token is x with probability
 *   p_spec(x) = min(p(x), q(x)) + (1 - beta) max(0, p(x) - q(x)) / R
 * (min(p(x), q(x)) when R = 0), which the page proves equals p(x).  x =
 * tokens[r].  Outputs (device float [B]): p_spec, and optionally beta and
 * p(x), q(x).  Single precision with compensated sums (about 1e-6
 * relative).  params: B, V, dtype, temperature (> 0), top_k, top_p and the
 * two row strides; p and q are filtered as in spec_verify (top-k keeping
 * every logit >= the k-th largest, then top-p keeping the smallest leading
 * set of equal-logit groups whose mass reaches top_p; a top-p crossing
 * within about 1e-6 of the mass may be placed either way); temperature 0 is
 * a point mass (SPEC_ERR_UNSUPPORTED); gamma_max and the other fields are
 * ignored.  A token outside [0, V), a row with NaN / +inf / no finite logit,
 * and (top-p) a row whose logits down to a depth bin past the crossing
 * number more than 4096 give NaN.  Asynchronous on stream.
 */
spec_status spec_law(const void *target_logits, const void *draft_logits, const int32_t *tokens,
                     const spec_params *params, float *p_spec, float *beta, float *p_token,
                     float *q_token, void *stream);

/*
 * spec_law with a workspace: filtered laws (top-k and / or top-p) run on the
 * strip-parallel kernel of spec_verify (each row's two logit rows cut into
 * pieces, read once; the kept sets selected exactly, as spec_verify selects
 * them), every row evaluated whatever its top-p region.  beta = sum min(p, q)
 * and R = sum max(0, p - q) are summed over p's kept set in single precision
 * (beta = 1 - R for a row whose candidate list overflowed: p sums to one).
 * Arguments, outputs and errors are those of spec_law; a call whose laws are
 * unfiltered, or whose workspace is NULL, misaligned (16 bytes) or smaller
 * than spec_law_workspace_size(params), runs spec_law itself.
 * params->cluster_size and list_capacity tune the pieces as for spec_verify.
 */
size_t spec_law_workspace_size(const spec_params *params);

spec_status spec_law_ws(const void *target_logits, const void *draft_logits,
                        const int32_t *tokens, const spec_params *params, float *p_spec,
                        float *beta, float *p_token, float *q_token, void *workspace,
                        size_t workspace_bytes, void *stream);

/*
 * Verification of a multi-stage draft cascade ("CS3602_FINAL_SpeDec",
 * 更多实现: several draft models in a chain, each drafting for the next
 * larger one, as the levels of a cache hierarchy serve each other).  The
 * page gives no algorithm; this is the plainest reading that keeps the
 * output law equal to the target's, with the verify step of spec_verify
 * (the same kernels) at every stage.
 *
 * Levels l = 0 .. L (n_levels = L + 1 >= 2): level 0 is the target, level L
 * the smallest draft model, which drew draft_tokens [B, gamma_max] (device
 * int32, contiguous) from its laws.  level_logits is a HOST array of
 * n_levels device pointers:
 *   level_logits[l], l < L   [B, gamma_max+1, V], strides target_pos_stride
 *                            and target_row_stride (shared by these levels):
 *                            one forward pass over the same drafts;
 *   level_logits[L]          [B, gamma_max, V], strides draft_pos_stride and
 *                            draft_row_stride (NULL allowed when greedy).
 * Stage k = 0 .. L-1 is one verify step of the tokens presented to it,
 * with draft level L-k, target level L-k-1 and the uniforms
 * uniforms[k] (device float32 [L, B, gamma_max+1, 2], contiguous; NULL when
 * greedy).  Stage 0 is presented the drafts (gamma_b of them, from
 * params->gamma_per_row or gamma_max).  After a stage, per row:
 *   - a rejection at slot a < n: the resampled token takes slot a and the
 *     next stage is presented the n = a + 1 tokens 0..a;
 *   - all n accepted: the bonus token is kept only at the last stage and
 *     only if no stage resampled (the tokens are then the original drafts);
 *     otherwise it is dropped and the next stage sees the same n tokens.
 * Outputs (device int32): out_tokens [B, gamma_max+1] (-1 after the
 * row's output), out_len [B] (1 .. gamma_b+1; 0 for a row in error);
 * optional stage_accepted [L, B] (each stage's accepted count; -1 for the
 * stages after the row's error) and row_status [B] (the stages' SPEC_ROW_*
 * bits, or-ed).  A row whose stage reports an error bit stops there.
 *
 * params: as for spec_verify (temperature, top_k, top_p and flags apply to
 * every stage).  workspace: required, 256-byte aligned, at least
 * spec_cascade_workspace_size(params, n_levels) bytes for the fastest
 * kernels (the cascade's own state first; with less room for the verify
 * step's part, the stages run on the cluster-per-row kernel).  Every
 * stage's arguments are checked before the first launch; asynchronous on
 * stream; B == 0 is a no-op.
 */
size_t spec_cascade_workspace_size(const spec_params *params, int32_t n_levels);

spec_status spec_cascade_verify(const void *const *level_logits, int32_t n_levels,
                                const int32_t *draft_tokens, const float *uniforms,
                                const spec_params *params, int32_t *out_tokens, int32_t *out_len,
                                int32_t *stage_accepted, int32_t *row_status, void *workspace,
                                size_t workspace_bytes, void *stream);

/* Human-readable name of a status code (static storage). */
const char *spec_status_string(spec_status status);

/* Copy the diagnostics block of a workspace to host counters[n] (synchronous
 * on the stream).  Counters: [0] positions where a candidate list overflowed
 * or missed the nucleus (exact slice-wide selection used instead), [1] draws
 * redone in float-float after the certified single-precision draw was
 * uncertain, [2] rows whose device-side waits timed out, [3] positions
 * where, under top-p without top-k, a tensor's candidate list was extended
 * from, or rebuilt by, a rescan of its logit row (counted once per stage). */
spec_status spec_read_diagnostics(const void *workspace, uint32_t *counters, int n,
                                  void *stream);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_VERIFY_H */
