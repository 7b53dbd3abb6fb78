// spec_cascade.cu -- verification of a multi-stage draft cascade
// ("CS3602_FINAL_SpeDec", 更多实现: several draft models in a chain, each
// one drafting for the next larger one, as the levels of a cache hierarchy
// serve each other).
//
// Level 0 is the target, level L the smallest draft model; every level but
// the smallest scored the smallest model's drafts in one forward pass.
// Stage k = 0 .. L-1 verifies the tokens presented to it (draft laws of
// level L-k, target laws of level L-k-1) with the verify step itself, i.e.
// the same kernels spec_verify runs.  Between stages one thread per row:
//   - a rejection at slot a < n puts the resampled token at slot a and cuts
//     the presented count to a + 1 (the later slots' laws were computed after
//     the original drafts, which no longer stand);
//   - when all n tokens are accepted, the bonus draw is kept only at the last
//     stage and only if no stage resampled; else it is discarded.
// Rows in error stop: later stages see gamma_b = -1 (rejected by the verify
// step without reading a logit) and the row's output is empty.
#include <cuda_runtime.h>

#include <cstdint>

#include "spec_verify.h"
#include "sv_verify.h"

namespace {

constexpr int CK_NT = 256;
constexpr int32_t kFlagError = 1;
constexpr int32_t kFlagResampled = 2;
constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// The cascade's own state at the start of the workspace (each array on a
// 256-byte boundary), then the verify step's workspace.
struct State {
  int32_t *tok;    // [B, gamma_max] presented tokens
  int32_t *n;      // [B] presented count (the stage's gamma_b); -1 after an error
  int32_t *acc;    // [B] the stage's accepted_len (when the caller keeps none)
  int32_t *next;   // [B] the stage's next_token
  int32_t *st;     // [B] the stage's row status
  int32_t *flags;  // [B] kFlag* bits
};

size_t state_bytes(int64_t B, int64_t gm) {
  return align_up(static_cast<size_t>(B * gm) * 4) + 5 * align_up(static_cast<size_t>(B) * 4);
}

State carve(void *ws, int64_t B, int64_t gm) {
  char *p = static_cast<char *>(ws);
  State s;
  s.tok = reinterpret_cast<int32_t *>(p);
  p += align_up(static_cast<size_t>(B * gm) * 4);
  int32_t **rows[5] = {&s.n, &s.acc, &s.next, &s.st, &s.flags};
  for (int32_t **r : rows) {
    *r = reinterpret_cast<int32_t *>(p);
    p += align_up(static_cast<size_t>(B) * 4);
  }
  return s;
}

__global__ void __launch_bounds__(CK_NT)
    cascade_init_kernel(const int32_t *draft_tokens, const int32_t *gamma_per_row, State S,
                        int32_t *row_status, int B, int gm) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * CK_NT + threadIdx.x;
  if (i < static_cast<int64_t>(B) * gm) S.tok[i] = draft_tokens[i];
  if (i < B) {
    S.n[i] = gamma_per_row ? gamma_per_row[i] : gm;
    S.flags[i] = 0;
    if (row_status) row_status[i] = 0;
  }
}

// After stage k: fold the stage's results into the row's state; the last
// stage also writes the output (out_tokens [B, gm+1], out_len [B]).
__global__ void __launch_bounds__(CK_NT)
    cascade_update_kernel(State S, const int32_t *acc, int32_t *stage_acc, int32_t *row_status,
                          int32_t *out_tokens, int32_t *out_len, int B, int gm, int last) {
  const int b = static_cast<int>(blockIdx.x) * CK_NT + static_cast<int>(threadIdx.x);
  if (b >= B) return;
  int32_t f = S.flags[b];
  int32_t n = S.n[b];
  int32_t bonus = -1;
  if (f & kFlagError) {
    if (stage_acc) stage_acc[b] = -1;
  } else {
    const int32_t st = S.st[b];
    if (row_status) row_status[b] |= st;
    const int32_t a = acc[b], t = S.next[b];
    // a stage result without an error bit has 0 <= a <= n <= gm and t >= 0
    if ((st & SPEC_ROW_ERROR_MASK) || a < 0 || a > n || n > gm || t < 0) {
      f |= kFlagError;
    } else if (a < n) {
      S.tok[static_cast<int64_t>(b) * gm + a] = t;
      n = a + 1;
      f |= kFlagResampled;
    } else if (last && !(f & kFlagResampled)) {
      bonus = t;
    }
    if (f & kFlagError) n = -1;
    S.n[b] = n;
    S.flags[b] = f;
  }
  if (!last) return;
  const bool err = (f & kFlagError) != 0;
  const int32_t len = err ? 0 : n + (bonus >= 0 ? 1 : 0);
  int32_t *o = out_tokens + static_cast<int64_t>(b) * (gm + 1);
  const int32_t *tk = S.tok + static_cast<int64_t>(b) * gm;
  for (int j = 0; j <= gm; ++j) o[j] = j < len ? (j < n ? tk[j] : bonus) : -1;
  out_len[b] = len;
}

// The verify parameters of stage k: target = level L-k-1, draft = level L-k
// (the smallest level keeps the caller's draft strides; the others share
// the target strides), gamma_b = the presented counts.
spec_params stage_params(const spec_params &p, int k, const int32_t *n) {
  spec_params s = p;
  if (k > 0) {
    s.draft_pos_stride = p.target_pos_stride;
    s.draft_row_stride = p.target_row_stride;
  }
  s.gamma_per_row = n;
  return s;
}

}  // namespace

extern "C" {

size_t spec_cascade_workspace_size(const spec_params *params, int32_t n_levels) {
  if (!params || n_levels < 2 || params->B < 0 || params->gamma_max < 0) return 0;
  size_t v = spec_verify_workspace_size(params);
  spec_params s = stage_params(*params, 1, nullptr);
  const size_t v1 = spec_verify_workspace_size(&s);
  if (v1 > v) v = v1;
  return state_bytes(params->B, params->gamma_max) + v;
}

spec_status spec_cascade_verify(const void *const *level_logits, int32_t n_levels,
                                const int32_t *draft_tokens, const float *uniforms,
                                const spec_params *params, int32_t *out_tokens, int32_t *out_len,
                                int32_t *stage_accepted, int32_t *row_status, void *workspace,
                                size_t workspace_bytes, void *stream) {
  if (!params || !level_logits || n_levels < 2) return SPEC_ERR_INVALID_ARG;
  const spec_params &p = *params;
  if (p.B < 0 || p.gamma_max < 0) return SPEC_ERR_INVALID_ARG;
  if (p.B == 0) return SPEC_OK;
  if (!out_tokens || !out_len || (p.gamma_max > 0 && !draft_tokens)) return SPEC_ERR_INVALID_ARG;
  const int L = n_levels - 1;
  for (int l = 0; l < L; ++l)
    if (!level_logits[l]) return SPEC_ERR_INVALID_ARG;
  const int64_t B = p.B, gm = p.gamma_max;
  const size_t own = state_bytes(B, gm);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0 ||
      workspace_bytes < own)
    return SPEC_ERR_WORKSPACE;
  const State S = carve(workspace, B, gm);
  void *vws = workspace_bytes > own ? static_cast<char *>(workspace) + own : nullptr;
  const size_t vws_bytes = workspace_bytes - own;
  // every stage's arguments are checked before the first launch
  const int64_t ustage = B * (gm + 1) * 2;
  for (int k = 0; k < L; ++k) {
    const spec_params s = stage_params(p, k, S.n);
    const spec_status c = sv::check_verify_args(
        level_logits[L - k - 1], level_logits[L - k], S.tok, uniforms ? uniforms + k * ustage : nullptr,
        &s, stage_accepted ? stage_accepted + k * B : S.acc, S.next, vws, vws ? vws_bytes : 0,
        false);
    if (c != SPEC_OK) return c;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t init_n = B * gm > B ? B * gm : B;
  cascade_init_kernel<<<static_cast<unsigned>((init_n + CK_NT - 1) / CK_NT), CK_NT, 0, st>>>(
      draft_tokens, p.gamma_per_row, S, row_status, p.B, p.gamma_max);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  const unsigned rows_grid = static_cast<unsigned>((B + CK_NT - 1) / CK_NT);
  for (int k = 0; k < L; ++k) {
    const spec_params s = stage_params(p, k, S.n);
    int32_t *acc = stage_accepted ? stage_accepted + k * B : S.acc;
    spec_debug dbg = {nullptr, nullptr, nullptr, S.st};
    const spec_status r = spec_verify(level_logits[L - k - 1], level_logits[L - k], S.tok,
                                      uniforms ? uniforms + k * ustage : nullptr, &s, acc, S.next,
                                      &dbg, vws, vws ? vws_bytes : 0, stream);
    if (r != SPEC_OK) return r;
    cascade_update_kernel<<<rows_grid, CK_NT, 0, st>>>(S, acc, stage_accepted ? acc : nullptr,
                                                       row_status, out_tokens, out_len, p.B,
                                                       p.gamma_max, k == L - 1 ? 1 : 0);
    if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  }
  return SPEC_OK;
}

}  // extern "C"
