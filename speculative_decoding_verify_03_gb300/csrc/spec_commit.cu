// spec_commit.cu -- the step after the verify: append the accepted draft
// tokens and the next token to each row's sequence, give the key/value
// cache length both models keep, and adapt the row's draft length with an
// additive-increase / multiplicative-decrease controller ("Prepare
// speculative sampling", steps 3-4; "CS3602_FINAL_SpeDec", 更多实现, the
// dynamic gamma).  One warp per row: lane j writes the j-th new token.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "spec_verify.h"

namespace {

constexpr int CM_NT = 256;           // threads per CTA
constexpr int CM_ROWS = CM_NT / 32;  // rows per CTA

struct CP {
  const int32_t *acc, *next, *tok, *gam;
  int32_t *seq, *seq_len, *kv_len, *gnext;
  int64_t stride;
  int32_t B, gm, cap;
  int32_t gmin, gmax, inc;
  float dec;
};

__global__ void __launch_bounds__(CM_NT) commit_kernel(const __grid_constant__ CP P) {
  const int lane = threadIdx.x & 31;
  const int b = static_cast<int>(blockIdx.x) * CM_ROWS + static_cast<int>(threadIdx.x >> 5);
  if (b >= P.B) return;
  const int g0 = P.gam ? P.gam[b] : P.gm;
  const int g = min(max(g0, 0), P.gm);
  const int a = P.acc[b], t = P.next[b];
  const int L = P.seq_len[b];
  const bool ok = g0 == g && a >= 0 && a <= g && t >= 0 && L >= 0;
  const int n = ok ? min(a + 1, max(0, P.cap - L)) : 0;  // tokens written
  int32_t *row = P.seq + static_cast<int64_t>(b) * P.stride + (ok ? L : 0);
  const int32_t *drafts = P.tok + static_cast<int64_t>(b) * P.gm;
  for (int j = lane; j < n; j += 32) row[j] = j < a ? drafts[j] : t;
  if (lane == 0) {
    const int nl = L + n;
    P.seq_len[b] = ok ? nl : L;
    if (P.kv_len) P.kv_len[b] = ok ? min(L + a, nl) : L;
    if (P.gnext) {
      const int up = g + P.inc;
      const int down = static_cast<int>(floorf(__fmul_rn(static_cast<float>(g), P.dec)));
      P.gnext[b] = min(max(ok && a == g ? up : down, P.gmin), P.gmax);
    }
  }
}

}  // namespace

extern "C" spec_status spec_commit(int32_t B, int32_t gamma_max, const int32_t *accepted_len,
                                   const int32_t *next_token, const int32_t *draft_tokens,
                                   const int32_t *gamma_per_row, int32_t *seq,
                                   int64_t seq_row_stride, int32_t seq_capacity,
                                   int32_t *seq_len, int32_t *kv_len, int32_t *gamma_next,
                                   const spec_aimd *aimd, void *stream) {
  if (B < 0 || gamma_max < 0 || seq_capacity < 0 || seq_row_stride < seq_capacity)
    return SPEC_ERR_INVALID_ARG;
  if (B == 0) return SPEC_OK;
  if (!accepted_len || !next_token || !seq || !seq_len) return SPEC_ERR_INVALID_ARG;
  if (gamma_max > 0 && !draft_tokens) return SPEC_ERR_INVALID_ARG;
  CP P = {};
  if (gamma_next) {
    if (!aimd || aimd->gamma_min < 0 || aimd->gamma_max < aimd->gamma_min || aimd->increase < 0 ||
        !(aimd->decrease >= 0.0f && aimd->decrease <= 1.0f))
      return SPEC_ERR_INVALID_ARG;
    P.gmin = aimd->gamma_min;
    P.gmax = aimd->gamma_max;
    P.inc = aimd->increase;
    P.dec = aimd->decrease;
  }
  P.acc = accepted_len;
  P.next = next_token;
  P.tok = draft_tokens;
  P.gam = gamma_per_row;
  P.seq = seq;
  P.seq_len = seq_len;
  P.kv_len = kv_len;
  P.gnext = gamma_next;
  P.stride = seq_row_stride;
  P.B = B;
  P.gm = gamma_max;
  P.cap = seq_capacity;
  const unsigned grid = static_cast<unsigned>((static_cast<int64_t>(B) + CM_ROWS - 1) / CM_ROWS);
  commit_kernel<<<grid, CM_NT, 0, static_cast<cudaStream_t>(stream)>>>(P);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
