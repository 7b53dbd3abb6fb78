// spec_law.cu -- the law of the speculative sampler's emitted token, for
// scoring ("CS3602_FINAL_SpeDec", section 2 困惑度测试 (PPL): with the
// acceptance rate beta = sum_x min(p(x), q(x)) and the residual law
// p'(x) = max(0, p(x) - q(x)) / sum_x' max(0, p(x') - q(x')), a token is
// emitted with probability min(p(x), q(x)) + (1 - beta) p'(x), which the
// page proves equals p(x)).  One CTA per row: a pass over both logit rows
// for the maxima and normalisers (an online softmax per thread, then a block
// merge), a second pass for beta and the residual normaliser, then the law
// at the row's token; 1024 threads per row and 16-byte loads when rows are
// aligned.  Unfiltered tempered laws only.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "spec_verify.h"
#include "sv_common.cuh"

namespace {

using sv::bf16_to_f32;
using sv::ex2_approx;

constexpr int LW_NT = 1024;  // a whole row per CTA; two CTAs fill an SM
constexpr int LW_NW = LW_NT / 32;

struct LP {
  const void *tgt, *drf;
  const int32_t *tok;
  float *pspec, *beta, *px, *qx;
  int64_t t_row, d_row;
  int32_t B, V;
  float c2;  // log2(e) / T
};

template <typename E>
__device__ __forceinline__ float lw_get(const E *g, int64_t j);
template <>
__device__ __forceinline__ float lw_get<float>(const float *g, int64_t j) { return g[j]; }
template <>
__device__ __forceinline__ float lw_get<uint16_t>(const uint16_t *g, int64_t j) {
  return bf16_to_f32(g[j]);
}

// Kahan step: s + x with compensation c.
__device__ __forceinline__ void kahan(float &s, float &c, float x) {
  const float t = __fsub_rn(x, c), u = __fadd_rn(s, t);
  c = __fsub_rn(__fsub_rn(u, s), t);
  s = u;
}

// Online softmax state: the maximum m (scaled by c2) and sum of 2^{y - m}.
struct On {
  float m, s, c;
  __device__ void init() {
    m = -INFINITY;
    s = 0.0f;
    c = 0.0f;
  }
  // several values at once: one rescale for their maximum
  template <int N>
  __device__ __forceinline__ void add_n(const float (&y)[N]) {
    float ym = y[0];
#pragma unroll
    for (int e = 1; e < N; ++e) ym = fmaxf(ym, y[e]);
    if (ym > m) {
      const float r = m == -INFINITY ? 0.0f : ex2_approx(__fsub_rn(m, ym));
      s = __fmul_rn(s, r);
      c = __fmul_rn(c, r);
      m = ym;
    }
#pragma unroll
    for (int e = 0; e < N; ++e)
      if (y[e] != -INFINITY) kahan(s, c, ex2_approx(__fsub_rn(y[e], m)));
  }
  __device__ __forceinline__ void add(float y) {
    if (y > m) {  // rescale what was summed so far
      const float r = m == -INFINITY ? 0.0f : ex2_approx(__fsub_rn(m, y));
      s = __fmul_rn(s, r);
      c = __fmul_rn(c, r);
      m = y;
    }
    if (y != -INFINITY) kahan(s, c, ex2_approx(__fsub_rn(y, m)));
    else if (y != y) kahan(s, c, y);  // NaN propagates
  }
};

// Merge of the block's online states: (M, Z) with Z = sum 2^{y - M}.
__device__ void on_merge(On o, float *sm, float &M, float &Z) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  float s = __fsub_rn(o.s, o.c);
  float m = o.m;
#pragma unroll
  for (int k = 16; k; k >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, k), os = __shfl_xor_sync(0xffffffffu, s, k);
    const float nm = fmaxf(m, om);
    // a thread with nothing summed adds 0; a NaN sum stays NaN (its maximum
    // may still be -inf when its only values were NaN)
    const float a = s == 0.0f ? 0.0f : __fmul_rn(s, ex2_approx(__fsub_rn(m, nm)));
    const float b = os == 0.0f ? 0.0f : __fmul_rn(os, ex2_approx(__fsub_rn(om, nm)));
    m = nm;
    s = __fadd_rn(a, b);
  }
  if (lane == 0) {
    sm[2 * wid] = m;
    sm[2 * wid + 1] = s;
  }
  __syncthreads();
  M = -INFINITY;
  for (int w = 0; w < LW_NW; ++w) M = fmaxf(M, sm[2 * w]);
  Z = 0.0f;
  for (int w = 0; w < LW_NW; ++w) {
    const float sw = sm[2 * w + 1];
    if (sw != 0.0f) Z = __fadd_rn(Z, __fmul_rn(sw, ex2_approx(__fsub_rn(sm[2 * w], M))));
  }
  __syncthreads();
}

__device__ float block_sum(float v, float *sm) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int k = 16; k; k >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, k));
  if (lane == 0) sm[wid] = v;
  __syncthreads();
  float s = 0.0f;
  for (int w = 0; w < LW_NW; ++w) s = __fadd_rn(s, sm[w]);
  __syncthreads();
  return s;
}

// 16-byte vectors of logits: 4 fp32 or 8 bf16.
template <typename E>
struct LVec;
template <>
struct LVec<float> {
  static constexpr int N = 4;
  __device__ static __forceinline__ void get(const uint4 &v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
};
template <>
struct LVec<uint16_t> {
  static constexpr int N = 8;
  __device__ static __forceinline__ void get(const uint4 &v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[2 * j] = __uint_as_float(w[j] << 16);
      f[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
  }
};

template <typename E, bool VEC>
__global__ void __launch_bounds__(LW_NT) law_kernel(const __grid_constant__ LP P) {
  __shared__ float sm[2 * LW_NW];
  const int r = blockIdx.x;
  const E *zt = static_cast<const E *>(P.tgt) + static_cast<int64_t>(r) * P.t_row;
  const E *zd = static_cast<const E *>(P.drf) + static_cast<int64_t>(r) * P.d_row;
  constexpr int N = LVec<E>::N;
  const int nv = VEC ? P.V / N : 0;  // whole vectors; the rest element by element
  // pass 1: maxima and normalisers of both tempered laws (base 2, scaled)
  On a, b;
  a.init();
  b.init();
#pragma unroll 4
  for (int v = threadIdx.x; v < nv; v += LW_NT) {
    float f[N], g[N];
    LVec<E>::get(__ldg(reinterpret_cast<const uint4 *>(zt) + v), f);
    LVec<E>::get(__ldg(reinterpret_cast<const uint4 *>(zd) + v), g);
#pragma unroll
    for (int e = 0; e < N; ++e) {
      f[e] = __fmul_rn(f[e], P.c2);
      g[e] = __fmul_rn(g[e], P.c2);
    }
    a.add_n(f);
    b.add_n(g);
  }
  for (int j = nv * N + threadIdx.x; j < P.V; j += LW_NT) {
    a.add(__fmul_rn(lw_get<E>(zt, j), P.c2));
    b.add(__fmul_rn(lw_get<E>(zd, j), P.c2));
  }
  float Mp, Zp, Mq, Zq;
  on_merge(a, sm, Mp, Zp);
  on_merge(b, sm, Mq, Zq);
  const float rp = __frcp_rn(Zp), rq = __frcp_rn(Zq);
  // pass 2: beta = sum min(p, q) and the residual normaliser sum max(0, p - q)
  float s1 = 0.0f, c1 = 0.0f, s2 = 0.0f, c2 = 0.0f;
#pragma unroll 4
  for (int v = threadIdx.x; v < nv; v += LW_NT) {
    float f[N], g[N];
    LVec<E>::get(__ldg(reinterpret_cast<const uint4 *>(zt) + v), f);
    LVec<E>::get(__ldg(reinterpret_cast<const uint4 *>(zd) + v), g);
#pragma unroll
    for (int e = 0; e < N; ++e) {
      const float p = __fmul_rn(ex2_approx(__fsub_rn(__fmul_rn(f[e], P.c2), Mp)), rp);
      const float q = __fmul_rn(ex2_approx(__fsub_rn(__fmul_rn(g[e], P.c2), Mq)), rq);
      kahan(s1, c1, fminf(p, q));
      kahan(s2, c2, fmaxf(__fsub_rn(p, q), 0.0f));
    }
  }
  for (int j = nv * N + threadIdx.x; j < P.V; j += LW_NT) {
    const float p = __fmul_rn(ex2_approx(__fsub_rn(__fmul_rn(lw_get<E>(zt, j), P.c2), Mp)), rp);
    const float q = __fmul_rn(ex2_approx(__fsub_rn(__fmul_rn(lw_get<E>(zd, j), P.c2), Mq)), rq);
    kahan(s1, c1, fminf(p, q));
    kahan(s2, c2, fmaxf(__fsub_rn(p, q), 0.0f));
  }
  const float beta = block_sum(__fsub_rn(s1, c1), sm);
  const float R = block_sum(__fsub_rn(s2, c2), sm);
  if (threadIdx.x == 0) {
    const int x = P.tok[r];
    float out = __int_as_float(0x7fc00000), px = out, qx = out;
    if (x >= 0 && x < P.V) {
      px = __fmul_rn(ex2_approx(__fsub_rn(__fmul_rn(lw_get<E>(zt, x), P.c2), Mp)), rp);
      qx = __fmul_rn(ex2_approx(__fsub_rn(__fmul_rn(lw_get<E>(zd, x), P.c2), Mq)), rq);
      const float res = fmaxf(__fsub_rn(px, qx), 0.0f);
      out = fminf(px, qx);
      if (R > 0.0f) out = __fadd_rn(out, __fdiv_rn(__fmul_rn(__fsub_rn(1.0f, beta), res), R));
      if (px != px || qx != qx || beta != beta || R != R) out = __int_as_float(0x7fc00000);
    }
    P.pspec[r] = out;
    if (P.beta) P.beta[r] = beta;
    if (P.px) P.px[r] = px;
    if (P.qx) P.qx[r] = qx;
  }
}

}  // namespace

extern "C" spec_status spec_law(const void *target_logits, const void *draft_logits,
                                const int32_t *tokens, const spec_params *params, float *p_spec,
                                float *beta, float *p_token, float *q_token, void *stream) {
  if (!params) return SPEC_ERR_INVALID_ARG;
  const spec_params &p = *params;
  if (p.B < 0 || p.V < 1 || p.V > (1 << 24)) return SPEC_ERR_INVALID_ARG;
  if (p.dtype != SPEC_F32 && p.dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (!std::isfinite(p.temperature) || p.temperature < 0.0f || !(p.top_p > 0.0f) ||
      p.target_row_stride < p.V || p.draft_row_stride < p.V)
    return SPEC_ERR_INVALID_ARG;
  if (p.temperature < 1e-30f) return SPEC_ERR_UNSUPPORTED;  // greedy: a point mass
  if ((p.top_k > 0 && p.top_k < p.V) || p.top_p < 1.0f) return SPEC_ERR_UNSUPPORTED;
  if (p.B == 0) return SPEC_OK;
  if (!target_logits || !draft_logits || !tokens || !p_spec) return SPEC_ERR_INVALID_ARG;
  LP L = {};
  L.tgt = target_logits;
  L.drf = draft_logits;
  L.tok = tokens;
  L.pspec = p_spec;
  L.beta = beta;
  L.px = p_token;
  L.qx = q_token;
  L.t_row = p.target_row_stride;
  L.d_row = p.draft_row_stride;
  L.B = p.B;
  L.V = p.V;
  L.c2 = static_cast<float>(1.4426950408889634 / static_cast<double>(p.temperature));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int es = p.dtype == SPEC_F32 ? 4 : 2;
  const bool vec = (reinterpret_cast<uintptr_t>(target_logits) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(draft_logits) & 15) == 0 &&
                   (p.target_row_stride * es) % 16 == 0 && (p.draft_row_stride * es) % 16 == 0;
  const unsigned grid = static_cast<unsigned>(p.B);
  if (p.dtype == SPEC_F32) {
    if (vec)
      law_kernel<float, true><<<grid, LW_NT, 0, s>>>(L);
    else
      law_kernel<float, false><<<grid, LW_NT, 0, s>>>(L);
  } else {
    if (vec)
      law_kernel<uint16_t, true><<<grid, LW_NT, 0, s>>>(L);
    else
      law_kernel<uint16_t, false><<<grid, LW_NT, 0, s>>>(L);
  }
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
