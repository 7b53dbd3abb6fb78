// spec_law.cu -- the law of the speculative sampler's emitted token, for
// scoring ("CS3602_FINAL_SpeDec", section 2 困惑度测试 (PPL): with the
// acceptance rate beta = sum_x min(p(x), q(x)) and the residual law
// p'(x) = max(0, p(x) - q(x)) / sum_x' max(0, p(x') - q(x')), a token is
// emitted with probability min(p(x), q(x)) + (1 - beta) p'(x), which the
// page proves equals p(x)).  One CTA per row: a pass over both logit rows
// for the maxima and normalisers (an online softmax per thread, then a block
// merge), a second pass for beta and the residual normaliser, then the law
// at the row's token; 1024 threads per row and 16-byte loads when rows are
// aligned.  Filtered laws (top-k, top-p) run law_filt_kernel below.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "spec_verify.h"
#include "sv_common.cuh"
#include "sv_verify.h"

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

// ------------------------------------------------------------ filtered laws
// With top-k and / or top-p, p and q are the filtered tempered laws of
// spec_verify (temperature, then top-k keeping every logit >= the k-th
// largest, then top-p keeping the smallest leading set of equal-logit
// groups whose mass reaches top_p of the survivors'; "CS3602_FINAL_SpeDec",
// 项目结构 (utils.py) and 问题分析与讨论 item 2).  Per tensor: the k-th largest
// logit by a radix selection over order-preserving keys (four rounds of
// 256-bin histograms); the top-p region by a histogram of the survivors in
// depth bins (1/16 of a log2 unit below the maximum, the bins' masses in
// scaled integers) ending at a bin where the survivors' mass passes top_p
// by a margin; that region (at most LF_CAP logits) is sorted in shared
// memory and walked from the top for the first group reaching top_p of the
// survivors' mass (float-float prefix sums of single-precision weights: a
// crossing within about 1e-6 of the survivors' mass may be placed either
// way).  A row whose region exceeds LF_CAP logits gets NaN outputs.
constexpr int LF_CAP = 4096;  // sorted top-p region per tensor (entries)

struct LFShared {
  unsigned long long reg[2][LF_CAP];  // keys (value descending, index ascending)
  uint32_t hist[2][256];
  uint32_t mass[2][256];  // per depth bin: sum of round(2^12 w 2^{b/16}) (w 2^{b/16} in (0.95, 1])
  float f[2][LW_NW][2];
  int   sc[2][8];
  float fc[2][8];
};

__device__ __forceinline__ uint32_t lf_fkey(float x) {
  const uint32_t u = __float_as_uint(__fadd_rn(x, 0.0f));
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float lf_unkey(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// One value of either tensor (t: 0 target, 1 draft) at index j, scaled by c2.
template <typename E>
__device__ __forceinline__ float lf_y(const E *z, int64_t j, float c2) {
  return __fmul_rn(lw_get<E>(z, j), c2);
}

template <typename E>
__global__ void __launch_bounds__(LW_NT) law_filt_kernel(const __grid_constant__ LP P, int top_k,
                                                        float top_p) {
  extern __shared__ __align__(16) unsigned char lf_raw[];
  LFShared &sh = *reinterpret_cast<LFShared *>(lf_raw);
  __shared__ float sm[2 * LW_NW];
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const E *zs[2] = {static_cast<const E *>(P.tgt) + static_cast<int64_t>(r) * P.t_row,
                    static_cast<const E *>(P.drf) + static_cast<int64_t>(r) * P.d_row};
  const int V = P.V;
  const bool k_on = top_k > 0 && top_k < V, p_on = top_p < 1.0f;
  // maxima and the unfiltered normalisers
  float M[2], Zall[2];
  for (int t = 0; t < 2; ++t) {
    On o;
    o.init();
    for (int j = tid; j < V; j += LW_NT) o.add(lf_y<E>(zs[t], j, P.c2));
    on_merge(o, sm, M[t], Zall[t]);
  }
  // top-k: the exact k-th largest key (ties kept: every logit >= it survives)
  uint32_t kth[2] = {0u, 0u};  // 0: every key survives
  if (k_on) {
    uint32_t prefix[2] = {0u, 0u}, mask = 0u;
    int kr[2] = {top_k, top_k};
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int j = tid; j < 512; j += LW_NT) (&sh.hist[0][0])[j] = 0u;
      __syncthreads();
      for (int t = 0; t < 2; ++t)
        for (int j = tid; j < V; j += LW_NT) {
          const uint32_t k = lf_fkey(lw_get<E>(zs[t], j));
          if ((k & mask) == prefix[t]) atomicAdd(&sh.hist[t][(k >> shift) & 255u], 1u);
        }
      __syncthreads();
      if (wid < 2) {
        const int t = wid;
        // bins from the largest digit down: lane l holds digits 255 - 8l .. 248 - 8l
        uint32_t c8[8], loc = 0u;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          c8[q] = sh.hist[t][255 - (lane * 8 + q)];
          loc += c8[q];
        }
        uint32_t inc = loc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t u = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += u;
        }
        const uint32_t exc = inc - loc;
        const bool mine = exc < static_cast<uint32_t>(kr[t]) && static_cast<uint32_t>(kr[t]) <= inc;
        if (mine) {
          uint32_t before = exc;
          int d = -1;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if (d < 0) {
              if (before + c8[q] >= static_cast<uint32_t>(kr[t]))
                d = 255 - (lane * 8 + q);
              else
                before += c8[q];
            }
          }
          sh.sc[t][0] = d;
          sh.sc[t][1] = static_cast<int>(before);
        }
      }
      __syncthreads();
      for (int t = 0; t < 2; ++t) {
        prefix[t] |= static_cast<uint32_t>(sh.sc[t][0]) << shift;
        kr[t] -= sh.sc[t][1];
      }
      mask |= 255u << shift;
      __syncthreads();
    }
    kth[0] = prefix[0];
    kth[1] = prefix[1];
  }
  // the survivors' normalisers (Kahan sums of single-precision weights)
  float Zk[2];
  for (int t = 0; t < 2; ++t) {
    if (!k_on) {
      Zk[t] = Zall[t];
      continue;
    }
    float s = 0.0f, c = 0.0f;
    for (int j = tid; j < V; j += LW_NT) {
      const float z = lw_get<E>(zs[t], j);
      if (lf_fkey(z) >= kth[t]) kahan(s, c, ex2_approx(__fsub_rn(__fmul_rn(z, P.c2), M[t])));
    }
    Zk[t] = block_sum(__fsub_rn(s, c), sm);
  }
  // the kept sets: threshold tau (a key) and normaliser Zkeep
  uint32_t tau[2] = {kth[0], kth[1]};
  float Zkeep[2] = {Zk[0], Zk[1]};
  int fail = 0;
  if (p_on) {
    for (int j = tid; j < 512; j += LW_NT) {
      (&sh.hist[0][0])[j] = 0u;
      (&sh.mass[0][0])[j] = 0u;
    }
    __syncthreads();
    // depth bins of the survivors: 1/16 of a log2 unit below M; bin 255 the
    // rest (counted, its mass not summed)
    for (int t = 0; t < 2; ++t)
      for (int j = tid; j < V; j += LW_NT) {
        const float z = lw_get<E>(zs[t], j);
        if (z > -INFINITY && lf_fkey(z) >= kth[t]) {
          const float y = __fsub_rn(__fmul_rn(z, P.c2), M[t]);  // <= 0
          const float d = __fmul_rn(y, -16.0f);
          const int b = d < 255.0f ? static_cast<int>(d) : 255;
          atomicAdd(&sh.hist[t][b], 1u);
          if (b < 255)  // w 2^{b/16} = 2^{y + b/16}, in (0.95, 1]
            atomicAdd(&sh.mass[t][b], __float2uint_rn(__fmul_rn(
                                          ex2_approx(__fadd_rn(y, static_cast<float>(b) * 0.0625f)), 4096.0f)));
        }
      }
    __syncthreads();
    if (wid < 2) {
      const int t = wid;
      // the first bin where the survivors' mass (the bins' scaled sums, about
      // 1e-4 relative) passes top_p Zk by a margin of 1e-3 Zk
      const float need = __fmul_rn(Zk[t], __fadd_rn(top_p, 1e-3f));
      float c8[8], loc = 0.0f;
      uint32_t n8[8], nloc = 0u;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int b = lane * 8 + q;
        n8[q] = sh.hist[t][b];
        nloc += n8[q];
        c8[q] = __fmul_rn(__fmul_rn(static_cast<float>(sh.mass[t][b]), 2.44140625e-4f),
                          exp2f(-static_cast<float>(b) * 0.0625f));
        loc = __fadd_rn(loc, c8[q]);
      }
      float inc = loc;
      uint32_t ninc = nloc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, inc, o);
        const uint32_t un = __shfl_up_sync(0xffffffffu, ninc, o);
        if (lane >= o) {
          inc = __fadd_rn(inc, u);
          ninc += un;
        }
      }
      const float exc = __fsub_rn(inc, loc);
      const bool mine = exc < need && need <= inc;
      const uint32_t own = __ballot_sync(0xffffffffu, mine);
      if (mine) {
        float before = exc;
        uint32_t nb = ninc - nloc;
        int bh = -1;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (bh < 0) {
            before = __fadd_rn(before, c8[q]);
            nb += n8[q];
            if (before >= need) {
              bh = lane * 8 + q;
              sh.sc[t][2] = bh;
              sh.sc[t][3] = static_cast<int>(nb);
            }
          }
        }
      }
      if (lane == 0 && !own) {
        sh.sc[t][2] = 255;  // every survivor
        sh.sc[t][3] = static_cast<int>(ninc + 0u);
      }
      if (lane == 0) {
        sh.sc[t][4] = 0;
        sh.sc[t][6] = 0;
      }
    }
    __syncthreads();
    // collect the region (every survivor of the bins up to b_hi; with the
    // deepest bin, every survivor)
    for (int t = 0; t < 2; ++t) {
      const int bh = sh.sc[t][2];
      for (int j = tid; j < V; j += LW_NT) {
        const float z = lw_get<E>(zs[t], j);
        if (z > -INFINITY && lf_fkey(z) >= kth[t]) {
          const float d = __fmul_rn(__fsub_rn(M[t], __fmul_rn(z, P.c2)), 16.0f);
          const int b = d < 255.0f ? static_cast<int>(d) : 255;
          if (b <= bh) {
            const int pos = atomicAdd(&sh.sc[t][4], 1);
            if (pos < LF_CAP)
              sh.reg[t][pos] = (static_cast<unsigned long long>(~lf_fkey(z)) << 32) |
                               static_cast<uint32_t>(j);
          }
        }
      }
    }
    __syncthreads();
    const int n0 = sh.sc[0][4], n1 = sh.sc[1][4];
    fail = (n0 > LF_CAP || n1 > LF_CAP) ? 1 : 0;
    if (!fail) {
      // sort both regions (ascending keys = values descending, indices ascending)
      for (int t = 0; t < 2; ++t)
        for (int j = (t == 0 ? n0 : n1) + tid; j < LF_CAP; j += LW_NT) sh.reg[t][j] = ~0ull;
      __syncthreads();
      for (int k = 2; k <= LF_CAP; k <<= 1)
        for (int jj = k >> 1; jj > 0; jj >>= 1) {
          for (int m = tid; m < LF_CAP; m += LW_NT) {  // both tensors: LF_CAP/2 pairs each
            const int t = m >= LF_CAP / 2, mm = m - t * (LF_CAP / 2);
            const int lo = 2 * mm - (mm & (jj - 1)), hi = lo + jj;
            const bool up = (lo & k) == 0;
            const unsigned long long a = sh.reg[t][lo], b2 = sh.reg[t][hi];
            if ((a > b2) == up) {
              sh.reg[t][lo] = b2;
              sh.reg[t][hi] = a;
            }
          }
          __syncthreads();
        }
      // walk from the top (one warp per tensor): float-float prefix sums of
      // the weights; the first group of equal logits reaching top_p Zk
      if (wid < 2) {
        const int t = wid, n = t == 0 ? n0 : n1;
        const float target = __fmul_rn(top_p, Zk[t]);
        float hi = 0.0f, lo = 0.0f;  // carry (float-float)
        int cross = -1;
        for (int r0 = 0; r0 < n && cross < 0; r0 += 32) {
          const int j = r0 + lane;
          const float z = j < n ? lf_unkey(~static_cast<uint32_t>(sh.reg[t][j] >> 32)) : -INFINITY;
          const float w = j < n ? ex2_approx(__fsub_rn(__fmul_rn(z, P.c2), M[t])) : 0.0f;
          sv::ff inc = {w, 0.0f};
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            sv::ff u = {__shfl_up_sync(0xffffffffu, inc.hi, o), __shfl_up_sync(0xffffffffu, inc.lo, o)};
            if (lane >= o) inc = sv::ff_add(u, inc);
          }
          inc = sv::ff_add(sv::ff{hi, lo}, inc);
          const bool hit = j < n && __fadd_rn(inc.hi, inc.lo) >= target;
          const uint32_t bal = __ballot_sync(0xffffffffu, hit);
          if (bal) cross = r0 + __ffs(bal) - 1;
          hi = __shfl_sync(0xffffffffu, inc.hi, 31);
          lo = __shfl_sync(0xffffffffu, inc.lo, 31);
        }
        if (cross < 0) {  // the region's mass fell short of top_p: no law for this row
          if (lane == 0) sh.sc[t][6] = 1;
          cross = n - 1;
        }
        // the crossing group's end and the kept mass
        const uint32_t hk = static_cast<uint32_t>(sh.reg[t][cross] >> 32);
        sv::ff m = {0.0f, 0.0f};
        for (int j = lane; j < n; j += 32) {
          const uint32_t h = static_cast<uint32_t>(sh.reg[t][j] >> 32);
          if (h <= hk) {
            const float z = lf_unkey(~h);
            m = sv::ff_add(m, sv::ff{ex2_approx(__fsub_rn(__fmul_rn(z, P.c2), M[t])), 0.0f});
          }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          sv::ff u = {__shfl_xor_sync(0xffffffffu, m.hi, o), __shfl_xor_sync(0xffffffffu, m.lo, o)};
          m = sv::ff_add(m, u);
        }
        if (lane == 0) {
          sh.sc[t][5] = static_cast<int>(~hk);  // the kept key threshold
          sh.fc[t][0] = __fadd_rn(m.hi, m.lo);
        }
      }
      __syncthreads();
      for (int t = 0; t < 2; ++t) {
        tau[t] = static_cast<uint32_t>(sh.sc[t][5]);
        Zkeep[t] = sh.fc[t][0];
      }
      fail = sh.sc[0][6] | sh.sc[1][6];
    }
  }
  // beta = sum min(p, q) and R = sum max(0, p - q) over the kept sets
  const float rp = __frcp_rn(Zkeep[0]), rq = __frcp_rn(Zkeep[1]);
  float s1 = 0.0f, c1 = 0.0f, s2 = 0.0f, c2s = 0.0f;
  for (int j = tid; j < V; j += LW_NT) {
    const float a = lw_get<E>(zs[0], j), b = lw_get<E>(zs[1], j);
    const float p = lf_fkey(a) >= tau[0] && a > -INFINITY
                        ? __fmul_rn(ex2_approx(__fsub_rn(__fmul_rn(a, P.c2), M[0])), rp) : 0.0f;
    const float q = lf_fkey(b) >= tau[1] && b > -INFINITY
                        ? __fmul_rn(ex2_approx(__fsub_rn(__fmul_rn(b, P.c2), M[1])), rq) : 0.0f;
    kahan(s1, c1, fminf(p, q));
    kahan(s2, c2s, fmaxf(__fsub_rn(p, q), 0.0f));
  }
  const float beta = block_sum(__fsub_rn(s1, c1), sm);
  const float R = block_sum(__fsub_rn(s2, c2s), sm);
  if (tid == 0) {
    const int x = P.tok[r];
    const float nan = __int_as_float(0x7fc00000);
    float out = nan, px = nan, qx = nan;
    const bool bad = fail || M[0] != M[0] || M[1] != M[1] || !(M[0] > -INFINITY) ||
                     !(M[1] > -INFINITY) || M[0] == INFINITY || M[1] == INFINITY ||
                     Zall[0] != Zall[0] || Zall[1] != Zall[1];
    if (!bad && x >= 0 && x < V) {
      const float a = lw_get<E>(zs[0], x), b = lw_get<E>(zs[1], x);
      px = lf_fkey(a) >= tau[0] && a > -INFINITY
               ? __fmul_rn(ex2_approx(__fsub_rn(__fmul_rn(a, P.c2), M[0])), rp) : 0.0f;
      qx = lf_fkey(b) >= tau[1] && b > -INFINITY
               ? __fmul_rn(ex2_approx(__fsub_rn(__fmul_rn(b, P.c2), M[1])), rq) : 0.0f;
      out = fminf(px, qx);
      if (R > 0.0f)
        out = __fadd_rn(out, __fdiv_rn(__fmul_rn(__fsub_rn(1.0f, beta), fmaxf(__fsub_rn(px, qx), 0.0f)), R));
    }
    P.pspec[r] = out;
    if (P.beta) P.beta[r] = bad ? nan : beta;
    if (P.px) P.px[r] = px;
    if (P.qx) P.qx[r] = qx;
  }
}

}  // namespace

namespace sv {

spec_status law_check_args(const void *target_logits, const void *draft_logits,
                           const int32_t *tokens, const spec_params *params, const float *p_spec) {
  if (!params) return SPEC_ERR_INVALID_ARG;
  const spec_params &p = *params;
  if (p.B < 0 || p.V < 1 || p.V > (1 << 24)) return SPEC_ERR_INVALID_ARG;
  if (p.dtype != SPEC_F32 && p.dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (!std::isfinite(p.temperature) || p.temperature < 0.0f || !(p.top_p > 0.0f) ||
      p.target_row_stride < p.V || p.draft_row_stride < p.V)
    return SPEC_ERR_INVALID_ARG;
  if (p.temperature < 1e-30f) return SPEC_ERR_UNSUPPORTED;  // greedy: a point mass
  if (p.cluster_size < 0 || p.cluster_size > 16 || p.list_capacity < 0 || p.list_capacity > 8192)
    return SPEC_ERR_INVALID_ARG;
  if (p.B == 0) return SPEC_OK;
  if (!target_logits || !draft_logits || !tokens || !p_spec) return SPEC_ERR_INVALID_ARG;
  return SPEC_OK;
}

}  // namespace sv

extern "C" spec_status spec_law(const void *target_logits, const void *draft_logits,
                                const int32_t *tokens, const spec_params *params, float *p_spec,
                                float *beta, float *p_token, float *q_token, void *stream) {
  const spec_status chk = sv::law_check_args(target_logits, draft_logits, tokens, params, p_spec);
  if (chk != SPEC_OK) return chk;
  const spec_params &p = *params;
  const bool filtered = (p.top_k > 0 && p.top_k < p.V) || p.top_p < 1.0f;
  if (p.B == 0) return SPEC_OK;
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
  if (filtered) {
    const size_t smem = sizeof(LFShared);
    auto f = p.dtype == SPEC_F32 ? law_filt_kernel<float> : law_filt_kernel<uint16_t>;
    static bool attr_done[2] = {false, false};
    if (!attr_done[p.dtype]) {
      if (cudaFuncSetAttribute(reinterpret_cast<const void *>(f),
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem)) != cudaSuccess)
        return SPEC_ERR_CUDA;
      attr_done[p.dtype] = true;
    }
    f<<<grid, LW_NT, smem, s>>>(L, p.top_k, p.top_p);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
  }
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
