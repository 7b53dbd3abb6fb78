// spec_verify.cu -- speculative-sampling verification on GB300 (sm_103a).
//
// One thread-block cluster of C CTAs verifies one row (sequence).  The
// vocabulary is split into C contiguous slices, one per CTA; each CTA
// streams its slice of the target (and draft) logits of one position from
// HBM into shared memory with 128-bit loads, and the cluster exchanges
// per-CTA partial results (maxima, sums, counts, candidate lists) through
// distributed shared memory.  Positions are walked in order and the walk
// stops at the first rejection, so the logits of later positions are never
// read.  Method: "Text Generation via Speculative Sampling, KV Caching, and
// OpenVINO", section "Prepare speculative sampling" (steps 3 and 4), and
// "CS3602_FINAL_SpeDec", section "2. 困惑度测试(PPL)" (acceptance
// min(1, p/q), residual norm(max(0, p - q))).
//
// Per position and tensor (p from the target row, q from the draft row):
//   pass 1 (HBM -> SMEM): max, first argmax, NaN / +inf / finite flags, and
//          the per-thread maxima that bound the top-k threshold from below;
//   filters: top-k / top-p thresholds on the raw logit (ties kept), found
//          on a candidate list gathered from the cluster (fast path) or by
//          an exact bisection over order-preserving keys (fallback);
//   normaliser Z over the kept set; p(x), q(x); accept iff u < p(x)/q(x);
//   at the first rejection (or the bonus position) an inverse-CDF draw in
//   vocabulary order, in float-float arithmetic.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "spec_verify.h"
#include "sv_common.cuh"

// Phase timing for development builds (-DSV_PHASE_PROFILE): thread 0 of
// each row's first CTA accumulates clock64() deltas per phase into a global
// array sv_phase_cycles[16].
#ifdef SV_PHASE_PROFILE
__device__ unsigned long long sv_phase_cycles[16];
#define SV_PHASE(id)                                                         \
  do {                                                                       \
    if (k.rank == 0 && threadIdx.x == 0) {                                   \
      const long long now_ = clock64();                                      \
      atomicAdd(&sv_phase_cycles[id], static_cast<unsigned long long>(now_ - t_ph_)); \
      t_ph_ = now_;                                                          \
    }                                                                        \
  } while (0)
#else
#define SV_PHASE(id) \
  do {               \
  } while (0)
#endif

namespace sv {

constexpr int NT = 256;          // threads per CTA
constexpr int NW = NT / kWarp;   // warps per CTA
constexpr int MAXC = 8;          // largest cluster
constexpr int XSLOTS = 4;        // rotating exchange slots
constexpr int XWORDS = 48;       // 32-bit words per exchange slot
constexpr int NBINS = 256;       // histogram bins of the list selection
constexpr int NBANDS = 16;       // depth bands of the top-p candidate window
constexpr int SAMPLE_EVERY = 8;  // band counts look at every 8th element

constexpr uint32_t F_BAD = 1u, F_FINITE = 2u;  // pass-1 flags

enum : int {
  ST_BAD_TOKEN = SPEC_ROW_BAD_TOKEN,
  ST_BAD_LOGIT = SPEC_ROW_BAD_LOGIT,
  ST_NO_FINITE = SPEC_ROW_NO_FINITE,
  ST_Q_ZERO = SPEC_ROW_Q_ZERO,
  ST_BAD_GAMMA = SPEC_ROW_BAD_GAMMA,
  ST_BAD_UNIFORM = SPEC_ROW_BAD_UNIFORM,
  ST_ERROR = SPEC_ROW_ERROR_MASK
};

// Kernel arguments (passed by value as a grid constant).
struct KP {
  const void *tgt, *drf;
  const int32_t *tok;
  const float *uni;
  const int32_t *gam;
  int64_t t_pos, t_row, d_pos, d_row;
  int64_t u_row, u_pos;      // uniform strides (floats)
  int32_t u_acc, u_draw;     // offsets of the acceptance / draw uniform
  int32_t B, gm, V, L;       // L = slice length per CTA (multiple of 8)
  int32_t greedy;
  float invT_hi, invT_lo;    // 1/T as float-float
  float c2;                  // log2(e)/T for the fast exponential
  float T;                   // temperature
  int32_t k_on, top_k, p_on;
  float top_p;
  int32_t cap;               // candidate-list capacity (0: lists off)
  int32_t fp_shift;          // fixed-point scale 2^fp_shift of masses
  int32_t r_warp;            // per-warp rank of the top-k lower bound
  int32_t *acc, *next;
  float *p_dbg, *q_dbg, *res_dbg;
  int32_t *st_dbg;
  unsigned int *diag;
  uint32_t off_stage_t, off_stage_d, off_lp, off_lq, off_w, off_hist;
};

// Distribution of one tensor at one position: keep z >= tau, weight
// e^{(z - m)/T}, normaliser Z.
struct Dist {
  float m;
  float tau;
  ff Z;       // normaliser
  ff rZ;      // 1 / Z
  float rzf;  // 1 / Z in single precision (fast draw)
  float zerr; // bound of the relative error of Z (0 when Z is float-float exact)
  int list;   // 1: the kept set is inside the candidate list
  int n;      // list length
};

__device__ __forceinline__ void set_Z(Dist &D, ff Z, float zerr) {
  D.Z = Z;
  D.rZ = ff_div(ff{1.0f, 0.0f}, Z);
  D.rzf = D.rZ.hi;
  D.zerr = zerr;
}

// Bound of the relative error of a fast weight 2^y (y = (z - m) * log2(e)/T
// rounded three times, then ex2.approx): 2^-21 for the approximation plus
// ln(2) * 3 * 2^-24 * |y| for the rounded exponent.
constexpr float kExpErr0 = 4.8e-7f;
constexpr float kExpErr1 = 1.3e-7f;

// ------------------------------------------------------------ element I/O
template <typename E>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int kPerVec = 4;
  __device__ static __forceinline__ float get(float v) { return canon(v); }
};
template <>
struct Elem<uint16_t> {
  static constexpr int kPerVec = 8;
  __device__ static __forceinline__ float get(uint16_t v) { return canon(bf16_to_f32(v)); }
};

__device__ __forceinline__ uint4 ldg_stream(const uint4 *p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

template <typename E>
__device__ __forceinline__ void unpack(const uint4 &v, float *out);
template <>
__device__ __forceinline__ void unpack<float>(const uint4 &v, float *o) {
  o[0] = canon(__uint_as_float(v.x));
  o[1] = canon(__uint_as_float(v.y));
  o[2] = canon(__uint_as_float(v.z));
  o[3] = canon(__uint_as_float(v.w));
}
template <>
__device__ __forceinline__ void unpack<uint16_t>(const uint4 &v, float *o) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    o[2 * j] = canon(__uint_as_float(w[j] << 16));
    o[2 * j + 1] = canon(__uint_as_float(w[j] & 0xffff0000u));
  }
}

// Pass-1 statistics of one thread.
struct TStat {
  float mx;
  int mi;      // first index of mx (vocabulary index)
  uint32_t fl;
  __device__ void init() {
    mx = -INFINITY;
    mi = INT_MAX;
    fl = 0;
  }
  __device__ __forceinline__ void add(float z, int idx) {
    if (z != z || z == INFINITY)
      fl |= F_BAD;
    else if (z != -INFINITY)
      fl |= F_FINITE;
    if (z > mx) {
      mx = z;
      mi = idx;
    }
  }
};

// Stream slice [lo, lo+n) of one logit row into shared memory (if `keep`)
// and accumulate pass-1 statistics.  Each thread visits its elements in
// increasing index order, so "first index of the maximum" needs no tie test.
template <typename E, bool VEC>
__device__ __forceinline__ void load_slice(const E *__restrict__ g, E *s, int n, int lo,
                                           bool keep, TStat &st) {
  const int tid = threadIdx.x;
  if (VEC) {
    constexpr int EPV = Elem<E>::kPerVec;
    const int nv = n / EPV;
    const uint4 *gv = reinterpret_cast<const uint4 *>(g);
    uint4 *sv4 = reinterpret_cast<uint4 *>(s);
    constexpr int U = 4;
    for (int v0 = tid; v0 < nv; v0 += NT * U) {
      uint4 buf[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * NT;
        if (v < nv) buf[u] = ldg_stream(gv + v);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * NT;
        if (v < nv) {
          if (keep) sv4[v] = buf[u];
          float f[EPV];
          unpack<E>(buf[u], f);
#pragma unroll
          for (int j = 0; j < EPV; ++j) st.add(f[j], lo + v * EPV + j);
        }
      }
    }
    for (int j = nv * EPV + tid; j < n; j += NT) {  // ragged tail
      const E e = g[j];
      if (keep) s[j] = e;
      st.add(Elem<E>::get(e), lo + j);
    }
  } else {
    for (int j = tid; j < n; j += NT) {
      const E e = g[j];
      if (keep) s[j] = e;
      st.add(Elem<E>::get(e), lo + j);
    }
  }
}

// -------------------------------------------------------------- the block
struct Blk {
  uint32_t *xch;      // [XSLOTS][XWORDS] own exchange slots
  uint32_t *gat;      // [MAXC * XWORDS] gathered peer words
  uint64_t *red;      // [NW * 4] reduction scratch
  int32_t *scal;      // misc scalars
  uint32_t C, rank;
  int slot;
};

// Publish words[0..nw) of this CTA, synchronise the cluster, gather the
// words of every CTA into gat[c * nw + j].  All threads call it.
__device__ __forceinline__ void exchange(Blk &k, const uint32_t *words, int nw) {
  uint32_t *mine = k.xch + k.slot * XWORDS;
  if (threadIdx.x < nw) mine[threadIdx.x] = words[threadIdx.x];
  cluster_sync();
  for (int t = threadIdx.x; t < static_cast<int>(k.C) * nw; t += NT) {
    const uint32_t peer = t / nw, w = t % nw;
    k.gat[t] = dsmem_ld_u32(dsmem_addr(smem_u32(k.xch + k.slot * XWORDS + w), peer));
  }
  __syncthreads();
  k.slot = (k.slot + 1) % XSLOTS;
}

__device__ __forceinline__ double gat_f64(const Blk &k, int c, int nw, int w) {
  const uint64_t lo = k.gat[c * nw + w], hi = k.gat[c * nw + w + 1];
  return __longlong_as_double(static_cast<long long>(lo | (hi << 32)));
}
__device__ __forceinline__ uint64_t gat_u64(const Blk &k, int c, int nw, int w) {
  return static_cast<uint64_t>(k.gat[c * nw + w]) |
         (static_cast<uint64_t>(k.gat[c * nw + w + 1]) << 32);
}
__device__ __forceinline__ void put_f64(uint32_t *w, double d) {
  const uint64_t u = static_cast<uint64_t>(__double_as_longlong(d));
  w[0] = static_cast<uint32_t>(u);
  w[1] = static_cast<uint32_t>(u >> 32);
}
__device__ __forceinline__ void put_u64(uint32_t *w, uint64_t u) {
  w[0] = static_cast<uint32_t>(u);
  w[1] = static_cast<uint32_t>(u >> 32);
}

// Block sums in a fixed order (deterministic).  Every thread gets the result.
__device__ __forceinline__ double block_sum_f64(Blk &k, double v) {
  v = warp_sum_f64(v);
  double *r = reinterpret_cast<double *>(k.red);
  if ((threadIdx.x & 31) == 0) r[threadIdx.x >> 5] = v;
  __syncthreads();
  double s = 0.0;
#pragma unroll
  for (int w = 0; w < NW; ++w) s += r[w];
  __syncthreads();
  return s;
}
__device__ __forceinline__ uint64_t block_sum_u64(Blk &k, uint64_t v) {
  v = warp_sum_u64(v);
  if ((threadIdx.x & 31) == 0) k.red[threadIdx.x >> 5] = v;
  __syncthreads();
  uint64_t s = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) s += k.red[w];
  __syncthreads();
  return s;
}
__device__ __forceinline__ void block_sum2_u64(Blk &k, uint64_t &a, uint64_t &b) {
  a = warp_sum_u64(a);
  b = warp_sum_u64(b);
  if ((threadIdx.x & 31) == 0) {
    k.red[threadIdx.x >> 5] = a;
    k.red[NW + (threadIdx.x >> 5)] = b;
  }
  __syncthreads();
  uint64_t sa = 0, sb = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    sa += k.red[w];
    sb += k.red[NW + w];
  }
  __syncthreads();
  a = sa;
  b = sb;
}
// Exclusive scan of float-float values in thread order; returns the prefix
// of this thread and writes the block total.
__device__ __forceinline__ ff block_scan_ff(Blk &k, ff v, ff &total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  ff inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    ff u;
    u.hi = __shfl_up_sync(0xffffffffu, inc.hi, o);
    u.lo = __shfl_up_sync(0xffffffffu, inc.lo, o);
    if (lane >= o) inc = ff_add(u, inc);
  }
  float *r = reinterpret_cast<float *>(k.red);
  if (lane == 31) {
    r[2 * w] = inc.hi;
    r[2 * w + 1] = inc.lo;
  }
  __syncthreads();
  ff base = {0.0f, 0.0f}, tot = {0.0f, 0.0f};
#pragma unroll
  for (int j = 0; j < NW; ++j) {
    const ff x = {r[2 * j], r[2 * j + 1]};
    if (j < w) base = ff_add(base, x);
    tot = ff_add(tot, x);
  }
  __syncthreads();
  total = tot;
  ff excl;
  excl.hi = __shfl_up_sync(0xffffffffu, inc.hi, 1);
  excl.lo = __shfl_up_sync(0xffffffffu, inc.lo, 1);
  if (lane == 0) excl = {0.0f, 0.0f};
  return ff_add(base, excl);
}
__device__ __forceinline__ ff block_sum_ff(Blk &k, ff v) {
  ff tot;
  (void)block_scan_ff(k, v, tot);
  return tot;
}
__device__ __forceinline__ int block_max_i32(Blk &k, int v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  int *r = reinterpret_cast<int *>(k.red);
  if ((threadIdx.x & 31) == 0) r[threadIdx.x >> 5] = v;
  __syncthreads();
  int m = INT_MIN;
#pragma unroll
  for (int w = 0; w < NW; ++w) m = max(m, r[w]);
  __syncthreads();
  return m;
}

// ----------------------------------------------------------- the weights
// y = (z - m)/T in float-float.  z - m is exact as a float-float (TwoSum).
__device__ __forceinline__ ff scaled_gap(const KP &P, float z, float m) {
  const ff d = two_sum(z, -m);
  return ff_mul(d, ff{P.invT_hi, P.invT_lo});
}
// Accurate e^{(z - m)/T} (0 for z = -inf).
__device__ __forceinline__ ff weight_ff(const KP &P, float z, float m) {
  if (z == -INFINITY) return {0.0f, 0.0f};
  return ff_exp(scaled_gap(P, z, m));
}
// Fast e^{(z - m)/T} (single precision, ~2^-22 relative; 0 below 2^-126).
__device__ __forceinline__ float weight_fast(const KP &P, float z, float m) {
  return ex2_approx(__fmul_rn(__fsub_rn(z, m), P.c2));
}

template <typename E>
__device__ __forceinline__ float stage_get(const E *s, int j) {
  return Elem<E>::get(s[j]);
}

// ------------------------------------------------------- slice-mode parts
// Z of both tensors over their kept sets, fast single precision (used for
// p(x)/q(x) in the acceptance test when the support is the whole slice).
// With `bands`, also a histogram of depth bands (nats below the maximum) of
// every SAMPLE_EVERY-th element: an estimate of how many tokens a top-p
// candidate window of each depth would hold.  Returns the cluster totals in
// zall_t / zall_d and the band counts in bt[] / bd[] (cumulative).
__constant__ float kBandDepth[NBANDS] = {1.f, 2.f, 3.f, 4.f, 5.f, 6.f, 7.f, 8.f,
                                         9.f, 10.f, 11.f, 12.f, 14.f, 16.f, 20.f, 24.f};

template <typename E>
__device__ void slice_Z_fast(const KP &P, Blk &k, const E *st, const E *sd, int n,
                             Dist &dt, Dist &dd, bool dod, bool bands, double &zall_t,
                             double &zall_d, int *bt, int *bd, int *bh /* smem [2][NBANDS+1] */) {
  if (bands) {
    for (int j = threadIdx.x; j < 2 * (NBANDS + 1); j += NT) bh[j] = 0;
    __syncthreads();
  }
  // compensated (Kahan) single-precision sums, plus a running error bound
  float zt = 0.0f, ct = 0.0f, et = 0.0f, zd = 0.0f, cd = 0.0f, ed = 0.0f;
  int it = 0;
  for (int j = threadIdx.x; j < n; j += NT, ++it) {
    const bool smp = bands && (it % SAMPLE_EVERY) == 0;
    const float a = stage_get(st, j);
    if (a >= dt.tau) {
      const float y = __fmul_rn(__fsub_rn(a, dt.m), P.c2);
      const float e = ex2_approx(y);
      const float t = __fsub_rn(e, ct), s2 = __fadd_rn(zt, t);
      ct = __fsub_rn(__fsub_rn(s2, zt), t);
      zt = s2;
      et = __fmaf_rn(e, __fmaf_rn(fabsf(y), kExpErr1, kExpErr0), et);
    }
    if (smp && a == a) {
      const float d = __fmul_rn(__fsub_rn(dt.m, a), P.invT_hi);
      int band = 0;
      while (band < NBANDS && !(d < kBandDepth[band])) ++band;
      atomicAdd(&bh[band], 1);
    }
    if (dod) {
      const float b = stage_get(sd, j);
      if (b >= dd.tau) {
        const float y = __fmul_rn(__fsub_rn(b, dd.m), P.c2);
        const float e = ex2_approx(y);
        const float t = __fsub_rn(e, cd), s2 = __fadd_rn(zd, t);
        cd = __fsub_rn(__fsub_rn(s2, zd), t);
        zd = s2;
        ed = __fmaf_rn(e, __fmaf_rn(fabsf(y), kExpErr1, kExpErr0), ed);
      }
      if (smp && b == b) {
        const float d = __fmul_rn(__fsub_rn(dd.m, b), P.invT_hi);
        int band = 0;
        while (band < NBANDS && !(d < kBandDepth[band])) ++band;
        atomicAdd(&bh[NBANDS + 1 + band], 1);
      }
    }
  }
  const ff Zt = block_sum_ff(k, quick_two_sum(zt, -ct));
  const ff Zd = block_sum_ff(k, quick_two_sum(zd, -cd));
  const double Et = block_sum_f64(k, static_cast<double>(et));
  const double Ed = block_sum_f64(k, static_cast<double>(ed));
  constexpr int NWD = 8 + 2 * NBANDS;
  uint32_t w[NWD];
  w[0] = __float_as_uint(Zt.hi);
  w[1] = __float_as_uint(Zt.lo);
  w[2] = __float_as_uint(Zd.hi);
  w[3] = __float_as_uint(Zd.lo);
  put_f64(w + 4, Et);
  put_f64(w + 6, Ed);
  if (bands) {
    __syncthreads();
    for (int j = 0; j < NBANDS; ++j) {
      w[8 + j] = static_cast<uint32_t>(bh[j]);
      w[8 + NBANDS + j] = static_cast<uint32_t>(bh[NBANDS + 1 + j]);
    }
  } else {
    for (int j = 8; j < NWD; ++j) w[j] = 0;
  }
  exchange(k, w, NWD);
  ff st_ = {0.0f, 0.0f}, sd_ = {0.0f, 0.0f};
  double et_ = 0.0, ed_ = 0.0;
  for (uint32_t c = 0; c < k.C; ++c) {
    const uint32_t *g = k.gat + c * NWD;
    st_ = ff_add(st_, ff{__uint_as_float(g[0]), __uint_as_float(g[1])});
    sd_ = ff_add(sd_, ff{__uint_as_float(g[2]), __uint_as_float(g[3])});
    et_ += gat_f64(k, c, NWD, 4);
    ed_ += gat_f64(k, c, NWD, 6);
  }
  if (bands) {
    int ct2 = 0, cd2 = 0;
    for (int j = 0; j < NBANDS; ++j) {
      for (uint32_t c = 0; c < k.C; ++c) {
        ct2 += static_cast<int>(k.gat[c * NWD + 8 + j]);
        cd2 += static_cast<int>(k.gat[c * NWD + 8 + NBANDS + j]);
      }
      bt[j] = ct2;
      bd[j] = cd2;
    }
  }
  zall_t = ff_to_double(st_);
  zall_d = ff_to_double(sd_);
  // relative error bound: the weights' bound plus the compensated sums'
  set_Z(dt, st_, static_cast<float>(et_ / zall_t) + 2.4e-7f);
  if (dod) set_Z(dd, sd_, static_cast<float>(ed_ / zall_d) + 2.4e-7f);
}

// Fixed-point weight of the top-p mass comparisons: round(e * 2^shift).
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }
__device__ __forceinline__ uint64_t to_fixed(ff e, int shift) {
  const float sc = pow2f(shift);  // exact scaling
  return __float2ull_rn(__fmul_rn(e.hi, sc)) +
         static_cast<uint64_t>(__float2ll_rn(__fmul_rn(e.lo, sc)));
}

// target = ceil(top_p * tot), exactly, with top_p = m24 / 2^sh.
__device__ __forceinline__ uint64_t ceil_scale(float top_p, uint64_t tot) {
  int e;
  const float fr = frexpf(top_p, &e);  // top_p = fr * 2^e, fr in [0.5, 1)
  const uint64_t m24 = static_cast<uint64_t>(ldexpf(fr, 24));
  const int sh = 24 - e;
  const uint64_t hi = __umul64hi(m24, tot), lo = m24 * tot;
  uint64_t q, rem;
  if (sh >= 64) {
    q = hi >> (sh - 64);
    rem = (lo != 0) || ((hi & ((1ull << (sh - 64)) - 1)) != 0);
  } else {
    q = (lo >> sh) | (sh ? (hi << (64 - sh)) : 0);
    rem = (lo & ((1ull << sh) - 1)) != 0;
  }
  return q + (rem ? 1 : 0);
}

// Exact threshold search over the cluster's slices: the largest key K such
// that the weight of {key(z) >= K} reaches the target (top-k: weight 1;
// top-p: fixed-point mass of the top-k survivors).  Binary search over the
// 32-bit key space, one pass + one cluster exchange per step, both tensors
// in lock-step.  The result is always the key of an existing element.
template <typename E>
__device__ void slice_bisect(const KP &P, Blk &k, const E *st, const E *sd, int n,
                             Dist &dt, Dist &dd, bool dot, bool dod, bool mass) {
  uint64_t tgt_t = static_cast<uint64_t>(P.top_k), tgt_d = tgt_t;
  const float sc = pow2f(P.fp_shift);
  if (mass) {
    uint64_t a = 0, b = 0;
    for (int j = threadIdx.x; j < n; j += NT) {
      if (dot) {
        const float x = stage_get(st, j);
        if (x >= dt.tau) a += __float2ull_rn(__fmul_rn(weight_fast(P, x, dt.m), sc));
      }
      if (dod) {
        const float y = stage_get(sd, j);
        if (y >= dd.tau) b += __float2ull_rn(__fmul_rn(weight_fast(P, y, dd.m), sc));
      }
    }
    block_sum2_u64(k, a, b);
    uint32_t w[4];
    put_u64(w, a);
    put_u64(w + 2, b);
    exchange(k, w, 4);
    uint64_t ta = 0, tb = 0;
    for (uint32_t c = 0; c < k.C; ++c) {
      ta += gat_u64(k, c, 4, 0);
      tb += gat_u64(k, c, 4, 2);
    }
    tgt_t = ceil_scale(P.top_p, ta);
    tgt_d = ceil_scale(P.top_p, tb);
  }
  uint64_t lo_t = 0, hi_t = 1ull << 32, lo_d = 0, hi_d = 1ull << 32;
  const uint32_t kt0 = fkey(dt.tau), kd0 = fkey(dd.tau);
  for (int it = 0; it < 32; ++it) {
    const uint64_t mt = (lo_t + hi_t) >> 1, md = (lo_d + hi_d) >> 1;
    uint64_t a = 0, b = 0;
    for (int j = threadIdx.x; j < n; j += NT) {
      if (dot) {
        const float x = stage_get(st, j);
        const uint32_t kx = fkey(x);
        if (x == x && kx >= mt && kx >= kt0)
          a += mass ? __float2ull_rn(__fmul_rn(weight_fast(P, x, dt.m), sc)) : 1ull;
      }
      if (dod) {
        const float y = stage_get(sd, j);
        const uint32_t ky = fkey(y);
        if (y == y && ky >= md && ky >= kd0)
          b += mass ? __float2ull_rn(__fmul_rn(weight_fast(P, y, dd.m), sc)) : 1ull;
      }
    }
    block_sum2_u64(k, a, b);
    uint32_t w[4];
    put_u64(w, a);
    put_u64(w + 2, b);
    exchange(k, w, 4);
    uint64_t sa = 0, sb = 0;
    for (uint32_t c = 0; c < k.C; ++c) {
      sa += gat_u64(k, c, 4, 0);
      sb += gat_u64(k, c, 4, 2);
    }
    if (sa >= tgt_t) lo_t = mt; else hi_t = mt;
    if (sb >= tgt_d) lo_d = md; else hi_d = md;
  }
  if (dot) dt.tau = fmaxf(dt.tau, key_to_f(static_cast<uint32_t>(lo_t)));
  if (dod) dd.tau = fmaxf(dd.tau, key_to_f(static_cast<uint32_t>(lo_d)));
}

// Exact Z (float-float) over the kept sets of the slices.
template <typename E>
__device__ void slice_Z_exact(const KP &P, Blk &k, const E *st, const E *sd, int n,
                              Dist &dt, Dist &dd, bool dot, bool dod) {
  ff a = {0.0f, 0.0f}, b = {0.0f, 0.0f};
  for (int j = threadIdx.x; j < n; j += NT) {
    if (dot) {
      const float x = stage_get(st, j);
      if (x >= dt.tau) a = ff_add(a, weight_ff(P, x, dt.m));
    }
    if (dod) {
      const float y = stage_get(sd, j);
      if (y >= dd.tau) b = ff_add(b, weight_ff(P, y, dd.m));
    }
  }
  a = block_sum_ff(k, a);
  b = block_sum_ff(k, b);
  uint32_t w[4] = {__float_as_uint(a.hi), __float_as_uint(a.lo), __float_as_uint(b.hi),
                   __float_as_uint(b.lo)};
  exchange(k, w, 4);
  ff sa = {0.0f, 0.0f}, sb = {0.0f, 0.0f};
  for (uint32_t c = 0; c < k.C; ++c) {
    sa = ff_add(sa, ff{__uint_as_float(k.gat[c * 4]), __uint_as_float(k.gat[c * 4 + 1])});
    sb = ff_add(sb, ff{__uint_as_float(k.gat[c * 4 + 2]), __uint_as_float(k.gat[c * 4 + 3])});
  }
  if (dot) set_Z(dt, sa, 0.0f);
  if (dod) set_Z(dd, sb, 0.0f);
}

// The draw weight of one token from its target / draft logits: p_v (bonus)
// or max(0, p_v - q_v) (residual, "max_fn" of "Prepare autoregressive
// sampling", normalised by the caller's inverse CDF).
__device__ __forceinline__ ff draw_weight_of(const KP &P, float x, float y, const Dist &dt,
                                             const Dist &dd, bool residual) {
  if (!(x >= dt.tau)) return {0.0f, 0.0f};
  ff p = ff_mul(weight_ff(P, x, dt.m), dt.rZ);
  if (!residual) return p;
  if (y >= dd.tau) p = ff_sub(p, ff_mul(weight_ff(P, y, dd.m), dd.rZ));
  return p.hi > 0.0f ? p : ff{0.0f, 0.0f};
}

template <typename E>
__device__ __forceinline__ ff draw_weight(const KP &P, const E *st, const E *sd, int j,
                                          const Dist &dt, const Dist &dd, bool residual) {
  return draw_weight_of(P, stage_get(st, j), residual ? stage_get(sd, j) : 0.0f, dt, dd,
                        residual);
}

// Inverse-CDF draw over the cluster's slices in vocabulary order.  Each
// thread owns a contiguous chunk of its CTA's slice.  Returns the token (all
// CTAs), or -1 when the total weight is 0; *Wout = the total weight.
template <typename E>
__device__ int slice_draw(const KP &P, Blk &k, const E *st, const E *sd, int n, int lo,
                          const Dist &dt, const Dist &dd, bool residual, float u, ff *Wout) {
  int ch = (n + NT - 1) / NT;
  ch |= 1;  // odd chunk length: conflict-free shared-memory strides
  const int j0 = min(n, static_cast<int>(threadIdx.x) * ch), j1 = min(n, j0 + ch);
  ff s = {0.0f, 0.0f};
  int lastpos = -1;
  for (int j = j0; j < j1; ++j) {
    const ff w = draw_weight(P, st, sd, j, dt, dd, residual);
    if (w.hi > 0.0f) lastpos = lo + j;
    s = ff_add(s, w);
  }
  ff ctot;
  const ff pre = block_scan_ff(k, s, ctot);
  const int clast = block_max_i32(k, lastpos);
  uint32_t w[3] = {__float_as_uint(ctot.hi), __float_as_uint(ctot.lo),
                   static_cast<uint32_t>(clast)};
  exchange(k, w, 3);
  ff W = {0.0f, 0.0f}, mybase = {0.0f, 0.0f};
  int glast = -1;
  for (uint32_t c = 0; c < k.C; ++c) {
    const ff x = {__uint_as_float(k.gat[c * 3]), __uint_as_float(k.gat[c * 3 + 1])};
    if (c < k.rank) mybase = ff_add(mybase, x);
    W = ff_add(W, x);
    glast = max(glast, static_cast<int>(k.gat[c * 3 + 2]));
  }
  *Wout = W;
  if (!(W.hi > 0.0f)) return -1;
  const ff target = ff_mul_f(W, u);
  if (threadIdx.x == 0) k.scal[8] = -1;
  __syncthreads();
  const ff a = ff_add(mybase, pre), b = ff_add(a, s);
  if (!ff_lt(target, a) && ff_lt(target, b)) {
    ff c = a;
    int tok = -1;
    for (int j = j0; j < j1; ++j) {
      const ff wj = draw_weight(P, st, sd, j, dt, dd, residual);
      if (wj.hi > 0.0f) tok = lo + j;
      c = ff_add(c, wj);
      if (ff_lt(target, c) && wj.hi > 0.0f) break;
    }
    k.scal[8] = tok;
  }
  __syncthreads();
  // broadcast the owner's token (or -1) to every CTA
  uint32_t v = static_cast<uint32_t>(k.scal[8]);
  exchange(k, &v, 1);
  int tok = -1;
  for (uint32_t c = 0; c < k.C; ++c) tok = max(tok, static_cast<int>(k.gat[c]));
  if (tok < 0) tok = glast;  // rounding left the target past the last weight
  return tok;
}

// Single-precision draw weight and a bound of its absolute error (the
// certified fast draw): p_v = 2^{y} / Z with y rounded as in weight_fast,
// relative error <= kExpErr0 + kExpErr1 |y| + zerr + 2^-22 (the reciprocal);
// the residual's subtraction adds (p + q) 2^-24.
__device__ __forceinline__ void fast_weight(const KP &P, float x, float y, const Dist &dt,
                                            const Dist &dd, bool residual, float &w,
                                            float &err) {
  w = 0.0f;
  err = 0.0f;
  if (!(x >= dt.tau)) return;
  const float yx = __fmul_rn(__fsub_rn(x, dt.m), P.c2);
  const float p = __fmul_rn(ex2_approx(yx), dt.rzf);
  const float ep = __fmul_rn(p, __fmaf_rn(fabsf(yx), kExpErr1, kExpErr0 + dt.zerr + 2.4e-7f));
  if (!residual) {
    w = p;
    err = ep;
    return;
  }
  float q = 0.0f, eq = 0.0f;
  if (y >= dd.tau) {
    const float yy = __fmul_rn(__fsub_rn(y, dd.m), P.c2);
    q = __fmul_rn(ex2_approx(yy), dd.rzf);
    eq = __fmul_rn(q, __fmaf_rn(fabsf(yy), kExpErr1, kExpErr0 + dd.zerr + 2.4e-7f));
  }
  const float d = __fsub_rn(p, q);
  w = d > 0.0f ? d : 0.0f;
  err = __fadd_rn(__fadd_rn(ep, eq), __fmul_rn(__fadd_rn(p, q), 6.0e-8f));
}

// Certified single-precision inverse-CDF draw over the slices.  Sums run in
// float-float over single-precision weights; D bounds the total absolute
// error of the weights, so every prefix sum and the target u*W are within D
// of their exact values.  The token is returned only when the target lies
// more than 2D (plus a rounding slack) inside its CDF interval; otherwise
// -2 (uncertain: the caller redraws exactly).  -1: total weight 0.
template <typename E>
__device__ int slice_draw_fast(const KP &P, Blk &k, const E *st, const E *sd, int n, int lo,
                               const Dist &dt, const Dist &dd, bool residual, float u,
                               float *Wf) {
  int ch = (n + NT - 1) / NT;
  ch |= 1;
  const int j0 = min(n, static_cast<int>(threadIdx.x) * ch), j1 = min(n, j0 + ch);
  ff s = {0.0f, 0.0f};
  float dsum = 0.0f;
  int lastpos = -1;
  for (int j = j0; j < j1; ++j) {
    float w, e;
    fast_weight(P, stage_get(st, j), residual ? stage_get(sd, j) : 0.0f, dt, dd, residual, w, e);
    if (w > 0.0f) lastpos = lo + j;
    s = ff_add_f(s, w);
    dsum = __fadd_rn(dsum, e);
  }
  ff ctot;
  const ff pre = block_scan_ff(k, s, ctot);
  const float cerr = static_cast<float>(block_sum_f64(k, static_cast<double>(dsum)));
  const int clast = block_max_i32(k, lastpos);
  uint32_t w4[4] = {__float_as_uint(ctot.hi), __float_as_uint(ctot.lo), __float_as_uint(cerr),
                    static_cast<uint32_t>(clast)};
  exchange(k, w4, 4);
  ff W = {0.0f, 0.0f}, mybase = {0.0f, 0.0f};
  float D = 0.0f;
  for (uint32_t c = 0; c < k.C; ++c) {
    const ff x = {__uint_as_float(k.gat[c * 4]), __uint_as_float(k.gat[c * 4 + 1])};
    if (c < k.rank) mybase = ff_add(mybase, x);
    W = ff_add(W, x);
    D = __fadd_rn(D, __uint_as_float(k.gat[c * 4 + 2]));
  }
  *Wf = W.hi + W.lo;
  if (!(W.hi > 0.0f)) return -1;
  // absolute slack: flushed subnormal weights and float-float rounding
  const float slack = __fmaf_rn(W.hi, 1e-12f, static_cast<float>(P.V) * 4e-38f *
                                                  (dt.rzf + (residual ? dd.rzf : 0.0f)));
  const ff target = ff_mul_f(W, u);
  if (threadIdx.x == 0) {
    k.scal[8] = -1;
    k.scal[10] = 0;
  }
  __syncthreads();
  const ff a = ff_add(mybase, pre), b = ff_add(a, s);
  if (!ff_lt(target, a) && ff_lt(target, b)) {
    ff c = a;
    int tok = -1;
    float margin = 0.0f;
    for (int j = j0; j < j1; ++j) {
      float w, e;
      fast_weight(P, stage_get(st, j), residual ? stage_get(sd, j) : 0.0f, dt, dd, residual, w, e);
      const ff cp = c;
      c = ff_add_f(c, w);
      if (w > 0.0f && ff_lt(target, c)) {
        tok = lo + j;
        const ff l = ff_sub(target, cp), h = ff_sub(c, target);
        margin = fminf(l.hi + l.lo, h.hi + h.lo);
        break;
      }
    }
    k.scal[8] = tok;
    k.scal[10] = (tok >= 0 && margin > __fmaf_rn(2.0f, D, slack)) ? 1 : 0;
  }
  __syncthreads();
  uint32_t v2[2] = {static_cast<uint32_t>(k.scal[8]), static_cast<uint32_t>(k.scal[10])};
  __syncthreads();
  exchange(k, v2, 2);
  int tok = -1, cert = 0;
  for (uint32_t c = 0; c < k.C; ++c) {
    const int t = static_cast<int>(k.gat[c * 2]);
    if (t >= 0) {
      tok = t;
      cert = static_cast<int>(k.gat[c * 2 + 1]);
    }
  }
  return (tok >= 0 && cert) ? tok : -2;
}

// --------------------------------------------------------- list-mode parts
// Candidate lists: every CTA of the cluster holds the same index-ordered
// list of the tokens whose logit is >= a candidate threshold, gathered from
// all slices.  p-list entries carry the target and draft logits of the
// token, q-list entries the draft logit.
struct Lists {
  int *p_idx;
  float *p_zp, *p_zq;
  int *q_idx;
  float *q_zq;
  uint64_t *w;     // [cap] fixed-point weights
  uint64_t *hist;  // [NBINS]
};

// Per-warp counts of {z >= cand} over contiguous warp segments of the slice.
// Sets the CTA totals and this warp's exclusive base (index order).
template <typename E>
__device__ void count_pass(Blk &k, const E *st, const E *sd, int n, float ct, float cd,
                           bool dot, bool dod, int *wc /* smem [2*NW] */, int &tot_t,
                           int &tot_d, int &base_t, int &base_d) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = (n + NW - 1) / NW;
  const int s0 = min(n, w * seg), s1 = min(n, s0 + seg);
  int a = 0, b = 0;
  for (int j0 = s0; j0 < s1; j0 += 32) {
    const int j = j0 + lane;
    bool ft = false, fd = false;
    if (j < s1) {
      if (dot) ft = stage_get(st, j) >= ct;
      if (dod) fd = stage_get(sd, j) >= cd;
    }
    a += __popc(__ballot_sync(0xffffffffu, ft));
    b += __popc(__ballot_sync(0xffffffffu, fd));
  }
  if (lane == 0) {
    wc[w] = a;
    wc[NW + w] = b;
  }
  __syncthreads();
  tot_t = tot_d = base_t = base_d = 0;
  for (int j = 0; j < NW; ++j) {
    if (j < w) {
      base_t += wc[j];
      base_d += wc[NW + j];
    }
    tot_t += wc[j];
    tot_d += wc[NW + j];
  }
  __syncthreads();
}

// Write the candidates into the lists of every CTA of the cluster at the
// positions given by the cluster offsets and warp bases (index order).
template <typename E>
__device__ void write_pass(Blk &k, const Lists &L, const E *st, const E *sd, int n, int lo,
                           float ct, float cd, bool dot, bool dod, bool has_draft, int pos_t,
                           int pos_d) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = (n + NW - 1) / NW;
  const int s0 = min(n, w * seg), s1 = min(n, s0 + seg);
  const uint32_t lt = (1u << lane) - 1u;
  for (int j0 = s0; j0 < s1; j0 += 32) {
    const int j = j0 + lane;
    float zt = 0.0f, zd = 0.0f;
    bool ft = false, fd = false;
    if (j < s1) {
      zt = stage_get(st, j);
      if (has_draft) zd = stage_get(sd, j);
      ft = dot && zt >= ct;
      fd = dod && zd >= cd;
    }
    const uint32_t mt = __ballot_sync(0xffffffffu, ft), md = __ballot_sync(0xffffffffu, fd);
    if (ft) {
      const int pos = pos_t + __popc(mt & lt);
      const uint32_t ai = smem_u32(L.p_idx + pos), ap = smem_u32(L.p_zp + pos),
                     aq = smem_u32(L.p_zq + pos);
      for (uint32_t c = 0; c < k.C; ++c) {
        dsmem_st_u32(dsmem_addr(ai, c), static_cast<uint32_t>(lo + j));
        dsmem_st_u32(dsmem_addr(ap, c), __float_as_uint(zt));
        dsmem_st_u32(dsmem_addr(aq, c), __float_as_uint(zd));
      }
    }
    if (fd) {
      const int pos = pos_d + __popc(md & lt);
      const uint32_t ai = smem_u32(L.q_idx + pos), aq = smem_u32(L.q_zq + pos);
      for (uint32_t c = 0; c < k.C; ++c) {
        dsmem_st_u32(dsmem_addr(ai, c), static_cast<uint32_t>(lo + j));
        dsmem_st_u32(dsmem_addr(aq, c), __float_as_uint(zd));
      }
    }
    pos_t += __popc(mt);
    pos_d += __popc(md);
  }
}

__device__ __forceinline__ void block_minmax(Blk &k, float &lo, float &hi) {
  lo = warp_min(lo);
  hi = warp_max(hi);
  float *r = reinterpret_cast<float *>(k.red);
  if ((threadIdx.x & 31) == 0) {
    r[2 * (threadIdx.x >> 5)] = lo;
    r[2 * (threadIdx.x >> 5) + 1] = hi;
  }
  __syncthreads();
  lo = INFINITY;
  hi = -INFINITY;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    lo = fminf(lo, r[2 * w]);
    hi = fmaxf(hi, r[2 * w + 1]);
  }
  __syncthreads();
}

// Bins of [lo, hi], bin 0 holding hi.  Monotone (non-increasing in v):
// every step is a correctly rounded operation applied to a monotone input.
// Halving first keeps hi - lo finite for any finite pair.
struct BinMap {
  float hh, sc;
  bool deg;
};
__device__ __forceinline__ BinMap bin_map(float lo, float hi) {
  BinMap m;
  m.hh = 0.5f * hi;
  const float span = __fsub_rn(m.hh, 0.5f * lo);
  m.sc = __fdiv_rn(static_cast<float>(NBINS), span);
  m.deg = !(span > 0.0f) || !(m.sc < INFINITY);
  return m;
}
__device__ __forceinline__ int value_bin(float v, const BinMap &m) {
  if (m.deg) return v >= 2.0f * m.hh ? 0 : NBINS - 1;
  const float t = __fmul_rn(__fsub_rn(m.hh, 0.5f * v), m.sc);
  return min(NBINS - 1, static_cast<int>(t));
}

// Threshold selection on a list (block level, each CTA independently): the
// largest value v such that the weight of entries with value >= v reaches
// `target` (top-k: weight 1 per entry; top-p: w[j]).  Refines a 256-bin
// value histogram of the current range, bins ordered from the largest value
// down; integer weights make the result exact and independent of the order
// of the shared-memory atomics.  Returns -inf if the whole list falls short.
__device__ float list_select(Blk &k, const float *val, int n, const uint64_t *w,
                             uint64_t target, uint64_t *hist) {
  float lo = INFINITY, hi = -INFINITY;
  for (int j = threadIdx.x; j < n; j += NT)
    if (!w || w[j]) {
      lo = fminf(lo, val[j]);
      hi = fmaxf(hi, val[j]);
    }
  block_minmax(k, lo, hi);
  if (!(lo <= hi)) return -INFINITY;  // empty
  uint64_t above = 0;
  for (int iter = 0; iter <= n + 1; ++iter) {  // each step drops >= 1 distinct value
    if (lo == hi) {
      // every remaining entry has this value; does the target fall here?
      uint64_t s = 0;
      for (int j = threadIdx.x; j < n; j += NT)
        if ((!w || w[j]) && val[j] == lo) s += w ? w[j] : 1ull;
      s = block_sum_u64(k, s);
      return (above + s >= target) ? lo : -INFINITY;
    }
    const BinMap bm = bin_map(lo, hi);
    for (int j = threadIdx.x; j < NBINS; j += NT) hist[j] = 0;
    __syncthreads();
    for (int j = threadIdx.x; j < n; j += NT) {
      const float v = val[j];
      if ((!w || w[j]) && v >= lo && v <= hi)
        atomicAdd(reinterpret_cast<unsigned long long *>(&hist[value_bin(v, bm)]),
                  static_cast<unsigned long long>(w ? w[j] : 1ull));
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      uint64_t loc = 0;
#pragma unroll
      for (int q = 0; q < NBINS / 32; ++q) loc += hist[lane * (NBINS / 32) + q];
      uint64_t inc = loc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint64_t u = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += u;
      }
      const uint32_t reach = __ballot_sync(0xffffffffu, above + inc >= target);
      if (lane == 0) k.scal[9] = -1;
      __syncwarp();
      if (reach && lane == __ffs(reach) - 1) {
        uint64_t cum = above + inc - loc;
        int bsel = lane * (NBINS / 32);
        for (int q = 0; q < NBINS / 32; ++q) {
          const uint64_t hq = hist[lane * (NBINS / 32) + q];
          if (cum + hq >= target) {
            bsel = lane * (NBINS / 32) + q;
            break;
          }
          cum += hq;
        }
        k.scal[9] = bsel;
        reinterpret_cast<uint64_t *>(k.scal)[6] = cum;  // weight strictly above the bin
      }
    }
    __syncthreads();
    const int bsel = k.scal[9];
    const uint64_t nabove = reinterpret_cast<uint64_t *>(k.scal)[6];
    __syncthreads();
    if (bsel < 0) return -INFINITY;  // the list's total falls short of the target
    float nlo = INFINITY, nhi = -INFINITY;
    for (int j = threadIdx.x; j < n; j += NT) {
      const float v = val[j];
      if ((!w || w[j]) && v >= lo && v <= hi && value_bin(v, bm) == bsel) {
        nlo = fminf(nlo, v);
        nhi = fmaxf(nhi, v);
      }
    }
    block_minmax(k, nlo, nhi);
    lo = nlo;
    hi = nhi;
    above = nabove;
  }
  return lo;  // not reached
}

// Filters and normaliser of one tensor from its list.  `zall` is the
// normaliser over the whole vocabulary (top-p without top-k).  Returns false
// if the list cannot hold the kept set (the nucleus reaches below it).
__device__ bool list_dist(const KP &P, Blk &k, const float *val, int n, Dist &D,
                          uint64_t *w, uint64_t *hist, double zall) {
  float tau = -INFINITY;
  if (P.k_on) {
    tau = list_select(k, val, n, nullptr, static_cast<uint64_t>(P.top_k), hist);
    if (tau == -INFINITY) return false;
  }
  if (P.p_on) {
    uint64_t s = 0;
    for (int j = threadIdx.x; j < n; j += NT) {
      const float v = val[j];
      w[j] = (v >= tau) ? to_fixed(weight_ff(P, v, D.m), P.fp_shift) : 0ull;
      s += w[j];
    }
    s = block_sum_u64(k, s);  // (the block sum's barrier also publishes w[])
    const uint64_t znorm = P.k_on ? s : to_fixed(ff_from_double(zall), P.fp_shift);
    const uint64_t target = ceil_scale(P.top_p, znorm);
    if (s < target) {
      if (!P.k_on) return false;  // the nucleus is not inside the candidate window
      // rounding: the kept set's own mass falls short; keep it whole
    } else {
      tau = fmaxf(tau, list_select(k, val, n, w, target, hist));
    }
  }
  ff z = {0.0f, 0.0f};
  for (int j = threadIdx.x; j < n; j += NT)
    if (val[j] >= tau) z = ff_add(z, weight_ff(P, val[j], D.m));
  set_Z(D, block_sum_ff(k, z), 0.0f);
  D.tau = tau;
  D.list = 1;
  D.n = n;
  return true;
}

// Inverse-CDF draw over the p-list (index order), redundantly in every CTA.
__device__ int list_draw(const KP &P, Blk &k, const Lists &L, int n, const Dist &dt,
                         const Dist &dd, bool residual, float u, ff *Wout) {
  int ch = (n + NT - 1) / NT;
  ch |= 1;
  const int j0 = min(n, static_cast<int>(threadIdx.x) * ch), j1 = min(n, j0 + ch);
  ff s = {0.0f, 0.0f};
  int lastpos = -1;
  for (int j = j0; j < j1; ++j) {
    const ff wj = draw_weight_of(P, L.p_zp[j], L.p_zq[j], dt, dd, residual);
    if (wj.hi > 0.0f) lastpos = L.p_idx[j];
    s = ff_add(s, wj);
  }
  ff W;
  const ff pre = block_scan_ff(k, s, W);
  const int glast = block_max_i32(k, lastpos);
  *Wout = W;
  if (!(W.hi > 0.0f)) return -1;
  const ff target = ff_mul_f(W, u);
  if (threadIdx.x == 0) k.scal[8] = -1;
  __syncthreads();
  const ff b = ff_add(pre, s);
  if (!ff_lt(target, pre) && ff_lt(target, b)) {
    ff c = pre;
    int tok = -1;
    for (int j = j0; j < j1; ++j) {
      const ff wj = draw_weight_of(P, L.p_zp[j], L.p_zq[j], dt, dd, residual);
      if (wj.hi > 0.0f) tok = L.p_idx[j];
      c = ff_add(c, wj);
      if (ff_lt(target, c) && wj.hi > 0.0f) break;
    }
    k.scal[8] = tok;
  }
  __syncthreads();
  int tok = k.scal[8];
  __syncthreads();
  if (tok < 0) tok = glast;
  return tok;
}

// --------------------------------------------------------------- the kernel
template <typename E, bool VEC>
__global__ void __launch_bounds__(NT, 2) verify_kernel(const __grid_constant__ KP P) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ uint32_t xch[XSLOTS * XWORDS];
  __shared__ uint32_t gat[MAXC * XWORDS];
  __shared__ uint64_t red[NW * 4];
  __shared__ __align__(8) int32_t scal[16];
  __shared__ int wcnt[2 * NW];
  __shared__ int bandh[2 * (NBANDS + 1)];

  Blk k;
  k.xch = xch;
  k.gat = gat;
  k.red = red;
  k.scal = scal;
  k.C = cluster_size();
  k.rank = cluster_rank();
  k.slot = 0;

  const int b = blockIdx.x / k.C;
  const int lo = static_cast<int>(k.rank) * P.L;
  const int n = max(0, min(P.V, lo + P.L) - lo);
  E *st = reinterpret_cast<E *>(smem + P.off_stage_t);
  E *sd = reinterpret_cast<E *>(smem + P.off_stage_d);
  Lists Ls;
  Ls.p_idx = reinterpret_cast<int *>(smem + P.off_lp);
  Ls.p_zp = reinterpret_cast<float *>(Ls.p_idx + P.cap);
  Ls.p_zq = Ls.p_zp + P.cap;
  Ls.q_idx = reinterpret_cast<int *>(smem + P.off_lq);
  Ls.q_zq = reinterpret_cast<float *>(Ls.q_idx + P.cap);
  Ls.w = reinterpret_cast<uint64_t *>(smem + P.off_w);
  Ls.hist = reinterpret_cast<uint64_t *>(smem + P.off_hist);
  const E *tg = static_cast<const E *>(P.tgt);
  const E *dg = static_cast<const E *>(P.drf);

  int status = 0, acc = 0, next = -1;
  float resid = 0.0f;
#ifdef SV_PHASE_PROFILE
  long long t_ph_ = clock64();
#endif
  const int gb = P.gam ? P.gam[b] : P.gm;
  bool done = false;
  if (gb < 0 || gb > P.gm) {
    status = ST_BAD_GAMMA;
    done = true;
  }

  for (int i = 0; !done && i <= gb; ++i) {
    const bool bonus = (i == gb);
    const bool two = !P.greedy && !bonus;  // is the draft row needed?
    int x = -1;
    if (!bonus) {
      x = P.tok[static_cast<int64_t>(b) * P.gm + i];
      if (x < 0 || x >= P.V) status |= ST_BAD_TOKEN;
    }
    const float *ui = P.uni + static_cast<int64_t>(b) * P.u_row + static_cast<int64_t>(i) * P.u_pos;
    float u0 = 0.0f;
    if (two) {
      u0 = ui[P.u_acc];
      if (!(u0 >= 0.0f && u0 < 1.0f)) status |= ST_BAD_UNIFORM;
    }

    // ---- pass 1: HBM -> SMEM, statistics
    TStat a, c;
    a.init();
    c.init();
    const E *trow = tg + static_cast<int64_t>(b) * P.t_row + static_cast<int64_t>(i) * P.t_pos + lo;
    load_slice<E, VEC>(trow, st, n, lo, !P.greedy, a);
    if (two) {
      const E *drow = dg + static_cast<int64_t>(b) * P.d_row + static_cast<int64_t>(i) * P.d_pos + lo;
      load_slice<E, VEC>(drow, sd, n, lo, true, c);
    }
    // per-warp lower bound of the top-k threshold: r-th largest lane maximum
    float tht = -INFINITY, thd = -INFINITY;
    if (P.r_warp > 0) {
      float va = a.mx, vc = c.mx;
      const int lane = threadIdx.x & 31;
      for (int r = 0; r < P.r_warp; ++r) {
        const float ma = warp_max(va), mc = warp_max(vc);
        tht = ma;
        thd = mc;
        const uint32_t ba = __ballot_sync(0xffffffffu, va == ma);
        const uint32_t bc = __ballot_sync(0xffffffffu, vc == mc);
        if (lane == __ffs(ba) - 1) va = -INFINITY;
        if (lane == __ffs(bc) - 1) vc = -INFINITY;
      }
    }
    // block reduction of the statistics
    {
      float am = a.mx, cm = c.mx;
      int ai = a.mi;
      warp_argmax(am, ai);
      cm = warp_max(cm);
      const uint32_t af = warp_or(a.fl), cf = warp_or(c.fl);
      uint32_t *r = reinterpret_cast<uint32_t *>(red);
      const int w = threadIdx.x >> 5;
      if ((threadIdx.x & 31) == 0) {
        r[w * 8 + 0] = __float_as_uint(am);
        r[w * 8 + 1] = static_cast<uint32_t>(ai);
        r[w * 8 + 2] = af;
        r[w * 8 + 3] = __float_as_uint(cm);
        r[w * 8 + 4] = cf;
        r[w * 8 + 5] = __float_as_uint(tht);
        r[w * 8 + 6] = __float_as_uint(thd);
      }
      __syncthreads();
      uint32_t wd[7];
      if (threadIdx.x == 0) {
        float bm = -INFINITY, dm = -INFINITY, t1 = INFINITY, t2 = INFINITY;
        int bi = INT_MAX;
        uint32_t bf = 0, df = 0;
        for (int j = 0; j < NW; ++j) {
          const float v = __uint_as_float(r[j * 8 + 0]);
          const int vi = static_cast<int>(r[j * 8 + 1]);
          if (v > bm || (v == bm && vi < bi)) {
            bm = v;
            bi = vi;
          }
          bf |= r[j * 8 + 2];
          dm = fmaxf(dm, __uint_as_float(r[j * 8 + 3]));
          df |= r[j * 8 + 4];
          t1 = fminf(t1, __uint_as_float(r[j * 8 + 5]));
          t2 = fminf(t2, __uint_as_float(r[j * 8 + 6]));
        }
        wd[0] = __float_as_uint(bm);
        wd[1] = static_cast<uint32_t>(bi);
        wd[2] = bf;
        wd[3] = __float_as_uint(dm);
        wd[4] = df;
        wd[5] = __float_as_uint(t1);
        wd[6] = __float_as_uint(t2);
        for (int j = 0; j < 7; ++j) scal[j] = static_cast<int32_t>(wd[j]);
      }
      __syncthreads();
      for (int j = 0; j < 7; ++j) wd[j] = static_cast<uint32_t>(scal[j]);
      exchange(k, wd, 7);
    }
    SV_PHASE(0);  // load + pass-1 reduction + exchange
    // cluster-wide statistics (identical in every CTA)
    Dist dt, dd;
    int amax = INT_MAX;
    float thc_t = INFINITY, thc_d = INFINITY;
    {
      float bm = -INFINITY, dm = -INFINITY;
      uint32_t bf = 0, df = 0;
      for (uint32_t cc = 0; cc < k.C; ++cc) {
        const uint32_t *g = gat + cc * 7;
        const float v = __uint_as_float(g[0]);
        const int vi = static_cast<int>(g[1]);
        if (v > bm || (v == bm && vi < amax)) {
          bm = v;
          amax = vi;
        }
        bf |= g[2];
        dm = fmaxf(dm, __uint_as_float(g[3]));
        df |= g[4];
        thc_t = fminf(thc_t, __uint_as_float(g[5]));
        thc_d = fminf(thc_d, __uint_as_float(g[6]));
      }
      if (bf & F_BAD) status |= ST_BAD_LOGIT;
      if (!(bf & F_FINITE)) status |= ST_NO_FINITE;
      if (two) {
        if (df & F_BAD) status |= ST_BAD_LOGIT;
        if (!(df & F_FINITE)) status |= ST_NO_FINITE;
      }
      dt.m = bm;
      dd.m = dm;
      dt.tau = dd.tau = -INFINITY;
      dt.list = dd.list = 0;
      dt.n = dd.n = 0;
      set_Z(dt, ff{1.0f, 0.0f}, 0.0f);
      dd = dt;
      dd.m = dm;
    }
    if (status & ST_ERROR) break;

    if (P.greedy) {
      if (!bonus && amax == x) continue;
      acc = i;
      next = amax;
      done = true;
      break;
    }

    // ---- filters and normalisers (sampling)
    const bool filt = P.k_on || P.p_on;
    bool lt = false, ld = false;  // kept set held by the candidate list
    if (filt && P.cap > 0) {
      float ct = -INFINITY, cd = -INFINITY;
      double zall_t = 0.0, zall_d = 0.0;
      if (P.k_on) {
        ct = thc_t;  // <= the k-th largest logit (per-warp maxima bound)
        cd = thc_d;
      } else {
        // top-p alone: Z over the vocabulary, and a window deep enough to
        // hold the nucleus but small enough for the list (sampled estimate)
        int bt[NBANDS], bd[NBANDS];
        slice_Z_fast<E>(P, k, st, sd, n, dt, dd, two, true, zall_t, zall_d, bt, bd, bandh);
        const int lim = P.cap / (2 * SAMPLE_EVERY);
        int jt = -1, jd = -1;
        for (int j = 0; j < NBANDS; ++j) {
          if (bt[j] <= lim) jt = j;
          if (bd[j] <= lim) jd = j;
        }
        if (jt >= 0) ct = __fsub_rn(dt.m, __fmul_rn(kBandDepth[jt], P.T));
        if (jd >= 0) cd = __fsub_rn(dd.m, __fmul_rn(kBandDepth[jd], P.T));
      }
      const bool vt = ct > -INFINITY, vd = two && cd > -INFINITY;
      int tot_t, tot_d, base_t, base_d;
      count_pass<E>(k, st, sd, n, ct, cd, vt, vd, wcnt, tot_t, tot_d, base_t, base_d);
      uint32_t cw[2] = {static_cast<uint32_t>(tot_t), static_cast<uint32_t>(tot_d)};
      exchange(k, cw, 2);
      int off_t = 0, off_d = 0, all_t = 0, all_d = 0;
      for (uint32_t cc = 0; cc < k.C; ++cc) {
        if (cc < k.rank) {
          off_t += static_cast<int>(gat[cc * 2]);
          off_d += static_cast<int>(gat[cc * 2 + 1]);
        }
        all_t += static_cast<int>(gat[cc * 2]);
        all_d += static_cast<int>(gat[cc * 2 + 1]);
      }
      lt = vt && all_t <= P.cap;
      ld = vd && all_d <= P.cap;
      if (lt || ld) {
        write_pass<E>(k, Ls, st, sd, n, lo, ct, cd, lt, ld, two, off_t + base_t, off_d + base_d);
        cluster_sync();
        SV_PHASE(1);  // Z/bands + count + write lists
        if (lt) lt = list_dist(P, k, Ls.p_zp, all_t, dt, Ls.w, Ls.hist, zall_t);
        if (ld) ld = list_dist(P, k, Ls.q_zq, all_d, dd, Ls.w, Ls.hist, zall_d);
      }
    }
    SV_PHASE(2);  // list selection
    const bool need_t = !lt, need_d = two && !ld;
    if (filt && (need_t || need_d)) {
      // exact slice-wide selection for the tensors without a list
      if (P.k_on) slice_bisect<E>(P, k, st, sd, n, dt, dd, need_t, need_d, false);
      if (P.p_on) slice_bisect<E>(P, k, st, sd, n, dt, dd, need_t, need_d, true);
      slice_Z_exact<E>(P, k, st, sd, n, dt, dd, need_t, need_d);
      if (P.diag && k.rank == 0 && threadIdx.x == 0) atomicAdd(P.diag + 0, 1u);
    } else if (!filt) {
      double z0, z1;
      slice_Z_fast<E>(P, k, st, sd, n, dt, dd, two, false, z0, z1, nullptr, nullptr, bandh);
    }

    SV_PHASE(3);  // slice fallback / fast Z
    if (bonus) {
      float u1 = ui[P.u_draw];
      if (!(u1 >= 0.0f && u1 < 1.0f)) {
        status |= ST_BAD_UNIFORM;
        break;
      }
      ff W;
      if (lt) {
        next = list_draw(P, k, Ls, dt.n, dt, dd, false, u1, &W);
      } else {
        float Wf;
        next = slice_draw_fast<E>(P, k, st, sd, n, lo, dt, dd, false, u1, &Wf);
        if (next < 0) {  // uncertain: exact redraw
          if (!filt) slice_Z_exact<E>(P, k, st, sd, n, dt, dd, true, false);
          next = slice_draw<E>(P, k, st, sd, n, lo, dt, dd, false, u1, &W);
          if (P.diag && k.rank == 0 && threadIdx.x == 0) atomicAdd(P.diag + 1, 1u);
        }
      }
      acc = gb;
      done = true;
      break;
    }

    // ---- acceptance test: u < p(x)/q(x)
    const int64_t toff = static_cast<int64_t>(b) * P.t_row + static_cast<int64_t>(i) * P.t_pos + x;
    const int64_t doff = static_cast<int64_t>(b) * P.d_row + static_cast<int64_t>(i) * P.d_pos + x;
    const float zx = Elem<E>::get(tg[toff]);
    const float wx = Elem<E>::get(dg[doff]);
    const bool kp = zx >= dt.tau && zx != -INFINITY;
    const bool kq = wx >= dd.tau && wx != -INFINITY;
    const ff yp = scaled_gap(P, zx, dt.m), yq = scaled_gap(P, wx, dd.m);
    bool accept;
    if (kq) {
      // p(x)/q(x) = e^{yp - yq} * Zq / Zp: one exponential, no underflow
      ff ratio = {0.0f, 0.0f};
      if (kp) ratio = ff_mul(ff_exp(ff_sub(yp, yq)), ff_mul(dd.Z, dt.rZ));
      accept = ff_lt(ff_make(u0), ratio);
    } else {
      status |= ST_Q_ZERO;
      accept = kp;
    }
    if (k.rank == 0 && threadIdx.x == 0) {
      if (P.p_dbg) {
        const ff px = kp ? ff_mul(ff_exp(yp), dt.rZ) : ff{0.0f, 0.0f};
        P.p_dbg[static_cast<int64_t>(b) * P.gm + i] = px.hi + px.lo;
      }
      if (P.q_dbg) {
        const ff qx = kq ? ff_mul(ff_exp(yq), dd.rZ) : ff{0.0f, 0.0f};
        P.q_dbg[static_cast<int64_t>(b) * P.gm + i] = qx.hi + qx.lo;
      }
    }
    if (accept) continue;

    SV_PHASE(4);  // acceptance
    // ---- first rejection: draw from norm(max(0, p - q))
    const float u1 = ui[P.u_draw];
    if (!(u1 >= 0.0f && u1 < 1.0f)) {
      status |= ST_BAD_UNIFORM;
      break;
    }
    ff W;
    int tok;
    if (lt) {
      tok = list_draw(P, k, Ls, dt.n, dt, dd, true, u1, &W);
      resid = W.hi + W.lo;  // residual mass sum max(0, p - q)
      if (tok < 0) tok = list_draw(P, k, Ls, dt.n, dt, dd, false, u1, &W);
    } else {
      float Wf;
      tok = slice_draw_fast<E>(P, k, st, sd, n, lo, dt, dd, true, u1, &Wf);
      resid = Wf;
      if (tok < 0) {  // uncertain, or an (almost) empty residual: exact redraw
        if (!filt) slice_Z_exact<E>(P, k, st, sd, n, dt, dd, true, !ld);
        tok = slice_draw<E>(P, k, st, sd, n, lo, dt, dd, true, u1, &W);
        resid = W.hi + W.lo;
        if (tok < 0) tok = slice_draw<E>(P, k, st, sd, n, lo, dt, dd, false, u1, &W);
        if (P.diag && k.rank == 0 && threadIdx.x == 0) atomicAdd(P.diag + 1, 1u);
      }
    }
    acc = i;
    next = tok;
    done = true;
    break;
  }
  SV_PHASE(5);  // draw (or greedy exit)
  if (status & ST_ERROR) {
    acc = 0;
    next = -1;
  }
  if (k.rank == 0 && threadIdx.x == 0) {
    if (P.acc) P.acc[b] = acc;
    P.next[b] = next;
    if (P.st_dbg) P.st_dbg[b] = status;
    if (P.res_dbg) P.res_dbg[b] = (status & ST_ERROR) ? 0.0f : resid;
  }
  cluster_sync();  // no CTA leaves while a peer may still read its shared memory
}

// Debug p/q outputs are NaN unless a position is evaluated.
__global__ void fill_nan_kernel(float *p, int64_t n) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) p[i] = __int_as_float(0x7fc00000);
}

}  // namespace sv

// ====================================================================== host
namespace {

using namespace sv;

constexpr size_t kStageBudget = 96 * 1024;  // bytes of staged logits per CTA
constexpr size_t kMaxSmem = 200 * 1024;      // dynamic shared memory per CTA
constexpr int kDiagWords = 4;

int sm_count() {
  static int n = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  });
  return n;
}

template <typename E, bool VEC>
cudaError_t prepare_kernel() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(verify_kernel<E, VEC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kMaxSmem));
  });
  return err;
}

template <typename E, bool VEC>
int active_clusters(int C, size_t smem) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(C) * 64u, 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = static_cast<unsigned>(C);
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, verify_kernel<E, VEC>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <typename E, bool VEC>
spec_status launch_one(const KP &kp, int C, size_t smem, cudaStream_t stream) {
  if (prepare_kernel<E, VEC>() != cudaSuccess) return SPEC_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(kp.B) * static_cast<unsigned>(C), 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = static_cast<unsigned>(C);
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, verify_kernel<E, VEC>, kp);
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

inline int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

struct Plan {
  int C = 1;
  int L = 0;
  int cap = 0;
  int64_t off_lp = 0, off_lq = 0, off_w = 0, off_hist = 0;
  size_t smem = 0;
  bool vec = false;
};

// Shared-memory plan for a given cluster size.
Plan plan_for(const spec_params &p, bool sampling, int es, bool aligned, int C) {
  Plan pl;
  pl.C = C;
  pl.L = static_cast<int>(align_up((static_cast<int64_t>(p.V) + C - 1) / C, 8));
  pl.vec = aligned;
  const bool filt = sampling && ((p.top_k > 0 && p.top_k < p.V) || p.top_p < 1.0f);
  pl.cap = !filt ? 0 : (p.list_capacity > 0 ? p.list_capacity
                                           : ((p.top_k > 0 && p.top_k < p.V) ? 1024 : 2048));
  const int64_t stage = sampling ? 2 * align_up(static_cast<int64_t>(pl.L) * es, 16) : 0;
  pl.off_lp = stage;
  pl.off_lq = pl.off_lp + 12ll * pl.cap;
  pl.off_w = align_up(pl.off_lq + 8ll * pl.cap, 16);
  pl.off_hist = pl.off_w + 8ll * pl.cap;
  pl.smem = static_cast<size_t>(pl.cap ? pl.off_hist + 8ll * NBINS : stage);
  return pl;
}

// Cluster size: the one that minimises (waves of resident clusters) x (slice
// length + a fixed per-position cost), among those whose slices fit.
template <typename E, bool VEC>
Plan choose_plan(const spec_params &p, bool sampling, int es, bool aligned) {
  if (p.cluster_size) return plan_for(p, sampling, es, aligned, p.cluster_size);
  if (prepare_kernel<E, VEC>() != cudaSuccess) return plan_for(p, sampling, es, aligned, MAXC);
  Plan best;
  double best_cost = 0.0;
  bool have = false;
  for (int C = 1; C <= MAXC; C *= 2) {
    const Plan pl = plan_for(p, sampling, es, aligned, C);
    if (pl.smem > kMaxSmem) continue;
    const int act = active_clusters<E, VEC>(C, pl.smem);
    if (act <= 0) continue;
    const int64_t waves = (static_cast<int64_t>(p.B) + act - 1) / act;
    const double cost = static_cast<double>(waves) * (static_cast<double>(pl.L) + 3000.0);
    if (!have || cost < best_cost) {
      best = pl;
      best_cost = cost;
      have = true;
    }
  }
  return have ? best : plan_for(p, sampling, es, aligned, MAXC);
}

// Plans are cached per problem shape (the occupancy queries cost host time).
Plan cached_plan(const spec_params &p, bool sampling, int es, bool aligned) {
  using Key = std::tuple<int, int, int, int, int, int, int, int, int>;
  static std::mutex mu;
  static std::map<Key, Plan> cache;
  const bool k_on = p.top_k > 0 && p.top_k < p.V;
  const Key key{p.B, p.V, p.dtype, sampling ? 1 : 0, aligned ? 1 : 0, p.cluster_size,
                p.list_capacity, k_on ? 1 : 0, p.top_p < 1.0f ? 1 : 0};
  {
    std::lock_guard<std::mutex> g(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  Plan pl;
  if (p.dtype == SPEC_F32)
    pl = aligned ? choose_plan<float, true>(p, sampling, es, aligned)
                 : choose_plan<float, false>(p, sampling, es, aligned);
  else
    pl = aligned ? choose_plan<uint16_t, true>(p, sampling, es, aligned)
                 : choose_plan<uint16_t, false>(p, sampling, es, aligned);
  std::lock_guard<std::mutex> g(mu);
  if (cache.size() > 4096) cache.clear();
  cache[key] = pl;
  return pl;
}

spec_status run_verify(const void *target, const void *draft, const int32_t *tokens,
                       const float *uniforms, const spec_params *pp, int32_t *acc,
                       int32_t *next, const spec_debug *dbg, void *ws, size_t ws_bytes,
                       cudaStream_t stream, bool sample_mode) {
  if (!pp) return SPEC_ERR_INVALID_ARG;
  const spec_params p = *pp;
  if (p.B < 0 || p.gamma_max < 0 || p.V < 1 || p.V > (1 << 24)) return SPEC_ERR_INVALID_ARG;
  if (p.B == 0) return SPEC_OK;
  if (p.dtype != SPEC_F32 && p.dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (!std::isfinite(p.temperature) || p.temperature < 0.0f) return SPEC_ERR_INVALID_ARG;
  if (p.temperature > 0.0f && p.temperature < 1e-30f) return SPEC_ERR_INVALID_ARG;
  if (!(p.top_p > 0.0f)) return SPEC_ERR_INVALID_ARG;  // also NaN
  if (p.flags != 0) return SPEC_ERR_INVALID_ARG;
  if (p.cluster_size != 0 && p.cluster_size != 1 && p.cluster_size != 2 &&
      p.cluster_size != 4 && p.cluster_size != 8)
    return SPEC_ERR_INVALID_ARG;
  if (p.list_capacity < 0) return SPEC_ERR_INVALID_ARG;
  if (p.target_pos_stride < 0 || p.target_row_stride < 0 || p.draft_pos_stride < 0 ||
      p.draft_row_stride < 0)
    return SPEC_ERR_INVALID_ARG;
  if (static_cast<int64_t>(p.B) * 8 > INT32_MAX) return SPEC_ERR_INVALID_ARG;
  const bool greedy = p.temperature == 0.0f;
  if (!target || !next) return SPEC_ERR_INVALID_ARG;
  if (!sample_mode) {
    if (!acc) return SPEC_ERR_INVALID_ARG;
    if (p.gamma_max > 0 && !tokens) return SPEC_ERR_INVALID_ARG;
    if (!greedy && p.gamma_max > 0 && !draft) return SPEC_ERR_INVALID_ARG;
  } else if (p.gamma_max != 0) {
    return SPEC_ERR_INVALID_ARG;
  }
  if (!greedy && !uniforms) return SPEC_ERR_INVALID_ARG;
  if (ws && (ws_bytes < kDiagWords * sizeof(uint32_t) ||
             (reinterpret_cast<uintptr_t>(ws) & 15) != 0))
    return SPEC_ERR_WORKSPACE;

  const int es = p.dtype == SPEC_F32 ? 4 : 2;
  const bool sampling = !greedy;
  const bool aligned =
      (reinterpret_cast<uintptr_t>(target) & 15) == 0 &&
      (!draft || (reinterpret_cast<uintptr_t>(draft) & 15) == 0) &&
      (p.target_pos_stride * es) % 16 == 0 && (p.target_row_stride * es) % 16 == 0 &&
      (p.draft_pos_stride * es) % 16 == 0 && (p.draft_row_stride * es) % 16 == 0;
  const Plan pl = cached_plan(p, sampling, es, aligned);
  if (pl.smem > kMaxSmem) return SPEC_ERR_UNSUPPORTED;  // vocabulary too large to stage

  KP kp;
  std::memset(&kp, 0, sizeof kp);
  kp.tgt = target;
  kp.drf = draft ? draft : target;
  kp.tok = tokens;
  kp.uni = uniforms;
  kp.gam = sample_mode ? nullptr : p.gamma_per_row;
  kp.t_pos = p.target_pos_stride;
  kp.t_row = p.target_row_stride;
  kp.d_pos = p.draft_pos_stride;
  kp.d_row = p.draft_row_stride;
  if (sample_mode) {
    kp.u_row = 1;
    kp.u_pos = 0;
    kp.u_acc = 0;
    kp.u_draw = 0;
  } else {
    kp.u_row = 2 * (static_cast<int64_t>(p.gamma_max) + 1);
    kp.u_pos = 2;
    kp.u_acc = 0;
    kp.u_draw = 1;
  }
  kp.B = p.B;
  kp.gm = p.gamma_max;
  kp.V = p.V;
  kp.L = pl.L;
  kp.greedy = greedy ? 1 : 0;
  if (sampling) {
    const double invT = 1.0 / static_cast<double>(p.temperature);
    kp.invT_hi = static_cast<float>(invT);
    kp.invT_lo = static_cast<float>(invT - static_cast<double>(kp.invT_hi));
    kp.c2 = static_cast<float>(1.4426950408889634 * invT);
    kp.T = p.temperature;
  }
  kp.k_on = (p.top_k > 0 && p.top_k < p.V) ? 1 : 0;
  kp.top_k = p.top_k;
  kp.p_on = p.top_p < 1.0f ? 1 : 0;
  kp.top_p = p.top_p;
  kp.cap = pl.cap;
  {
    int bits = 0;
    while ((1ll << bits) <= static_cast<int64_t>(p.V)) ++bits;
    kp.fp_shift = 62 - bits;
  }
  kp.r_warp = 0;
  if (kp.k_on && pl.cap > 0) {
    const int r = (p.top_k + pl.C * NW - 1) / (pl.C * NW);
    kp.r_warp = r <= 32 ? r : 0;  // 0: no bound, the exact slice selection is used
  }
  kp.acc = acc;
  kp.next = next;
  if (dbg) {
    kp.p_dbg = dbg->p_draft;
    kp.q_dbg = dbg->q_draft;
    kp.res_dbg = dbg->residual_mass;
    kp.st_dbg = dbg->row_status;
  }
  kp.diag = static_cast<unsigned int *>(ws);
  kp.off_stage_t = 0;
  kp.off_stage_d = static_cast<uint32_t>(align_up(static_cast<int64_t>(pl.L) * es, 16));
  kp.off_lp = static_cast<uint32_t>(pl.off_lp);
  kp.off_lq = static_cast<uint32_t>(pl.off_lq);
  kp.off_w = static_cast<uint32_t>(pl.off_w);
  kp.off_hist = static_cast<uint32_t>(pl.off_hist);

  if (dbg && p.gamma_max > 0) {
    const int64_t nn = static_cast<int64_t>(p.B) * p.gamma_max;
    const unsigned blocks = static_cast<unsigned>((nn + 255) / 256);
    if (dbg->p_draft) fill_nan_kernel<<<blocks, 256, 0, stream>>>(dbg->p_draft, nn);
    if (dbg->q_draft) fill_nan_kernel<<<blocks, 256, 0, stream>>>(dbg->q_draft, nn);
    if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  }
  if (p.dtype == SPEC_F32)
    return pl.vec ? launch_one<float, true>(kp, pl.C, pl.smem, stream)
                  : launch_one<float, false>(kp, pl.C, pl.smem, stream);
  return pl.vec ? launch_one<uint16_t, true>(kp, pl.C, pl.smem, stream)
                : launch_one<uint16_t, false>(kp, pl.C, pl.smem, stream);
}

}  // namespace

#ifdef SV_PHASE_PROFILE
extern "C" int sv_phase_read(unsigned long long *host, int reset) {
  if (cudaMemcpyFromSymbol(host, sv_phase_cycles, 16 * sizeof(unsigned long long)) != cudaSuccess)
    return 1;
  if (reset) {
    unsigned long long z[16] = {0};
    if (cudaMemcpyToSymbol(sv_phase_cycles, z, sizeof z) != cudaSuccess) return 1;
  }
  return 0;
}
#endif

extern "C" {

size_t spec_verify_workspace_size(const spec_params *) { return kDiagWords * sizeof(uint32_t); }

spec_status spec_verify(const void *target_logits, const void *draft_logits,
                        const int32_t *draft_tokens, const float *uniforms,
                        const spec_params *params, int32_t *accepted_len, int32_t *next_token,
                        const spec_debug *debug, void *workspace, size_t workspace_bytes,
                        void *stream) {
  return run_verify(target_logits, draft_logits, draft_tokens, uniforms, params, accepted_len,
                    next_token, debug, workspace, workspace_bytes,
                    static_cast<cudaStream_t>(stream), false);
}

spec_status spec_sample(const void *logits, const float *u, const spec_params *params,
                        int32_t *tokens, int32_t *row_status, void *stream) {
  spec_debug d = {nullptr, nullptr, nullptr, row_status};
  return run_verify(logits, nullptr, nullptr, u, params, nullptr, tokens, &d, nullptr, 0,
                    static_cast<cudaStream_t>(stream), true);
}

const char *spec_status_string(spec_status s) {
  switch (s) {
    case SPEC_OK: return "SPEC_OK";
    case SPEC_ERR_INVALID_ARG: return "SPEC_ERR_INVALID_ARG: invalid parameter or pointer";
    case SPEC_ERR_UNSUPPORTED: return "SPEC_ERR_UNSUPPORTED: not supported by this build or device";
    case SPEC_ERR_WORKSPACE: return "SPEC_ERR_WORKSPACE: workspace too small or misaligned";
    case SPEC_ERR_CUDA: return "SPEC_ERR_CUDA: a CUDA runtime call failed";
  }
  return "unknown spec_status";
}

spec_status spec_read_diagnostics(const void *workspace, uint32_t *counters, int n,
                                  void *stream) {
  if (!workspace || !counters || n < 0) return SPEC_ERR_INVALID_ARG;
  const int m = n < kDiagWords ? n : kDiagWords;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(counters, workspace, m * sizeof(uint32_t), cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return SPEC_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SPEC_ERR_CUDA;
  for (int i = m; i < n; ++i) counters[i] = 0;
  return SPEC_OK;
}

}  // extern "C"
