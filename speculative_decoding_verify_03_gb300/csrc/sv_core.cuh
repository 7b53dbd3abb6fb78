// sv_core.cuh -- device code shared by the verify kernels (sm_103a): kernel
// parameters, per-position distributions, element I/O and staging, block and
// group reductions, the weights e^{(z-m)/T} in single precision (with error
// bounds) and float-float, and the exact slice-wide selection, normaliser
// and inverse-CDF draw.  The slice routines read their elements through
// plain pointers, so a slice may be staged in shared memory or read in place
// from global memory (a one-CTA "cluster").
#pragma once

#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <type_traits>

#include "spec_verify.h"
#include "sv_common.cuh"

namespace sv {

constexpr int MAXNW = 8;          // warps per CTA at most
constexpr int MAXC = 8;           // largest cluster
constexpr int XSLOTS = 4;         // rotating exchange slots
constexpr int XWORDS = 48;        // 32-bit words per exchange slot
constexpr int NBINS = 256;        // histogram bins of the list selection
constexpr int NBANDS = 16;        // depth bands of the top-p candidate window
constexpr int SAMPLE_EVERY = 8;   // band counts look at every 8th element
constexpr int NCH = 1;            // bulk-copy chunks per tensor and position
constexpr int FP_SHIFT = 31;      // masses in fixed point: round(e * 2^31)
constexpr int SMALL_LIST = 256;   // lists up to this size: all-pairs selection
constexpr int SORT_MAX = 512;     // lists up to this size: sorted selection
constexpr int SMALL_SORTED = 128; // ... from this size up (shorter: all-pairs)
constexpr int TOPR = 4;           // per-warp top lane maxima for the top-k bound
constexpr uint32_t kWaitPolls = 1u << 22;  // bounded mbarrier waits

constexpr uint32_t F_BAD = 1u, F_FINITE = 2u, F_TIMEOUT = 4u;  // pass-1 flags

enum : int {
  ST_BAD_TOKEN = SPEC_ROW_BAD_TOKEN,
  ST_BAD_LOGIT = SPEC_ROW_BAD_LOGIT,
  ST_NO_FINITE = SPEC_ROW_NO_FINITE,
  ST_Q_ZERO = SPEC_ROW_Q_ZERO,
  ST_BAD_GAMMA = SPEC_ROW_BAD_GAMMA,
  ST_BAD_UNIFORM = SPEC_ROW_BAD_UNIFORM,
  ST_TIMEOUT = SPEC_ROW_WAIT_TIMEOUT,
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
  int32_t kc;                // per-CTA rank of the top-k lower bound (0: none)
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
  ff Z;        // normaliser: compensated single precision, or float-float if exact
  ff rZ;       // 1 / Z in float-float (valid when exact)
  float rzf;   // 1 / Z in single precision
  float zerr;  // bound of the relative error of Z and rzf (0 when exact)
  int exact;   // Z is float-float accurate
  int list;    // 1: the kept set is inside the candidate list
  int n;       // list length
};

// Every logit kept, maximum m, normaliser 1 until computed.
__device__ __forceinline__ void dist_init(Dist &D, float m) {
  D.m = m;
  D.tau = -INFINITY;
  D.Z = D.rZ = ff{1.0f, 0.0f};
  D.rzf = 1.0f;
  D.zerr = 0.0f;
  D.exact = 0;
  D.list = 0;
  D.n = 0;
}

// Fast normaliser with its relative error bound (the reciprocal of the high
// part adds at most 2^-23).
__device__ __forceinline__ void set_Zf(Dist &D, ff Z, float zerr) {
  D.Z = Z;
  D.rzf = __frcp_rn(Z.hi);
  D.zerr = __fadd_rn(zerr, 1.2e-7f);
  D.exact = 0;
}
// Float-float normaliser (exact paths).
static __device__ __forceinline__ void set_Zx(Dist &D, ff Z) {
  D.Z = Z;
  D.rZ = ff_div(ff{1.0f, 0.0f}, Z);
  D.rzf = D.rZ.hi;
  D.zerr = 0.0f;
  D.exact = 1;
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

// Raw values (-0 kept): comparisons and exponentials do not distinguish
// -0 from +0; only the order-preserving keys need the canonical form.
template <typename E>
__device__ __forceinline__ void unpack(const uint4 &v, float *out);
template <>
__device__ __forceinline__ void unpack<float>(const uint4 &v, float *o) {
  o[0] = __uint_as_float(v.x);
  o[1] = __uint_as_float(v.y);
  o[2] = __uint_as_float(v.z);
  o[3] = __uint_as_float(v.w);
}
template <>
__device__ __forceinline__ void unpack<uint16_t>(const uint4 &v, float *o) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    o[2 * j] = __uint_as_float(w[j] << 16);
    o[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
  }
}
__device__ __forceinline__ float raw_of(float v) { return v; }
__device__ __forceinline__ float raw_of(uint16_t v) { return bf16_to_f32(v); }

template <typename E>
__device__ __forceinline__ float stage_raw(const E *s, int j) {
  return raw_of(s[j]);
}
template <typename E>
__device__ __forceinline__ float stage_get(const E *s, int j) {
  return Elem<E>::get(s[j]);
}

// Pass-1 statistics of one thread: the maximum (NaN ignored), a NaN flag,
// and with ARG the first index of the maximum (greedy mode).
template <bool ARG>
struct TStat {
  float mx;
  float mxn;  // without ARG: the NaN-propagating maximum (NaN iff a NaN was seen)
  int mi;
  uint32_t nan, to;
  __device__ void init() {
    mx = -INFINITY;
    mxn = -INFINITY;
    mi = INT_MAX;
    nan = 0;
    to = 0;
  }
  __device__ __forceinline__ void add(float z, int idx) {
    if (ARG) {
      nan |= (z != z) ? 1u : 0u;
      if (z > mx) {
        mx = z;
        mi = idx;
      }
    } else {
      mx = fmaxf(mx, z);
      mxn = max_nan(mxn, z);
    }
  }
  // NaN or +inf: bad; nothing above -inf: no finite logit
  __device__ __forceinline__ uint32_t flags() const {
    const bool any_nan = ARG ? nan != 0u : mxn != mxn;
    return ((any_nan || mx == INFINITY) ? F_BAD : 0u) | (mx > -INFINITY ? F_FINITE : 0u) |
           (to ? F_TIMEOUT : 0u);
  }
};

// Pass-1 statistics of one thread for top-p without top-k: the maximum, the
// second largest value seen (with the maximum: two elements >= it), the
// NaN-propagating maximum and the timeout flag.  A NaN makes the row an
// error row, so the second largest need not be exact then.
struct TStat2 {
  float mx, mx2, mxn;
  int mi;  // unused (no argmax)
  uint32_t to;
  __device__ void init() {
    mx = -INFINITY;
    mx2 = -INFINITY;
    mxn = -INFINITY;
    mi = INT_MAX;
    to = 0;
  }
  __device__ __forceinline__ void add(float z, int) {
    mx2 = fmaxf(mx2, fminf(mx, z));
    mx = fmaxf(mx, z);
    mxn = max_nan(mxn, z);
  }
  __device__ __forceinline__ uint32_t flags() const {
    return ((mxn != mxn || mx == INFINITY) ? F_BAD : 0u) | (mx > -INFINITY ? F_FINITE : 0u) |
           (to ? F_TIMEOUT : 0u);
  }
};

// Bulk-copy chunk boundaries (in elements) of a slice of n elements: the
// 16-byte-aligned body [0, nb) in NCH pieces; the tail [nb, n) is loaded by
// threads.
template <typename E>
struct Chunks {
  int ce[NCH + 1];
  int nb;
  __device__ void make(int n) {
    constexpr int EPV = Elem<E>::kPerVec;
    nb = (n / EPV) * EPV;
    const int per = ((nb + NCH - 1) / NCH + EPV - 1) / EPV * EPV;
#pragma unroll
    for (int c = 0; c <= NCH; ++c) ce[c] = min(nb, c * per);
  }
};

// Thread 0: start the bulk copies of one slice.
template <typename E>
__device__ __forceinline__ void issue_slice(const E *g, E *s, const Chunks<E> &ch,
                                            uint64_t *bars) {
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    const int a = ch.ce[c], b = ch.ce[c + 1];
    if (b > a) {
      const uint32_t bytes = static_cast<uint32_t>(b - a) * sizeof(E);
      mbar_arrive_tx(&bars[c], bytes);
      bulk_g2s(s + a, g + a, bytes, &bars[c]);
    }
  }
}

// Wait for each chunk of a staged slice and fold it into the statistics,
// then load and fold the ragged tail.  Every thread of the CTA calls it.
// Each thread visits its elements in increasing index order ("first index
// of the maximum" needs no tie test).
template <typename E, typename ST>
__device__ __forceinline__ void scan_slice(const E *g, E *s, const Chunks<E> &ch, int n,
                                           int lo, uint64_t *bars, uint32_t parity, ST &st) {
  constexpr int EPV = Elem<E>::kPerVec;
  const uint4 *s4 = reinterpret_cast<const uint4 *>(s);
#pragma unroll 1
  for (int c = 0; c < NCH; ++c) {
    const int a = ch.ce[c], b = ch.ce[c + 1];
    if (b <= a) continue;
    // one thread waits for the chunk; the block waits on the CTA barrier,
    // which also orders the chunk's shared-memory contents for every thread
    if (threadIdx.x == 0 && !mbar_wait_sleep(&bars[c], parity, kWaitPolls)) st.to = 1;
    __syncthreads();
    for (int v = a / EPV + static_cast<int>(threadIdx.x); v < b / EPV;
         v += static_cast<int>(blockDim.x)) {
      const uint4 x = s4[v];
      float f[EPV];
      unpack<E>(x, f);
#pragma unroll
      for (int j = 0; j < EPV; ++j) st.add(f[j], lo + v * EPV + j);
    }
  }
  for (int j = ch.nb + static_cast<int>(threadIdx.x); j < n; j += static_cast<int>(blockDim.x)) {
    const E e = g[j];
    s[j] = e;
    st.add(raw_of(e), lo + j);
  }
}

// Unaligned rows: plain loads into shared memory.
template <typename E, typename ST>
__device__ __forceinline__ void load_slice_plain(const E *__restrict__ g, E *s, int n, int lo,
                                                 ST &st) {
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const E e = g[j];
    s[j] = e;
    st.add(raw_of(e), lo + j);
  }
}

// NaN-propagating maximum of one 16-byte vector of logits: 8 bfloat16 values
// through packed bf16x2 maxima, or 4 floats.
template <typename E>
__device__ __forceinline__ float vec_max_nan(const uint4 &v);
template <>
__device__ __forceinline__ float vec_max_nan<float>(const uint4 &v) {
  return max_nan(max_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                 max_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
}
template <>
__device__ __forceinline__ float vec_max_nan<uint16_t>(const uint4 &v) {
  uint32_t a, b;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(a) : "r"(v.x), "r"(v.y));
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(b) : "r"(v.z), "r"(v.w));
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(a) : "r"(a), "r"(b));
  return max_nan(__uint_as_float(a << 16), __uint_as_float(a & 0xffff0000u));
}

// Pass 1 of a staged slice for top-p alone, per 16-byte vector: the
// vector's NaN-propagating maximum, and per thread the two largest vector
// maxima (two distinct elements: a thread holds at least two elements >=
// its second value), a NaN flag and the maximum.  Waits on the chunk's
// bulk copy like scan_slice; the ragged tail is loaded by threads.
template <typename E>
__device__ __forceinline__ void scan_slice_top2(const E *g, E *s, const Chunks<E> &ch, int n,
                                                uint64_t *bars, uint32_t parity, TStat2 &st) {
  constexpr int EPV = Elem<E>::kPerVec;
  const uint4 *s4 = reinterpret_cast<const uint4 *>(s);
#pragma unroll 1
  for (int c = 0; c < NCH; ++c) {
    const int a = ch.ce[c], b = ch.ce[c + 1];
    if (b <= a) continue;
    if (threadIdx.x == 0 && !mbar_wait_sleep(&bars[c], parity, kWaitPolls)) st.to = 1;
    __syncthreads();
    for (int v = a / EPV + static_cast<int>(threadIdx.x); v < b / EPV;
         v += static_cast<int>(blockDim.x)) {
      const float m = vec_max_nan<E>(s4[v]);
      st.mxn = max_nan(st.mxn, m);
      st.mx2 = fmaxf(st.mx2, fminf(st.mx, m));
      st.mx = fmaxf(st.mx, m);
    }
  }
  for (int j = ch.nb + static_cast<int>(threadIdx.x); j < n; j += static_cast<int>(blockDim.x)) {
    const E e = g[j];
    s[j] = e;
    st.add(raw_of(e), j);
  }
}

// -------------------------------------------------------------- the block
struct Blk {
  uint32_t *xch;  // [XSLOTS][XWORDS] own exchange slots
  uint32_t *gat;  // [MAXC * XWORDS] gathered peer words
  uint64_t *red;  // [MAXNW * 4] reduction scratch
  int32_t *scal;  // misc scalars [32]
  uint32_t C, rank;
  int slot, nt, nw;
};

__device__ __forceinline__ uint32_t *xslot(Blk &k) { return k.xch + k.slot * XWORDS; }

// The words of this CTA's current slot (written before the call) are
// published: synchronise the cluster, gather every CTA's first nw words into
// gat[c * nw + j].  All threads call it.
__device__ __forceinline__ void xsync(Blk &k, int nw) {
  if (k.C == 1) {  // a lone CTA: its own slot, no cluster barrier
    __syncthreads();
    for (int t = threadIdx.x; t < nw; t += k.nt) k.gat[t] = k.xch[k.slot * XWORDS + t];
    __syncthreads();
    k.slot = (k.slot + 1) % XSLOTS;
    return;
  }
  cluster_sync();
  for (int t = threadIdx.x; t < static_cast<int>(k.C) * nw; t += k.nt) {
    const uint32_t peer = t / nw, w = t % nw;
    k.gat[t] = dsmem_ld_u32(dsmem_addr(smem_u32(k.xch + k.slot * XWORDS + w), peer));
  }
  __syncthreads();
  k.slot = (k.slot + 1) % XSLOTS;
}
// Convenience: every thread holds the same words[]; publish and gather.
__device__ __forceinline__ void exchange(Blk &k, const uint32_t *words, int nw) {
  if (static_cast<int>(threadIdx.x) < nw) xslot(k)[threadIdx.x] = words[threadIdx.x];
  xsync(k, nw);
}

__device__ __forceinline__ uint64_t gat_u64(const Blk &k, int c, int nw, int w) {
  return static_cast<uint64_t>(k.gat[c * nw + w]) |
         (static_cast<uint64_t>(k.gat[c * nw + w + 1]) << 32);
}
__device__ __forceinline__ void put_u64(uint32_t *w, uint64_t u) {
  w[0] = static_cast<uint32_t>(u);
  w[1] = static_cast<uint32_t>(u >> 32);
}

// Thread groups: the whole block (barrier 0) or half of it (named barriers
// 1 and 2), so that the p and q candidate lists are processed concurrently.
struct Grp {
  int t, n, bar;
  uint64_t *red;  // [MAXNW * 2]
  int32_t *sc;    // [8]
};
__device__ __forceinline__ void gsync(const Grp &g) {
  if (g.bar)
    named_sync(g.bar, g.n);
  else
    __syncthreads();
}
__device__ __forceinline__ Grp whole_block(const Blk &k) {
  Grp g;
  g.t = threadIdx.x;
  g.n = k.nt;
  g.bar = 0;
  g.red = k.red;
  g.sc = k.scal + 16;
  return g;
}

// Group reductions in a fixed order (deterministic); all members get the result.
__device__ __forceinline__ uint64_t g_sum_u64(const Grp &g, uint64_t v) {
  v = warp_sum_u64(v);
  if ((g.t & 31) == 0) g.red[g.t >> 5] = v;
  gsync(g);
  uint64_t s = 0;
  for (int w = 0; w < g.n / 32; ++w) s += g.red[w];
  gsync(g);
  return s;
}
__device__ __forceinline__ ff warp_sum_ff(ff v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    ff u;
    u.hi = __shfl_xor_sync(0xffffffffu, v.hi, o);
    u.lo = __shfl_xor_sync(0xffffffffu, v.lo, o);
    v = ff_add(v, u);  // commutative: both lanes of a pair get the same sum
  }
  return v;
}
__device__ __forceinline__ ff g_sum_ff(const Grp &g, ff v) {
  v = warp_sum_ff(v);
  float *r = reinterpret_cast<float *>(g.red);
  if ((g.t & 31) == 0) {
    r[2 * (g.t >> 5)] = v.hi;
    r[2 * (g.t >> 5) + 1] = v.lo;
  }
  gsync(g);
  ff s = {0.0f, 0.0f};
  for (int w = 0; w < g.n / 32; ++w) s = ff_add(s, ff{r[2 * w], r[2 * w + 1]});
  gsync(g);
  return s;
}
__device__ __forceinline__ float g_sum_f(const Grp &g, float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  float *r = reinterpret_cast<float *>(g.red);
  if ((g.t & 31) == 0) r[g.t >> 5] = v;
  gsync(g);
  float s = 0.0f;
  for (int w = 0; w < g.n / 32; ++w) s = __fadd_rn(s, r[w]);
  gsync(g);
  return s;
}
__device__ __forceinline__ void g_minmax(const Grp &g, float &lo, float &hi) {
  lo = warp_min(lo);
  hi = warp_max(hi);
  float *r = reinterpret_cast<float *>(g.red);
  if ((g.t & 31) == 0) {
    r[2 * (g.t >> 5)] = lo;
    r[2 * (g.t >> 5) + 1] = hi;
  }
  gsync(g);
  lo = INFINITY;
  hi = -INFINITY;
  for (int w = 0; w < g.n / 32; ++w) {
    lo = fminf(lo, r[2 * w]);
    hi = fmaxf(hi, r[2 * w + 1]);
  }
  gsync(g);
}
__device__ __forceinline__ float g_max_f(const Grp &g, float v) {
  float lo = INFINITY;
  g_minmax(g, lo, v);
  return v;
}
__device__ __forceinline__ int g_max_i32(const Grp &g, int v) {
  v = warp_max_i32(v);
  int *r = reinterpret_cast<int *>(g.red);
  if ((g.t & 31) == 0) r[g.t >> 5] = v;
  gsync(g);
  int m = INT_MIN;
  for (int w = 0; w < g.n / 32; ++w) m = max(m, r[w]);
  gsync(g);
  return m;
}
// Exclusive scan of float-float values in thread order over the group.
__device__ __forceinline__ ff g_scan_ff(const Grp &g, ff v, ff &total) {
  const int lane = g.t & 31, w = g.t >> 5;
  ff inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    ff u;
    u.hi = __shfl_up_sync(0xffffffffu, inc.hi, o);
    u.lo = __shfl_up_sync(0xffffffffu, inc.lo, o);
    if (lane >= o) inc = ff_add(u, inc);
  }
  float *r = reinterpret_cast<float *>(g.red);
  if (lane == 31) {
    r[2 * w] = inc.hi;
    r[2 * w + 1] = inc.lo;
  }
  gsync(g);
  ff base = {0.0f, 0.0f}, tot = {0.0f, 0.0f};
  for (int j = 0; j < g.n / 32; ++j) {
    const ff x = {r[2 * j], r[2 * j + 1]};
    if (j < w) base = ff_add(base, x);
    tot = ff_add(tot, x);
  }
  gsync(g);
  total = tot;
  ff excl;
  excl.hi = __shfl_up_sync(0xffffffffu, inc.hi, 1);
  excl.lo = __shfl_up_sync(0xffffffffu, inc.lo, 1);
  if (lane == 0) excl = {0.0f, 0.0f};
  return ff_add(base, excl);
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
// Fast weight and a bound of its relative error (0 for z = -inf).
__device__ __forceinline__ float fw(const KP &P, float z, float m, float &eps) {
  if (z == -INFINITY) {
    eps = 0.0f;
    return 0.0f;
  }
  const float y = __fmul_rn(__fsub_rn(z, m), P.c2);
  eps = __fmaf_rn(fabsf(y), kExpErr1, kExpErr0);
  return ex2_approx(y);
}
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }
// Fixed-point weight round(e * 2^FP_SHIFT) of e in [0, 1].
__device__ __forceinline__ uint32_t to_fixed(ff e) {
  const float sc = pow2f(FP_SHIFT);
  const float x = __fadd_rn(__fmul_rn(e.hi, sc), __fmul_rn(e.lo, sc));
  return __float2uint_rn(x);
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

// ------------------------------------------------------- slice-mode parts
// Z of both tensors over their kept sets, fast single precision with
// compensated sums and a running bound of the error (used for p(x)/q(x) when
// the support is the whole vocabulary, and by the certified draw).  With
// `bands`, also a histogram of depth bands (nats below the maximum) of every
// SAMPLE_EVERY-th element: an estimate of how many tokens a top-p candidate
// window of each depth holds (cumulative counts in bt[] / bd[]).
static __constant__ float kBandDepth[NBANDS] = {1.f, 2.f, 3.f, 4.f, 5.f, 6.f, 7.f, 8.f,
                                         9.f, 10.f, 11.f, 12.f, 14.f, 16.f, 20.f, 24.f};

__device__ __forceinline__ int band_of(float d) {
  int band = 0;
  while (band < NBANDS && !(d < kBandDepth[band])) ++band;
  return band;
}

template <typename E>
__device__ __forceinline__ void slice_Z_fast(const KP &P, Blk &k, const E *st, const E *sd, int n, Dist &dt,
                             Dist &dd, bool dod, bool bands, ff &zall_t, ff &zall_d, int *bt,
                             int *bd, int *bh /* smem [2][NBANDS+1] */) {
  const Grp g = whole_block(k);
  if (bands) {
    for (int j = threadIdx.x; j < 2 * (NBANDS + 1); j += k.nt) bh[j] = 0;
    __syncthreads();
  }
  float zt = 0.0f, ct = 0.0f, et = 0.0f, zd = 0.0f, cd = 0.0f, ed = 0.0f;
  int it = 0;
  for (int j = threadIdx.x; j < n; j += k.nt, ++it) {
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
    if (smp && a == a) atomicAdd(&bh[band_of(__fmul_rn(__fsub_rn(dt.m, a), P.invT_hi))], 1);
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
      if (smp && b == b)
        atomicAdd(&bh[NBANDS + 1 + band_of(__fmul_rn(__fsub_rn(dd.m, b), P.invT_hi))], 1);
    }
  }
  const ff Zt = g_sum_ff(g, quick_two_sum(zt, -ct));
  const ff Zd = g_sum_ff(g, quick_two_sum(zd, -cd));
  const float Et = g_sum_f(g, et), Ed = g_sum_f(g, ed);
  constexpr int NWD = 6 + 2 * NBANDS;
  if (threadIdx.x == 0) {
    uint32_t *w = xslot(k);
    w[0] = __float_as_uint(Zt.hi);
    w[1] = __float_as_uint(Zt.lo);
    w[2] = __float_as_uint(Zd.hi);
    w[3] = __float_as_uint(Zd.lo);
    w[4] = __float_as_uint(Et);
    w[5] = __float_as_uint(Ed);
    for (int j = 0; j < NBANDS; ++j) {
      w[6 + j] = bands ? static_cast<uint32_t>(bh[j]) : 0u;
      w[6 + NBANDS + j] = bands ? static_cast<uint32_t>(bh[NBANDS + 1 + j]) : 0u;
    }
  }
  xsync(k, NWD);
  ff st_ = {0.0f, 0.0f}, sd_ = {0.0f, 0.0f};
  float et_ = 0.0f, ed_ = 0.0f;
  for (uint32_t c = 0; c < k.C; ++c) {
    const uint32_t *w = k.gat + c * NWD;
    st_ = ff_add(st_, ff{__uint_as_float(w[0]), __uint_as_float(w[1])});
    sd_ = ff_add(sd_, ff{__uint_as_float(w[2]), __uint_as_float(w[3])});
    et_ = __fadd_rn(et_, __uint_as_float(w[4]));
    ed_ = __fadd_rn(ed_, __uint_as_float(w[5]));
  }
  if (bands) {
    int c1 = 0, c2 = 0;
    for (int j = 0; j < NBANDS; ++j) {
      for (uint32_t c = 0; c < k.C; ++c) {
        c1 += static_cast<int>(k.gat[c * NWD + 6 + j]);
        c2 += static_cast<int>(k.gat[c * NWD + 6 + NBANDS + j]);
      }
      bt[j] = c1;
      bd[j] = c2;
    }
  }
  zall_t = st_;
  zall_d = sd_;
  // relative error bound of Z: the weights' bound plus the compensated sums'
  set_Zf(dt, st_, __fadd_rn(__fdiv_rn(et_, st_.hi), 2.4e-7f));
  if (dod) set_Zf(dd, sd_, __fadd_rn(__fdiv_rn(ed_, sd_.hi), 2.4e-7f));
}

// Exact threshold search over the cluster's slices: the largest key K such
// that the weight of {key(z) >= K} reaches the target (top-k: weight 1;
// top-p: fixed-point mass of the top-k survivors).  Binary search over the
// 32-bit key space, one pass + one cluster exchange per step, both tensors
// in lock-step.  The result is always the key of an existing element.
template <typename E>
__device__ __noinline__ void slice_bisect(const KP &P, Blk &k, const E *st, const E *sd, int n, Dist &dt,
                             Dist &dd, bool dot, bool dod, bool mass) {
  const Grp g = whole_block(k);
  uint64_t tgt_t = static_cast<uint64_t>(P.top_k), tgt_d = tgt_t;
  const float sc = pow2f(FP_SHIFT);
  if (mass) {
    uint64_t a = 0, b = 0;
    for (int j = threadIdx.x; j < n; j += k.nt) {
      if (dot) {
        const float x = stage_get(st, j);
        if (x >= dt.tau) a += __float2uint_rn(__fmul_rn(weight_fast(P, x, dt.m), sc));
      }
      if (dod) {
        const float y = stage_get(sd, j);
        if (y >= dd.tau) b += __float2uint_rn(__fmul_rn(weight_fast(P, y, dd.m), sc));
      }
    }
    a = g_sum_u64(g, a);
    b = g_sum_u64(g, b);
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
    for (int j = threadIdx.x; j < n; j += k.nt) {
      if (dot) {
        const float x = stage_get(st, j);
        const uint32_t kx = fkey(x);
        if (x == x && kx >= mt && kx >= kt0)
          a += mass ? __float2uint_rn(__fmul_rn(weight_fast(P, x, dt.m), sc)) : 1u;
      }
      if (dod) {
        const float y = stage_get(sd, j);
        const uint32_t ky = fkey(y);
        if (y == y && ky >= md && ky >= kd0)
          b += mass ? __float2uint_rn(__fmul_rn(weight_fast(P, y, dd.m), sc)) : 1u;
      }
    }
    a = g_sum_u64(g, a);
    b = g_sum_u64(g, b);
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
__device__ __noinline__ void slice_Z_exact(const KP &P, Blk &k, const E *st, const E *sd, int n, Dist &dt,
                              Dist &dd, bool dot, bool dod) {
  const Grp g = whole_block(k);
  ff a = {0.0f, 0.0f}, b = {0.0f, 0.0f};
  for (int j = threadIdx.x; j < n; j += k.nt) {
    if (dot) {
      const float x = stage_get(st, j);
      if (x >= dt.tau) a = ff_add(a, weight_ff(P, x, dt.m));
    }
    if (dod) {
      const float y = stage_get(sd, j);
      if (y >= dd.tau) b = ff_add(b, weight_ff(P, y, dd.m));
    }
  }
  a = g_sum_ff(g, a);
  b = g_sum_ff(g, b);
  uint32_t w[4] = {__float_as_uint(a.hi), __float_as_uint(a.lo), __float_as_uint(b.hi),
                   __float_as_uint(b.lo)};
  exchange(k, w, 4);
  ff sa = {0.0f, 0.0f}, sb = {0.0f, 0.0f};
  for (uint32_t c = 0; c < k.C; ++c) {
    sa = ff_add(sa, ff{__uint_as_float(k.gat[c * 4]), __uint_as_float(k.gat[c * 4 + 1])});
    sb = ff_add(sb, ff{__uint_as_float(k.gat[c * 4 + 2]), __uint_as_float(k.gat[c * 4 + 3])});
  }
  if (dot) set_Zx(dt, sa);
  if (dod) set_Zx(dd, sb);
}

// The draw weight of one token from its target / draft logits: p_v (bonus)
// or max(0, p_v - q_v) (residual: "max_fn" of "Prepare autoregressive
// sampling", normalised by the inverse CDF).
__device__ __forceinline__ ff draw_weight_of(const KP &P, float x, float y, const Dist &dt,
                                             const Dist &dd, bool residual) {
  if (!(x >= dt.tau)) return {0.0f, 0.0f};
  ff p = ff_mul(weight_ff(P, x, dt.m), dt.rZ);
  if (!residual) return p;
  if (y >= dd.tau) p = ff_sub(p, ff_mul(weight_ff(P, y, dd.m), dd.rZ));
  return p.hi > 0.0f ? p : ff{0.0f, 0.0f};
}

// Inverse-CDF draw over the cluster's slices in vocabulary order, float-float.
// Each thread owns a contiguous chunk of its CTA's slice.  Returns the token
// (all CTAs), or -1 when the total weight is 0; *Wout = the total weight.
template <typename E>
__device__ __noinline__ int slice_draw(const KP &P, Blk &k, const E *st, const E *sd, int n, int lo,
                          const Dist &dt, const Dist &dd, bool residual, float u, ff *Wout) {
  const Grp g = whole_block(k);
  int ch = (n + k.nt - 1) / k.nt;
  ch |= 1;  // odd chunk length: conflict-free shared-memory strides
  const int j0 = min(n, static_cast<int>(threadIdx.x) * ch), j1 = min(n, j0 + ch);
  ff s = {0.0f, 0.0f};
  int lastpos = -1;
  for (int j = j0; j < j1; ++j) {
    const ff w = draw_weight_of(P, stage_get(st, j), residual ? stage_get(sd, j) : 0.0f, dt,
                                dd, residual);
    if (w.hi > 0.0f) lastpos = lo + j;
    s = ff_add(s, w);
  }
  ff ctot;
  const ff pre = g_scan_ff(g, s, ctot);
  const int clast = g_max_i32(g, lastpos);
  uint32_t w3[3] = {__float_as_uint(ctot.hi), __float_as_uint(ctot.lo),
                    static_cast<uint32_t>(clast)};
  exchange(k, w3, 3);
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
      const ff wj = draw_weight_of(P, stage_get(st, j), residual ? stage_get(sd, j) : 0.0f, dt,
                                   dd, residual);
      if (wj.hi > 0.0f) tok = lo + j;
      c = ff_add(c, wj);
      if (ff_lt(target, c) && wj.hi > 0.0f) break;
    }
    k.scal[8] = tok;
  }
  __syncthreads();
  uint32_t v = static_cast<uint32_t>(k.scal[8]);
  __syncthreads();
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
__device__ __forceinline__ int slice_draw_fast(const KP &P, Blk &k, const E *st, const E *sd, int n, int lo,
                               const Dist &dt, const Dist &dd, bool residual, float u,
                               float *Wf) {
  const Grp g = whole_block(k);
  int ch = (n + k.nt - 1) / k.nt;
  ch |= 1;
  const int j0 = min(n, static_cast<int>(threadIdx.x) * ch), j1 = min(n, j0 + ch);
  ff s = {0.0f, 0.0f};
  float dsum = 0.0f;
  for (int j = j0; j < j1; ++j) {
    float w, e;
    fast_weight(P, stage_get(st, j), residual ? stage_get(sd, j) : 0.0f, dt, dd, residual, w, e);
    s = ff_add_f(s, w);
    dsum = __fadd_rn(dsum, e);
  }
  ff ctot;
  const ff pre = g_scan_ff(g, s, ctot);
  const float cerr = g_sum_f(g, dsum);
  uint32_t w3[3] = {__float_as_uint(ctot.hi), __float_as_uint(ctot.lo), __float_as_uint(cerr)};
  exchange(k, w3, 3);
  ff W = {0.0f, 0.0f}, mybase = {0.0f, 0.0f};
  float D = 0.0f;
  for (uint32_t c = 0; c < k.C; ++c) {
    const ff x = {__uint_as_float(k.gat[c * 3]), __uint_as_float(k.gat[c * 3 + 1])};
    if (c < k.rank) mybase = ff_add(mybase, x);
    W = ff_add(W, x);
    D = __fadd_rn(D, __uint_as_float(k.gat[c * 3 + 2]));
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
      fast_weight(P, stage_get(st, j), residual ? stage_get(sd, j) : 0.0f, dt, dd, residual, w,
                  e);
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

}  // namespace sv
