// spec_verify.cu -- speculative-sampling verification on GB300 (sm_103a).
//
// One thread-block cluster of C CTAs verifies one row (sequence).  The
// vocabulary is split into C contiguous slices, one per CTA.  For each
// position, each CTA's slice of the target (and draft) logits is staged in
// shared memory by one-dimensional bulk copies (TMA) in NCH chunks, each
// chunk processed as soon as its mbarrier completes; the cluster exchanges
// per-CTA partial results (maxima, sums, counts, candidate lists) through
// distributed shared memory.  Positions are walked in order and the walk
// stops at the first rejection, so later positions are never read.
// Method: "Text Generation via Speculative Sampling, KV Caching, and
// OpenVINO", section "Prepare speculative sampling" (steps 3 and 4), and
// "CS3602_FINAL_SpeDec", section "2. 困惑度测试(PPL)" (acceptance
// min(1, p/q), residual norm(max(0, p - q))).
//
// Per position and tensor (p from the target row, q from the draft row):
//   pass 1 (HBM -> SMEM): max, first argmax, NaN / +inf / finite flags, and
//          per-warp top-4 of the per-thread maxima, whose k_c-th largest
//          bounds each CTA's share of the top-k from below;
//   filters: top-k / top-p thresholds on the raw logit (ties kept), found
//          on a candidate list gathered from the cluster (fast path) or by
//          an exact bisection over order-preserving keys (fallback);
//   normaliser Z over the kept set; accept iff u < p(x)/q(x);
//   at the first rejection (or the bonus position) an inverse-CDF draw in
//   vocabulary order: over the list in float-float, or over the slices in
//   single precision with a certified error bound (float-float if the
//   uniform falls within the bound of a CDF boundary).
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <type_traits>

#include "spec_verify.h"
#include "sv_core.cuh"
#include "sv_row.h"
#include "sv_strip.h"
#include "sv_verify.h"

// Phase timing for development builds (-DSV_PHASE_PROFILE): thread 0 of
// each row's first CTA accumulates clock64() deltas per phase into a global
// array sv_phase_cycles[16].
#ifdef SV_PHASE_PROFILE
__device__ unsigned long long sv_phase_cycles[16];
#define SV_PHASE(id)                                                                       \
  do {                                                                                     \
    if (k.rank == 0 && threadIdx.x == 0) {                                                 \
      const long long now_ = clock64();                                                    \
      atomicAdd(&sv_phase_cycles[id], static_cast<unsigned long long>(now_ - t_ph_));      \
      t_ph_ = now_;                                                                        \
    }                                                                                      \
  } while (0)
#else
#define SV_PHASE(id) \
  do {               \
  } while (0)
#endif

namespace sv {

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
  uint32_t *w_p, *w_q;        // [cap] fixed-point weights
  uint64_t *hist_p, *hist_q;  // [NBINS]
  uint64_t *key_p, *key_q;    // [SORT_MAX] sort keys
};

// Warp segments of a slice: contiguous, starting on a 16-byte vector.
template <typename E>
__device__ __forceinline__ void warp_segment(const Blk &k, int n, int &s0, int &s1) {
  const int w = threadIdx.x >> 5;
  const int seg = ((n + k.nw - 1) / k.nw + 7) & ~7;
  s0 = min(n, w * seg);
  s1 = min(n, s0 + seg);
}

// Number of elements >= t in one 16-byte vector.
__device__ __forceinline__ int vcount(const uint4 &x, float t, float) {
  return (__uint_as_float(x.x) >= t) + (__uint_as_float(x.y) >= t) + (__uint_as_float(x.z) >= t) +
         (__uint_as_float(x.w) >= t);
}
__device__ __forceinline__ int vcount(const uint4 &x, float t, uint16_t) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  int c = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e)
    c += (__uint_as_float(w[e] << 16) >= t) + (__uint_as_float(w[e] & 0xffff0000u) >= t);
  return c;
}

// Per-warp counts of {z >= cand} over the warp segments (vector loads, no
// ordering needed).  Sets the CTA totals and this warp's exclusive base.
template <typename E>
__device__ __forceinline__ void count_pass(const Blk &k, const E *st, const E *sd, int n,
                                           float ct, float cd, bool dot, bool dod, int *wc,
                                           int &tot_t, int &tot_d, int &base_t, int &base_d) {
  constexpr int EPV = Elem<E>::kPerVec;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int s0, s1;
  warp_segment<E>(k, n, s0, s1);
  const uint4 *vt = reinterpret_cast<const uint4 *>(st), *vd = reinterpret_cast<const uint4 *>(sd);
  const int q1 = s1 / EPV;
  int a = 0, b = 0;
#pragma unroll 4
  for (int q = s0 / EPV + lane; q < q1; q += 32) {
    if (dot) a += vcount(vt[q], ct, E());
    if (dod) b += vcount(vd[q], cd, E());
  }
  for (int j = max(s0, q1 * EPV) + lane; j < s1; j += 32) {  // ragged end of the last segment
    if (dot) a += stage_raw(st, j) >= ct;
    if (dod) b += stage_raw(sd, j) >= cd;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
  }
  if (lane == 0) {
    wc[w] = a;
    wc[MAXNW + w] = b;
  }
  __syncthreads();
  tot_t = tot_d = base_t = base_d = 0;
  for (int j = 0; j < k.nw; ++j) {
    if (j < w) {
      base_t += wc[j];
      base_d += wc[MAXNW + j];
    }
    tot_t += wc[j];
    tot_d += wc[MAXNW + j];
  }
  __syncthreads();
}

// Write this CTA's candidates, in index order, into its own lists at the
// cluster-wide positions (cluster offset + warp base + rank).  Vector rows:
// each lane takes one 16-byte vector; rows without a candidate are skipped.
template <typename E>
__device__ __forceinline__ void write_pass(const Blk &k, const Lists &L, const E *st, const E *sd,
                                           int n, int lo, float ct, float cd, bool dot, bool dod,
                                           bool has_draft, int pos_t, int pos_d) {
  constexpr int EPV = Elem<E>::kPerVec;
  const int lane = threadIdx.x & 31;
  int s0, s1;
  warp_segment<E>(k, n, s0, s1);
  const int q1 = s1 / EPV;
  // full vector rows of 32 lanes (the ragged end is handled element-wise)
  for (int q0 = s0 / EPV; q0 < q1; q0 += 32) {
    const int q = q0 + lane;
    uint32_t mt = 0, md = 0;
    float ft[EPV], fd[EPV];
    if (q < q1) {
      unpack<E>(reinterpret_cast<const uint4 *>(st)[q], ft);
      if (has_draft) unpack<E>(reinterpret_cast<const uint4 *>(sd)[q], fd);
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        if (!has_draft) fd[e] = 0.0f;
        if (dot && ft[e] >= ct) mt |= 1u << e;
        if (dod && fd[e] >= cd) md |= 1u << e;
      }
    }
    const int ctn = __popc(mt), cdn = __popc(md);
    if (!__any_sync(0xffffffffu, ctn | cdn)) continue;
    int it = ctn, id = cdn;  // inclusive scans over the lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, it, o), v = __shfl_up_sync(0xffffffffu, id, o);
      if (lane >= o) {
        it += u;
        id += v;
      }
    }
    int pt = pos_t + it - ctn, pd = pos_d + id - cdn;
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      const int idx = lo + q * EPV + e;
      if (mt & (1u << e)) {
        L.p_idx[pt] = idx;
        L.p_zp[pt] = ft[e];
        L.p_zq[pt] = fd[e];
        ++pt;
      }
      if (md & (1u << e)) {
        L.q_idx[pd] = idx;
        L.q_zq[pd] = fd[e];
        ++pd;
      }
    }
    pos_t += __shfl_sync(0xffffffffu, it, 31);
    pos_d += __shfl_sync(0xffffffffu, id, 31);
  }
  // ragged end: element-wise in index order
  for (int j0 = max(s0, q1 * EPV); j0 < s1; j0 += 32) {
    const int j = j0 + lane;
    float zt = 0.0f, zd = 0.0f;
    bool bt = false, bd = false;
    if (j < s1) {
      zt = stage_raw(st, j);
      if (has_draft) zd = stage_raw(sd, j);
      bt = dot && zt >= ct;
      bd = dod && zd >= cd;
    }
    const uint32_t lt = (1u << lane) - 1u;
    const uint32_t mt = __ballot_sync(0xffffffffu, bt), md = __ballot_sync(0xffffffffu, bd);
    if (bt) {
      const int pos = pos_t + __popc(mt & lt);
      L.p_idx[pos] = lo + j;
      L.p_zp[pos] = zt;
      L.p_zq[pos] = zd;
    }
    if (bd) {
      const int pos = pos_d + __popc(md & lt);
      L.q_idx[pos] = lo + j;
      L.q_zq[pos] = zd;
    }
    pos_t += __popc(mt);
    pos_d += __popc(md);
  }
}

// After a cluster barrier: copy the other CTAs' regions of the lists (same
// positions in their shared memory) into this CTA's lists.  off[c] / cnt[c]:
// region of CTA c.  Independent remote loads, one entry per thread.
__device__ __forceinline__ void pull_lists(const Blk &k, const Lists &L, const int *off_t,
                                           const int *off_d, int all_t, int all_d, bool dot,
                                           bool dod) {
  const int me0t = off_t[k.rank], me1t = off_t[k.rank + 1];
  const int me0d = off_d[k.rank], me1d = off_d[k.rank + 1];
  if (dot) {
    for (int j = threadIdx.x; j < all_t; j += k.nt) {
      if (j >= me0t && j < me1t) continue;
      uint32_t c = 0;
      while (j >= off_t[c + 1]) ++c;
      L.p_idx[j] = static_cast<int>(dsmem_ld_u32(dsmem_addr(smem_u32(L.p_idx + j), c)));
      L.p_zp[j] = __uint_as_float(dsmem_ld_u32(dsmem_addr(smem_u32(L.p_zp + j), c)));
      L.p_zq[j] = __uint_as_float(dsmem_ld_u32(dsmem_addr(smem_u32(L.p_zq + j), c)));
    }
  }
  if (dod) {
    for (int j = threadIdx.x; j < all_d; j += k.nt) {
      if (j >= me0d && j < me1d) continue;
      uint32_t c = 0;
      while (j >= off_d[c + 1]) ++c;
      L.q_idx[j] = static_cast<int>(dsmem_ld_u32(dsmem_addr(smem_u32(L.q_idx + j), c)));
      L.q_zq[j] = __uint_as_float(dsmem_ld_u32(dsmem_addr(smem_u32(L.q_zq + j), c)));
    }
  }
}

// Threshold selection on a list: the largest value v such that the weight
// of entries with value >= v reaches `target` (top-k: weight 1 per entry;
// top-p: w[j]); -inf if the whole list falls short.  Short lists: every
// entry counts the weight at or above it (exact, one pass of n^2/size).
// Long lists: a 256-bin value histogram of the current range is refined
// around the bin where the cumulative weight from the top crosses the
// target; integer weights make both exact and order-independent.
__device__ __forceinline__ float g_select(const Grp &g, const float *val, const uint32_t *w, int n,
                          uint64_t target, uint64_t *hist) {
  if (n <= SMALL_LIST) {
    float best = -INFINITY;
    for (int j = g.t; j < n; j += g.n) {
      if (w && !w[j]) continue;
      const float vj = val[j];
      uint64_t s = 0;
      for (int i = 0; i < n; ++i)
        if (val[i] >= vj) s += w ? w[i] : 1u;
      if (s >= target && vj > best) best = vj;
    }
    return g_max_f(g, best);
  }
  float lo = INFINITY, hi = -INFINITY;
  for (int j = g.t; j < n; j += g.n)
    if (!w || w[j]) {
      lo = fminf(lo, val[j]);
      hi = fmaxf(hi, val[j]);
    }
  g_minmax(g, lo, hi);
  if (!(lo <= hi)) return -INFINITY;
  uint64_t above = 0;
  for (int iter = 0; iter <= n + 1; ++iter) {  // each step drops >= 1 distinct value
    if (lo == hi) {
      uint64_t s = 0;
      for (int j = g.t; j < n; j += g.n)
        if ((!w || w[j]) && val[j] == lo) s += w ? w[j] : 1u;
      s = g_sum_u64(g, s);
      return (above + s >= target) ? lo : -INFINITY;
    }
    const BinMap bm = bin_map(lo, hi);
    for (int j = g.t; j < NBINS; j += g.n) hist[j] = 0;
    gsync(g);
    for (int j = g.t; j < n; j += g.n) {
      const float v = val[j];
      if ((!w || w[j]) && v >= lo && v <= hi)
        atomicAdd(reinterpret_cast<unsigned long long *>(&hist[value_bin(v, bm)]),
                  static_cast<unsigned long long>(w ? w[j] : 1u));
    }
    gsync(g);
    if (g.t < 32) {
      const int lane = g.t;
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
      if (lane == 0) g.sc[0] = -1;
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
        g.sc[0] = bsel;
        reinterpret_cast<uint64_t *>(g.sc)[1] = cum;  // weight strictly above the bin
      }
    }
    gsync(g);
    const int bsel = g.sc[0];
    const uint64_t nabove = reinterpret_cast<const uint64_t *>(g.sc)[1];
    gsync(g);
    if (bsel < 0) return -INFINITY;
    float nlo = INFINITY, nhi = -INFINITY;
    for (int j = g.t; j < n; j += g.n) {
      const float v = val[j];
      if ((!w || w[j]) && v >= lo && v <= hi && value_bin(v, bm) == bsel) {
        nlo = fminf(nlo, v);
        nhi = fmaxf(nhi, v);
      }
    }
    g_minmax(g, nlo, nhi);
    lo = nlo;
    hi = nhi;
    above = nabove;
  }
  return lo;  // not reached
}

// Sort the list's entries by value, largest first (ties by list position):
// a bitonic network over N = next power of two >= n keys
// ~(key(value) << 32 | position), ascending.  Group-level, in shared memory.
__device__ __forceinline__ int g_sort_desc(const Grp &g, const float *val, int n, uint64_t *key) {
  int N = 1;
  while (N < n) N <<= 1;
  for (int j = g.t; j < N; j += g.n)
    key[j] = j < n ? ~((static_cast<uint64_t>(fkey(canon(val[j]))) << 32) |
                       static_cast<uint32_t>(~j))
                   : ~0ull;
  gsync(g);
  for (int kk = 2; kk <= N; kk <<= 1) {
    for (int jj = kk >> 1; jj > 0; jj >>= 1) {
      for (int t = g.t; t < N / 2; t += g.n) {
        const int i = (t / jj) * 2 * jj + (t % jj), l = i + jj;
        const uint64_t a = key[i], b = key[l];
        const bool up = (i & kk) == 0;
        if ((a > b) == up) {
          key[i] = b;
          key[l] = a;
        }
      }
      gsync(g);
    }
  }
  return N;
}
__device__ __forceinline__ int sorted_pos(uint64_t k) {
  return static_cast<int>(~static_cast<uint32_t>(~k));
}

// Filters and normaliser from a sorted list (n <= SORT_MAX): top-k is the
// k-th value, top-p the first rank where the cumulative fixed-point mass
// reaches the target; the same certification as g_list_fast.
__device__ int g_list_sorted(const KP &P, const Grp &g, const float *val, int n, float m,
                             uint32_t *w, uint64_t *key, ff zall, float zall_err, float &tau_out,
                             ff &Z_out, float &zerr_out) {
  g_sort_desc(g, val, n, key);
  float tau = -INFINITY;
  int state = 1;
  if (P.k_on) {
    if (n < P.top_k) return 0;
    tau = val[sorted_pos(key[P.top_k - 1])];
  }
  if (P.p_on) {
    const float sc = pow2f(FP_SHIFT);
    // fixed-point weights in rank order (0 below the top-k threshold)
    uint64_t s = 0;
    float E = 0.0f;
    for (int r = g.t; r < n; r += g.n) {
      const float v = val[sorted_pos(key[r])];
      uint32_t wr = 0;
      if (v >= tau) {
        float eps;
        const float e = __fmul_rn(fw(P, v, m, eps), sc);
        wr = __float2uint_rn(e);
        E = __fmaf_rn(e, eps, __fadd_rn(E, 0.5f));
      }
      w[r] = wr;
      s += wr;
    }
    s = g_sum_u64(g, s);
    E = g_sum_f(g, E);
    uint64_t znorm = s;
    float EZ = E;
    if (!P.k_on) {
      znorm = __float2ull_rn(__fmul_rn(zall.hi, sc)) +
              static_cast<uint64_t>(__float2ll_rn(__fmul_rn(zall.lo, sc)));
      EZ = __fmaf_rn(__fmul_rn(zall.hi, sc), zall_err, 2.0f);
    }
    const uint64_t target = ceil_scale(P.top_p, znorm);
    const uint64_t slack =
        static_cast<uint64_t>(__fmul_rn(__fmaf_rn(P.top_p, EZ, E), 1.01f)) + 4ull;
    if (s < target) {
      if (!P.k_on) return (s + slack >= target) ? 2 : 0;
    } else {
      // inclusive prefix of w over ranks: each thread a contiguous chunk
      const int ch = (n + g.n - 1) / g.n;
      const int r0 = min(n, g.t * ch), r1 = min(n, r0 + ch);
      uint64_t loc = 0;
      for (int r = r0; r < r1; ++r) loc += w[r];
      // exclusive scan of the chunk sums over the group
      uint64_t inc = loc;
      const int lane = g.t & 31, wi = g.t >> 5;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint64_t u = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += u;
      }
      if (lane == 31) g.red[wi] = inc;
      gsync(g);
      uint64_t base = 0;
      for (int j = 0; j < wi; ++j) base += g.red[j];
      gsync(g);
      uint64_t cum = base + inc - loc;
      if (g.t == 0) g.sc[0] = -1;
      gsync(g);
      for (int r = r0; r < r1; ++r) {
        const uint64_t before = cum;
        cum += w[r];
        if (before < target && cum >= target) g.sc[0] = r;  // the crossing rank (unique)
      }
      gsync(g);
      const int rc = g.sc[0];
      gsync(g);
      const float tp = val[sorted_pos(key[rc])];
      // masses strictly above and at-or-above the threshold value
      uint64_t mhi = 0, mlo = 0;
      for (int r = g.t; r < n; r += g.n) {
        const float v = val[sorted_pos(key[r])];
        if (v >= tp) mhi += w[r];
        if (v > tp) mlo += w[r];
      }
      mhi = g_sum_u64(g, mhi);
      mlo = g_sum_u64(g, mlo);
      if (!(mhi >= target + slack && mlo + slack < target)) state = 2;
      tau = fmaxf(tau, tp);
    }
  }
  float zs = 0.0f, zc = 0.0f, ze = 0.0f;
  for (int j = g.t; j < n; j += g.n) {
    const float v = val[j];
    if (v >= tau) {
      float eps;
      const float e = fw(P, v, m, eps);
      const float t = __fsub_rn(e, zc), s2 = __fadd_rn(zs, t);
      zc = __fsub_rn(__fsub_rn(s2, zs), t);
      zs = s2;
      ze = __fmaf_rn(e, eps, ze);
    }
  }
  Z_out = g_sum_ff(g, quick_two_sum(zs, -zc));
  ze = g_sum_f(g, ze);
  tau_out = tau;
  zerr_out = __fadd_rn(__fdiv_rn(ze, Z_out.hi), 4.8e-7f);
  return state;
}

// Filters and normaliser of one tensor from its list in single precision,
// with every decision checked against a bound of its rounding error.
// `zall` (relative error zall_err) normalises top-p without top-k.
// Returns 1 (done), 0 (the nucleus reaches below the list), or 2 (a top-p
// mass comparison fell within its error bound: redo it exactly).
__device__ __forceinline__ int g_list_fast(const KP &P, const Grp &g, const float *val, int n, float m,
                           uint32_t *w, uint64_t *hist, ff zall, float zall_err,
                           float &tau_out, ff &Z_out, float &zerr_out) {
  float tau = -INFINITY;
  int state = 1;
  if (P.k_on) {
    tau = g_select(g, val, nullptr, n, static_cast<uint64_t>(P.top_k), hist);
    if (tau == -INFINITY) return 0;
  }
  if (P.p_on) {
    const float sc = pow2f(FP_SHIFT);
    uint64_t s = 0;
    float E = 0.0f;  // bound of the total error of the fixed-point weights
    for (int j = g.t; j < n; j += g.n) {
      const float v = val[j];
      uint32_t wj = 0;
      if (v >= tau) {
        float eps;
        const float e = __fmul_rn(fw(P, v, m, eps), sc);
        wj = __float2uint_rn(e);
        E = __fmaf_rn(e, eps, __fadd_rn(E, 0.5f));
      }
      w[j] = wj;
      s += wj;
    }
    s = g_sum_u64(g, s);  // (its barrier also publishes w[])
    E = g_sum_f(g, E);
    uint64_t znorm = s;
    float EZ = E;
    if (!P.k_on) {
      znorm = __float2ull_rn(__fmul_rn(zall.hi, sc)) +
              static_cast<uint64_t>(__float2ll_rn(__fmul_rn(zall.lo, sc)));
      EZ = __fmaf_rn(__fmul_rn(zall.hi, sc), zall_err, 2.0f);
    }
    const uint64_t target = ceil_scale(P.top_p, znorm);
    const uint64_t slack =
        static_cast<uint64_t>(__fmul_rn(__fmaf_rn(P.top_p, EZ, E), 1.01f)) + 4ull;
    if (s < target) {
      if (!P.k_on) return (s + slack >= target) ? 2 : 0;
    } else {
      const float tp = g_select(g, val, w, n, target, hist);
      uint64_t mhi = 0, mlo = 0;
      for (int j = g.t; j < n; j += g.n) {
        if (val[j] >= tp) mhi += w[j];
        if (val[j] > tp) mlo += w[j];
      }
      mhi = g_sum_u64(g, mhi);
      mlo = g_sum_u64(g, mlo);
      if (!(mhi >= target + slack && mlo + slack < target)) state = 2;
      tau = fmaxf(tau, tp);
    }
  }
  float zs = 0.0f, zc = 0.0f, ze = 0.0f;
  for (int j = g.t; j < n; j += g.n) {
    const float v = val[j];
    if (v >= tau) {
      float eps;
      const float e = fw(P, v, m, eps);
      const float t = __fsub_rn(e, zc), s2 = __fadd_rn(zs, t);
      zc = __fsub_rn(__fsub_rn(s2, zs), t);
      zs = s2;
      ze = __fmaf_rn(e, eps, ze);
    }
  }
  Z_out = g_sum_ff(g, quick_two_sum(zs, -zc));
  ze = g_sum_f(g, ze);
  tau_out = tau;
  zerr_out = __fadd_rn(__fdiv_rn(ze, Z_out.hi), 4.8e-7f);
  return state;
}

// The same in float-float (exact path): `zall` must then be exact too.
// Returns false if the list cannot hold the kept set.
__device__ __noinline__ bool g_list_exact(const KP &P, const Grp &g, const float *val, int n,
                                          float m, uint32_t *w, uint64_t *hist, ff zall,
                                          float &tau_out, ff &Z_out) {
  float tau = -INFINITY;
  if (P.k_on) {
    tau = g_select(g, val, nullptr, n, static_cast<uint64_t>(P.top_k), hist);
    if (tau == -INFINITY) return false;
  }
  if (P.p_on) {
    uint64_t s = 0;
    for (int j = g.t; j < n; j += g.n) {
      const float v = val[j];
      w[j] = (v >= tau) ? to_fixed(weight_ff(P, v, m)) : 0u;
      s += w[j];
    }
    s = g_sum_u64(g, s);  // (its barrier also publishes w[])
    uint64_t znorm = s;
    if (!P.k_on) {
      const float sc = pow2f(FP_SHIFT);
      znorm = __float2ull_rn(__fmul_rn(zall.hi, sc)) +
              static_cast<uint64_t>(__float2ll_rn(__fmul_rn(zall.lo, sc)));
    }
    const uint64_t target = ceil_scale(P.top_p, znorm);
    if (s < target) {
      if (!P.k_on) return false;  // the nucleus is not inside the candidate window
      // rounding: the kept set's own mass falls short; keep it whole
    } else {
      tau = fmaxf(tau, g_select(g, val, w, n, target, hist));
    }
  }
  ff z = {0.0f, 0.0f};
  for (int j = g.t; j < n; j += g.n)
    if (val[j] >= tau) z = ff_add(z, weight_ff(P, val[j], m));
  Z_out = g_sum_ff(g, z);
  tau_out = tau;
  return true;
}


// Float-float normaliser of a list-mode distribution (exact paths).
__device__ __noinline__ void list_make_exact(const KP &P, const Grp &g, const float *val, int n,
                                             Dist &D) {
  ff z = {0.0f, 0.0f};
  for (int j = g.t; j < n; j += g.n)
    if (val[j] >= D.tau) z = ff_add(z, weight_ff(P, val[j], D.m));
  set_Zx(D, g_sum_ff(g, z));
}

// Certified single-precision inverse-CDF draw over the p-list (index
// order), redundantly in every CTA: as slice_draw_fast, without the cluster
// exchange.  Returns the token, -1 (total weight 0) or -2 (uncertain).
__device__ __forceinline__ int list_draw_fast(const KP &P, Blk &k, const Lists &L, int n, const Dist &dt,
                              const Dist &dd, bool residual, float u, float *Wf) {
  const Grp g = whole_block(k);
  int ch = (n + k.nt - 1) / k.nt;
  ch |= 1;
  const int j0 = min(n, static_cast<int>(threadIdx.x) * ch), j1 = min(n, j0 + ch);
  ff s = {0.0f, 0.0f};
  float dsum = 0.0f;
  for (int j = j0; j < j1; ++j) {
    float w, e;
    fast_weight(P, L.p_zp[j], L.p_zq[j], dt, dd, residual, w, e);
    s = ff_add_f(s, w);
    dsum = __fadd_rn(dsum, e);
  }
  ff W;
  const ff pre = g_scan_ff(g, s, W);
  const float D = g_sum_f(g, dsum);
  *Wf = W.hi + W.lo;
  if (!(W.hi > 0.0f)) return -1;
  const float slack = __fmaf_rn(W.hi, 1e-12f, static_cast<float>(n) * 4e-38f *
                                                  (dt.rzf + (residual ? dd.rzf : 0.0f)));
  const ff target = ff_mul_f(W, u);
  if (threadIdx.x == 0) {
    k.scal[8] = -1;
    k.scal[10] = 0;
  }
  __syncthreads();
  const ff b = ff_add(pre, s);
  if (!ff_lt(target, pre) && ff_lt(target, b)) {
    ff c = pre;
    int tok = -1;
    float margin = 0.0f;
    for (int j = j0; j < j1; ++j) {
      float w, e;
      fast_weight(P, L.p_zp[j], L.p_zq[j], dt, dd, residual, w, e);
      const ff cp = c;
      c = ff_add_f(c, w);
      if (w > 0.0f && ff_lt(target, c)) {
        tok = L.p_idx[j];
        const ff l = ff_sub(target, cp), h = ff_sub(c, target);
        margin = fminf(l.hi + l.lo, h.hi + h.lo);
        break;
      }
    }
    k.scal[8] = tok;
    k.scal[10] = (tok >= 0 && margin > __fmaf_rn(2.0f, D, slack)) ? 1 : 0;
  }
  __syncthreads();
  const int tok = k.scal[8], cert = k.scal[10];
  __syncthreads();
  return (tok >= 0 && cert) ? tok : -2;
}

// Inverse-CDF draw over the p-list (index order), redundantly in every CTA.
__device__ __noinline__ int list_draw(const KP &P, Blk &k, const Lists &L, int n, const Dist &dt,
                         const Dist &dd, bool residual, float u, ff *Wout) {
  const Grp g = whole_block(k);
  int ch = (n + k.nt - 1) / k.nt;
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
  const ff pre = g_scan_ff(g, s, W);
  const int glast = g_max_i32(g, lastpos);
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
template <typename E, bool VEC, int NT>
__global__ void __launch_bounds__(NT, NT == 128 ? 4 : 2) verify_kernel(const __grid_constant__ KP P) {
  constexpr int NW = NT / kWarp;
  static_assert(NW >= 2 && NW <= MAXNW, "2 to 8 warps per CTA");
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint32_t xch[XSLOTS * XWORDS];
  __shared__ uint32_t gat[MAXC * XWORDS];
  __shared__ uint64_t red[MAXNW * 4];
  __shared__ uint64_t gred[2][MAXNW * 2];
  __shared__ __align__(8) int32_t scal[32];
  __shared__ __align__(8) int32_t gsc[2][8];
  __shared__ int wcnt[2 * MAXNW];
  __shared__ int bandh[2 * (NBANDS + 1)];
  __shared__ float cand[2][MAXNW * TOPR];
  __shared__ uint32_t wstat[MAXNW * 8];
  __shared__ __align__(8) uint64_t bars[2 * NCH];
  __shared__ float lres[2][5];  // list results: state, tau, Z.hi, Z.lo, zerr

  Blk k;
  k.xch = xch;
  k.gat = gat;
  k.red = red;
  k.scal = scal;
  k.C = cluster_size();
  k.rank = cluster_rank();
  k.slot = 0;
  k.nt = NT;
  k.nw = NW;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;

  const int b = blockIdx.x / k.C;
  const int lo = static_cast<int>(k.rank) * P.L;
  const int n = max(0, min(P.V, lo + P.L) - lo);
  E *st = reinterpret_cast<E *>(smem + P.off_stage_t);
  E *sd = reinterpret_cast<E *>(smem + P.off_stage_d);
  Lists Ls;
  Ls.p_idx = reinterpret_cast<int *>(smem + P.off_lp);
  Ls.p_zp = reinterpret_cast<float *>(Ls.p_idx + P.cap);
  Ls.p_zq = Ls.p_zp + P.cap;
  Ls.q_idx = reinterpret_cast<int *>(Ls.p_zq + P.cap);
  Ls.q_zq = reinterpret_cast<float *>(Ls.q_idx + P.cap);
  Ls.w_p = reinterpret_cast<uint32_t *>(smem + P.off_w);
  Ls.w_q = Ls.w_p + P.cap;
  Ls.key_p = reinterpret_cast<uint64_t *>(smem + P.off_hist);
  Ls.key_q = Ls.key_p + SORT_MAX;
  Ls.hist_p = Ls.key_q + SORT_MAX;
  Ls.hist_q = Ls.hist_p + NBINS;
  const E *tg = static_cast<const E *>(P.tgt);
  const E *dg = static_cast<const E *>(P.drf);

  Chunks<E> ch;
  ch.make(n);
  uint32_t ph_t = 0, ph_d = 0;
  bool timed_out = false;
  if (VEC) {
    if (tid == 0) {
      for (int j = 0; j < 2 * NCH; ++j) mbar_init(&bars[j], 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
  }

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

    // ---- pass 1: HBM -> SMEM (bulk copies), statistics
    __syncthreads();  // every reader of the staging buffers is done
    const E *trow = tg + static_cast<int64_t>(b) * P.t_row + static_cast<int64_t>(i) * P.t_pos + lo;
    const E *drow = dg + static_cast<int64_t>(b) * P.d_row + static_cast<int64_t>(i) * P.d_pos + lo;
    // pass 1 in its greedy (first argmax) or sampling (max only) form
    float a_mx, c_mx;
    int a_mi;
    uint32_t a_fl, c_fl;
    {
      auto run = [&](auto arg_tag) {
        constexpr bool ARG = decltype(arg_tag)::value;
        TStat<ARG> a, c;
        a.init();
        c.init();
        if (VEC) {
          if (tid == 0) {
            fence_proxy_async();
            issue_slice<E>(trow, st, ch, bars);
            if (two) issue_slice<E>(drow, sd, ch, bars + NCH);
          }
          scan_slice<E>(trow, st, ch, n, lo, bars, ph_t, a);
          ph_t ^= 1u;
          if (two) {
            scan_slice<E>(drow, sd, ch, n, lo, bars + NCH, ph_d, c);
            ph_d ^= 1u;
          }
          if (a.to | c.to) timed_out = true;
        } else {
          load_slice_plain<E>(trow, st, n, lo, a);
          if (two) load_slice_plain<E>(drow, sd, n, lo, c);
        }
        a_mx = a.mx;
        a_mi = ARG ? a.mi : INT_MAX;
        a_fl = a.flags();
        c_mx = c.mx;
        c_fl = c.flags();
      };
      if (P.greedy)
        run(std::true_type{});
      else
        run(std::false_type{});
    }
    {
      float am = a_mx;
      int ai = a_mi;
      warp_argmax(am, ai);
      const uint32_t af = warp_or(a_fl), cf = warp_or(c_fl);
      const float cm = warp_max(c_mx);
      if (lane == 0) {
        wstat[wid * 8 + 0] = __float_as_uint(am);
        wstat[wid * 8 + 1] = static_cast<uint32_t>(ai);
        wstat[wid * 8 + 2] = af;
        wstat[wid * 8 + 3] = __float_as_uint(cm);
        wstat[wid * 8 + 4] = cf;
      }
      if (P.kc > 0) {  // per-warp top-TOPR of the per-thread maxima
        float va = a_mx, vc = c_mx;
#pragma unroll
        for (int r = 0; r < TOPR; ++r) {
          const float ma = warp_max(va), mc = warp_max(vc);
          if (lane == r) {
            cand[0][wid * TOPR + r] = ma;
            cand[1][wid * TOPR + r] = mc;
          }
          const uint32_t ba = __ballot_sync(0xffffffffu, va == ma);
          const uint32_t bc = __ballot_sync(0xffffffffu, vc == mc);
          if (lane == __ffs(ba) - 1) va = -INFINITY;
          if (lane == __ffs(bc) - 1) vc = -INFINITY;
        }
      }
      __syncthreads();
      if (wid < 2) {  // warp 0: target statistics; warp 1: draft statistics
        const int o = wid ? 3 : 0;
        float v = lane < NW ? __uint_as_float(wstat[lane * 8 + o]) : -INFINITY;
        int vi = (lane < NW && !wid) ? static_cast<int>(wstat[lane * 8 + 1]) : INT_MAX;
        uint32_t f = lane < NW ? wstat[lane * 8 + o + (wid ? 1 : 2)] : 0u;
        if (wid == 0)
          warp_argmax(v, vi);
        else
          v = warp_max(v);
        f = warp_or(f);
        float th = -INFINITY;
        if (P.kc > 0) {
          // k_c-th largest of this CTA's per-warp top lane maxima: at least
          // k_c elements of the slice are >= it
          float cv = lane < NW * TOPR ? cand[wid][lane] : -INFINITY;
          cv = warp_sort_desc(cv);
          th = __shfl_sync(0xffffffffu, cv, P.kc - 1);
        }
        if (lane == 0) {
          uint32_t *xs = xslot(k);
          if (wid == 0) {
            xs[0] = __float_as_uint(v);
            xs[1] = static_cast<uint32_t>(vi);
            xs[2] = f;
            xs[5] = __float_as_uint(th);
          } else {
            xs[3] = __float_as_uint(v);
            xs[4] = f;
            xs[6] = __float_as_uint(th);
          }
        }
      }
      xsync(k, 7);
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
      if ((bf | df) & F_TIMEOUT) status |= ST_TIMEOUT;
      if (bf & F_BAD) status |= ST_BAD_LOGIT;
      if (!(bf & F_FINITE)) status |= ST_NO_FINITE;
      if (two) {
        if (df & F_BAD) status |= ST_BAD_LOGIT;
        if (!(df & F_FINITE)) status |= ST_NO_FINITE;
      }
      dt.m = bm;
      dt.tau = -INFINITY;
      dt.list = 0;
      dt.n = 0;
      dt.Z = dt.rZ = ff{1.0f, 0.0f};
      dt.rzf = 1.0f;
      dt.zerr = 0.0f;
      dt.exact = 0;
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
    int all_t = 0, all_d = 0;
    if (filt && P.cap > 0) {
      float ct = -INFINITY, cd = -INFINITY;
      ff zall_t = {0.0f, 0.0f}, zall_d = {0.0f, 0.0f};
      if (P.k_on) {
        ct = thc_t;  // <= the k-th largest logit
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
      SV_PHASE(6);  // (top-p window)
      const bool vt = ct > -INFINITY, vd = two && cd > -INFINITY;
      int tot_t, tot_d, base_t, base_d;
      count_pass<E>(k, st, sd, n, ct, cd, vt, vd, wcnt, tot_t, tot_d, base_t, base_d);
      SV_PHASE(7);  // count pass
      uint32_t cw[2] = {static_cast<uint32_t>(tot_t), static_cast<uint32_t>(tot_d)};
      exchange(k, cw, 2);
      SV_PHASE(8);  // count exchange
      int offt[MAXC + 1], offd[MAXC + 1];
      offt[0] = offd[0] = 0;
      for (uint32_t cc = 0; cc < k.C; ++cc) {
        offt[cc + 1] = offt[cc] + static_cast<int>(gat[cc * 2]);
        offd[cc + 1] = offd[cc] + static_cast<int>(gat[cc * 2 + 1]);
      }
      all_t = offt[k.C];
      all_d = offd[k.C];
      lt = vt && all_t <= P.cap;
      ld = vd && all_d <= P.cap;
      if (lt || ld) {
        write_pass<E>(k, Ls, st, sd, n, lo, ct, cd, lt, ld, two, offt[k.rank] + base_t,
                      offd[k.rank] + base_d);
        SV_PHASE(9);  // write pass
        cluster_sync();
        pull_lists(k, Ls, offt, offd, all_t, all_d, lt, ld);
        __syncthreads();
        SV_PHASE(1);  // list sync
        // the p and q lists are processed by the two halves of the block
        const bool split = lt && ld;
        const int half = NT / 2;
        Grp g;
        if (split) {
          const int side = tid < half ? 0 : 1;
          g.t = tid - side * half;
          g.n = half;
          g.bar = 1 + side;
          g.red = gred[side];
          g.sc = gsc[side];
        } else {
          g.t = tid;
          g.n = NT;
          g.bar = 0;
          g.red = gred[0];
          g.sc = gsc[0];
        }
        for (int side = 0; side < 2; ++side) {
          const bool mine = split ? (tid < half) == (side == 0) : true;
          const bool want = side == 0 ? lt : ld;
          if (!mine || !want) continue;
          float tau, zerr;
          ff Z;
          const float *val = side == 0 ? Ls.p_zp : Ls.q_zq;
          const int nn = side == 0 ? all_t : all_d;
          const Dist &D = side == 0 ? dt : dd;
          uint32_t *w = side == 0 ? Ls.w_p : Ls.w_q;
          const ff za = side == 0 ? zall_t : zall_d;
          const int state =
              (nn > SMALL_SORTED && nn <= SORT_MAX)
                  ? g_list_sorted(P, g, val, nn, D.m, w, side == 0 ? Ls.key_p : Ls.key_q, za,
                                  D.zerr, tau, Z, zerr)
                  : g_list_fast(P, g, val, nn, D.m, w, side == 0 ? Ls.hist_p : Ls.hist_q, za,
                                D.zerr, tau, Z, zerr);
          if (g.t == 0) {
            lres[side][0] = static_cast<float>(state);
            lres[side][1] = tau;
            lres[side][2] = Z.hi;
            lres[side][3] = Z.lo;
            lres[side][4] = zerr;
          }
        }
        __syncthreads();
        const int st_t = lt ? static_cast<int>(lres[0][0]) : 0;
        const int st_d = ld ? static_cast<int>(lres[1][0]) : 0;
        if (st_t == 1) {
          dt.tau = lres[0][1];
          set_Zf(dt, ff{lres[0][2], lres[0][3]}, lres[0][4]);
        }
        if (st_d == 1) {
          dd.tau = lres[1][1];
          set_Zf(dd, ff{lres[1][2], lres[1][3]}, lres[1][4]);
        }
        __syncthreads();
        if (st_t == 2 || st_d == 2) {
          // a top-p comparison was within its error bound: redo it in
          // float-float (with an exact vocabulary normaliser for top-p alone)
          if (!P.k_on) {
            Dist xt = dt, xd = dd;
            slice_Z_exact<E>(P, k, st, sd, n, xt, xd, st_t == 2, st_d == 2);
            zall_t = xt.Z;
            zall_d = xd.Z;
          }
          const Grp gw = whole_block(k);
          for (int side = 0; side < 2; ++side) {
            if ((side == 0 ? st_t : st_d) != 2) continue;
            float tau;
            ff Z;
            const bool ok =
                side == 0 ? g_list_exact(P, gw, Ls.p_zp, all_t, dt.m, Ls.w_p, Ls.hist_p, zall_t,
                                         tau, Z)
                          : g_list_exact(P, gw, Ls.q_zq, all_d, dd.m, Ls.w_q, Ls.hist_q, zall_d,
                                         tau, Z);
            Dist &D = side == 0 ? dt : dd;
            if (ok) {
              D.tau = tau;
              set_Zx(D, Z);
            }
            if (side == 0) lt = ok; else ld = ok;
          }
          if (P.diag && k.rank == 0 && tid == 0) atomicAdd(P.diag + 3, 1u);
        }
        if (st_t == 0) lt = false;
        if (st_d == 0) ld = false;
        if (lt) {
          dt.list = 1;
          dt.n = all_t;
        }
        if (ld) {
          dd.list = 1;
          dd.n = all_d;
        }
      }
    }
    SV_PHASE(2);  // list selection
    const bool need_t = !lt, need_d = two && !ld;
    if (filt && (need_t || need_d)) {
      // exact slice-wide selection for the tensors without a list
      if (P.k_on) slice_bisect<E>(P, k, st, sd, n, dt, dd, need_t, need_d, false);
      if (P.p_on) slice_bisect<E>(P, k, st, sd, n, dt, dd, need_t, need_d, true);
      slice_Z_exact<E>(P, k, st, sd, n, dt, dd, need_t, need_d);
      if (P.diag && k.rank == 0 && tid == 0) atomicAdd(P.diag + 0, 1u);
    } else if (!filt) {
      ff z0, z1;
      slice_Z_fast<E>(P, k, st, sd, n, dt, dd, two, false, z0, z1, nullptr, nullptr, bandh);
    }
    SV_PHASE(3);  // slice fallback / fast Z

    // exact normalisers on demand (rare paths)
    auto make_exact = [&](bool wt, bool wd) {
      const Grp gw = whole_block(k);
      if (wt && !dt.exact) {
        if (dt.list)
          list_make_exact(P, gw, Ls.p_zp, dt.n, dt);
        else
          slice_Z_exact<E>(P, k, st, sd, n, dt, dd, true, false);
      }
      if (wd && !dd.exact) {
        if (dd.list)
          list_make_exact(P, gw, Ls.q_zq, dd.n, dd);
        else
          slice_Z_exact<E>(P, k, st, sd, n, dt, dd, false, true);
      }
    };

    if (bonus) {
      const float u1 = ui[P.u_draw];
      if (!(u1 >= 0.0f && u1 < 1.0f)) {
        status |= ST_BAD_UNIFORM;
        break;
      }
      float Wf;
      next = lt ? list_draw_fast(P, k, Ls, dt.n, dt, dd, false, u1, &Wf)
                : slice_draw_fast<E>(P, k, st, sd, n, lo, dt, dd, false, u1, &Wf);
      if (next < 0) {  // uncertain: exact redraw
        ff W;
        make_exact(true, false);
        next = lt ? list_draw(P, k, Ls, dt.n, dt, dd, false, u1, &W)
                  : slice_draw<E>(P, k, st, sd, n, lo, dt, dd, false, u1, &W);
        if (P.diag && k.rank == 0 && tid == 0) atomicAdd(P.diag + 1, 1u);
      }
      acc = gb;
      done = true;
      break;
    }

    // ---- acceptance test: u < p(x)/q(x), single precision with an error
    // bound, decided exactly when u falls within the bound (warp 0)
    const int64_t toff = static_cast<int64_t>(b) * P.t_row + static_cast<int64_t>(i) * P.t_pos + x;
    const int64_t doff = static_cast<int64_t>(b) * P.d_row + static_cast<int64_t>(i) * P.d_pos + x;
    if (wid == 0) {
      const float zx = raw_of(tg[toff]);
      const float wx = raw_of(dg[doff]);
      const bool kp = zx >= dt.tau && zx != -INFINITY;
      const bool kq = wx >= dd.tau && wx != -INFINITY;
      int verdict;  // 1 accept, 0 reject, 2 uncertain
      float pdbg = 0.0f, qdbg = 0.0f;
      const float yp = __fmul_rn(__fsub_rn(zx, dt.m), P.c2);
      const float yq = __fmul_rn(__fsub_rn(wx, dd.m), P.c2);
      if (kp) pdbg = __fmul_rn(ex2_approx(yp), dt.rzf);
      if (kq) qdbg = __fmul_rn(ex2_approx(yq), dd.rzf);
      if (!kq) {
        verdict = kp ? 1 : 0;  // the limit of min(1, p/q) as q -> 0
      } else if (!kp) {
        verdict = 0;  // ratio 0
      } else if (u0 == 0.0f) {
        verdict = 1;  // 0 < p/q
      } else {
        const float d = __fsub_rn(yp, yq);
        const float r = __fmul_rn(ex2_approx(d), __fmul_rn(dd.Z.hi, dt.rzf));
        const float eps = __fadd_rn(
            __fmaf_rn(__fadd_rn(__fadd_rn(fabsf(yp), fabsf(yq)), fabsf(d)), kExpErr1, kExpErr0),
            __fadd_rn(__fadd_rn(dt.zerr, dd.zerr), 1.2e-6f));
        if (r == INFINITY || u0 < __fmul_rn(r, 1.0f - eps))
          verdict = 1;
        else if (u0 >= __fmul_rn(r, 1.0f + eps) && r > 0.0f)
          verdict = 0;
        else
          verdict = 2;
      }
      if (lane == 0) {
        scal[11] = verdict;
        scal[12] = kq ? 0 : ST_Q_ZERO;
        if (k.rank == 0) {
          if (P.p_dbg) P.p_dbg[static_cast<int64_t>(b) * P.gm + i] = pdbg;
          if (P.q_dbg) P.q_dbg[static_cast<int64_t>(b) * P.gm + i] = qdbg;
        }
      }
    }
    __syncthreads();
    int verdict = scal[11];
    status |= scal[12];
    __syncthreads();
    if (verdict == 2) {  // exact decision in float-float
      make_exact(true, true);
      if (wid == 0) {
        const float zx = raw_of(tg[toff]);
        const float wx = raw_of(dg[doff]);
        const ff yp = scaled_gap(P, zx, dt.m), yq = scaled_gap(P, wx, dd.m);
        const ff ratio = ff_mul(ff_exp(ff_sub(yp, yq)), ff_mul(dd.Z, dt.rZ));
        if (lane == 0) scal[11] = ff_lt(ff_make(u0), ratio) ? 1 : 0;
      }
      __syncthreads();
      verdict = scal[11];
      __syncthreads();
      if (P.diag && k.rank == 0 && tid == 0) atomicAdd(P.diag + 1, 1u);
    }
    SV_PHASE(4);  // acceptance
    if (verdict == 1) continue;

    // ---- first rejection: draw from norm(max(0, p - q))
    const float u1 = ui[P.u_draw];
    if (!(u1 >= 0.0f && u1 < 1.0f)) {
      status |= ST_BAD_UNIFORM;
      break;
    }
    float Wf;
    int tok = lt ? list_draw_fast(P, k, Ls, dt.n, dt, dd, true, u1, &Wf)
                 : slice_draw_fast<E>(P, k, st, sd, n, lo, dt, dd, true, u1, &Wf);
    resid = Wf;  // residual mass sum max(0, p - q)
    if (tok < 0) {  // uncertain, or an (almost) empty residual: exact redraw
      ff W;
      make_exact(true, true);
      tok = lt ? list_draw(P, k, Ls, dt.n, dt, dd, true, u1, &W)
               : slice_draw<E>(P, k, st, sd, n, lo, dt, dd, true, u1, &W);
      resid = W.hi + W.lo;
      if (tok < 0)
        tok = lt ? list_draw(P, k, Ls, dt.n, dt, dd, false, u1, &W)
                 : slice_draw<E>(P, k, st, sd, n, lo, dt, dd, false, u1, &W);
      if (P.diag && k.rank == 0 && tid == 0) atomicAdd(P.diag + 1, 1u);
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
  if (k.rank == 0 && tid == 0) {
    if (P.acc) P.acc[b] = acc;
    P.next[b] = next;
    if (P.st_dbg) P.st_dbg[b] = status;
    if (P.res_dbg) P.res_dbg[b] = (status & ST_ERROR) ? 0.0f : resid;
    if ((status & ST_TIMEOUT) && P.diag) atomicAdd(P.diag + 2, 1u);
  }
  if (VEC && timed_out && tid == 0) {
    // let copies that outlived a timed-out wait land before the CTA exits
    for (int j = 0; j < NCH; ++j) (void)mbar_wait(&bars[j], ph_t ^ 1u, kWaitPolls);
    for (int j = 0; j < NCH; ++j) (void)mbar_wait(&bars[NCH + j], ph_d ^ 1u, kWaitPolls);
  }
  cluster_sync();  // no CTA leaves while a peer may still read its shared memory
}

// Debug p/q outputs are NaN unless a position is evaluated.
__global__ void fill_nan_kernel(float *p, int64_t n) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) p[i] = __int_as_float(0x7fc00000);
}

}  // namespace sv

namespace sv {

constexpr int kDiagWords = 4;  // see spec_read_diagnostics

spec_status check_verify_args(const void *target, const void *draft, const int32_t *tokens,
                              const float *uniforms, const spec_params *pp, const int32_t *acc,
                              const int32_t *next, const void *ws, size_t ws_bytes,
                              bool sample_mode) {
  if (!pp) return SPEC_ERR_INVALID_ARG;
  const spec_params p = *pp;
  if (p.B < 0 || p.gamma_max < 0 || p.V < 1 || p.V > (1 << 24)) return SPEC_ERR_INVALID_ARG;
  if (p.B == 0) return SPEC_OK;
  if (p.dtype != SPEC_F32 && p.dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (!std::isfinite(p.temperature) || p.temperature < 0.0f) return SPEC_ERR_INVALID_ARG;
  if (p.temperature > 0.0f && p.temperature < 1e-30f) return SPEC_ERR_INVALID_ARG;
  if (!(p.top_p > 0.0f)) return SPEC_ERR_INVALID_ARG;  // also NaN
  if ((p.flags & ~SPEC_FLAG_CLUSTER_KERNEL) != 0) return SPEC_ERR_INVALID_ARG;
  if (p.cluster_size != 0 && p.cluster_size != 1 && p.cluster_size != 2 &&
      p.cluster_size != 4 && p.cluster_size != 8)
    return SPEC_ERR_INVALID_ARG;
  if (p.list_capacity < 0 || p.list_capacity > 8192) return SPEC_ERR_INVALID_ARG;
  if (p.target_pos_stride < 0 || p.target_row_stride < 0 || p.draft_pos_stride < 0 ||
      p.draft_row_stride < 0)
    return SPEC_ERR_INVALID_ARG;
  if (static_cast<int64_t>(p.B) * MAXC > INT32_MAX) return SPEC_ERR_INVALID_ARG;
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
  return SPEC_OK;
}

}  // namespace sv


// ====================================================================== host
namespace {

using namespace sv;

constexpr size_t kMaxSmem = 200 * 1024;  // dynamic shared memory per CTA


using KernelFn = void (*)(KP);

template <typename E, bool VEC, int NT>
KernelFn kernel_ptr() {
  return verify_kernel<E, VEC, NT>;
}

KernelFn pick_kernel(int dtype, bool vec, int nt) {
  if (dtype == SPEC_F32) {
    if (vec) return nt == 256 ? kernel_ptr<float, true, 256>() : kernel_ptr<float, true, 128>();
    return nt == 256 ? kernel_ptr<float, false, 256>() : kernel_ptr<float, false, 128>();
  }
  if (vec) return nt == 256 ? kernel_ptr<uint16_t, true, 256>() : kernel_ptr<uint16_t, true, 128>();
  return nt == 256 ? kernel_ptr<uint16_t, false, 256>() : kernel_ptr<uint16_t, false, 128>();
}

cudaError_t prepare_kernel(KernelFn f) {
  static std::mutex mu;
  static std::map<KernelFn, cudaError_t> done;
  std::lock_guard<std::mutex> g(mu);
  auto it = done.find(f);
  if (it != done.end()) return it->second;
  const cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void *>(f),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kMaxSmem));
  done[f] = e;
  return e;
}

cudaLaunchConfig_t launch_cfg(int C, int nt, size_t smem, unsigned grid, cudaStream_t stream,
                              cudaLaunchAttribute *at) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(nt), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = static_cast<unsigned>(C);
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cfg;
}

int active_clusters(KernelFn f, int C, int nt, size_t smem) {
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = launch_cfg(C, nt, smem, static_cast<unsigned>(C) * 64u, nullptr, at);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void *>(f), &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

inline int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

struct Plan {
  int C = 1, NT = 256, L = 0, cap = 0;
  int64_t off_d = 0, off_lp = 0, off_w = 0, off_hist = 0;
  size_t smem = 0;
  bool vec = false;
};

// Shared-memory plan for a cluster size and block size.
Plan plan_for(const spec_params &p, bool sampling, int es, bool aligned, int C, int nt) {
  Plan pl;
  pl.C = C;
  pl.NT = nt;
  pl.L = static_cast<int>(align_up((static_cast<int64_t>(p.V) + C - 1) / C, 8));
  pl.vec = aligned;
  const bool filt = sampling && ((p.top_k > 0 && p.top_k < p.V) || p.top_p < 1.0f);
  const bool k_on = p.top_k > 0 && p.top_k < p.V;
  int auto_cap = 2048;
  if (k_on) {  // the top-k candidates number about k plus a margin
    auto_cap = 256;
    while (auto_cap < 2 * p.top_k + 64 && auto_cap < 8192) auto_cap *= 2;
  }
  pl.cap = !filt ? 0 : (p.list_capacity > 0 ? (p.list_capacity + 3) & ~3 : auto_cap);
  const int64_t one = align_up(static_cast<int64_t>(pl.L) * es, 128);
  pl.off_d = one;
  const int64_t stage = sampling ? 2 * one : one;
  pl.off_lp = stage;
  pl.off_w = align_up(pl.off_lp + 20ll * pl.cap, 16);
  pl.off_hist = align_up(pl.off_w + 8ll * pl.cap, 16);
  // sort keys for lists up to SORT_MAX; value histograms for longer lists
  pl.smem = static_cast<size_t>(
      pl.cap ? pl.off_hist + 2ll * 8 * SORT_MAX + (pl.cap > SORT_MAX ? 2ll * 8 * NBINS : 0)
             : stage);
  return pl;
}

// Block size: 256 threads for long slices, 128 for short ones.  Cluster
// size: the one that minimises (waves of resident clusters) x (slice length
// + a fixed per-position cost), among those whose slices fit.
Plan choose_plan(const spec_params &p, bool sampling, int es, bool aligned) {
  auto nt_for = [&](int C) {
    const int64_t L = (static_cast<int64_t>(p.V) + C - 1) / C;
    return L >= 4096 ? 256 : 128;
  };
  if (p.cluster_size) {
    const int C = p.cluster_size;
    return plan_for(p, sampling, es, aligned, C, nt_for(C));
  }
  Plan best;
  double best_cost = 0.0;
  bool have = false;
  for (int C = 1; C <= MAXC; C *= 2) {
    const int nt = nt_for(C);
    const Plan pl = plan_for(p, sampling, es, aligned, C, nt);
    if (pl.smem > kMaxSmem) continue;
    KernelFn f = pick_kernel(p.dtype, aligned, nt);
    if (prepare_kernel(f) != cudaSuccess) continue;
    const int act = active_clusters(f, C, nt, pl.smem);
    if (act <= 0) continue;
    const int64_t waves = (static_cast<int64_t>(p.B) + act - 1) / act;
    const double cost = static_cast<double>(waves) * (static_cast<double>(pl.L) * es + 6000.0);
    if (!have || cost < best_cost) {
      best = pl;
      best_cost = cost;
      have = true;
    }
  }
  return have ? best : plan_for(p, sampling, es, aligned, MAXC, nt_for(MAXC));
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
  const Plan pl = choose_plan(p, sampling, es, aligned);
  std::lock_guard<std::mutex> g(mu);
  if (cache.size() > 4096) cache.clear();
  cache[key] = pl;
  return pl;
}

// The kernel arguments of a verify call (sample_mode: of spec_sample), and
// whether every row starts on a 16-byte boundary (*aligned_out).
KP make_kp(const spec_params &p, const void *target, const void *draft, const int32_t *tokens,
           const float *uniforms, int32_t *acc, int32_t *next, const spec_debug *dbg, void *ws,
           bool sample_mode, bool *aligned_out) {
  const int es = p.dtype == SPEC_F32 ? 4 : 2;
  const bool greedy = p.temperature == 0.0f;
  const bool sampling = !greedy;
  *aligned_out =
      (reinterpret_cast<uintptr_t>(target) & 15) == 0 &&
      (!draft || (reinterpret_cast<uintptr_t>(draft) & 15) == 0) &&
      (p.target_pos_stride * es) % 16 == 0 && (p.target_row_stride * es) % 16 == 0 &&
      (p.draft_pos_stride * es) % 16 == 0 && (p.draft_row_stride * es) % 16 == 0;
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
  kp.acc = acc;
  kp.next = next;
  if (dbg) {
    kp.p_dbg = dbg->p_draft;
    kp.q_dbg = dbg->q_draft;
    kp.res_dbg = dbg->residual_mass;
    kp.st_dbg = dbg->row_status;
  }
  kp.diag = static_cast<unsigned int *>(ws);

  return kp;
}

spec_status run_verify(const void *target, const void *draft, const int32_t *tokens,
                       const float *uniforms, const spec_params *pp, int32_t *acc,
                       int32_t *next, const spec_debug *dbg, void *ws, size_t ws_bytes,
                       cudaStream_t stream, bool sample_mode) {
  const spec_status chk =
      check_verify_args(target, draft, tokens, uniforms, pp, acc, next, ws, ws_bytes, sample_mode);
  if (chk != SPEC_OK) return chk;
  const spec_params p = *pp;
  if (p.B == 0) return SPEC_OK;
  const bool force_cluster = (p.flags & SPEC_FLAG_CLUSTER_KERNEL) != 0;
  const bool greedy = p.temperature == 0.0f;
  const bool sampling = !greedy;
  bool aligned = false;
  KP kp = make_kp(p, target, draft, tokens, uniforms, acc, next, dbg, ws, sample_mode, &aligned);
  const int es = p.dtype == SPEC_F32 ? 4 : 2;

  // Small vocabularies, greedy or unfiltered: the warp-per-row kernel
  // (spec_row.cu), which needs no workspace.
  if (!force_cluster && row_eligible(p))
    return row_launch(kp, p.dtype, aligned, ws, ws_bytes, p, stream);

  // With a large enough workspace, the strip-parallel kernel (spec_strip.cu)
  // handles greedy and top-k problems.
  if (ws && !force_cluster) {
    const StripPlan sp = strip_plan(p);
    if (sp.ok && ws_bytes >= sp.ws_bytes) return strip_launch(kp, sp, ws, aligned, stream);
  }

  // the cluster-per-row kernel
  const Plan pl = cached_plan(p, sampling, es, aligned);
  if (pl.smem > kMaxSmem) return SPEC_ERR_UNSUPPORTED;  // vocabulary too large to stage
  kp.L = pl.L;
  kp.cap = pl.cap;
  kp.kc = 0;
  if (kp.k_on && pl.cap > 0) {
    const int kc = (p.top_k + pl.C - 1) / pl.C;
    kp.kc = kc <= (pl.NT / 32) * TOPR ? kc : 0;  // 0: no bound, exact slice selection
  }
  kp.off_stage_t = 0;
  kp.off_stage_d = static_cast<uint32_t>(pl.off_d);
  kp.off_lp = static_cast<uint32_t>(pl.off_lp);
  kp.off_w = static_cast<uint32_t>(pl.off_w);
  kp.off_hist = static_cast<uint32_t>(pl.off_hist);

  if (dbg && p.gamma_max > 0) {
    const int64_t nn = static_cast<int64_t>(p.B) * p.gamma_max;
    const unsigned blocks = static_cast<unsigned>((nn + 255) / 256);
    if (dbg->p_draft) fill_nan_kernel<<<blocks, 256, 0, stream>>>(dbg->p_draft, nn);
    if (dbg->q_draft) fill_nan_kernel<<<blocks, 256, 0, stream>>>(dbg->q_draft, nn);
    if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  }
  KernelFn f = pick_kernel(p.dtype, pl.vec, pl.NT);
  if (prepare_kernel(f) != cudaSuccess) return SPEC_ERR_CUDA;
  cudaLaunchAttribute at[1];
  cudaLaunchConfig_t cfg = launch_cfg(pl.C, pl.NT, pl.smem,
                                      static_cast<unsigned>(p.B) * static_cast<unsigned>(pl.C),
                                      stream, at);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, f, kp);
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
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

// The fixed device block behind spec_verify_noalloc: a static device array
// (allocated with the module, never by a call).
namespace {
constexpr size_t kNoAllocBytes = 64ull << 20;
static __device__ __align__(256) unsigned char noalloc_block[kNoAllocBytes];
constexpr int kMaxDevices = 64;

// Device address of the block on the current device (looked up once per
// device), or nullptr.
void *noalloc_base() {
  static std::mutex mu;
  static void *base[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> g(mu);
  if (!base[dev] && cudaGetSymbolAddress(&base[dev], noalloc_block) != cudaSuccess) {
    cudaGetLastError();
    base[dev] = nullptr;
  }
  return base[dev];
}
}  // namespace

extern "C" {

spec_status spec_verify_noalloc(const void *target_logits, const void *draft_logits,
                                const int32_t *draft_tokens, const float *uniforms,
                                const spec_params *params, int32_t *accepted_len,
                                int32_t *next_token, const spec_debug *debug, void *stream) {
  if (!params) return SPEC_ERR_INVALID_ARG;
  if (spec_verify_workspace_size(params) > kNoAllocBytes) return SPEC_ERR_WORKSPACE;
  void *ws = noalloc_base();
  if (!ws) return SPEC_ERR_CUDA;
  return run_verify(target_logits, draft_logits, draft_tokens, uniforms, params, accepted_len,
                    next_token, debug, ws, kNoAllocBytes, static_cast<cudaStream_t>(stream),
                    false);
}

size_t spec_verify_workspace_size(const spec_params *params) {
  const size_t diag = sv::kDiagWords * sizeof(uint32_t);
  if (!params) return diag;
  if (params->flags & SPEC_FLAG_CLUSTER_KERNEL) return diag;
  if (row_eligible(*params)) {  // the warp-per-row kernel (and its deferred-row list)
    const size_t d = row_defer_bytes(*params);
    return d > diag ? d : diag;
  }
  const StripPlan sp = strip_plan(*params);
  return sp.ok && sp.ws_bytes > diag ? sp.ws_bytes : diag;
}

spec_status spec_verify(const void *target_logits, const void *draft_logits,
                        const int32_t *draft_tokens, const float *uniforms,
                        const spec_params *params, int32_t *accepted_len, int32_t *next_token,
                        const spec_debug *debug, void *workspace, size_t workspace_bytes,
                        void *stream) {
  return run_verify(target_logits, draft_logits, draft_tokens, uniforms, params, accepted_len,
                    next_token, debug, workspace, workspace_bytes,
                    static_cast<cudaStream_t>(stream), false);
}

}  // extern "C"

namespace {
// The verify-shaped parameters of a law evaluation: one position per row
// (the row's target and draft logits at position 0), no draft lengths.
spec_params law_verify_params(const spec_params &p) {
  spec_params q = p;
  q.gamma_max = 1;
  q.target_pos_stride = p.V;
  q.draft_pos_stride = p.V;
  q.gamma_per_row = nullptr;
  q.flags = 0;
  return q;
}
bool law_filtered(const spec_params &p) {
  return p.temperature > 0.0f && ((p.top_k > 0 && p.top_k < p.V) || p.top_p < 1.0f);
}
}  // namespace

extern "C" {

size_t spec_law_workspace_size(const spec_params *params) {
  if (!params || !law_filtered(*params) || params->B < 1) return 0;
  const StripPlan pl = strip_plan(law_verify_params(*params), true);
  return pl.ok ? pl.ws_bytes : 0;
}

spec_status spec_law_ws(const void *target_logits, const void *draft_logits,
                        const int32_t *tokens, const spec_params *params, float *p_spec,
                        float *beta, float *p_token, float *q_token, void *workspace,
                        size_t workspace_bytes, void *stream) {
  const spec_status chk = law_check_args(target_logits, draft_logits, tokens, params, p_spec);
  if (chk != SPEC_OK) return chk;
  const spec_params &p = *params;
  if (p.B == 0) return SPEC_OK;
  const spec_params q = law_verify_params(p);
  const StripPlan pl = law_filtered(p) ? strip_plan(q, true) : StripPlan();
  if (!pl.ok || !workspace || workspace_bytes < pl.ws_bytes ||
      (reinterpret_cast<uintptr_t>(workspace) & 15) != 0)
    return spec_law(target_logits, draft_logits, tokens, params, p_spec, beta, p_token, q_token,
                    stream);
  bool aligned = false;
  const KP kp = make_kp(q, target_logits, draft_logits, tokens, nullptr, nullptr, nullptr, nullptr,
                        workspace, false, &aligned);
  float *const outs[4] = {p_spec, beta, p_token, q_token};
  return strip_launch(kp, pl, workspace, aligned, static_cast<cudaStream_t>(stream), outs);
}

spec_status spec_sample(const void *logits, const float *u, const spec_params *params,
                        int32_t *tokens, int32_t *row_status, void *stream) {
  spec_debug d = {nullptr, nullptr, nullptr, row_status};
  return run_verify(logits, nullptr, nullptr, u, params, nullptr, tokens, &d, nullptr, 0,
                    static_cast<cudaStream_t>(stream), true);
}

size_t spec_sample_workspace_size(const spec_params *params) {
  return spec_verify_workspace_size(params);
}

spec_status spec_sample_ws(const void *logits, const float *u, const spec_params *params,
                           int32_t *tokens, int32_t *row_status, void *workspace,
                           size_t workspace_bytes, void *stream) {
  spec_debug d = {nullptr, nullptr, nullptr, row_status};
  return run_verify(logits, nullptr, nullptr, u, params, nullptr, tokens, &d, workspace,
                    workspace_bytes, static_cast<cudaStream_t>(stream), true);
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
  const int m = n < sv::kDiagWords ? n : sv::kDiagWords;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(counters, workspace, m * sizeof(uint32_t), cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return SPEC_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SPEC_ERR_CUDA;
  for (int i = m; i < n; ++i) counters[i] = 0;
  return SPEC_OK;
}

}  // extern "C"
