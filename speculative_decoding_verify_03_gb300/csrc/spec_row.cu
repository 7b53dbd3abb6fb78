// spec_row.cu -- the verify step for small vocabularies, one warp per row.
//
// The method is the one of the other kernels: speculative sampling as in
// "Prepare speculative sampling" (OpenVINO notebook; steps 2-4: accept
// draft token x_i with probability min(1, p(x_i)/q(x_i)); at the first
// rejection draw from norm(max(0, p - q)); when every draft token is accepted
// draw the bonus token from p) and "CS3602_FINAL_SpeDec" section 2 (the
// output law of that rule is p).  Greedy decoding accepts while the target
// argmax equals the draft token.
//
// With V <= 1024 a whole row position (target and draft logits) fits in one
// warp's registers, 32 logits per lane, lane l holding the contiguous indices
// [32 l, 32 l + 32).  A warp walks the positions of its row in order and
// stops at the first rejection, so positions after it are never read.  There
// is no shared memory, no CTA barrier and no workspace: the only cross-lane
// traffic is shuffles.  The arithmetic is certified single precision with a
// float-float redo, as in the other kernels: the normalisers are compensated
// sums with an error bound, the acceptance ratio carries a relative error
// bound, and the inverse-CDF draw runs float-float prefix sums over
// single-precision weights whose absolute errors are summed; a decision
// closer to its boundary than the bound is recomputed in float-float.
// The sampling path keeps a row position in local memory (L1-resident) and
// runs rolled loops over it: fully unrolled per-element code made the
// kernel wait on instruction fetch; the greedy path keeps its logits in
// registers.
// Top-k / top-p are not handled here (the candidate-list kernels do that).
//
// When the call provides a workspace, a CTA of two warps walks each row
// instead (16 contiguous logits a thread, the same certified arithmetic),
// and a row whose decision is uncertain is handed to a second kernel that
// finishes it in float-float with 256 threads; without a workspace the warp
// per row redoes its uncertain decisions itself.
#include <cuda_runtime.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <climits>
#include <cmath>

#include "spec_verify.h"
#include "sv_core.cuh"
#include "sv_row.h"

// Phase timing for development builds (-DSV_PHASE_PROFILE): thread 0 of each
// row CTA accumulates clock64() deltas per phase, and counts, into a global
// array read by sv_row_phase_read().
#ifdef SV_PHASE_PROFILE
__device__ unsigned long long sv_row_cycles[64];
#define RC_PHASE(id)                                                                       \
  do {                                                                                     \
    if (threadIdx.x == 0) {                                                                \
      const long long now_ = clock64();                                                    \
      atomicAdd(&sv_row_cycles[id], static_cast<unsigned long long>(now_ - t_ph_));        \
      atomicAdd(&sv_row_cycles[32 + (id)], 1ull);                                          \
      t_ph_ = now_;                                                                        \
    }                                                                                      \
  } while (0)
#define RC_PHASE_START long long t_ph_ = clock64()
#else
#define RC_PHASE(id) \
  do {               \
  } while (0)
#define RC_PHASE_START \
  do {                 \
  } while (0)
#endif

namespace sv {

namespace {

// One warp per CTA: a CTA ends with its row, so long rows (many accepted
// positions) hold no other row's slot.
constexpr int RW_NT = 32;               // threads per CTA
constexpr int RW_ROWS = RW_NT / kWarp;  // rows per CTA (one per warp)
constexpr int RW_PL = kRowMaxV / kWarp; // logits per lane
constexpr unsigned RW_FULL = 0xffffffffu;
static_assert(RW_PL == 32, "32 logits per lane");

// A lane's logits, passed by value to the out-of-line (rare) paths so that
// the caller's copy stays in registers.
struct Lane32 {
  float v[RW_PL];
};

// The logits [32 lane, 32 lane + 32) of one row position (-inf past V).
template <typename E, bool VEC>
__device__ __forceinline__ void rw_load(const E *g, int V, int lane, float (&z)[RW_PL]) {
  const int v0 = lane * RW_PL;
  if (VEC && v0 + RW_PL <= V) {
    constexpr int EPV = Elem<E>::kPerVec;
    const uint4 *g4 = reinterpret_cast<const uint4 *>(g + v0);
#pragma unroll
    for (int j = 0; j < RW_PL / EPV; ++j) {
      float f[EPV];
      unpack<E>(__ldg(g4 + j), f);
#pragma unroll
      for (int e = 0; e < EPV; ++e) z[j * EPV + e] = canon(f[e]);
    }
  } else {
#pragma unroll
    for (int k = 0; k < RW_PL; ++k) z[k] = v0 + k < V ? Elem<E>::get(g[v0 + k]) : -INFINITY;
  }
}

// NaN-propagating warp maximum.
__device__ __forceinline__ float rw_max_nan(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = max_nan(v, __shfl_xor_sync(RW_FULL, v, o));
  return v;
}

__device__ __forceinline__ float rw_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(RW_FULL, v, o));
  return v;
}

// Row flags (pass-1 semantics of the other kernels): NaN or +inf is bad;
// nothing above -inf means no finite logit.  *m = the NaN-ignoring maximum.
__device__ __forceinline__ uint32_t rw_flags(const float (&z)[RW_PL], float *m) {
  float mx = -INFINITY, mxn = -INFINITY;
#pragma unroll 4
  for (int k = 0; k < RW_PL; ++k) {
    mx = fmaxf(mx, z[k]);
    mxn = max_nan(mxn, z[k]);
  }
  mx = warp_max(mx);
  mxn = rw_max_nan(mxn);
  *m = mx;
  return ((mxn != mxn || mx == INFINITY) ? F_BAD : 0u) | (mx > -INFINITY ? F_FINITE : 0u);
}

// The element at index x of the row (every lane gets it).
__device__ __forceinline__ float rw_at(const float (&z)[RW_PL], int x) {
  return __shfl_sync(RW_FULL, z[x & (RW_PL - 1)], x / RW_PL);
}

// Fast normalisers of the target row and the draft row (compensated sums of
// single-precision weights, each with a bound of its relative error), the
// two chains side by side; dd is set only when two.
__device__ __forceinline__ void rw_Z_fast2(const KP &P, const float (&z)[RW_PL],
                                           const float (&w)[RW_PL], bool two, Dist &dt,
                                           Dist &dd) {
  float s0 = 0.0f, c0 = 0.0f, E0 = 0.0f, s1 = 0.0f, c1 = 0.0f, E1 = 0.0f;
#pragma unroll 4
  for (int k = 0; k < RW_PL; ++k) {
    float eps0, eps1;
    const float e0 = fw(P, z[k], dt.m, eps0);
    const float e1 = fw(P, w[k], dd.m, eps1);  // w is all -inf when !two
    const float t0 = __fsub_rn(e0, c0), u0 = __fadd_rn(s0, t0);
    const float t1 = __fsub_rn(e1, c1), u1 = __fadd_rn(s1, t1);
    c0 = __fsub_rn(__fsub_rn(u0, s0), t0);
    c1 = __fsub_rn(__fsub_rn(u1, s1), t1);
    s0 = u0;
    s1 = u1;
    E0 = __fmaf_rn(e0, eps0, E0);
    E1 = __fmaf_rn(e1, eps1, E1);
  }
  const ff Z0 = warp_sum_ff(quick_two_sum(s0, -c0));
  const ff Z1 = warp_sum_ff(quick_two_sum(s1, -c1));
  E0 = rw_sum(E0);
  E1 = rw_sum(E1);
  set_Zf(dt, Z0, __fadd_rn(__fdiv_rn(E0, Z0.hi), 2.4e-7f));
  if (two) set_Zf(dd, Z1, __fadd_rn(__fdiv_rn(E1, Z1.hi), 2.4e-7f));
}

// Float-float weight e^{(z - m)/T} (0 for -inf and underflow): the
// branch-free core of ff_exp with the out-of-range inputs selected away, so
// that the unrolled loops below run several exponentials side by side.
__device__ __forceinline__ ff rw_weight_ff(const KP &P, float z, float m) {
  const ff y = scaled_gap(P, z, m);
  const bool lo = !(y.hi > -104.0f), hi = y.hi > 88.0f;  // NaN: lo
  const ff yc = {lo ? -104.0f : (hi ? 88.0f : y.hi), (lo || hi) ? 0.0f : y.lo};
  const ff e = ff_exp_core(yc);
  if (z == -INFINITY || lo) return {0.0f, 0.0f};
  return hi ? ff{__int_as_float(0x7f800000), 0.0f} : e;
}

// Exact (float-float) normalisers of the target and, if two, the draft row.
struct RwZ {
  ff t, d;
};
__device__ __noinline__ RwZ rw_exact_Z(const KP &P, const Lane32 z, const Lane32 w, float mt,
                                       float md, bool two) {
  ff a = {0.0f, 0.0f}, c = {0.0f, 0.0f};
#pragma unroll 4
  for (int k = 0; k < RW_PL; ++k) {
    a = ff_add(a, rw_weight_ff(P, z.v[k], mt));
    if (two) c = ff_add(c, rw_weight_ff(P, w.v[k], md));
  }
  return {warp_sum_ff(a), warp_sum_ff(c)};
}
__device__ __forceinline__ Lane32 rw_copy(const float (&z)[RW_PL]) {
  Lane32 c;
#pragma unroll 4
  for (int k = 0; k < RW_PL; ++k) c.v[k] = z[k];
  return c;
}

// Single-precision draw weight w (p, or max(0, p - q)) of one token and a
// bound of its absolute error; exactly zero for a -inf logit.
__device__ __forceinline__ void rw_weight(const KP &P, float x, float y, const Dist &dt,
                                          const Dist &dd, bool residual, float &w, float &err) {
  w = 0.0f;
  err = 0.0f;
  if (x == -INFINITY) return;
  const float yx = __fmul_rn(__fsub_rn(x, dt.m), P.c2);
  const float p = __fmul_rn(ex2_approx(yx), dt.rzf);
  const float ep = __fmul_rn(p, __fmaf_rn(fabsf(yx), kExpErr1, kExpErr0 + dt.zerr + 2.4e-7f));
  if (!residual) {
    w = p;
    err = ep;
    return;
  }
  float q = 0.0f, eq = 0.0f;
  if (y != -INFINITY) {
    const float yy = __fmul_rn(__fsub_rn(y, dd.m), P.c2);
    q = __fmul_rn(ex2_approx(yy), dd.rzf);
    eq = __fmul_rn(q, __fmaf_rn(fabsf(yy), kExpErr1, kExpErr0 + dd.zerr + 2.4e-7f));
  }
  const float d = __fsub_rn(p, q);
  w = d > 0.0f ? d : 0.0f;
  err = __fadd_rn(__fadd_rn(ep, eq), __fmul_rn(__fadd_rn(p, q), 6.0e-8f));
}

// Exclusive float-float scan of the lanes' values; *total = the sum.
__device__ __forceinline__ ff rw_scan_ff(ff v, ff *total) {
  const int lane = threadIdx.x & 31;
  ff inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    ff u;
    u.hi = __shfl_up_sync(RW_FULL, inc.hi, o);
    u.lo = __shfl_up_sync(RW_FULL, inc.lo, o);
    if (lane >= o) inc = ff_add(u, inc);
  }
  total->hi = __shfl_sync(RW_FULL, inc.hi, 31);
  total->lo = __shfl_sync(RW_FULL, inc.lo, 31);
  ff ex;
  ex.hi = __shfl_up_sync(RW_FULL, inc.hi, 1);
  ex.lo = __shfl_up_sync(RW_FULL, inc.lo, 1);
  if (lane == 0) ex = {0.0f, 0.0f};
  return ex;
}

// Certified inverse-CDF draw in vocabulary order: the smallest v with
// u * W < C_v (C the prefix sums of the weights).  Float-float prefix sums
// over single-precision weights; the token is returned only when u * W lies
// more than twice the summed weight error (plus a rounding slack) inside its
// CDF interval; -2: uncertain, -1: total weight 0.  *Wf = the total weight.
__device__ __forceinline__ int rw_draw_fast(const KP &P, const float (&z)[RW_PL],
                                            const float (&w)[RW_PL], const Dist &dt,
                                            const Dist &dd, bool residual, float u, float *Wf) {
  const int lane = threadIdx.x & 31;
  // the lane's weights in four groups of 8 (group sums kept for the walk)
  ff gsum[4];
  ff s = {0.0f, 0.0f};
  float dsum = 0.0f;
#pragma unroll 1
  for (int g = 0; g < 4; ++g) {
    ff t = {0.0f, 0.0f};
#pragma unroll 4
    for (int kk = 0; kk < 8; ++kk) {
      float wk, ek;
      rw_weight(P, z[g * 8 + kk], w[g * 8 + kk], dt, dd, residual, wk, ek);
      t = ff_add_f(t, wk);
      dsum = __fadd_rn(dsum, ek);
    }
    gsum[g] = t;
    s = ff_add(s, t);
  }
  ff W;
  const ff a = rw_scan_ff(s, &W);
  const float D = rw_sum(dsum);
  *Wf = __fadd_rn(W.hi, W.lo);
  if (!(W.hi > 0.0f)) return -1;
  const float slack = __fmaf_rn(W.hi, 1e-12f, static_cast<float>(P.V) * 4e-38f *
                                                  (dt.rzf + (residual ? dd.rzf : 0.0f)));
  const ff target = ff_mul_f(W, u);
  const bool own = !ff_lt(target, a) && ff_lt(target, ff_add(a, s));
  int tok = -1, cert = 0;
  if (own) {
    ff c = a;
    int g = 0;
    for (; g < 3; ++g) {  // the group holding the target
      const ff cn = ff_add(c, gsum[g]);
      if (ff_lt(target, cn)) break;
      c = cn;
    }
    for (int kk = 0; kk < 8; ++kk) {
      const int k = g * 8 + kk;
      float wk, ek;
      rw_weight(P, z[k], w[k], dt, dd, residual, wk, ek);
      const ff cp = c;
      c = ff_add_f(c, wk);
      if (wk > 0.0f && ff_lt(target, c)) {
        tok = lane * RW_PL + k;
        const ff l = ff_sub(target, cp), h = ff_sub(c, target);
        cert = fminf(__fadd_rn(l.hi, l.lo), __fadd_rn(h.hi, h.lo)) > __fmaf_rn(2.0f, D, slack);
        break;
      }
    }
  }
  const uint32_t bal = __ballot_sync(RW_FULL, tok >= 0);
  if (!bal) return -2;
  const int L = __ffs(bal) - 1;
  tok = __shfl_sync(RW_FULL, tok, L);
  cert = __shfl_sync(RW_FULL, cert, L);
  return cert ? tok : -2;
}

// The same draw in float-float, from float-float weights computed once: the
// normalisers (set exact in dt and dd), then the weights max(0, p - q) (or p)
// and their prefix sums.  Returns the token, the last positive weight when
// rounding leaves u * W past it, or -1 (total weight 0); *Wf = the total.
__device__ __noinline__ int rw_draw_exact(const KP &P, const Lane32 z, const Lane32 w, float mt,
                                          float md, bool residual, float u, float *Wf) {
  const int lane = threadIdx.x & 31;
  ff ep[RW_PL], eq[RW_PL];
  ff a = {0.0f, 0.0f}, c = {0.0f, 0.0f};
#pragma unroll 4
  for (int k = 0; k < RW_PL; ++k) {
    ep[k] = rw_weight_ff(P, z.v[k], mt);
    eq[k] = residual ? rw_weight_ff(P, w.v[k], md) : ff{0.0f, 0.0f};
    a = ff_add(a, ep[k]);
    c = ff_add(c, eq[k]);
  }
  const ff rZt = ff_div(ff{1.0f, 0.0f}, warp_sum_ff(a));
  const ff rZd = residual ? ff_div(ff{1.0f, 0.0f}, warp_sum_ff(c)) : ff{0.0f, 0.0f};
  ff s = {0.0f, 0.0f};
  int last = -1;
  for (int k = 0; k < RW_PL; ++k) {
    ff p = ff_mul(ep[k], rZt);
    if (residual) p = ff_sub(p, ff_mul(eq[k], rZd));
    ep[k] = p.hi > 0.0f ? p : ff{0.0f, 0.0f};
    if (ep[k].hi > 0.0f) last = lane * RW_PL + k;
    s = ff_add(s, ep[k]);
  }
  ff W;
  const ff a0 = rw_scan_ff(s, &W);
  last = warp_max_i32(last);
  *Wf = __fadd_rn(W.hi, W.lo);
  if (!(W.hi > 0.0f)) return -1;
  const ff target = ff_mul_f(W, u);
  int tok = -1;
  if (!ff_lt(target, a0) && ff_lt(target, ff_add(a0, s))) {
    ff cc = a0;
    for (int k = 0; k < RW_PL; ++k) {
      if (ep[k].hi > 0.0f) tok = lane * RW_PL + k;
      cc = ff_add(cc, ep[k]);
      if (ep[k].hi > 0.0f && ff_lt(target, cc)) break;
    }
  }
  const uint32_t bal = __ballot_sync(RW_FULL, tok >= 0);
  if (!bal) return last;
  return __shfl_sync(RW_FULL, tok, __ffs(bal) - 1);
}

// Rows whose certified decision was uncertain can be handed to a second
// kernel (when the call has a workspace): the warp records (row, position,
// status so far) and stops; row_redo_kernel finishes the row from that
// position in float-float with a whole CTA, so that one uncertain row no
// longer holds a lone warp for the time of 64 float-float exponentials a lane.
struct RowDefer {
  uint32_t *count;  // rows deferred (nullptr: uncertain decisions are redone in the warp)
  int4 *list;       // [B]: row, position, status, 0
};

__device__ __forceinline__ void rw_defer(const RowDefer &D, int b, int i, int status) {
  if ((threadIdx.x & 31) == 0) {
    const uint32_t k = atomicAdd(D.count, 1u);
    D.list[k] = make_int4(b, i, status, 0);
  }
}

__device__ void rw_bad_row(const KP &P, int b) {
  if (P.acc) P.acc[b] = 0;
  P.next[b] = -1;
  if (P.st_dbg) P.st_dbg[b] = ST_BAD_GAMMA;
  if (P.res_dbg) P.res_dbg[b] = 0.0f;
  const float nan = __int_as_float(0x7fc00000);
  for (int j = 0; j < P.gm; ++j) {
    if (P.p_dbg) P.p_dbg[static_cast<int64_t>(b) * P.gm + j] = nan;
    if (P.q_dbg) P.q_dbg[static_cast<int64_t>(b) * P.gm + j] = nan;
  }
}

template <typename E, bool VEC>
__global__ void __launch_bounds__(RW_NT) row_kernel(const __grid_constant__ KP P, RowDefer D) {
  const int lane = threadIdx.x & 31;
  const int b = static_cast<int>(blockIdx.x) * RW_ROWS + static_cast<int>(threadIdx.x >> 5);
  if (b >= P.B) return;
  const int gb = P.gam ? P.gam[b] : P.gm;
  if (gb < 0 || gb > P.gm) {
    if (lane == 0) rw_bad_row(P, b);
    return;
  }
  const E *tb = static_cast<const E *>(P.tgt) + static_cast<int64_t>(b) * P.t_row;
  const E *db = static_cast<const E *>(P.drf) + static_cast<int64_t>(b) * P.d_row;
  const float *ub = P.uni ? P.uni + static_cast<int64_t>(b) * P.u_row : nullptr;
  int status = 0, token = -1, r = gb, tested = 0;
  float resid = 0.0f;
  for (int i = 0; i <= gb; ++i) {
    const bool bonus = i == gb;
    int x = -1;
    if (!bonus) {
      x = P.tok[static_cast<int64_t>(b) * P.gm + i];
      if (x < 0 || x >= P.V) status |= ST_BAD_TOKEN;
    }
    if (P.greedy) {
      // the first maximum in index order, and the row flags (registers)
      float zg[RW_PL];
      rw_load<E, VEC>(tb + static_cast<int64_t>(i) * P.t_pos, P.V, lane, zg);
      float v = -INFINITY;
      int vi = INT_MAX;
      bool nan = false;
#pragma unroll
      for (int k = 0; k < RW_PL; ++k) {
        nan |= zg[k] != zg[k];
        if (zg[k] > v) {
          v = zg[k];
          vi = lane * RW_PL + k;
        }
      }
      warp_argmax(v, vi);
      nan = __any_sync(RW_FULL, nan);
      if (nan || v == INFINITY) status |= ST_BAD_LOGIT;
      if (!(v > -INFINITY)) status |= ST_NO_FINITE;
      if (status & ST_ERROR) {
        r = i;
        break;
      }
      if (!bonus && vi == x) continue;  // accepted
      token = vi;
      r = i;
      break;
    }
    // both rows' loads in flight together (one memory latency per position)
    float z[RW_PL], w[RW_PL];
    rw_load<E, VEC>(tb + static_cast<int64_t>(i) * P.t_pos, P.V, lane, z);
    if (!bonus) {
      rw_load<E, VEC>(db + static_cast<int64_t>(i) * P.d_pos, P.V, lane, w);
    } else {
#pragma unroll 4
      for (int k = 0; k < RW_PL; ++k) w[k] = -INFINITY;
    }
    float mt;
    const uint32_t ft = rw_flags(z, &mt);
    if (ft & F_BAD) status |= ST_BAD_LOGIT;
    if (!(ft & F_FINITE)) status |= ST_NO_FINITE;
    float md = -INFINITY;
    if (!bonus) {
      const uint32_t fd = rw_flags(w, &md);
      if (fd & F_BAD) status |= ST_BAD_LOGIT;
      if (!(fd & F_FINITE)) status |= ST_NO_FINITE;
    }
    const float *ui = ub + static_cast<int64_t>(i) * P.u_pos;
    float u0 = 0.0f;
    if (!bonus) {
      u0 = ui[P.u_acc];
      if (!(u0 >= 0.0f && u0 < 1.0f)) status |= ST_BAD_UNIFORM;
    }
    if (status & ST_ERROR) {
      r = i;
      break;
    }
    Dist dt, dd;
    dist_init(dt, mt);
    dist_init(dd, md);
    rw_Z_fast2(P, z, w, !bonus, dt, dd);
    if (!bonus) {
      // acceptance u < p(x)/q(x): single precision with an error bound, in
      // float-float when u falls within the bound
      const float zx = rw_at(z, x), wx = rw_at(w, x);
      const bool kp = zx != -INFINITY, kq = wx != -INFINITY;
      const float yp = __fmul_rn(__fsub_rn(zx, dt.m), P.c2);
      const float yq = __fmul_rn(__fsub_rn(wx, dd.m), P.c2);
      const float pf = kp ? __fmul_rn(ex2_approx(yp), dt.rzf) : 0.0f;
      const float qf = kq ? __fmul_rn(ex2_approx(yq), dd.rzf) : 0.0f;
      int v;
      if (!kq) {
        v = kp ? 1 : 0;  // the limit of min(1, p/q) as q -> 0
      } else if (!kp) {
        v = 0;
      } else if (u0 == 0.0f) {
        v = 1;
      } else {
        const float d = __fsub_rn(yp, yq);
        const float rr = __fmul_rn(ex2_approx(d), __fmul_rn(dd.Z.hi, dt.rzf));
        const float eps = __fadd_rn(
            __fmaf_rn(__fadd_rn(__fadd_rn(fabsf(yp), fabsf(yq)), fabsf(d)), kExpErr1, kExpErr0),
            __fadd_rn(__fadd_rn(dt.zerr, dd.zerr), 1.2e-6f));
        if (rr == INFINITY || u0 < __fmul_rn(rr, 1.0f - eps))
          v = 1;
        else if (u0 >= __fmul_rn(rr, 1.0f + eps) && rr > 0.0f)
          v = 0;
        else
          v = 2;
      }
      if (v == 2 && D.count) {  // to the second kernel
        rw_defer(D, b, i, status);
        return;
      }
      if (v == 2) {  // exact decision in float-float
        const RwZ X = rw_exact_Z(P, rw_copy(z), rw_copy(w), dt.m, dd.m, true);
        set_Zx(dt, X.t);
        set_Zx(dd, X.d);
        const ff ratio = ff_mul(ff_exp(ff_sub(scaled_gap(P, zx, dt.m), scaled_gap(P, wx, dd.m))),
                                ff_mul(dd.Z, dt.rZ));
        v = ff_lt(ff_make(u0), ratio) ? 1 : 0;
        if (P.diag && lane == 0) atomicAdd(P.diag + 1, 1u);
      }
      if (!kq) status |= ST_Q_ZERO;
      tested = i + 1;
      if (lane == 0) {
        if (P.p_dbg) P.p_dbg[static_cast<int64_t>(b) * P.gm + i] = pf;
        if (P.q_dbg) P.q_dbg[static_cast<int64_t>(b) * P.gm + i] = qf;
      }
      if (v) continue;  // accepted
    }
    // the draw at position i: the residual at a rejection, p at the bonus
    r = i;
    const float u1 = ui[P.u_draw];
    if (!(u1 >= 0.0f && u1 < 1.0f)) {
      status |= ST_BAD_UNIFORM;
      break;
    }
    const bool residual = !bonus;
    float W = 0.0f, Wp = 0.0f;
    int t1 = rw_draw_fast(P, z, w, dt, dd, residual, u1, &W);
    if (t1 < 0 && D.count) {  // to the second kernel (it redoes position i whole)
      rw_defer(D, b, i, status);
      return;
    }
    if (t1 < 0) {  // uncertain, or an (almost) empty residual: exact redraw
      const Lane32 lz = rw_copy(z), lw = rw_copy(w);
      t1 = rw_draw_exact(P, lz, lw, dt.m, dd.m, residual, u1, &W);
      if (t1 < 0) t1 = rw_draw_exact(P, lz, lw, dt.m, dd.m, false, u1, &Wp);  // empty residual
      if (P.diag && lane == 0) atomicAdd(P.diag + 1, 1u);
    }
    token = t1;
    if (residual) resid = W;
    break;
  }
  if (lane == 0) {
    const bool err = (status & ST_ERROR) != 0;
    if (P.acc) P.acc[b] = err ? 0 : r;
    P.next[b] = err ? -1 : token;
    if (P.st_dbg) P.st_dbg[b] = status;
    if (P.res_dbg) P.res_dbg[b] = err ? 0.0f : resid;
    const float nan = __int_as_float(0x7fc00000);
    for (int j = tested; j < P.gm; ++j) {
      if (P.p_dbg) P.p_dbg[static_cast<int64_t>(b) * P.gm + j] = nan;
      if (P.q_dbg) P.q_dbg[static_cast<int64_t>(b) * P.gm + j] = nan;
    }
  }
}

// ------------------------------------------------------------ second pass
constexpr int RD_NT = 256;                // threads per CTA
constexpr int RD_PT = kRowMaxV / RD_NT;   // logits per thread (contiguous)
static_assert(RD_PT * RD_NT == kRowMaxV, "the CTA covers the largest vocabulary");

struct RdShared {
  ff red[RD_NT / 32];
  float fx[4];
  int ix[4];
};

__device__ __forceinline__ ff rd_sum(ff v, RdShared &sh) {
  v = warp_sum_ff(v);
  if ((threadIdx.x & 31) == 0) sh.red[threadIdx.x >> 5] = v;
  __syncthreads();
  ff t = {0.0f, 0.0f};
#pragma unroll
  for (int k = 0; k < RD_NT / 32; ++k) t = ff_add(t, sh.red[k]);
  __syncthreads();
  return t;
}
__device__ __forceinline__ float rd_max(float v, RdShared &sh) {
  v = warp_max(v);
  if ((threadIdx.x & 31) == 0) sh.red[threadIdx.x >> 5].hi = v;
  __syncthreads();
  float t = -INFINITY;
#pragma unroll
  for (int k = 0; k < RD_NT / 32; ++k) t = fmaxf(t, sh.red[k].hi);
  __syncthreads();
  return t;
}
// Exclusive scan in thread order (= vocabulary order: thread t holds the
// indices [RD_PT t, RD_PT (t + 1))); *total = the sum.
__device__ __forceinline__ ff rd_scan(ff v, RdShared &sh, ff *total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  ff inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    ff u;
    u.hi = __shfl_up_sync(RW_FULL, inc.hi, o);
    u.lo = __shfl_up_sync(RW_FULL, inc.lo, o);
    if (lane >= o) inc = ff_add(u, inc);
  }
  if (lane == 31) sh.red[w] = inc;
  __syncthreads();
  ff base = {0.0f, 0.0f}, tot = {0.0f, 0.0f};
#pragma unroll
  for (int k = 0; k < RD_NT / 32; ++k) {
    if (k < w) base = ff_add(base, sh.red[k]);
    tot = ff_add(tot, sh.red[k]);
  }
  __syncthreads();
  ff ex;
  ex.hi = __shfl_up_sync(RW_FULL, inc.hi, 1);
  ex.lo = __shfl_up_sync(RW_FULL, inc.lo, 1);
  if (lane == 0) ex = {0.0f, 0.0f};
  *total = tot;
  return ff_add(base, ex);
}

// The deferred rows, one CTA each (a grid-stride loop over the list): the
// row's walk from the recorded position in float-float throughout (the
// normalisers, the acceptance ratio, the residual or bonus weights and their
// prefix sums), with the conventions of the warp kernel's exact paths.
template <typename E>
__global__ void __launch_bounds__(RD_NT) row_redo_kernel(const __grid_constant__ KP P, RowDefer D) {
  __shared__ RdShared sh;
  const int tid = threadIdx.x;
  // the programmatic dependent of the first kernel: its deferred rows are
  // complete and visible once it has finished
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint32_t cnt = *reinterpret_cast<volatile const uint32_t *>(D.count);
  RC_PHASE_START;
  for (uint32_t e = blockIdx.x; e < cnt; e += gridDim.x) {
    RC_PHASE(9);  // redo: between rows
    const int4 rec = D.list[e];
    const int b = rec.x, i0 = rec.y;
    int status = rec.z, token = -1, r = i0, tested = i0;
    float resid = 0.0f;
    const int gb = P.gam ? P.gam[b] : P.gm;
    const E *tb = static_cast<const E *>(P.tgt) + static_cast<int64_t>(b) * P.t_row;
    const E *db = static_cast<const E *>(P.drf) + static_cast<int64_t>(b) * P.d_row;
    const float *ub = P.uni + static_cast<int64_t>(b) * P.u_row;
    for (int i = i0; i <= gb; ++i) {
      const bool bonus = i == gb;
      int x = -1;
      if (!bonus) {
        x = P.tok[static_cast<int64_t>(b) * P.gm + i];
        if (x < 0 || x >= P.V) status |= ST_BAD_TOKEN;
      }
      float zt[RD_PT], zd[RD_PT];
      bool bad = false;
      float mx = -INFINITY, mxd = -INFINITY;
#pragma unroll
      for (int k = 0; k < RD_PT; ++k) {
        const int v = tid * RD_PT + k;
        zt[k] = v < P.V ? Elem<E>::get(tb[static_cast<int64_t>(i) * P.t_pos + v]) : -INFINITY;
        zd[k] = (v < P.V && !bonus) ? Elem<E>::get(db[static_cast<int64_t>(i) * P.d_pos + v])
                                    : -INFINITY;
        bad |= zt[k] != zt[k] || zt[k] == INFINITY || zd[k] != zd[k] || zd[k] == INFINITY;
        mx = fmaxf(mx, zt[k]);
        mxd = fmaxf(mxd, zd[k]);
      }
      if (__syncthreads_or(bad ? 1 : 0)) status |= ST_BAD_LOGIT;
      RC_PHASE(10);  // redo: loads + flags
      const float mt = rd_max(mx, sh), md = rd_max(mxd, sh);
      RC_PHASE(11);  // redo: maxima
      if (!(mt > -INFINITY) || (!bonus && !(md > -INFINITY))) status |= ST_NO_FINITE;
      const float *ui = ub + static_cast<int64_t>(i) * P.u_pos;
      float u0 = 0.0f;
      if (!bonus) {
        u0 = ui[P.u_acc];
        if (!(u0 >= 0.0f && u0 < 1.0f)) status |= ST_BAD_UNIFORM;
      }
      if (status & ST_ERROR) {
        r = i;
        break;
      }
      ff et[RD_PT], ed[RD_PT];
      ff st = {0.0f, 0.0f}, sd = {0.0f, 0.0f};
#pragma unroll
      for (int k = 0; k < RD_PT; ++k) {
        et[k] = rw_weight_ff(P, zt[k], mt);
        ed[k] = bonus ? ff{0.0f, 0.0f} : rw_weight_ff(P, zd[k], md);
        st = ff_add(st, et[k]);
        sd = ff_add(sd, ed[k]);
      }
      const ff Zt = rd_sum(st, sh);
      const ff Zd = bonus ? ff{1.0f, 0.0f} : rd_sum(sd, sh);
      const ff rZt = ff_div(ff{1.0f, 0.0f}, Zt);
      const ff rZd = ff_div(ff{1.0f, 0.0f}, Zd);
      RC_PHASE(12);  // redo: float-float weights + normalisers
      if (!bonus) {
        // the token's weights, from the thread holding index x
        if (tid == x / RD_PT) {
          sh.fx[0] = et[x % RD_PT].hi;
          sh.fx[1] = et[x % RD_PT].lo;
          sh.fx[2] = ed[x % RD_PT].hi;
          sh.fx[3] = ed[x % RD_PT].lo;
        }
        __syncthreads();
        const ff px = ff_mul(ff{sh.fx[0], sh.fx[1]}, rZt);
        const ff qx = ff_mul(ff{sh.fx[2], sh.fx[3]}, rZd);
        __syncthreads();
        int v;
        if (!(qx.hi > 0.0f)) {
          v = px.hi > 0.0f ? 1 : 0;  // the limit of min(1, p/q) as q -> 0
          status |= ST_Q_ZERO;
        } else if (!(px.hi > 0.0f)) {
          v = 0;
        } else {
          v = ff_lt(ff_make(u0), ff_div(px, qx)) ? 1 : 0;
        }
        if (tid == 0) {
          if (P.p_dbg) P.p_dbg[static_cast<int64_t>(b) * P.gm + i] = __fadd_rn(px.hi, px.lo);
          if (P.q_dbg) P.q_dbg[static_cast<int64_t>(b) * P.gm + i] = __fadd_rn(qx.hi, qx.lo);
        }
        tested = i + 1;
        RC_PHASE(13);  // redo: acceptance
        if (v) continue;  // accepted
      }
      // the draw at position i: the residual at a rejection, p at the bonus
      r = i;
      const float u1 = ui[P.u_draw];
      if (!(u1 >= 0.0f && u1 < 1.0f)) {
        status |= ST_BAD_UNIFORM;
        break;
      }
      for (int pass = 0; pass < 2; ++pass) {
        const bool residual = !bonus && pass == 0;
        ff wk[RD_PT], s = {0.0f, 0.0f};
        int last = -1;
#pragma unroll
        for (int k = 0; k < RD_PT; ++k) {
          ff p = ff_mul(et[k], rZt);
          if (residual) p = ff_sub(p, ff_mul(ed[k], rZd));
          wk[k] = p.hi > 0.0f ? p : ff{0.0f, 0.0f};
          if (wk[k].hi > 0.0f) last = tid * RD_PT + k;
          s = ff_add(s, wk[k]);
        }
        ff W;
        const ff a0 = rd_scan(s, sh, &W);
        if (residual) resid = __fadd_rn(W.hi, W.lo);
        if (!(W.hi > 0.0f)) continue;  // an empty residual: draw from p
        const ff target = ff_mul_f(W, u1);
        if (tid == 0) {
          sh.ix[0] = -1;
          sh.ix[1] = -1;
        }
        __syncthreads();
        if (!ff_lt(target, a0) && ff_lt(target, ff_add(a0, s))) {
          ff c = a0;
          int tok = -1;
#pragma unroll
          for (int k = 0; k < RD_PT; ++k) {
            if (tok < 0) {
              if (wk[k].hi > 0.0f) c = ff_add(c, wk[k]);
              if (wk[k].hi > 0.0f && ff_lt(target, c)) tok = tid * RD_PT + k;
            }
          }
          if (tok >= 0) sh.ix[0] = tok;
        }
        atomicMax(&sh.ix[1], last);
        __syncthreads();
        token = sh.ix[0] >= 0 ? sh.ix[0] : sh.ix[1];  // rounding past the end: the last weight
        __syncthreads();
        RC_PHASE(14);  // redo: draw
        break;
      }
      break;
    }
    if (tid == 0) {
      const bool err = (status & ST_ERROR) != 0;
      if (P.acc) P.acc[b] = err ? 0 : r;
      P.next[b] = err ? -1 : token;
      if (P.st_dbg) P.st_dbg[b] = status;
      if (P.res_dbg) P.res_dbg[b] = err ? 0.0f : resid;
      const float nan = __int_as_float(0x7fc00000);
      for (int j = tested; j < P.gm; ++j) {
        if (P.p_dbg) P.p_dbg[static_cast<int64_t>(b) * P.gm + j] = nan;
        if (P.q_dbg) P.q_dbg[static_cast<int64_t>(b) * P.gm + j] = nan;
      }
    }
    __syncthreads();
    RC_PHASE(8);  // redo: one deferred row
  }
}

// ------------------------------------------ one CTA of two warps per row
// The same walk and certified single-precision arithmetic as row_kernel,
// with a row spread over 64 threads (16 contiguous logits each, so thread
// order is vocabulary order): four times shorter per-thread chains and
// 24 rows per SM.  Uncertain decisions are deferred to row_redo_kernel
// (the kernel runs only when the call provides the deferred-row list).
constexpr int RC_NT = 64;
constexpr int RC_PT = kRowMaxV / RC_NT;  // logits per thread
static_assert(RC_PT == 16, "16 logits per thread");

struct RcShared {
  float mx[2][2];  // per warp: target and draft maxima
  float zx[2];     // the token's target and draft logits (from the slice's owner)
  ff zs[2][2];     // per warp: the normalisers' partial sums
  float ys[2][2];  // per warp: sum e y (y <= 0) of each tensor, for the error bounds
  ff ds[2];        // per warp: the draw weights' sums
  float de[2][3];  // per warp: sum p y, sum q y (y <= 0), sum p + q
  int tok[2];      // the drawn token and whether it is certified
};

// The row kernel keeps each position's logits in shared memory, not in
// registers: a thread's slice of both rows, [RC_PT t, RC_PT t + RC_PT), is
// copied there with 16-byte asynchronous copies (element loads for a ragged
// or unaligned slice, -inf past the vocabulary), and read back in chunks of
// four by each pass.  The 16-byte chunks are interleaved over the threads
// (chunk c of thread t at chunk c * RC_NT + t), so that a warp's loads of
// its threads' chunk c fall in distinct banks.  A thread reads only its own
// slice, except the token's logits after a CTA barrier; with 40 registers a
// thread, 24 rows fit an SM.
template <typename E>
__device__ __forceinline__ int rc_index(int t, int k) {  // element k of thread t's slice
  constexpr int PER = 16 / static_cast<int>(sizeof(E));
  return ((k / PER) * RC_NT + t) * PER + (k % PER);
}
template <typename E, bool VEC>
__device__ __forceinline__ void rc_stage(const E *g, int V, int t, E *s) {
  const int v0 = t * RC_PT;
  if (VEC && v0 + RC_PT <= V) {
    constexpr int PER = 16 / static_cast<int>(sizeof(E));
#pragma unroll
    for (int j = 0; j < RC_PT / PER; ++j) {
      const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(s + rc_index<E>(t, j * PER)));
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(g + v0 + j * PER)
                   : "memory");
    }
  } else {
    for (int k = 0; k < RC_PT; ++k) {
      const int j = rc_index<E>(t, k);
      if (v0 + k < V) {
        s[j] = g[v0 + k];
      } else if (sizeof(E) == 4) {
        reinterpret_cast<float *>(s)[j] = -INFINITY;
      } else {
        reinterpret_cast<uint16_t *>(s)[j] = 0xff80u;  // bfloat16 -inf
      }
    }
  }
}
__device__ __forceinline__ void rc_stage_wait() {
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}
// Elements [4 c, 4 c + 4) of thread t's staged slice.
template <typename E>
__device__ __forceinline__ void rc_chunk(const E *s, int t, int c, float (&f)[4]);
template <>
__device__ __forceinline__ void rc_chunk<float>(const float *s, int t, int c, float (&f)[4]) {
  const float4 v = *reinterpret_cast<const float4 *>(s + rc_index<float>(t, 4 * c));
  f[0] = v.x;
  f[1] = v.y;
  f[2] = v.z;
  f[3] = v.w;
}
template <>
__device__ __forceinline__ void rc_chunk<uint16_t>(const uint16_t *s, int t, int c,
                                                   float (&f)[4]) {
  const uint2 v = *reinterpret_cast<const uint2 *>(s + rc_index<uint16_t>(t, 4 * c));
  f[0] = __uint_as_float(v.x << 16);
  f[1] = __uint_as_float(v.x & 0xffff0000u);
  f[2] = __uint_as_float(v.y << 16);
  f[3] = __uint_as_float(v.y & 0xffff0000u);
}
// The staged logit of vocabulary index j.
template <typename E>
__device__ __forceinline__ float rc_elem(const E *s, int j) {
  const int k = rc_index<E>(j / RC_PT, j % RC_PT);
  return sizeof(E) == 4 ? reinterpret_cast<const float *>(s)[k]
                        : __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t *>(s)[k]) << 16);
}

// Sum of a thread's weights e = 2^y, y = max(((z - m) c2), -256) (NaN kept)
// of one staged slice in four interleaved sums (k mod 4; two lanes per
// packed operation), and sum e y for the error bound.  An fp32 slice is
// overwritten with its weights (the draw reads them instead of recomputing
// 2^y; nothing reads the logits afterwards).
template <typename E>
__device__ __forceinline__ void rc_wsum(E *s, int t, float m, float c2, float &S, float &Y) {
  const f2 M2 = f2_pack(m, m), C2 = f2_pack(c2, c2);
  f2 a01 = f2_pack(0.0f, 0.0f), a23 = a01, yy = a01;
#pragma unroll
  for (int c = 0; c < RC_PT / 4; ++c) {
    float f[4];
    rc_chunk<E>(s, t, c, f);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float ya, yb;
      f2_unpack(f2_mul(f2_sub(f2_pack(f[2 * h], f[2 * h + 1]), M2), C2), ya, yb);
      ya = max_nan(ya, -256.0f);
      yb = max_nan(yb, -256.0f);
      const f2 e2 = f2_pack(ex2_approx(ya), ex2_approx(yb));
      if (h) a23 = f2_add(a23, e2); else a01 = f2_add(a01, e2);
      yy = f2_fma(e2, f2_pack(ya, yb), yy);
      if constexpr (sizeof(E) == 4) f2_unpack(e2, f[2 * h], f[2 * h + 1]);
    }
    if constexpr (sizeof(E) == 4)
      *reinterpret_cast<float4 *>(s + rc_index<E>(t, 4 * c)) = make_float4(f[0], f[1], f[2], f[3]);
  }
  float a, b, c, d;
  f2_unpack(a01, a, b);
  f2_unpack(a23, c, d);
  S = __fadd_rn(__fadd_rn(a, b), __fadd_rn(c, d));
  f2_unpack(yy, a, b);
  Y = __fadd_rn(a, b);
}

// The draw weight of one element from its stored weights e_t, e_d (fp32
// rows): p = e_t / Z_t, and max(0, p - q) with q = e_d / Z_d (residual).
// The same roundings as rc_draw_w.
__device__ __forceinline__ float rc_cached_w(float et, float ed, float rzt, float rzd,
                                             bool residual) {
  const float p = __fmul_rn(et, rzt);
  if (!residual) return p;
  return fmaxf(__fsub_rn(p, __fmul_rn(ed, rzd)), 0.0f);
}

// The draw weight of one element: max(0, p - q) (residual) or p, with the
// bound terms p, p y_p, q, q y_q (y clamped at -256: the weight is 0 there).
__device__ __forceinline__ float rc_draw_w(float z, float w, const Dist &dt, const Dist &dd,
                                           float c2, bool residual, float &sp, float &sq,
                                           float &py, float &qy) {
  const float yt = fmaxf(__fmul_rn(__fsub_rn(z, dt.m), c2), -256.0f);
  const float p = __fmul_rn(ex2_approx(yt), dt.rzf);
  sp = __fadd_rn(sp, p);
  py = __fmaf_rn(p, yt, py);
  if (!residual) return p;
  const float yd = fmaxf(__fmul_rn(__fsub_rn(w, dd.m), c2), -256.0f);
  const float q = __fmul_rn(ex2_approx(yd), dd.rzf);
  sq = __fadd_rn(sq, q);
  qy = __fmaf_rn(q, yd, qy);
  return fmaxf(__fsub_rn(p, q), 0.0f);
}

template <typename E, bool VEC>
__global__ void __launch_bounds__(RC_NT, 24) row_cta_kernel(const __grid_constant__ KP P, RowDefer D) {
  __shared__ RcShared sh;
  extern __shared__ __align__(16) unsigned char rc_dyn[];
  E *zs = reinterpret_cast<E *>(rc_dyn);  // [kRowMaxV] target, then [kRowMaxV] draft
  E *wsd = zs + kRowMaxV;
  const int t = threadIdx.x, lane = t & 31, wp = t >> 5;
  const int v0 = t * RC_PT;
  const int b = static_cast<int>(blockIdx.x);
  // launched as the programmatic dependent of the counter clear: the second
  // kernel may launch once every CTA has started; CTA 0 waits for the clear
  // so that this grid cannot complete before it (the second kernel waits
  // for this grid only)
  asm volatile("griddepcontrol.launch_dependents;");
  if (b == 0 && t == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
  const int gb = P.gam ? P.gam[b] : P.gm;
  if (gb < 0 || gb > P.gm) {
    if (t == 0) rw_bad_row(P, b);
    return;
  }
  const E *tb = static_cast<const E *>(P.tgt) + static_cast<int64_t>(b) * P.t_row;
  const E *db = static_cast<const E *>(P.drf) + static_cast<int64_t>(b) * P.d_row;
  const float *ub = P.uni + static_cast<int64_t>(b) * P.u_row;
  const float c2 = P.c2;
  int status = 0, token = -1, r = gb, tested = 0;
  float resid = 0.0f;
  RC_PHASE_START;
  for (int i = 0; i <= gb; ++i) {
    const bool bonus = i == gb;
    int x = -1;
    if (!bonus) {
      x = P.tok[static_cast<int64_t>(b) * P.gm + i];
      if (x < 0 || x >= P.V) status |= ST_BAD_TOKEN;
    }
    // the thread's slices of both rows (the previous position's are no longer
    // read by any thread: the last barrier of that position is behind us)
    rc_stage<E, VEC>(tb + static_cast<int64_t>(i) * P.t_pos, P.V, t, zs);
    if (!bonus) rc_stage<E, VEC>(db + static_cast<int64_t>(i) * P.d_pos, P.V, t, wsd);
    rc_stage_wait();
    // the token's logits, published by the thread whose slice holds them (its
    // own copies are complete; the others read them after the barrier below)
    const bool xin = x >= 0 && x < P.V;
    if (xin && t == x / RC_PT) {
      sh.zx[0] = rc_elem<E>(zs, x);
      sh.zx[1] = rc_elem<E>(wsd, x);
    }
    // maxima (NaN ignored here; a NaN shows in the normaliser)
    float mt = -INFINITY, md = -INFINITY;
#pragma unroll
    for (int c = 0; c < RC_PT / 4; ++c) {
      float f[4];
      rc_chunk<E>(zs, t, c, f);
      mt = fmaxf(fmaxf(mt, fmaxf(f[0], f[1])), fmaxf(f[2], f[3]));
      if (!bonus) {
        rc_chunk<E>(wsd, t, c, f);
        md = fmaxf(fmaxf(md, fmaxf(f[0], f[1])), fmaxf(f[2], f[3]));
      }
    }
    RC_PHASE(0);  // loads + per-thread maxima
    mt = warp_max(mt);
    if (!bonus) md = warp_max(md);
    if (lane == 0) {
      sh.mx[wp][0] = mt;
      sh.mx[wp][1] = md;
    }
    __syncthreads();
    const float zx = xin ? sh.zx[0] : 0.0f;
    const float wx = xin ? sh.zx[1] : 0.0f;
    mt = fmaxf(sh.mx[0][0], sh.mx[1][0]);
    md = fmaxf(sh.mx[0][1], sh.mx[1][1]);
    RC_PHASE(1);  // maxima: warp reductions + barrier
    // no finite logit (the other kernels' rule; a NaN among them is bad),
    // from the logits before the normalisers overwrite fp32 slices
    if (!(mt > -INFINITY) || (!bonus && !(md > -INFINITY))) {  // uniform
      status |= ST_NO_FINITE;
      bool nan = false;
      for (int k = 0; k < RC_PT; ++k) {
        const float a = rc_elem<E>(zs, v0 + k);
        nan |= a != a;
        if (!bonus) {
          const float c = rc_elem<E>(wsd, v0 + k);
          nan |= c != c;
        }
      }
      if (__syncthreads_or(nan)) status |= ST_BAD_LOGIT;
    }
    // normalisers: each thread sums its weights in four interleaved
    // single-precision sums (depth 5: relative error <= 5 2^-24), the
    // threads' sums in float-float; the weights' error bound e (k0 + k1 |y|)
    // summed as k0 sum e - k1 sum e y.  A NaN logit makes its weight, and so
    // Z, NaN.
    ff Zt, Zd = {1.0f, 0.0f};
    float yst, ysd = 0.0f;
    {
      float S0, y0, S1 = 0.0f, y1 = 0.0f;
      rc_wsum<E>(zs, t, mt, c2, S0, y0);
      if (!bonus) rc_wsum<E>(wsd, t, md, c2, S1, y1);
      const ff Z0 = warp_sum_ff(ff{S0, 0.0f});
      y0 = rw_sum(y0);
      ff Z1 = {0.0f, 0.0f};
      if (!bonus) {
        Z1 = warp_sum_ff(ff{S1, 0.0f});
        y1 = rw_sum(y1);
      }
      if (lane == 0) {
        sh.zs[wp][0] = Z0;
        sh.zs[wp][1] = Z1;
        sh.ys[wp][0] = y0;
        sh.ys[wp][1] = y1;
      }
      __syncthreads();
      Zt = ff_add(sh.zs[0][0], sh.zs[1][0]);
      yst = __fadd_rn(sh.ys[0][0], sh.ys[1][0]);
      if (!bonus) {
        Zd = ff_add(sh.zs[0][1], sh.zs[1][1]);
        ysd = __fadd_rn(sh.ys[0][1], sh.ys[1][1]);
      }
    }
    // row flags: NaN or +inf is bad (the other kernels' rule)
    const bool tfin = mt > -INFINITY && mt < INFINITY;
    const bool dfin = md > -INFINITY && md < INFINITY;
    if (mt == INFINITY || (!bonus && md == INFINITY)) status |= ST_BAD_LOGIT;
    if ((tfin && Zt.hi != Zt.hi) || (!bonus && dfin && Zd.hi != Zd.hi)) status |= ST_BAD_LOGIT;
    const float *ui = ub + static_cast<int64_t>(i) * P.u_pos;
    float u0 = 0.0f;
    if (!bonus) {
      u0 = ui[P.u_acc];
      if (!(u0 >= 0.0f && u0 < 1.0f)) status |= ST_BAD_UNIFORM;
    }
    if (status & ST_ERROR) {
      r = i;
      break;
    }
    Dist dt, dd;
    dist_init(dt, mt);
    dist_init(dd, md);
    {
      const float Et = __fmaf_rn(__fmul_rn(Zt.hi, 1.001f), kExpErr0, -__fmul_rn(yst, kExpErr1));
      set_Zf(dt, Zt, __fadd_rn(__fdiv_rn(Et, Zt.hi), 3.6e-7f));
      if (!bonus) {
        const float Ed = __fmaf_rn(__fmul_rn(Zd.hi, 1.001f), kExpErr0, -__fmul_rn(ysd, kExpErr1));
        set_Zf(dd, Zd, __fadd_rn(__fdiv_rn(Ed, Zd.hi), 3.6e-7f));
      }
    }
    RC_PHASE(2);  // normalisers: weights, sums, barrier
    if (!bonus) {
      // acceptance u < p(x)/q(x), certified; uncertain: deferred
      const bool kp = zx != -INFINITY, kq = wx != -INFINITY;
      const float yp = __fmul_rn(__fsub_rn(zx, dt.m), c2);
      const float yq = __fmul_rn(__fsub_rn(wx, dd.m), c2);
      const float pf = kp ? __fmul_rn(ex2_approx(yp), dt.rzf) : 0.0f;
      const float qf = kq ? __fmul_rn(ex2_approx(yq), dd.rzf) : 0.0f;
      int v;
      if (!kq) {
        v = kp ? 1 : 0;
      } else if (!kp) {
        v = 0;
      } else if (u0 == 0.0f) {
        v = 1;
      } else {
        const float d = __fsub_rn(yp, yq);
        const float rr = __fmul_rn(ex2_approx(d), __fmul_rn(dd.Z.hi, dt.rzf));
        const float eps = __fadd_rn(
            __fmaf_rn(__fadd_rn(__fadd_rn(fabsf(yp), fabsf(yq)), fabsf(d)), kExpErr1, kExpErr0),
            __fadd_rn(__fadd_rn(dt.zerr, dd.zerr), 1.2e-6f));
        if (rr == INFINITY || u0 < __fmul_rn(rr, 1.0f - eps))
          v = 1;
        else if (u0 >= __fmul_rn(rr, 1.0f + eps) && rr > 0.0f)
          v = 0;
        else
          v = 2;
      }
      if (v == 2) {
        if (t == 0) {
          asm volatile("griddepcontrol.wait;" ::: "memory");  // the count is clear
          const uint32_t k = atomicAdd(D.count, 1u);
          D.list[k] = make_int4(b, i, status, 0);
        }
        return;
      }
      if (!kq) status |= ST_Q_ZERO;
      tested = i + 1;
      if (t == 0) {
        if (P.p_dbg) P.p_dbg[static_cast<int64_t>(b) * P.gm + i] = pf;
        if (P.q_dbg) P.q_dbg[static_cast<int64_t>(b) * P.gm + i] = qf;
      }
      RC_PHASE(3);  // acceptance
      // accepted: the next position restages the slices (every thread read
      // the token's logits before the normalisers' barrier)
      if (v) continue;
    }
    // the draw at position i, certified; uncertain or empty: deferred.  The
    // weights (the residual max(0, p - q) at a rejection, p at the bonus
    // position) are summed per thread in four interleaved single-precision
    // sums, the threads' sums scanned in float-float; the owner of the
    // target walks its weights in float-float.  Bound of the weights' errors:
    // p (k0 + k1 |y_p| + zerr_p + 2.4e-7) + q (likewise) + 6e-8 (p + q), from
    // the sums of p, q, p y_p and q y_q; the per-thread sums' rounding
    // (depth 5) is covered by 3.6e-7 W.  fp32 rows read the weights 2^y the
    // normalisers stored, and take those sums from the normalisers' (sum p =
    // Z_t / Z_t, sum p y_p = (sum e y) / Z_t); bf16 rows recompute 2^y and
    // sum them here.
    r = i;
    const float u1 = ui[P.u_draw];
    if (!(u1 >= 0.0f && u1 < 1.0f)) {
      status |= ST_BAD_UNIFORM;
      break;
    }
    const bool residual = !bonus;
    constexpr bool kCached = sizeof(E) == 4;  // the slices hold the weights 2^y
    float sp = 0.0f, sq = 0.0f, py = 0.0f, qy = 0.0f;
    float a4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int c = 0; c < RC_PT / 4; ++c) {
      float fz[4], fw[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      rc_chunk<E>(zs, t, c, fz);
      if (residual) rc_chunk<E>(wsd, t, c, fw);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float w;
        if constexpr (kCached)
          w = rc_cached_w(fz[e], fw[e], dt.rzf, dd.rzf, residual);
        else
          w = rc_draw_w(fz[e], fw[e], dt, dd, c2, residual, sp, sq, py, qy);
        a4[e] = __fadd_rn(a4[e], w);
      }
    }
    const float sm = __fadd_rn(__fadd_rn(a4[0], a4[1]), __fadd_rn(a4[2], a4[3]));
    // exclusive scan over the 64 threads in thread (= vocabulary) order
    ff inc = {sm, 0.0f};
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      ff u;
      u.hi = __shfl_up_sync(RW_FULL, inc.hi, o);
      u.lo = __shfl_up_sync(RW_FULL, inc.lo, o);
      if (lane >= o) inc = ff_add(u, inc);
    }
    if constexpr (!kCached) {
      sp = rw_sum(sp);
      sq = residual ? rw_sum(sq) : 0.0f;
      py = rw_sum(py);
      qy = residual ? rw_sum(qy) : 0.0f;
      if (lane == 0) {
        sh.de[wp][0] = py;
        sh.de[wp][1] = qy;
        sh.de[wp][2] = __fadd_rn(sp, sq);
      }
    }
    if (lane == 31) sh.ds[wp] = inc;
    if (t == 0) {
      sh.tok[0] = -1;
      sh.tok[1] = 0;
    }
    __syncthreads();
    ff a;
    a.hi = __shfl_up_sync(RW_FULL, inc.hi, 1);
    a.lo = __shfl_up_sync(RW_FULL, inc.lo, 1);
    if (lane == 0) a = {0.0f, 0.0f};
    if (wp == 1) a = ff_add(sh.ds[0], a);
    const ff W = ff_add(sh.ds[0], sh.ds[1]);
    // Dw: the weights' error bound, with the larger of the two tensors'
    // relative constants on sum (p + q), plus the per-thread sums' rounding
    float Dw;
    {
      float PY, QY, PQ;
      if constexpr (kCached) {
        // sum p = Z_t / Z_t and sum q are one up to 2^-23 and the relative
        // error of Z (1.2e-6 together, within the factor 1.001 below); the
        // sums of e y are still in shared memory
        PY = __fmul_rn(__fadd_rn(sh.ys[0][0], sh.ys[1][0]), dt.rzf);
        QY = residual ? __fmul_rn(__fadd_rn(sh.ys[0][1], sh.ys[1][1]), dd.rzf) : 0.0f;
        PQ = residual ? 2.0f : 1.0f;
      } else {
        PY = __fadd_rn(sh.de[0][0], sh.de[1][0]);
        QY = __fadd_rn(sh.de[0][1], sh.de[1][1]);
        PQ = __fadd_rn(sh.de[0][2], sh.de[1][2]);
      }
      const float kp = __fadd_rn(kExpErr0, __fadd_rn(dt.zerr, 2.4e-7f));
      const float kq = residual ? __fadd_rn(kExpErr0, __fadd_rn(dd.zerr, 2.4e-7f)) : 0.0f;
      const float wsum = __fmaf_rn(fmaxf(kp, kq), PQ, -__fmul_rn(kExpErr1, __fadd_rn(PY, QY)));
      Dw = __fmul_rn(__fadd_rn(__fmaf_rn(PQ, 6.0e-8f, wsum), __fmul_rn(W.hi, 3.6e-7f)), 1.001f);
    }
    if (residual) resid = __fadd_rn(W.hi, W.lo);
    if (!(W.hi > 0.0f)) {  // an (almost) empty residual: to the second kernel
      if (t == 0) {
        asm volatile("griddepcontrol.wait;" ::: "memory");  // the count is clear
        const uint32_t k = atomicAdd(D.count, 1u);
        D.list[k] = make_int4(b, i, status, 0);
      }
      return;
    }
    const float slack = __fmaf_rn(W.hi, 1e-12f, static_cast<float>(P.V) * 4e-38f *
                                                    (dt.rzf + (residual ? dd.rzf : 0.0f)));
    const ff target = ff_mul_f(W, u1);
    if (!ff_lt(target, a) && ff_lt(target, ff_add_f(a, sm))) {
      ff cc = a;
      int tk = -1, cert = 0;
      float d0 = 0.0f, d1 = 0.0f, d2 = 0.0f, d3 = 0.0f;  // (the bound terms: unused here)
      for (int k = 0; k < RC_PT; ++k) {
        if (tk < 0) {
          const float zk = rc_elem<E>(zs, v0 + k), wk0 = residual ? rc_elem<E>(wsd, v0 + k) : 0.0f;
          float wk;
          if constexpr (kCached)
            wk = rc_cached_w(zk, wk0, dt.rzf, dd.rzf, residual);
          else
            wk = rc_draw_w(zk, wk0, dt, dd, c2, residual, d0, d1, d2, d3);
          const ff cp = cc;
          cc = ff_add_f(cc, wk);
          if (wk > 0.0f && ff_lt(target, cc)) {
            tk = v0 + k;
            const ff l = ff_sub(target, cp), h = ff_sub(cc, target);
            // the error of t - C (t = u W, C a boundary) is u dR - (1 - u) dC,
            // dC and dR the errors of the sums before and after the boundary:
            // at most Dw in size
            cert = fminf(__fadd_rn(l.hi, l.lo), __fadd_rn(h.hi, h.lo)) > __fadd_rn(Dw, slack);
          }
        }
      }
      if (tk >= 0) {
        sh.tok[0] = tk;
        sh.tok[1] = cert;
      }
    }
    __syncthreads();
    token = sh.tok[0];
    RC_PHASE(4);  // draw
    if (token < 0 || !sh.tok[1]) {
      if (t == 0) {
        asm volatile("griddepcontrol.wait;" ::: "memory");  // the count is clear
        const uint32_t k = atomicAdd(D.count, 1u);
        D.list[k] = make_int4(b, i, status, 0);
      }
      return;
    }
    break;
  }
  if (t == 0) {
    const bool err = (status & ST_ERROR) != 0;
    if (P.acc) P.acc[b] = err ? 0 : r;
    P.next[b] = err ? -1 : token;
    if (P.st_dbg) P.st_dbg[b] = status;
    if (P.res_dbg) P.res_dbg[b] = err ? 0.0f : resid;
    const float nan = __int_as_float(0x7fc00000);
    for (int j = tested; j < P.gm; ++j) {
      if (P.p_dbg) P.p_dbg[static_cast<int64_t>(b) * P.gm + j] = nan;
      if (P.q_dbg) P.q_dbg[static_cast<int64_t>(b) * P.gm + j] = nan;
    }
  }
}

// Clears the deferred-row count; lets the row kernel launch at once (it
// waits for this grid before its first use of the count).
__global__ void row_clear(uint32_t *count) {
  asm volatile("griddepcontrol.launch_dependents;");
  if (threadIdx.x == 0) *count = 0u;
}

using RowFn = void (*)(KP, RowDefer);

RowFn row_fn(int dtype, bool vec) {
  if (dtype == SPEC_F32) return vec ? row_kernel<float, true> : row_kernel<float, false>;
  return vec ? row_kernel<uint16_t, true> : row_kernel<uint16_t, false>;
}
RowFn cta_fn(int dtype, bool vec) {
  if (dtype == SPEC_F32) return vec ? row_cta_kernel<float, true> : row_cta_kernel<float, false>;
  return vec ? row_cta_kernel<uint16_t, true> : row_cta_kernel<uint16_t, false>;
}
RowFn redo_fn(int dtype) {
  return dtype == SPEC_F32 ? row_redo_kernel<float> : row_redo_kernel<uint16_t>;
}

// The row kernel keeps 8 KB of rows per CTA in shared memory: ask for the
// largest shared-memory carveout, so that 24 CTAs fit an SM (once per kernel).
cudaError_t cta_prepare(RowFn f) {
  static std::mutex mu;
  static std::map<RowFn, cudaError_t> done;
  std::lock_guard<std::mutex> lk(mu);
  auto it = done.find(f);
  if (it != done.end()) return it->second;
  const cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void *>(f),
                                             cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  done[f] = e;
  return e;
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
      n = v;
    else
      n = 132;
  }
  return n;
}

}  // namespace

bool row_eligible(const spec_params &p) {
  if (p.V < 1 || p.V > kRowMaxV || p.cluster_size != 0) return false;
  if (p.dtype != SPEC_F32 && p.dtype != SPEC_BF16) return false;
  if (p.temperature == 0.0f) return true;  // greedy: the filters cannot change the argmax
  const bool k_on = p.top_k > 0 && p.top_k < p.V;
  const bool p_on = p.top_p < 1.0f;
  return !k_on && !p_on;
}

size_t row_defer_bytes(const spec_params &p) {
  if (p.temperature == 0.0f || p.B < 1) return 0;  // greedy decisions are never uncertain
  return kRowDeferOffset + static_cast<size_t>(p.B) * sizeof(int4);
}

spec_status row_launch(const KP &kp, int dtype, bool vec, void *ws, size_t ws_bytes,
                       const spec_params &p, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>((static_cast<int64_t>(kp.B) + RW_ROWS - 1) / RW_ROWS);
  RowDefer D = {nullptr, nullptr};
  const size_t need = row_defer_bytes(p);
  if (ws && need && ws_bytes >= need) {
    char *w = static_cast<char *>(ws);
    D.count = reinterpret_cast<uint32_t *>(w + kRowDeferOffset - 16);
    D.list = reinterpret_cast<int4 *>(w + kRowDeferOffset);
  }
  if (!D.count) {  // a warp per row, uncertain decisions redone in the warp
    row_fn(dtype, vec)<<<grid, RW_NT, 0, stream>>>(kp, D);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
  }
  // a CTA of two warps per row, uncertain rows to the second kernel: the
  // counter clear, then both kernels as programmatic dependents (each waits
  // for its predecessor where it needs its results)
  row_clear<<<1, 32, 0, stream>>>(D.count);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  const RowFn cf = cta_fn(dtype, vec);
  if (cta_prepare(cf) != cudaSuccess) return SPEC_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(kp.B));
  cfg.blockDim = dim3(RC_NT);
  cfg.dynamicSmemBytes = 2 * kRowMaxV * (dtype == SPEC_F32 ? 4 : 2);
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, cf, kp, D) != cudaSuccess) return SPEC_ERR_CUDA;
  cfg.dynamicSmemBytes = 0;
  cfg.gridDim = dim3(static_cast<unsigned>(std::min<int64_t>(kp.B, sm_count())));
  cfg.blockDim = dim3(RD_NT);
  if (cudaLaunchKernelEx(&cfg, redo_fn(dtype), kp, D) != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}

}  // namespace sv

#ifdef SV_PHASE_PROFILE
extern "C" int sv_row_phase_read(unsigned long long *host, int reset) {
  if (cudaMemcpyFromSymbol(host, sv_row_cycles, 64 * sizeof(unsigned long long)) != cudaSuccess)
    return 1;
  if (reset) {
    unsigned long long z[64] = {0};
    if (cudaMemcpyToSymbol(sv_row_cycles, z, sizeof z) != cudaSuccess) return 1;
  }
  return 0;
}
#endif
