// sv_common.cuh -- device helpers for the verify kernels (sm_103a):
// cluster / distributed-shared-memory primitives in inline PTX, warp
// reductions, order-preserving keys and float-float ("double-float")
// arithmetic with an accurate exponential.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

constexpr int kWarp = 32;

// ---------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// All threads of all CTAs of the cluster arrive, then wait.  Release /
// acquire order shared-memory writes across the cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ uint32_t dsmem_ld_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void dsmem_st_u32(uint32_t a, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// Named barrier over `n` threads (a multiple of 32) of the CTA.
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// ------------------------------------------------- mbarriers and bulk copies
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
// Arrive (count 1) and add `bytes` to the transaction count of this phase.
__device__ __forceinline__ void mbar_arrive_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// One-dimensional bulk copy global -> this CTA's shared memory (TMA); its
// completion is signalled on `bar`.  Addresses and size: multiples of 16 B.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// Wait until the phase with the given parity has completed; gives up after
// `limit` polls and returns false (the caller records the timeout).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t limit) {
  const uint32_t a = smem_u32(bar);
  for (uint32_t it = 0; it < limit; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}
// The same wait for one thread of a CTA (the rest of the block waits on a
// CTA barrier and issues nothing): between polls the thread sleeps, 32 ns at
// first, doubling up to 256 ns, so that a wait of a few microseconds costs
// a few dozen instructions instead of thousands.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t limit) {
  const uint32_t a = smem_u32(bar);
  uint32_t ns = 32;
  for (uint32_t it = 0; it < limit; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    if (ok) return true;
    __nanosleep(ns);
    ns = ns < 256 ? 2 * ns : 256;
  }
  return false;
}
// Maximum that propagates NaN.
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
// Order this thread's earlier generic shared-memory accesses before later
// asynchronous-proxy (bulk copy) writes to shared memory.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------- warps
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ uint32_t warp_or(uint32_t v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v |= __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ int warp_max_i32(int v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
// Sort one value per lane in descending order across the warp (bitonic).
__device__ __forceinline__ float warp_sort_desc(float v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const float o = __shfl_xor_sync(0xffffffffu, v, j);
      const bool desc = (lane & k) == 0 || k == 32;
      const bool lower = (lane & j) == 0;
      v = (lower == desc) ? fmaxf(v, o) : fminf(v, o);
    }
  }
  return v;
}
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// (value, index) maximum with the lowest index winning ties.
__device__ __forceinline__ void warp_argmax(float &v, int &i) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, v, o);
    int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (ov > v || (ov == v && oi < i)) {
      v = ov;
      i = oi;
    }
  }
}

// ------------------------------------------------------------------ values
// Logits are read as float with -0 folded into +0, so that equal values
// have equal bit patterns and keys.
__device__ __forceinline__ float canon(float x) { return __fadd_rn(x, 0.0f); }
__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
// Monotone map float -> uint32 (NaN excluded): a < b  <=>  key(a) < key(b).
__device__ __forceinline__ uint32_t fkey(float x) {
  uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_to_f(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}

// 2^x with the MUFU approximation (flushes results below 2^-126 to 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------ packed single precision
// Two single-precision values in one 64-bit register pair, for the packed
// (two-lane) add / subtract / multiply / fused multiply-add of sm_100 and
// later: each lane is rounded exactly as the scalar operation.
using f2 = unsigned long long;
__device__ __forceinline__ f2 f2_pack(float a, float b) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(f2 v, float &a, float &b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ f2 f2_add(f2 a, f2 b) {
  f2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2 f2_sub(f2 a, f2 b) {
  f2 r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2 f2_mul(f2 a, f2 b) {
  f2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c) {
  f2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// -------------------------------------------------------- float-float math
// A value hi + lo with |lo| <= ulp(hi)/2 (Dekker 1971; Knuth's TwoSum).
// Every operation uses explicitly rounded intrinsics so that the compiler
// cannot contract or reassociate the error terms.
struct ff {
  float hi, lo;
};

__device__ __forceinline__ ff ff_make(float a) { return {a, 0.0f}; }
__device__ __forceinline__ ff ff_neg(ff a) { return {-a.hi, -a.lo}; }
__device__ __forceinline__ ff two_sum(float a, float b) {
  float s = __fadd_rn(a, b);
  float bb = __fsub_rn(s, a);
  float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}
__device__ __forceinline__ ff quick_two_sum(float a, float b) {  // |a| >= |b|
  float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ ff ff_add(ff a, ff b) {
  ff s = two_sum(a.hi, b.hi);
  ff t = two_sum(a.lo, b.lo);
  s.lo = __fadd_rn(s.lo, t.hi);
  s = quick_two_sum(s.hi, s.lo);
  s.lo = __fadd_rn(s.lo, t.lo);
  return quick_two_sum(s.hi, s.lo);
}
__device__ __forceinline__ ff ff_sub(ff a, ff b) { return ff_add(a, ff_neg(b)); }
__device__ __forceinline__ ff ff_add_f(ff a, float b) {
  ff s = two_sum(a.hi, b);
  s.lo = __fadd_rn(s.lo, a.lo);
  return quick_two_sum(s.hi, s.lo);
}
__device__ __forceinline__ ff ff_mul(ff a, ff b) {
  float p = __fmul_rn(a.hi, b.hi);
  float e = __fmaf_rn(a.hi, b.hi, -p);
  e = __fmaf_rn(a.hi, b.lo, e);
  e = __fmaf_rn(a.lo, b.hi, e);
  return quick_two_sum(p, e);
}
__device__ __forceinline__ ff ff_mul_f(ff a, float b) {
  float p = __fmul_rn(a.hi, b);
  float e = __fmaf_rn(a.hi, b, -p);
  e = __fmaf_rn(a.lo, b, e);
  return quick_two_sum(p, e);
}
// a / b by two Newton-style correction steps on the quotient.
__device__ __forceinline__ ff ff_div(ff a, ff b) {
  float q1 = __fdiv_rn(a.hi, b.hi);
  ff r = ff_sub(a, ff_mul_f(b, q1));
  float q2 = __fdiv_rn(r.hi, b.hi);
  r = ff_sub(r, ff_mul_f(b, q2));
  float q3 = __fdiv_rn(r.hi, b.hi);
  return ff_add_f(quick_two_sum(q1, q2), q3);
}
// a < b (both normalised).
__device__ __forceinline__ bool ff_lt(ff a, ff b) {
  return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo);
}
__device__ __forceinline__ ff ff_from_double(double d) {
  float hi = __double2float_rn(d);
  return {hi, __double2float_rn(d - static_cast<double>(hi))};
}
__device__ __forceinline__ double ff_to_double(ff a) {
  return static_cast<double>(a.hi) + static_cast<double>(a.lo);
}

// e^x in float-float (relative error ~1e-14 for x in [-87, 88]).
// Method: Cody-Waite reduction x = k ln2 + r with ln2 split into three
// floats (the first with 16 significant bits so k*LN2_A is exact for
// |k| < 256), then the Taylor series of e^r (|r| <= 0.347) to degree 11
// (truncation < 1e-14), terms of degree >= 7 in single precision, the rest
// in float-float, and a final scaling by 2^k.  The constants are ln 2 and
// 1/n!, split into floats from their exact values.
// ff_exp_core takes x.hi in [-104, 88] (branch-free, for callers that
// interleave several); ff_exp handles every input.
__device__ __forceinline__ ff ff_exp_core(ff x) {
  constexpr float LN2_A = 0x1.62e4p-1f;
  constexpr float LN2_B = 0x1.7f7d1cp-20f;
  constexpr float LN2_C = 0x1.ef357ap-45f;
  const float k = rintf(__fmul_rn(x.hi, 1.44269504f));
  ff r = ff_add_f(x, -__fmul_rn(k, LN2_A));
  {
    float p = __fmul_rn(k, LN2_B);
    ff kb = {p, __fmaf_rn(k, LN2_B, -p)};
    r = ff_sub(r, kb);
  }
  r = ff_add_f(r, -__fmul_rn(k, LN2_C));
  const float rh = r.hi;
  float t = 0x1.ae6456p-26f;                 // 1/11!
  t = __fmaf_rn(t, rh, 0x1.27e4fcp-22f);     // 1/10!
  t = __fmaf_rn(t, rh, 0x1.71de3ap-19f);     // 1/9!
  t = __fmaf_rn(t, rh, 0x1.a01a02p-16f);     // 1/8!
  t = __fmaf_rn(t, rh, 0x1.a01a02p-13f);     // 1/7!
  ff s = {t, 0.0f};
  s = ff_add(ff_mul(s, r), ff{0x1.6c16c2p-10f, -0x1.27d27ep-35f});  // 1/6!
  s = ff_add(ff_mul(s, r), ff{0x1.111112p-7f, -0x1.dddddep-32f});   // 1/5!
  s = ff_add(ff_mul(s, r), ff{0x1.555556p-5f, -0x1.555556p-30f});   // 1/4!
  s = ff_add(ff_mul(s, r), ff{0x1.555556p-3f, -0x1.555556p-28f});   // 1/3!
  s = ff_add(ff_mul(s, r), ff{0.5f, 0.0f});
  s = ff_add(ff_mul(s, r), ff{1.0f, 0.0f});
  s = ff_add(ff_mul(s, r), ff{1.0f, 0.0f});
  const int ki = static_cast<int>(k);
  return {ldexpf(s.hi, ki), ldexpf(s.lo, ki)};
}
static __device__ __noinline__ ff ff_exp(ff x) {
  if (!(x.hi > -104.0f)) return {0.0f, 0.0f};  // also -inf and NaN inputs
  if (x.hi > 88.0f) return {__int_as_float(0x7f800000), 0.0f};
  return ff_exp_core(x);
}

}  // namespace sv
