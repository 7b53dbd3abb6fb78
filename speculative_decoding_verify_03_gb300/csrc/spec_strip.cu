// spec_strip.cu -- strip-parallel speculative-sampling verification on
// GB300 (sm_103a).
//
// A strip is one row of logits: (sequence b, position i, tensor t), t = 0
// the target row i, t = 1 the draft row i (sampling, i < gamma_b).  Each
// strip is cut into C pieces of L elements and every piece is one CTA.  The
// grid is numbered position-major, so the pieces of early positions are
// scheduled first; a CTA whose sequence already ended at an earlier
// position (a per-sequence hint in the workspace) exits at once, so the
// early exit of the sequential walk is kept while all sequences and pieces
// run in parallel.
//
// Per piece: bulk copies (TMA, 1-D) stage the piece in shared memory; pass 1
// folds max, first argmax and NaN / +inf / finite flags, and takes a lower
// bound theta of the piece's k-th largest logit (the ceil(k/NW)-th largest
// of each warp's per-thread maxima, minimum over the warps: at least k
// elements are >= theta); pass 2 writes every element >= theta to the
// workspace as a candidate.  A piece's theta bounds the strip's k-th largest
// logit too, so the largest theta of the strip's pieces is a common bound.
//
// The last CTA to finish a position (an atomic arrival count) decides it
// (method: "Text Generation via Speculative Sampling, KV Caching, and
// OpenVINO", section "Prepare speculative sampling", steps 3 and 4;
// "CS3602_FINAL_SpeDec", section "2. 困惑度测试(PPL)"): it merges and sorts
// the candidates of p and q, applies top-k and top-p exactly (thresholds on
// the raw logit, ties kept, float-float masses), tests u < p(x)/q(x) in
// float-float, and at a rejection (or the bonus position) draws from
// norm(max(0, p - q)) (or p) by the inverse CDF in vocabulary order over
// the kept set.  When a candidate list overflowed, the exact slice-wide
// bisection, normaliser and draw run over the strip in place in global
// memory.  Each decision sets bits of a per-sequence mask (decided /
// ending positions); the decision that completes the prefix up to the first
// ending position writes the sequence's outputs.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>

#include "spec_verify.h"
#include "sv_core.cuh"
#include "sv_strip.h"

// Phase timing for development builds (-DSV_PHASE_PROFILE): thread 0 of
// each CTA accumulates clock64() deltas per phase, and counts, into a global
// array read by sv_strip_phase_read().
#ifdef SV_PHASE_PROFILE
__device__ unsigned long long sv_strip_cycles[64];
#define SP_PHASE(id)                                                                       \
  do {                                                                                     \
    if (threadIdx.x == 0) {                                                                \
      const long long now_ = clock64();                                                    \
      atomicAdd(&sv_strip_cycles[id], static_cast<unsigned long long>(now_ - t_ph_));      \
      atomicAdd(&sv_strip_cycles[32 + (id)], 1ull);                                        \
      t_ph_ = now_;                                                                        \
    }                                                                                      \
  } while (0)
#define SP_PHASE_START long long t_ph_ = clock64()
// a mark inside a helper, with its own timer variable
#define SP_MARK_START(t) long long t = clock64()
#define SP_MARK(id, t)                                                                     \
  do {                                                                                     \
    if (threadIdx.x == 0) {                                                                \
      const long long now_ = clock64();                                                    \
      atomicAdd(&sv_strip_cycles[id], static_cast<unsigned long long>(now_ - (t)));        \
      atomicAdd(&sv_strip_cycles[32 + (id)], 1ull);                                        \
      (t) = now_;                                                                          \
    }                                                                                      \
  } while (0)
// timeline (ns): [0] first CTA start, [1] last CTA exit; per position i: [2+2i] first and
// [3+2i] last decision, [20+i] last piece arrival, [36+i] first piece start
__device__ unsigned long long sv_strip_tl[64];
__device__ __forceinline__ unsigned long long sp_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
#define SP_TL_MIN(j) atomicMin(&sv_strip_tl[j], sp_now())
#define SP_TL_MAX(j) atomicMax(&sv_strip_tl[j], sp_now())
#else
#define SP_PHASE(id) \
  do {               \
  } while (0)
#define SP_PHASE_START \
  do {                 \
  } while (0)
#define SP_MARK_START(t) \
  do {                   \
  } while (0)
#define SP_MARK(id, t) \
  do {                 \
  } while (0)
#define SP_TL_MIN(j) \
  do {               \
  } while (0)
#define SP_TL_MAX(j) \
  do {               \
  } while (0)
#endif

namespace sv {

constexpr int SP_NT = 256;                  // threads per CTA
constexpr int SP_NW = SP_NT / kWarp;        // warps per CTA
constexpr int SP_MAXC = 16;                 // pieces per strip at most
constexpr int SP_UCAP = 2048;               // merged candidates per tensor and position
constexpr int SP_KCAP = 256;                // kept top-k entries per tensor (warp sort)
constexpr int SP_PIECE_BYTES = 112 * 1024;  // target piece size
constexpr uint32_t F_OVER = 8u;             // piece flag: its candidates overflowed
constexpr uint32_t FULL = 0xffffffffu;
static_assert(SP_NT == 256, "one thread per histogram bin");

// Dynamic shared memory of a deciding CTA (the piece data is dead by then).
constexpr size_t SP_DEC_SMEM = (2 * SP_UCAP + 3 * SP_KCAP) * 8 + 2 * 256 * 4 + SP_KCAP * (4 + 8);

// Top-p without top-k.  Each piece publishes the candidates at or above PH,
// a bound that at least SP_NW * SP_TOPP_K of its logits reach (about 1.5x
// that many candidates), and the single-precision sum of the weights of its
// logits below PH; the decider merges at most SP_TOPP_UCAP candidates per
// tensor.
constexpr int SP_TOPP_K = 40;  // rank in a warp's 64 largest lane values
constexpr int SP_TOPP_UCAP = 2048;
constexpr int SP_TOPP_BIN = 256;  // entries of the crossing bin ranked directly
constexpr int SP_TOPP_CAPC = 1024;
// The extension's first attempt collects the logits within this many depth
// bins (1/16 of a log2 unit each) below Theta.
constexpr float kExtBand = 8.0f;
// List masses in fixed point: a weight e in [0, 1] as round(e 2^40) (u64;
// sums of up to 2^23 weights fit, and integer sums are order-independent).
constexpr float kFix = 1099511627776.0f;  // 2^40
constexpr float kFixInv = 9.094947017729282e-13f;  // 2^-40
// Decider shared memory (top-p alone): U [2][UCAP] keys (the kept lists are
// compacted in place), K2 [UCAP], bin masses [2][256] u64, bin counts
// [2][256] u32, yb [UCAP] f32, wb [UCAP] ff, crossing-bin entries [2][2][256].
constexpr size_t SP_DEC_SMEM_P = (2 * SP_TOPP_UCAP + SP_TOPP_UCAP) * 8 + 2 * 256 * 8 +
                                 2 * 256 * 4 + SP_TOPP_UCAP * 4 + SP_TOPP_UCAP * 8 +
                                 4 * SP_TOPP_BIN * 8;

struct SP {
  KP k;                      // tensors, strides, filters, outputs
  int32_t C, L, T, NP;       // pieces, piece length, tensors per position, positions per row
  int32_t capc;              // candidates per piece
  int32_t r, r2;             // ranks of the per-warp lower bounds (k-th and ceil(k/C)-th)
  int32_t kc;                // ceil(top_k / C); top-p alone: candidates aimed at per piece
  int32_t topp;              // top-p without top-k (temperature > 0)
  int32_t law;               // spec_law: the law at the token, one position per row
  float *lps, *lbeta, *lpx, *lqx;  // its outputs [B]
  int32_t off_cb;            // shared-memory offset of the piece's candidate copy
  uint32_t *arrive;          // [B * NP] arrivals per position
  uint32_t *hint;            // [B] NP - (first ending position seen), 0 = none
  unsigned long long *mask;  // [B] bits 0..31 decided, 32..63 ending positions
  uint4 *dec;                // [B * NP * 2] decision records
  uint4 *hdr;                // [items] piece headers
  uint4 *hdr2;               // [items] top-p alone: tail weight sum (ff) and its error bound
  unsigned long long *cand;  // [items * capc] candidate keys
};

// Per-tensor result of the list selection (written by the tensor's warp).
struct LRes {
  float m, tau, Zhi, Zlo, zerr;
  int n;      // kept entries (a prefix of the sorted list)
  int exact;  // Z is float-float exact
  int ok;     // 1: the kept set is the list's first n entries; 2 (the rescan):
              // tau and Z are known but the kept set is not listed (draws
              // run over the strip); 0: neither (slice fallback)
};

struct SpShared {
  uint32_t xch[XSLOTS * XWORDS];
  uint32_t gat[XWORDS];
  uint64_t red[MAXNW * 4];
  int32_t scal[32];
  uint4 hdr[2][SP_MAXC];
  uint4 hdr2[2][SP_MAXC];
  ff xs[2][4], xa[2][4], xm[2][2];  // extension band walk: warp scans and sums, group masses
  int xj[2][3];                     // extension band walk: crossing, group first and last
  float wv[SP_NW], wth[SP_NW], wph[SP_NW];
  int wi[SP_NW];
  uint32_t wf[SP_NW];
  int wcnt[SP_NW];
  int cnt[2];
  LRes lr[2];
  float pq[2];
  float pre[4];  // prefetched for a decision: u0, u1, z(x), w(x)
  int pre_x;
  uint32_t hist[256];
  uint32_t umin;
  // top-p alone
  float wz[SP_NW][3];       // per-warp tail sums (hi, lo) and error bounds
  uint64_t gs[2][4];        // per-warp list masses of each side
  uint64_t ga[2][4];        // per-warp masses of the values >= Theta (then: before b*)
  float ge[2][4];           // per-warp weight error bounds of each side
  int gc[2][4];             // per-warp counts (compaction)
  struct TP {
    int ok, exact, bstar, nb, nkeep, blo, nbelow, deficit;
    float theta, tau;
    uint64_t cum_before, tfix, slack, zkeep, amass;
    float Zt_hi, Zt_lo, Et;  // tail of the normaliser
    float El;                // list weights' error bound
    uint64_t slist;          // list mass (fixed point)
  } tp[2];
};

// Candidate keys sort ascending as (value descending, index ascending).
__device__ __forceinline__ uint64_t cand_key(float v, int idx) {
  return (static_cast<uint64_t>(~fkey(canon(v))) << 32) | static_cast<uint32_t>(idx);
}
__device__ __forceinline__ float key_val(uint64_t k) {
  return key_to_f(~static_cast<uint32_t>(k >> 32));
}
__device__ __forceinline__ int key_idx(uint64_t k) {
  return static_cast<int>(static_cast<uint32_t>(k));
}

template <typename E>
__device__ __forceinline__ const E *strip_row(const KP &P, int b, int i, int t) {
  return t == 0 ? static_cast<const E *>(P.tgt) + static_cast<int64_t>(b) * P.t_row +
                      static_cast<int64_t>(i) * P.t_pos
                : static_cast<const E *>(P.drf) + static_cast<int64_t>(b) * P.d_row +
                      static_cast<int64_t>(i) * P.d_pos;
}

// The first ending position r of a sequence once positions 0..r are all
// decided, else -1.
__device__ __forceinline__ int first_end(unsigned long long M) {
  const uint32_t ends = static_cast<uint32_t>(M >> 32), dec = static_cast<uint32_t>(M);
  if (!ends) return -1;
  const int r = __ffs(ends) - 1;
  const uint32_t need = r == 31 ? 0xffffffffu : ((1u << (r + 1)) - 1u);
  return (dec & need) == need ? r : -1;
}


// Atomics with acquire-release order at GPU scope (the release publishes
// this CTA's earlier writes, the acquire makes the other CTAs' visible).
__device__ __forceinline__ uint32_t atom_add_acqrel(uint32_t *a, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(a), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ unsigned long long atom_or_acqrel(unsigned long long *a,
                                                             unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.acq_rel.gpu.global.or.b64 %0, [%1], %2;" : "=l"(old) : "l"(a), "l"(v) : "memory");
  return old;
}

// ------------------------------------------------------------ warp helpers
__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int m) {
  const uint32_t lo = __shfl_xor_sync(FULL, static_cast<uint32_t>(v), m);
  const uint32_t hi = __shfl_xor_sync(FULL, static_cast<uint32_t>(v >> 32), m);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ ff shfl_ff(ff v, int src) {
  return {__shfl_sync(FULL, v.hi, src), __shfl_sync(FULL, v.lo, src)};
}
__device__ __forceinline__ ff shfl_up_ff(ff v, int o) {
  return {__shfl_up_sync(FULL, v.hi, o), __shfl_up_sync(FULL, v.lo, o)};
}
// Inclusive scan over the lanes in lane order (deterministic).
__device__ __forceinline__ ff warp_scan_ff(ff v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const ff u = shfl_up_ff(v, o);
    if (lane >= o) v = ff_add(u, v);
  }
  return v;
}
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(FULL, v, o));
  return v;
}

// Bitonic sort of N = 32 NPL keys held by one warp (element s*32 + lane in
// v[s]), ascending.
template <int NPL>
__device__ __forceinline__ void warp_bitonic(uint64_t (&v)[NPL]) {
  const int lane = threadIdx.x & 31;
  constexpr int N = 32 * NPL;
#pragma unroll
  for (int kk = 2; kk <= N; kk <<= 1) {
#pragma unroll
    for (int jj = kk >> 1; jj > 0; jj >>= 1) {
      if (jj >= 32) {
#pragma unroll
        for (int s = 0; s < NPL; ++s) {
          const int s2 = s ^ (jj >> 5);
          if (s2 > s) {
            const bool up = ((s * 32 + lane) & kk) == 0;
            const uint64_t a = v[s], b = v[s2];
            const bool sw = (a > b) == up;
            v[s] = sw ? b : a;
            v[s2] = sw ? a : b;
          }
        }
      } else {
#pragma unroll
        for (int s = 0; s < NPL; ++s) {
          const uint64_t o = shfl_xor_u64(v[s], jj);
          const bool up = ((s * 32 + lane) & kk) == 0;
          const bool lower = (lane & jj) == 0;
          const uint64_t lo = v[s] < o ? v[s] : o, hi = v[s] < o ? o : v[s];
          v[s] = (lower == up) ? lo : hi;
        }
      }
    }
  }
}
template <int NPL>
__device__ __forceinline__ void warp_sort_run(uint64_t *keys, int n) {
  const int lane = threadIdx.x & 31;
  uint64_t v[NPL];
#pragma unroll
  for (int s = 0; s < NPL; ++s) {
    const int j = s * 32 + lane;
    v[s] = j < n ? keys[j] : ~0ull;
  }
  warp_bitonic<NPL>(v);
  __syncwarp();
#pragma unroll
  for (int s = 0; s < NPL; ++s) {
    const int j = s * 32 + lane;
    if (j < n) keys[j] = v[s];
  }
  __syncwarp();
}
// Sort keys[0..n) (shared memory, n <= SP_KCAP) ascending, one warp.
__device__ __noinline__ void warp_sort(uint64_t *keys, int n) {
  if (n <= 32)
    warp_sort_run<1>(keys, n);
  else if (n <= 64)
    warp_sort_run<2>(keys, n);
  else if (n <= 128)
    warp_sort_run<4>(keys, n);
  else
    warp_sort_run<8>(keys, n);
}

// The k-th smallest high word h_j = keys[j] >> 32 over j < n (1 <= k <= n),
// one warp: four rounds of 8-bit digits, each a 256-bin histogram (hist[])
// of the entries that match the digits chosen so far.  *n_le receives the
// number of entries with h_j <= the result (ties included).
__device__ __noinline__ uint32_t warp_select(const uint64_t *keys, int n, int k, uint32_t *hist,
                                             int *n_le) {
  const int lane = threadIdx.x & 31;
  uint32_t prefix = 0u, mask = 0u;
  int kr = k, eq = 0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int j = lane; j < 256; j += 32) hist[j] = 0u;
    __syncwarp();
    for (int j0 = 0; j0 < n; j0 += 32) {
      const int j = j0 + lane;
      bool in = false;
      uint32_t d = 0u;
      if (j < n) {
        const uint32_t h = static_cast<uint32_t>(keys[j] >> 32);
        in = (h & mask) == prefix;
        d = (h >> shift) & 255u;
      }
      const uint32_t act = __ballot_sync(FULL, in);
      if (in) {
        const uint32_t grp = __match_any_sync(act, d);
        if (lane == __ffs(grp) - 1) atomicAdd(&hist[d], static_cast<uint32_t>(__popc(grp)));
      }
    }
    __syncwarp();
    uint32_t c[8], loc = 0u;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      c[q] = hist[lane * 8 + q];
      loc += c[q];
    }
    uint32_t incl = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t u = __shfl_up_sync(FULL, incl, o);
      if (lane >= o) incl += u;
    }
    const uint32_t excl = incl - loc;
    const bool mine = excl < static_cast<uint32_t>(kr) && static_cast<uint32_t>(kr) <= incl;
    const int owner = __ffs(__ballot_sync(FULL, mine)) - 1;
    uint32_t d = 0u, before = excl, e = 0u;
    if (mine) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (e == 0u) {
          if (before + c[q] >= static_cast<uint32_t>(kr)) {
            d = static_cast<uint32_t>(lane * 8 + q);
            e = c[q];
          } else {
            before += c[q];
          }
        }
      }
    }
    d = __shfl_sync(FULL, d, owner);
    before = __shfl_sync(FULL, before, owner);
    e = __shfl_sync(FULL, e, owner);
    kr -= static_cast<int>(before);
    eq = static_cast<int>(e);
    prefix |= d << shift;
    mask |= 255u << shift;
    __syncwarp();
  }
  *n_le = (k - kr) + eq;
  return prefix;
}

// The k-th smallest key (value descending, index ascending) of keys[0..n),
// all with values in [lo, hi], one warp: a 256-bin value histogram (bin 0
// holds the largest values) locates the bin of the k-th entry, whose
// entries (at most 32) are ranked directly.  Returns false when that bin
// holds more than 32 entries (the caller uses the radix select).  On
// success *th = the high word of the k-th key and *n_le = the number of
// entries whose high word is <= it (the values >= the k-th value).
__device__ __noinline__ bool warp_select_bins(const uint64_t *keys, int n, int k, float lo,
                                              float hi, uint32_t *hist, uint64_t *tmp,
                                              uint32_t *th, int *n_le) {
  const int lane = threadIdx.x & 31;
  if (!(lo > -INFINITY) || !(hi < INFINITY)) return false;
  const BinMap bm = bin_map(lo, hi);
  for (int j = lane; j < 256; j += 32) hist[j] = 0u;
  __syncwarp();
  for (int j0 = 0; j0 < n; j0 += 32) {
    const int j = j0 + lane;
    const bool in = j < n;
    const int d = in ? value_bin(key_val(keys[j]), bm) : 0;
    const uint32_t act = __ballot_sync(FULL, in);
    if (in) {
      const uint32_t grp = __match_any_sync(act, d);
      if (lane == __ffs(grp) - 1) atomicAdd(&hist[d], static_cast<uint32_t>(__popc(grp)));
    }
  }
  __syncwarp();
  uint32_t c[8], loc = 0u;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    c[q] = hist[lane * 8 + q];
    loc += c[q];
  }
  uint32_t incl = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += u;
  }
  const uint32_t excl = incl - loc;
  const bool mine = excl < static_cast<uint32_t>(k) && static_cast<uint32_t>(k) <= incl;
  const int owner = __ffs(__ballot_sync(FULL, mine)) - 1;
  int d = 0;
  uint32_t before = excl, e = 0u;
  if (mine) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (e == 0u) {
        if (before + c[q] >= static_cast<uint32_t>(k)) {
          d = lane * 8 + q;
          e = c[q];
        } else {
          before += c[q];
        }
      }
    }
  }
  d = __shfl_sync(FULL, d, owner);
  before = __shfl_sync(FULL, before, owner);
  e = __shfl_sync(FULL, e, owner);
  __syncwarp();
  if (e > 32u) return false;
  // the bin's entries, one per lane
  int w = 0;
  for (int j0 = 0; j0 < n; j0 += 32) {
    const int j = j0 + lane;
    const bool in = j < n && value_bin(key_val(keys[j]), bm) == d;
    const uint32_t bal = __ballot_sync(FULL, in);
    if (in) tmp[w + __popc(bal & ((1u << lane) - 1u))] = keys[j];
    w += __popc(bal);
  }
  __syncwarp();
  const uint64_t mine_k = lane < static_cast<int>(e) ? tmp[lane] : ~0ull;
  int rank = 0;
  for (int q = 0; q < static_cast<int>(e); ++q) {
    rank += tmp[q] < mine_k ? 1 : 0;
  }
  const int want = k - static_cast<int>(before) - 1;  // 0-based rank within the bin
  const uint32_t sel = __ballot_sync(FULL, lane < static_cast<int>(e) && rank == want);
  const uint32_t t = static_cast<uint32_t>(__shfl_sync(FULL, static_cast<uint32_t>(mine_k >> 32), __ffs(sel) - 1));
  const uint32_t le = __ballot_sync(FULL, lane < static_cast<int>(e) && static_cast<uint32_t>(mine_k >> 32) <= t);
  *th = t;
  *n_le = static_cast<int>(before) + __popc(le);
  __syncwarp();
  return true;
}

constexpr float kU = 5.9604645e-8f;  // 2^-24: unit roundoff of single precision

__device__ __forceinline__ float warp_scan_f(float v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float u = __shfl_up_sync(FULL, v, o);
    if (lane >= o) v = __fadd_rn(u, v);
  }
  return v;
}

// Filters and normaliser of one tensor from its kept top-k entries
// K[0..nk) (sorted: value descending), one warp.  Top-p keeps the smallest
// leading set of equal-value groups whose mass reaches top_p of the
// survivors' mass.  Single precision: a sum of nonnegative weights computed
// along a chain of d additions is within d 2^-24 of its total (plus the
// weights' own error E); a top-p crossing within that bound is redone in
// float-float.
__device__ __forceinline__ void warp_dist(const KP &P, const uint64_t *K, int nk, LRes *out) {
  const int lane = threadIdx.x & 31;
  SP_MARK_START(t_m_);
  const float m = key_val(K[0]);
  const int rows = (nk + 31) >> 5;  // nk <= SP_KCAP = 8 rows
  // weights of the ranks r = s*32 + lane, their sum and error bound
  float e[8], v[8];
  float z = 0.0f, E = 0.0f;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int r = s * 32 + lane;
    e[s] = 0.0f;
    v[s] = -INFINITY;
    if (s < rows && r < nk) {
      float eps;
      v[s] = key_val(K[r]);
      e[s] = fw(P, v[s], m, eps);
      z = __fadd_rn(z, e[s]);
      E = __fmaf_rn(e[s], eps, E);
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    z = __fadd_rn(z, __shfl_xor_sync(FULL, z, o));
    E = __fadd_rn(E, __shfl_xor_sync(FULL, E, o));
  }
  SP_MARK(17, t_m_);  // dist: weights + sums
  int nkeep = nk, exact = 0;
  float tau = key_val(K[nk - 1]);
  float Zk = z;  // normaliser of the kept set
  ff Zx = {0.0f, 0.0f};
  if (P.p_on) {
    // first rank where the prefix mass reaches top_p * Z, certified
    const float target = __fmul_rn(z, P.top_p);
    const float zr = __fmul_rn(static_cast<float>(rows + 6) * kU, z);
    const float dp = __fmaf_rn(static_cast<float>(rows + 7) * kU, z, E);
    const float slack = __fmaf_rn(__fmaf_rn(P.top_p, __fadd_rn(E, zr), dp), 1.01f, z * kU);
    int rc = -1;
    bool cert = false;
    float carry = 0.0f;
    float pre[8];
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      pre[s] = 0.0f;
      if (s < rows) {
        const float incl = __fadd_rn(carry, warp_scan_f(e[s]));
        pre[s] = incl;
        if (rc < 0) {
          float before = __shfl_up_sync(FULL, incl, 1);
          if (lane == 0) before = carry;
          const int r = s * 32 + lane;
          const bool hit = r < nk && before < target && !(incl < target);
          const uint32_t bal = __ballot_sync(FULL, hit);
          if (bal) {
            const int L = __ffs(bal) - 1;
            rc = s * 32 + L;
            const bool ok = __fsub_rn(incl, target) > slack && __fsub_rn(target, before) > slack;
            cert = __shfl_sync(FULL, ok ? 1 : 0, L) != 0;
          }
        }
        carry = __shfl_sync(FULL, incl, 31);
      }
    }
    SP_MARK(18, t_m_);  // dist: top-p scan
    if (!cert) {
      // exact: float-float weights and prefix masses
      exact = 1;
      ff ze = {0.0f, 0.0f};
      for (int r = lane; r < nk; r += 32) ze = ff_add(ze, weight_ff(P, key_val(K[r]), m));
      ze = warp_sum_ff(ze);
      const ff tx = ff_mul_f(ze, P.top_p);
      rc = nk - 1;  // rounding left the mass short: keep the survivors
      ff cx = {0.0f, 0.0f};
      for (int r0 = 0; r0 < nk; r0 += 32) {
        const int r = r0 + lane;
        const ff w = r < nk ? weight_ff(P, key_val(K[r]), m) : ff{0.0f, 0.0f};
        const ff incl = ff_add(cx, warp_scan_ff(w));
        ff before = shfl_up_ff(incl, 1);
        if (lane == 0) before = cx;
        const uint32_t bal =
            __ballot_sync(FULL, r < nk && ff_lt(before, tx) && !ff_lt(incl, tx));
        if (bal) {
          rc = r0 + __ffs(bal) - 1;
          break;
        }
        cx = shfl_ff(incl, 31);
      }
    }
    tau = key_val(K[rc]);
    // kept ranks: the values >= tau (a prefix)
    int cnt = 0;
#pragma unroll
    for (int s = 0; s < 8; ++s) cnt += __popc(__ballot_sync(FULL, s < rows && v[s] >= tau));
    nkeep = cnt;
    if (exact) {
      for (int r = lane; r < nkeep; r += 32) Zx = ff_add(Zx, weight_ff(P, key_val(K[r]), m));
      Zx = warp_sum_ff(Zx);
    } else {
      // the prefix mass at rank nkeep - 1
      const int sr = (nkeep - 1) >> 5, lr = (nkeep - 1) & 31;
      float pk = 0.0f;
#pragma unroll
      for (int s = 0; s < 8; ++s)
        if (s == sr) pk = pre[s];
      Zk = __shfl_sync(FULL, pk, lr);
    }
  }
  SP_MARK(19, t_m_);  // dist: kept count, normaliser
  if (lane == 0) {
    out->m = m;
    out->tau = tau;
    out->Zhi = exact ? Zx.hi : Zk;
    out->Zlo = exact ? Zx.lo : 0.0f;
    // E bounds the weights' error for every subset; the sums' rounding adds
    // at most rows + 7 units
    out->zerr = exact ? 0.0f
                      : __fadd_rn(__fadd_rn(__fdiv_rn(E, Zk), static_cast<float>(rows + 7) * kU),
                                  4.8e-7f);
    out->n = nkeep;
    out->exact = exact;
    out->ok = 1;
  }
  __syncwarp();
}

// Float-float normaliser of a list-mode distribution (exact paths), one warp.
__device__ __noinline__ ff warp_exact_Z(const KP &P, const uint64_t *K, int n, float m) {
  const int lane = threadIdx.x & 31;
  ff z = {0.0f, 0.0f};
  for (int r = lane; r < n; r += 32) z = ff_add(z, weight_ff(P, key_val(K[r]), m));
  return warp_sum_ff(z);
}
__device__ __forceinline__ void warp_make_exact(const KP &P, const uint64_t *K, Dist &D) {
  set_Zx(D, warp_exact_Z(P, K, D.n, D.m));
}

// Inverse-CDF draw over the p-list in vocabulary order (K2: index-sorted
// (index, rank) pairs of the n kept p-ranks; yb[rank]: the draft logit of
// that token), one warp.  fast: certified single precision, returns the
// token, -1 (total weight 0) or -2 (a CDF boundary within the error bound);
// exact: float-float, returns the token (the last positive weight when
// rounding leaves the target past it) or -1.  wb: n weights of scratch.
__device__ __noinline__ int warp_list_draw_exact(const KP &P, const uint64_t *Kp,
                                                 const uint64_t *K2, const float *yb, int n,
                                                 const Dist &dt, const Dist &dd, bool residual,
                                                 float u, float *Wout, ff *wb);
__device__ __forceinline__ int warp_list_draw(const KP &P, const uint64_t *Kp, const uint64_t *K2,
                                              const float *yb, int n, const Dist &dt,
                                              const Dist &dd, bool residual, float u, bool fast,
                                              float *Wout, ff *wb) {
  const int lane = threadIdx.x & 31;
  if (fast) {
    // single precision: weights with absolute error bounds e_j; sums along
    // chains of at most rows + 7 additions
    float s = 0.0f, D = 0.0f;
    float *wf = reinterpret_cast<float *>(wb);
    for (int j = lane; j < n; j += 32) {
      const int r = static_cast<int>(static_cast<uint32_t>(K2[j]));
      const float x = key_val(Kp[r]);
      const float y = residual ? yb[r] : 0.0f;
      float w, e;
      fast_weight(P, x, y, dt, dd, residual, w, e);
      wf[j] = w;
      s = __fadd_rn(s, w);
      D = __fadd_rn(D, e);
    }
    __syncwarp();
    const float W = warp_sum_f(s);
    const int rows = (n + 31) >> 5;
    D = __fmaf_rn(static_cast<float>(rows + 7) * kU, W, warp_sum_f(D));
    *Wout = W;
    if (!(W > 0.0f)) return -1;
    const float target = __fmul_rn(W, u);
    const float need = __fmaf_rn(2.0f, D, __fmaf_rn(2.0f * kU, W, static_cast<float>(n) * 4e-38f *
                                                         (dt.rzf + (residual ? dd.rzf : 0.0f))));
    float carry = 0.0f;
    for (int j0 = 0; j0 < n; j0 += 32) {
      const int j = j0 + lane;
      const float w = j < n ? wf[j] : 0.0f;
      const float incl = __fadd_rn(carry, warp_scan_f(w));
      float before = __shfl_up_sync(FULL, incl, 1);
      if (lane == 0) before = carry;
      const bool hit = j < n && w > 0.0f && !(target < before) && target < incl;
      const uint32_t bal = __ballot_sync(FULL, hit);
      if (bal) {
        const int L = __ffs(bal) - 1;
        const float margin = fminf(__fsub_rn(target, before), __fsub_rn(incl, target));
        const int ok = __shfl_sync(FULL, margin > need ? 1 : 0, L);
        const int tok = __shfl_sync(FULL, j < n ? static_cast<int>(K2[j] >> 32) : -1, L);
        return ok ? tok : -2;
      }
      carry = __shfl_sync(FULL, incl, 31);
    }
    return -2;
  }
  // copies: the distributions of the caller stay in registers
  const Dist a = dt, c = dd;
  return warp_list_draw_exact(P, Kp, K2, yb, n, a, c, residual, u, Wout, wb);
}
__device__ __noinline__ int warp_list_draw_exact(const KP &P, const uint64_t *Kp,
                                                 const uint64_t *K2, const float *yb, int n,
                                                 const Dist &dt, const Dist &dd, bool residual,
                                                 float u, float *Wout, ff *wb) {
  const int lane = threadIdx.x & 31;
  // float-float
  ff s = {0.0f, 0.0f};
  int last = -1;
  for (int j = lane; j < n; j += 32) {
    const int v = static_cast<int>(K2[j] >> 32), r = static_cast<int>(static_cast<uint32_t>(K2[j]));
    const float x = key_val(Kp[r]);
    const float y = residual ? yb[r] : 0.0f;
    const ff w = draw_weight_of(P, x, y, dt, dd, residual);
    if (w.hi > 0.0f) last = max(last, v);
    wb[j] = w;
    s = ff_add(s, w);
  }
  __syncwarp();
  const ff W = warp_sum_ff(s);
#pragma unroll
  for (int o = 16; o; o >>= 1) last = max(last, __shfl_xor_sync(FULL, last, o));
  *Wout = __fadd_rn(W.hi, W.lo);
  if (!(W.hi > 0.0f)) return -1;
  const ff target = ff_mul_f(W, u);
  ff carry = {0.0f, 0.0f};
  for (int j0 = 0; j0 < n; j0 += 32) {
    const int j = j0 + lane;
    const ff w = j < n ? wb[j] : ff{0.0f, 0.0f};
    const ff incl = ff_add(carry, warp_scan_ff(w));
    ff before = shfl_up_ff(incl, 1);
    if (lane == 0) before = carry;
    const bool hit = j < n && w.hi > 0.0f && !ff_lt(target, before) && ff_lt(target, incl);
    const uint32_t bal = __ballot_sync(FULL, hit);
    if (bal) {
      const int L = __ffs(bal) - 1;
      return __shfl_sync(FULL, j < n ? static_cast<int>(K2[j] >> 32) : -1, L);
    }
    carry = shfl_ff(incl, 31);
  }
  return last;
}

// Ascending bitonic sort of a[0..N) (N a power of two; pad with ~0) by nt
// threads of a group (thread t) that synchronise on named barrier `bar`.
__device__ __noinline__ void group_bitonic(uint64_t *a, int N, int t, int nt, int bar) {
  for (int k = 2; k <= N; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int m = t; m < (N >> 1); m += nt) {
        const int lo = 2 * m - (m & (j - 1)), hi = lo + j;
        const bool up = (lo & k) == 0;
        const uint64_t x = a[lo], y = a[hi];
        if ((x > y) == up) {
          a[lo] = y;
          a[hi] = x;
        }
      }
      named_sync(bar, nt);
    }
  }
}

// Inclusive scan of u64 values over the lanes, in lane order.
__device__ __forceinline__ uint64_t warp_scan_u64(uint64_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t u = static_cast<uint64_t>(__shfl_up_sync(FULL, static_cast<long long>(v), o));
    if (lane >= o) v += u;
  }
  return v;
}

// Weights with the temperature passed in registers (for the out-of-line
// top-p helpers, which would otherwise reload the launch parameters through
// a generic pointer inside their loops): fast e^{(z - m)/T} with its error
// bound (c2 = log2(e)/T), and the float-float weight (1/T = ih + il).
__device__ __forceinline__ float fw_c(float c2, float z, float m, float &eps) {
  if (z == -INFINITY) {
    eps = 0.0f;
    return 0.0f;
  }
  const float y = __fmul_rn(__fsub_rn(z, m), c2);
  eps = __fmaf_rn(fabsf(y), kExpErr1, kExpErr0);
  return ex2_approx(y);
}
__device__ __forceinline__ ff wff_c(float ih, float il, float z, float m) {
  if (z == -INFINITY) return {0.0f, 0.0f};
  return ff_exp(ff_mul(two_sum(z, -m), ff{ih, il}));
}

// round(x 2^40) for x in [0, 2^20) as an integer, from the float's bits (the
// float-to-64-bit-integer conversion runs on the slow double-precision pipe).
__device__ __forceinline__ uint64_t to_fix40(float x) {
  const uint32_t u = __float_as_uint(x);
  const int e = static_cast<int>(u >> 23) - 127 + 40;  // x 2^40 = m 2^(e - 23)
  const uint64_t m = (u & 0x7fffffu) | 0x800000u;
  if (x <= 0.0f || e < -1) return 0ull;  // below 2^-41: rounds to 0
  if (e >= 23) return m << (e - 23);
  const int sh = 23 - e;  // 1 .. 24: round to nearest, ties up
  return (m + (1ull << (sh - 1))) >> sh;
}

// A fixed-point mass (units of 2^-40) as float-float.
__device__ __forceinline__ ff fix_to_ff(uint64_t x) {
  const float hi = __ull2float_rn(x);
  const long long r = static_cast<long long>(x - __float2ull_rn(hi));
  return quick_two_sum(__fmul_rn(hi, kFixInv), __fmul_rn(__ll2float_rn(r), kFixInv));
}

// Filters and normalisers of both tensors of a position under top-p alone
// (whole CTA; side s = threads [128 s, 128 s + 128) handles tensor s < T).
// The pieces published every logit >= PH_c (their candidates) and the sum
// of the weights below PH_c (their tails), so Z = tails + the candidates'
// weights, and the logits >= Theta = max_c PH_c are all present: when their
// mass reaches top_p Z, the top-p crossing (the first group of equal logits,
// from the largest, where the cumulative mass reaches top_p Z) lies among
// them.  Fast path: single-precision weights summed in fixed point (exact,
// order-independent integer sums), a 256-bin mass histogram of the values
// >= Theta to find the crossing bin, whose entries are ranked and walked;
// accepted when the crossing's margins exceed the error bound.  Otherwise
// the candidates are sorted and walked in float-float (only the tails keep
// single-precision error).  Writes sh.lr[s] (ok = 0: the caller takes the
// exact slice-wide path) and leaves the kept list (value >= tau) in
// U[s * SP_TOPP_UCAP ...]: in candidate order (fast) or sorted (exact).
__device__ __noinline__ void topp_lists(const SP &S, SpShared &sh, int T, int64_t hb,
                                        const float *Mx, const float *Th, const uint32_t *fl,
                                        uint64_t *U, uint64_t *hm, uint32_t *hc, uint64_t *bs) {
  const int tid = threadIdx.x, s = tid >> 7, lt = tid & 127, lane = tid & 31,
            w4 = (tid >> 5) & 3;
  // launch parameters in registers
  const int C = S.C, capc = S.capc;
  const unsigned long long *cand = S.cand;
  const float c2 = S.k.c2, ih = S.k.invT_hi, il = S.k.invT_lo, top_p = S.k.top_p;
  SP_MARK_START(t_tl_);
  int offs[SP_MAXC + 1];
  offs[0] = 0;
#pragma unroll
  for (int q = 0; q < SP_MAXC; ++q)
    offs[q + 1] = offs[q] + ((q < C && s < T) ? static_cast<int>(sh.hdr[s][q].x & 0xffffffu) : 0);
  const int n = offs[SP_MAXC];
  const bool act = s < T && !(fl[s] & F_OVER) && n <= SP_TOPP_UCAP;
  int nmax = 0;  // uniform loop bound of the compaction
  for (int t2 = 0; t2 < T; ++t2) {
    int m2 = 0;
    for (int q = 0; q < C; ++q) m2 += static_cast<int>(sh.hdr[t2][q].x & 0xffffffu);
    nmax = max(nmax, m2);
  }
  nmax = min(nmax, SP_TOPP_UCAP);
  const float M = s < T ? Mx[s] : 0.0f, Theta = s < T ? Th[s] : 0.0f;
  uint64_t *Us = U + s * SP_TOPP_UCAP;
  // the side's 2 KB of bin space: [256] u32 approximate bin masses (each
  // weight over its bin's largest weight, times 2^12), then [256] the
  // reciprocals of the bins' largest weights; [256] u32 exact bin counts
  uint32_t *hus = reinterpret_cast<uint32_t *>(hm + s * 256);
  float *wtop = reinterpret_cast<float *>(hm + s * 256) + 256;
  uint32_t *hcs = hc + s * 256;
  uint64_t *bsg = bs + s * 2 * SP_TOPP_BIN, *bss = bsg + SP_TOPP_BIN;
  const bool thfin = Theta > -INFINITY;
  const BinMap bm = bin_map(thfin ? Theta : M, M);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int b = lt + 128 * h;
    hus[b] = 0u;
    hcs[b] = 0u;
    // the largest value of bin b: 2 (hh - b / sc) (bin 0 holds M)
    const float vt = (b == 0 || bm.deg) ? M : fminf(M, 2.0f * __fsub_rn(bm.hh, __fdiv_rn(static_cast<float>(b), bm.sc)));
    const float wt = ex2_approx(__fmul_rn(__fsub_rn(vt, M), c2));
    wtop[b] = wt > 0.0f ? __frcp_rn(wt) : 0.0f;  // the reciprocal (0: an empty weight range)
  }
  if (lt == 0) {
    sh.tp[s].ok = 0;
    sh.tp[s].exact = 0;
    sh.tp[s].amass = ~0ull;  // set once the list's sums are complete
    sh.tp[s].deficit = 0;
    sh.gc[s][0] = 0;
  }
  __syncthreads();
  // gather (piece order, then each piece's order), weights, bins; exact
  // fixed-point sums of all weights and of the weights >= Theta
  uint64_t fsum = 0ull, asum = 0ull;
  float esum = 0.0f;
  constexpr int GPT = SP_TOPP_UCAP / 128;  // entries per thread at most
  if (act) {
    {
      uint64_t kv[GPT];  // every load of the thread in flight at once (one L2 round trip)
#pragma unroll
      for (int u = 0; u < GPT; ++u) {
        const int j = u * 128 + lt;
        kv[u] = ~0ull;
        if (j < n) {
          int c = 0;
#pragma unroll
          for (int q = 1; q < SP_MAXC; ++q)
            if (q < C && j >= offs[q]) c = q;
          kv[u] = __ldcg(cand + (hb + s * C + c) * capc + (j - offs[c]));
        }
      }
#pragma unroll
      for (int u = 0; u < GPT; ++u) {
        const int j = u * 128 + lt;
        if (j < n) {
          const uint64_t key = kv[u];
          Us[j] = key;
          const float z = key_val(key);
          float eps;
          const float e = fw_c(c2, z, M, eps);
          const uint64_t f = to_fix40(e);
          fsum += f;
          esum = __fmaf_rn(e, eps, esum);
          if (z >= Theta) {
            asum += f;
            const int b = thfin ? value_bin(z, bm) : 0;
            atomicAdd(&hus[b], __float2uint_rn(__fmul_rn(__fmul_rn(e, wtop[b]), 4096.0f)));
            atomicAdd(&hcs[b], 1u);
          }
        }
      }
    }
  }
  fsum = warp_sum_u64(fsum);
  asum = warp_sum_u64(asum);
  esum = warp_sum_f(esum);
  if (lane == 0) {
    sh.gs[s][w4] = fsum;
    sh.ge[s][w4] = esum;
    sh.ga[s][w4] = asum;
  }
  __syncthreads();
  SP_MARK(14, t_tl_);  // top-p lists: gather + weights + bins
  // the normaliser, the target top_p Z and the crossing bin (one warp per side)
  if (act && w4 == 0) {
    uint64_t sl = 0ull;
    float el = 0.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      sl += sh.gs[s][q];
      el = __fadd_rn(el, sh.ge[s][q]);
    }
    ff zt = {0.0f, 0.0f};
    float et = 0.0f;
    for (int c = 0; c < C; ++c) {
      const uint4 h = sh.hdr[s][c], h2 = sh.hdr2[s][c];
      const float zh = __uint_as_float(h2.x);
      if (zh > 0.0f) {
        const float y = __fmul_rn(__fsub_rn(__uint_as_float(h.y), M), c2);
        const float fac = ex2_approx(y);
        const float ferr = __fmaf_rn(fabsf(y), kExpErr1, kExpErr0);
        zt = ff_add(zt, ff_mul_f(ff{zh, __uint_as_float(h2.y)}, fac));
        et = __fadd_rn(et, __fmul_rn(__fmaf_rn(zh, ferr, __uint_as_float(h2.z)), fac));
      }
    }
    // weights rounded to 2^-41 each; tail factors' rounding
    el = __fadd_rn(el, static_cast<float>(n) * 4.6e-13f);
    const ff Z = ff_add(zt, fix_to_ff(sl));
    const float EZ = __fmaf_rn(Z.hi, 1e-12f, __fadd_rn(et, el));
    const ff Tt = ff_mul_f(Z, top_p);
    const long long tfix = __float2ll_rn(__fmul_rn(Tt.hi, kFix)) +
                           __float2ll_rn(__fmul_rn(Tt.lo, kFix));
    const float slackf = __fmul_rn(__fmaf_rn(top_p, EZ, el), 1.01f);
    const uint64_t slack = __float2ull_ru(__fmul_rn(slackf, kFix)) + 8ull;
    uint64_t A = 0ull;  // the exact mass of the values >= Theta
#pragma unroll
    for (int q = 0; q < 4; ++q) A += sh.ga[s][q];
    const uint64_t tf = tfix > 0 ? static_cast<uint64_t>(tfix) : 0ull;
    // the crossing bin from the approximate bin masses (2^-13 relative):
    // the first bin where the cumulative mass reaches top_p Z; the walk
    // checks it against exact sums
    const float tgt = __fmul_rn(static_cast<float>(tf), kFixInv);
    float c8[8], loc = 0.0f;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int bq = lane * 8 + q;
      c8[q] = wtop[bq] > 0.0f ? __fmul_rn(__fmul_rn(static_cast<float>(hus[bq]), 2.44140625e-4f),
                                          __frcp_rn(wtop[bq]))
                              : 0.0f;
      loc = __fadd_rn(loc, c8[q]);
    }
    const float incl = warp_scan_f(loc);
    const float excl = __fsub_rn(incl, loc);
    const bool mine = excl < tgt && tgt <= incl;
    uint32_t own = __ballot_sync(FULL, mine);
    int bstar = -1;
    if (mine) {
      float before = excl;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (bstar < 0) {
          before = __fadd_rn(before, c8[q]);
          if (before >= tgt) bstar = lane * 8 + q;
        }
      }
    }
    if (!own) {  // rounding left the target past the last bin: the last non-empty bin
      int lastb = -1;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (hcs[lane * 8 + q]) lastb = lane * 8 + q;
      own = __ballot_sync(FULL, lastb >= 0);
      bstar = lastb;
      if (own) own = 1u << (31 - __clz(own));
    }
    int nbefore = 0, nwalk = 0;
    if (own) {
      const int L = __ffs(own) - 1;
      bstar = __shfl_sync(FULL, bstar, L);
      // entries of the bins before b* - 1, and of the bins b*-1 .. b*+1
      int cnt = 0, cw = 0;
      for (int b = lane; b < 256; b += 32) {
        cnt += b < max(0, bstar - 1) ? static_cast<int>(hcs[b]) : 0;
        cw += (b >= bstar - 1 && b <= bstar + 1) ? static_cast<int>(hcs[b]) : 0;
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        cnt += __shfl_xor_sync(FULL, cnt, o);
        cw += __shfl_xor_sync(FULL, cw, o);
      }
      nbefore = cnt;
      nwalk = cw;
    }
    if (lane == 0) {
      auto &tp = sh.tp[s];
      tp.ok = (own != 0u && A >= tf + slack) ? 1 : 0;
      tp.deficit = (A >= tf + slack) ? 0 : 1;
      tp.bstar = bstar;
      tp.nb = nwalk;
      tp.blo = max(0, bstar - 1);
      tp.nbelow = nbefore;
      tp.tfix = tf;
      tp.slack = slack;
      tp.amass = A;
      tp.theta = Theta;
      tp.Zt_hi = zt.hi;
      tp.Zt_lo = zt.lo;
      tp.Et = et;
      tp.El = el;
      tp.slist = sl;
    }
  }
  __syncthreads();
  SP_MARK(11, t_tl_);  // top-p lists: normaliser + crossing bin
  // fast path: rank the crossing bin's entries and walk them
  const int okf = act ? sh.tp[s].ok : 0;
  const int nb = sh.tp[s].nb, bstar = sh.tp[s].bstar;
  const int blo = sh.tp[s].blo;  // the first bin walked
  const bool walk = okf && nb <= SP_TOPP_BIN;
  {
    // the entries of the bins b*-1 .. b*+1 (the estimate of b* may be one
    // bin off), and the exact mass of the bins before them
    uint64_t cb = 0ull;
    if (walk) {
      for (int j = lt; j < n; j += 128) {
        const uint64_t key = Us[j];
        const float z = key_val(key);
        if (z >= Theta) {
          const int bz = thfin ? value_bin(z, bm) : 0;
          if (bz >= blo && bz <= bstar + 1) {
            const int pos = atomicAdd(&sh.gc[s][0], 1);
            if (pos < SP_TOPP_BIN) bsg[pos] = key;
          } else if (bz < blo) {
            float eps;
            cb += to_fix40(fw_c(c2, z, M, eps));
          }
        }
      }
    }
    cb = warp_sum_u64(cb);
    if (lane == 0) sh.ga[s][w4] = cb;
  }
  __syncthreads();
  if (walk && lt == 0) {
    uint64_t cb = 0ull;
#pragma unroll
    for (int q = 0; q < 4; ++q) cb += sh.ga[s][q];
    sh.tp[s].cum_before = cb;
  }
  __syncthreads();
  if (walk) {
    for (int j = lt; j < nb; j += 128) {
      const uint64_t kk = bsg[j];
      int rank = 0;
      for (int l = 0; l < nb; ++l) rank += bsg[l] < kk ? 1 : 0;
      bss[rank] = kk;
    }
  }
  __syncthreads();
  if (walk && w4 == 0) {
    const uint64_t tf = sh.tp[s].tfix, slack = sh.tp[s].slack;
    uint64_t carry = sh.tp[s].cum_before;
    int cross = -1;
    for (int r0 = 0; r0 < nb && cross < 0; r0 += 32) {
      const int r = r0 + lane;
      uint64_t f = 0ull;
      if (r < nb) {
        float eps;
        f = to_fix40(fw_c(c2, key_val(bss[r]), M, eps));
      }
      const uint64_t incl = carry + warp_scan_u64(f);
      const bool hit = r < nb && incl - f < tf && incl >= tf;
      const uint32_t bal = __ballot_sync(FULL, hit);
      if (bal) cross = r0 + __ffs(bal) - 1;
      carry = static_cast<uint64_t>(__shfl_sync(FULL, static_cast<long long>(incl), 31));
    }
    int ok = 0;
    if (cross >= 0) {
      const uint32_t hk = static_cast<uint32_t>(bss[cross] >> 32);
      // the group of equal values around the crossing entry: [g0, g1]
      int g0 = nb, g1 = -1;
      uint64_t mA = 0ull, mB = 0ull;
      for (int r = lane; r < nb; r += 32) {
        const uint32_t h = static_cast<uint32_t>(bss[r] >> 32);
        float eps;
        const uint64_t f = to_fix40(fw_c(c2, key_val(bss[r]), M, eps));
        if (h == hk) {
          g0 = min(g0, r);
          g1 = max(g1, r);
        }
        if (h < hk) mA += f;   // larger values: before the group
        if (h <= hk) mB += f;  // up to the group's end
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        g0 = min(g0, __shfl_xor_sync(FULL, g0, o));
        g1 = max(g1, __shfl_xor_sync(FULL, g1, o));
      }
      mA = warp_sum_u64(mA);
      mB = warp_sum_u64(mB);
      const uint64_t cumA = sh.tp[s].cum_before + mA, cumB = sh.tp[s].cum_before + mB;
      ok = (tf > cumA && tf - cumA > slack && cumB > tf && cumB - tf > slack) ? 1 : 0;
      if (lane == 0 && ok) {
        sh.tp[s].tau = key_val(bss[g0]);
        sh.tp[s].nkeep = sh.tp[s].nbelow + g1 + 1;
        sh.tp[s].zkeep = cumB;
      }
    }
    if (lane == 0) sh.tp[s].exact = ok ? 0 : 1;  // 1: take the float-float path
  }
  __syncthreads();
  SP_MARK(16, t_tl_);  // top-p lists: crossing bin ranked and walked
  const bool fast = walk && sh.tp[s].exact == 0;
  const bool exf = act && okf && !fast;
#ifdef SV_PHASE_PROFILE
  if (lt == 0 && s < T) {
    atomicAdd(&sv_strip_cycles[29], 1ull);
    atomicAdd(&sv_strip_cycles[26], static_cast<unsigned long long>(n));
    if (act && okf) atomicAdd(&sv_strip_cycles[27], static_cast<unsigned long long>(nb));
    if (exf) atomicAdd(&sv_strip_cycles[24], 1ull);
    if (act && okf && nb > SP_TOPP_BIN) atomicAdd(&sv_strip_cycles[25], 1ull);
    if (!(act && okf)) atomicAdd(&sv_strip_cycles[28], 1ull);
    if (!act) atomicAdd(&sv_strip_cycles[31], 1ull);  // overflowed lists
  }
#endif
  // fast: compact the kept entries (value >= tau) to the front, stably
  {
    const uint32_t kmax = fast ? ~fkey(canon(sh.tp[s].tau)) : 0u;
    int run = 0;
    for (int base = 0; base < nmax; base += 128) {
      const int j = base + lt;
      const uint64_t key = (fast && j < n) ? Us[j] : ~0ull;
      const bool pred = fast && j < n && static_cast<uint32_t>(key >> 32) <= kmax;
      const uint32_t bal = __ballot_sync(FULL, pred);
      if (lane == 0) sh.gc[s][w4] = __popc(bal);
      __syncthreads();
      int wb = 0, tot = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int x = sh.gc[s][q];
        wb += q < w4 ? x : 0;
        tot += x;
      }
      if (pred) Us[run + wb + __popc(bal & ((1u << lane) - 1u))] = key;
      run += tot;
      __syncthreads();
    }
  }
  SP_MARK(30, t_tl_);  // top-p lists: compaction
  // exact: sort every candidate, float-float normaliser and walk
  int Nx = 128;
  while (Nx < n && Nx < SP_TOPP_UCAP) Nx <<= 1;
  if (exf)
    for (int j = n + lt; j < Nx; j += 128) Us[j] = ~0ull;
  __syncthreads();
  if (exf) group_bitonic(Us, Nx, lt, 128, 1 + s);
  __syncthreads();
  if (exf) {
    ff a = {0.0f, 0.0f};
    for (int j = lt; j < n; j += 128) a = ff_add(a, wff_c(ih, il, key_val(Us[j]), M));
    a = warp_sum_ff(a);
    if (lane == 0) {
      sh.ge[s][w4] = a.hi;
      reinterpret_cast<float *>(&sh.gs[s][w4])[0] = a.lo;
    }
  }
  __syncthreads();
  if (exf && w4 == 0) {
    ff zl = {0.0f, 0.0f};
#pragma unroll
    for (int q = 0; q < 4; ++q)
      zl = ff_add(zl, ff{sh.ge[s][q], reinterpret_cast<const float *>(&sh.gs[s][q])[0]});
    const ff Z = ff_add(ff{sh.tp[s].Zt_hi, sh.tp[s].Zt_lo}, zl);
    const float E = __fmaf_rn(Z.hi, 1e-12f, sh.tp[s].Et);
    const ff Tt = ff_mul_f(Z, top_p);
    const float slack = __fmaf_rn(top_p, E, __fmul_rn(Z.hi, 1e-12f));
    ff carry = {0.0f, 0.0f};
    int cross = -1;
    bool below = false;
    for (int r0 = 0; r0 < n && cross < 0 && !below; r0 += 32) {
      const int r = r0 + lane;
      const float z = r < n ? key_val(Us[r]) : -INFINITY;
      const bool in = r < n && z >= Theta;
      const ff w = in ? wff_c(ih, il, z, M) : ff{0.0f, 0.0f};
      const ff incl = ff_add(carry, warp_scan_ff(w));
      ff bef = shfl_up_ff(incl, 1);
      if (lane == 0) bef = carry;
      const uint32_t bal = __ballot_sync(FULL, in && ff_lt(bef, Tt) && !ff_lt(incl, Tt));
      if (bal) cross = r0 + __ffs(bal) - 1;
      below = __ballot_sync(FULL, r < n && !in) != 0u;
      carry = shfl_ff(incl, 31);
    }
    int ok = 0;
    if (cross >= 0) {
      const uint32_t hk = static_cast<uint32_t>(Us[cross] >> 32);
      int g0 = n, g1 = -1;
      ff mA = {0.0f, 0.0f}, mB = {0.0f, 0.0f};
      for (int r0 = 0; r0 < n; r0 += 32) {
        const int r = r0 + lane;
        const uint32_t h = r < n ? static_cast<uint32_t>(Us[r] >> 32) : 0xffffffffu;
        const bool inB = r < n && h <= hk;
        const ff w = inB ? wff_c(ih, il, key_val(Us[r]), M) : ff{0.0f, 0.0f};
        if (r < n && h == hk) {
          g0 = min(g0, r);
          g1 = max(g1, r);
        }
        mB = ff_add(mB, w);
        if (h < hk) mA = ff_add(mA, w);
        if (__ballot_sync(FULL, r < n && h > hk)) break;  // sorted: the rest is smaller
      }
      mA = warp_sum_ff(mA);
      mB = warp_sum_ff(mB);
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        g0 = min(g0, __shfl_xor_sync(FULL, g0, o));
        g1 = max(g1, __shfl_xor_sync(FULL, g1, o));
      }
      const ff dA = ff_sub(Tt, mA), dB = ff_sub(mB, Tt);
      // certified; or the top-p mass lies within 1e-6 Z of the group's
      // boundary whatever the rounding (a boundary case: any consistent
      // choice is a valid reading), and the walk's own choice stands
      ok = ((dA.hi > slack && dB.hi > slack) || __fmul_rn(2.0f, slack) < __fmul_rn(Z.hi, 1e-6f)) ? 1 : 0;
      if (lane == 0 && ok) {
        sh.tp[s].tau = key_val(Us[g0]);
        sh.tp[s].nkeep = g1 + 1;
        sh.tp[s].Zt_hi = mB.hi;  // the kept set's normaliser (float-float)
        sh.tp[s].Zt_lo = mB.lo;
      }
    }
    if (lane == 0) sh.tp[s].ok = ok;
  }
  __syncthreads();
  if (s < T && lt == 0) {
    LRes *out = &sh.lr[s];
    const auto &tp = sh.tp[s];
    out->m = M;
    if (!act || !tp.ok) {
      out->ok = 0;
    } else if (fast) {
      const ff zk = fix_to_ff(tp.zkeep);
      out->tau = tp.tau;
      out->Zhi = zk.hi;
      out->Zlo = zk.lo;
      out->zerr = __fadd_rn(__fdiv_rn(tp.El, zk.hi), 2.4e-7f);
      out->n = tp.nkeep;
      out->exact = 0;
      out->ok = 1;
    } else {
      out->tau = tp.tau;
      out->Zhi = tp.Zt_hi;
      out->Zlo = tp.Zt_lo;
      out->zerr = 0.0f;
      out->n = tp.nkeep;
      out->exact = 1;
      out->ok = 1;
    }
  }
  __syncthreads();
}

// The depth of z below the bound th, in 1/16 of a log2 unit of weight
// (monotone non-increasing in z; NaN for NaN).
__device__ __forceinline__ float band_depth(float th, float z, float c2) {
  return __fmul_rn(__fmul_rn(__fsub_rn(th, z), c2), 16.0f);
}

// One element of a strip row in the rescan: the weight e^{(z - M)/T} and
// its depth bin (1/8 of a log2 unit per bin below M; bin 255 holds the rest).
__device__ __forceinline__ void rescan_elem(float c2, float z, float M, float &w, float &y,
                                            int &bin) {
  y = __fmul_rn(__fsub_rn(z, M), c2);
  w = z > -INFINITY ? ex2_approx(y) : 0.0f;
  const float d = __fmul_rn(y, -8.0f);
  bin = (z > -INFINITY && d < 255.0f) ? static_cast<int>(d) : 255;
}

// Visit the elements of a strip row (global memory) in index order per
// thread: 16-byte vectors (GL loads in flight) when the row is aligned,
// element loads otherwise.  fn(value, index).
template <typename E, int GL = 8, typename Fn>
__device__ __forceinline__ void rescan_row(const E *g, int V, int t, int nt, Fn &&fn) {
  constexpr int EPV = Elem<E>::kPerVec;
  int done = 0;
  if ((reinterpret_cast<uintptr_t>(g) & 15u) == 0) {
    const uint4 *g4 = reinterpret_cast<const uint4 *>(g);
    const int nv = V / EPV;
    for (int v0 = 0; v0 < nv; v0 += GL * nt) {
      uint4 x[GL];
#pragma unroll
      for (int u = 0; u < GL; ++u) {
        const int v = v0 + u * nt + t;
        if (v < nv) x[u] = __ldcg(g4 + v);
      }
#pragma unroll
      for (int u = 0; u < GL; ++u) {
        const int v = v0 + u * nt + t;
        if (v < nv) {
          float f[EPV];
          unpack<E>(x[u], f);
#pragma unroll
          for (int e = 0; e < EPV; ++e) fn(f[e], v * EPV + e);
        }
      }
    }
    done = nv * EPV;
  }
  for (int j = done + t; j < V; j += nt) fn(raw_of(g[j]), j);
}

// Sort the side's list Us[0..tot) (descending values) and walk it in
// float-float against top_p Z: the first group of equal logits where the
// cumulative mass reaches top_p Z, certified (or within 1e-6 Z of it).  The
// list must hold every logit >= its smallest entry.  Writes sh.lr[s] (ok = 0
// when no group reaches top_p Z or the walk is within the error bound).
// Whole CTA (side s = threads [128 s, 128 s + 128) works on tensor s when
// go); wx: [UCAP] float-float scratch of the side.
__device__ __noinline__ void ext_sort_walk(const SP &S, SpShared &sh, int s, bool go, int tot,
                                           float M, uint64_t *Us, ff *wx) {
  const int tid = threadIdx.x, lt = tid & 127, lane = tid & 31, w4 = (tid >> 5) & 3;
  const float ih = S.k.invT_hi, il = S.k.invT_lo, top_p = S.k.top_p;
  int N = 128;
  while (N < tot && N < SP_TOPP_UCAP) N <<= 1;
  if (go)
    for (int j = tot + lt; j < N; j += 128) Us[j] = ~0ull;
  __syncthreads();
  if (go) group_bitonic(Us, N, lt, 128, 1 + s);
  __syncthreads();
  // the float-float weights of the sorted list, by the side's threads
  if (go)
    for (int j = lt; j < tot; j += 128) wx[j] = wff_c(ih, il, key_val(Us[j]), M);
  __syncthreads();
  if (go && w4 == 0) {
    const ff Z = ff_add(ff{sh.tp[s].Zt_hi, sh.tp[s].Zt_lo}, fix_to_ff(sh.tp[s].slist));
    const float EZ = __fmaf_rn(Z.hi, 1e-12f, __fadd_rn(sh.tp[s].Et, sh.tp[s].El));
    const ff Tt = ff_mul_f(Z, top_p);
    const float slack = __fmaf_rn(top_p, EZ, __fmul_rn(Z.hi, 1e-12f));
    ff carry = {0.0f, 0.0f};
    int cross = -1;
    for (int r0 = 0; r0 < tot && cross < 0; r0 += 32) {
      const int r = r0 + lane;
      const ff w = r < tot ? wx[r] : ff{0.0f, 0.0f};
      const ff incl = ff_add(carry, warp_scan_ff(w));
      ff bef = shfl_up_ff(incl, 1);
      if (lane == 0) bef = carry;
      const uint32_t bal = __ballot_sync(FULL, r < tot && ff_lt(bef, Tt) && !ff_lt(incl, Tt));
      if (bal) cross = r0 + __ffs(bal) - 1;
      carry = shfl_ff(incl, 31);
    }
    int ok = 0;
    if (cross >= 0) {
      const uint32_t hk = static_cast<uint32_t>(Us[cross] >> 32);
      int g0 = tot, g1 = -1;
      ff mA = {0.0f, 0.0f}, mB = {0.0f, 0.0f};
      for (int r0 = 0; r0 < tot; r0 += 32) {
        const int r = r0 + lane;
        const uint32_t h = r < tot ? static_cast<uint32_t>(Us[r] >> 32) : 0xffffffffu;
        const bool inB = r < tot && h <= hk;
        const ff w = inB ? wx[r] : ff{0.0f, 0.0f};
        if (r < tot && h == hk) {
          g0 = min(g0, r);
          g1 = max(g1, r);
        }
        mB = ff_add(mB, w);
        if (h < hk) mA = ff_add(mA, w);
        if (__ballot_sync(FULL, r < tot && h > hk)) break;
      }
      mA = warp_sum_ff(mA);
      mB = warp_sum_ff(mB);
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        g0 = min(g0, __shfl_xor_sync(FULL, g0, o));
        g1 = max(g1, __shfl_xor_sync(FULL, g1, o));
      }
      const ff dA = ff_sub(Tt, mA), dB = ff_sub(mB, Tt);
      // certified; or the top-p mass lies within 1e-6 Z of the group's
      // boundary whatever the rounding (a boundary case: any consistent
      // choice is a valid reading), and the walk's own choice stands
      ok = ((dA.hi > slack && dB.hi > slack) || __fmul_rn(2.0f, slack) < __fmul_rn(Z.hi, 1e-6f)) ? 1 : 0;
      if (lane == 0 && ok) {
        LRes *out = &sh.lr[s];
        out->m = M;
        out->tau = key_val(Us[g0]);
        out->Zhi = mB.hi;
        out->Zlo = mB.lo;
        out->zerr = 0.0f;
        out->n = g1 + 1;
        out->exact = 1;
      }
    }
    if (lane == 0) sh.lr[s].ok = ok;
#ifdef SV_PHASE_PROFILE
    if (lane == 0 && !ok) atomicAdd(&sv_strip_cycles[59], 1ull);
#endif
  }
  __syncthreads();
}

// The walk of an extension's band.  The side's list holds Us[0..nkeep) (the
// logits >= Theta, in any order) and Us[nkeep..tot) (the band below Theta,
// in any order), and every logit down to the band's lower edge is present.
// The band is sorted (descending) in the scratch keys and copied back; the
// masses are float-float: A (the logits >= Theta) by a block sum, the
// band's prefix sums by a block scan in sorted order (thread t holds a
// contiguous chunk); the first band entry where A plus the prefix reaches
// top_p Z gives the crossing group, certified as in ext_sort_walk.  Writes
// sh.lr[s] (ok = 0 when the band does not reach top_p Z, or A alone does, or
// the walk is within the error bound).  Whole CTA; side s = threads
// [128 s, 128 s + 128) works when go.  keys: [UCAP] u64 scratch of the side.
__device__ __noinline__ void ext_band_walk(const SP &S, SpShared &sh, int s, bool go, int nkeep,
                                           int tot, float M, uint64_t *Us, uint64_t *keys) {
  const int tid = threadIdx.x, lt = tid & 127, lane = tid & 31, w4 = (tid >> 5) & 3;
  const float ih = S.k.invT_hi, il = S.k.invT_lo, top_p = S.k.top_p;
  const int nb = go ? tot - nkeep : 0;
  int N = 32;
  while (N < nb && N < SP_TOPP_UCAP) N <<= 1;
  if (go) {
    for (int j = lt; j < N; j += 128) keys[j] = j < nb ? Us[nkeep + j] : ~0ull;
    if (lt == 0) {
      sh.xj[s][0] = INT_MAX;
      sh.xj[s][1] = INT_MAX;
      sh.xj[s][2] = -1;
    }
  }
  __syncthreads();
  if (go) group_bitonic(keys, N, lt, 128, 1 + s);
  __syncthreads();
  // A, and the band chunk sums
  ff a = {0.0f, 0.0f}, loc = {0.0f, 0.0f};
  const int q = (nb + 127) / 128;
  const int j0 = min(nb, lt * q), j1 = min(nb, j0 + q);
  if (go) {
    for (int j = lt; j < nkeep; j += 128) a = ff_add(a, wff_c(ih, il, key_val(Us[j]), M));
    for (int j = j0; j < j1; ++j) loc = ff_add(loc, wff_c(ih, il, key_val(keys[j]), M));
  }
  a = warp_sum_ff(a);
  const ff incl = warp_scan_ff(loc);
  ff ex = shfl_up_ff(incl, 1);
  if (lane == 0) ex = ff{0.0f, 0.0f};
  if (go && lane == 31) sh.xs[s][w4] = incl;
  if (go && lane == 0) sh.xa[s][w4] = a;
  __syncthreads();
  ff A = {0.0f, 0.0f}, run = {0.0f, 0.0f}, Tt = {0.0f, 0.0f}, Z = {0.0f, 0.0f};
  float slack = 0.0f;
  if (go) {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      A = ff_add(A, sh.xa[s][w]);
      if (w < w4) run = ff_add(run, sh.xs[s][w]);
    }
    run = ff_add(A, ff_add(run, ex));  // the mass before this thread's chunk
    Z = ff_add(ff{sh.tp[s].Zt_hi, sh.tp[s].Zt_lo}, fix_to_ff(sh.tp[s].slist));
    const float EZ = __fmaf_rn(Z.hi, 1e-12f, __fadd_rn(sh.tp[s].Et, sh.tp[s].El));
    Tt = ff_mul_f(Z, top_p);
    slack = __fmaf_rn(top_p, EZ, __fmul_rn(Z.hi, 1e-12f));
    // the crossing: the first entry whose cumulative mass reaches top_p Z
    ff r = run;
    for (int j = j0; j < j1; ++j) {
      const ff nr = ff_add(r, wff_c(ih, il, key_val(keys[j]), M));
      if (ff_lt(r, Tt) && !ff_lt(nr, Tt)) atomicMin(&sh.xj[s][0], j);
      r = nr;
    }
  }
  __syncthreads();
  const int cross = go ? sh.xj[s][0] : INT_MAX;
  const bool found = go && cross < nb;
  // the crossing group (equal values are contiguous in the sorted band), and
  // the sorted band back into the list
  if (found) {
    const uint32_t hk = static_cast<uint32_t>(keys[cross] >> 32);
    for (int j = j0; j < j1; ++j)
      if (static_cast<uint32_t>(keys[j] >> 32) == hk) {
        atomicMin(&sh.xj[s][1], j);
        atomicMax(&sh.xj[s][2], j);
      }
  }
  if (go)
    for (int j = lt; j < nb; j += 128) Us[nkeep + j] = keys[j];
  __syncthreads();
  // the masses above the group (mA) and through it (mB), by the chunks' owners
  if (found) {
    const int g0 = sh.xj[s][1], g1 = sh.xj[s][2];
    ff r = run;
    for (int j = j0; j < j1; ++j) {
      if (j == g0) sh.xm[s][0] = r;
      r = ff_add(r, wff_c(ih, il, key_val(keys[j]), M));
      if (j == g1) sh.xm[s][1] = r;
    }
  }
  __syncthreads();
  if (go && lt == 0) {
    int ok = 0;
    if (found) {
      const int g0 = sh.xj[s][1], g1 = sh.xj[s][2];
      const ff mA = sh.xm[s][0], mB = sh.xm[s][1];
      const ff dA = ff_sub(Tt, mA), dB = ff_sub(mB, Tt);
      // certified; or the top-p mass lies within 1e-6 Z of the group's
      // boundary whatever the rounding (a boundary case: any consistent
      // choice is a valid reading), and the walk's own choice stands
      ok = ((dA.hi > slack && dB.hi > slack) || __fmul_rn(2.0f, slack) < __fmul_rn(Z.hi, 1e-6f))
               ? 1
               : 0;
      if (ok) {
        LRes *out = &sh.lr[s];
        out->m = M;
        out->tau = key_val(keys[g0]);
        out->Zhi = mB.hi;
        out->Zlo = mB.lo;
        out->zerr = 0.0f;
        out->n = nkeep + g1 + 1;
        out->exact = 1;
      }
    }
    sh.lr[s].ok = ok;
#ifdef SV_PHASE_PROFILE
    if (!ok) atomicAdd(&sv_strip_cycles[59], 1ull);
#endif
  }
  __syncthreads();
}

// Top-p alone, when the candidates were complete (no overflow) but the
// logits >= Theta did not reach top_p Z: extend the list downwards (whole
// CTA; side s handles tensor s when need0 / need1).  The normaliser Z and
// the exact mass A of the logits >= Theta are known from the list phase.
// The list is compacted to the logits >= Theta; one pass over the strip row
// counts the logits below Theta in depth bins (1/16 of a log2 unit below
// Theta: the weights of bin b lie within w(Theta) [2^{-(b+1)/16}, 2^{-b/16}]);
// the lower bounds of the bin masses give the first bin b_hi past which the
// cumulative mass surely
// exceeds top_p Z; a second pass appends every logit below Theta of the bins
// up to b_hi; the list is sorted and walked in float-float against top_p Z.
// Writes sh.lr[s] (ok = 0 when the list would exceed SP_TOPP_UCAP or the
// walk is within the error bound) and leaves the kept list, sorted, in U.
template <typename E>
__device__ __noinline__ void topp_extend(const SP &S, SpShared &sh, int T, int b, int i,
                                         int need0, int need1, const float *Mx, uint64_t *U,
                                         uint32_t *hc, ff *wx0, ff *wx1) {
  const int tid = threadIdx.x, s = tid >> 7, lt = tid & 127, lane = tid & 31,
            w4 = (tid >> 5) & 3;
  bool act = s < T && (s == 0 ? need0 : need1);
  const float M = Mx[s < T ? s : 0];
  const int V = S.k.V, C = S.C;
  const float c2 = S.k.c2, top_p = S.k.top_p;
  uint64_t *Us = U + s * SP_TOPP_UCAP;
  uint32_t *cnt = hc + s * 256;
  ff *wx = s == 0 ? wx0 : wx1;  // [UCAP] float-float weights of the side
  const float Theta = sh.tp[s].theta;
  SP_MARK_START(t_ex_);
  int n = 0, nmax = 0;
  for (int t2 = 0; t2 < T; ++t2) {
    int m2 = 0;
    for (int q = 0; q < C; ++q) m2 += static_cast<int>(sh.hdr[t2][q].x & 0xffffffu);
    if (t2 == s) n = m2;
    nmax = max(nmax, m2);
  }
  nmax = min(nmax, SP_TOPP_UCAP);
  cnt[lt] = 0u;
  cnt[lt + 128] = 0u;
  if (lt == 0) {
    sh.tp[s].ok = 0;
    sh.gc[s][0] = 0;
  }
  // compact the list to the logits >= Theta (stable, in place)
  {
    const uint32_t kmax = ~fkey(canon(Theta));
    int run = 0;
    for (int base = 0; base < nmax; base += 128) {
      const int j = base + lt;
      const uint64_t key = (act && j < n) ? Us[j] : ~0ull;
      const bool pred = act && j < n && static_cast<uint32_t>(key >> 32) <= kmax;
      const uint32_t bal = __ballot_sync(FULL, pred);
      if (lane == 0) sh.gc[s][w4] = __popc(bal);
      __syncthreads();
      int wb = 0, tot = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int x = sh.gc[s][q];
        wb += q < w4 ? x : 0;
        tot += x;
      }
      if (pred) Us[run + wb + __popc(bal & ((1u << lane) - 1u))] = key;
      run += tot;
      __syncthreads();
    }
    if (lt == 0) sh.tp[s].nkeep = run;  // the logits >= Theta
  }
  if (lt == 0) sh.gc[s][0] = 0;
  __syncthreads();
  SP_MARK(17, t_ex_);  // extension: compaction
  // First attempt: the band of kExtBand bins just below Theta, where the
  // crossing usually lies.  One pass over the strip row appends the band's
  // logits (few: one shared atomic each) after the kept ones, and the band
  // is sorted and walked when the list fits.  The list then holds every
  // logit down to the band's lower edge (the depth is monotone in the
  // logit), so a crossing found in it is the row's.  When one tensor alone
  // needs it, every thread of the CTA reads its row.
  {
    const bool single = (need0 != 0) != (need1 != 0);
    const int ps = single ? (need0 ? 0 : 1) : s;
    const bool pact = (single || act) && ps < T;
    const int pt = single ? tid : lt, pn = single ? SP_NT : 128;
    const float Thp = sh.tp[ps < T ? ps : 0].theta;
    uint64_t *Up = U + ps * SP_TOPP_UCAP;
    const int basep = pact ? sh.tp[ps].nkeep : 0;
    if (pact) {
      rescan_row<E>(strip_row<E>(S.k, b, i, ps), V, pt, pn, [&](float z, int j) {
        if (z < Thp && z > -INFINITY && band_depth(Thp, z, c2) < kExtBand) {
          const int pos = basep + atomicAdd(&sh.gc[ps][0], 1);
          if (pos < SP_TOPP_UCAP) Up[pos] = cand_key(z, j);
        }
      });
    }
    __syncthreads();
    const int totb = act ? sh.tp[s].nkeep + sh.gc[s][0] : 0;
    ext_band_walk(S, sh, s, act && totb <= SP_TOPP_UCAP, act ? sh.tp[s].nkeep : 0, totb, M, Us,
                  reinterpret_cast<uint64_t *>(wx));
  }
  SP_MARK(17, t_ex_);  // extension: band pass + walk (with the compaction)
  // the sides whose band missed the crossing (or overflowed the list) go on
  // to the depth histogram
  need0 = need0 && !sh.lr[0].ok;
  need1 = need1 && T > 1 && !sh.lr[1].ok;
  if (!need0 && !need1) return;  // uniform: both flags are in shared memory
  act = s < T && (s == 0 ? need0 : need1);
  if (lt == 0) sh.gc[s][0] = 0;
  __syncthreads();
  // the passes over the strip: when one tensor alone needs them, every
  // thread of the CTA works on it (twice the loads in flight)
  const bool single = (need0 != 0) != (need1 != 0);
  const int ps = single ? (need0 ? 0 : 1) : s;
  const bool pact = single || act;
  const int pt = single ? tid : lt, pn = single ? SP_NT : 128;
  const E *gp = strip_row<E>(S.k, b, i, ps < T ? ps : 0);
  const float Thp = sh.tp[ps].theta;
  uint32_t *cntp = hc + ps * 256;
  uint64_t *Up = U + ps * SP_TOPP_UCAP;
  // pass 1: depth bins below Theta (1/16 of a log2 unit each; bin 255 holds
  // the rest) of the logits below Theta
  if (pact) {
    rescan_row<E>(gp, V, pt, pn, [&](float z, int) {
      if (z < Thp && z > -INFINITY) {
        // the deepest bin is neither bounded nor collected: not counted
        const float d = __fmul_rn(__fmul_rn(__fsub_rn(Thp, z), c2), 16.0f);
        if (d < 255.0f) atomicAdd(&cntp[static_cast<int>(d)], 1u);
      }
    });
  }
  __syncthreads();
  if (act && w4 == 0) {
    const ff Z = ff_add(ff{sh.tp[s].Zt_hi, sh.tp[s].Zt_lo}, fix_to_ff(sh.tp[s].slist));
    const float EZ = __fmaf_rn(Z.hi, 1e-12f, __fadd_rn(sh.tp[s].Et, sh.tp[s].El));
    // a lower bound of A (the fixed-point sums are exact; the weights' error)
    const float A = __fsub_rn(__fmul_rn(__ull2float_rd(sh.tp[s].amass), kFixInv), sh.tp[s].El);
    const float need = __fmaf_rn(top_p, __fadd_rn(Z.hi, EZ), __fmul_rn(Z.hi, 1e-6f));
    // lower bounds of the bins' masses: a weight of bin b is at least
    // w(Theta) 2^{-(b+1)/16} (the depth's rounding widens each bin a little)
    const float wth = __fmul_rn(ex2_approx(__fmul_rn(__fsub_rn(Theta, M), c2)), 0.9999f);
    float c8[8], loc = 0.0f;
    uint32_t n8[8], nloc = 0u;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int bq = lane * 8 + q;
      n8[q] = cnt[bq];
      nloc += n8[q];
      c8[q] = bq < 255 ? __fmul_rn(static_cast<float>(n8[q]),
                                   __fmul_rn(exp2f(-static_cast<float>(bq + 1) * 0.0625f), wth))
                       : 0.0f;
      loc = __fadd_rn(loc, c8[q]);
    }
    const float incl = __fadd_rn(A, warp_scan_f(loc));
    const float excl = __fsub_rn(incl, loc);
    uint32_t nincl = nloc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t u = __shfl_up_sync(FULL, nincl, o);
      if (lane >= o) nincl += u;
    }
    const bool mine = excl < need && need <= incl;
    const uint32_t own = __ballot_sync(FULL, mine);
    int bhi = -1;
    uint32_t nnew = 0u;
    if (mine) {
      float before = excl;
      uint32_t nb = nincl - nloc;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (bhi < 0) {
          before = __fadd_rn(before, c8[q]);
          nb += n8[q];
          if (before >= need) {
            bhi = lane * 8 + q;
            nnew = nb;
          }
        }
      }
    }
    if (own) {
      const int L = __ffs(own) - 1;
      bhi = __shfl_sync(FULL, bhi, L);
      nnew = __shfl_sync(FULL, nnew, L);
    }
    if (lane == 0) {
      const int tot = sh.tp[s].nkeep + static_cast<int>(nnew);
      sh.tp[s].ok = (own != 0u && tot <= SP_TOPP_UCAP) ? 1 : 0;
#ifdef SV_PHASE_PROFILE
      if (own == 0u) atomicAdd(&sv_strip_cycles[58], 1ull);
      if (own != 0u && tot > SP_TOPP_UCAP) atomicAdd(&sv_strip_cycles[60], 1ull);
      if (A >= need) atomicAdd(&sv_strip_cycles[61], 1ull);
#endif
      sh.tp[s].bstar = bhi;
      sh.tp[s].nb = tot;
    }
  }
  __syncthreads();
  SP_MARK(18, t_ex_);  // extension: pass 1 + bins
  const bool go = act && sh.tp[s].ok;
  // (an idle side's fields are not set: use none of them)
  const int tot = go ? sh.tp[s].nb : 0;
  // pass 2: append the logits below Theta of the bins up to b_hi
  {
    const bool gop = pact && ps < T && sh.tp[ps].ok;
    const int bhip = gop ? sh.tp[ps].bstar : -1, basep = gop ? sh.tp[ps].nkeep : 0;
    if (gop) {
      rescan_row<E>(gp, V, pt, pn, [&](float z, int j) {
        if (z < Thp && z > -INFINITY) {
          const float d = __fmul_rn(__fmul_rn(__fsub_rn(Thp, z), c2), 16.0f);
          if ((d < 255.0f ? static_cast<int>(d) : 255) <= bhip) {
            const int pos = basep + atomicAdd(&sh.gc[ps][0], 1);
            if (pos < SP_TOPP_UCAP) Up[pos] = cand_key(z, j);
          }
        }
      });
    }
  }
  __syncthreads();
  SP_MARK(19, t_ex_);  // extension: pass 2
  ext_sort_walk(S, sh, s, go, tot, M, Us, wx);
  SP_MARK(12, t_ex_);  // extension: sort + walk
}

// Exact top-p of a tensor whose candidates could not hold its nucleus (top-p
// alone; whole CTA, side s = threads [128 s, 128 s + 128) handles tensor s
// when need0 / need1): one pass over the strip row gives Z (the weights
// above 2^-16 in float-float, the rest in compensated single precision with
// its error bound) and a mass histogram of the weights in depth bins that
// locates a bin b* past the top-p crossing and a bin b_lo before it.  A
// second pass collects every element of the bins up to b* (all values above
// b*'s lower edge), which are sorted and walked in float-float against
// top_p Z, and the kept list is left, sorted, in U (ok = 1).  When that
// region exceeds SP_TOPP_UCAP but the bins b_lo .. b* do not, the pass sums
// the weights of the bins before b_lo in float-float instead (all of them
// lie before the crossing) and collects the window b_lo .. b* alone; the
// walk starts from that sum, and the result is tau and Z without a list
// (ok = 2: the draw runs over the strip).  ok = 0 when the window exceeds
// SP_TOPP_UCAP too, the crossing lies in the deepest bin, or the walk finds
// no crossing: the caller then takes the slice-wide path.
template <typename E>
__device__ __noinline__ void topp_rescan(const SP &S, SpShared &sh, int T, int b, int i,
                                         int need0, int need1, const float *Mx, uint64_t *U,
                                         uint64_t *hm, uint32_t *hc) {
  const int tid = threadIdx.x, s = tid >> 7, lt = tid & 127, lane = tid & 31,
            w4 = (tid >> 5) & 3;
  const bool act = s < T && (s == 0 ? need0 : need1);
  const E *g = strip_row<E>(S.k, b, i, s < T ? s : 0);
  const float M = Mx[s < T ? s : 0];
  // launch parameters in registers
  const int V = S.k.V;
  const float c2 = S.k.c2, ih = S.k.invT_hi, il = S.k.invT_lo, top_p = S.k.top_p;
  uint64_t *Us = U + s * SP_TOPP_UCAP;
  uint64_t *hms = hm + s * 256;
  uint32_t *hcs = hc + s * 256;
  hms[lt] = 0ull;
  hms[lt + 128] = 0ull;
  hcs[lt] = 0u;
  hcs[lt + 128] = 0u;
  if (lt == 0) {
    sh.tp[s].ok = 0;
    sh.gc[s][0] = 0;
  }
  __syncthreads();
  // pass 1: the total weight Z (compensated per-thread sums, then a fixed
  // order) with the weights' error bound, and bin masses that only locate
  // the crossing bin: in bin b a weight times 2^{b/8} lies in (0.91, 1], kept
  // as round(2^12 w 2^{b/8}) in 32-bit integer sums (order-independent; a
  // relative precision of 2^-13); the deepest bin is not summed
  float err = 0.0f, zs = 0.0f, zc = 0.0f;
  ff zx = {0.0f, 0.0f};  // float-float sum of the weights above 2^-16
  // the side's 2 KB of bin space: [256] u32 scaled masses, then [256] 2^{b/8}
  uint32_t *hus = reinterpret_cast<uint32_t *>(hms);
  float *bsc = reinterpret_cast<float *>(hms) + 256;
  bsc[lt] = exp2f(static_cast<float>(lt) * 0.125f);
  bsc[lt + 128] = exp2f(static_cast<float>(lt + 128) * 0.125f);
  __syncthreads();
  if (act) {
    rescan_row<E>(g, V, lt, 128, [&](float z, int) {
      float w, y;
      int bin;
      rescan_elem(c2, z, M, w, y, bin);
      if (w > 0.0f) {
        if (y > -16.0f) {
          // weights above 2^-16 in float-float: the normaliser's error then
          // comes from the small weights alone
          zx = ff_add(zx, wff_c(ih, il, z, M));
        } else {
          const float t = __fsub_rn(w, zc), s2 = __fadd_rn(zs, t);
          zc = __fsub_rn(__fsub_rn(s2, zs), t);
          zs = s2;
          err = __fmaf_rn(w, __fmaf_rn(fabsf(y), kExpErr1, kExpErr0), err);
        }
        if (bin < 255) {
          atomicAdd(&hus[bin], __float2uint_rn(__fmul_rn(__fmul_rn(w, bsc[bin]), 4096.0f)));
          atomicAdd(&hcs[bin], 1u);
        }
      }
    });
  }
  const ff zsum = warp_sum_ff(quick_two_sum(zs, -zc));
  const ff zxs = warp_sum_ff(zx);
  err = warp_sum_f(err);
  if (lane == 0) {
    sh.ge[s][w4] = err;
    reinterpret_cast<float *>(&sh.gs[s][w4])[0] = zsum.hi;
    reinterpret_cast<float *>(&sh.gs[s][w4])[1] = zsum.lo;
    reinterpret_cast<float *>(&sh.ga[s][w4])[0] = zxs.hi;
    reinterpret_cast<float *>(&sh.ga[s][w4])[1] = zxs.lo;
  }
  __syncthreads();
  if (act && w4 == 0) {
    float e = 0.0f;
    ff Zs = {0.0f, 0.0f}, Zx = {0.0f, 0.0f};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      e = __fadd_rn(e, sh.ge[s][q]);
      const float *zq = reinterpret_cast<const float *>(&sh.gs[s][q]);
      Zs = ff_add(Zs, ff{zq[0], zq[1]});
      const float *xq = reinterpret_cast<const float *>(&sh.ga[s][q]);
      Zx = ff_add(Zx, ff{xq[0], xq[1]});
    }
    // the small weights' compensated sums: two units; weights flushed below
    // 2^-126; the float-float sums' rounding
    e = __fadd_rn(__fmaf_rn(Zs.hi, 2.4e-7f, e), static_cast<float>(V) * 1.2e-38f);
    const ff Z = ff_add(Zx, Zs);
    e = __fmaf_rn(Z.hi, 1e-12f, e);
    // the crossing bin, located with a margin over the bin masses' rounding
    // (2^-13 relative, and at most 256 float additions): the first bin where
    // the cumulative mass reaches top_p Z + 2^-10 Z
    const float tgt = __fmaf_rn(Z.hi, top_p, __fmul_rn(Z.hi, 9.765625e-4f));
    // and the first bin b_lo where it reaches top_p Z - 2^-10 Z: the bins
    // before it lie wholly before the crossing (0 when none qualifies)
    const float tgl = __fmaf_rn(Z.hi, top_p, -__fmul_rn(Z.hi, 9.765625e-4f));
    float c8[8], loc = 0.0f;
    uint32_t n8[8], nloc = 0u;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int bq = lane * 8 + q;
      c8[q] = __fdiv_rn(__fmul_rn(static_cast<float>(hus[bq]), 2.44140625e-4f), bsc[bq]);
      n8[q] = hcs[bq];
      loc = __fadd_rn(loc, c8[q]);
      nloc += n8[q];
    }
    const float incl = warp_scan_f(loc);
    const float excl = __fsub_rn(incl, loc);
    uint32_t nincl = nloc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t u = __shfl_up_sync(FULL, nincl, o);
      if (lane >= o) nincl += u;
    }
    const bool mine = excl < tgt && tgt <= incl;
    const uint32_t own = __ballot_sync(FULL, mine);
    int bstar = -1;
    uint32_t nreg = 0u;  // elements of the bins up to b*
    if (mine) {
      float before = excl;
      uint32_t nb = nincl - nloc;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (bstar < 0) {
          before = __fadd_rn(before, c8[q]);
          nb += n8[q];
          if (before >= tgt) {
            bstar = lane * 8 + q;
            nreg = nb;
          }
        }
      }
    }
    if (own) {
      const int L = __ffs(own) - 1;
      bstar = __shfl_sync(FULL, bstar, L);
      nreg = __shfl_sync(FULL, nreg, L);
    }
    const bool mlo = excl < tgl && tgl <= incl;
    const uint32_t olo = __ballot_sync(FULL, mlo);
    int blo = -1;
    uint32_t nlow = 0u;  // elements of the bins before b_lo
    if (mlo) {
      float before = excl;
      uint32_t nb = nincl - nloc;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (blo < 0) {
          before = __fadd_rn(before, c8[q]);
          if (before >= tgl) {
            blo = lane * 8 + q;
            nlow = nb;
          }
          nb += n8[q];
        }
      }
    }
    if (olo) {
      const int L = __ffs(olo) - 1;
      blo = __shfl_sync(FULL, blo, L);
      nlow = __shfl_sync(FULL, nlow, L);
    }
    if (blo < 0 || blo > bstar) {  // (rounding) the window from bin 0
      blo = 0;
      nlow = 0u;
    }
    if (lane == 0) {
      const uint32_t cap = static_cast<uint32_t>(SP_TOPP_UCAP);
      int mode = 0;
      if (own != 0u && bstar >= 0 && bstar < 255) mode = nreg <= cap ? 1 : (nreg - nlow <= cap ? 2 : 0);
      sh.tp[s].ok = mode;
      sh.tp[s].bstar = bstar;
      sh.tp[s].nb = static_cast<int>(mode == 2 ? nreg - nlow : nreg);
      sh.tp[s].blo = mode == 2 ? blo : 0;
      sh.tp[s].Zt_hi = Z.hi;
      sh.tp[s].Zt_lo = Z.lo;
      sh.tp[s].Et = e;
    }
  }
  __syncthreads();
  const int mode = act ? sh.tp[s].ok : 0;  // uniform over the side's warps
  const bool go = mode != 0;
  const int bstar = go ? sh.tp[s].bstar : -1, nreg = go ? sh.tp[s].nb : 0;
  const int blo = mode == 2 ? sh.tp[s].blo : 0;
  ff above = {0.0f, 0.0f};  // window mode: the weights of the bins before b_lo
  if (go) {
    rescan_row<E>(g, V, lt, 128, [&](float z, int j) {
      float w, y;
      int bin;
      rescan_elem(c2, z, M, w, y, bin);
      if (w > 0.0f && bin <= bstar) {
        if (bin < blo) {
          above = ff_add(above, wff_c(ih, il, z, M));
        } else {
          const int pos = atomicAdd(&sh.gc[s][0], 1);
          if (pos < SP_TOPP_UCAP) Us[pos] = cand_key(z, j);
        }
      }
    });
  }
  if (mode == 2) {
    above = warp_sum_ff(above);
    if (lane == 0) {
      reinterpret_cast<float *>(&sh.ga[s][w4])[0] = above.hi;
      reinterpret_cast<float *>(&sh.ga[s][w4])[1] = above.lo;
    }
  }
  __syncthreads();
  if (go)
    for (int j = nreg + lt; j < SP_TOPP_UCAP; j += 128) Us[j] = ~0ull;
  __syncthreads();
  if (go) group_bitonic(Us, SP_TOPP_UCAP, lt, 128, 1 + s);
  __syncthreads();
  if (go && w4 == 0) {
    const ff Z = {sh.tp[s].Zt_hi, sh.tp[s].Zt_lo};
    const float Eb = __fmaf_rn(Z.hi, 1e-12f, sh.tp[s].Et);
    const ff Tt = ff_mul_f(Z, top_p);
    // window mode: the walk starts from the mass before b_lo, a float-float
    // sum of up to V / 128 terms per thread (relative error under 1.1e-14
    // per addition)
    ff A = {0.0f, 0.0f};
    if (mode == 2) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float *aq = reinterpret_cast<const float *>(&sh.ga[s][q]);
        A = ff_add(A, ff{aq[0], aq[1]});
      }
    }
    const float slack = __fmaf_rn(
        A.hi, __fmul_rn(static_cast<float>(V / 128 + 32), 1.1e-14f),
        __fmaf_rn(top_p, Eb, __fmul_rn(Z.hi, 1e-12f)));
    ff carry = A;
    int cross = -1;
    for (int r0 = 0; r0 < nreg && cross < 0; r0 += 32) {
      const int r = r0 + lane;
      const ff w = r < nreg ? wff_c(ih, il, key_val(Us[r]), M) : ff{0.0f, 0.0f};
      const ff incl = ff_add(carry, warp_scan_ff(w));
      ff bef = shfl_up_ff(incl, 1);
      if (lane == 0) bef = carry;
      const uint32_t bal = __ballot_sync(FULL, r < nreg && ff_lt(bef, Tt) && !ff_lt(incl, Tt));
      if (bal) cross = r0 + __ffs(bal) - 1;
      carry = shfl_ff(incl, 31);
    }
    int ok = 0;
    if (cross >= 0) {
      const uint32_t hk = static_cast<uint32_t>(Us[cross] >> 32);
      int g0 = nreg, g1 = -1;
      ff mA = {0.0f, 0.0f}, mB = {0.0f, 0.0f};
      for (int r0 = 0; r0 < nreg; r0 += 32) {
        const int r = r0 + lane;
        const uint32_t h = r < nreg ? static_cast<uint32_t>(Us[r] >> 32) : 0xffffffffu;
        const bool inB = r < nreg && h <= hk;
        const ff w = inB ? wff_c(ih, il, key_val(Us[r]), M) : ff{0.0f, 0.0f};
        if (r < nreg && h == hk) {
          g0 = min(g0, r);
          g1 = max(g1, r);
        }
        mB = ff_add(mB, w);
        if (h < hk) mA = ff_add(mA, w);
        if (__ballot_sync(FULL, r < nreg && h > hk)) break;
      }
      mA = ff_add(A, warp_sum_ff(mA));
      mB = ff_add(A, warp_sum_ff(mB));
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        g0 = min(g0, __shfl_xor_sync(FULL, g0, o));
        g1 = max(g1, __shfl_xor_sync(FULL, g1, o));
      }
      const ff dA = ff_sub(Tt, mA), dB = ff_sub(mB, Tt);
      // certified; or the top-p mass lies within 1e-6 Z of the group's
      // boundary whatever the rounding (a boundary case: any consistent
      // choice is a valid reading), and the walk's own choice stands
      ok = ((dA.hi > slack && dB.hi > slack) || __fmul_rn(2.0f, slack) < __fmul_rn(Z.hi, 1e-6f)) ? 1 : 0;
      if (lane == 0 && ok) {
        LRes *out = &sh.lr[s];
        out->m = M;
        out->tau = key_val(Us[g0]);
        out->Zhi = mB.hi;
        out->Zlo = mB.lo;
        out->zerr = 0.0f;
        out->n = mode == 2 ? 0 : g1 + 1;
        out->exact = 1;
      }
    }
    if (lane == 0) sh.lr[s].ok = ok ? mode : 0;
  }
  __syncthreads();
}

__device__ void strip_bad_row(const SP &S, int b) {
  const KP &P = S.k;
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

// Outputs of sequence b: positions 0..r are decided, r is the first ending.
__device__ void strip_finalize(const SP &S, int b, int r) {
  const KP &P = S.k;
  const uint4 *d = S.dec + 2 * static_cast<int64_t>(b) * S.NP;
  int status = 0;
  for (int j = 0; j <= r; ++j) status |= static_cast<int>(__ldcg(d + 2 * j).x);
  const uint4 d0 = __ldcg(d + 2 * r), d1 = __ldcg(d + 2 * r + 1);
  const bool err = (status & ST_ERROR) != 0;
  if (P.acc) P.acc[b] = err ? 0 : r;
  P.next[b] = err ? -1 : static_cast<int>(d0.y);
  if (P.st_dbg) P.st_dbg[b] = status;
  if (P.res_dbg) P.res_dbg[b] = err ? 0.0f : __uint_as_float(d1.x);
  if (P.p_dbg || P.q_dbg) {
    const float nan = __int_as_float(0x7fc00000);
    for (int j = 0; j < P.gm; ++j) {
      float pv = nan, qv = nan;
      if (j <= r) {
        const uint4 e0 = __ldcg(d + 2 * j), e1 = __ldcg(d + 2 * j + 1);
        if (e1.y) {
          pv = __uint_as_float(e0.z);
          qv = __uint_as_float(e0.w);
        }
      }
      if (P.p_dbg) P.p_dbg[static_cast<int64_t>(b) * P.gm + j] = pv;
      if (P.q_dbg) P.q_dbg[static_cast<int64_t>(b) * P.gm + j] = qv;
    }
  }
  if ((status & ST_TIMEOUT) && P.diag) atomicAdd(P.diag + 2, 1u);
}

// Four warps (128 threads) gather the candidates >= bound of the C pieces of
// tensor tt into U, unordered (shared-memory count sh.cnt[tt], which may
// exceed SP_UCAP: overflow).
__device__ __forceinline__ void group_gather(const SP &S, SpShared &sh, int tt, int64_t hb,
                                             float bound, uint64_t *U) {
  const int t = threadIdx.x & 127;
  int offs[SP_MAXC + 1];
  offs[0] = 0;
#pragma unroll
  for (int q = 0; q < SP_MAXC; ++q)
    offs[q + 1] = offs[q] + (q < S.C ? static_cast<int>(sh.hdr[tt][q].x & 0xffffffu) : 0);
  const int total = offs[SP_MAXC];
  const uint32_t kmax = ~fkey(canon(bound));  // key >> 32 <= kmax  <=>  value >= bound
  for (int j0 = 0; j0 < total; j0 += 128 * 4) {
    uint64_t kv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = j0 + u * 128 + t;
      kv[u] = ~0ull;
      if (j < total) {
        int c = 0;
#pragma unroll
        for (int q = 1; q < SP_MAXC; ++q)
          if (j >= offs[q] && q < S.C) c = q;
        kv[u] = __ldcg(S.cand + (hb + tt * S.C + c) * S.capc + (j - offs[c]));
      }
    }
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool pass = kv[u] != ~0ull && static_cast<uint32_t>(kv[u] >> 32) <= kmax;
      const uint32_t bal = __ballot_sync(FULL, pass);
      if (bal) {  // one shared-memory atomic per warp and batch
        int base = 0;
        if (lane == __ffs(bal) - 1) base = atomicAdd(&sh.cnt[tt], __popc(bal));
        base = __shfl_sync(FULL, base, __ffs(bal) - 1);
        const int pos = base + __popc(bal & ((1u << lane) - 1u));
        if (pass && pos < SP_UCAP) U[pos] = kv[u];
      }
    }
  }
}

// One warp: from the gathered candidates U[0..n) of tensor tt (every value
// >= bound, every value >= the strip's k-th largest among them), the kept
// top-k set sorted by value (into K) and its filters and normaliser
// (sh.lr[tt]).  Short lists are sorted whole; long ones go through an exact
// selection first.
__device__ __forceinline__ void warp_tensor_list(const SP &S, SpShared &sh, int tt, int n,
                                                 float bound, float hi, uint64_t *U, uint64_t *K,
                                                 uint32_t *hist, bool sorted) {
  const KP &P = S.k;
  const int lane = threadIdx.x & 31;
  LRes *out = &sh.lr[tt];
  if (n > SP_UCAP || n < P.top_k) {
    if (lane == 0) out->ok = 0;
    __syncwarp();
    return;
  }
  int nk;
  if (sorted) {
    // K holds the n entries sorted (value descending): the kept set is the
    // prefix of the values >= the k-th
    const float tk = key_val(K[P.top_k - 1]);
    int c = 0;
    for (int r = lane; r < n; r += 32) c += key_val(K[r]) >= tk ? 1 : 0;
#pragma unroll
    for (int o = 16; o; o >>= 1) c += __shfl_xor_sync(FULL, c, o);
    nk = c;
  } else {
    uint32_t th;
    if (!warp_select_bins(U, n, P.top_k, bound, hi, hist, K, &th, &nk))
      th = warp_select(U, n, P.top_k, hist, &nk);
    if (nk > SP_KCAP) {
      if (lane == 0) out->ok = 0;
      __syncwarp();
      return;
    }
    int w = 0;
    for (int j0 = 0; j0 < n; j0 += 32) {
      const int j = j0 + lane;
      const bool keep = j < n && static_cast<uint32_t>(U[j] >> 32) <= th;
      const uint32_t bal = __ballot_sync(FULL, keep);
      if (keep) K[w + __popc(bal & ((1u << lane) - 1u))] = U[j];
      w += __popc(bal);
    }
    __syncwarp();
    warp_sort(K, nk);
  }
  warp_dist(P, K, nk, out);
}

// A tensor's distribution from its list result.
__device__ __forceinline__ void apply_list(Dist &D, const LRes &R) {
  D.m = R.m;
  D.tau = R.tau;
  if (R.exact)
    set_Zx(D, ff{R.Zhi, R.Zlo});
  else
    set_Zf(D, ff{R.Zhi, R.Zlo}, R.zerr);
  D.list = 1;
  D.n = R.n;
}

// A rescan's cut without a list (ok = 2): the threshold and the exact
// normaliser, the kept set read from the strip.
__device__ __forceinline__ void apply_cut(Dist &D, const LRes &R) {
  D.m = R.m;
  D.tau = R.tau;
  set_Zx(D, ff{R.Zhi, R.Zlo});
  D.list = 0;
  D.n = 0;
}

// The decision at position i of sequence b (whole CTA; the piece data of
// this CTA is no longer needed, its shared memory holds the lists).  It and
// the helpers of its common path are inlined into the kernel: there the
// launch parameters are constant-bank operands, while a called function
// reads them through a generic pointer, one memory load each.  The
// distributions dt and dd reach out-of-line (rare) paths only as copies, so
// they stay in registers.
template <typename E>
__device__ __forceinline__ void strip_decide(const SP &S, SpShared &sh, unsigned char *smem,
                                             int b, int i, int gb) {
  const KP &P = S.k;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  SP_PHASE_START;
  const bool bonus = i == gb;
  const bool two = !P.greedy && !bonus;
  const int T = two ? 2 : 1;
  const int64_t hb = (static_cast<int64_t>(i) * P.B + b) * S.T * S.C;
  for (int j = tid; j < T * S.C; j += SP_NT) {
    sh.hdr[j / S.C][j % S.C] = __ldcg(S.hdr + hb + j);
    if (S.topp) sh.hdr2[j / S.C][j % S.C] = __ldcg(S.hdr2 + hb + j);
  }
  if (tid == 0) sh.cnt[0] = sh.cnt[1] = 0;
  // token, uniforms and the logits of the token: read by the piece ahead
  int x = -1, status = 0;
  float u0 = 0.0f;
  if (!bonus) {
    x = sh.pre_x;
    if (x < 0 || x >= P.V) status |= ST_BAD_TOKEN;
  }
  if (two) {
    u0 = sh.pre[0];
    if (!(u0 >= 0.0f && u0 < 1.0f)) status |= ST_BAD_UNIFORM;
  }
  const float zx = sh.pre[2], wx = sh.pre[3];
  __syncthreads();
  float m[2] = {-INFINITY, -INFINITY}, bnd[2] = {-INFINITY, -INFINITY};
  uint32_t fl[2] = {0u, 0u};
  float amv = -INFINITY;
  int am = INT_MAX;
  for (int tt = 0; tt < T; ++tt) {
    float th = -INFINITY, ph = INFINITY;
    for (int cc = 0; cc < S.C; ++cc) {
      const uint4 h = sh.hdr[tt][cc];
      const float mv = __uint_as_float(h.y);
      fl[tt] |= h.x >> 24;
      m[tt] = fmaxf(m[tt], mv);
      if (P.greedy) {
        if (mv > amv) {  // pieces in index order: the first maximum wins
          amv = mv;
          am = static_cast<int>(h.z);
        }
      } else {
        th = fmaxf(th, __uint_as_float(h.z));
        ph = fminf(ph, __uint_as_float(h.w));
      }
    }
    // both are lower bounds of the strip's k-th largest logit
    bnd[tt] = fmaxf(th, ph);
    if (fl[tt] & F_TIMEOUT) status |= ST_TIMEOUT;
    if (fl[tt] & F_BAD) status |= ST_BAD_LOGIT;
    if (!(fl[tt] & F_FINITE)) status |= ST_NO_FINITE;
  }
  int term = 1, token = -1, tested = 0;
  float pdbg = 0.0f, qdbg = 0.0f, resid = 0.0f;
  float lbeta = 0.0f, lres = 0.0f;  // spec_law: beta and R at the position
  SP_PHASE(5);  // decider: headers
  if (status & ST_ERROR) {
    // the sequence ends here with an error
  } else if (P.greedy) {
    if (!bonus && am == x)
      term = 0;
    else
      token = am;
  } else {
    uint64_t *U = reinterpret_cast<uint64_t *>(smem);  // [2][SP_UCAP]
    uint64_t *K = U + 2 * SP_UCAP;                     // [2][SP_KCAP]
    uint64_t *K2 = K + 2 * SP_KCAP;                    // [SP_KCAP]
    uint32_t *hist = reinterpret_cast<uint32_t *>(K2 + SP_KCAP);  // [2][256]
    float *yb = reinterpret_cast<float *>(hist + 2 * 256);         // [SP_KCAP]
    ff *wb = reinterpret_cast<ff *>(yb + SP_KCAP);                  // [SP_KCAP]
    uint64_t *Kp = K, *Kq = K + SP_KCAP;  // the kept lists of p and q
    const E *gt = strip_row<E>(P, b, i, 0);
    const E *gd = two ? strip_row<E>(P, b, i, 1) : gt;
    const int side = wid >> 2;
    if (S.topp) {
      // top-p alone: U [2][SP_TOPP_UCAP] (the kept lists in place), K2, bin
      // masses and counts, yb, wb, crossing-bin entries
      K2 = U + 2 * SP_TOPP_UCAP;
      uint64_t *hm = K2 + SP_TOPP_UCAP;
      uint32_t *hc = reinterpret_cast<uint32_t *>(hm + 2 * 256);
      yb = reinterpret_cast<float *>(hc + 2 * 256);
      wb = reinterpret_cast<ff *>(yb + SP_TOPP_UCAP);
      uint64_t *bs = reinterpret_cast<uint64_t *>(wb + SP_TOPP_UCAP);
      Kp = U;
      Kq = U + SP_TOPP_UCAP;
      topp_lists(S, sh, T, hb, m, bnd, fl, U, hm, hc, bs);
      SP_PHASE(20);  // decider: top-p lists
      // a complete list whose logits >= Theta missed the nucleus: extend it
      // downwards from the strip
      int need0 = sh.lr[0].ok == 0 && sh.tp[0].amass != ~0ull && sh.tp[0].deficit;
      int need1 = T > 1 && sh.lr[1].ok == 0 && sh.tp[1].amass != ~0ull && sh.tp[1].deficit;
      if (need0 || need1) {
        // scratch for the weights: K2 (side 0) and wb (side 1), free until
        // the draw
        topp_extend<E>(S, sh, T, b, i, need0, need1, m, U, hc, reinterpret_cast<ff *>(K2), wb);
        if (P.diag && tid == 0) atomicAdd(P.diag + 3, 1u);
        SP_PHASE(22);  // decider: top-p extension
      }
      // still missing (an overflowed list, or an extension that failed):
      // rescan those strips whole
      need0 = sh.lr[0].ok == 0;
      need1 = T > 1 && sh.lr[1].ok == 0;
      if (need0 || need1) {
        topp_rescan<E>(S, sh, T, b, i, need0, need1, m, U, hm, hc);
        if (P.diag && tid == 0) atomicAdd(P.diag + 3, 1u);
        SP_PHASE(13);  // decider: top-p rescan
      }
    } else {
      // gather the candidates >= the bound of each tensor into U (unordered):
      // warps 0-3 for p, 4-7 for q
      if (side < T && !(fl[side] & F_OVER)) group_gather(S, sh, side, hb, bnd[side], U + side * SP_UCAP);
      __syncthreads();
      SP_PHASE(14);  // decider: gather
      // short lists: sorted by rank, every thread of the tensor's 128 ranking
      // its entries against all (keys are distinct: the ranks permute 0..n-1)
      const int ns = side < T ? sh.cnt[side] : 0;
      const bool rsort = side < T && !(fl[side] & F_OVER) && ns >= P.top_k && ns <= SP_KCAP;
      if (rsort) {
        const uint64_t *Us = U + side * SP_UCAP;
        uint64_t *Ks = K + side * SP_KCAP;
        for (int j = tid & 127; j < ns; j += 128) {
          const uint64_t kk = Us[j];
          int rank = 0;
#pragma unroll 8
          for (int l = 0; l < ns; ++l) rank += Us[l] < kk ? 1 : 0;
          Ks[rank] = kk;
        }
      }
      __syncthreads();
      SP_PHASE(11);  // decider: gather + rank sort
      if ((wid & 3) == 0 && side < T) {
        if (fl[side] & F_OVER) {
          if (lane == 0) sh.lr[side].ok = 0;
        } else {
          warp_tensor_list(S, sh, side, ns, bnd[side], m[side], U + side * SP_UCAP,
                           K + side * SP_KCAP, hist + side * 256, rsort);
        }
      }
      SP_PHASE(20);  // decider: p list (warp 0)
      __syncthreads();
    }
    SP_PHASE(6);  // decider: kept sets + filters
    Dist dt, dd;
    dist_init(dt, m[0]);
    dist_init(dd, m[1]);
    const int ok0 = sh.lr[0].ok, ok1 = two ? sh.lr[1].ok : 0;
    const bool lt = ok0 == 1, ld = ok1 == 1;
    if (lt) apply_list(dt, sh.lr[0]);
    if (ld) apply_list(dd, sh.lr[1]);
    if (ok0 == 2) apply_cut(dt, sh.lr[0]);
    if (ok1 == 2) apply_cut(dd, sh.lr[1]);
    Blk k;
    k.xch = sh.xch;
    k.gat = sh.gat;
    k.red = sh.red;
    k.scal = sh.scal;
    k.C = 1;
    k.rank = 0;
    k.slot = 0;
    k.nt = SP_NT;
    k.nw = SP_NW;
    // the slice-wide selection for a tensor with neither a list nor a cut
    const bool ft = ok0 == 0, fd = two && ok1 == 0;
    if (ft || fd) {
      // exact selection over the whole strip, read in place
      Dist t0 = dt, t1 = dd;  // copies: dt and dd stay in registers
      if (P.k_on) slice_bisect<E>(P, k, gt, gd, P.V, t0, t1, ft, fd, false);
      if (P.p_on) slice_bisect<E>(P, k, gt, gd, P.V, t0, t1, ft, fd, true);
      slice_Z_exact<E>(P, k, gt, gd, P.V, t0, t1, ft, fd);
      dt = t0;
      dd = t1;
      if (P.diag && tid == 0) atomicAdd(P.diag, 1u);
      SP_PHASE(7);  // decider: slice-wide fallback
    }
    // the draw's inputs, ahead of the acceptance test: warp 1 sorts the kept
    // p-ranks by token index, warps 2-3 read the draft logits of those tokens
    if (lt) {
      if (wid >= 1 && wid <= 3 && !S.topp) {
        if (dt.n <= 128) {
          // the kept p-ranks in token order, by ranking the token indices
          for (int r = tid - 32; r < dt.n; r += 96) {
            const int v = key_idx(Kp[r]);
            int rank = 0;
#pragma unroll 8
            for (int l = 0; l < dt.n; ++l) rank += key_idx(Kp[l]) < v ? 1 : 0;
            K2[rank] = (static_cast<uint64_t>(static_cast<uint32_t>(v)) << 32) |
                       static_cast<uint32_t>(r);
          }
        } else {
          // longer lists (top-p alone): a bitonic sort of (index, rank) pairs
          int N = 256;
          while (N < dt.n && N < SP_KCAP) N <<= 1;
          for (int r = tid - 32; r < N; r += 96)
            K2[r] = r < dt.n ? (static_cast<uint64_t>(static_cast<uint32_t>(key_idx(Kp[r]))) << 32) |
                                   static_cast<uint32_t>(r)
                             : ~0ull;
          named_sync(5, 96);
          group_bitonic(K2, N, tid - 32, 96, 5);
        }
      } else if (two && wid >= 4) {
        for (int r = tid - 128; r < dt.n; r += 128) yb[r] = raw_of(gd[key_idx(Kp[r])]);
      }
    }
    int verdict = 0;
    if (!bonus) {
      // acceptance u < p(x)/q(x): single precision with an error bound, in
      // float-float when u falls within the bound (warp 0)
      if (wid == 0) {
        const bool kp = zx >= dt.tau && zx != -INFINITY;
        const bool kq = wx >= dd.tau && wx != -INFINITY;
        const float yp = __fmul_rn(__fsub_rn(zx, dt.m), P.c2);
        const float yq = __fmul_rn(__fsub_rn(wx, dd.m), P.c2);
        float pf = kp ? __fmul_rn(ex2_approx(yp), dt.rzf) : 0.0f;
        float qf = kq ? __fmul_rn(ex2_approx(yq), dd.rzf) : 0.0f;
        int v;
        if (!kq) {
          v = kp ? 1 : 0;  // the limit of min(1, p/q) as q -> 0
        } else if (!kp) {
          v = 0;
        } else if (u0 == 0.0f) {
          v = 1;
        } else {
          const float d = __fsub_rn(yp, yq);
          const float r = __fmul_rn(ex2_approx(d), __fmul_rn(dd.Z.hi, dt.rzf));
          const float eps = __fadd_rn(
              __fmaf_rn(__fadd_rn(__fadd_rn(fabsf(yp), fabsf(yq)), fabsf(d)), kExpErr1,
                        kExpErr0),
              __fadd_rn(__fadd_rn(dt.zerr, dd.zerr), 1.2e-6f));
          if (r == INFINITY || u0 < __fmul_rn(r, 1.0f - eps))
            v = 1;
          else if (u0 >= __fmul_rn(r, 1.0f + eps) && r > 0.0f)
            v = 0;
          else
            v = 2;
        }
        if (v == 2) {  // exact decision in float-float
          if (!dt.exact) warp_make_exact(P, Kp, dt);
          if (!dd.exact) warp_make_exact(P, Kq, dd);
          const ff ratio = ff_mul(ff_exp(ff_sub(scaled_gap(P, zx, dt.m), scaled_gap(P, wx, dd.m))),
                                  ff_mul(dd.Z, dt.rZ));
          v = ff_lt(ff_make(u0), ratio) ? 1 : 0;
          if (P.diag && lane == 0) atomicAdd(P.diag + 1, 1u);
        }
        if (lane == 0) {
          sh.scal[2] = v;
          sh.scal[3] = kq ? 0 : ST_Q_ZERO;
          sh.pq[0] = pf;
          sh.pq[1] = qf;
        }
      }
      SP_PHASE(21);  // decider: acceptance test (warp 0)
      __syncthreads();
      verdict = sh.scal[2];
      status |= sh.scal[3];
      pdbg = sh.pq[0];
      qdbg = sh.pq[1];
      tested = 1;
    }
    if (bonus) __syncthreads();  // K2 ready
    SP_PHASE(8);  // decider: acceptance
    if (S.law) {
      // spec_law: beta = sum min(p, q) and R = sum max(0, p - q), over p's
      // kept set (min and the positive part vanish off it), from p's kept
      // list and the draft logits of its tokens; without the list, R by the
      // slice-wide residual sum and beta = 1 - R (p sums to one)
      if (lt) {
        if (wid == 0) {
          float bs = 0.0f, rs = 0.0f;
          for (int r = lane; r < dt.n; r += 32) {
            const float p = __fmul_rn(ex2_approx(__fmul_rn(__fsub_rn(key_val(Kp[r]), dt.m), P.c2)),
                                      dt.rzf);
            const float y = yb[r];
            const float q = (y >= dd.tau && y != -INFINITY)
                                ? __fmul_rn(ex2_approx(__fmul_rn(__fsub_rn(y, dd.m), P.c2)), dd.rzf)
                                : 0.0f;
            bs = __fadd_rn(bs, fminf(p, q));
            rs = __fadd_rn(rs, fmaxf(__fsub_rn(p, q), 0.0f));
          }
          bs = warp_sum_f(bs);
          rs = warp_sum_f(rs);
          if (lane == 0) {
            sh.pq[0] = bs;
            sh.pq[1] = rs;
          }
        }
        __syncthreads();
        lbeta = sh.pq[0];
        lres = sh.pq[1];
      } else {
        if (dd.list && !dd.exact && wid == 0) warp_make_exact(P, Kq, dd);
        if (dd.list) {
          if (wid == 0 && lane == 0) {
            sh.pq[0] = dd.Z.hi;
            sh.pq[1] = dd.Z.lo;
          }
          __syncthreads();
          set_Zx(dd, ff{sh.pq[0], sh.pq[1]});
        }
        ff W = {0.0f, 0.0f};
        Dist t0 = dt, t1 = dd;
        slice_draw<E>(P, k, gt, gd, P.V, 0, t0, t1, true, 0.5f, &W);
        lres = __fadd_rn(W.hi, W.lo);
        lbeta = __fsub_rn(1.0f, lres);
      }
    } else if (verdict) {
      term = 0;
    } else {
      if (!bonus && tid == 0) atomicMax(S.hint + b, static_cast<uint32_t>(S.NP - i));
      const float u1 = sh.pre[1];
      if (!(u1 >= 0.0f && u1 < 1.0f)) {
        status |= ST_BAD_UNIFORM;
      } else {
        const bool residual = !bonus;
        int tok = -1;
        if (lt) {
          if (S.topp) {
            // the kept p-ranks in token order (top-p alone: built only when
            // a draw follows), by all threads
            if (dt.n <= 192) {
              for (int r = tid; r < dt.n; r += SP_NT) {
                const int v = key_idx(Kp[r]);
                int rank = 0;
                for (int l = 0; l < dt.n; ++l) rank += key_idx(Kp[l]) < v ? 1 : 0;
                K2[rank] = (static_cast<uint64_t>(static_cast<uint32_t>(v)) << 32) |
                           static_cast<uint32_t>(r);
              }
              __syncthreads();
            } else {
              int N = 128;
              while (N < dt.n && N < SP_TOPP_UCAP) N <<= 1;
              for (int r = tid; r < N; r += SP_NT)
                K2[r] = r < dt.n ? (static_cast<uint64_t>(static_cast<uint32_t>(key_idx(Kp[r]))) << 32) |
                                       static_cast<uint32_t>(r)
                                 : ~0ull;
              __syncthreads();
              group_bitonic(K2, N, tid, SP_NT, 0);
            }
          }
          if (wid == 0) {
            float W = 0.0f, Wp = 0.0f;
            int t1 = warp_list_draw(P, Kp, K2, yb, dt.n, dt, dd, residual, u1, true, &W, wb);
            if (t1 < 0) {  // uncertain, or an (almost) empty residual: exact redraw
              if (!dt.exact) warp_make_exact(P, Kp, dt);
              if (residual && dd.list && !dd.exact) warp_make_exact(P, Kq, dd);
              t1 = warp_list_draw(P, Kp, K2, yb, dt.n, dt, dd, residual, u1, false, &W, wb);
              if (t1 < 0)  // empty residual: draw from p
                t1 = warp_list_draw(P, Kp, K2, yb, dt.n, dt, dd, false, u1, false, &Wp, wb);
              if (P.diag && lane == 0) atomicAdd(P.diag + 1, 1u);
            }
            if (lane == 0) {
              sh.scal[4] = t1;
              sh.pq[0] = W;
            }
          }
          __syncthreads();
          tok = sh.scal[4];
          if (residual) resid = sh.pq[0];
        } else {
          if (dd.list && !dd.exact && residual && wid == 0) warp_make_exact(P, Kq, dd);
          if (dd.list && residual) {
            if (wid == 0 && lane == 0) {
              sh.pq[0] = dd.Z.hi;
              sh.pq[1] = dd.Z.lo;
            }
            __syncthreads();
            set_Zx(dd, ff{sh.pq[0], sh.pq[1]});
          }
          ff W = {0.0f, 0.0f};
          Dist t0 = dt, t1 = dd;
          tok = slice_draw<E>(P, k, gt, gd, P.V, 0, t0, t1, residual, u1, &W);
          if (residual) resid = __fadd_rn(W.hi, W.lo);
          if (tok < 0) tok = slice_draw<E>(P, k, gt, gd, P.V, 0, t0, t1, false, u1, &W);
        }
        token = tok;
      }
      SP_PHASE(9);  // decider: draw
    }
  }
  if (S.law) {
    // the law at the token (NaN for a row in error): min(p, q) + (1 - beta)
    // max(0, p - q) / R, min(p, q) when R = 0
    if (tid == 0) {
      const float nan = __int_as_float(0x7fc00000);
      const bool err = (status & ST_ERROR) != 0;
      float ps = fminf(pdbg, qdbg);
      if (lres > 0.0f)
        ps = __fadd_rn(ps, __fdiv_rn(__fmul_rn(__fsub_rn(1.0f, lbeta), fmaxf(__fsub_rn(pdbg, qdbg), 0.0f)),
                                     lres));
      S.lps[b] = err ? nan : ps;
      if (S.lbeta) S.lbeta[b] = err ? nan : lbeta;
      if (S.lpx) S.lpx[b] = err ? nan : pdbg;
      if (S.lqx) S.lqx[b] = err ? nan : qdbg;
    }
    return;
  }
  if (tid == 0) {
    if (term) atomicMax(S.hint + b, static_cast<uint32_t>(S.NP - i));
    const int64_t di = 2 * (static_cast<int64_t>(b) * S.NP + i);
    S.dec[di] = make_uint4(static_cast<uint32_t>(status), static_cast<uint32_t>(token),
                           __float_as_uint(pdbg), __float_as_uint(qdbg));
    S.dec[di + 1] = make_uint4(__float_as_uint(resid), static_cast<uint32_t>(tested), 0u, 0u);
    const unsigned long long bits = (1ull << i) | (term ? (1ull << (32 + i)) : 0ull);
    const unsigned long long old = atom_or_acqrel(S.mask + b, bits);
    SP_PHASE(23);  // decider: decision stores + mask atomic
    const int r = first_end(old | bits);
    if (r >= 0 && first_end(old) < 0) strip_finalize(S, b, r);
    SP_TL_MIN(2 + 2 * i);
    SP_TL_MAX(3 + 2 * i);
  }
  SP_PHASE(10);  // decider: publish + finalise
}

template <typename E, bool VEC>
__global__ void __launch_bounds__(SP_NT, 2) strip_kernel(const __grid_constant__ SP S) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ SpShared sh;
  __shared__ __align__(8) uint64_t bars[NCH];
  const KP &P = S.k;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  SP_PHASE_START;
  const int per_pos = P.B * S.T * S.C;
  const int i = static_cast<int>(blockIdx.x) / per_pos;
  int rem = static_cast<int>(blockIdx.x) - i * per_pos;
  const int b = rem / (S.T * S.C);
  rem -= b * S.T * S.C;
  const int t = rem / S.C, c = rem - t * S.C;
  const int gb = P.gam ? P.gam[b] : P.gm;
  if (gb < 0 || gb > P.gm) {
    if (i == 0 && t == 0 && c == 0 && tid == 0) strip_bad_row(S, b);
    return;
  }
  if (i > gb || (t == 1 && i == gb)) return;
  const int lo = c * S.L;
  const int n = min(P.V, lo + S.L) - lo;
  const E *g = strip_row<E>(P, b, i, t) + lo;
  E *st = reinterpret_cast<E *>(smem);
  Chunks<E> ch;
  ch.make(n);
  if (tid == 0) {
    int skip = 0;
    if (i > 0) {  // position 0 is always evaluated
      asm volatile("griddepcontrol.wait;" ::: "memory");  // the counters are clear
      const uint32_t h = *reinterpret_cast<const volatile uint32_t *>(S.hint + b);
      skip = (h != 0u && S.NP - static_cast<int>(h) < i) ? 1 : 0;
    }
    sh.scal[0] = skip;
    sh.cnt[0] = 0;
    if (VEC && !skip) {
      for (int j = 0; j < NCH; ++j) mbar_init(&bars[j], 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      fence_proxy_async();
      issue_slice<E>(g, st, ch, bars);
    }
  }
  __syncthreads();
  if (sh.scal[0]) {  // an earlier position ended this sequence
    SP_PHASE(0);  // skipped CTAs
    if (tid == 0) SP_TL_MAX(1);
    return;
  }
  SP_PHASE(15);  // started CTAs: entry
  if (tid == 0 && i < 16) {
    SP_TL_MIN(0);
    SP_TL_MIN(36 + i);
  }

  // inputs of a possible decision, loaded now and used at the end of the
  // piece (their latency overlaps the passes)
  int pre_x = -1;
  float pre_u0 = 0.0f, pre_u1 = 0.0f, pre_zx = 0.0f, pre_wx = 0.0f;
  if (tid == 32) {
    if (i < gb) pre_x = P.tok[static_cast<int64_t>(b) * P.gm + i];
    if (!P.greedy && !S.law) {
      const float *ui = P.uni + static_cast<int64_t>(b) * P.u_row + static_cast<int64_t>(i) * P.u_pos;
      if (i < gb) pre_u0 = ui[P.u_acc];
      pre_u1 = ui[P.u_draw];
    }
  }
  // pass 1
  float mx, mx2 = -INFINITY;
  int mi = INT_MAX;
  uint32_t fl;
  if (S.topp) {
    TStat2 s;
    s.init();
    if (VEC)
      scan_slice_top2<E>(g, st, ch, n, bars, 0u, s);
    else
      load_slice_plain<E>(g, st, n, lo, s);
    mx = s.mx;
    mx2 = s.mx2;
    fl = s.flags();
  } else if (P.greedy) {
    TStat<true> s;
    s.init();
    if (VEC)
      scan_slice<E>(g, st, ch, n, lo, bars, 0u, s);
    else
      load_slice_plain<E>(g, st, n, lo, s);
    mx = s.mx;
    mi = s.mi;
    fl = s.flags();
  } else {
    TStat<false> s;
    s.init();
    if (VEC)
      scan_slice<E>(g, st, ch, n, lo, bars, 0u, s);
    else
      load_slice_plain<E>(g, st, n, lo, s);
    mx = s.mx;
    fl = s.flags();
  }
  if (tid == 32 && !P.greedy && i < gb && pre_x >= 0 && pre_x < P.V) {
    pre_zx = raw_of(strip_row<E>(P, b, i, 0)[pre_x]);
    pre_wx = raw_of(strip_row<E>(P, b, i, 1)[pre_x]);
  }
  SP_PHASE(1);  // piece: load + pass 1
  // lower bounds of the piece's k-th and ceil(k/C)-th largest logits: at
  // least NW * r (NW * r2) elements are >= the minimum over the warps of
  // the r-th (r2-th) largest per-thread maximum
  float th = -INFINITY, ph = -INFINITY;
  if (S.topp) {
    // the warp's 64 values (each lane's largest and second largest: distinct
    // elements of its share) sorted; at least S.kc elements of the warp's
    // share are >= the kc-th largest of them, so at least SP_NW * S.kc
    // elements of the piece are >= the minimum over the warps
    uint64_t v2[2] = {(static_cast<uint64_t>(~fkey(canon(mx))) << 32) | static_cast<uint32_t>(lane),
                      (static_cast<uint64_t>(~fkey(canon(mx2))) << 32) | static_cast<uint32_t>(32 + lane)};
    warp_bitonic<2>(v2);
    const int r = S.kc - 1;
    const uint64_t kr = __shfl_sync(FULL, r >= 32 ? v2[1] : v2[0], r & 31);
    th = key_to_f(~static_cast<uint32_t>(kr >> 32));
    ph = th;
  } else if (!P.greedy) {
    const float srt = warp_sort_desc(mx);
    th = __shfl_sync(FULL, srt, S.r - 1);
    ph = __shfl_sync(FULL, srt, S.r2 - 1);
  }
  {
    float wm = mx;
    int wmi = mi;
    if (P.greedy)
      warp_argmax(wm, wmi);
    else
      wm = warp_max(wm);
    const uint32_t wfl = warp_or(fl);
    if (lane == 0) {
      sh.wv[wid] = wm;
      sh.wi[wid] = wmi;
      sh.wf[wid] = wfl;
      sh.wth[wid] = th;
      sh.wph[wid] = ph;
    }
  }
  __syncthreads();
  float M = -INFINITY, TH = INFINITY, PH = INFINITY;
  int MI = INT_MAX;
  uint32_t F = 0u;
#pragma unroll
  for (int w = 0; w < SP_NW; ++w) {
    const float v = sh.wv[w];
    const int vi = sh.wi[w];
    if (v > M || (v == M && vi < MI)) {
      M = v;
      MI = vi;
    }
    F |= sh.wf[w];
    TH = fminf(TH, sh.wth[w]);
    PH = fminf(PH, sh.wph[w]);
  }
  SP_PHASE(2);  // piece: reductions + bounds
  // pass 2: the candidates >= TH (at least top_k of them), written to the
  // workspace and to a shared-memory copy, in thread order (deterministic)
  const int64_t slot = blockIdx.x;
  int cnt = 0;
  ff zt = {0.0f, 0.0f};  // top-p alone: weight sum of the logits below PH, and its bound
  float zte = 0.0f;
  if (S.topp) {
    unsigned long long *gc = S.cand + slot * S.capc;
    constexpr int EPV = Elem<E>::kPerVec;
    const uint4 *s4 = reinterpret_cast<const uint4 *>(st);
    const int nv = n / EPV;
    // one sweep: mark the thread's vectors whose maximum reaches TH, and sum
    // the weights e^{(z - M)/T} of the logits below TH (the tail): each
    // vector's weights by a tree of depth log2(EPV), the vector sums
    // compensated; the weights' error bound sum_e e (k0 + k1 |y|) from
    // sum e and sum e y (y <= 0)
    uint64_t hm = 0;
    float zs = 0.0f, zc = 0.0f, zy = 0.0f;
    {
      // two lanes per packed operation (each rounded as the scalar one: the
      // same values, and the tree adds in the same pairs)
      const f2 M2 = f2_pack(M, M), C2 = f2_pack(P.c2, P.c2);
      f2 zy2 = f2_pack(0.0f, 0.0f);
      int it = 0;
      for (int v = tid; v < nv; v += SP_NT, ++it) {
        float f[EPV];
        f2 w2[EPV / 2];
        const uint4 raw = s4[v];
        unpack<E>(raw, f);
        hm |= static_cast<uint64_t>(vec_max_nan<E>(raw) >= TH ? 1u : 0u) << it;
#pragma unroll
        for (int e = 0; e < EPV; e += 2) {
          float y0, y1;
          f2_unpack(f2_mul(f2_sub(f2_pack(f[e], f[e + 1]), M2), C2), y0, y1);
          const float x0 = f[e] < TH ? ex2_approx(y0) : 0.0f;
          const float x1 = f[e + 1] < TH ? ex2_approx(y1) : 0.0f;
          w2[e / 2] = f2_pack(x0, x1);
          zy2 = f2_fma(w2[e / 2], f2_pack(fmaxf(y0, -256.0f), fmaxf(y1, -256.0f)), zy2);
        }
        // the tree: w[e] + w[e + h] for h = EPV/2 .. 1, the first levels on pairs
#pragma unroll
        for (int h = EPV / 4; h; h >>= 1)
#pragma unroll
          for (int e = 0; e < h; ++e) w2[e] = f2_add(w2[e], w2[e + h]);
        float w0, w1;
        f2_unpack(w2[0], w0, w1);
        const float t = __fsub_rn(__fadd_rn(w0, w1), zc), s2 = __fadd_rn(zs, t);
        zc = __fsub_rn(__fsub_rn(s2, zs), t);
        zs = s2;
      }
      float za, zb;
      f2_unpack(zy2, za, zb);
      zy = __fadd_rn(za, zb);
    }
    const int jt = nv * EPV + tid;
    const float ftail = jt < n ? stage_raw(st, jt) : -INFINITY;
    if (jt < n && ftail < TH) {
      const float y = __fmul_rn(__fsub_rn(ftail, M), P.c2);
      const float x = ex2_approx(y);
      zy = __fmaf_rn(x, fmaxf(y, -256.0f), zy);
      const float t = __fsub_rn(x, zc), s2 = __fadd_rn(zs, t);
      zc = __fsub_rn(__fsub_rn(s2, zs), t);
      zs = s2;
    }
    // the candidates: the logits >= TH
    const float PHt = TH;
    // the candidates >= PHt, in thread order, then index order
    const bool tail = jt < n && ftail >= PHt;
    int ct = tail ? 1 : 0;
    for (uint64_t h = hm; h; h &= h - 1) {
      const int v = tid + (__ffsll(static_cast<long long>(h)) - 1) * SP_NT;
      float f[EPV];
      unpack<E>(s4[v], f);
#pragma unroll
      for (int e = 0; e < EPV; ++e) ct += f[e] >= PHt ? 1 : 0;
    }
    int incl = ct;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(FULL, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) sh.wcnt[wid] = incl;
    __syncthreads();
    int base = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < SP_NW; ++w) {
      const int x = sh.wcnt[w];
      base += w < wid ? x : 0;
      tot += x;
    }
    if (ct) {
      int pos = base + incl - ct;
      for (uint64_t h = hm; h; h &= h - 1) {
        const int v = tid + (__ffsll(static_cast<long long>(h)) - 1) * SP_NT;
        float f[EPV];
        unpack<E>(s4[v], f);
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          if (f[e] >= PHt) {
            if (pos < S.capc) gc[pos] = cand_key(f[e], lo + v * EPV + e);
            ++pos;
          }
        }
      }
      if (tail && pos < S.capc) gc[pos] = cand_key(ftail, lo + jt);
    }
    cnt = tot;
    if (cnt > S.capc) {
      F |= F_OVER;
      cnt = S.capc;
    }
    // weights' bound k0 sum e + k1 sum e |y|
    const float ze = __fmaf_rn(__fmul_rn(zs, 1.001f), kExpErr0, -__fmul_rn(zy, kExpErr1));
    const ff zwf = warp_sum_ff(quick_two_sum(zs, -zc));
    const float zew = warp_sum_f(ze);
    if (lane == 0) {
      sh.wz[wid][0] = zwf.hi;
      sh.wz[wid][1] = zwf.lo;
      sh.wz[wid][2] = zew;
    }
    __syncthreads();
#pragma unroll
    for (int w = 0; w < SP_NW; ++w) {
      zt = ff_add(zt, ff{sh.wz[w][0], sh.wz[w][1]});
      zte = __fadd_rn(zte, sh.wz[w][2]);
    }
    // the rounding of the vector sums' trees (log2(EPV) units each) and of
    // the compensated sums (two units), and weights flushed to zero below
    // 2^-126
    zte = __fadd_rn(__fmaf_rn(zt.hi, 6.0e-7f, zte), static_cast<float>(n) * 1.2e-38f);
    TH = PHt;
    PH = PHt;
  } else if (!P.greedy) {
    unsigned long long *gc = S.cand + slot * S.capc;
    uint64_t *cb = reinterpret_cast<uint64_t *>(smem + S.off_cb);
    constexpr int EPV = Elem<E>::kPerVec;
    const uint4 *s4 = reinterpret_cast<const uint4 *>(st);
    const int nv = n / EPV;
    // one sweep marks the thread's vectors whose maximum reaches TH (bit j:
    // its j-th vector; a piece of at most 192 KB gives each thread at most 48
    // vectors); the candidates are then counted and written from the marked
    // vectors only (a few in a hundred)
    uint64_t hm = 0;
    {
      int it = 0;
      for (int v = tid; v < nv; v += SP_NT, ++it) {
        float f[EPV];
        unpack<E>(s4[v], f);
        float vm = f[0];
#pragma unroll
        for (int e = 1; e < EPV; ++e) vm = fmaxf(vm, f[e]);
        hm |= static_cast<uint64_t>(vm >= TH ? 1u : 0u) << it;
      }
    }
    SP_PHASE(12);  // piece: pass 2 sweep
    // the tail (fewer than EPV elements, staged by their own threads)
    const int jt = nv * EPV + tid;
    const float ftail = jt < n ? stage_raw(st, jt) : -INFINITY;
    const bool tail = jt < n && ftail >= TH;
    int ct = tail ? 1 : 0;
    for (uint64_t h = hm; h; h &= h - 1) {
      const int v = tid + (__ffsll(static_cast<long long>(h)) - 1) * SP_NT;
      float f[EPV];
      unpack<E>(s4[v], f);
#pragma unroll
      for (int e = 0; e < EPV; ++e) ct += f[e] >= TH ? 1 : 0;
    }
    int incl = ct;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(FULL, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) sh.wcnt[wid] = incl;
    __syncthreads();
    int base = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < SP_NW; ++w) {
      const int x = sh.wcnt[w];
      base += w < wid ? x : 0;
      tot += x;
    }
    if (ct) {
      // thread order, then index order
      int pos = base + incl - ct;
      for (uint64_t h = hm; h; h &= h - 1) {
        const int v = tid + (__ffsll(static_cast<long long>(h)) - 1) * SP_NT;
        float f[EPV];
        unpack<E>(s4[v], f);
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          if (f[e] >= TH) {
            if (pos < S.capc) {
              const uint64_t kk = cand_key(f[e], lo + v * EPV + e);
              gc[pos] = kk;
              cb[pos] = kk;
            }
            ++pos;
          }
        }
      }
      if (tail && pos < S.capc) {
        const uint64_t kk = cand_key(ftail, lo + jt);
        gc[pos] = kk;
        cb[pos] = kk;
      }
    }
    cnt = tot;
    SP_PHASE(13);  // piece: pass 2 count + write
    if (cnt > S.capc) {
      F |= F_OVER;
      cnt = S.capc;
    }
    // a tighter bound of the piece's ceil(k/C)-th largest logit: the least
    // candidate in the bin of a value histogram of the candidates where the
    // count from the top reaches ceil(k/C) (that many elements are >= it)
    if (!(F & F_OVER) && TH > -INFINITY && M > TH && cnt >= S.kc) {
      const BinMap bm = bin_map(TH, M);
      sh.hist[tid] = 0u;  // SP_NT == 256 bins
      if (tid == 0) sh.umin = 0xffffffffu;
      __syncthreads();
      for (int j = tid; j < cnt; j += SP_NT) atomicAdd(&sh.hist[value_bin(key_val(cb[j]), bm)], 1u);
      __syncthreads();
      if (wid == 0) {
        uint32_t c8[8], loc = 0u;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          c8[q] = sh.hist[lane * 8 + q];
          loc += c8[q];
        }
        uint32_t incl = loc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t u = __shfl_up_sync(FULL, incl, o);
          if (lane >= o) incl += u;
        }
        const uint32_t excl = incl - loc;
        const uint32_t kc = static_cast<uint32_t>(S.kc);
        if (excl < kc && kc <= incl) {
          // the first bin (from the top) where the count reaches kc
          uint32_t before = excl;
          int d = -1;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if (d < 0) {
              if (before + c8[q] >= kc)
                d = lane * 8 + q;
              else
                before += c8[q];
            }
          }
          sh.scal[5] = d;
        }
      }
      __syncthreads();
      const int dsel = sh.scal[5];
      for (int j = tid; j < cnt; j += SP_NT) {
        const float v = key_val(cb[j]);
        if (value_bin(v, bm) == dsel) atomicMin(&sh.umin, fkey(v));
      }
      __syncthreads();
      PH = fmaxf(PH, key_to_f(sh.umin));
    }
  }
  SP_PHASE(3);  // piece: pass 2
  if (tid == 0) {
    S.hdr[slot] = make_uint4(static_cast<uint32_t>(cnt) | (F << 24), __float_as_uint(M),
                             P.greedy ? static_cast<uint32_t>(MI) : __float_as_uint(TH),
                             __float_as_uint(PH));
    if (S.topp)
      S.hdr2[slot] = make_uint4(__float_as_uint(zt.hi), __float_as_uint(zt.lo),
                                __float_as_uint(zte), 0u);
  }
  if (tid == 32) {
    sh.pre_x = pre_x;
    sh.pre[0] = pre_u0;
    sh.pre[1] = pre_u1;
    sh.pre[2] = pre_zx;
    sh.pre[3] = pre_wx;
  }
  __syncthreads();
  if (tid == 0) {
    if (i == 0) asm volatile("griddepcontrol.wait;" ::: "memory");  // the counters are clear
    const int need = (S.T == 2 && i < gb) ? 2 * S.C : S.C;
    const uint32_t old = atom_add_acqrel(S.arrive + static_cast<int64_t>(b) * S.NP + i, 1u);
    sh.scal[1] = static_cast<int>(old) == need - 1 ? 1 : 0;
  }
  __syncthreads();
  if (tid == 0 && i < 16) SP_TL_MAX(20 + i);
  SP_PHASE(4);  // piece: header + fence + arrival
  if (sh.scal[1]) strip_decide<E>(S, sh, smem, b, i, gb);
  if (VEC && (F & F_TIMEOUT) && tid == 0) {
    // let copies that outlived a timed-out wait land before the CTA exits
    for (int j = 0; j < NCH; ++j) (void)mbar_wait(&bars[j], 0u, kWaitPolls);
  }
  if (tid == 0) SP_TL_MAX(1);
}

}  // namespace sv

#ifdef SV_PHASE_PROFILE
extern "C" int sv_strip_tl_read(unsigned long long *host, int reset) {
  if (cudaMemcpyFromSymbol(host, sv_strip_tl, 64 * sizeof(unsigned long long)) != cudaSuccess)
    return 1;
  if (reset) {
    unsigned long long z[64];
    for (int j = 0; j < 64; ++j) z[j] = (j == 0 || (j >= 2 && j < 20 && j % 2 == 0) || j >= 36) ? ~0ull : 0ull;
    if (cudaMemcpyToSymbol(sv_strip_tl, z, sizeof z) != cudaSuccess) return 1;
  }
  return 0;
}
extern "C" int sv_strip_phase_read(unsigned long long *host, int reset) {
  if (cudaMemcpyFromSymbol(host, sv_strip_cycles, 64 * sizeof(unsigned long long)) != cudaSuccess)
    return 1;
  if (reset) {
    unsigned long long z[64] = {0};
    if (cudaMemcpyToSymbol(sv_strip_cycles, z, sizeof z) != cudaSuccess) return 1;
  }
  return 0;
}
#endif

namespace sv {

namespace {

inline int64_t aup(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

using StripFn = void (*)(SP);

// Clears the per-call counters; lets the verify grid launch at once (it
// waits for this grid before its first counter access).
__global__ void strip_clear(uint32_t *p, int n) {
  asm volatile("griddepcontrol.launch_dependents;");
  for (int j = static_cast<int>(blockIdx.x * blockDim.x + threadIdx.x); j < n;
       j += static_cast<int>(gridDim.x * blockDim.x))
    p[j] = 0u;
}

StripFn strip_fn(int dtype, bool vec) {
  if (dtype == SPEC_F32) return vec ? strip_kernel<float, true> : strip_kernel<float, false>;
  return vec ? strip_kernel<uint16_t, true> : strip_kernel<uint16_t, false>;
}

cudaError_t strip_prepare(StripFn f) {
  static std::mutex mu;
  static std::map<StripFn, cudaError_t> done;
  std::lock_guard<std::mutex> lk(mu);
  auto it = done.find(f);
  if (it != done.end()) return it->second;
  const cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void *>(f),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             200 * 1024);
  done[f] = e;
  return e;
}

}  // namespace

StripPlan strip_plan(const spec_params &p, bool law) {
  StripPlan s;
  if (p.B < 1 || p.V < 1 || p.V > (1 << 24) || p.gamma_max < 0 || p.gamma_max > 31) return s;
  if (p.dtype != SPEC_F32 && p.dtype != SPEC_BF16) return s;
  const bool greedy = p.temperature == 0.0f;
  const bool k_on = p.top_k > 0 && p.top_k < p.V;
  const bool topp = !greedy && !k_on && p.top_p < 1.0f;
  if (!greedy && !topp && !(k_on && p.top_k <= SP_NW * kWarp)) return s;
  const int64_t es = p.dtype == SPEC_F32 ? 4 : 2;
  int C = p.cluster_size > 0
              ? p.cluster_size
              : static_cast<int>((static_cast<int64_t>(p.V) * es + SP_PIECE_BYTES - 1) /
                                 SP_PIECE_BYTES);
  C = std::max(1, std::min(C, SP_MAXC));
  const int64_t L = aup((static_cast<int64_t>(p.V) + C - 1) / C, 8);
  C = static_cast<int>((p.V + L - 1) / L);
  if (L * es > 192 * 1024) return s;  // a piece is staged in shared memory
  s.dtype = p.dtype;
  s.C = C;
  s.L = static_cast<int>(L);
  s.T = (greedy || p.gamma_max == 0) ? 1 : 2;  // no draft slot: the target alone
  s.NP = law ? 1 : p.gamma_max + 1;
  s.law = law;
  s.topp = topp;
  s.r = (greedy || topp) ? 0 : (p.top_k + SP_NW - 1) / SP_NW;
  s.r2 = (greedy || topp) ? 0 : ((p.top_k + C - 1) / C + SP_NW - 1) / SP_NW;
  int capc = 0;
  if (topp) {
    capc = p.list_capacity > 0 ? p.list_capacity : SP_TOPP_CAPC;
  } else if (!greedy) {
    capc = 256;
    while (capc < 4 * p.top_k) capc *= 2;
    if (p.list_capacity > 0) capc = p.list_capacity;
  }
  s.kc = greedy ? 0 : (topp ? SP_TOPP_K : (p.top_k + C - 1) / C);
  s.capc = capc;
  s.items = static_cast<int64_t>(s.NP) * p.B * s.T * s.C;
  if (s.items > INT32_MAX) return s;
  const size_t stage = static_cast<size_t>(aup(L * es, 128));
  s.off_cb = stage;  // the piece's candidate copy follows its staged slice
  s.smem = greedy ? stage
                  : std::max(stage + static_cast<size_t>(capc) * 8,
                             topp ? SP_DEC_SMEM_P : SP_DEC_SMEM);
  size_t o = 16;  // diagnostics counters (kept across calls)
  s.off_ctr = o;
  s.off_arrive = o;
  o += static_cast<size_t>(p.B) * s.NP * 4;
  s.off_hint = o;
  o += static_cast<size_t>(p.B) * 4;
  o = static_cast<size_t>(aup(static_cast<int64_t>(o), 8));
  s.off_mask = o;
  o += static_cast<size_t>(p.B) * 8;
  s.ctr_bytes = o - s.off_ctr;
  o = static_cast<size_t>(aup(static_cast<int64_t>(o), 16));
  s.off_dec = o;
  o += static_cast<size_t>(p.B) * s.NP * 32;
  s.off_hdr = o;
  o += static_cast<size_t>(s.items) * 16;
  s.off_hdr2 = o;
  if (topp) o += static_cast<size_t>(s.items) * 16;
  s.off_cand = o;
  o += static_cast<size_t>(s.items) * s.capc * 8;
  s.ws_bytes = o;
  s.ok = true;
  return s;
}

spec_status strip_launch(const KP &kp, const StripPlan &pl, void *ws, bool vec,
                         cudaStream_t stream, float *const *law_out) {
  SP S;
  std::memset(&S, 0, sizeof S);
  S.k = kp;
  S.k.diag = static_cast<unsigned int *>(ws);
  S.C = pl.C;
  S.L = pl.L;
  S.T = pl.T;
  S.NP = pl.NP;
  S.capc = pl.capc;
  S.r = pl.r;
  S.r2 = pl.r2;
  S.kc = pl.kc;
  S.topp = pl.topp ? 1 : 0;
  S.law = pl.law ? 1 : 0;
  if (pl.law) {
    if (!law_out || !law_out[0]) return SPEC_ERR_INVALID_ARG;
    S.lps = law_out[0];
    S.lbeta = law_out[1];
    S.lpx = law_out[2];
    S.lqx = law_out[3];
  }
  S.off_cb = static_cast<int32_t>(pl.off_cb);
  char *w = static_cast<char *>(ws);
  S.arrive = reinterpret_cast<uint32_t *>(w + pl.off_arrive);
  S.hint = reinterpret_cast<uint32_t *>(w + pl.off_hint);
  S.mask = reinterpret_cast<unsigned long long *>(w + pl.off_mask);
  S.dec = reinterpret_cast<uint4 *>(w + pl.off_dec);
  S.hdr = reinterpret_cast<uint4 *>(w + pl.off_hdr);
  S.hdr2 = reinterpret_cast<uint4 *>(w + pl.off_hdr2);
  S.cand = reinterpret_cast<unsigned long long *>(w + pl.off_cand);
  const StripFn f = strip_fn(pl.dtype, vec);
  if (strip_prepare(f) != cudaSuccess) return SPEC_ERR_CUDA;
  const int nw = static_cast<int>(pl.ctr_bytes / 4);
  strip_clear<<<static_cast<unsigned>(std::min(64, (nw + 255) / 256)), 256, 0, stream>>>(
      reinterpret_cast<uint32_t *>(w + pl.off_ctr), nw);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(pl.items));
  cfg.blockDim = dim3(SP_NT);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, f, S) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace sv
