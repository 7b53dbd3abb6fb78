// sv_strip.h -- host interface of the strip-parallel verify kernel
// (spec_strip.cu), used by the C ABI in spec_verify.cu.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "spec_verify.h"

namespace sv {

struct KP;

// Launch plan of the strip path for one problem shape.
struct StripPlan {
  bool ok = false;     // the strip path handles this problem
  int dtype = 0;       // spec_dtype of the logits
  int C = 1;           // pieces per strip
  int L = 0;           // piece length (elements, multiple of 8)
  int T = 1;           // tensors per position (1 greedy, 2 sampling)
  int NP = 1;          // positions per row (gamma_max + 1)
  int capc = 0;        // candidate capacity per piece
  int r = 0, r2 = 0;   // ranks of the per-warp lower bounds (k-th, ceil(k/C)-th)
  int kc = 0;          // ceil(top_k / C); top-p alone: candidates aimed at per piece
  bool topp = false;   // top-p without top-k
  bool law = false;    // the law at one token per row (spec_law): one position per row
  size_t off_cb = 0;   // shared-memory offset of a piece's candidate copy
  int64_t items = 0;   // CTAs of one launch
  size_t smem = 0;     // dynamic shared memory per CTA
  size_t off_ctr = 0, ctr_bytes = 0;  // counters cleared before each launch
  size_t off_arrive = 0, off_hint = 0, off_mask = 0, off_dec = 0, off_hdr = 0, off_hdr2 = 0,
         off_cand = 0;
  size_t ws_bytes = 0;  // workspace the launch needs
};

// Plan of the strip path (ok = false: use the cluster kernel).  Depends on
// the shape and filters only, not on pointers.  law: the emitted-token law
// of spec_law, one position per row (p.gamma_max must be 1: the row's
// target and draft logits are position 0; sampling with top-k or top-p).
StripPlan strip_plan(const spec_params &p, bool law = false);

// Enqueue the strip path on `stream`: clear the counters, launch the kernel.
// kp holds the tensors, strides, filters and outputs (as for the cluster
// kernel); ws is the caller's workspace (>= plan.ws_bytes, 16-byte aligned).
// law_out (plan.law): device float [B] p_spec, beta, p(x), q(x) (each may
// be null but p_spec).
spec_status strip_launch(const KP &kp, const StripPlan &plan, void *ws, bool vec,
                         cudaStream_t stream, float *const *law_out = nullptr);

}  // namespace sv
