// sv_row.h -- host interface of the warp-per-row verify kernel (spec_row.cu)
// for small vocabularies, used by the C ABI in spec_verify.cu.
#pragma once

#include <cuda_runtime.h>

#include "spec_verify.h"

namespace sv {

struct KP;

// Largest vocabulary of the warp-per-row kernel: 32 logits per lane.
constexpr int kRowMaxV = 1024;

// The warp-per-row kernel handles this problem: a vocabulary of at most
// kRowMaxV, and greedy or unfiltered sampling (no top-k, no top-p).
bool row_eligible(const spec_params &p);

// Workspace offset of the deferred-row list (the diagnostics words and the
// list's counter come first).
constexpr size_t kRowDeferOffset = 32;

// Workspace bytes that let the warp-per-row kernel hand its uncertain rows
// to a second kernel (0: greedy problems never need it).
size_t row_defer_bytes(const spec_params &p);

// Enqueue the warp-per-row kernel on `stream`.  kp holds the tensors,
// strides, temperature and outputs as for the other kernels; dtype: the
// spec_dtype of the logits; vec: every row starts on a 16-byte boundary.
// With a workspace of row_defer_bytes(p), rows whose certified decision is
// uncertain are finished by a second kernel (one CTA per row, float-float);
// without one, the row's warp redoes the decision itself.
spec_status row_launch(const KP &kp, int dtype, bool vec, void *ws, size_t ws_bytes,
                       const spec_params &p, cudaStream_t stream);

}  // namespace sv
