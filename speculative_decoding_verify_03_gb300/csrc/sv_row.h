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

// Enqueue the warp-per-row kernel on `stream`.  kp holds the tensors,
// strides, temperature and outputs as for the other kernels; dtype: the
// spec_dtype of the logits; vec: every row starts on a 16-byte boundary.
spec_status row_launch(const KP &kp, int dtype, bool vec, cudaStream_t stream);

}  // namespace sv
