// sv_verify.h -- host helpers of the verify entry points (spec_verify.cu)
// shared with the other entry points of the library.
#pragma once

#include <cstddef>
#include <cstdint>

#include "spec_verify.h"

namespace sv {

// The argument checks of spec_verify (sample_mode: those of spec_sample):
// SPEC_OK when a call with these arguments would be enqueued (or is a
// no-op), else the status spec_verify returns, before any launch.
spec_status check_verify_args(const void *target, const void *draft, const int32_t *tokens,
                              const float *uniforms, const spec_params *p, const int32_t *acc,
                              const int32_t *next, const void *ws, size_t ws_bytes,
                              bool sample_mode);

// The argument checks of spec_law: SPEC_OK when a call with these arguments
// would be enqueued (or is a no-op), else the status it returns.
spec_status law_check_args(const void *target_logits, const void *draft_logits,
                           const int32_t *tokens, const spec_params *params, const float *p_spec);

}  // namespace sv
