// kda_internal.h -- host-side helpers shared by the library's translation units
// (not exported).
#pragma once

#include <stdint.h>

#include "kda_solve_tril.h"

namespace kda {

// The host-side argument checks of kda_solve_tril that do not involve the
// workspace: dtypes, shape limits, the packed/dense layout rules, null
// pointers, 16-byte alignment and overlap of A and Ai.  Makes no CUDA call.
kda_status_t validate_solve(const void *A, const void *Ai, const int32_t *cu, int32_t num_seqs, int64_t B,
                            int64_t T, int32_t H, int32_t in_dt, int32_t out_dt);

}  // namespace kda
