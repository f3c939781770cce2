// ssd_fused.cuh -- the fused plan: one persistent tensor-core kernel that
// keeps every chunk state on chip (declarations; see fused_tc.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "../../include/ssd.h"

namespace ssd {

bool fused_supported(const ssd_fwd_args *a);
const char *fused_unsupported_reason(const ssd_fwd_args *a);
bool fused_preferred(const ssd_fwd_args *a);
size_t fused_workspace_size(const ssd_fwd_args *a);
// cu_dev (device, nseq + 1 offsets): packed variable-length sequences along L
// of a B = 1 call, states indexed by sequence; NULL for the regular layout.
cudaError_t run_fused(const ssd_fwd_args *a, cudaStream_t s, const long long *cu_dev = nullptr, int nseq = 0);

}  // namespace ssd
