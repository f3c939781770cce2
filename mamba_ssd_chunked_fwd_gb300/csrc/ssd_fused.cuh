// ssd_fused.cuh -- the fused plan: one persistent tensor-core kernel that
// keeps every chunk state on chip (declarations; see fused_tc.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "../../include/ssd.h"

namespace ssd {

bool fused_supported(const ssd_fwd_args *a);
// The fused kernel can apply the gated RMSNorm in its store stage: z given and
// at most 4 heads per group (a cluster of up to 2 CTAs, one per head pair).
bool fused_norm_supported(const ssd_fwd_args *a);
const char *fused_unsupported_reason(const ssd_fwd_args *a);
bool fused_preferred(const ssd_fwd_args *a);
size_t fused_workspace_size(const ssd_fwd_args *a);
cudaError_t run_fused(const ssd_fwd_args *a, cudaStream_t s);
// Packed variable-length sequences along L of a B = 1 call (cu: host, nseq + 1
// offsets; states indexed by sequence).  The workspace holds the error word,
// the offsets and the host-built schedule of units over CTAs.
size_t fused_varlen_workspace_size(const ssd_fwd_args *a, int64_t nseq);
cudaError_t run_fused_varlen(const ssd_fwd_args *a, const int64_t *cu, int nseq, cudaStream_t s);

}  // namespace ssd
