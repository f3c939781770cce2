// fused_tc.cu -- the fused plan (placeholder until the tensor-core kernel
// lands): reports every shape as unsupported.
#include "ssd_fused.cuh"

namespace ssd {

bool fused_supported(const ssd_fwd_args *) { return false; }
const char *fused_unsupported_reason(const ssd_fwd_args *) { return "fused plan not built"; }
bool fused_preferred(const ssd_fwd_args *) { return false; }
size_t fused_workspace_size(const ssd_fwd_args *) { return 256; }
cudaError_t run_fused(const ssd_fwd_args *, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace ssd
