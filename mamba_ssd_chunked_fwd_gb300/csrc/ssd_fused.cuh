// ssd_fused.cuh -- the fused plan: one persistent tensor-core kernel that
// keeps every chunk state on chip (declarations; see fused_tc.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

#include "../../include/ssd.h"
#include "ssd_internal.cuh"

namespace ssd {

// TMA descriptor of a [batch, tokens, features] tensor of dtype io (an
// IoType), boxes of 128 bytes x 64 tokens x 1, 128-byte swizzle or none, zero
// fill past the end of the sequence.
cudaError_t encode_tile_map(CUtensorMap *m, const void *base, int io, int64_t feats, int64_t L, int64_t B,
                            bool swizzle);

// The segment passes of the fused plan at N = 128 (segstate.cu): the state
// entering each segment s >= 1 into seg_states [B, nseg, H, P, N], with
// seg_decay [B, H, nseg] as scratch.  Nothing is launched when nseg < 2.
struct SegMaps {
    CUtensorMap x, b;
};
int segment_max_len();
bool segment_smem_fits(int io, int seg_len);
cudaError_t launch_segment_passes(const Params &p, int io, bool bf16, float *seg_states, float *seg_decay,
                                  unsigned int *err, int sms, cudaStream_t s);

bool fused_supported(const ssd_fwd_args *a);
// Packed sequences take the fused plan at N = 64 only.
bool fused_varlen_supported(const ssd_fwd_args *a);
// The causal conv1d in front of the SSD runs inside the fused kernel at N = 64.
bool fused_conv_supported(const ssd_fwd_args *a);
// Segments the fused walk cuts each sequence into (1 at N = 64).
int fused_segments(const ssd_fwd_args *a);
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
