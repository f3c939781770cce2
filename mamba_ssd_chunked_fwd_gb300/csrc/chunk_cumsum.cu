// chunk_cumsum.cu -- step 1 of the chunked SSD forward (ops-transformer
// MambaV2 article, section 4.2 "mamba2_chunk_cumsum"): processed step
// d_t = clamp(softplus(dt + dt_bias)) and the inclusive cumulative sum of
// d_t * A[h] inside each chunk.
//
// One CTA per (chunk k, batch b, tile of 16 heads).  dt is [B,L,H] with the
// head index fastest, so the load reads 16 heads of a token as one segment.
// The scan runs sequentially per head (one thread each), in token order:
// past the end of a ragged sequence the step is exactly 0, so the sum holds
// its last value bit for bit.  Both outputs go out through shared memory as
// contiguous [B,H,c,Q] rows.
#include "ssd_internal.cuh"

namespace ssd {

namespace {

constexpr int kHeadsPerCta = 16;
constexpr int kThreads = 256;
constexpr int kMaxQ = 256;

__global__ void __launch_bounds__(kThreads)
chunk_cumsum_kernel(Params p, float *__restrict__ dtp, float *__restrict__ cs) {
    __shared__ float d_s[kHeadsPerCta][kMaxQ + 1];
    __shared__ float c_s[kHeadsPerCta][kMaxQ + 1];
    const int k = blockIdx.x, b = blockIdx.y, h0 = blockIdx.z * kHeadsPerCta;
    const int Q = p.Q, L = p.L, H = p.H;
    const int nh = min(kHeadsPerCta, H - h0);

    for (int e = threadIdx.x; e < kHeadsPerCta * Q; e += kThreads) {
        const int hh = e % kHeadsPerCta, i = e / kHeadsPerCta;
        const int t = k * Q + i, h = h0 + hh;
        float d = 0.f;
        if (t < L && hh < nh) d = dt_processed(p, __ldg(p.dt + ((size_t)b * L + t) * H + h), h);
        d_s[hh][i] = d;
    }
    __syncthreads();
    if (threadIdx.x < nh) {
        const int hh = threadIdx.x;
        const float a = __ldg(p.A + h0 + hh);
        float run = 0.f;
        for (int i = 0; i < Q; ++i) {
            run = fmaf(d_s[hh][i], a, run);
            c_s[hh][i] = run;
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < nh * Q; e += kThreads) {
        const int hh = e / Q, i = e % Q;
        const size_t row = (((size_t)b * H + h0 + hh) * p.nchunks + k) * Q;
        dtp[row + i] = d_s[hh][i];
        cs[row + i] = c_s[hh][i];
    }
}

}  // namespace

cudaError_t launch_chunk_cumsum(const Params &p, float *dtp, float *cs, cudaStream_t s) {
    if (p.Q > kMaxQ) return cudaErrorInvalidValue;
    dim3 grid(p.nchunks, p.B, (p.H + kHeadsPerCta - 1) / kHeadsPerCta);
    chunk_cumsum_kernel<<<grid, kThreads, 0, s>>>(p, dtp, cs);
    return cudaGetLastError();
}

}  // namespace ssd
