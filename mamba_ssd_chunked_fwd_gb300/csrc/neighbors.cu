// neighbors.cu -- the two operators around the SSD on the pages
// (ops-transformer MambaV2 article, sections 1.4, 4.1 and 4.6):
//
//   causal conv1d + SiLU   out[b,d,t] = silu(bias[d] + sum_k w[d,k] x[b,d,t-(W-1)+k])
//                          (depthwise along the sequence, x = 0 before t = 0)
//   gated RMSNorm          v = x * silu(z);  out = v / sqrt(mean_group(v^2) + eps) * w
//                          over `groups` runs of D/groups consecutive channels
//
// Both are HBM-bound elementwise-plus-reduction passes, fp32 arithmetic.
//   conv1d: one CTA per (1024-token tile, channel, batch); the tile and its
//           W-1 token halo go through shared memory, loads and stores are
//           coalesced along the sequence.
//   RMSNorm: one warp per (row, group); the group's sum of squares is a warp
//           reduction, a second pass (from L1/L2) writes the output.
#include "ssd_internal.cuh"

namespace ssd {

namespace {

constexpr int kConvThreads = 256;
constexpr int kConvPer = 4;  // outputs per thread
constexpr int kConvTile = kConvThreads * kConvPer;
constexpr int kMaxW = 8;

template <int IO>
__global__ void __launch_bounds__(kConvThreads)
causal_conv1d_kernel(int S, int D, int W, const void *x, const float *__restrict__ w, const float *__restrict__ bias,
                     int silu, void *out) {
    __shared__ float xs[kConvTile + kMaxW - 1];
    const int s0 = blockIdx.x * kConvTile, d = blockIdx.y, b = blockIdx.z;
    const size_t row = ((size_t)b * D + d) * S;
    const int halo = W - 1;
    for (int i = threadIdx.x; i < kConvTile + halo; i += kConvThreads) {
        const int t = s0 - halo + i;
        xs[i] = (t >= 0 && t < S) ? ld_io<IO>(x, row + t) : 0.f;
    }
    float wk[kMaxW];
#pragma unroll
    for (int k = 0; k < kMaxW; ++k) wk[k] = k < W ? __ldg(w + (size_t)d * W + k) : 0.f;
    const float bv = bias ? __ldg(bias + d) : 0.f;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kConvPer; ++i) {
        const int j = threadIdx.x + kConvThreads * i;  // output within the tile
        const int t = s0 + j;
        if (t >= S) continue;
        float acc = bv;
#pragma unroll
        for (int k = 0; k < kMaxW; ++k)
            if (k < W) acc = fmaf(wk[k], xs[j + k], acc);  // xs[j + k] is x[t - (W-1) + k]
        if (silu) acc = acc / (1.f + expf(-acc));
        st_io<IO>(out, row + t, acc);
    }
}

template <int IO>
__global__ void __launch_bounds__(256)
gated_rmsnorm_kernel(long long rows, int D, int groups, float eps, const void *x, const void *z,
                     const float *__restrict__ w, void *out) {
    const long long wid = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);  // (row, group)
    const int lane = threadIdx.x & 31;
    if (wid >= rows * groups) return;
    const long long r = wid / groups;
    const int g = (int)(wid % groups);
    const int gs = D / groups;
    const size_t base = (size_t)r * D + (size_t)g * gs;
    float ss = 0.f;
    for (int i = lane; i < gs; i += 32) {
        const float zv = ld_io<IO>(z, base + i);
        const float v = ld_io<IO>(x, base + i) * (zv / (1.f + expf(-zv)));
        ss = fmaf(v, v, ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float inv = rsqrtf(ss / (float)gs + eps);
    for (int i = lane; i < gs; i += 32) {
        const float zv = ld_io<IO>(z, base + i);
        const float v = ld_io<IO>(x, base + i) * (zv / (1.f + expf(-zv)));
        st_io<IO>(out, base + i, v * inv * __ldg(w + g * gs + i));
    }
}

}  // namespace

cudaError_t launch_causal_conv1d(int B, int D, int S, int W, int io, const void *x, const float *w,
                                 const float *bias, int silu, void *out, cudaStream_t s) {
    const dim3 grid((unsigned)((S + kConvTile - 1) / kConvTile), (unsigned)D, (unsigned)B);
    switch (io) {
        case IO_F32: causal_conv1d_kernel<IO_F32><<<grid, kConvThreads, 0, s>>>(S, D, W, x, w, bias, silu, out); break;
        case IO_F16: causal_conv1d_kernel<IO_F16><<<grid, kConvThreads, 0, s>>>(S, D, W, x, w, bias, silu, out); break;
        case IO_BF16: causal_conv1d_kernel<IO_BF16><<<grid, kConvThreads, 0, s>>>(S, D, W, x, w, bias, silu, out); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_gated_rmsnorm(long long rows, int D, int groups, float eps, int io, const void *x, const void *z,
                                 const float *w, void *out, cudaStream_t s) {
    const long long warps = rows * groups;
    const unsigned blocks = (unsigned)((warps + 7) / 8);
    switch (io) {
        case IO_F32: gated_rmsnorm_kernel<IO_F32><<<blocks, 256, 0, s>>>(rows, D, groups, eps, x, z, w, out); break;
        case IO_F16: gated_rmsnorm_kernel<IO_F16><<<blocks, 256, 0, s>>>(rows, D, groups, eps, x, z, w, out); break;
        case IO_BF16: gated_rmsnorm_kernel<IO_BF16><<<blocks, 256, 0, s>>>(rows, D, groups, eps, x, z, w, out); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace ssd
