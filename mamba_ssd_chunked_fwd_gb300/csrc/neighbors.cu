// neighbors.cu -- the two operators around the SSD on the pages
// (ops-transformer MambaV2 article, sections 1.4, 4.1 and 4.6):
//
//   causal conv1d + SiLU   out[b,d,t] = silu(bias[d] + sum_k w[d,k] x[b,d,t-(W-1)+k])
//                          (depthwise along the sequence, x = 0 before t = 0)
//   gated RMSNorm          v = x * silu(z);  out = v / sqrt(mean_group(v^2) + eps) * w
//                          over `groups` runs of D/groups consecutive channels
//
// Both are HBM-bound elementwise-plus-reduction passes, fp32 arithmetic.  The
// conv1d also exists for token-major activations ([B, S, C], the layout of a
// Mamba-2 block's x, B and C), which the SSD forward uses when it runs the
// convolution in front of itself outside the fused kernel.
//   conv1d: one CTA per (1024-token tile, 4 channels, batch); each channel's
//           tile and its W-1 token halo go through shared memory, loads and
//           stores are coalesced along the sequence (16 bytes per thread when
//           fp32 rows allow it), 16 KB of loads in flight per CTA.
//   RMSNorm: one warp per (row, group); the group's values stay in registers
//           (up to 512 channels per group; wider groups take a second pass
//           from L1/L2) and its sum of squares is a warp reduction.
#include "ssd_internal.cuh"

namespace ssd {

namespace {

constexpr int kConvThreads = 256;
constexpr int kConvPer = 4;  // consecutive outputs per thread and channel
constexpr int kConvTile = kConvThreads * kConvPer;
constexpr int kConvRows = 4;  // channels per CTA
constexpr int kMaxW = 8;
constexpr int kPad = 8;       // the halo slot in front of each channel's tile (>= W-1, keeps float4 alignment)

// VEC: fp32 rows with S % 4 == 0 (16-byte aligned rows): float4 loads and stores,
// the taps in KT (4 or 8, >= W) slots.
template <int IO, bool VEC, int KT = kMaxW>
__global__ void __launch_bounds__(kConvThreads)
causal_conv1d_kernel(int S, int D, int W, const void *x, const float *__restrict__ w, const float *__restrict__ bias,
                     int silu, void *out) {
    __shared__ __align__(16) float xs[kConvRows][kPad + kConvTile];
    const int s0 = blockIdx.x * kConvTile, d0 = blockIdx.y * kConvRows, b = blockIdx.z;
    const int halo = W - 1;
    // tiles: xs[r][kPad + i] = x[t = s0 + i], xs[r][kPad - m] = x[s0 - m] for m <= W-1 (halo), 0 before
#pragma unroll
    for (int r = 0; r < kConvRows; ++r) {
        const int d = d0 + r;
        if (d >= D) break;
        const size_t row = ((size_t)b * D + d) * S;
        if (VEC) {
            const int t = s0 + 4 * threadIdx.x;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < S) v = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(x) + row + t));
            *reinterpret_cast<float4 *>(&xs[r][kPad + 4 * threadIdx.x]) = v;
        } else {
#pragma unroll
            for (int i = 0; i < kConvPer; ++i) {
                const int j = threadIdx.x + kConvThreads * i, t = s0 + j;
                xs[r][kPad + j] = t < S ? ld_io<IO>(x, row + t) : 0.f;
            }
        }
        if (threadIdx.x < kPad) {  // the whole pad: the halo, zeros in front of it (read with zero taps)
            const int m = threadIdx.x, t = s0 - kPad + m;
            xs[r][m] = (m >= kPad - halo && t >= 0) ? ld_io<IO>(x, row + t) : 0.f;
        }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kConvRows; ++r) {
        const int d = d0 + r;
        if (d >= D) break;
        const size_t row = ((size_t)b * D + d) * S;
        const float bv = bias ? __ldg(bias + d) : 0.f;
        float o[kConvPer];
        if (VEC) {
            // The thread's 4 consecutive outputs need x[t - (W-1) .. t + 3]: the (KT + 4) / 4
            // aligned float4 from xs[r][4 tid + 8 - KT] on (bank-conflict free).  The taps sit
            // right-aligned in KT slots (wr[j] = w[j - (KT - W)], zeros before), so output i is
            // sum_j wr[j] win[1 + i + j] with compile-time indices.
            float wr[KT];
#pragma unroll
            for (int j = 0; j < KT; ++j) wr[j] = j >= KT - W ? __ldg(w + (size_t)d * W + j - (KT - W)) : 0.f;
            float win[KT + 4];
#pragma unroll
            for (int q = 0; q < (KT + 4) / 4; ++q) {
                const float4 v = *reinterpret_cast<const float4 *>(&xs[r][4 * threadIdx.x + kPad - KT + 4 * q]);
                win[4 * q] = v.x; win[4 * q + 1] = v.y; win[4 * q + 2] = v.z; win[4 * q + 3] = v.w;
            }
#pragma unroll
            for (int i = 0; i < kConvPer; ++i) {
                float acc = bv;
#pragma unroll
                for (int j = 0; j < KT; ++j) acc = fmaf(wr[j], win[1 + i + j], acc);
                if (silu) acc = __fdividef(acc, 1.f + __expf(-acc));  // a few ulp; 0 below -87 (the limit)
                o[i] = acc;
            }
        } else {
            float wk[kMaxW];
#pragma unroll
            for (int k = 0; k < kMaxW; ++k) wk[k] = k < W ? __ldg(w + (size_t)d * W + k) : 0.f;
#pragma unroll
            for (int i = 0; i < kConvPer; ++i) {
                const int j = threadIdx.x + kConvThreads * i;  // outputs strided by the block
                float acc = bv;
#pragma unroll
                for (int k = 0; k < kMaxW; ++k)
                    if (k < W) acc = fmaf(wk[k], xs[r][kPad - halo + j + k], acc);  // x[t - (W-1) + k]
                if (silu) acc = acc / (1.f + expf(-acc));
                o[i] = acc;
            }
        }
        if (VEC) {
            const int t = s0 + 4 * threadIdx.x;
            if (t < S)
                *reinterpret_cast<float4 *>(static_cast<float *>(out) + row + t) = make_float4(o[0], o[1], o[2], o[3]);
        } else {
#pragma unroll
            for (int i = 0; i < kConvPer; ++i) {
                const int t = s0 + threadIdx.x + kConvThreads * i;
                if (t < S) st_io<IO>(out, row + t, o[i]);
            }
        }
    }
}

// PER: values each lane keeps in registers (PER * 32 >= the group size), 0 for
// groups wider than 512 channels (second pass).  The gate uses the fast
// exponential and division (a few ulp; 0 for z below -87, the limit).
template <int IO, int PER>
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
    if constexpr (PER > 0) {
        float v[PER];
#pragma unroll
        for (int k = 0; k < PER; ++k) {  // every load first
            const int i = lane + 32 * k;
            v[k] = 0.f;
            if (i < gs) {
                const float zv = ld_io<IO>(z, base + i);
                v[k] = ld_io<IO>(x, base + i) * __fdividef(zv, 1.f + __expf(-zv));
            }
        }
#pragma unroll
        for (int k = 0; k < PER; ++k) ss = fmaf(v[k], v[k], ss);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float inv = rsqrtf(ss / (float)gs + eps);
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            const int i = lane + 32 * k;
            if (i < gs) st_io<IO>(out, base + i, v[k] * inv * __ldg(w + g * gs + i));
        }
    } else {
        for (int i = lane; i < gs; i += 32) {
            const float zv = ld_io<IO>(z, base + i);
            const float v = ld_io<IO>(x, base + i) * __fdividef(zv, 1.f + __expf(-zv));
            ss = fmaf(v, v, ss);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float inv = rsqrtf(ss / (float)gs + eps);
        for (int i = lane; i < gs; i += 32) {  // second pass, from L1/L2
            const float zv = ld_io<IO>(z, base + i);
            const float v = ld_io<IO>(x, base + i) * __fdividef(zv, 1.f + __expf(-zv));
            st_io<IO>(out, base + i, v * inv * __ldg(w + g * gs + i));
        }
    }
}

// Groups of 32, 64 or 128 channels: one warp covers GPW groups (256 channels,
// PER = group size / 32 values per lane and group), so that a warp keeps 2 KB
// of loads in flight; each group's sum of squares reduces over the warp as in
// the kernel above (per-lane partial, then the xor tree).
template <int IO, int PER, int GPW>
__global__ void __launch_bounds__(256)
gated_rmsnorm_multi_kernel(long long rows, int D, int groups, float eps, const void *x, const void *z,
                           const float *__restrict__ w, void *out) {
    constexpr int kGs = 32 * PER, kVpl = PER * GPW;
    const long long wid = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);  // (row, block of GPW groups)
    const int lane = threadIdx.x & 31;
    const int spans = groups / GPW;
    if (wid >= rows * spans) return;
    const long long r = wid / spans;
    const int g0 = (int)(wid % spans) * GPW;
    const size_t base = (size_t)r * D + (size_t)g0 * kGs;
    float v[kVpl];
#pragma unroll
    for (int k = 0; k < kVpl; ++k) {  // every load first
        const float zv = ld_io<IO>(z, base + lane + 32 * k);
        v[k] = ld_io<IO>(x, base + lane + 32 * k) * __fdividef(zv, 1.f + __expf(-zv));
    }
    float inv[GPW];
#pragma unroll
    for (int j = 0; j < GPW; ++j) {
        float ss = 0.f;
#pragma unroll
        for (int k = j * PER; k < (j + 1) * PER; ++k) ss = fmaf(v[k], v[k], ss);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        inv[j] = rsqrtf(ss / (float)kGs + eps);
    }
#pragma unroll
    for (int k = 0; k < kVpl; ++k) {
        const int i = lane + 32 * k;
        st_io<IO>(out, base + i, v[k] * inv[k / PER] * __ldg(w + (size_t)g0 * kGs + i));
    }
}

// 4 consecutive channels of one token row as floats (16 bytes fp32, 8 bytes 16-bit).
template <int IO>
__device__ __forceinline__ void load4(const void *base, size_t i, float (&v)[4]) {
    if (IO == IO_F32) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(base) + i));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    } else {
        const uint2 u = __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(base) + i));
        const uint32_t wd[2] = {u.x, u.y};
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float2 f;
            if (IO == IO_BF16) f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&wd[q]));
            else f = __half22float2(*reinterpret_cast<const __half2 *>(&wd[q]));
            v[2 * q] = f.x; v[2 * q + 1] = f.y;
        }
    }
}

template <int IO>
__device__ __forceinline__ void store4(void *base, size_t i, const float (&v)[4]) {
    if (IO == IO_F32) {
        *reinterpret_cast<float4 *>(static_cast<float *>(base) + i) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
        uint2 u;
        if (IO == IO_BF16) {
            __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
            u.x = *reinterpret_cast<uint32_t *>(&a); u.y = *reinterpret_cast<uint32_t *>(&b);
        } else {
            __half2 a = __floats2half2_rn(v[0], v[1]), b = __floats2half2_rn(v[2], v[3]);
            u.x = *reinterpret_cast<uint32_t *>(&a); u.y = *reinterpret_cast<uint32_t *>(&b);
        }
        *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(base) + i) = u;
    }
}

// Token-major causal conv1d + SiLU, the layout of a Mamba-2 block's x, B and C:
//   out[b,t,c] = silu(bias[c] + sum_{k<W} w[c,k] x[b,t-(W-1)+k,c]).
// A thread owns 4 consecutive channels over kTokRun consecutive tokens: it
// reads the 3 tokens before its run once and slides the window in registers.
// A warp's 32 threads cover 128 channels of one token row, so every load and
// store is coalesced.  Taps sit right-aligned in 4 slots (slot 3 = the current
// token), so every register index is a constant.
constexpr int kTokRun = 16;
template <int IO>
__global__ void __launch_bounds__(256)
conv_tokens_kernel(int S, int C, int W, const void *x, const float *__restrict__ w, const float *__restrict__ bias,
                   int silu, void *out) {
    const int c = (blockIdx.x * 256 + threadIdx.x) * 4;
    if (c >= C) return;
    const int t0 = blockIdx.y * kTokRun;
    const size_t row0 = (size_t)blockIdx.z * S;
    float wk[4][4], bj[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int sl = 0; sl < 4; ++sl) {
            const int k = sl - (4 - W);
            wk[sl][j] = k >= 0 ? __ldg(w + (size_t)(c + j) * W + k) : 0.f;
        }
        bj[j] = bias ? __ldg(bias + c + j) : 0.f;
    }
    float win[3][4];  // tokens t-3, t-2, t-1 of the current output token t
#pragma unroll
    for (int m = 0; m < 3; ++m) {
        const int t = t0 - 3 + m;
        if (t >= 0) load4<IO>(x, (row0 + t) * C + c, win[m]);
        else win[m][0] = win[m][1] = win[m][2] = win[m][3] = 0.f;
    }
#pragma unroll 4
    for (int i = 0; i < kTokRun; ++i) {
        const int t = t0 + i;
        if (t >= S) break;
        float v[4], o[4];
        load4<IO>(x, (row0 + t) * C + c, v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float a = bj[j];
            a = fmaf(wk[0][j], win[0][j], a);
            a = fmaf(wk[1][j], win[1][j], a);
            a = fmaf(wk[2][j], win[2][j], a);
            a = fmaf(wk[3][j], v[j], a);
            // 16-bit outputs: the one-MUFU SiLU (its error is below the output's rounding)
            o[j] = !silu ? a : IO == IO_F32 ? silu_fast(a) : silu_tanh(a);
            win[0][j] = win[1][j];
            win[1][j] = win[2][j];
            win[2][j] = v[j];
        }
        store4<IO>(out, (row0 + t) * C + c, o);
    }
}

}  // namespace

cudaError_t launch_conv_tokens(int B, int S, int C, int W, int io, const void *x, const float *w, const float *bias,
                               int silu, void *out, cudaStream_t s) {
    if (C % 4 != 0 || W < 1 || W > 4) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)((C / 4 + 255) / 256), (unsigned)((S + kTokRun - 1) / kTokRun), (unsigned)B);
    switch (io) {
        case IO_F32: conv_tokens_kernel<IO_F32><<<grid, 256, 0, s>>>(S, C, W, x, w, bias, silu, out); break;
        case IO_F16: conv_tokens_kernel<IO_F16><<<grid, 256, 0, s>>>(S, C, W, x, w, bias, silu, out); break;
        case IO_BF16: conv_tokens_kernel<IO_BF16><<<grid, 256, 0, s>>>(S, C, W, x, w, bias, silu, out); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_causal_conv1d(int B, int D, int S, int W, int io, const void *x, const float *w,
                                 const float *bias, int silu, void *out, cudaStream_t s) {
    const dim3 grid((unsigned)((S + kConvTile - 1) / kConvTile), (unsigned)((D + kConvRows - 1) / kConvRows),
                    (unsigned)B);
    const bool vec = S % 4 == 0 && reinterpret_cast<uintptr_t>(x) % 16 == 0 && reinterpret_cast<uintptr_t>(out) % 16 == 0;
    switch (io) {
        case IO_F32:
            if (vec && W <= 4)
                causal_conv1d_kernel<IO_F32, true, 4><<<grid, kConvThreads, 0, s>>>(S, D, W, x, w, bias, silu, out);
            else if (vec)
                causal_conv1d_kernel<IO_F32, true, 8><<<grid, kConvThreads, 0, s>>>(S, D, W, x, w, bias, silu, out);
            else causal_conv1d_kernel<IO_F32, false><<<grid, kConvThreads, 0, s>>>(S, D, W, x, w, bias, silu, out);
            break;
        case IO_F16: causal_conv1d_kernel<IO_F16, false><<<grid, kConvThreads, 0, s>>>(S, D, W, x, w, bias, silu, out); break;
        case IO_BF16: causal_conv1d_kernel<IO_BF16, false><<<grid, kConvThreads, 0, s>>>(S, D, W, x, w, bias, silu, out); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_gated_rmsnorm(long long rows, int D, int groups, float eps, int io, const void *x, const void *z,
                                 const float *w, void *out, cudaStream_t s) {
    const int gs = D / groups;
    const int gpw = (gs == 32 || gs == 64 || gs == 128) ? 256 / gs : 1;
    if (gpw > 1 && groups % gpw == 0) {  // several groups per warp
        const long long mwarps = rows * (groups / gpw);
        const unsigned mblocks = (unsigned)((mwarps + 7) / 8);
#define SSD_RMS_MULTI(PER, GPW)                                                                                   \
    switch (io) {                                                                                                 \
        case IO_F32: gated_rmsnorm_multi_kernel<IO_F32, PER, GPW><<<mblocks, 256, 0, s>>>(rows, D, groups, eps, x, z, w, out); break; \
        case IO_F16: gated_rmsnorm_multi_kernel<IO_F16, PER, GPW><<<mblocks, 256, 0, s>>>(rows, D, groups, eps, x, z, w, out); break; \
        case IO_BF16: gated_rmsnorm_multi_kernel<IO_BF16, PER, GPW><<<mblocks, 256, 0, s>>>(rows, D, groups, eps, x, z, w, out); break; \
        default: return cudaErrorInvalidValue;                                                                    \
    }
        if (gs == 32) { SSD_RMS_MULTI(1, 8) }
        else if (gs == 64) { SSD_RMS_MULTI(2, 4) }
        else { SSD_RMS_MULTI(4, 2) }
#undef SSD_RMS_MULTI
        return cudaGetLastError();
    }
    const long long warps = rows * groups;
    const unsigned blocks = (unsigned)((warps + 7) / 8);
#define SSD_RMS_LAUNCH(PER)                                                                                  \
    switch (io) {                                                                                            \
        case IO_F32: gated_rmsnorm_kernel<IO_F32, PER><<<blocks, 256, 0, s>>>(rows, D, groups, eps, x, z, w, out); break; \
        case IO_F16: gated_rmsnorm_kernel<IO_F16, PER><<<blocks, 256, 0, s>>>(rows, D, groups, eps, x, z, w, out); break; \
        case IO_BF16: gated_rmsnorm_kernel<IO_BF16, PER><<<blocks, 256, 0, s>>>(rows, D, groups, eps, x, z, w, out); break; \
        default: return cudaErrorInvalidValue;                                                               \
    }
    if (gs <= 32) { SSD_RMS_LAUNCH(1) }
    else if (gs <= 64) { SSD_RMS_LAUNCH(2) }
    else if (gs <= 128) { SSD_RMS_LAUNCH(4) }
    else if (gs <= 256) { SSD_RMS_LAUNCH(8) }
    else if (gs <= 512) { SSD_RMS_LAUNCH(16) }
    else { SSD_RMS_LAUNCH(0) }
#undef SSD_RMS_LAUNCH
    return cudaGetLastError();
}

}  // namespace ssd
