// decode.cu -- one recurrent step of the SSD for a single new token per
// sequence, continuing from a carried state: the "final_state for the decode
// stage" use of the ops-transformer MambaV2 article (section 4.4,
// chunk_state_passing outputs).  For every (b, h), g = h / (H/G):
//
//   d      = clamp(softplus(dt[b,h] + dt_bias[h]))
//   S[p,:] = exp(d A[h]) S[p,:] + d x[b,h,p] B[b,g,:]       (in place, fp32)
//   y[p]   = (S[p,:] . C[b,g,:] + D[h] x[b,h,p]) * silu(z[b,h,p])
//
// All arithmetic is fp32 on the CUDA cores: the step reads and writes the
// [P,N] state once and does 4 flops per state element, so it is bound by HBM.
// One CTA of 128 threads per (b, h).  When N is 4, 8, ..., 128 the state is
// moved as float4: thread t owns float4 number t + 128 k of the [P,N] block
// (so a warp covers whole consecutive rows, 512 contiguous bytes per access),
// issues all its loads before any arithmetic, and a row's dot product with C
// is a shuffle reduction over the N/4 lanes holding that row.  Other N take a
// scalar kernel (warp per row, lane per column).
#include "ssd_internal.cuh"

namespace ssd {

namespace {

constexpr int kDecodeThreads = 128;
constexpr int kMaxNPerLane = 4;  // N <= 128

template <int IO>
__global__ void __launch_bounds__(kDecodeThreads)
decode_step_kernel(DecodeParams p) {
    const int bh = blockIdx.x;
    const int b = bh / p.H, h = bh % p.H;
    const int g = h / (p.H / p.G);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    float u = p.dt[bh];
    if (p.dt_bias) u += __ldg(p.dt_bias + h);
    float d = p.dt_softplus ? softplus_f(u) : u;
    if (p.has_limit) d = fminf(fmaxf(d, p.dt_min), p.dt_max);
    const float a = expf(d * __ldg(p.A + h));
    const float Dh = p.D ? __ldg(p.D + h) : 0.f;

    // this lane's columns of B and C
    float Bv[kMaxNPerLane], Cv[kMaxNPerLane];
    const size_t bc0 = ((size_t)b * p.G + g) * p.N;
#pragma unroll
    for (int j = 0; j < kMaxNPerLane; ++j) {
        const int n = lane + 32 * j;
        Bv[j] = n < p.N ? ld_io<IO>(p.Bm, bc0 + n) : 0.f;
        Cv[j] = n < p.N ? ld_io<IO>(p.Cm, bc0 + n) : 0.f;
    }

    float *S = p.state + (size_t)bh * p.P * p.N;
    const size_t xr0 = (size_t)bh * p.P;
    for (int row = warp; row < p.P; row += kDecodeThreads / 32) {
        const float xv = ld_io<IO>(p.x, xr0 + row);
        const float dx = d * xv;
        float *Sr = S + (size_t)row * p.N;
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < kMaxNPerLane; ++j) {
            const int n = lane + 32 * j;
            if (n < p.N) {
                const float s = fmaf(a, Sr[n], dx * Bv[j]);
                Sr[n] = s;
                acc = fmaf(s, Cv[j], acc);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) {
            float yv = acc;
            if (p.D) yv = fmaf(Dh, xv, yv);
            if (p.z) yv *= silu_f(ld_io<IO>(p.z, xr0 + row));
            st_io<IO>(p.y, xr0 + row, yv);
        }
    }
}

// Vectorised step for N = 4 * LPR, LPR (lanes per row) a power of two <= 32.
template <int IO, int LPR>
__global__ void __launch_bounds__(kDecodeThreads)
decode_step_vec_kernel(DecodeParams p) {
    constexpr int kBatch = 8;  // float4 per thread held at once
    const int bh = blockIdx.x;
    const int b = bh / p.H, h = bh % p.H;
    const int g = h / (p.H / p.G);
    const int t = threadIdx.x;

    float u = p.dt[bh];
    if (p.dt_bias) u += __ldg(p.dt_bias + h);
    float d = p.dt_softplus ? softplus_f(u) : u;
    if (p.has_limit) d = fminf(fmaxf(d, p.dt_min), p.dt_max);
    const float a = expf(d * __ldg(p.A + h));
    const float Dh = p.D ? __ldg(p.D + h) : 0.f;

    // the thread's four columns never change: (t + 128 k) % LPR == t % LPR
    const int c4 = t % LPR;
    const size_t bc0 = ((size_t)b * p.G + g) * p.N + 4 * c4;
    float Bv[4], Cv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        Bv[e] = ld_io<IO>(p.Bm, bc0 + e);
        Cv[e] = ld_io<IO>(p.Cm, bc0 + e);
    }

    float4 *S = reinterpret_cast<float4 *>(p.state + (size_t)bh * p.P * p.N);
    const size_t xr0 = (size_t)bh * p.P;
    const int total4 = p.P * LPR;  // float4 in the [P,N] block
    for (int base = 0; base < total4; base += kDecodeThreads * kBatch) {
        float4 sv[kBatch];
        float xv[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {  // every load first
            const int f = base + t + kDecodeThreads * k;
            if (f < total4) {
                sv[k] = S[f];
                xv[k] = ld_io<IO>(p.x, xr0 + f / LPR);
            }
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int f = base + t + kDecodeThreads * k;
            const bool in = f < total4;  // uniform across a row's LPR lanes
            float acc = 0.f;
            if (in) {
                const float dx = d * xv[k];
                float4 s4 = sv[k];
                s4.x = fmaf(a, s4.x, dx * Bv[0]);
                s4.y = fmaf(a, s4.y, dx * Bv[1]);
                s4.z = fmaf(a, s4.z, dx * Bv[2]);
                s4.w = fmaf(a, s4.w, dx * Bv[3]);
                S[f] = s4;
                acc = s4.x * Cv[0];
                acc = fmaf(s4.y, Cv[1], acc);
                acc = fmaf(s4.z, Cv[2], acc);
                acc = fmaf(s4.w, Cv[3], acc);
            }
#pragma unroll
            for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (in && c4 == 0) {
                const int row = f / LPR;
                float yv = acc;
                if (p.D) yv = fmaf(Dh, xv[k], yv);
                if (p.z) yv *= silu_f(ld_io<IO>(p.z, xr0 + row));
                st_io<IO>(p.y, xr0 + row, yv);
            }
        }
    }
}

template <int IO>
cudaError_t launch_io(const DecodeParams &p, cudaStream_t s) {
    const dim3 grid((unsigned)(p.B * p.H));
    switch (p.N) {
        case 4: decode_step_vec_kernel<IO, 1><<<grid, kDecodeThreads, 0, s>>>(p); break;
        case 8: decode_step_vec_kernel<IO, 2><<<grid, kDecodeThreads, 0, s>>>(p); break;
        case 16: decode_step_vec_kernel<IO, 4><<<grid, kDecodeThreads, 0, s>>>(p); break;
        case 32: decode_step_vec_kernel<IO, 8><<<grid, kDecodeThreads, 0, s>>>(p); break;
        case 64: decode_step_vec_kernel<IO, 16><<<grid, kDecodeThreads, 0, s>>>(p); break;
        case 128: decode_step_vec_kernel<IO, 32><<<grid, kDecodeThreads, 0, s>>>(p); break;
        default: decode_step_kernel<IO><<<grid, kDecodeThreads, 0, s>>>(p); break;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_step(const DecodeParams &p, int io, cudaStream_t s) {
    // the float4 kernels need a 16-byte aligned state; any other takes the scalar kernel
    const bool vec = (reinterpret_cast<uintptr_t>(p.state) % 16) == 0;
    const dim3 grid((unsigned)(p.B * p.H));
    switch (io) {
        case IO_F32:
            if (vec) return launch_io<IO_F32>(p, s);
            decode_step_kernel<IO_F32><<<grid, kDecodeThreads, 0, s>>>(p);
            break;
        case IO_F16:
            if (vec) return launch_io<IO_F16>(p, s);
            decode_step_kernel<IO_F16><<<grid, kDecodeThreads, 0, s>>>(p);
            break;
        case IO_BF16:
            if (vec) return launch_io<IO_BF16>(p, s);
            decode_step_kernel<IO_BF16><<<grid, kDecodeThreads, 0, s>>>(p);
            break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace ssd
