// chunk_state.cu -- step 2 of the chunked SSD forward (ops-transformer
// MambaV2 article, section 4.3 "mamba2_chunk_state"): the state each chunk
// produces from a zero start,
//     states[b,k,h,p,n] = sum_i w_i x[b,kQ+i,h,p] B[b,kQ+i,g,n],
//     w_i = exp(cs[k,Q-1] - cs[k,i]) * dtp[k,i]   (exponent <= 0: no overflow).
//
// CUDA-core fp32 version (the exact plan): one CTA per (chunk, batch*head),
// 256 threads as a 16 x 16 grid over (p, n), each owning a strided
// (P/16) x (N/16) block of the [P,N] output.  Tokens stream through shared
// memory 32 at a time.  Grid: x = batch*head, y = chunk.  MT (4 or 8) bounds
// the block at compile time, so P, N <= 64 issue no idle multiply-adds; with
// MT = 4 a thread owns the consecutive p = 4 tp .. 4 tp + 3, n = 4 tn .. 4 tn + 3
// and reads each token's operands as two float4 (one broadcast per 16 lanes).
#include "ssd_internal.cuh"

namespace ssd {

namespace {

constexpr int kThreads = 256;
constexpr int kTok = 32;
constexpr int kMaxDim = 128;

template <int IO, int MT>
__global__ void __launch_bounds__(kThreads)
chunk_state_kernel(Params p, const float *__restrict__ dtp, const float *__restrict__ cs,
                   float *__restrict__ states) {
    __shared__ __align__(16) float xs[kTok][kMaxDim];
    __shared__ __align__(16) float bs[kTok][kMaxDim];
    __shared__ float w_s[kTok];
    const int k = blockIdx.y;
    const int bh = blockIdx.x;
    const int b = bh / p.H, h = bh % p.H, g = h / p.hpg;
    const int P = p.P, N = p.N, Q = p.Q, L = p.L;
    const int PT = P >> 4, NT = N >> 4;
    const int tn = threadIdx.x & 15, tp = threadIdx.x >> 4;
    const size_t crow = (((size_t)b * p.H + h) * p.nchunks + k) * Q;
    const float cs_last = __ldg(cs + crow + Q - 1);

    float acc[MT][MT];
#pragma unroll
    for (int a = 0; a < MT; ++a)
#pragma unroll
        for (int c = 0; c < MT; ++c) acc[a][c] = 0.f;

    for (int i0 = 0; i0 < Q; i0 += kTok) {
        const int ntok = min(kTok, Q - i0);
        if (threadIdx.x < kTok) {
            const int i = i0 + threadIdx.x;
            float w = 0.f;
            if (threadIdx.x < ntok && k * Q + i < L)
                w = expf(cs_last - __ldg(cs + crow + i)) * __ldg(dtp + crow + i);
            w_s[threadIdx.x] = w;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < kTok * P; e += kThreads) {
            const int i = e / P, pp = e % P;
            const int t = k * Q + i0 + i;
            float v = 0.f;
            if (i < ntok && t < L) v = ld_io<IO>(p.x, (((size_t)b * L + t) * p.H + h) * P + pp) * w_s[i];
            xs[i][pp] = v;
        }
        for (int e = threadIdx.x; e < kTok * N; e += kThreads) {
            const int i = e / N, n = e % N;
            const int t = k * Q + i0 + i;
            float v = 0.f;
            if (i < ntok && t < L) v = ld_io<IO>(p.Bm, (((size_t)b * L + t) * p.G + g) * N + n);
            bs[i][n] = v;
        }
        __syncthreads();
        for (int i = 0; i < ntok; ++i) {
            float xv[MT], bv[MT];
            if constexpr (MT == 4) {
                const float4 x4 = *reinterpret_cast<const float4 *>(&xs[i][4 * tp]);
                const float4 b4 = *reinterpret_cast<const float4 *>(&bs[i][4 * tn]);
                xv[0] = x4.x; xv[1] = x4.y; xv[2] = x4.z; xv[3] = x4.w;
                bv[0] = b4.x; bv[1] = b4.y; bv[2] = b4.z; bv[3] = b4.w;
            } else {
#pragma unroll
                for (int a = 0; a < MT; ++a) xv[a] = (a < PT) ? xs[i][tp + 16 * a] : 0.f;
#pragma unroll
                for (int c = 0; c < MT; ++c) bv[c] = (c < NT) ? bs[i][tn + 16 * c] : 0.f;
            }
#pragma unroll
            for (int a = 0; a < MT; ++a)
#pragma unroll
                for (int c = 0; c < MT; ++c) acc[a][c] = fmaf(xv[a], bv[c], acc[a][c]);
        }
        __syncthreads();
    }

    float *out = states + ((((size_t)b * p.nchunks + k) * p.H + h) * P) * N;
    if constexpr (MT == 4) {  // rows 4 tp + a, columns 4 tn .. 4 tn + 3 (beyond P or N: not stored)
#pragma unroll
        for (int a = 0; a < 4; ++a)
            if (4 * tp + a < P && 4 * tn < N)
                *reinterpret_cast<float4 *>(out + (size_t)(4 * tp + a) * N + 4 * tn) =
                    make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
    } else {
#pragma unroll
        for (int a = 0; a < MT; ++a)
#pragma unroll
            for (int c = 0; c < MT; ++c)
                if (a < PT && c < NT) out[(size_t)(tp + 16 * a) * N + tn + 16 * c] = acc[a][c];
    }
}

// chunk, P, N <= 64: the chunk's tokens in one pass.  Every global load is
// issued first (thread: column tid % 64 of rows tid / 64 + 4 q, coalesced),
// then x is scaled by its token's weight into shared memory and the same
// 4 x 4 float4 tiles as above accumulate over the tokens.
template <int IO>
__global__ void __launch_bounds__(kThreads)
chunk_state64_kernel(Params p, const float *__restrict__ dtp, const float *__restrict__ cs,
                     float *__restrict__ states) {
    constexpr int kM = 64;
    __shared__ __align__(16) float xs[kM][kM];  // w_i x_i, [token][p]
    __shared__ __align__(16) float bs[kM][kM];  // B_i, [token][n]
    __shared__ float w_s[kM];
    const int k = blockIdx.y, bh = blockIdx.x, tid = threadIdx.x;
    const int b = bh / p.H, h = bh % p.H, g = h / p.hpg;
    const int P = p.P, N = p.N, Q = p.Q, L = p.L;
    const size_t crow = (((size_t)b * p.H + h) * p.nchunks + k) * Q;
    if (tid < kM) {
        const int i = tid;
        float w = 0.f;
        if (i < Q && k * Q + i < L) w = expf(__ldg(cs + crow + Q - 1) - __ldg(cs + crow + i)) * __ldg(dtp + crow + i);
        w_s[i] = w;
    }
    constexpr int kPer = kM * kM / kThreads;  // 16
    const int col = tid & (kM - 1), r0 = tid >> 6;
    float rx[kPer], rb[kPer];
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        const int i = r0 + 4 * q, t = k * Q + i;
        const bool in = i < Q && t < L;
        rx[q] = in && col < P ? ld_io<IO>(p.x, (((size_t)b * L + t) * p.H + h) * P + col) : 0.f;
        rb[q] = in && col < N ? ld_io<IO>(p.Bm, (((size_t)b * L + t) * p.G + g) * N + col) : 0.f;
    }
    __syncthreads();  // w_s
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        const int i = r0 + 4 * q;
        xs[i][col] = rx[q] * w_s[i];
        bs[i][col] = rb[q];
    }
    __syncthreads();
    const int tn = tid & 15, tp = tid >> 4;
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[a][c] = 0.f;
#pragma unroll 8
    for (int i = 0; i < Q; ++i) {
        const float4 x4 = *reinterpret_cast<const float4 *>(&xs[i][4 * tp]);
        const float4 b4 = *reinterpret_cast<const float4 *>(&bs[i][4 * tn]);
        const float xv[4] = {x4.x, x4.y, x4.z, x4.w}, bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[a][c] = fmaf(xv[a], bv[c], acc[a][c]);
    }
    float *out = states + ((((size_t)b * p.nchunks + k) * p.H + h) * P) * N;
#pragma unroll
    for (int a = 0; a < 4; ++a)
        if (4 * tp + a < P && 4 * tn < N)
            *reinterpret_cast<float4 *>(out + (size_t)(4 * tp + a) * N + 4 * tn) =
                make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
}

}  // namespace

cudaError_t launch_chunk_state(const Params &p, int io, const float *dtp, const float *cs,
                               float *states, cudaStream_t s) {
    if (p.P > kMaxDim || p.N > kMaxDim || (p.P & 15) || (p.N & 15)) return cudaErrorInvalidValue;
    dim3 grid(p.B * p.H, p.nchunks);
    // the float4 stores of the 4-wide variants need a 16-byte aligned output
    const bool small = p.P <= 64 && p.N <= 64 && reinterpret_cast<uintptr_t>(states) % 16 == 0;
    if (small && p.Q <= 64) {
        switch (io) {
            case IO_F32: chunk_state64_kernel<IO_F32><<<grid, kThreads, 0, s>>>(p, dtp, cs, states); break;
            case IO_F16: chunk_state64_kernel<IO_F16><<<grid, kThreads, 0, s>>>(p, dtp, cs, states); break;
            case IO_BF16: chunk_state64_kernel<IO_BF16><<<grid, kThreads, 0, s>>>(p, dtp, cs, states); break;
            default: return cudaErrorInvalidValue;
        }
        return cudaGetLastError();
    }
#define SSD_STATE_LAUNCH(IOV)                                                                  \
    if (small) chunk_state_kernel<IOV, 4><<<grid, kThreads, 0, s>>>(p, dtp, cs, states);       \
    else chunk_state_kernel<IOV, 8><<<grid, kThreads, 0, s>>>(p, dtp, cs, states);
    switch (io) {
        case IO_F32: SSD_STATE_LAUNCH(IO_F32) break;
        case IO_F16: SSD_STATE_LAUNCH(IO_F16) break;
        case IO_BF16: SSD_STATE_LAUNCH(IO_BF16) break;
        default: return cudaErrorInvalidValue;
    }
#undef SSD_STATE_LAUNCH
    return cudaGetLastError();
}

}  // namespace ssd
