// chunk_scan.cu -- step 4 of the chunked SSD forward (ops-transformer
// MambaV2 article, section 4.5 "mamba2_chunk_scan"): the output of chunk k
// from the state entering it,
//     y_i = exp(cs_i) * sum_n C[i,n] S_k[p,n]                       (inter-chunk)
//         + sum_{j<=i} (sum_n C[i,n] B[j,n]) exp(cs_i - cs_j) dtp_j x[j,p]  (intra)
//         + D[h] x[i,p],   then  y *= silu(z[i,p]).
// The decay is only ever formed as exp(cs_i - cs_j) with j <= i (exponent
// <= 0), after the causal mask.
//
// CUDA-core fp32 version (the exact plan).  One CTA per (batch*head, chunk,
// tile of 32 tokens); 256 threads as 16 token rows x 16 head-dim lanes, each
// owning 2 x (P/16) outputs.  C of the tile stays in shared memory; the
// state, then B / x tiles of 32 tokens, stream through it.  MT (4 or 8) bounds
// the per-thread outputs at compile time, so P <= 64 issues no idle work.
#include "ssd_internal.cuh"

namespace ssd {

namespace {

constexpr int kThreads = 256;
constexpr int kTI = 32;       // output tokens per CTA
constexpr int kTJ = 32;       // source tokens per step
constexpr int kNC = 16;       // state columns per step of the inter-chunk part
constexpr int kMaxDim = 128;
constexpr int kMaxQ = 256;

struct ScanSmem {
    float cs[kMaxQ];
    float dtp[kMaxQ];
    float C[kTI][kMaxDim + 1];
    union {
        float S[kMaxDim][kNC + 1];
        struct {
            float B[kTJ][kMaxDim + 1];
            float X[kTJ][kMaxDim];
        } bx;
    } u;
    float M[kTI][kTJ + 1];
};

template <int IO, int MT>
__global__ void __launch_bounds__(kThreads)
chunk_scan_kernel(Params p, const float *__restrict__ dtp, const float *__restrict__ cs,
                  const float *__restrict__ states) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ScanSmem &sm = *reinterpret_cast<ScanSmem *>(smem_raw);
    const int bh = blockIdx.x, k = blockIdx.y, i0 = blockIdx.z * kTI;
    const int b = bh / p.H, h = bh % p.H, g = h / p.hpg;
    const int P = p.P, N = p.N, Q = p.Q, L = p.L, H = p.H;
    const int PT = P >> 4;
    const int tp = threadIdx.x & 15, ti = threadIdx.x >> 4;
    const int tok0 = k * Q;  // first token of the chunk
    if (i0 >= Q) return;
    const int nI = min(kTI, Q - i0);
    const size_t crow = (((size_t)b * H + h) * p.nchunks + k) * Q;

    for (int i = threadIdx.x; i < Q; i += kThreads) {
        sm.cs[i] = __ldg(cs + crow + i);
        sm.dtp[i] = __ldg(dtp + crow + i);
    }
    for (int e = threadIdx.x; e < kTI * N; e += kThreads) {
        const int i = e / N, n = e % N;
        const int t = tok0 + i0 + i;
        float v = 0.f;
        if (i < nI && t < L) v = ld_io<IO>(p.Cm, (((size_t)b * L + t) * p.G + g) * N + n);
        sm.C[i][n] = v;
    }

    float acc[2][MT];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int a = 0; a < MT; ++a) acc[m][a] = 0.f;

    // inter-chunk part: C_i . S_k[p, :]
    const float *S = states + ((((size_t)b * p.nchunks + k) * H + h) * P) * N;
    for (int n0 = 0; n0 < N; n0 += kNC) {
        __syncthreads();
        for (int e = threadIdx.x; e < P * kNC; e += kThreads) {
            const int pp = e / kNC, n = e % kNC;
            sm.u.S[pp][n] = __ldg(S + (size_t)pp * N + n0 + n);
        }
        __syncthreads();
#pragma unroll 4
        for (int n = 0; n < kNC; ++n) {
            const float c0 = sm.C[ti][n0 + n], c1 = sm.C[ti + 16][n0 + n];
#pragma unroll
            for (int a = 0; a < MT; ++a) {
                if (a < PT) {
                    const float sv = sm.u.S[tp + 16 * a][n];
                    acc[0][a] = fmaf(c0, sv, acc[0][a]);
                    acc[1][a] = fmaf(c1, sv, acc[1][a]);
                }
            }
        }
    }
    {
        const float e0 = expf(sm.cs[min(i0 + ti, Q - 1)]);
        const float e1 = expf(sm.cs[min(i0 + ti + 16, Q - 1)]);
#pragma unroll
        for (int a = 0; a < MT; ++a) {
            acc[0][a] *= e0;
            acc[1][a] *= e1;
        }
    }

    // intra-chunk part: source tokens j <= i
    const int jend = i0 + nI;  // exclusive
    for (int j0 = 0; j0 < jend; j0 += kTJ) {
        const int nJ = min(kTJ, jend - j0);
        __syncthreads();
        for (int e = threadIdx.x; e < kTJ * N; e += kThreads) {
            const int j = e / N, n = e % N;
            const int t = tok0 + j0 + j;
            float v = 0.f;
            if (j < nJ && t < L) v = ld_io<IO>(p.Bm, (((size_t)b * L + t) * p.G + g) * N + n);
            sm.u.bx.B[j][n] = v;
        }
        for (int e = threadIdx.x; e < kTJ * P; e += kThreads) {
            const int j = e / P, pp = e % P;
            const int t = tok0 + j0 + j;
            float v = 0.f;
            if (j < nJ && t < L) v = ld_io<IO>(p.x, (((size_t)b * L + t) * H + h) * P + pp);
            sm.u.bx.X[j][pp] = v;
        }
        __syncthreads();
        // M[i,j] = (C_i . B_j) * exp(cs_i - cs_j) * dtp_j  for j <= i, else 0
        {
            const int i = threadIdx.x >> 3;  // 0..31
            const int jl = threadIdx.x & 7;
            float cb[4] = {0.f, 0.f, 0.f, 0.f};
            for (int n = 0; n < N; ++n) {
                const float cv = sm.C[i][n];
#pragma unroll
                for (int q = 0; q < 4; ++q) cb[q] = fmaf(cv, sm.u.bx.B[jl + 8 * q][n], cb[q]);
            }
            const int ig = i0 + i;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int jg = j0 + jl + 8 * q;
                float m = 0.f;
                if (jg <= ig && i < nI && jl + 8 * q < nJ)
                    m = cb[q] * expf(sm.cs[ig] - sm.cs[jg]) * sm.dtp[jg];
                sm.M[i][jl + 8 * q] = m;
            }
        }
        __syncthreads();
#pragma unroll 4
        for (int j = 0; j < kTJ; ++j) {
            const float m0 = sm.M[ti][j], m1 = sm.M[ti + 16][j];
#pragma unroll
            for (int a = 0; a < MT; ++a) {
                if (a < PT) {
                    const float xv = sm.u.bx.X[j][tp + 16 * a];
                    acc[0][a] = fmaf(m0, xv, acc[0][a]);
                    acc[1][a] = fmaf(m1, xv, acc[1][a]);
                }
            }
        }
    }

    // epilogue: D skip, z gate, store
    const float Dh = p.D ? __ldg(p.D + h) : 0.f;
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        const int i = ti + 16 * m;
        const int t = tok0 + i0 + i;
        if (i >= nI || t >= L) continue;
        const size_t rowoff = (((size_t)b * L + t) * H + h) * P;
#pragma unroll
        for (int a = 0; a < MT; ++a) {
            if (a >= PT) continue;
            const int pp = tp + 16 * a;
            float v = acc[m][a];
            if (p.D) v = fmaf(Dh, ld_io<IO>(p.x, rowoff + pp), v);
            if (p.z) v *= silu_f(ld_io<IO>(p.z, rowoff + pp));
            st_io<IO>(p.y, rowoff + pp, v);
        }
    }
}

template <int IO, int MT>
cudaError_t run_scan(const Params &p, const float *dtp, const float *cs, const float *states, dim3 grid, size_t smem,
                     cudaStream_t s) {
    const cudaError_t err =
        cudaFuncSetAttribute(chunk_scan_kernel<IO, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    chunk_scan_kernel<IO, MT><<<grid, kThreads, smem, s>>>(p, dtp, cs, states);
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_chunk_scan(const Params &p, int io, const float *dtp, const float *cs,
                              const float *states, cudaStream_t s) {
    if (p.P > kMaxDim || p.N > kMaxDim || (p.P & 15) || (p.N % kNC) || p.Q > kMaxQ)
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(ScanSmem);
    dim3 grid(p.B * p.H, p.nchunks, (p.Q + kTI - 1) / kTI);
    const bool small = p.P <= 64;
    cudaError_t err = cudaSuccess;
    switch (io) {
        case IO_F32: err = small ? run_scan<IO_F32, 4>(p, dtp, cs, states, grid, smem, s)
                                 : run_scan<IO_F32, 8>(p, dtp, cs, states, grid, smem, s); break;
        case IO_F16: err = small ? run_scan<IO_F16, 4>(p, dtp, cs, states, grid, smem, s)
                                 : run_scan<IO_F16, 8>(p, dtp, cs, states, grid, smem, s); break;
        case IO_BF16: err = small ? run_scan<IO_BF16, 4>(p, dtp, cs, states, grid, smem, s)
                                  : run_scan<IO_BF16, 8>(p, dtp, cs, states, grid, smem, s); break;
        default: return cudaErrorInvalidValue;
    }
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace ssd
