// bwd.cu -- the SSD backward (the backward chain named in the "Mamba-2 SSD
// for Ascend NPU" README, "Limitations and roadmap"), chunked like the
// forward (ops-transformer MambaV2 article, sections 4.2-4.5) and run in fp32
// on the CUDA cores.  With S_k the state entering chunk k (recomputed by the
// forward's first three steps), cs the within-chunk cumulative d*A and Q the
// chunk length, the loss L = sum_t dy_t . y_t + <dfinal, final_state> gives:
//
//   adjoint at each chunk end (reverse state passing):
//     G_{c-1} = dfinal,   G_{k-1} = exp(cs_last[k]) G_k + sum_i exp(cs_i) dyp_i (outer) C_i,
//     dh0 = exp(cs_last[0]) G_0 + sum_{i in chunk 0} exp(cs_i) dyp_i (outer) C_i
//   within chunk k (E[i,j] = exp(cs_i - cs_j) for j <= i, else 0;
//     CB = C B^T, DX = dyp x^T, both Q x Q):
//     dx_t = d_t (sum_i E[i,t] CB[i,t] dyp_i + exp(cs_last - cs_t) G_k B_t) + D dyp_t
//     dB_t = d_t (sum_i E[i,t] DX[i,t] C_i + exp(cs_last - cs_t) G_k^T x_t)   (per head; heads of a group summed)
//     dC_i = exp(cs_i) S_k^T dyp_i + sum_j E[i,j] DX[i,j] d_j B_j              (per head; summed)
//     dd_t = x_t . (dx_t - D dyp_t) / d_t + A sum_{s >= t} dcs_s, where
//     dcs_i = exp(cs_i) C_i . (S_k^T dyp_i) + R_i - K_i - w_i
//             + [i = Q-1] (exp(cs_last) <G_k, S_k> + sum_j w_j),
//       v[i,j] = E[i,j] CB[i,j] DX[i,j] d_j, R_i = sum_j v[i,j], K_j = sum_i v[i,j],
//       w_j = exp(cs_last - cs_j) d_j x_j . (G_k B_j)
//     dA += d_t sum_{s >= t} dcs_s,  dD += dyp_t . x_t,
//     ddt_t = dd_t softplus'(dt_t + bias) (0 outside the dt_limit clamp),  dbias += ddt_t
//   and the gate: dyp = dy silu(z), dz = dy (y before the gate) silu'(z).
//
// Every sum runs in a fixed order (no floating atomics): results are bitwise
// reproducible.  Shapes: chunk <= 64, P <= 64, N <= 64.
#include "ssd_internal.cuh"

namespace ssd {

namespace {

constexpr int kThreads = 256;
constexpr int kMax = 64;  // chunk, P, N

// ---- gate: dyp = dy * silu(z),  dz = dy * ypre * silu'(z) ----
template <int IO>
__global__ void bwd_gate_kernel(Params p, const void *dy, const void *ypre, float *dyp, void *dz, size_t count) {
    const size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= count) return;
    const float g = ld_io<IO>(dy, e);
    if (!p.z) {
        dyp[e] = g;
        return;
    }
    const float zv = ld_io<IO>(p.z, e);
    const float sg = 1.f / (1.f + expf(-zv));
    dyp[e] = g * zv * sg;
    st_io<IO>(dz, e, g * ld_io<IO>(ypre, e) * sg * (1.f + zv * (1.f - sg)));
}

// 16 outputs per thread as a 4 x 4 register tile of a 64 x 64 result: rows
// r0 + 16 a, columns c0 + 16 b (r0 = tid / 16, c0 = tid % 16), so that a warp's
// loads of one operand are broadcast and of the other conflict-free (rows of
// 65 floats).  acc[a][b] += sum_k A(r, k) * B(c, k) over k < K.
template <class FA, class FB>
__device__ __forceinline__ void tile4x4(float (&acc)[4][4], int K, int r0, int c0, FA fa, FB fb) {
    for (int k = 0; k < K; ++k) {
        float av[4], bv[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) av[a] = fa(r0 + 16 * a, k);
#pragma unroll
        for (int b = 0; b < 4; ++b) bv[b] = fb(c0 + 16 * b, k);
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(av[a], bv[b], acc[a][b]);
    }
}

__device__ __forceinline__ void zero4x4(float (&acc)[4][4]) {
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
}

// ---- per chunk: sum_i exp(cs_i) dyp_i (outer) C_i  [P,N] ----
template <int IO>
__global__ void __launch_bounds__(kThreads)
bwd_chunk_adjoint_kernel(Params p, const float *__restrict__ cs, const float *__restrict__ dyp,
                         float *__restrict__ adj) {
    __shared__ float ds[kMax][kMax + 1];  // [i][p]
    __shared__ float cc[kMax][kMax + 1];  // [i][n]
    const int k = blockIdx.y, bh = blockIdx.x;
    const int b = bh / p.H, h = bh % p.H, g = h / p.hpg;
    const int P = p.P, N = p.N, Q = p.Q, L = p.L;
    const size_t crow = (((size_t)b * p.H + h) * p.nchunks + k) * Q;
    for (int e = threadIdx.x; e < Q * P; e += kThreads) {
        const int i = e / P, pp = e % P, t = k * Q + i;
        ds[i][pp] = t < L ? dyp[(((size_t)b * L + t) * p.H + h) * P + pp] * expf(__ldg(cs + crow + i)) : 0.f;
    }
    for (int e = threadIdx.x; e < Q * N; e += kThreads) {
        const int i = e / N, n = e % N, t = k * Q + i;
        cc[i][n] = t < L ? ld_io<IO>(p.Cm, (((size_t)b * L + t) * p.G + g) * N + n) : 0.f;
    }
    __syncthreads();
    const int r0 = threadIdx.x >> 4, c0 = threadIdx.x & 15;
    float acc[4][4];
    zero4x4(acc);
    tile4x4(acc, Q, r0, c0, [&](int pp, int i) { return ds[i][pp]; }, [&](int n, int i) { return cc[i][n]; });
    float *out = adj + ((((size_t)b * p.nchunks + k) * p.H + h) * P) * N;
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int pp = r0 + 16 * a, n = c0 + 16 * c;
            if (pp < P && n < N) out[(size_t)pp * N + n] = acc[a][c];
        }
}

// ---- reverse state passing: adj[k] <- G_k (adjoint at the end of chunk k), dh0 ----
// Four consecutive elements per thread; the next chunk's values are loaded
// before the current ones are stored.
__global__ void __launch_bounds__(kThreads)
bwd_state_passing_kernel(Params p, const float *__restrict__ cs, const float *__restrict__ dfinal,
                         float *__restrict__ adj, float *__restrict__ dh0) {
    const int bh = blockIdx.x;
    const int b = bh / p.H, h = bh % p.H;
    const int PN = p.P * p.N;
    const int e = (blockIdx.y * kThreads + threadIdx.x) * 4;
    if (e >= PN) return;
    const int c = p.nchunks;
    const size_t crow = ((size_t)b * p.H + h) * c;
    const size_t kstride = (size_t)p.H * PN;
    float *base = adj + (((size_t)b * c) * p.H + h) * PN + e;
    float4 gs = make_float4(0.f, 0.f, 0.f, 0.f);
    if (dfinal) gs = __ldg(reinterpret_cast<const float4 *>(dfinal + ((size_t)b * p.H + h) * PN + e));
    float4 nxt = *reinterpret_cast<const float4 *>(base + (size_t)(c - 1) * kstride);
    for (int k = c - 1; k >= 0; --k) {
        const float4 loc = nxt;
        if (k > 0) nxt = *reinterpret_cast<const float4 *>(base + (size_t)(k - 1) * kstride);
        *reinterpret_cast<float4 *>(base + (size_t)k * kstride) = gs;
        const float a = expf(__ldg(cs + (crow + k) * p.Q + p.Q - 1));
        gs.x = fmaf(a, gs.x, loc.x);
        gs.y = fmaf(a, gs.y, loc.y);
        gs.z = fmaf(a, gs.z, loc.z);
        gs.w = fmaf(a, gs.w, loc.w);
    }
    if (dh0) *reinterpret_cast<float4 *>(dh0 + ((size_t)b * p.H + h) * PN + e) = gs;
}

// ---- within one chunk: dx, dB, dC (per head), ddt, and partial dA, dD, dbias ----
struct ChunkSmem {
    float x[kMax][kMax + 1], dy[kMax][kMax + 1], B[kMax][kMax + 1], C[kMax][kMax + 1];
    float S[kMax][kMax + 1], Gm[kMax][kMax + 1];
    float CB[kMax][kMax + 1], DX[kMax][kMax + 1], V[kMax][kMax + 1];
    float T[kMax][kMax + 1];  // dxs, then S^T dyp
    float GB[kMax][kMax + 1];
    float cs[kMax], d[kMax], ecs[kMax], el[kMax], dd1[kMax], w[kMax], z[kMax], dcs[kMax], u[kMax];
    float red[kThreads];
};

template <int IO>
__global__ void __launch_bounds__(kThreads)
bwd_chunk_kernel(Params p, const float *__restrict__ dtp, const float *__restrict__ cs,
                 const float *__restrict__ states, const float *__restrict__ adj, const float *__restrict__ dyp,
                 void *dx, float *__restrict__ ddt, float *__restrict__ dBh, float *__restrict__ dCh,
                 float *__restrict__ partA, float *__restrict__ partD, float *__restrict__ partBias) {
    extern __shared__ unsigned char smem_raw[];
    ChunkSmem &sm = *reinterpret_cast<ChunkSmem *>(smem_raw);
    const int k = blockIdx.y, bh = blockIdx.x;
    const int b = bh / p.H, h = bh % p.H, g = h / p.hpg;
    const int P = p.P, N = p.N, Q = p.Q, L = p.L, tid = threadIdx.x;
    const int r0 = tid >> 4, c0 = tid & 15;  // 4 x 4 tiles of 64 x 64 results
    const size_t crow = (((size_t)b * p.H + h) * p.nchunks + k) * Q;
    const size_t st_off = ((((size_t)b * p.nchunks + k) * p.H + h) * P) * N;
    const float A = __ldg(p.A + h);
    const float Dh = p.D ? __ldg(p.D + h) : 0.f;

    // (1) tiles; past L: x, dy, B, C = 0 and d = 0 (cs keeps its last value)
    for (int e = tid; e < Q; e += kThreads) {
        const bool in = k * Q + e < L;
        sm.cs[e] = __ldg(cs + crow + e);
        sm.d[e] = in ? __ldg(dtp + crow + e) : 0.f;
        float u = in ? __ldg(p.dt + ((size_t)b * L + k * Q + e) * p.H + h) : 0.f;
        if (p.dt_bias) u += __ldg(p.dt_bias + h);
        sm.u[e] = u;
    }
    for (int e = tid; e < Q * P; e += kThreads) {
        const int i = e / P, pp = e % P, t = k * Q + i;
        const size_t o = (((size_t)b * L + t) * p.H + h) * P + pp;
        sm.x[i][pp] = t < L ? ld_io<IO>(p.x, o) : 0.f;
        sm.dy[i][pp] = t < L ? dyp[o] : 0.f;
    }
    for (int e = tid; e < Q * N; e += kThreads) {
        const int i = e / N, n = e % N, t = k * Q + i;
        const size_t o = (((size_t)b * L + t) * p.G + g) * N + n;
        sm.B[i][n] = t < L ? ld_io<IO>(p.Bm, o) : 0.f;
        sm.C[i][n] = t < L ? ld_io<IO>(p.Cm, o) : 0.f;
    }
    for (int e = tid; e < P * N; e += kThreads) {
        sm.S[e / N][e % N] = __ldg(states + st_off + e);
        sm.Gm[e / N][e % N] = __ldg(adj + st_off + e);
    }
    __syncthreads();
    const float cs_last = sm.cs[Q - 1];
    for (int e = tid; e < Q; e += kThreads) {
        sm.ecs[e] = expf(sm.cs[e]);
        sm.el[e] = expf(cs_last - sm.cs[e]);
    }
    // (2) CB = C B^T, DX = dyp x^T, then the masked decay: CB <- E CB, DX <- E DX,
    //     V = E CB DX d_j  (rows i, columns j of 4 x 4 tiles; past Q: unused)
    {
        float cb[4][4], dxm[4][4];
        zero4x4(cb);
        zero4x4(dxm);
        tile4x4(cb, N, r0, c0, [&](int i, int n) { return sm.C[i][n]; }, [&](int j, int n) { return sm.B[j][n]; });
        tile4x4(dxm, P, r0, c0, [&](int i, int pp) { return sm.dy[i][pp]; },
                [&](int j, int pp) { return sm.x[j][pp]; });
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int i = r0 + 16 * a, j = c0 + 16 * c;
                if (i < Q && j < Q) {
                    const float E = j <= i ? expf(sm.cs[i] - sm.cs[j]) : 0.f;
                    const float a1 = E * cb[a][c];
                    sm.V[i][j] = a1 * dxm[a][c] * sm.d[j];
                    sm.CB[i][j] = a1;
                    sm.DX[i][j] = E * dxm[a][c];
                }
            }
    }
    __syncthreads();
    // (4) T = dxs = (E CB)^T dyp + el (G B) ; GB = G B_t  (rows t, columns p)
    // (5) dB_t = d_t ((E DX)^T C + el G^T x_t)  (rows t, columns n)
    {
        float acc[4][4], gb[4][4];
        zero4x4(acc);
        zero4x4(gb);
        tile4x4(acc, Q, r0, c0, [&](int t, int i) { return sm.CB[i][t]; }, [&](int pp, int i) { return sm.dy[i][pp]; });
        tile4x4(gb, N, r0, c0, [&](int t, int n) { return sm.B[t][n]; }, [&](int pp, int n) { return sm.Gm[pp][n]; });
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int t = r0 + 16 * a, pp = c0 + 16 * c;
                if (t < Q && pp < P) {
                    sm.GB[t][pp] = gb[a][c];
                    sm.T[t][pp] = fmaf(sm.el[t], gb[a][c], acc[a][c]);
                }
            }
        zero4x4(acc);
        zero4x4(gb);
        tile4x4(acc, Q, r0, c0, [&](int t, int i) { return sm.DX[i][t]; }, [&](int n, int i) { return sm.C[i][n]; });
        tile4x4(gb, P, r0, c0, [&](int t, int pp) { return sm.x[t][pp]; }, [&](int n, int pp) { return sm.Gm[pp][n]; });
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int t = r0 + 16 * a, n = c0 + 16 * c;
                if (t < Q && n < N && k * Q + t < L)
                    dBh[(((size_t)b * L + k * Q + t) * p.H + h) * N + n] = sm.d[t] * fmaf(sm.el[t], gb[a][c], acc[a][c]);
            }
    }
    __syncthreads();
    // dx, and per token dd1 = x . dxs, z = x . GB
    for (int e = tid; e < Q * P; e += kThreads) {
        const int t = e / P, pp = e % P;
        if (k * Q + t < L)
            st_io<IO>(dx, (((size_t)b * L + k * Q + t) * p.H + h) * P + pp,
                      fmaf(sm.d[t], sm.T[t][pp], Dh * sm.dy[t][pp]));
    }
    if (tid < Q) {
        float a = 0.f, zz = 0.f;
        for (int pp = 0; pp < P; ++pp) {
            a = fmaf(sm.x[tid][pp], sm.T[tid][pp], a);
            zz = fmaf(sm.x[tid][pp], sm.GB[tid][pp], zz);
        }
        sm.dd1[tid] = a;
        sm.z[tid] = zz;
    }
    __syncthreads();
    // (6) dC_i = ecs_i (S^T dyp_i) + (E DX d) B ; T <- S^T dyp  (rows i, columns n)
    {
        float sd[4][4], acc[4][4];
        zero4x4(sd);
        zero4x4(acc);
        tile4x4(sd, P, r0, c0, [&](int i, int pp) { return sm.dy[i][pp]; }, [&](int n, int pp) { return sm.S[pp][n]; });
        tile4x4(acc, Q, r0, c0, [&](int i, int j) { return sm.DX[i][j] * sm.d[j]; },
                [&](int n, int j) { return sm.B[j][n]; });
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int i = r0 + 16 * a, n = c0 + 16 * c;
                if (i < Q && n < N) {
                    sm.T[i][n] = sd[a][c];
                    if (k * Q + i < L)
                        dCh[(((size_t)b * L + k * Q + i) * p.H + h) * N + n] = fmaf(sm.ecs[i], sd[a][c], acc[a][c]);
                }
            }
    }
    // <G, S> (fixed-order block reduction)
    {
        float part = 0.f;
        for (int e = tid; e < P * N; e += kThreads) part = fmaf(sm.Gm[e / N][e % N], sm.S[e / N][e % N], part);
        sm.red[tid] = part;
    }
    __syncthreads();
    for (int s = kThreads / 2; s > 0; s >>= 1) {
        if (tid < s) sm.red[tid] += sm.red[tid + s];
        __syncthreads();
    }
    const float gs = sm.red[0];
    // (7) u_i = C_i . T_i ; dcs ; per-token raw-dt gradient factor
    if (tid < Q) {
        float uu = 0.f;
        for (int n = 0; n < N; ++n) uu = fmaf(sm.C[tid][n], sm.T[tid][n], uu);
        float R = 0.f, K = 0.f;
        for (int j = 0; j < Q; ++j) R += sm.V[tid][j];
        for (int i = 0; i < Q; ++i) K += sm.V[i][tid];
        const float w = sm.el[tid] * sm.d[tid] * sm.z[tid];
        sm.w[tid] = w;
        sm.dcs[tid] = sm.ecs[tid] * uu + R - K - w;
        // d(raw dt) / d(d): softplus' = sigmoid, 0 outside the clamp
        const float u = sm.u[tid];
        const float dpre = p.dt_softplus ? softplus_f(u) : u;
        float f = (p.has_limit && (dpre < p.dt_min || dpre > p.dt_max)) ? 0.f : 1.f;
        if (p.dt_softplus) f *= 1.f / (1.f + expf(-u));
        sm.u[tid] = f;
    }
    __syncthreads();
    if (tid == 0) {
        float wsum = 0.f;
        for (int j = 0; j < Q; ++j) wsum += sm.w[j];
        sm.dcs[Q - 1] += expf(cs_last) * gs + wsum;
        // reverse cumsum; dd, dA, dbias (fixed order)
        float run = 0.f, sA = 0.f, sBias = 0.f, sD = 0.f;
        for (int t = Q - 1; t >= 0; --t) {
            run += sm.dcs[t];
            sm.dcs[t] = run;
        }
        for (int t = 0; t < Q; ++t) {
            sD += sm.DX[t][t];  // E = 1 on the diagonal: dyp_t . x_t
            if (k * Q + t >= L) continue;
            sA = fmaf(sm.d[t], sm.dcs[t], sA);
            sBias = fmaf(fmaf(A, sm.dcs[t], sm.dd1[t]), sm.u[t], sBias);
        }
        const size_t pi = ((size_t)b * p.nchunks + k) * p.H + h;
        partA[pi] = sA;
        partD[pi] = sD;
        partBias[pi] = sBias;
    }
    __syncthreads();
    for (int t = tid; t < Q; t += kThreads)
        if (k * Q + t < L) ddt[((size_t)b * L + k * Q + t) * p.H + h] = fmaf(A, sm.dcs[t], sm.dd1[t]) * sm.u[t];
}

// ---- dB, dC: heads of a group summed; dA, dD, dbias: (batch, chunk) summed ----
template <int IO>
__global__ void bwd_group_sum_kernel(Params p, const float *__restrict__ perhead, void *out) {
    const size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x;  // element of [B,L,G,N]
    const size_t total = (size_t)p.B * p.L * p.G * p.N;
    if (e >= total) return;
    const int n = e % p.N;
    const size_t bt = e / ((size_t)p.G * p.N);
    const int g = (e / p.N) % p.G;
    float acc = 0.f;
    for (int hh = 0; hh < p.hpg; ++hh) acc += perhead[(bt * p.H + g * p.hpg + hh) * p.N + n];
    st_io<IO>(out, e, acc);
}

__global__ void bwd_head_sum_kernel(Params p, const float *__restrict__ partA, const float *__restrict__ partD,
                                    const float *__restrict__ partBias, float *dA, float *dD, float *dbias) {
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= p.H) return;
    float a = 0.f, dv = 0.f, bv = 0.f;
    for (int bk = 0; bk < p.B * p.nchunks; ++bk) {
        const size_t i = (size_t)bk * p.H + h;
        a += partA[i];
        dv += partD[i];
        bv += partBias[i];
    }
    dA[h] = a;
    if (dD) dD[h] = dv;
    if (dbias) dbias[h] = bv;
}

}  // namespace

size_t bwd_chunk_smem_bytes() { return sizeof(ChunkSmem); }

cudaError_t launch_bwd(const Params &p, int io, const BwdBuffers &w, cudaStream_t s) {
    const size_t count = (size_t)p.B * p.L * p.H * p.P;
    const unsigned eb = (unsigned)((count + 255) / 256);
    switch (io) {
        case IO_F32: bwd_gate_kernel<IO_F32><<<eb, 256, 0, s>>>(p, w.dy, w.ypre, w.dyp, w.dz, count); break;
        case IO_F16: bwd_gate_kernel<IO_F16><<<eb, 256, 0, s>>>(p, w.dy, w.ypre, w.dyp, w.dz, count); break;
        case IO_BF16: bwd_gate_kernel<IO_BF16><<<eb, 256, 0, s>>>(p, w.dy, w.ypre, w.dyp, w.dz, count); break;
        default: return cudaErrorInvalidValue;
    }
    const dim3 grid(p.B * p.H, p.nchunks);
    switch (io) {
        case IO_F32: bwd_chunk_adjoint_kernel<IO_F32><<<grid, kThreads, 0, s>>>(p, w.cs, w.dyp, w.adj); break;
        case IO_F16: bwd_chunk_adjoint_kernel<IO_F16><<<grid, kThreads, 0, s>>>(p, w.cs, w.dyp, w.adj); break;
        case IO_BF16: bwd_chunk_adjoint_kernel<IO_BF16><<<grid, kThreads, 0, s>>>(p, w.cs, w.dyp, w.adj); break;
    }
    const int PN = p.P * p.N;  // a multiple of 256: P, N are multiples of 16
    bwd_state_passing_kernel<<<dim3(p.B * p.H, (PN / 4 + kThreads - 1) / kThreads), kThreads, 0, s>>>(
        p, w.cs, w.dfinal, w.adj, w.dh0);
    const int smem = (int)sizeof(ChunkSmem);
    cudaError_t e;
    switch (io) {
        case IO_F32:
            if ((e = cudaFuncSetAttribute(bwd_chunk_kernel<IO_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          smem)) != cudaSuccess)
                return e;
            bwd_chunk_kernel<IO_F32><<<grid, kThreads, smem, s>>>(p, w.dtp, w.cs, w.states, w.adj, w.dyp, w.dx,
                                                                  w.ddt, w.dBh, w.dCh, w.partA, w.partD, w.partBias);
            break;
        case IO_F16:
            if ((e = cudaFuncSetAttribute(bwd_chunk_kernel<IO_F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          smem)) != cudaSuccess)
                return e;
            bwd_chunk_kernel<IO_F16><<<grid, kThreads, smem, s>>>(p, w.dtp, w.cs, w.states, w.adj, w.dyp, w.dx,
                                                                  w.ddt, w.dBh, w.dCh, w.partA, w.partD, w.partBias);
            break;
        case IO_BF16:
            if ((e = cudaFuncSetAttribute(bwd_chunk_kernel<IO_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          smem)) != cudaSuccess)
                return e;
            bwd_chunk_kernel<IO_BF16><<<grid, kThreads, smem, s>>>(p, w.dtp, w.cs, w.states, w.adj, w.dyp, w.dx,
                                                                   w.ddt, w.dBh, w.dCh, w.partA, w.partD, w.partBias);
            break;
    }
    const size_t gtotal = (size_t)p.B * p.L * p.G * p.N;
    const unsigned gb = (unsigned)((gtotal + 255) / 256);
    switch (io) {
        case IO_F32:
            bwd_group_sum_kernel<IO_F32><<<gb, 256, 0, s>>>(p, w.dBh, w.dB);
            bwd_group_sum_kernel<IO_F32><<<gb, 256, 0, s>>>(p, w.dCh, w.dC);
            break;
        case IO_F16:
            bwd_group_sum_kernel<IO_F16><<<gb, 256, 0, s>>>(p, w.dBh, w.dB);
            bwd_group_sum_kernel<IO_F16><<<gb, 256, 0, s>>>(p, w.dCh, w.dC);
            break;
        case IO_BF16:
            bwd_group_sum_kernel<IO_BF16><<<gb, 256, 0, s>>>(p, w.dBh, w.dB);
            bwd_group_sum_kernel<IO_BF16><<<gb, 256, 0, s>>>(p, w.dCh, w.dC);
            break;
    }
    bwd_head_sum_kernel<<<(p.H + 127) / 128, 128, 0, s>>>(p, w.partA, w.partD, w.partBias, w.dA, w.dD, w.dbias);
    return cudaGetLastError();
}

}  // namespace ssd
