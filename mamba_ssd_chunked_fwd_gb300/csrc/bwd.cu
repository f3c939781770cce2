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
    {
        // every global load issued before the shared-memory stores; 0 outside (Q, P, N) and past L
        constexpr int kPer = kMax * kMax / kThreads;
        float rd[kPer], rc[kPer], re[kPer];
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int e = threadIdx.x + kThreads * q, i = e >> 6, col = e & (kMax - 1), t = k * Q + i;
            const bool row_in = i < Q && t < L;
            rd[q] = row_in && col < P ? __ldg(dyp + (((size_t)b * L + t) * p.H + h) * P + col) : 0.f;
            rc[q] = row_in && col < N ? ld_io<IO>(p.Cm, (((size_t)b * L + t) * p.G + g) * N + col) : 0.f;
            re[q] = row_in ? __ldg(cs + crow + i) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int e = threadIdx.x + kThreads * q, i = e >> 6, col = e & (kMax - 1);
            ds[i][col] = rd[q] * expf(re[q]);
            cc[i][col] = rc[q];
        }
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
// Row sums of 4 x 4 tiles reduce over the 16 lanes that share a tile row
// (a half warp); column sums over the two tile rows of a warp, then over the
// 8 warps through shared memory in warp order.  Every order is fixed.
struct ChunkSmem {
    float x[kMax][kMax + 1], dy[kMax][kMax + 1], B[kMax][kMax + 1], C[kMax][kMax + 1];
    float S[kMax][kMax + 1], Gm[kMax][kMax + 1];
    float CB[kMax][kMax + 1];  // E CB (masked decayed C B^T)
    float DX[kMax][kMax + 1];  // E DX d_j (masked decayed dyp x^T, column j scaled by d_j)
    float Kp[kThreads / 32][kMax];
    float cs[kMax], d[kMax], ecs[kMax], el[kMax], dd1[kMax], w[kMax], z[kMax], dcs[kMax], u[kMax];
    float R[kMax], uu[kMax], dxd[kMax];
    float red[kThreads / 32];
};

// sum over the 16 lanes of a half warp (lanes sharing a tile row)
__device__ __forceinline__ float half_warp_sum(float v) {
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

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
    const int lane = tid & 31, warp = tid >> 5;
    const int r0 = tid >> 4, c0 = tid & 15;  // 4 x 4 tiles of 64 x 64 results
    const size_t crow = (((size_t)b * p.H + h) * p.nchunks + k) * Q;
    const size_t st_off = ((((size_t)b * p.nchunks + k) * p.H + h) * P) * N;
    const float A = __ldg(p.A + h);
    const float Dh = p.D ? __ldg(p.D + h) : 0.f;

    // (1) tiles, every global load issued before the shared-memory stores.
    //     Outside (Q, P, N) and past L: 0, and d = 0 (cs keeps its last value).
    if (tid < kMax) {
        const int e = tid;
        const bool inq = e < Q, in = inq && k * Q + e < L;
        const float c = inq ? __ldg(cs + crow + e) : 0.f;
        float u = in ? __ldg(p.dt + ((size_t)b * L + k * Q + e) * p.H + h) : 0.f;
        if (p.dt_bias) u += __ldg(p.dt_bias + h);
        sm.cs[e] = c;
        sm.d[e] = in ? __ldg(dtp + crow + e) : 0.f;
        sm.u[e] = u;
    }
    {
        constexpr int kPer = kMax * kMax / kThreads;  // 16 elements per thread and tile
        float rx[kPer], rdy[kPer], rb[kPer], rc[kPer], rs[kPer], rg[kPer];
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int e = tid + kThreads * q, i = e >> 6, col = e & (kMax - 1), t = k * Q + i;
            const bool row_in = i < Q && t < L;
            const size_t ox = (((size_t)b * L + t) * p.H + h) * P + col;
            const size_t ob = (((size_t)b * L + t) * p.G + g) * N + col;
            rx[q] = row_in && col < P ? ld_io<IO>(p.x, ox) : 0.f;
            rdy[q] = row_in && col < P ? __ldg(dyp + ox) : 0.f;
            rb[q] = row_in && col < N ? ld_io<IO>(p.Bm, ob) : 0.f;
            rc[q] = row_in && col < N ? ld_io<IO>(p.Cm, ob) : 0.f;
            const bool sin = i < P && col < N;  // i: state row p, col: n
            rs[q] = sin ? __ldg(states + st_off + (size_t)i * N + col) : 0.f;
            rg[q] = sin ? __ldg(adj + st_off + (size_t)i * N + col) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int e = tid + kThreads * q, i = e >> 6, col = e & (kMax - 1);
            sm.x[i][col] = rx[q];
            sm.dy[i][col] = rdy[q];
            sm.B[i][col] = rb[q];
            sm.C[i][col] = rc[q];
            sm.S[i][col] = rs[q];
            sm.Gm[i][col] = rg[q];
        }
    }
    __syncthreads();
    const float cs_last = sm.cs[Q - 1];
    if (tid < kMax) {
        const int e = tid;
        sm.ecs[e] = e < Q ? expf(sm.cs[e]) : 0.f;
        sm.el[e] = e < Q ? expf(cs_last - sm.cs[e]) : 0.f;
    }
    // (2) CB = C B^T, DX = dyp x^T, then the masked decay: CB <- E CB,
    //     DX <- E DX d_j; V = E CB DX d_j only as its row sums R and column sums K
    {
        float cb[4][4], dxm[4][4];
        zero4x4(cb);
        zero4x4(dxm);
        tile4x4(cb, N, r0, c0, [&](int i, int n) { return sm.C[i][n]; }, [&](int j, int n) { return sm.B[j][n]; });
        tile4x4(dxm, P, r0, c0, [&](int i, int pp) { return sm.dy[i][pp]; },
                [&](int j, int pp) { return sm.x[j][pp]; });
        float rp[4] = {0.f, 0.f, 0.f, 0.f}, cp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int i = r0 + 16 * a, j = c0 + 16 * c;
                const float E = (i < Q && j <= i) ? expf(sm.cs[i] - sm.cs[j]) : 0.f;
                const float a1 = E * cb[a][c], dm = E * dxm[a][c] * sm.d[j];
                const float v = a1 * dxm[a][c] * sm.d[j];
                rp[a] += v;
                cp[c] += v;
                sm.CB[i][j] = a1;
                sm.DX[i][j] = dm;
                if (i == j) sm.dxd[i] = dxm[a][c];  // E = 1 on the diagonal: dyp_i . x_i
            }
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const float r = half_warp_sum(rp[a]);
            if (c0 == 0) sm.R[r0 + 16 * a] = r;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const float s = cp[c] + __shfl_xor_sync(0xffffffffu, cp[c], 16);  // tile rows 2w and 2w+1
            if (lane < 16) sm.Kp[warp][c0 + 16 * c] = s;
        }
    }
    __syncthreads();
    // (4) dxs = (E CB)^T dyp + el (G B)  (rows t, columns p) -> dx = d dxs + D dyp,
    //     dd1_t = x_t . dxs_t, z_t = x_t . (G B_t)
    // (5) dB_t = (E DX d)^T C + d_t el_t G^T x_t  (rows t, columns n)
    {
        float acc[4][4], gb[4][4];
        zero4x4(acc);
        zero4x4(gb);
        tile4x4(acc, Q, r0, c0, [&](int t, int i) { return sm.CB[i][t]; }, [&](int pp, int i) { return sm.dy[i][pp]; });
        tile4x4(gb, N, r0, c0, [&](int t, int n) { return sm.B[t][n]; }, [&](int pp, int n) { return sm.Gm[pp][n]; });
        float dp[4] = {0.f, 0.f, 0.f, 0.f}, zp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int t = r0 + 16 * a, pp = c0 + 16 * c;
                const float T = fmaf(sm.el[t], gb[a][c], acc[a][c]);
                const float xv = sm.x[t][pp];
                dp[a] = fmaf(xv, T, dp[a]);
                zp[a] = fmaf(xv, gb[a][c], zp[a]);
                if (t < Q && pp < P && k * Q + t < L)
                    st_io<IO>(dx, (((size_t)b * L + k * Q + t) * p.H + h) * P + pp,
                              fmaf(sm.d[t], T, Dh * sm.dy[t][pp]));
            }
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const float s1 = half_warp_sum(dp[a]), s2 = half_warp_sum(zp[a]);
            if (c0 == 0) {
                sm.dd1[r0 + 16 * a] = s1;
                sm.z[r0 + 16 * a] = s2;
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
                    dBh[(((size_t)b * L + k * Q + t) * p.H + h) * N + n] =
                        fmaf(sm.d[t] * sm.el[t], gb[a][c], acc[a][c]);
            }
    }
    // (6) dC_i = ecs_i (S^T dyp_i) + (E DX d) B ;  uu_i = C_i . (S^T dyp_i)  (rows i, columns n)
    {
        float sd[4][4], acc[4][4];
        zero4x4(sd);
        zero4x4(acc);
        tile4x4(sd, P, r0, c0, [&](int i, int pp) { return sm.dy[i][pp]; }, [&](int n, int pp) { return sm.S[pp][n]; });
        tile4x4(acc, Q, r0, c0, [&](int i, int j) { return sm.DX[i][j]; }, [&](int n, int j) { return sm.B[j][n]; });
        float up[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int i = r0 + 16 * a, n = c0 + 16 * c;
                up[a] = fmaf(sm.C[i][n], sd[a][c], up[a]);
                if (i < Q && n < N && k * Q + i < L)
                    dCh[(((size_t)b * L + k * Q + i) * p.H + h) * N + n] = fmaf(sm.ecs[i], sd[a][c], acc[a][c]);
            }
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const float s = half_warp_sum(up[a]);
            if (c0 == 0) sm.uu[r0 + 16 * a] = s;
        }
    }
    // <G, S>: per warp, then over the warps in order
    {
        float part = 0.f;
        for (int e = tid; e < kMax * kMax; e += kThreads) part = fmaf(sm.Gm[e >> 6][e & 63], sm.S[e >> 6][e & 63], part);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if (lane == 0) sm.red[warp] = part;
    }
    __syncthreads();
    float gs = 0.f;
#pragma unroll
    for (int q = 0; q < kThreads / 32; ++q) gs += sm.red[q];
    // (7) dcs and the per-token raw-dt gradient factor
    if (tid < Q) {
        float K = 0.f;
#pragma unroll
        for (int q = 0; q < kThreads / 32; ++q) K += sm.Kp[q][tid];
        const float w = sm.el[tid] * sm.d[tid] * sm.z[tid];
        sm.w[tid] = w;
        sm.dcs[tid] = sm.ecs[tid] * sm.uu[tid] + sm.R[tid] - K - w;
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
            sD += sm.dxd[t];
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
