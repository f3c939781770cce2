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

__device__ __forceinline__ void zero4x4(float (&acc)[4][4]) {
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
}

// ---- 4 x 4 register tiles over shared operands (adjoint and chunk kernels) ----
// Every product is a 64 x 64 result in 4 x 4 register tiles: thread (r0, c0)
// = (tid / 16, tid % 16) owns rows 4 r0 .. 4 r0 + 3 and columns 4 c0 .. 4 c0 + 3,
// and each step of the contraction reads one float4 of each operand from
// shared memory.  Operands are 64 x 64 fp32 in one of two layouts:
//   N: element (r, c) at [r][c];
//   T: element (r, c) at row c, 16-byte chunk (r / 4) ^ s(c) with
//      s(c) = (c % 8) ^ ((c / 4) % 8), so that four consecutive r at one c are
//      one aligned float4.  16-byte accesses are served 8 lanes at a time, and
//      s keeps those 8 lanes on 8 different bank groups in every pattern used
//      here: one row at 8 consecutive chunks, one chunk of 8 consecutive rows,
//      and one chunk of rows 4 j + o for 8 consecutive j.
// A product sum_k A(r, k) B(c, k) reads A as row k, chunk r0 (the same float4
// for a half warp) and B as row k, chunk c0.
__device__ __forceinline__ int tsw(int row, int chunk) {
    return row * kMax + 4 * (chunk ^ ((row & 7) ^ ((row >> 2) & 7)));
}
__device__ __forceinline__ float4 ld4n(const float *m, int row, int chunk) {
    return *reinterpret_cast<const float4 *>(m + row * kMax + 4 * chunk);
}
__device__ __forceinline__ float4 ld4t(const float *m, int row, int chunk) {
    return *reinterpret_cast<const float4 *>(m + tsw(row, chunk));
}
__device__ __forceinline__ void st4n(float *m, int row, int chunk, float4 v) {
    *reinterpret_cast<float4 *>(m + row * kMax + 4 * chunk) = v;
}
__device__ __forceinline__ void st4t(float *m, int row, int chunk, float4 v) {
    *reinterpret_cast<float4 *>(m + tsw(row, chunk)) = v;
}
__device__ __forceinline__ float f4(const float4 &v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }

// acc[a][b] += sum_{k0 <= k < k1} A(4 r0 + a, k) B(4 c0 + b, k); fa(k), fb(k)
// return the float4s; k1 - k0 is a multiple of 4.
template <class FA, class FB>
__device__ __forceinline__ void tile4v(float (&acc)[4][4], int k0, int k1, FA fa, FB fb) {
#pragma unroll 8
    for (int k = k0; k < k1; ++k) {
        const float4 av = fa(k), bv = fb(k);
        const float ar[4] = {av.x, av.y, av.z, av.w}, br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(ar[a], br[b], acc[a][b]);
    }
}

// sum over the 16 lanes of a half warp (lanes sharing a tile's rows)
__device__ __forceinline__ float half_warp_sum(float v) {
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}


// ---- per chunk: sum_i exp(cs_i) dyp_i (outer) C_i  [P,N] ----
template <int IO>
__global__ void __launch_bounds__(kThreads)
bwd_chunk_adjoint_kernel(Params p, const float *__restrict__ cs, const float *__restrict__ dyp,
                         float *__restrict__ adj) {
    __shared__ __align__(16) float ds[kMax * kMax];  // exp(cs_i) dyp_i, [i][p] (N)
    __shared__ __align__(16) float cc[kMax * kMax];  // C, [i][n] (N)
    __shared__ float e_s[kMax];                      // exp(cs_i)
    const int k = blockIdx.y, bh = blockIdx.x;
    const int b = bh / p.H, h = bh % p.H, g = h / p.hpg;
    const int P = p.P, N = p.N, Q = p.Q, L = p.L, tid = threadIdx.x;
    const size_t crow = (((size_t)b * p.H + h) * p.nchunks + k) * Q;
    if (tid < kMax) e_s[tid] = tid < Q ? expf(__ldg(cs + crow + tid)) : 0.f;
    // every global load issued before the shared-memory stores; 0 outside (Q, P, N) and past L
    constexpr int kPer = kMax * kMax / kThreads;
    const int col = tid & (kMax - 1), rb = tid >> 6;
    float rd[kPer], rc[kPer];
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        const int i = rb * kPer + q, t = k * Q + i;
        const bool row_in = i < Q && t < L;
        rd[q] = row_in && col < P ? __ldg(dyp + (((size_t)b * L + t) * p.H + h) * P + col) : 0.f;
        rc[q] = row_in && col < N ? ld_io<IO>(p.Cm, (((size_t)b * L + t) * p.G + g) * N + col) : 0.f;
    }
    __syncthreads();  // e_s
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        const int i = rb * kPer + q;
        ds[i * kMax + col] = rd[q] * e_s[i];
        cc[i * kMax + col] = rc[q];
    }
    __syncthreads();
    const int r0 = tid >> 4, c0 = tid & 15;
    float acc[4][4];
    zero4x4(acc);
    tile4v(acc, 0, Q, [&](int i) { return ld4n(ds, i, r0); }, [&](int i) { return ld4n(cc, i, c0); });
    float *out = adj + ((((size_t)b * p.nchunks + k) * p.H + h) * P) * N;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int pp = 4 * r0 + a;
        if (pp < P && 4 * c0 < N)
            *reinterpret_cast<float4 *>(out + (size_t)pp * N + 4 * c0) =
                make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
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
// Row sums of a tile reduce over the 16 lanes that share its rows (a half
// warp); column sums over the two tile rows of a warp, then over the 8 warps
// through shared memory in warp order.  Every order is fixed.  The masked
// products stop at the warp's own rows: (E CB)[i][t] and (E DX)[i][t] vanish
// for i < t.
struct ChunkSmem {
    float xt[kMax * kMax], dyt[kMax * kMax], dy[kMax * kMax];  // x^T, dyp^T (T); dyp (N)
    float Bt[kMax * kMax], B[kMax * kMax], Ct[kMax * kMax], C[kMax * kMax];
    float S[kMax * kMax], G[kMax * kMax], Gt[kMax * kMax];  // S, G [p][n] (N); G^T (T)
    float CB[kMax * kMax];                                  // E CB (N)
    float DX[kMax * kMax], DXt[kMax * kMax];                // E DX d_j (N and T)
    float Kp[kThreads / 32][kMax];
    float cs[kMax], d[kMax], ecs[kMax], el[kMax], dd1[kMax], w[kMax], z[kMax], dcs[kMax], u[kMax];
    float R[kMax], uu[kMax], dxd[kMax];
    float red[kThreads / 32];
};

// One cache line into L2 (a hint: no alignment rule, no completion).
__device__ __forceinline__ void prefetch_line_l2(const void *q) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(q));
}

// Ask L2 for every operand line of the chunk kernel's CTA (bh, k): its rows of
// x, dyp, B, C and dt (one row per thread of each quarter of the CTA), its cs
// and dtp vectors and its state and adjoint blocks.
template <int IO>
__device__ __forceinline__ void bwd_chunk_prefetch(const Params &p, const float *dtp, const float *cs,
                                                   const float *states, const float *adj, const float *dyp, int bh,
                                                   int k, int tid) {
    constexpr int kIo = IO == IO_F32 ? 4 : 2;
    const int P = p.P, N = p.N, Q = p.Q, L = p.L;
    const int b = bh / p.H, h = bh - b * p.H, g = h / p.hpg;
    const int i = tid & (kMax - 1), which = tid >> 6;  // 4 groups of 64 rows
    const int t = k * Q + i;
    if (i < Q && t < L) {
        const unsigned char *row;
        int bytes;
        if (which == 0) {
            row = static_cast<const unsigned char *>(p.x) + (((size_t)b * L + t) * p.H + h) * P * kIo;
            bytes = P * kIo;
        } else if (which == 1) {
            row = reinterpret_cast<const unsigned char *>(dyp + (((size_t)b * L + t) * p.H + h) * P);
            bytes = P * 4;
            prefetch_line_l2(p.dt + ((size_t)b * L + t) * p.H + h);
        } else {
            row = static_cast<const unsigned char *>(which == 2 ? p.Bm : p.Cm) +
                  (((size_t)b * L + t) * p.G + g) * N * kIo;
            bytes = N * kIo;
        }
        for (int o = 0; o < bytes; o += 128) prefetch_line_l2(row + o);
        prefetch_line_l2(row + bytes - 1);
    }
    const size_t crow = (((size_t)b * p.H + h) * p.nchunks + k) * Q;
    if (tid == 0) {
        prefetch_line_l2(cs + crow);
        prefetch_line_l2(cs + crow + Q - 1);
        prefetch_line_l2(dtp + crow);
        prefetch_line_l2(dtp + crow + Q - 1);
    }
    // the state and adjoint blocks: P N floats each, contiguous
    const size_t st = ((((size_t)b * p.nchunks + k) * p.H + h) * P) * N;
    const int bytes = P * N * 4, lines = (bytes + 127) / 128;
    for (int l = tid; l < 2 * lines; l += kThreads) {
        const float *base = (l < lines ? states : adj) + st;
        const int o = (l < lines ? l : l - lines) * 128;
        prefetch_line_l2(reinterpret_cast<const unsigned char *>(base) + (o < bytes ? o : bytes - 1));
    }
}

template <int IO>
__global__ void __launch_bounds__(kThreads)
bwd_chunk_kernel(Params p, const float *__restrict__ dtp, const float *__restrict__ cs,
                 const float *__restrict__ states, const float *__restrict__ adj, const float *__restrict__ dyp,
                 void *dx, float *__restrict__ ddt, float *__restrict__ dBh, float *__restrict__ dCh,
                 float *__restrict__ partA, float *__restrict__ partD, float *__restrict__ partBias, int wave) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ChunkSmem &sm = *reinterpret_cast<ChunkSmem *>(smem_raw);
    const int k = blockIdx.y, bh = blockIdx.x;
    const int b = bh / p.H, h = bh % p.H, g = h / p.hpg;
    const int P = p.P, N = p.N, Q = p.Q, L = p.L, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int r0 = tid >> 4, c0 = tid & 15;
    const size_t crow = (((size_t)b * p.H + h) * p.nchunks + k) * Q;
    const size_t st_off = ((((size_t)b * p.nchunks + k) * p.H + h) * P) * N;
    const float A = __ldg(p.A + h);
    const float Dh = p.D ? __ldg(p.D + h) : 0.f;

    // One CTA fills an SM, so the CTA that follows it there would start by
    // waiting on the memory with nothing to overlap.  CTAs start in linear
    // order (blockIdx.x fastest), one wave (`wave` CTAs) apart on the SMs, so
    // this one asks L2 for the operands of the CTA a wave after it.
    {
        const long long nxt = (long long)k * gridDim.x + bh + wave;
        if (wave > 0 && nxt < (long long)gridDim.x * gridDim.y)
            bwd_chunk_prefetch<IO>(p, dtp, cs, states, adj, dyp, (int)(nxt % gridDim.x), (int)(nxt / gridDim.x),
                                   tid);
    }

    // (1) operands, every global load issued before the shared-memory stores.
    //     Outside (Q, P, N) and past L: 0, and d = 0 (cs keeps its last value).
    //     Thread: column col of rows 16 rb .. 16 rb + 15 (coalesced rows; four
    //     float4 of consecutive rows for the T copies).
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
        constexpr int kPer = kMax * kMax / kThreads;  // 16
        const int col = tid & (kMax - 1), rb = tid >> 6;
        float rx[kPer], rdy[kPer], rb_[kPer], rc[kPer], rs[kPer], rg[kPer];
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int i = rb * kPer + q, t = k * Q + i;
            const bool row_in = i < Q && t < L;
            const size_t ox = (((size_t)b * L + t) * p.H + h) * P + col;
            const size_t ob = (((size_t)b * L + t) * p.G + g) * N + col;
            rx[q] = row_in && col < P ? ld_io<IO>(p.x, ox) : 0.f;
            rdy[q] = row_in && col < P ? __ldg(dyp + ox) : 0.f;
            rb_[q] = row_in && col < N ? ld_io<IO>(p.Bm, ob) : 0.f;
            rc[q] = row_in && col < N ? ld_io<IO>(p.Cm, ob) : 0.f;
            const bool sin = i < P && col < N;  // state row p = i, column n = col
            rs[q] = sin ? __ldg(states + st_off + (size_t)i * N + col) : 0.f;
            rg[q] = sin ? __ldg(adj + st_off + (size_t)i * N + col) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int i = rb * kPer + q;
            sm.dy[i * kMax + col] = rdy[q];
            sm.B[i * kMax + col] = rb_[q];
            sm.C[i * kMax + col] = rc[q];
            sm.S[i * kMax + col] = rs[q];
            sm.G[i * kMax + col] = rg[q];
        }
#pragma unroll
        for (int m = 0; m < kPer / 4; ++m) {
            const int ch = rb * (kPer / 4) + m;  // chunk of rows 16 rb + 4 m .. + 3
            st4t(sm.xt, col, ch, make_float4(rx[4 * m], rx[4 * m + 1], rx[4 * m + 2], rx[4 * m + 3]));
            st4t(sm.dyt, col, ch, make_float4(rdy[4 * m], rdy[4 * m + 1], rdy[4 * m + 2], rdy[4 * m + 3]));
            st4t(sm.Bt, col, ch, make_float4(rb_[4 * m], rb_[4 * m + 1], rb_[4 * m + 2], rb_[4 * m + 3]));
            st4t(sm.Ct, col, ch, make_float4(rc[4 * m], rc[4 * m + 1], rc[4 * m + 2], rc[4 * m + 3]));
            st4t(sm.Gt, col, ch, make_float4(rg[4 * m], rg[4 * m + 1], rg[4 * m + 2], rg[4 * m + 3]));
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
        tile4v(cb, 0, N, [&](int n) { return ld4t(sm.Ct, n, r0); }, [&](int n) { return ld4t(sm.Bt, n, c0); });
        tile4v(dxm, 0, P, [&](int pp) { return ld4t(sm.dyt, pp, r0); }, [&](int pp) { return ld4t(sm.xt, pp, c0); });
        float rp[4] = {0.f, 0.f, 0.f, 0.f}, cp[4] = {0.f, 0.f, 0.f, 0.f};
        float dm[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int i = 4 * r0 + a;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int j = 4 * c0 + c;
                const float E = (i < Q && j <= i) ? expf(sm.cs[i] - sm.cs[j]) : 0.f;
                const float dj = sm.d[j];
                const float a1 = E * cb[a][c];
                dm[a][c] = E * dxm[a][c] * dj;
                const float v = a1 * dxm[a][c] * dj;
                rp[a] += v;
                cp[c] += v;
                cb[a][c] = a1;
                if (i == j) sm.dxd[i] = dxm[a][c];  // E = 1 on the diagonal: dyp_i . x_i
            }
            st4n(sm.CB, i, c0, make_float4(cb[a][0], cb[a][1], cb[a][2], cb[a][3]));
            st4n(sm.DX, i, c0, make_float4(dm[a][0], dm[a][1], dm[a][2], dm[a][3]));
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) st4t(sm.DXt, 4 * c0 + c, r0, make_float4(dm[0][c], dm[1][c], dm[2][c], dm[3][c]));
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const float r = half_warp_sum(rp[a]);
            if (c0 == 0) sm.R[4 * r0 + a] = r;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const float s = cp[c] + __shfl_xor_sync(0xffffffffu, cp[c], 16);  // tile rows 2w and 2w+1
            if (lane < 16) sm.Kp[warp][4 * c0 + c] = s;
        }
    }
    __syncthreads();
    const int tri_lo = 8 * warp;                              // first row of the warp's tiles
    const int tri_hi = min(8 * warp + 8, Q);                  // one past its last row (within Q)
    // (4) dxs = (E CB)^T dyp + el (G B)  (rows t, columns p) -> dx = d dxs + D dyp,
    //     dd1_t = x_t . dxs_t, z_t = x_t . (G B_t).  (E CB)[i][t] = 0 for i < t.
    {
        float acc[4][4], gb[4][4];
        zero4x4(acc);
        zero4x4(gb);
        tile4v(acc, tri_lo < Q ? tri_lo : Q, Q, [&](int i) { return ld4n(sm.CB, i, r0); },
               [&](int i) { return ld4n(sm.dy, i, c0); });
        tile4v(gb, 0, N, [&](int n) { return ld4t(sm.Bt, n, r0); }, [&](int n) { return ld4t(sm.Gt, n, c0); });
        float4 xx[4], dd[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) xx[c] = ld4t(sm.xt, 4 * c0 + c, r0);  // x at rows 4 r0 .., column 4 c0 + c
#pragma unroll
        for (int a = 0; a < 4; ++a) dd[a] = ld4n(sm.dy, 4 * r0 + a, c0);
        float dp[4] = {0.f, 0.f, 0.f, 0.f}, zp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int t = 4 * r0 + a;
            const float elt = sm.el[t], dt_ = sm.d[t];
            const bool row_ok = t < Q && k * Q + t < L;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int pp = 4 * c0 + c;
                const float T = fmaf(elt, gb[a][c], acc[a][c]);
                const float xv = f4(xx[c], a);
                dp[a] = fmaf(xv, T, dp[a]);
                zp[a] = fmaf(xv, gb[a][c], zp[a]);
                if (row_ok && pp < P)
                    st_io<IO>(dx, (((size_t)b * L + k * Q + t) * p.H + h) * P + pp, fmaf(dt_, T, Dh * f4(dd[a], c)));
            }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const float s1 = half_warp_sum(dp[a]), s2 = half_warp_sum(zp[a]);
            if (c0 == 0) {
                sm.dd1[4 * r0 + a] = s1;
                sm.z[4 * r0 + a] = s2;
            }
        }
    }
    // (5) dB_t = (E DX d)^T C + d_t el_t G^T x_t  (rows t, columns n).  (E DX)[i][t] = 0 for i < t.
    {
        float acc[4][4], gb[4][4];
        zero4x4(acc);
        zero4x4(gb);
        tile4v(acc, tri_lo < Q ? tri_lo : Q, Q, [&](int i) { return ld4n(sm.DX, i, r0); },
               [&](int i) { return ld4n(sm.C, i, c0); });
        tile4v(gb, 0, P, [&](int pp) { return ld4t(sm.xt, pp, r0); }, [&](int pp) { return ld4n(sm.G, pp, c0); });
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int t = 4 * r0 + a;
            if (t < Q && k * Q + t < L && 4 * c0 < N) {
                const float f = sm.d[t] * sm.el[t];
                float4 o;
                o.x = fmaf(f, gb[a][0], acc[a][0]);
                o.y = fmaf(f, gb[a][1], acc[a][1]);
                o.z = fmaf(f, gb[a][2], acc[a][2]);
                o.w = fmaf(f, gb[a][3], acc[a][3]);
                *reinterpret_cast<float4 *>(dBh + (((size_t)b * L + k * Q + t) * p.H + h) * N + 4 * c0) = o;
            }
        }
    }
    // (6) dC_i = ecs_i (S^T dyp_i) + (E DX d) B ;  uu_i = C_i . (S^T dyp_i)  (rows i, columns n).
    //     (E DX)[i][j] = 0 for j > i.
    {
        float sd[4][4], acc[4][4];
        zero4x4(sd);
        zero4x4(acc);
        tile4v(sd, 0, P, [&](int pp) { return ld4t(sm.dyt, pp, r0); }, [&](int pp) { return ld4n(sm.S, pp, c0); });
        tile4v(acc, 0, tri_hi > 0 ? tri_hi : 0, [&](int j) { return ld4t(sm.DXt, j, r0); },
               [&](int j) { return ld4n(sm.B, j, c0); });
        float up[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int i = 4 * r0 + a;
            const float4 cv = ld4n(sm.C, i, c0);
            up[a] = fmaf(cv.x, sd[a][0], fmaf(cv.y, sd[a][1], fmaf(cv.z, sd[a][2], fmaf(cv.w, sd[a][3], up[a]))));
            if (i < Q && k * Q + i < L && 4 * c0 < N) {
                const float e = sm.ecs[i];
                float4 o;
                o.x = fmaf(e, sd[a][0], acc[a][0]);
                o.y = fmaf(e, sd[a][1], acc[a][1]);
                o.z = fmaf(e, sd[a][2], acc[a][2]);
                o.w = fmaf(e, sd[a][3], acc[a][3]);
                *reinterpret_cast<float4 *>(dCh + (((size_t)b * L + k * Q + i) * p.H + h) * N + 4 * c0) = o;
            }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const float s = half_warp_sum(up[a]);
            if (c0 == 0) sm.uu[4 * r0 + a] = s;
        }
    }
    // <G, S>: per warp, then over the warps in order
    {
        float part = 0.f;
#pragma unroll
        for (int q = 0; q < kMax * kMax / 4 / kThreads; ++q) {
            const int e4 = tid + kThreads * q;  // float4 index
            const float4 gv = reinterpret_cast<const float4 *>(sm.G)[e4];
            const float4 sv = reinterpret_cast<const float4 *>(sm.S)[e4];
            part = fmaf(gv.x, sv.x, fmaf(gv.y, sv.y, fmaf(gv.z, sv.z, fmaf(gv.w, sv.w, part))));
        }
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
    // the tail below gives each of the 32 lanes two tokens: it needs Q <= 64 and an even Q
    static_assert(kMax <= 64 && kMax % 2 == 0, "the one-warp tail covers at most 2 x 32 tokens");
    if (warp == 0) {
        // tokens 2 lane and 2 lane + 1 (Q is even): the last token's extra terms, the reverse
        // cumulative sum of dcs (a shuffle scan of the pair sums), then dA, dD, dbias partials;
        // every sum in a fixed order
        const int t0 = 2 * lane, t1 = t0 + 1;
        const bool q0 = t0 < Q, q1 = t1 < Q;
        float wsum = (q0 ? sm.w[t0] : 0.f) + (q1 ? sm.w[t1] : 0.f);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
        const float d0 = q0 ? sm.dcs[t0] : 0.f;
        float d1 = q1 ? sm.dcs[t1] : 0.f;
        if (t1 == Q - 1) d1 += expf(cs_last) * gs + wsum;
        const float pr = d0 + d1;
        float S = pr;  // sum of the pair sums of lanes >= this one
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_down_sync(0xffffffffu, S, off);
            if (lane + off < 32) S += o;
        }
        float excl = __shfl_down_sync(0xffffffffu, S, 1);  // lanes > this one
        if (lane == 31) excl = 0.f;
        const float R1 = d1 + excl, R0 = d0 + R1;
        if (q0) sm.dcs[t0] = R0;
        if (q1) sm.dcs[t1] = R1;
        const bool in0 = q0 && k * Q + t0 < L, in1 = q1 && k * Q + t1 < L;
        float sA = (in0 ? sm.d[t0] * R0 : 0.f) + (in1 ? sm.d[t1] * R1 : 0.f);
        float sBias = (in0 ? fmaf(A, R0, sm.dd1[t0]) * sm.u[t0] : 0.f) + (in1 ? fmaf(A, R1, sm.dd1[t1]) * sm.u[t1] : 0.f);
        float sD = (q0 ? sm.dxd[t0] : 0.f) + (q1 ? sm.dxd[t1] : 0.f);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            sA += __shfl_xor_sync(0xffffffffu, sA, off);
            sBias += __shfl_xor_sync(0xffffffffu, sBias, off);
            sD += __shfl_xor_sync(0xffffffffu, sD, off);
        }
        if (lane == 0) {
            const size_t pi = ((size_t)b * p.nchunks + k) * p.H + h;
            partA[pi] = sA;
            partD[pi] = sD;
            partBias[pi] = sBias;
        }
    }
    __syncthreads();
    for (int t = tid; t < Q; t += kThreads)
        if (k * Q + t < L) ddt[((size_t)b * L + k * Q + t) * p.H + h] = fmaf(A, sm.dcs[t], sm.dd1[t]) * sm.u[t];
}

// ---- dB, dC: heads of a group summed; dA, dD, dbias: (batch, chunk) summed ----
// Four consecutive n per thread (N is a multiple of 16), heads in order.
template <int IO>
__global__ void bwd_group_sum_kernel(Params p, const float *__restrict__ perhead, void *out) {
    const size_t e4 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;  // float4 of [B,L,G,N]
    const int N4 = p.N / 4;
    if (e4 >= (size_t)p.B * p.L * p.G * N4) return;
    const int n4 = (int)(e4 % N4);
    const int g = (int)((e4 / N4) % p.G);
    const size_t bt = e4 / ((size_t)p.G * N4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int hh = 0; hh < p.hpg; ++hh) {
        const float4 v = __ldg(reinterpret_cast<const float4 *>(perhead + (bt * p.H + g * p.hpg + hh) * p.N) + n4);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
    }
    const size_t e = e4 * 4;
    st_io<IO>(out, e, acc.x);
    st_io<IO>(out, e + 1, acc.y);
    st_io<IO>(out, e + 2, acc.z);
    st_io<IO>(out, e + 3, acc.w);
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
    // without z the gate is the identity: fp32 dy is read in place
    const float *dyp = w.dyp;
    if (!p.z && io == IO_F32) {
        dyp = static_cast<const float *>(w.dy);
    } else {
        switch (io) {
            case IO_F32: bwd_gate_kernel<IO_F32><<<eb, 256, 0, s>>>(p, w.dy, w.ypre, w.dyp, w.dz, count); break;
            case IO_F16: bwd_gate_kernel<IO_F16><<<eb, 256, 0, s>>>(p, w.dy, w.ypre, w.dyp, w.dz, count); break;
            case IO_BF16: bwd_gate_kernel<IO_BF16><<<eb, 256, 0, s>>>(p, w.dy, w.ypre, w.dyp, w.dz, count); break;
            default: return cudaErrorInvalidValue;
        }
    }
    const dim3 grid(p.B * p.H, p.nchunks);
    switch (io) {
        case IO_F32: bwd_chunk_adjoint_kernel<IO_F32><<<grid, kThreads, 0, s>>>(p, w.cs, dyp, w.adj); break;
        case IO_F16: bwd_chunk_adjoint_kernel<IO_F16><<<grid, kThreads, 0, s>>>(p, w.cs, dyp, w.adj); break;
        case IO_BF16: bwd_chunk_adjoint_kernel<IO_BF16><<<grid, kThreads, 0, s>>>(p, w.cs, dyp, w.adj); break;
    }
    const int PN = p.P * p.N;  // a multiple of 256: P, N are multiples of 16
    bwd_state_passing_kernel<<<dim3(p.B * p.H, (PN / 4 + kThreads - 1) / kThreads), kThreads, 0, s>>>(
        p, w.cs, w.dfinal, w.adj, w.dh0);
    const int smem = (int)sizeof(ChunkSmem);
    cudaError_t e;
    int dev = 0, wave = 0;  // CTAs resident at once: one per SM
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&wave, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess) {
        (void)cudaGetLastError();
        wave = 0;  // no prefetch
    }
    switch (io) {
        case IO_F32:
            if ((e = cudaFuncSetAttribute(bwd_chunk_kernel<IO_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          smem)) != cudaSuccess)
                return e;
            bwd_chunk_kernel<IO_F32><<<grid, kThreads, smem, s>>>(p, w.dtp, w.cs, w.states, w.adj, dyp, w.dx,
                                                                  w.ddt, w.dBh, w.dCh, w.partA, w.partD, w.partBias, wave);
            break;
        case IO_F16:
            if ((e = cudaFuncSetAttribute(bwd_chunk_kernel<IO_F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          smem)) != cudaSuccess)
                return e;
            bwd_chunk_kernel<IO_F16><<<grid, kThreads, smem, s>>>(p, w.dtp, w.cs, w.states, w.adj, dyp, w.dx,
                                                                  w.ddt, w.dBh, w.dCh, w.partA, w.partD, w.partBias, wave);
            break;
        case IO_BF16:
            if ((e = cudaFuncSetAttribute(bwd_chunk_kernel<IO_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          smem)) != cudaSuccess)
                return e;
            bwd_chunk_kernel<IO_BF16><<<grid, kThreads, smem, s>>>(p, w.dtp, w.cs, w.states, w.adj, dyp, w.dx,
                                                                   w.ddt, w.dBh, w.dCh, w.partA, w.partD, w.partBias, wave);
            break;
    }
    const size_t gtotal = (size_t)p.B * p.L * p.G * p.N / 4;
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
