// chunk_tc.cu -- tensor-core (tcgen05, sm_103a) versions of step 2
// (chunk_state) and step 4 (chunk_scan) of the chunked SSD forward
// (ops-transformer MambaV2 article, sections 4.3 and 4.5), used by the
// chunked plan when the operands are fp16 / bf16.  They take the shapes the
// fused kernel does not: N = 64 or 128 and chunks of 128 or 256 tokens, where
// (batch x group) alone is too little parallelism for a chunk-sequential
// kernel, so every chunk gets its own CTAs and the states go through HBM.
//
// Both kernels pair two heads of a group along the MMA's M = 128 rows
// (rows = (head, p), P = 64), exactly like the fused kernel, and write their
// operands into the no-swizzle 8x16-byte block layout of tc_ptx.cuh straight
// from the row-major global tensors.  256 threads: warp w reads TMEM lanes
// 32 (w % 4) .. +31 and the column half w / 4.  Two CTAs fit on an SM; each
// waits for its own MMAs, and the other CTA's work fills the gaps.
//
// chunk_state:  CTA = (unit (b, g, head pair), chunk k)
//     dS[(h,p), n] = sum_j Xw[j, (h,p)] B[j, n],  Xw = exp(cs_last - cs_j) dt_j x_j
//     64 tokens at a time: Xw^T (MN-major) x B (MN-major), fp32 in TMEM.
//
// chunk_scan:   CTA = (unit, chunk k, 128-token output tile i0)
//     Yint^T = sum over 64-token source blocks jb <= tile:
//              blockdiag(X_h0^T, X_h1^T) x [M_h0^T ; M_h1^T]
//              M_h[i,j] = (C_i . B_j) exp(cs_i - cs_j) dt_j   (j <= i)
//              with C_i . B_j = G from its own MMA (M = 128 rows i)
//     Yoff^T = S_in x C^T
//     y_i    = exp(cs_i) Yoff + Yint (+ D x_i) (* silu(z_i))
#include "ssd_internal.cuh"
#include "tc_operands.cuh"
#include "tc_ptx.cuh"

namespace ssd {

namespace {

using tcop::ex2_approx;
using tcop::load8;
using tcop::st_shared_v4;
using tcop::store8;

constexpr int kP = 64;
constexpr int kThreads = 256;
constexpr uint64_t kWaitNs = 2000000000ull;  // an mbarrier wait gives up after 2 s
constexpr int kMaxQ = 256;

template <int IO>
__host__ __device__ constexpr size_t io_bytes() { return IO == IO_F32 ? 4 : 2; }

__device__ __forceinline__ void report_timeout(unsigned int *err) {
    if (err) atomicOr(err, 2u);
}

// ------------------------------------------------------------------ chunk_state

template <int N>
struct StateSmem {
    static constexpr uint32_t XT = 0;                    // Xw^T, MN-major, 128 x 64 j (16 KB)
    static constexpr uint32_t BM = 16384;                // B, MN-major (MN = n, K = j), 64 x N
    static constexpr uint32_t W = BM + 64 * N * 2;       // w[2][kMaxQ] floats
    static constexpr uint32_t BYTES = W + 2 * kMaxQ * 4 + 1024;
};

template <int IO, bool BF16, int N>
__global__ void __launch_bounds__(kThreads, 2)
chunk_state_tc_kernel(const __grid_constant__ Params p, const float *__restrict__ dtp,
                      const float *__restrict__ cs, float *__restrict__ states, unsigned int *err) {
    using SM = StateSmem<N>;
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t mma_bar;
    __shared__ uint32_t tmem_slot;
    const uint32_t raw = tc::smem_addr(smem_raw);
    unsigned char *sm = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sbase = tc::smem_addr(sm);
    float *w_s = reinterpret_cast<float *>(sm + SM::W);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int pairs = p.hpg >> 1;
    const int unit = blockIdx.x, k = blockIdx.y;
    const int pair = unit % pairs, bg = unit / pairs;
    const int g = bg % p.G, b = bg / p.G;
    const int h0 = g * p.hpg + 2 * pair;
    const int Q = p.Q, L = p.L, H = p.H;
    const uint32_t bar = tc::smem_addr(&mma_bar);

    if (tid == 0) {
        tc::mbar_init(bar, 1);
        tc::mbar_init_fence();
    }
    if (warp == 0) {
        tc::tmem_alloc(tc::smem_addr(&tmem_slot), N);
        tc::tmem_relinquish();
    }
    // pull the chunk's x rows (both heads) and B rows into L2 now; the 64-token
    // blocks below then load from L2 instead of waiting on HBM one by one
    for (int i = tid; i < Q; i += kThreads) {
        const int t = k * Q + i;
        if (t < L) {
            tc::prefetch_l2(static_cast<const char *>(p.x) + (((size_t)b * L + t) * H + h0) * kP * io_bytes<IO>(),
                            2 * kP * io_bytes<IO>());
            tc::prefetch_l2(static_cast<const char *>(p.Bm) + (((size_t)b * L + t) * p.G + g) * N * io_bytes<IO>(),
                            N * io_bytes<IO>());
        }
    }
    // w[h][i] = exp(cs[Q-1] - cs[i]) * dtp[i] (exponent <= 0)
    for (int e = tid; e < 2 * Q; e += kThreads) {
        const int h = e / Q, i = e % Q;
        const size_t row = (((size_t)b * H + h0 + h) * p.nchunks + k) * Q;
        w_s[h * kMaxQ + i] = expf(__ldg(cs + row + Q - 1) - __ldg(cs + row + i)) * __ldg(dtp + row + i);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_slot;
    constexpr uint32_t ID = tc::idesc_f16(128, N, BF16, true, true);
    bool timed_out = false;

    for (int jb = 0; jb < Q / 64; ++jb) {
        const int t0 = k * Q + jb * 64;
#pragma unroll
        for (int it = 0; it < 4; ++it) {  // x: (token, head, 8 p) items
            const int e = tid + kThreads * it;
            const int jl = e & 7, c16 = (e >> 3) & 15, jg = e >> 7;
            const int h = c16 >> 3, po = c16 & 7, t = t0 + jg * 8 + jl;
            float v[8];
            load8<IO>(p.x, (((size_t)b * L + t) * H + h0 + h) * kP + 8 * po, t < L, v);
            const float w = w_s[h * kMaxQ + jb * 64 + jg * 8 + jl];
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] *= w;
            store8(sbase + SM::XT + (jg * 16 + 8 * h + po) * 128 + jl * 16, v, BF16);
        }
#pragma unroll
        for (int it = 0; it < N / 32; ++it) {  // B: (token, 8 n) items
            const int e = tid + kThreads * it;
            const int jl = e & 7, ng = (e >> 3) & (N / 8 - 1), jg = e / N;
            const int t = t0 + jg * 8 + jl;
            float v[8];
            load8<IO>(p.Bm, (((size_t)b * L + t) * p.G + g) * N + 8 * ng, t < L, v);
            store8(sbase + SM::BM + (ng * 8 + jg) * 128 + jl * 16, v, BF16);
        }
        tc::fence_smem_to_async();
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                tc::mma_f16(tmem, tc::desc(sbase + SM::XT + ks * 4096, 2048, 128),
                            tc::desc(sbase + SM::BM + ks * 256, 128, 1024), ID, (jb | ks) != 0);
            tc::commit(bar);
        }
        if (!timed_out && !tc::mbar_wait(bar, jb & 1, kWaitNs)) timed_out = true;
        tc::fence_after_sync();
    }

    // states[b, k, h, p, n] from TMEM: lane (h, p), columns n
    {
        const int quarter = warp & 3, half = warp >> 2;
        const int row = quarter * 32 + lane;
        const int h = row >> 6, pp = row & 63;
        float *dst = states + ((((size_t)b * p.nchunks + k) * H + h0 + h) * kP + pp) * N;
        const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
#pragma unroll
        for (int c = 0; c < N / 32; ++c) {
            const int n0 = half * (N / 2) + 16 * c;
            float v[16];
            tc::tmem_ld16(tl + n0, v);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                *reinterpret_cast<float4 *>(dst + n0 + 4 * q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
    }
    if (timed_out) report_timeout(err);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, N);
}

// ------------------------------------------------------------------ chunk_scan

template <int N>
struct ScanSmem {
    static constexpr uint32_t CI = 0;                 // C of the 128-token tile, K-major, 128 x N
    static constexpr uint32_t U = 128 * N * 2;        // union: [B_j (64 x N) | Xcat (24 KB)], then S (128 x N)
    static constexpr uint32_t BJ = U;
    static constexpr uint32_t XC = U + 64 * N * 2;
    static constexpr uint32_t U_BYTES = (64 * N * 2 + 24576) > 128 * N * 2 ? (64 * N * 2 + 24576) : 128 * N * 2;
    static constexpr uint32_t MC = U + U_BYTES;       // Mcat, K-major, 128 i x 128 (h', j), 32 KB
    static constexpr uint32_t VEC = MC + 32768;       // cs2[2][kMaxQ], dt[2][kMaxQ], cs[2][kMaxQ]
    static constexpr uint32_t BYTES = VEC + 3 * 2 * kMaxQ * 4 + 1024;
};

template <int IO, bool BF16, int N>
__global__ void __launch_bounds__(kThreads, 2)
chunk_scan_tc_kernel(const __grid_constant__ Params p, const float *__restrict__ dtp,
                     const float *__restrict__ cs, const float *__restrict__ states, unsigned int *err) {
    using SM = ScanSmem<N>;
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t mma_bar;
    __shared__ uint32_t tmem_slot;
    const uint32_t raw = tc::smem_addr(smem_raw);
    unsigned char *sm = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sbase = tc::smem_addr(sm);
    float *cs2_s = reinterpret_cast<float *>(sm + SM::VEC);
    float *dt_s = cs2_s + 2 * kMaxQ;
    float *cs_s = dt_s + 2 * kMaxQ;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int pairs = p.hpg >> 1;
    const int unit = blockIdx.x, k = blockIdx.y, i0 = blockIdx.z * 128;
    const int pair = unit % pairs, bg = unit / pairs;
    const int g = bg % p.G, b = bg / p.G;
    const int h0 = g * p.hpg + 2 * pair;
    const int Q = p.Q, L = p.L, H = p.H;
    const uint32_t bar = tc::smem_addr(&mma_bar);
    constexpr float kLog2e = 1.4426950408889634f;

    if (tid == 0) {
        tc::mbar_init(bar, 1);
        tc::mbar_init_fence();
    }
    if (warp == 0) {
        tc::tmem_alloc(tc::smem_addr(&tmem_slot), 256);
        tc::tmem_relinquish();
    }
    // pull everything this CTA reads after C into L2 now: x and B rows of the
    // source blocks, z rows of the tile, the two heads' entering states
    for (int i = tid; i < i0 + 128; i += kThreads) {
        const int t = k * Q + i;
        if (t < L) {
            const size_t xrow = (((size_t)b * L + t) * H + h0) * kP * io_bytes<IO>();
            tc::prefetch_l2(static_cast<const char *>(p.x) + xrow, 2 * kP * io_bytes<IO>());
            tc::prefetch_l2(static_cast<const char *>(p.Bm) + (((size_t)b * L + t) * p.G + g) * N * io_bytes<IO>(),
                            N * io_bytes<IO>());
            if (p.z && i >= i0) tc::prefetch_l2(static_cast<const char *>(p.z) + xrow, 2 * kP * io_bytes<IO>());
        }
    }
    if (tid < 2 * kP * N * 4 / 16384) {  // 16 KB pieces of the 2 x [P, N] fp32 states
        const char *st = reinterpret_cast<const char *>(states + (((size_t)b * p.nchunks + k) * H + h0) * kP * N);
        tc::prefetch_l2(st + (size_t)tid * 16384, 16384);
    }
    for (int e = tid; e < 2 * Q; e += kThreads) {
        const int h = e / Q, i = e % Q;
        const size_t row = (((size_t)b * H + h0 + h) * p.nchunks + k) * Q;
        const float c = __ldg(cs + row + i);
        cs_s[h * kMaxQ + i] = c;
        cs2_s[h * kMaxQ + i] = c * kLog2e;
        dt_s[h * kMaxQ + i] = __ldg(dtp + row + i);
    }
    // C of the output tile, K-major (rows i, K = n)
#pragma unroll
    for (int it = 0; it < N / 16; ++it) {
        const int e = tid + kThreads * it;
        const int il = e & 7, ng = (e >> 3) & (N / 8 - 1), ig = e / N;
        const int t = k * Q + i0 + ig * 8 + il;
        float v[8];
        load8<IO>(p.Cm, (((size_t)b * L + t) * p.G + g) * N + 8 * ng, t < L, v);
        store8(sbase + SM::CI + (ng * 16 + ig) * 128 + il * 16, v, BF16);
    }
    // the zero block between the two heads' x tiles (MN groups 8..15 of Xcat)
    for (int e = tid; e < 8 * 8 * 8; e += kThreads) {
        const int jg = e >> 6, mg = 8 + ((e >> 3) & 7), rr = e & 7;
        st_shared_v4(sbase + SM::XC + (jg * 24 + mg) * 128 + rr * 16, 0u, 0u, 0u, 0u);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_slot;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    constexpr uint32_t ID_G = tc::idesc_f16(128, 64, BF16, false, false);    // G: 128 i x 64 j
    constexpr uint32_t ID_Y = tc::idesc_f16(128, 128, BF16, true, false);    // Yint: 128 (h,p) x 128 i
    constexpr uint32_t ID_O = tc::idesc_f16(128, 128, BF16, false, false);   // Yoff: 128 (h,p) x 128 i
    constexpr uint32_t TM_YINT = 0, TM_G = 128, TM_YOFF = 128;
    bool timed_out = false;
    uint32_t phase = 0;

    const int nj = (i0 + 128) / 64;  // causal: source blocks up to the tile's last row
    for (int jb = 0; jb < nj; ++jb) {
        const int t0 = k * Q + jb * 64;
#pragma unroll
        for (int it = 0; it < N / 32; ++it) {  // B_j, K-major for G (rows j, K = n)
            const int e = tid + kThreads * it;
            const int jl = e & 7, ng = (e >> 3) & (N / 8 - 1), jg = e / N;
            const int t = t0 + jg * 8 + jl;
            float v[8];
            load8<IO>(p.Bm, (((size_t)b * L + t) * p.G + g) * N + 8 * ng, t < L, v);
            store8(sbase + SM::BJ + (ng * 8 + jg) * 128 + jl * 16, v, BF16);
        }
#pragma unroll
        for (int it = 0; it < 4; ++it) {  // x_j, MN-major, into [X_h0 | 0 | X_h1]
            const int e = tid + kThreads * it;
            const int jl = e & 7, c16 = (e >> 3) & 15, jg = e >> 7;
            const int h = c16 >> 3, po = c16 & 7, t = t0 + jg * 8 + jl;
            float v[8];
            load8<IO>(p.x, (((size_t)b * L + t) * H + h0 + h) * kP + 8 * po, t < L, v);
            store8(sbase + SM::XC + (jg * 24 + (h ? 16 + po : po)) * 128 + jl * 16, v, BF16);
        }
        tc::fence_smem_to_async();
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0) {  // G = C_i B_j^T
            tc::fence_after_sync();
#pragma unroll
            for (int ks = 0; ks < N / 16; ++ks)
                tc::mma_f16(tmem + TM_G, tc::desc(sbase + SM::CI + ks * 4096, 2048, 128),
                            tc::desc(sbase + SM::BJ + ks * 2048, 1024, 128), ID_G, ks > 0);
            tc::commit(bar);
        }
        if (!timed_out && !tc::mbar_wait(bar, phase, kWaitNs)) timed_out = true;
        phase ^= 1u;
        tc::fence_after_sync();
        {  // Mcat: M_h[i][j] for both heads, thread = row i, 32 columns j
            const int i = quarter * 32 + lane;
            const int ig = i0 + i;  // row within the chunk
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int j0 = half * 32 + 16 * c;
                float gv[16];
                tc::tmem_ld16(tl + TM_G + j0, gv);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float csi = cs2_s[h * kMaxQ + ig];
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        float m[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int jj = jb * 64 + j0 + 8 * q + e;  // source token within the chunk
                            const float v = gv[8 * q + e] * ex2_approx(csi - cs2_s[h * kMaxQ + jj]) *
                                            dt_s[h * kMaxQ + jj];
                            m[e] = (jj <= ig) ? v : 0.f;
                        }
                        const int kg = 8 * h + ((j0 + 8 * q) >> 3);
                        store8(sbase + SM::MC + (kg * 16 + (i >> 3)) * 128 + (i & 7) * 16, m, BF16);
                    }
                }
            }
        }
        tc::fence_smem_to_async();
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0) {  // Yint += blockdiag(X^T) Mcat
            tc::fence_after_sync();
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_f16(tmem + TM_YINT, tc::desc(sbase + SM::XC + hh * 1024 + ks * 6144, 3072, 128),
                                tc::desc(sbase + SM::MC + hh * 16384 + ks * 4096, 2048, 128), ID_Y,
                                (jb | hh | ks) != 0);
            tc::commit(bar);
        }
        if (!timed_out && !tc::mbar_wait(bar, phase, kWaitNs)) timed_out = true;
        phase ^= 1u;
        tc::fence_after_sync();
    }

    // S_in of both heads, K-major (rows (h, p), K = n), into the union region
#pragma unroll
    for (int it = 0; it < N / 16; ++it) {
        const int e = tid + kThreads * it;
        const int rr = e & 7, ng = (e >> 3) & (N / 8 - 1), mg = e / N;
        const int row = mg * 8 + rr, h = row >> 6, pp = row & 63;
        const float4 *src = reinterpret_cast<const float4 *>(
            states + ((((size_t)b * p.nchunks + k) * H + h0 + h) * kP + pp) * N + 8 * ng);
        const float4 a = __ldg(src), c = __ldg(src + 1);
        const float v[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
        store8(sbase + SM::U + (ng * 16 + mg) * 128 + rr * 16, v, BF16);
    }
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    if (tid == 0) {  // Yoff = S C_i^T
        tc::fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < N / 16; ++ks)
            tc::mma_f16(tmem + TM_YOFF, tc::desc(sbase + SM::U + ks * 4096, 2048, 128),
                        tc::desc(sbase + SM::CI + ks * 4096, 2048, 128), ID_O, ks > 0);
        tc::commit(bar);
    }
    if (!timed_out && !tc::mbar_wait(bar, phase, kWaitNs)) timed_out = true;
    tc::fence_after_sync();

    // epilogue: lane (h, p), 64 columns i of this thread's half
    {
        const int row = quarter * 32 + lane, h = row >> 6, pp = row & 63;
        const float Dh = p.D ? __ldg(p.D + h0 + h) : 0.f;
        const size_t step = (size_t)H * kP;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            const int ic = half * 64 + 16 * c;  // column within the tile
            float yo[16], yi[16];
            tc::tmem_ld16(tl + TM_YOFF + ic, yo);
            tc::tmem_ld16(tl + TM_YINT + ic, yi);
            const int tb = k * Q + i0 + ic;
            float ev[16];
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) ev[ii] = __expf(cs_s[h * kMaxQ + i0 + ic + ii]);  // cs <= 0
            const size_t off0 = (((size_t)b * L + tb) * H + h0 + h) * kP + pp;
            float v[16];
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) v[ii] = fmaf(ev[ii], yo[ii], yi[ii]);
            if (p.D) {
#pragma unroll
                for (int ii = 0; ii < 16; ++ii)
                    if (tb + ii < L) v[ii] = fmaf(Dh, ld_io<IO>(p.x, off0 + ii * step), v[ii]);
            }
            if (p.z) {
#pragma unroll
                for (int ii = 0; ii < 16; ++ii)
                    if (tb + ii < L) v[ii] *= silu_fast(ld_io<IO>(p.z, off0 + ii * step));
            }
#pragma unroll
            for (int ii = 0; ii < 16; ++ii)
                if (tb + ii < L) st_io<IO>(p.y, off0 + ii * step, v[ii]);
        }
    }
    if (timed_out) report_timeout(err);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

template <typename K>
cudaError_t set_smem(K kern, uint32_t bytes) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int IO, bool BF16, int N>
cudaError_t launch_state(const Params &p, const float *dtp, const float *cs, float *states, unsigned int *err,
                         cudaStream_t s) {
    auto kern = chunk_state_tc_kernel<IO, BF16, N>;
    cudaError_t e = set_smem(kern, StateSmem<N>::BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid(p.B * p.G * (p.hpg / 2), p.nchunks);
    kern<<<grid, kThreads, StateSmem<N>::BYTES, s>>>(p, dtp, cs, states, err);
    return cudaGetLastError();
}

template <int IO, bool BF16, int N>
cudaError_t launch_scan(const Params &p, const float *dtp, const float *cs, const float *states, unsigned int *err,
                        cudaStream_t s) {
    auto kern = chunk_scan_tc_kernel<IO, BF16, N>;
    cudaError_t e = set_smem(kern, ScanSmem<N>::BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid(p.B * p.G * (p.hpg / 2), p.nchunks, p.Q / 128);
    kern<<<grid, kThreads, ScanSmem<N>::BYTES, s>>>(p, dtp, cs, states, err);
    return cudaGetLastError();
}

template <int IO, bool BF16>
cudaError_t dispatch_state(const Params &p, const float *dtp, const float *cs, float *states, unsigned int *err,
                           cudaStream_t s) {
    return p.N == 64 ? launch_state<IO, BF16, 64>(p, dtp, cs, states, err, s)
                     : launch_state<IO, BF16, 128>(p, dtp, cs, states, err, s);
}

template <int IO, bool BF16>
cudaError_t dispatch_scan(const Params &p, const float *dtp, const float *cs, const float *states, unsigned int *err,
                          cudaStream_t s) {
    return p.N == 64 ? launch_scan<IO, BF16, 64>(p, dtp, cs, states, err, s)
                     : launch_scan<IO, BF16, 128>(p, dtp, cs, states, err, s);
}

}  // namespace

bool chunk_tc_state_supported(const Params &p, int ops) {
    return ops != SSD_OPS_F32 && p.P == kP && (p.N == 64 || p.N == 128) && p.Q % 64 == 0 && p.Q <= kMaxQ &&
           p.hpg % 2 == 0;
}

bool chunk_tc_scan_supported(const Params &p, int ops) {
    return ops != SSD_OPS_F32 && p.P == kP && (p.N == 64 || p.N == 128) && p.Q % 128 == 0 && p.Q <= kMaxQ &&
           p.hpg % 2 == 0;
}

cudaError_t launch_chunk_state_tc(const Params &p, int io, int ops, const float *dtp, const float *cs,
                                  float *states, unsigned int *err, cudaStream_t s) {
    const bool bf16 = ops == SSD_OPS_BF16;
    switch (io) {
        case IO_F32: return bf16 ? dispatch_state<IO_F32, true>(p, dtp, cs, states, err, s) : dispatch_state<IO_F32, false>(p, dtp, cs, states, err, s);
        case IO_F16: return bf16 ? dispatch_state<IO_F16, true>(p, dtp, cs, states, err, s) : dispatch_state<IO_F16, false>(p, dtp, cs, states, err, s);
        case IO_BF16: return bf16 ? dispatch_state<IO_BF16, true>(p, dtp, cs, states, err, s) : dispatch_state<IO_BF16, false>(p, dtp, cs, states, err, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_chunk_scan_tc(const Params &p, int io, int ops, const float *dtp, const float *cs,
                                 const float *states, unsigned int *err, cudaStream_t s) {
    const bool bf16 = ops == SSD_OPS_BF16;
    switch (io) {
        case IO_F32: return bf16 ? dispatch_scan<IO_F32, true>(p, dtp, cs, states, err, s) : dispatch_scan<IO_F32, false>(p, dtp, cs, states, err, s);
        case IO_F16: return bf16 ? dispatch_scan<IO_F16, true>(p, dtp, cs, states, err, s) : dispatch_scan<IO_F16, false>(p, dtp, cs, states, err, s);
        case IO_BF16: return bf16 ? dispatch_scan<IO_BF16, true>(p, dtp, cs, states, err, s) : dispatch_scan<IO_BF16, false>(p, dtp, cs, states, err, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace ssd
