// fused_tc.cu -- the fused plan: the whole chunked SSD forward (chunk_cumsum,
// chunk_state, state_passing, chunk_scan; ops-transformer MambaV2 article,
// sections 4.2-4.5) in one persistent sm_103a kernel whose chunk states never
// leave the chip.  This is the "remove state / y_diag materialisation" item
// of the "Mamba-2 SSD for Ascend NPU" README ("Limitations and roadmap"),
// re-designed for tcgen05 tensor cores with TMEM accumulators.
//
// Work unit: (batch b, group g, head pair).  One CTA (256 threads, 8 warps)
// walks the unit's chunks in order, carrying the fp32 [P,N] states of its two
// heads in registers.  Per chunk of Q = 64 tokens (P = N = 64):
//
//   G     = C B^T                  [Q x Q]   rows duplicated to M = 128
//   dS    = Xw^T B                 [2P x N]  Xw = exp(cs_last - cs_j) dt_j x_j
//   Yoff  = S C^T                  [2P x Q]  S = state entering the chunk
//   Yint  = blockdiag(X^T) Mcat    [2P x Q]  Mcat = [M_h0^T ; M_h1^T],
//           M_h[i,j] = G[i,j] exp(cs_i - cs_j) dt_j  (j <= i, else 0)
//   y_i   = exp(cs_i) Yoff + Yint (+ D x_i) (* silu(z_i))
//   S    <- exp(cs_last) S + dS
//
// All four products are tcgen05.mma kind::f16 (bf16 or fp16 operands, fp32
// accumulation in TMEM), M = 128, N = 64.  Rows of the transposed outputs are
// (head, p), so the two heads of the pair stack along M and share the C / B
// operands; the intra-chunk product reaches M = 128 with a zero block between
// the heads' x tiles.  Operands are written into shared memory in the
// no-swizzle block layout (see tc_ptx.cuh) straight from the natural
// row-major global layout: x, B and C tiles are MN- or K-major as they come,
// so no transposes are needed.  The next chunk's inputs are loaded into
// registers while the current chunk computes.
#include <stdio.h>

#include "ssd_fused.cuh"
#include "ssd_internal.cuh"
#include "tc_ptx.cuh"

namespace ssd {

namespace {

constexpr int kQ = 64, kN = 64, kP = 64;
constexpr int kThreads = 256;
constexpr uint64_t kWaitNs = 2000000000ull;  // an mbarrier wait gives up after 2 s

// shared-memory layout, bytes from a 1024-aligned base
constexpr uint32_t OFF_CB2 = 0;      // C twice (rows 0-63, 64-127), K-major, 16 KB
constexpr uint32_t OFF_BB = 16384;   // B blocks (j, n), 8 KB: K-major for G, MN-major for dS
constexpr uint32_t OFF_XT = 24576;   // Xw^T, MN-major, 128 (h,p) x 64 j, 16 KB
constexpr uint32_t OFF_XC = 40960;   // [X_h0 | 0 | X_h1], MN-major, 192 rows x 64 j, 24 KB
constexpr uint32_t OFF_MC = 65536;   // Mcat, K-major B operand, 64 i x 128 (h', j), 16 KB
constexpr uint32_t OFF_S = 81920;    // S, K-major, 128 (h,p) x 64 n, 16 KB
constexpr uint32_t OFF_VEC = 98304;  // per-chunk vectors
constexpr uint32_t SMEM_BYTES = OFF_VEC + 4096 + 1024;  // + alignment slack

// TMEM columns (256 allocated)
constexpr uint32_t TM_G = 0, TM_DS = 64, TM_YOFF = 128, TM_YINT = 192, TM_COLS = 256;

struct ChunkVec {
    float d[2][kQ];    // processed step
    float cs[2][kQ];   // within-chunk cumulative d*A
    float ecs[2][kQ];  // exp(cs)
    float w[2][kQ];    // exp(cs_last - cs) * d
    float a[2];        // exp(cs_last)
};

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool bf16) {
    if (bf16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&v);
    }
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint32_t saddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ void store8(uint32_t saddr, const float (&v)[8], bool bf16) {
    st_shared_v4(saddr, pack2(v[0], v[1], bf16), pack2(v[2], v[3], bf16), pack2(v[4], v[5], bf16),
                 pack2(v[6], v[7], bf16));
}

// 8 consecutive elements of a public tensor as floats (zeros when !valid)
template <int IO>
__device__ __forceinline__ void load8(const void *base, size_t off, bool valid, float (&v)[8]) {
    if (!valid) {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.f;
        return;
    }
    if (IO == IO_F32) {
        const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(base) + off);
        const float4 a = __ldg(p), b = __ldg(p + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(base) + off));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (IO == IO_BF16) {
                __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162 *>(&w[i]);
                float2 f = __bfloat1622float2(h);
                v[2 * i] = f.x; v[2 * i + 1] = f.y;
            } else {
                __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
                float2 f = __half22float2(h);
                v[2 * i] = f.x; v[2 * i + 1] = f.y;
            }
        }
    }
}

// Registers holding one chunk of inputs for this thread.
struct ChunkRegs {
    float x[4][8];   // 4 items of (token j, head h, 8 consecutive p)
    float bm[2][8];  // 2 items of (token j, 8 consecutive n)
    float cm[2][8];
    float dt;        // threads < 128: (head, token)
};

template <int IO>
__device__ __forceinline__ void load_chunk(const Params &p, int b, int g, int h0, int k, int tid,
                                           ChunkRegs &r) {
    const int tok0 = k * kQ;
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int e = tid + kThreads * it;
        const int jl = e & 7, c16 = (e >> 3) & 15, jg = e >> 7;
        const int h = c16 >> 3, po = c16 & 7, t = tok0 + jg * 8 + jl;
        load8<IO>(p.x, (((size_t)b * p.L + t) * p.H + h0 + h) * kP + 8 * po, t < p.L, r.x[it]);
    }
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int e = tid + kThreads * it;
        const int jl = e & 7, ng = (e >> 3) & 7, jg = e >> 6;
        const int t = tok0 + jg * 8 + jl;
        const size_t off = (((size_t)b * p.L + t) * p.G + g) * kN + 8 * ng;
        load8<IO>(p.Bm, off, t < p.L, r.bm[it]);
        load8<IO>(p.Cm, off, t < p.L, r.cm[it]);
    }
    r.dt = 0.f;
    if (tid < 2 * kQ) {
        const int h = tid >> 6, i = tid & 63, t = tok0 + i;
        if (t < p.L) r.dt = __ldg(p.dt + ((size_t)b * p.L + t) * p.H + h0 + h);
    }
}

template <int IO, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
ssd_fused_kernel(Params p, int n_units, unsigned int *err) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bars[3];
    __shared__ uint32_t tmem_slot;
    const uint32_t raw = tc::smem_addr(smem_raw);
    unsigned char *sm = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sbase = tc::smem_addr(sm);
    ChunkVec &V = *reinterpret_cast<ChunkVec *>(sm + OFF_VEC);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wg = warp >> 2, quarter = warp & 3;
    const int row = quarter * 32 + lane;  // TMEM lane owned by this thread
    const int my_h = row >> 6, my_p = row & 63;
    const int col0 = wg * 32;             // this thread's 32 columns of each 64-column region
    const uint32_t bar_g = tc::smem_addr(&bars[0]);
    const uint32_t bar_b = tc::smem_addr(&bars[1]);
    const uint32_t bar_c = tc::smem_addr(&bars[2]);

    if (tid == 0) {
        tc::mbar_init(bar_g, 1);
        tc::mbar_init(bar_b, 1);
        tc::mbar_init(bar_c, 1);
        tc::mbar_init_fence();
    }
    if (warp == 0) {
        tc::tmem_alloc(tc::smem_addr(&tmem_slot), TM_COLS);
        tc::tmem_relinquish();
    }
    // the zero block between the two heads' x tiles (MN groups 8..15 of Xcat)
    for (int e = tid; e < 8 * 8 * 8; e += kThreads) {  // 8 K groups x 8 MN groups x 8 rows of 16 B
        const int jg = e >> 6, mg = 8 + ((e >> 3) & 7), rr = e & 7;
        st_shared_v4(sbase + OFF_XC + (jg * 24 + mg) * 128 + rr * 16, 0u, 0u, 0u, 0u);
    }
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_slot;
    const uint32_t tlane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);

    constexpr uint32_t ID_KK = tc::idesc_f16(128, 64, BF16, false, false);
    constexpr uint32_t ID_MNMN = tc::idesc_f16(128, 64, BF16, true, true);
    constexpr uint32_t ID_MNK = tc::idesc_f16(128, 64, BF16, true, false);

    const int pairs = p.hpg >> 1;
    const int nchunks = p.nchunks;
    uint32_t parity = 0;
    bool timed_out = false;

    for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
        const int pair = unit % pairs;
        const int bg = unit / pairs;
        const int g = bg % p.G, b = bg / p.G;
        const int h0 = g * p.hpg + 2 * pair;

        // state of (head my_h, row my_p), columns n = col0 .. col0+31
        float S[32];
        if (p.h0) {
            const float4 *src = reinterpret_cast<const float4 *>(
                p.h0 + (((size_t)b * p.H + h0 + my_h) * kP + my_p) * kN + col0);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 v = __ldg(src + q);
                S[4 * q] = v.x; S[4 * q + 1] = v.y; S[4 * q + 2] = v.z; S[4 * q + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int n = 0; n < 32; ++n) S[n] = 0.f;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = S[8 * q + e];
            const int ng = (col0 >> 3) + q;
            store8(sbase + OFF_S + (ng * 16 + (row >> 3)) * 128 + (row & 7) * 16, v, BF16);
        }

        ChunkRegs cur;
        load_chunk<IO>(p, b, g, h0, 0, tid, cur);

        for (int k = 0; k < nchunks; ++k) {
            // ---- P1: processed step and within-chunk cumulative decay ----
            if (tid < 2 * kQ) {
                const int h = tid >> 6, i = tid & 63;
                V.d[h][i] = (k * kQ + i < p.L) ? dt_processed(p, cur.dt, h0 + h) : 0.f;
            }
            __syncthreads();
            if (warp < 2) {
                const int h = warp;
                const float A = __ldg(p.A + h0 + h);
                float v0 = V.d[h][lane] * A, v1 = V.d[h][lane + 32] * A;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float o0 = __shfl_up_sync(0xffffffffu, v0, off);
                    const float o1 = __shfl_up_sync(0xffffffffu, v1, off);
                    if (lane >= off) { v0 += o0; v1 += o1; }
                }
                v1 += __shfl_sync(0xffffffffu, v0, 31);
                V.cs[h][lane] = v0;
                V.cs[h][lane + 32] = v1;
            }
            __syncthreads();
            if (tid < 2 * kQ) {
                const int h = tid >> 6, i = tid & 63;
                const float c = V.cs[h][i], last = V.cs[h][kQ - 1];
                V.ecs[h][i] = expf(c);
                V.w[h][i] = expf(last - c) * V.d[h][i];
                if (i == 0) V.a[h] = expf(last);
            }
            __syncthreads();

            // ---- P2: operands into shared memory ----
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int e = tid + kThreads * it;
                const int jl = e & 7, c16 = (e >> 3) & 15, jg = e >> 7;
                const int h = c16 >> 3, po = c16 & 7;
                const int mgc = h ? 16 + po : po;
                store8(sbase + OFF_XC + (jg * 24 + mgc) * 128 + jl * 16, cur.x[it], BF16);
                const float w = V.w[h][jg * 8 + jl];
                float xs[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) xs[q] = cur.x[it][q] * w;
                store8(sbase + OFF_XT + (jg * 16 + 8 * h + po) * 128 + jl * 16, xs, BF16);
            }
#pragma unroll
            for (int it = 0; it < 2; ++it) {
                const int e = tid + kThreads * it;
                const int jl = e & 7, ng = (e >> 3) & 7, jg = e >> 6;
                store8(sbase + OFF_BB + (ng * 8 + jg) * 128 + jl * 16, cur.bm[it], BF16);
                store8(sbase + OFF_CB2 + (ng * 16 + jg) * 128 + jl * 16, cur.cm[it], BF16);
                store8(sbase + OFF_CB2 + (ng * 16 + jg + 8) * 128 + jl * 16, cur.cm[it], BF16);
            }
            if (k + 1 < nchunks) load_chunk<IO>(p, b, g, h0, k + 1, tid, cur);
            tc::fence_smem_to_async();
            tc::fence_before_sync();
            __syncthreads();

            // ---- P3: G, dS and Yoff on the tensor cores ----
            if (tid == 0) {
                tc::fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < kN / 16; ++ks)  // G = C B^T, K = n
                    tc::mma_f16(tmem + TM_G, tc::desc(sbase + OFF_CB2 + ks * 4096, 2048, 128),
                                tc::desc(sbase + OFF_BB + ks * 2048, 1024, 128), ID_KK, ks > 0);
                tc::commit(bar_g);
#pragma unroll
                for (int ks = 0; ks < kQ / 16; ++ks)  // dS = Xw^T B, K = j
                    tc::mma_f16(tmem + TM_DS, tc::desc(sbase + OFF_XT + ks * 4096, 2048, 128),
                                tc::desc(sbase + OFF_BB + ks * 256, 128, 1024), ID_MNMN, ks > 0);
#pragma unroll
                for (int ks = 0; ks < kN / 16; ++ks)  // Yoff = S C^T, K = n
                    tc::mma_f16(tmem + TM_YOFF, tc::desc(sbase + OFF_S + ks * 4096, 2048, 128),
                                tc::desc(sbase + OFF_CB2 + ks * 4096, 2048, 128), ID_KK, ks > 0);
                tc::commit(bar_b);
            }

            // ---- P4: masked, decayed C B^T -> Mcat ----
            if (!timed_out && !tc::mbar_wait(bar_g, parity, kWaitNs)) timed_out = true;
            tc::fence_after_sync();
            {
                float gv[32];
                tc::tmem_ld32(tlane + TM_G + col0, gv);
                const int i = row & 63, h = row >> 6;
                const float csi = V.cs[h][i];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float m[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int j = col0 + 8 * q + e;
                        m[e] = (j <= i) ? gv[8 * q + e] * expf(csi - V.cs[h][j]) * V.d[h][j] : 0.f;
                    }
                    const int kg = 8 * h + (col0 >> 3) + q;
                    store8(sbase + OFF_MC + (kg * 8 + (i >> 3)) * 128 + (i & 7) * 16, m, BF16);
                }
            }
            tc::fence_smem_to_async();
            tc::fence_before_sync();
            __syncthreads();

            // ---- P5: Yint = blockdiag(X^T) Mcat ----
            if (tid == 0) {
                tc::fence_after_sync();
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                    for (int ks = 0; ks < kQ / 16; ++ks)
                        tc::mma_f16(tmem + TM_YINT,
                                    tc::desc(sbase + OFF_XC + hh * 1024 + ks * 6144, 3072, 128),
                                    tc::desc(sbase + OFF_MC + hh * 8192 + ks * 2048, 1024, 128), ID_MNK,
                                    (hh | ks) != 0);
                tc::commit(bar_c);
            }

            // ---- P6: state update S <- exp(cs_last) S + dS ----
            if (!timed_out && !tc::mbar_wait(bar_b, parity, kWaitNs)) timed_out = true;
            tc::fence_after_sync();
            {
                float ds[32];
                tc::tmem_ld32(tlane + TM_DS + col0, ds);
                const float a = V.a[my_h];
#pragma unroll
                for (int n = 0; n < 32; ++n) S[n] = fmaf(a, S[n], ds[n]);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = S[8 * q + e];
                    const int ng = (col0 >> 3) + q;
                    store8(sbase + OFF_S + (ng * 16 + (row >> 3)) * 128 + (row & 7) * 16, v, BF16);
                }
            }

            // ---- P7: epilogue y = exp(cs) Yoff + Yint (+ D x) (* silu z) ----
            if (!timed_out && !tc::mbar_wait(bar_c, parity, kWaitNs)) timed_out = true;
            tc::fence_after_sync();
            {
                float yo[32], yi[32];
                tc::tmem_ld32(tlane + TM_YOFF + col0, yo);
                tc::tmem_ld32(tlane + TM_YINT + col0, yi);
                const int h = h0 + my_h;
                const float Dh = p.D ? __ldg(p.D + h) : 0.f;
#pragma unroll
                for (int ii = 0; ii < 32; ++ii) {
                    const int i = col0 + ii, t = k * kQ + i;
                    if (t >= p.L) continue;
                    const size_t off = (((size_t)b * p.L + t) * p.H + h) * kP + my_p;
                    float v = fmaf(V.ecs[my_h][i], yo[ii], yi[ii]);
                    if (p.D) v = fmaf(Dh, ld_io<IO>(p.x, off), v);
                    if (p.z) v *= silu_f(ld_io<IO>(p.z, off));
                    st_io<IO>(p.y, off, v);
                }
            }
            tc::fence_before_sync();
            parity ^= 1u;
        }

        if (p.final_state) {
            float4 *dst = reinterpret_cast<float4 *>(
                p.final_state + (((size_t)b * p.H + h0 + my_h) * kP + my_p) * kN + col0);
#pragma unroll
            for (int q = 0; q < 8; ++q) dst[q] = make_float4(S[4 * q], S[4 * q + 1], S[4 * q + 2], S[4 * q + 3]);
        }
        __syncthreads();
    }

    if (timed_out) atomicOr(err, 1u);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, TM_COLS);
}

int g_num_sms = 0;

int num_sms() {
    if (g_num_sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (g_num_sms <= 0) g_num_sms = 1;
    }
    return g_num_sms;
}

int64_t fused_units(const ssd_fwd_args *a) { return a->B * a->G * ((a->H / a->G) / 2); }

template <int IO, bool BF16>
cudaError_t launch_typed(const Params &p, int units, unsigned int *err, cudaStream_t s) {
    auto kern = ssd_fused_kernel<IO, BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int grid = units < num_sms() * per_sm ? units : num_sms() * per_sm;
    kern<<<grid, kThreads, SMEM_BYTES, s>>>(p, units, err);
    return cudaGetLastError();
}

}  // namespace

const char *fused_unsupported_reason(const ssd_fwd_args *a) {
    if (a->P != kP || a->N != kN || a->chunk != kQ) return "needs P = N = chunk = 64";
    if ((a->H / a->G) % 2 != 0) return "needs an even number of heads per group";
    if (a->ops == SSD_OPS_F32) return "needs fp16 or bf16 operands (the fp32 path is the chunked plan)";
    if (fused_units(a) > 0x7fffffffLL) return "too many (batch, group, head pair) units";
    return nullptr;
}

bool fused_supported(const ssd_fwd_args *a) { return fused_unsupported_reason(a) == nullptr; }

bool fused_preferred(const ssd_fwd_args *a) { return fused_units(a) >= num_sms(); }

size_t fused_workspace_size(const ssd_fwd_args *) { return 256; }

cudaError_t run_fused(const ssd_fwd_args *a, cudaStream_t s) {
    Params p;
    p.B = (int)a->B; p.L = (int)a->L; p.H = (int)a->H; p.P = (int)a->P; p.N = (int)a->N;
    p.G = (int)a->G; p.Q = (int)a->chunk;
    p.nchunks = (int)((a->L + a->chunk - 1) / a->chunk);
    p.hpg = (int)(a->H / a->G);
    p.x = a->x; p.dt = a->dt; p.A = a->A; p.Bm = a->Bm; p.Cm = a->Cm; p.D = a->D; p.z = a->z;
    p.dt_bias = a->dt_bias; p.h0 = a->initial_state; p.y = a->y; p.final_state = a->final_state;
    p.dt_softplus = a->dt_softplus ? 1 : 0;
    p.has_limit = !(a->dt_min == 0.f && isinf(a->dt_max) && a->dt_max > 0.f);
    p.dt_min = a->dt_min; p.dt_max = a->dt_max;
    unsigned int *err = static_cast<unsigned int *>(a->workspace);
    cudaError_t e = cudaMemsetAsync(err, 0, 256, s);
    if (e != cudaSuccess) return e;
    const int units = (int)fused_units(a);
    const bool bf16 = a->ops == SSD_OPS_BF16;
    switch (a->x_dtype) {
        case SSD_F32: return bf16 ? launch_typed<IO_F32, true>(p, units, err, s) : launch_typed<IO_F32, false>(p, units, err, s);
        case SSD_F16: return bf16 ? launch_typed<IO_F16, true>(p, units, err, s) : launch_typed<IO_F16, false>(p, units, err, s);
        case SSD_BF16: return bf16 ? launch_typed<IO_BF16, true>(p, units, err, s) : launch_typed<IO_BF16, false>(p, units, err, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace ssd
