// segstate.cu -- the segment passes that let the fused plan walk one sequence
// in parallel at state width N = 128, where (batch x group x head pair) alone
// is too few units for the GPU.  The sequence is cut into nseg segments of
// seg_len tokens (a multiple of 64); the fused kernel walks each segment from
// the state entering it, and these two kernels provide that state.  It is the
// chunked algorithm's inter-chunk recurrence (ops-transformer MambaV2 article,
// sections 4.3 and 4.4: chunk_state, then chunk_state_passing) taken over
// segments instead of chunks: the pages' chunk-parallel lesson (MindSpeed-Ops
// PR #101 page, the "aux" path for shapes whose batch x heads cannot fill
// the device) with the states of only nseg - 1 boundaries materialised.
//
// Pre-pass, one CTA per (batch b, group g, head pair, segment s < nseg - 1):
//     E_s[(h,p), n] = sum_{t in s} exp(sum_{t' in s, t' > t} d_t' A_h) d_t x_t[h,p] B_t[n]
//     a_s[h]        = sum_{t in s} d_t A_h
// E_s is the state segment s produces from a zero start; it is one tcgen05
// accumulation (M = 128 rows (head, p), N = 128, K = the segment's tokens in
// 64-token blocks) of bf16 / fp16 operands into an fp32 TMEM accumulator.
// The decay weight of every token is an exclusive suffix sum of d A taken
// backwards over the segment, so no large cumulative sums are subtracted.
// Warps 0-15 first compute the weights (eight warps per head, 8 consecutive
// tokens per thread), then convert the TMA-staged x and B tiles into
// operands (B moves as it is when it already has the operand type); warp 16
// issues the TMA copies into a ring of stages and prefetches the blocks after
// the ring into L2; warp 17 issues the MMAs.  Every handoff is
// an mbarrier whose wait gives up after 2 s (recorded in the workspace error
// word).
//
// Fold, one thread per 4 state elements of one (b, h):
//     S_in(0) = h0 (or 0),   S_in(s + 1) = exp(a_s) S_in(s) + E_s,
// written over E in place: seg_states[b, s] holds the state entering segment s.
#include "ssd_fused.cuh"
#include "ssd_internal.cuh"
#include "tc_operands.cuh"
#include "tc_ptx.cuh"
#include "tc_stage.cuh"

namespace ssd {

namespace {

using tcop::st_shared_v4;
using tcop::store8;
using tcstage::BOX_BYTES;
using tcstage::stage_read8;

constexpr int kNN = 128, kP = 64;
constexpr int kConvWarps = 16;
constexpr int kConvThreads = kConvWarps * 32;
constexpr int kTmaWarp = kConvWarps, kMmaWarp = kConvWarps + 1;
constexpr int kThreads = kConvThreads + 64;
constexpr uint64_t kWaitNs = 2000000000ull;

// shared memory (bytes from a 1024-aligned base): kStages staging stages of x
// (128 features) and B (128 features) of one 64-token block, two operand
// buffers of Xw^T (MN-major, 128 (h,p) x 64 j) and B (MN-major, 64 j x 128 n),
// then the weights w[2][seg_len].  The CTA streams its segment, so the stages
// in flight set its bandwidth: four with 16-bit tensors (32 KB each), two with
// fp32 (64 KB each; a third does not fit beside the operands).
template <int IO>
struct PreSmem {
    static constexpr int kStages = IO == IO_F32 ? 2 : 4;
    static constexpr uint32_t STG_BYTES = (IO == IO_F32 ? 4u : 2u) * BOX_BYTES;  // x or B of one block
    static constexpr uint32_t STG = 0;                          // stage i: x at STG + 2 i STG_BYTES, B after it
    static constexpr uint32_t XT = 2 * kStages * STG_BYTES;     // operand buffer i at XT + i OP_BYTES
    static constexpr uint32_t OP_BYTES = 16384 + 16384;         // Xw^T, then B
    static constexpr uint32_t W = XT + 2 * OP_BYTES;
    static constexpr uint32_t bytes(int seg_len) { return W + 2u * seg_len * 4u + 1024u; }
};

constexpr int kMaxStages = 4;
constexpr int kPrefetchAhead = 2;
constexpr int kMaxSegLen = 2048;
constexpr int kHeadThreads = kConvThreads / 2;  // weight threads per head
constexpr int kTokPerThread = kMaxSegLen / kHeadThreads;
static_assert(kMaxSegLen % kHeadThreads == 0, "whole tokens per weight thread");  // blocks past the ring's last stage requested into L2
enum { PB_FULL0 = 0, PB_EMPTY0 = kMaxStages, PB_OPS0 = 2 * kMaxStages, PB_DONE0 = PB_OPS0 + 2, PB_N = PB_DONE0 + 2 };

template <int IO, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
segment_state_kernel(const __grid_constant__ Params p, const __grid_constant__ SegMaps tm, float *seg_states,
                     float *seg_decay, unsigned int *err) {
    using SM = PreSmem<IO>;
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bars[PB_N];
    __shared__ uint32_t tmem_slot;
    __shared__ float warp_total[kConvWarps];
    const uint32_t raw = tc::smem_addr(smem_raw);
    unsigned char *sm = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sbase = tc::smem_addr(sm);
    float *w_s = reinterpret_cast<float *>(sm + SM::W);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int pairs = p.hpg >> 1, nsg = p.nseg - 1;  // the last segment needs no pre-pass
    int q = blockIdx.x;
    const int pair = q % pairs;
    q /= pairs;
    const int g = q % p.G;
    q /= p.G;
    const int s = q % nsg, b = q / nsg;
    const int h0 = g * p.hpg + 2 * pair;
    const int t0 = s * p.seg_len, nblk = p.seg_len / 64;
    const uint32_t bar0 = tc::smem_addr(&bars[0]);
    auto bar = [bar0](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    bool timed_out = false;
    auto wait = [&](int i, uint32_t parity) {
        if (!timed_out && !tc::mbar_wait(bar(i), parity, kWaitNs)) timed_out = true;
    };

    constexpr int NS = SM::kStages;
    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            tc::mbar_init(bar(PB_FULL0 + i), 1);
            tc::mbar_init(bar(PB_EMPTY0 + i), kConvWarps);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(bar(PB_OPS0 + i), kConvWarps);
            tc::mbar_init(bar(PB_DONE0 + i), 1);
        }
        tc::mbar_init_fence();
    }
    if (warp == kMmaWarp) {
        tc::tmem_alloc(tc::smem_addr(&tmem_slot), kNN);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    tc::pdl_launch_dependents();  // the fold may be scheduled once every pre-pass CTA is resident
    const uint32_t tmem = tmem_slot;
    constexpr int bw = IO == IO_F32 ? 32 : 64;  // features per 128-byte box

    if (warp == kTmaWarp) {
        if (lane == 0) {
            tc::prefetch_tensormap(&tm.x);
            tc::prefetch_tensormap(&tm.b);
            auto prefetch = [&](int j) {  // block j into L2 only
#pragma unroll
                for (int bx = 0; bx < 128 / bw; ++bx) {
                    tc::tma_prefetch_3d(&tm.x, h0 * kP + bx * bw, t0 + 64 * j, b);
                    tc::tma_prefetch_3d(&tm.b, g * kNN + bx * bw, t0 + 64 * j, b);
                }
            };
            for (int j = NS; j < NS + kPrefetchAhead && j < nblk; ++j) prefetch(j);
            for (int j = 0; j < nblk; ++j) {
                const int st = j % NS;
                if (j >= NS) wait(PB_EMPTY0 + st, ((j - NS) / NS) & 1u);
                if (j + NS + kPrefetchAhead < nblk) prefetch(j + NS + kPrefetchAhead);
                const uint32_t xdst = sbase + SM::STG + 2 * st * SM::STG_BYTES, bdst = xdst + SM::STG_BYTES;
                tc::mbar_arrive_expect_tx(bar(PB_FULL0 + st), 2 * SM::STG_BYTES);
#pragma unroll
                for (int bx = 0; bx < 128 / bw; ++bx) {
                    tc::tma_load_3d(xdst + bx * BOX_BYTES, &tm.x, h0 * kP + bx * bw, t0 + 64 * j, b, bar(PB_FULL0 + st));
                    tc::tma_load_3d(bdst + bx * BOX_BYTES, &tm.b, g * kNN + bx * bw, t0 + 64 * j, b, bar(PB_FULL0 + st));
                }
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            constexpr uint32_t ID = tc::idesc_f16(128, kNN, BF16, true, true);
            for (int j = 0; j < nblk; ++j) {
                const int ob = j & 1;
                wait(PB_OPS0 + ob, (j >> 1) & 1u);
                tc::fence_after_sync();
                const uint32_t xt = sbase + SM::XT + ob * SM::OP_BYTES, bb = xt + 16384;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)  // E += Xw^T B, K = 16 tokens per step
                    tc::mma_f16(tmem, tc::desc(xt + ks * 4096, 2048, 128), tc::desc(bb + ks * 256, 128, 1024), ID,
                                (j | ks) != 0);
                tc::commit(bar(PB_DONE0 + ob));
            }
        }
        __syncwarp();
    } else {
        // ---- weights: w_t = exp(sum of d A over the segment's tokens after t) d_t.
        // The first kHeadThreads threads take head h0, the rest h0 + 1, up to
        // kTokPerThread consecutive tokens each (every load issued before the
        // first use); the suffix sums run within the thread, then over the later
        // lanes of its warp, then over the later warps of its head, each in a
        // fixed order ----
        {
            constexpr int kT = kTokPerThread, kHW = kHeadThreads / 32;  // warps per head
            const int hh = tid / kHeadThreads, i = tid % kHeadThreads, h = h0 + hh;
            const int per = (p.seg_len + kHeadThreads - 1) / kHeadThreads;  // tokens per thread
            const int tb = i * per;
            float dv[kT], ex[kT];
#pragma unroll
            for (int m = 0; m < kT; ++m) {
                const int t = tb + m;
                dv[m] = (m < per && t < p.seg_len) ? __ldg(p.dt + ((size_t)b * p.L + t0 + t) * p.H + h) : 0.f;
            }
            const float A = __ldg(p.A + h);
            float run = 0.f;  // sum of d A over this thread's tokens after token m
#pragma unroll
            for (int m = kT - 1; m >= 0; --m) {
                const bool ok = m < per && tb + m < p.seg_len;
                const float d = ok ? dt_processed(p, dv[m], h) : 0.f;
                dv[m] = d;
                ex[m] = run;
                run += d * A;
            }
            float incl = run;  // over this lane and the later lanes of the warp
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float o = __shfl_down_sync(0xffffffffu, incl, off);
                if (lane + off < 32) incl += o;
            }
            float excl = __shfl_down_sync(0xffffffffu, incl, 1);
            if (lane == 31) excl = 0.f;
            if (lane == 0) warp_total[warp] = incl;
            tc::named_barrier(1, kConvThreads);
            float later = 0.f;  // the later warps of this head, from the segment's end backwards
            for (int q = kHW * hh + kHW - 1; q > warp; --q) later += warp_total[q];
            const float base = later + excl;
#pragma unroll
            for (int m = 0; m < kT; ++m)
                if (m < per && tb + m < p.seg_len) w_s[hh * p.seg_len + tb + m] = expf(ex[m] + base) * dv[m];
            if (i == 0) {
                float total = 0.f;
                for (int q = kHW * hh + kHW - 1; q >= kHW * hh; --q) total += warp_total[q];
                seg_decay[((size_t)b * p.H + h) * p.nseg + s] = total;
            }
        }
        tc::named_barrier(1, kConvThreads);

        // ---- operands: block j of x (scaled by w) and B, from the staging ring ----
        for (int j = 0; j < nblk; ++j) {
            const int st = j % NS, ob = j & 1;
            wait(PB_FULL0 + st, (j / NS) & 1u);
            if (j >= 2) wait(PB_DONE0 + ob, ((j - 2) >> 1) & 1u);  // the MMA of block j - 2 read this buffer
            const uint32_t xsrc = sbase + SM::STG + 2 * st * SM::STG_BYTES, bsrc = xsrc + SM::STG_BYTES;
            const uint32_t xt = sbase + SM::XT + ob * SM::OP_BYTES, bb = xt + 16384;
            constexpr bool kRawB = IO != IO_F32 && ((IO == IO_BF16) == BF16);  // B is the operand already
#pragma unroll
            for (int it = 0; it < 1024 / kConvThreads; ++it) {  // 64 tokens x 16 groups of 8 features
                const int e = tid + kConvThreads * it;
                const int jl = e & 7, c16 = (e >> 3) & 15, jg = e >> 7;
                const int r = jg * 8 + jl;
                float v[8];
                stage_read8<IO>(xsrc, r, c16, v);
                const float wv = w_s[(c16 >> 3) * p.seg_len + 64 * j + r];
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] *= wv;
                store8(xt + (jg * 16 + c16) * 128 + jl * 16, v, BF16);  // row (h, p) = 8 c16 + ..
                const uint32_t bdst = bb + (c16 * 8 + jg) * 128 + jl * 16;
                if constexpr (kRawB) {
                    const uint4 u = tcstage::stage_raw16(bsrc, r, c16);
                    st_shared_v4(bdst, u.x, u.y, u.z, u.w);
                } else {
                    stage_read8<IO>(bsrc, r, c16, v);
                    store8(bdst, v, BF16);
                }
            }
            tc::fence_smem_to_async();
            __syncwarp();
            if (lane == 0) {
                tc::mbar_arrive(bar(PB_EMPTY0 + st));
                tc::mbar_arrive(bar(PB_OPS0 + ob));
            }
        }

        // ---- E_s out of TMEM: warp w reads lanes 32 (w % 4) .. + 31, kCols columns from kCols (w / 4) ----
        constexpr int kCols = kNN / (kConvWarps / 4);
        wait(PB_DONE0 + ((nblk - 1) & 1), ((nblk - 1) >> 1) & 1u);
        tc::fence_after_sync();
        const int quarter = warp & 3, part = warp >> 2;
        const int row = quarter * 32 + lane, h = row >> 6, pp = row & 63;
        float *dst = seg_states + ((((size_t)b * p.nseg + s + 1) * p.H + h0 + h) * kP + pp) * kNN + kCols * part;
        const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + kCols * part;
#pragma unroll
        for (int c = 0; c < kCols / 16; ++c) {
            float v[16];
            tc::tmem_ld16(tl + 16 * c, v);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                reinterpret_cast<float4 *>(dst + 16 * c)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
    }

    if (timed_out) atomicOr(err, 4u);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == kMmaWarp) tc::tmem_dealloc(tmem, kNN);
}

// S_in(s + 1) = exp(a_s) S_in(s) + E_s over s = 0 .. nseg - 2, in place
__global__ void __launch_bounds__(256)
segment_fold_kernel(const Params p, const float *__restrict__ seg_decay, float *seg_states) {
    tc::pdl_launch_dependents();  // the walk may be scheduled; it waits for this grid before reading states
    tc::pdl_wait();               // the pre-pass has completed
    const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;
    const int PN = kP * kNN;
    const int e = (blockIdx.y * 256 + threadIdx.x) * 4;
    if (e >= PN) return;
    const size_t sstride = (size_t)p.H * PN;  // distance between segments
    float *base = seg_states + ((size_t)b * p.nseg * p.H + h) * PN + e;
    float4 st = make_float4(0.f, 0.f, 0.f, 0.f);
    if (p.h0) st = __ldg(reinterpret_cast<const float4 *>(p.h0 + ((size_t)b * p.H + h) * PN + e));
    const float *a = seg_decay + ((size_t)b * p.H + h) * p.nseg;
    float4 nxt = *reinterpret_cast<const float4 *>(base + sstride);
    for (int s = 1; s < p.nseg; ++s) {
        const float4 loc = nxt;
        if (s + 1 < p.nseg) nxt = *reinterpret_cast<const float4 *>(base + (size_t)(s + 1) * sstride);
        const float ea = expf(__ldg(a + s - 1));
        st.x = fmaf(ea, st.x, loc.x);
        st.y = fmaf(ea, st.y, loc.y);
        st.z = fmaf(ea, st.z, loc.z);
        st.w = fmaf(ea, st.w, loc.w);
        *reinterpret_cast<float4 *>(base + (size_t)s * sstride) = st;
    }
}

template <int IO, bool BF16>
cudaError_t launch_pre(const Params &p, float *seg_states, float *seg_decay, unsigned int *err, cudaStream_t s) {
    SegMaps tm;
    cudaError_t e;
    if ((e = encode_tile_map(&tm.x, p.x, IO, (int64_t)p.H * kP, p.L, p.B, true)) != cudaSuccess) return e;
    if ((e = encode_tile_map(&tm.b, p.Bm, IO, (int64_t)p.G * kNN, p.L, p.B, true)) != cudaSuccess) return e;
    const uint32_t smem = PreSmem<IO>::bytes(p.seg_len);
    auto kern = segment_state_kernel<IO, BF16>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
    const int ctas = p.B * p.G * (p.hpg / 2) * (p.nseg - 1);
    kern<<<ctas, kThreads, smem, s>>>(p, tm, seg_states, seg_decay, err);
    return cudaGetLastError();
}

}  // namespace

int segment_max_len() { return kMaxSegLen; }

bool segment_smem_fits(int io, int seg_len) {
    const uint32_t need = io == IO_F32 ? PreSmem<IO_F32>::bytes(seg_len) : PreSmem<IO_BF16>::bytes(seg_len);
    return seg_len % 64 == 0 && seg_len <= segment_max_len() && need <= 232448u - 256u;
}

cudaError_t launch_segment_passes(const Params &p, int io, bool bf16, float *seg_states, float *seg_decay,
                                  unsigned int *err, cudaStream_t s) {
    if (p.nseg < 2) return cudaSuccess;
    cudaError_t e;
    switch (io) {
        case IO_F32: e = bf16 ? launch_pre<IO_F32, true>(p, seg_states, seg_decay, err, s)
                              : launch_pre<IO_F32, false>(p, seg_states, seg_decay, err, s); break;
        case IO_F16: e = bf16 ? launch_pre<IO_F16, true>(p, seg_states, seg_decay, err, s)
                              : launch_pre<IO_F16, false>(p, seg_states, seg_decay, err, s); break;
        default: e = bf16 ? launch_pre<IO_BF16, true>(p, seg_states, seg_decay, err, s)
                          : launch_pre<IO_BF16, false>(p, seg_states, seg_decay, err, s); break;
    }
    if (e != cudaSuccess) return e;
    // programmatic dependent launch: the fold starts as the pre-pass's last CTAs
    // run and waits for it on the device (griddepcontrol.wait)
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(p.B * p.H, (kP * kNN / 4 + 255) / 256);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, segment_fold_kernel, p, static_cast<const float *>(seg_decay), seg_states);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace ssd
