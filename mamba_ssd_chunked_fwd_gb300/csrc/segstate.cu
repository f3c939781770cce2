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
// Pre-pass, one work item per (batch b, group g, head pair, segment s < nseg - 1),
// persistent CTAs (one per SM at most) walking the items:
//     E_s[(h,p), n] = sum_{t in s} exp(sum_{t' in s, t' > t} d_t' A_h) d_t x_t[h,p] B_t[n]
//     a_s[h]        = sum_{t in s} d_t A_h
// E_s is the state segment s produces from a zero start; it is one tcgen05
// accumulation (M = 128 rows (head, p), N = 128, K = the segment's tokens in
// 64-token blocks) of bf16 / fp16 operands into an fp32 TMEM accumulator.
// The decay weight of every token is an exclusive suffix sum of d A taken
// backwards over the segment, so no large cumulative sums are subtracted.
// Warps 0-15 first compute the weights (up to 4 consecutive tokens of both
// heads per thread), then convert the TMA-staged x tiles (and B, unless it
// already has the operand type) into operands; warp 16 issues the TMA copies
// into a ring of stages (and with fp32 tensors prefetches the blocks after
// the ring into L2); warp 17 issues the MMAs.  Every handoff is
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
// (128 features) and B (128 features) of one 64-token block, kOpBufs operand
// buffers, then the weights w[2][seg_len].  An operand buffer holds Xw^T
// (MN-major, 128 (h,p) x 64 j), and B (MN-major, 64 j x 128 n) after it unless
// B already has the operand type: the MMA then reads B from its staging tile
// (128-byte swizzled by the TMA, which is the MN-major 128-byte-swizzle operand
// layout) and the stage stays busy until that MMA completes.  Four stages of
// 16-bit tensors (32 KB each) or two of fp32 (64 KB each) are in flight.
template <int IO, bool BF16>
struct PreSmem {
    static constexpr bool kRawB = IO != IO_F32 && ((IO == IO_BF16) == BF16);
    static constexpr int kStages = IO == IO_F32 ? 2 : 4;
    static constexpr int kOpBufs = kRawB ? 4 : 2;
    static constexpr uint32_t STG_BYTES = (IO == IO_F32 ? 4u : 2u) * BOX_BYTES;  // x or B of one block
    static constexpr uint32_t STG = 0;                          // stage i: x at STG + 2 i STG_BYTES, B after it
    static constexpr uint32_t XT = 2 * kStages * STG_BYTES;     // operand buffer i at XT + i OP_BYTES
    static constexpr uint32_t OP_BYTES = kRawB ? 16384u : 32768u;
    static constexpr uint32_t W = XT + kOpBufs * OP_BYTES;
    static constexpr uint32_t bytes(int seg_len) { return W + 2u * seg_len * 4u + 1024u; }
};

constexpr int kMaxStages = 4, kMaxOpBufs = 4;
// blocks past the ring's last stage requested into L2: fp32 only (two stages in
// flight); with 16-bit tensors the four stages suffice and the extra TMA
// requests measured slower
constexpr int kPrefetchAhead = 2;
constexpr int kMaxSegLen = 2048;
constexpr int kTokPerThread = kMaxSegLen / kConvThreads;  // weight tokens per converter thread
static_assert(kMaxSegLen % kConvThreads == 0, "whole tokens per weight thread");

// mbarriers: staging stage full / empty, operand buffer full / consumed by the
// MMA, accumulator (one per TMEM buffer) complete
enum {
    PB_FULL0 = 0,
    PB_EMPTY0 = kMaxStages,
    PB_OPS0 = 2 * kMaxStages,
    PB_DONE0 = PB_OPS0 + kMaxOpBufs,
    PB_ACC0 = PB_DONE0 + kMaxOpBufs,
    PB_N = PB_ACC0 + 2
};

// A work item: (batch b, group g, head pair, segment s < nseg - 1), the head
// pair fastest so that CTAs running side by side share their B tiles in L2.
struct PreItem {
    int b, g, h0, s;
};
__device__ __forceinline__ PreItem pre_item(const Params &p, int q) {
    const int pairs = p.hpg >> 1, nsg = p.nseg - 1;
    PreItem it;
    const int pair = q % pairs;
    q /= pairs;
    it.g = q % p.G;
    q /= p.G;
    it.s = q % nsg;
    it.b = q / nsg;
    it.h0 = it.g * p.hpg + 2 * pair;
    return it;
}

// Persistent: CTA c runs items c, c + gridDim.x, ...  The TMA warp streams the
// blocks of all of its items through one ring; the MMA warp accumulates item i
// into TMEM buffer i % 2, so the next item's products run while the converter
// warps read item i out (after the first blocks of item i + 1, by which time
// its products are complete); the raw dt of item i + 1 is loaded while item i
// converts.
template <int IO, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
segment_state_kernel(const __grid_constant__ Params p, const __grid_constant__ SegMaps tm, float *seg_states,
                     float *seg_decay, unsigned int *err) {
    using SM = PreSmem<IO, BF16>;
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bars[PB_N];
    __shared__ uint32_t tmem_slot;
    __shared__ float warp_total[2][kConvWarps];
    const uint32_t raw = tc::smem_addr(smem_raw);
    unsigned char *sm = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sbase = tc::smem_addr(sm);
    float *w_s = reinterpret_cast<float *>(sm + SM::W);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int items = p.B * p.G * (p.hpg >> 1) * (p.nseg - 1);  // the last segment needs no pre-pass
    const int mine = static_cast<int>(blockIdx.x) < items ? (items - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int nblk = p.seg_len / 64;
    const uint32_t bar0 = tc::smem_addr(&bars[0]);
    auto bar = [bar0](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    bool timed_out = false;
    auto wait = [&](int i, uint32_t parity) {
        if (!timed_out && !tc::mbar_wait(bar(i), parity, kWaitNs)) timed_out = true;
    };

    constexpr int NS = SM::kStages, NOB = SM::kOpBufs;
    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            tc::mbar_init(bar(PB_FULL0 + i), 1);
            tc::mbar_init(bar(PB_EMPTY0 + i), SM::kRawB ? kConvWarps + 1 : kConvWarps);
        }
        for (int i = 0; i < NOB; ++i) {
            tc::mbar_init(bar(PB_OPS0 + i), kConvWarps);
            tc::mbar_init(bar(PB_DONE0 + i), 1);
        }
        for (int i = 0; i < 2; ++i) tc::mbar_init(bar(PB_ACC0 + i), 1);
        tc::mbar_init_fence();
    }
    if (warp == kMmaWarp) {
        tc::tmem_alloc(tc::smem_addr(&tmem_slot), 2 * kNN);
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
            const int total = mine * nblk;
            // block gj of this CTA's sequence: block gj % nblk of item blockIdx.x + (gj / nblk) gridDim.x;
            // items are decoded once each (the issuing thread paces the ring)
            int cur_li = -1, pf_li = -1;
            PreItem cur{}, pf{};
            auto item_for = [&](int gj, int &li_cache, PreItem &cache) -> const PreItem & {
                const int li = gj / nblk;
                if (li != li_cache) {
                    li_cache = li;
                    cache = pre_item(p, blockIdx.x + li * gridDim.x);
                }
                return cache;
            };
            auto boxes = [&](const PreItem &it, int gj, uint32_t xdst, uint32_t mbar, bool load) {
                const int tok = it.s * p.seg_len + 64 * (gj % nblk);
#pragma unroll
                for (int bx = 0; bx < 128 / bw; ++bx) {
                    if (load) {
                        tc::tma_load_3d(xdst + bx * BOX_BYTES, &tm.x, it.h0 * kP + bx * bw, tok, it.b, mbar);
                        tc::tma_load_3d(xdst + SM::STG_BYTES + bx * BOX_BYTES, &tm.b, it.g * kNN + bx * bw, tok, it.b,
                                        mbar);
                    } else {
                        tc::tma_prefetch_3d(&tm.x, it.h0 * kP + bx * bw, tok, it.b);
                        tc::tma_prefetch_3d(&tm.b, it.g * kNN + bx * bw, tok, it.b);
                    }
                }
            };
            constexpr int PF = IO == IO_F32 ? kPrefetchAhead : 0;
            for (int gj = NS; gj < NS + PF && gj < total; ++gj) boxes(item_for(gj, pf_li, pf), gj, 0u, 0u, false);
            for (int gj = 0; gj < total; ++gj) {
                const int st = gj % NS;
                if (gj >= NS) wait(PB_EMPTY0 + st, ((gj - NS) / NS) & 1u);
                if (PF > 0 && gj + NS + PF < total)
                    boxes(item_for(gj + NS + PF, pf_li, pf), gj + NS + PF, 0u, 0u, false);
                tc::mbar_arrive_expect_tx(bar(PB_FULL0 + st), 2 * SM::STG_BYTES);
                boxes(item_for(gj, cur_li, cur), gj, sbase + SM::STG + 2 * st * SM::STG_BYTES, bar(PB_FULL0 + st), true);
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            constexpr uint32_t ID = tc::idesc_f16(128, kNN, BF16, true, true);
            for (int li = 0; li < mine; ++li) {
                const uint32_t acc = tmem + static_cast<uint32_t>((li & 1) * kNN);
                for (int j = 0; j < nblk; ++j) {
                    const int gj = li * nblk + j, ob = gj % NOB;
                    wait(PB_OPS0 + ob, (gj / NOB) & 1u);
                    tc::fence_after_sync();
                    const uint32_t xt = sbase + SM::XT + ob * SM::OP_BYTES;
                    if constexpr (SM::kRawB) {
                        const int st = gj % NS;
                        wait(PB_FULL0 + st, (gj / NS) & 1u);  // (complete already: the converters saw it)
                        tc::fence_after_sync();
                        const uint32_t bst = sbase + SM::STG + (2 * st + 1) * SM::STG_BYTES;
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)  // E += Xw^T B, K = 16 tokens per step
                            tc::mma_f16(acc, tc::desc(xt + ks * 4096, 2048, 128),
                                        tc::desc_sw128(bst + ks * 2048, BOX_BYTES, 1024), ID, (j | ks) != 0);
                        tc::commit(bar(PB_DONE0 + ob));
                        tc::commit(bar(PB_EMPTY0 + st));
                    } else {
                        const uint32_t bb = xt + 16384;
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            tc::mma_f16(acc, tc::desc(xt + ks * 4096, 2048, 128), tc::desc(bb + ks * 256, 128, 1024),
                                        ID, (j | ks) != 0);
                        tc::commit(bar(PB_DONE0 + ob));
                    }
                }
                tc::commit(bar(PB_ACC0 + (li & 1)));
            }
        }
        __syncwarp();
    } else {
        constexpr int kT = kTokPerThread;
        const int per = (p.seg_len + kConvThreads - 1) / kConvThreads;  // tokens per thread
        const int tb = tid * per;
        const bool pair_aligned = (reinterpret_cast<uintptr_t>(p.dt) & 7u) == 0;  // h0 is even
        // raw dt of both heads of this thread's tokens of item li (the pair's two
        // values of a token are adjacent: one 8-byte load; every load in flight at once)
        auto load_dt = [&](int li, float2 (&dv)[kT]) {
            const PreItem it = pre_item(p, blockIdx.x + li * gridDim.x);
            const float *src = p.dt + ((size_t)it.b * p.L + it.s * p.seg_len + tb) * p.H + it.h0;
#pragma unroll
            for (int m = 0; m < kT; ++m) {
                dv[m] = make_float2(0.f, 0.f);
                if (m < per && tb + m < p.seg_len) {
                    const float *q = src + (size_t)m * p.H;
                    dv[m] = pair_aligned ? __ldg(reinterpret_cast<const float2 *>(q)) : make_float2(__ldg(q), __ldg(q + 1));
                }
            }
        };
        // E of item li out of TMEM buffer li % 2: warp w reads lanes 32 (w % 4) .. + 31,
        // kCols columns from kCols (w / 4)
        auto read_out = [&](int li) {
            constexpr int kCols = kNN / (kConvWarps / 4);
            wait(PB_ACC0 + (li & 1), (li >> 1) & 1u);
            tc::fence_after_sync();
            const PreItem it = pre_item(p, blockIdx.x + li * gridDim.x);
            const int quarter = warp & 3, part = warp >> 2;
            const int row = quarter * 32 + lane, h = row >> 6, pp = row & 63;
            float *dst = seg_states + ((((size_t)it.b * p.nseg + it.s + 1) * p.H + it.h0 + h) * kP + pp) * kNN +
                         kCols * part;
            const uint32_t tl =
                tmem + static_cast<uint32_t>((li & 1) * kNN) + (static_cast<uint32_t>(quarter * 32) << 16) + kCols * part;
#pragma unroll
            for (int c = 0; c < kCols / 16; ++c) {
                float v[16];
                tc::tmem_ld16(tl + 16 * c, v);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    reinterpret_cast<float4 *>(dst + 16 * c)[i] =
                        make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            }
            tc::fence_before_sync();  // the TMEM reads precede the next products into this buffer
        };

        float2 dv[kT];
        if (mine > 0) load_dt(0, dv);
        for (int li = 0; li < mine; ++li) {
            const PreItem it = pre_item(p, blockIdx.x + li * gridDim.x);
            // every converter is done with the previous item's weights
            tc::named_barrier(1, kConvThreads);
            // ---- weights: w_t = exp(sum of d A over the segment's tokens after t) d_t for
            // heads h0 and h0 + 1.  Thread i takes tokens i per .. i per + per - 1; the
            // suffix sums run within the thread, then over the later lanes of its warp,
            // then over the later warps, each in a fixed order ----
            {
                const float A0 = __ldg(p.A + it.h0), A1 = __ldg(p.A + it.h0 + 1);
                float ex0[kT], ex1[kT];
                float run0 = 0.f, run1 = 0.f;  // sums of d A over this thread's tokens after token m
#pragma unroll
                for (int m = kT - 1; m >= 0; --m) {
                    const bool ok = m < per && tb + m < p.seg_len;
                    const float d0 = ok ? dt_processed(p, dv[m].x, it.h0) : 0.f;
                    const float d1 = ok ? dt_processed(p, dv[m].y, it.h0 + 1) : 0.f;
                    dv[m] = make_float2(d0, d1);
                    ex0[m] = run0;
                    ex1[m] = run1;
                    run0 += d0 * A0;
                    run1 += d1 * A1;
                }
                float in0 = run0, in1 = run1;  // over this lane and the later lanes of the warp
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float o0 = __shfl_down_sync(0xffffffffu, in0, off);
                    const float o1 = __shfl_down_sync(0xffffffffu, in1, off);
                    if (lane + off < 32) {
                        in0 += o0;
                        in1 += o1;
                    }
                }
                float x0 = __shfl_down_sync(0xffffffffu, in0, 1), x1 = __shfl_down_sync(0xffffffffu, in1, 1);
                if (lane == 31) x0 = x1 = 0.f;
                if (lane == 0) {
                    warp_total[0][warp] = in0;
                    warp_total[1][warp] = in1;
                }
                tc::named_barrier(1, kConvThreads);
                float later0 = 0.f, later1 = 0.f;  // the later warps, from the segment's end backwards
                for (int q = kConvWarps - 1; q > warp; --q) {
                    later0 += warp_total[0][q];
                    later1 += warp_total[1][q];
                }
                const float base0 = later0 + x0, base1 = later1 + x1;
#pragma unroll
                for (int m = 0; m < kT; ++m)
                    if (m < per && tb + m < p.seg_len) {
                        w_s[tb + m] = expf(ex0[m] + base0) * dv[m].x;
                        w_s[p.seg_len + tb + m] = expf(ex1[m] + base1) * dv[m].y;
                    }
                if (tid < 2) {
                    float total = 0.f;
                    for (int q = kConvWarps - 1; q >= 0; --q) total += warp_total[tid][q];
                    seg_decay[((size_t)it.b * p.H + it.h0 + tid) * p.nseg + it.s] = total;
                }
            }
            tc::named_barrier(1, kConvThreads);
            if (li + 1 < mine) load_dt(li + 1, dv);  // consumed at the next item's weights

            // ---- operands: block j of x (scaled by w), and of B unless the MMA reads it staged ----
            for (int j = 0; j < nblk; ++j) {
                const int gj = li * nblk + j, st = gj % NS, ob = gj % NOB;
                wait(PB_FULL0 + st, (gj / NS) & 1u);
                if (gj >= NOB) wait(PB_DONE0 + ob, ((gj - NOB) / NOB) & 1u);  // the MMA of block gj - NOB read it
                const uint32_t xsrc = sbase + SM::STG + 2 * st * SM::STG_BYTES, bsrc = xsrc + SM::STG_BYTES;
                const uint32_t xt = sbase + SM::XT + ob * SM::OP_BYTES, bb = xt + 16384;
#pragma unroll
                for (int itn = 0; itn < 1024 / kConvThreads; ++itn) {  // 64 tokens x 16 groups of 8 features
                    const int e = tid + kConvThreads * itn;
                    const int jl = e & 7, c16 = (e >> 3) & 15, jg = e >> 7;
                    const int r = jg * 8 + jl;
                    float v[8];
                    stage_read8<IO>(xsrc, r, c16, v);
                    const float wv = w_s[(c16 >> 3) * p.seg_len + 64 * j + r];
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[i] *= wv;
                    store8(xt + (jg * 16 + c16) * 128 + jl * 16, v, BF16);  // row (h, p) = 8 c16 + ..
                    if constexpr (!SM::kRawB) {
                        stage_read8<IO>(bsrc, r, c16, v);
                        store8(bb + (c16 * 8 + jg) * 128 + jl * 16, v, BF16);
                    }
                }
                tc::fence_smem_to_async();
                __syncwarp();
                if (lane == 0) {
                    tc::mbar_arrive(bar(PB_EMPTY0 + st));
                    tc::mbar_arrive(bar(PB_OPS0 + ob));
                }
                // the previous item's products are complete by now: read it out
                if (li > 0 && j == (nblk > 1 ? 1 : 0)) read_out(li - 1);
            }
        }
        if (mine > 0) read_out(mine - 1);
    }

    if (timed_out) atomicOr(err, 4u);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == kMmaWarp) tc::tmem_dealloc(tmem, 2 * kNN);
}

// S_in(s + 1) = exp(a_s) S_in(s) + E_s over s = 0 .. nseg - 2, in place.  The
// E_s of up to kFoldBatch segments (and their decays) are loaded at once, so
// the chain costs one memory round trip per batch, not one per segment.
constexpr int kFoldBatch = 8;
__global__ void __launch_bounds__(256, 4)
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
    for (int s0 = 1; s0 < p.nseg; s0 += kFoldBatch) {
        const int cnt = p.nseg - s0 < kFoldBatch ? p.nseg - s0 : kFoldBatch;
        float4 loc[kFoldBatch];
        float ea[kFoldBatch];
#pragma unroll
        for (int i = 0; i < kFoldBatch; ++i)
            if (i < cnt) {
                loc[i] = *reinterpret_cast<const float4 *>(base + (size_t)(s0 + i) * sstride);
                ea[i] = __ldg(a + s0 + i - 1);
            }
#pragma unroll
        for (int i = 0; i < kFoldBatch; ++i)
            if (i < cnt) {
                const float d = expf(ea[i]);
                st.x = fmaf(d, st.x, loc[i].x);
                st.y = fmaf(d, st.y, loc[i].y);
                st.z = fmaf(d, st.z, loc[i].z);
                st.w = fmaf(d, st.w, loc[i].w);
                *reinterpret_cast<float4 *>(base + (size_t)(s0 + i) * sstride) = st;
            }
    }
}

template <int IO, bool BF16>
cudaError_t launch_pre(const Params &p, float *seg_states, float *seg_decay, unsigned int *err, int sms,
                       cudaStream_t s) {
    SegMaps tm;
    cudaError_t e;
    if ((e = encode_tile_map(&tm.x, p.x, IO, (int64_t)p.H * kP, p.L, p.B, true)) != cudaSuccess) return e;
    if ((e = encode_tile_map(&tm.b, p.Bm, IO, (int64_t)p.G * kNN, p.L, p.B, true)) != cudaSuccess) return e;
    const uint32_t smem = PreSmem<IO, BF16>::bytes(p.seg_len);
    auto kern = segment_state_kernel<IO, BF16>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
    const int items = p.B * p.G * (p.hpg / 2) * (p.nseg - 1);
    const int ctas = items < sms ? items : sms;  // persistent: one CTA per SM at most
    kern<<<ctas, kThreads, smem, s>>>(p, tm, seg_states, seg_decay, err);
    return cudaGetLastError();
}

}  // namespace

int segment_max_len() { return kMaxSegLen; }

bool segment_smem_fits(int io, int seg_len) {
    static_assert(PreSmem<IO_F32, true>::bytes(64) == PreSmem<IO_BF16, true>::bytes(64) &&
                      PreSmem<IO_F16, true>::bytes(64) == PreSmem<IO_BF16, true>::bytes(64),
                  "one size for every instantiation");
    const uint32_t need = PreSmem<IO_BF16, true>::bytes(seg_len);
    (void)io;
    return seg_len % 64 == 0 && seg_len <= segment_max_len() && need <= 232448u - 256u;
}

cudaError_t launch_segment_passes(const Params &p, int io, bool bf16, float *seg_states, float *seg_decay,
                                  unsigned int *err, int sms, cudaStream_t s) {
    if (p.nseg < 2) return cudaSuccess;
    cudaError_t e;
    switch (io) {
        case IO_F32: e = bf16 ? launch_pre<IO_F32, true>(p, seg_states, seg_decay, err, sms, s)
                              : launch_pre<IO_F32, false>(p, seg_states, seg_decay, err, sms, s); break;
        case IO_F16: e = bf16 ? launch_pre<IO_F16, true>(p, seg_states, seg_decay, err, sms, s)
                              : launch_pre<IO_F16, false>(p, seg_states, seg_decay, err, sms, s); break;
        default: e = bf16 ? launch_pre<IO_BF16, true>(p, seg_states, seg_decay, err, sms, s)
                          : launch_pre<IO_BF16, false>(p, seg_states, seg_decay, err, sms, s); break;
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
