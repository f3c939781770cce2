// fused_tc.cu -- the fused plan: the whole chunked SSD forward (chunk_cumsum,
// chunk_state, state_passing, chunk_scan; ops-transformer MambaV2 article,
// sections 4.2-4.5) in one persistent sm_103a kernel whose chunk states never
// leave the chip.  This is the "remove state / y_diag materialisation" item
// of the "Mamba-2 SSD for Ascend NPU" README ("Limitations and roadmap"),
// re-designed for tcgen05 tensor cores with TMEM accumulators.
//
// Work unit: (batch b, group g, head pair).  One CTA per SM walks units, and
// each unit's chunks in order, carrying the fp32 [P,N] states of its two heads
// in registers.  Packed variable-length input (the VARLEN instantiation) makes
// the unit (sequence s, group, head pair) over tokens [cu[s], cu[s+1]) of the
// single batch row: its chunks start at cu[s], tokens past its end enter with
// d = 0, and the y rows of its last chunk are written straight to global
// memory (a 64-row TMA store would overwrite the next sequence).  Per chunk of
// Q = 64 tokens (P = N = 64):
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
// row-major global layout (MN- or K-major as the tensors come), so nothing is
// transposed.
//
// Warp roles (640 threads, 20 warps): warps 0-15 compute (thread = TMEM lane
// (head, p) x 16 columns), warp 16 issues the MMAs and warp 17 the TMA copies
// (one thread each), warps 18-19 compute the per-chunk decay vectors of one
// head each, up to two chunks ahead.  Every handoff is an mbarrier, so no role
// waits for another's instruction issue, only for its results:
//
//   compute, chunk k:  wait VEC_FULL; A_k  wait STAGE; operands -> smem (arrive OPS_FULL)
//                      D_k-1 wait Y_FREE, Y_DONE; epilogue of chunk k-1 -> y staging
//                            (arrive Y_STAGED, VEC_EMPTY)           (overlaps G_k)
//                      B_k  wait G_DONE;  G -> Mcat             (arrive MCAT_FULL)
//                      C_k  wait DS_DONE; S <- a S + dS -> smem (arrive S_FULL)
//   MMA, chunk k:      wait OPS_FULL -> G (commit G_DONE);
//                      wait S_FULL -> dS, Yoff (commit DS_DONE);
//                      wait MCAT_FULL -> Yint (commit Y_DONE[k%2])
//   TMA, chunk k:      wait OPS_FULL -> load x, B, C of chunk k+1 (STAGE);
//                      wait Y_STAGED -> store y of chunk k-1, wait for its reads (arrive Y_FREE)
//   decay, chunk k:    wait VEC_EMPTY -> d, cumulative d A, exponentials (arrive VEC_FULL)
//
// Xcat and the Yoff / Yint TMEM accumulators are double-buffered, the
// per-chunk decay vectors triple-buffered; Mcat needs one buffer because the
// epilogue before it already waits for the previous intra-chunk MMA.  Every
// mbarrier wait gives up after 2 s (recorded in the workspace error word)
// instead of hanging.
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "ssd_fused.cuh"
#include "ssd_internal.cuh"
#include "tc_operands.cuh"
#include "tc_ptx.cuh"
#include "tc_stage.cuh"

namespace ssd {

namespace {

constexpr int kQ = 64, kP = 64;
constexpr int kComputeWarps = 16;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kMmaWarp = kComputeWarps;           // warp 16
constexpr int kTmaWarp = kComputeWarps + 1;       // warp 17
constexpr int kDecayWarp0 = kComputeWarps + 2;    // warps 18, 19
constexpr int kThreads = kComputeThreads + 4 * 32;  // 640
// the conv1d instantiation adds 4 warps that convolve the staged x, B, C tiles
constexpr int kConvWarp0 = kComputeWarps + 4;     // warps 20-23
constexpr int kConvWarps = 4;
constexpr int kThreadsConv = kThreads + kConvWarps * 32;  // 768
constexpr int kVecSlots = 3;
constexpr uint64_t kWaitNs = 2000000000ull;       // an mbarrier wait gives up after 2 s
constexpr uint32_t XC_BYTES = 24576;              // [X_h0 | 0 | X_h1], MN-major, 192 rows x 64 j
constexpr uint32_t VEC_BYTES = 2064;
// The gated instantiations (ZM 1: y * silu(z); ZM 2: then the gated RMSNorm)
// load each chunk's z tile by TMA into the y staging tile, where the epilogue
// reads z at the address it then writes y to; an mbarrier after the decay
// vectors marks its arrival.  ZM 2 adds the exchange of per-token sums of
// squares between the CTAs of a cluster that hold the head pairs of one norm
// group (a B/C group).
// Clusters of up to 2: at 8 heads per group (4 CTAs) the forward plus the
// standalone norm kernel measured faster (2.19 vs 2.39 ms at the large shape).
constexpr int kNormMaxRanks = 2;
constexpr uint32_t NORM_LPART = 0;     // [4 warpgroups][4 warps][16 tokens] fp32: per-warp sums
constexpr uint32_t NORM_RECV = 1024;   // [2 slots][kNormMaxRanks][64 tokens] fp32: per-CTA sums
constexpr uint32_t NORM_BARS = NORM_RECV + 2 * kNormMaxRanks * 64 * 4;  // [2 slots][4 warpgroups] mbarriers
constexpr uint32_t NORM_ZBAR = NORM_BARS + 2 * 4 * 8;                    // z tile arrived

// Shared-memory layout, bytes from a 1024-aligned base, for state width NN
// (64 or 128) and public dtype IO:
//   CB2    C twice (rows 0-63, 64-127), K-major, 128 x NN
//   BB     B blocks (j, n), 64 x NN: K-major for G, MN-major for dS
//   XT     Xw^T, MN-major, 128 (h,p) x 64 j, 16 KB
//   XC     kXcBufs x [X_h0 | 0 | X_h1], MN-major, 192 rows x 64 j
//   MC     Mcat, K-major B operand, 64 i x 128 (h', j), 16 KB
//   S      bf16 copy of the state, K-major, 128 (h,p) x NN (NN = 64 only)
//   TMA staging, boxes of 64 token rows x 128 bytes (8 KB each): one chunk's y
//   tile on its way out (not swizzled, the epilogue writes whole rows), and the
//   next chunk's x, B, C tiles on their way in (128-byte swizzled for
//   conflict-free column reads)
//   VEC    3 x ChunkVec, then the norm exchange (gated instantiations)
// At NN = 128 the state lives in TMEM (an fp32 accumulator and the bf16 copy
// that is the A operand of S C^T), and with fp32 I/O y is staged in the C
// staging tile and Xcat has one buffer: the layout then fits in 227 KB.
// NN = 64 keeps the layout the large training shape was tuned on.
// The conv1d instantiation (CV, N = 64) adds POST: the convolved x, B, C of a
// chunk in the operand dtype, laid out like 16-bit TMA staging tiles (x 2
// boxes, B and C one each), which the compute warps read while the next
// chunk's raw tiles land in the staging area; to make room its bf16 state copy
// lives in TMEM and Xcat has one buffer.
// DIRECT (N = 128 with 16-bit tensors already in the operand dtype): the
// products read x, B and C from two staging buffers just as the TMA wrote
// them (128-byte swizzle), so there are no operand copies of them (CB2, BB,
// XC) and the staging is double-buffered; buffer i at STGD + i * DStg::BUF:
//   DX  x of the pair as [head 0 box | zero box | head 1 box] (24 KB): the
//       intra product's block-diagonal A operand, each head's M half beside zeros
//   DB  B, two 64-feature boxes (16 KB)
//   DC  C twice, [c0 | c0 | c1 | c1] (32 KB): 128 rows for C B^T
struct DStg {
    static constexpr uint32_t DX = 0, DB = 3 * 8192, DC = DB + 2 * 8192, BUF = DC + 4 * 8192;
};
template <int NN, int IO, bool CV = false, bool DIRECT = false>
struct Smem {
    static constexpr bool kStateBfTmem = NN == 128 || CV;  // the bf16 copy of the state in TMEM
    static constexpr bool kAliasY = NN == 128 && IO == IO_F32;
    static constexpr int kXcBufs = DIRECT ? 0 : (kAliasY || CV) ? 1 : 2;
    static constexpr uint32_t CB2 = 0;
    static constexpr uint32_t BB = CB2 + (DIRECT ? 0 : 256 * NN);
    static constexpr uint32_t XT = BB + (DIRECT ? 0 : 128 * NN);
    static constexpr uint32_t XC = XT + 16384;
    static constexpr uint32_t MC = XC + kXcBufs * XC_BYTES;
    static constexpr uint32_t POST = MC + 16384;                 // x at POST, B at POST_B, C at POST_C
    static constexpr uint32_t POST_B = POST + 2 * 8192, POST_C = POST_B + 8192;
    static constexpr uint32_t S = POST + (CV ? 4 * 8192 : 0);
    static constexpr uint32_t STG_Y = S + (kStateBfTmem ? 0 : 256 * NN);
    static constexpr uint32_t Y_BYTES = NN == 64 ? 32768 : kAliasY ? 0 : (IO == IO_F32 ? 32768 : 16384);
    static constexpr uint32_t STG_X = STG_Y + Y_BYTES;
    static constexpr uint32_t X_BYTES = DIRECT ? 0 : NN == 64 ? 32768 : (IO == IO_F32 ? 32768 : 16384);
    static constexpr uint32_t STG_B = STG_X + X_BYTES;
    static constexpr uint32_t BC_BYTES = DIRECT ? 0 : NN == 64 ? 16384 : 64 * NN * (IO == IO_F32 ? 4 : 2);
    static constexpr uint32_t STG_C = STG_B + BC_BYTES;
    static constexpr uint32_t YSTAGE = kAliasY ? STG_C : STG_Y;  // where the epilogue stages y (and z)
    static constexpr uint32_t STGD = STG_C + BC_BYTES;
    static constexpr uint32_t VEC = STGD + (DIRECT ? 2 * DStg::BUF : 0);
    static constexpr uint32_t NORM = VEC + 3 * VEC_BYTES;
    static constexpr uint32_t BYTES = NORM + 1024;                    // + alignment slack
    static constexpr uint32_t BYTES_NORM = NORM + NORM_ZBAR + 16 + 1024;
    static_assert(STG_X % 1024 == 0 && STG_B % 1024 == 0 && STG_C % 1024 == 0 && POST % 1024 == 0 &&
                      STGD % 1024 == 0 && DStg::BUF % 1024 == 0,
                  "swizzled TMA boxes need 1 KB");
    static_assert(NORM % 16 == 0 && BYTES_NORM + 512 <= 232448, "the layout fits in shared memory");
};
static_assert(Smem<64, IO_F32>::VEC == 221184 && Smem<64, IO_BF16>::STG_C == 204800, "N = 64 layout unchanged");
// the launch sizes shared memory from the regular layout
static_assert(Smem<128, IO_BF16, false, true>::BYTES == Smem<128, IO_BF16>::BYTES &&
                  Smem<128, IO_BF16, false, true>::BYTES_NORM == Smem<128, IO_BF16>::BYTES_NORM &&
                  Smem<128, IO_F16, false, true>::BYTES == Smem<128, IO_F16>::BYTES &&
                  Smem<128, IO_F16, false, true>::BYTES_NORM == Smem<128, IO_F16>::BYTES_NORM,
              "the direct layout takes the same room");

// TMEM columns (512 allocated).  NN = 64: G 0-63, dS 64-127, Yoff / Yint in
// two buffers from 128.  NN = 128: G 0-63, the fp32 state 64-191 (dS is
// accumulated onto the decayed state there), Yoff 192 / 256, Yint 320 / 384,
// the bf16 state (A operand of S C^T, two values per column) 448-511.
constexpr uint32_t TM_G = 0, TM_DS = 64, TM_COLS = 512;
constexpr uint32_t TM_S32 = 64, TM_SBF = 448;  // (the conv1d instantiation at N = 64 keeps its bf16 state at 448 too)
template <int NN>
__device__ __forceinline__ uint32_t tm_yoff(int buf) { return NN == 64 ? 128u + 128u * buf : 192u + 64u * buf; }
template <int NN>
__device__ __forceinline__ uint32_t tm_yint(int buf) { return NN == 64 ? 192u + 128u * buf : 320u + 64u * buf; }

// mbarriers
enum {
    BAR_OPS_FULL = 0, BAR_MCAT_FULL, BAR_S_FULL, BAR_G_DONE, BAR_DS_DONE, BAR_Y_DONE0, BAR_Y_DONE1,
    BAR_STAGE_FULL, BAR_Y_STAGED, BAR_Y_FREE, BAR_VEC_FULL0, BAR_VEC_EMPTY0 = BAR_VEC_FULL0 + kVecSlots,
    BAR_CONV_DONE = BAR_VEC_EMPTY0 + kVecSlots, BAR_STG_FREE,
    BAR_DFULL0, BAR_DFREE0 = BAR_DFULL0 + 2,  // the direct layout's two staging buffers: loaded, read
    NBARS = BAR_DFREE0 + 2
};

// TMA descriptors of x [B,L,H*P] and B, C [B,L,G*N] as 3-D tensors
// (innermost first: features, tokens, batch), boxes of 128 bytes x 64 tokens.
struct TmaMaps {
    CUtensorMap x, b, c, y, z;  // z: gated instantiations only
};

// 16-byte aligned so that consecutive slots keep their float4 reads aligned
struct alignas(16) ChunkVec {
    float d[2][kQ];    // processed step
    float cs2[2][kQ];  // within-chunk cumulative d*A, times log2(e)
    float ecs[2][kQ];  // exp(cs)
    float w[2][kQ];    // exp(cs_last - cs) * d
    float a[2];        // exp(cs_last)
};
static_assert(sizeof(ChunkVec) % 16 == 0 && sizeof(ChunkVec) <= VEC_BYTES, "ChunkVec slots");

using tcop::ex2_approx;
using tcop::pack2;
using tcop::st_shared_v4;
using tcop::store8;
using tcstage::BOX_BYTES;
using tcstage::stage_raw16;
using tcstage::stage_read8;

// Shapes of one call, held in registers by every thread.
struct Dims {
    int L, H, G, hpg, nchunks;
};

// Tokens of one work unit: tensor batch b, state index sb (b, or the sequence
// for packed variable-length input), group g, first head h0, token offset t0
// and length len within the batch row, its number of chunks, and its segment
// (segmented walks, else 0).
struct Span {
    int b, sb, g, h0, t0, len, nch, seg;
};

// `unit` is the walk position: every CTA walks positions blockIdx.x,
// blockIdx.x + gridDim.x, ...; for packed sequences the host's schedule maps a
// position to the unit it runs there.  Segmented walks (SEG) order the units
// (batch, segment, group, head pair) with the head pair fastest, so that the
// CTAs running side by side share their B and C tiles in L2.
template <bool VARLEN, bool SEG = false>
__device__ __forceinline__ Span unit_span(const Params &p, const Dims &dm, int unit) {
    if (VARLEN) unit = p.sched_units[unit];
    const int pairs = dm.hpg >> 1;
    const int pair = unit % pairs, bg = unit / pairs;
    Span u;
    u.g = bg % dm.G;
    u.h0 = u.g * dm.hpg + 2 * pair;
    const int q = bg / dm.G;
    u.sb = q;
    u.seg = 0;
    if (VARLEN) {
        u.b = 0;
        u.t0 = (int)p.cu[q];
        u.len = (int)(p.cu[q + 1] - p.cu[q]);
        u.nch = (u.len + kQ - 1) / kQ;
    } else if (SEG) {
        u.seg = q % p.nseg;
        u.b = u.sb = q / p.nseg;
        u.t0 = u.seg * p.seg_len;
        u.len = min(p.seg_len, dm.L - u.t0);
        u.nch = (u.len + kQ - 1) / kQ;
    } else {
        u.b = q;
        u.t0 = 0;
        u.len = dm.L;
        u.nch = dm.nchunks;
    }
    return u;
}

// Decay warps' registers: raw dt of tokens lane and lane + 32 of a chunk.
struct DtRegs {
    float dt0, dt1;
};

__device__ __forceinline__ void load_dt(const Params &p, const Dims &dm, const Span &u, int h, int k, int lane,
                                        DtRegs &r) {
    const int t0 = k * kQ + lane, t1 = t0 + 32;  // tokens within the unit's sequence
    const float *row = p.dt + ((size_t)u.b * dm.L + u.t0) * dm.H + h;
    r.dt0 = t0 < u.len ? __ldg(row + (size_t)t0 * dm.H) : 0.f;
    r.dt1 = t1 < u.len ? __ldg(row + (size_t)t1 * dm.H) : 0.f;
}

// Decay vectors of one chunk for head hh (one warp): processed step, the
// within-chunk inclusive cumulative sum of d*A (warp scan over 64 tokens)
// and the exponentials the other phases need.  Tokens at or past `valid`
// (the end of the sequence) take d = 0.
__device__ __forceinline__ void decay_vectors(const Params &p, int h, int hh, int valid, int lane, float raw0,
                                              float raw1, ChunkVec &V) {
    const float d0 = (lane < valid) ? dt_processed(p, raw0, h) : 0.f;
    const float d1 = (lane + 32 < valid) ? dt_processed(p, raw1, h) : 0.f;
    const float A = __ldg(p.A + h);
    float v0 = d0 * A, v1 = d1 * A;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float o0 = __shfl_up_sync(0xffffffffu, v0, off);
        const float o1 = __shfl_up_sync(0xffffffffu, v1, off);
        if (lane >= off) { v0 += o0; v1 += o1; }
    }
    v1 += __shfl_sync(0xffffffffu, v0, 31);
    const float last = __shfl_sync(0xffffffffu, v1, 31);
    constexpr float kLog2e = 1.4426950408889634f;
    V.d[hh][lane] = d0;
    V.d[hh][lane + 32] = d1;
    V.cs2[hh][lane] = v0 * kLog2e;
    V.cs2[hh][lane + 32] = v1 * kLog2e;
    V.ecs[hh][lane] = expf(v0);
    V.ecs[hh][lane + 32] = expf(v1);
    V.w[hh][lane] = expf(last - v0) * d0;
    V.w[hh][lane + 32] = expf(last - v1) * d1;
    if (lane == 0) V.a[hh] = expf(last);
}

// One value of an unswizzled staging tile (fp32, or fp16 / bf16 bits).
template <int IO>
__device__ __forceinline__ float ld_stage(uint32_t a) {
    if (IO == IO_F32) {
        float v;
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
        return v;
    } else {
        uint16_t hb;
        asm volatile("ld.shared.b16 %0, [%1];" : "=h"(hb) : "r"(a));
        if (IO == IO_BF16) return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(&hb));
        return __half2float(*reinterpret_cast<const __half *>(&hb));
    }
}

// The z gate silu(z) of the staged-z epilogues: with a 16-bit y the one-MUFU
// form (its error is below y's rounding), with fp32 y the two-MUFU form.
template <int IO>
__device__ __forceinline__ float gate(float z) {
    return IO == IO_F32 ? silu_fast(z) : silu_tanh(z);
}

// y for one (head, p) and 8 consecutive tokens from tok_base, read from the
// TMEM accumulators of buffer bp and written into the y staging tile (rows of
// 128 bytes per box; the TMA store drops rows past L).  For packed sequences
// (VARLEN) tokens count from t0 in batch row 0, the sequence ends at len, and
// in its last chunk (`direct`) y goes straight to global memory for the
// tokens inside the sequence, since the rows past its end belong to the next.
// T = 16 reads both accumulators' 16 columns with one wait; T = 8 with two
// loads and two waits, fewer registers live (same-process A/B: T = 16 is 2.3 %
// faster at N = 128, 0.6 % slower at N = 64 with its register-resident state).
template <int IO, bool VARLEN, int ZM = 0, int NN = 64, bool SEG = false, int T = 8, bool FENCE = true>
__device__ __forceinline__ void epilogue_tokens(const Params &p, const Dims &dm, const ChunkVec &V, uint32_t tlane,
                                                int bp, int col, int b, int h0, int my_h, int my_p, int tok_base,
                                                uint32_t ystage, int t0, int len, bool direct) {
    static_assert(T == 8 || T == 16, "8 or 16 tokens col .. col + T - 1 of the chunk");
    if (!VARLEN && !SEG) {
        t0 = 0;
        len = dm.L;
    }
    float yo[T], yi[T];
    if constexpr (T == 16) {
        tc::tmem_ld16x2(tlane + tm_yoff<NN>(bp) + col, tlane + tm_yint<NN>(bp) + col, yo, yi);  // one wait
    } else {
        tc::tmem_ld8(tlane + tm_yoff<NN>(bp) + col, yo);
        tc::tmem_ld8(tlane + tm_yint<NN>(bp) + col, yi);
    }
    tc::fence_before_sync();
    const int i0 = tok_base % kQ;
    float ev[T];
#pragma unroll
    for (int q = 0; q < T / 4; ++q) {
        const float4 e = *reinterpret_cast<const float4 *>(&V.ecs[my_h][i0 + 4 * q]);
        ev[4 * q] = e.x; ev[4 * q + 1] = e.y; ev[4 * q + 2] = e.z; ev[4 * q + 3] = e.w;
    }
    const int h = h0 + my_h;
    const size_t step = (size_t)dm.H * kP;
    const size_t off0 = (((size_t)b * dm.L + t0 + tok_base) * dm.H + h) * kP + my_p;
    float v[T];
#pragma unroll
    for (int ii = 0; ii < T; ++ii) v[ii] = fmaf(ev[ii], yo[ii], yi[ii]);
    // (D x is in the intra-chunk product)
    if constexpr (ZM > 0) {  // z staged where y goes
        const int f = my_h * kP + my_p;
        const uint32_t a0 = IO == IO_F32 ? ystage + (f >> 5) * BOX_BYTES + i0 * 128 + (f & 31) * 4
                                         : ystage + (f >> 6) * BOX_BYTES + i0 * 128 + (f & 63) * 2;
#pragma unroll
        for (int ii = 0; ii < T; ++ii) v[ii] *= gate<IO>(ld_stage<IO>(a0 + ii * 128));
    } else if (p.z) {
        float zv[T];
#pragma unroll
        for (int ii = 0; ii < T; ++ii)
            zv[ii] = (tok_base + ii < len) ? ld_io<IO>(p.z, off0 + ii * step) : 0.f;
#pragma unroll
        for (int ii = 0; ii < T; ++ii) v[ii] *= gate<IO>(zv[ii]);
    }
    if (VARLEN && direct) {
#pragma unroll
        for (int ii = 0; ii < T; ++ii)
            if (tok_base + ii < len) st_io<IO>(p.y, off0 + ii * step, v[ii]);
        return;
    }
    const int f = my_h * kP + my_p;  // feature within the pair's 128
    const uint32_t a0 = IO == IO_F32 ? ystage + (f >> 5) * BOX_BYTES + i0 * 128 + (f & 31) * 4
                                     : ystage + (f >> 6) * BOX_BYTES + i0 * 128 + (f & 63) * 2;
#pragma unroll
    for (int ii = 0; ii < T; ++ii) {
        const uint32_t a = a0 + ii * 128;
        if (IO == IO_F32) {
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v[ii]));
        } else {
            uint16_t hbits;
            if (IO == IO_BF16) {
                __nv_bfloat16 hv = __float2bfloat16_rn(v[ii]);
                hbits = *reinterpret_cast<uint16_t *>(&hv);
            } else {
                __half hv = __float2half_rn(v[ii]);
                hbits = *reinterpret_cast<uint16_t *>(&hv);
            }
            asm volatile("st.shared.b16 [%0], %1;" ::"r"(a), "h"(hbits));
        }
    }
    // the staged y goes out by TMA: one proxy fence after the last of a thread's stores (a
    // fence per 8-token half measured 1.014 ms against 1.000 at the large training shape)
    if constexpr (FENCE) tc::fence_smem_to_async();
}

// Shared-memory addresses of the norm exchange and this CTA's place in it.
struct NormCtx {
    uint32_t lpart, recv, rbar;
    int cs, rank;  // CTAs per norm group (the cluster), this CTA's rank (= its head pair)
};

// NORM epilogue: y of this thread's feature for the 16 tokens col0 .. col0+15
// of the chunk (as epilogue_tokens with z staged; D x is already in the intra-chunk
// product), then the gated RMSNorm of the
// ops-transformer MambaV2 article, section 4.6: every token is divided by the
// root mean square of its cs * 128 gated features (the group's heads) and
// multiplied by the feature's weight.  The sum of squares runs over the warp's
// 32 features (shuffles), the warpgroup's 4 warps (shared memory), then the
// cs CTAs of the cluster (remote stores + an mbarrier per warpgroup and slot;
// two slots alternate by chunk).  Every CTA adds the cs partial sums in rank
// order, so all features of a group use bitwise the same scale.
template <int IO>
__device__ __forceinline__ void epilogue_norm(const Params &p, const Dims &dm, const ChunkVec &V, uint32_t tlane,
                                              int bp, int col0, int b, int h0, int my_h, int my_p, int tok_base,
                                              uint32_t ystage, const NormCtx &nc, uint32_t gp, int wg, int quarter,
                                              int lane, float wf, bool &timed_out) {
    const int f = my_h * kP + my_p;  // feature within the pair's 128
    auto stage_addr = [&](int ib) {  // token row ib of the staging tile, this feature
        return IO == IO_F32 ? ystage + (f >> 5) * BOX_BYTES + ib * 128 + (f & 31) * 4
                            : ystage + (f >> 6) * BOX_BYTES + ib * 128 + (f & 63) * 2;
    };
    float v[16];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        float yo[8], yi[8];
        tc::tmem_ld8(tlane + tm_yoff<64>(bp) + col0 + 8 * hf, yo);
        tc::tmem_ld8(tlane + tm_yint<64>(bp) + col0 + 8 * hf, yi);
        const float4 e0 = *reinterpret_cast<const float4 *>(&V.ecs[my_h][col0 + 8 * hf]);
        const float4 e1 = *reinterpret_cast<const float4 *>(&V.ecs[my_h][col0 + 8 * hf + 4]);
        const float ev[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
#pragma unroll
        for (int ii = 0; ii < 8; ++ii) v[8 * hf + ii] = fmaf(ev[ii], yo[ii], yi[ii]);
    }
    tc::fence_before_sync();  // (D x is in the intra-chunk product)
#pragma unroll
    for (int ii = 0; ii < 16; ++ii) v[ii] *= gate<IO>(ld_stage<IO>(stage_addr(col0 + ii)));  // z staged where y goes
    // per-token sum of squares over the warp's 32 features: halve the token set
    // at each shuffle step; lane l ends with token tk(l) (bits 4..1 of l), l and
    // l ^ 1 holding the same sum
    float e;
    {
        float a8[8], a4[4], a2[2];
        const bool u4 = lane & 16, u3 = lane & 8, u2 = lane & 4, u1 = lane & 2;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float lo = v[j] * v[j], hi = v[8 + j] * v[8 + j];
            a8[j] = (u4 ? hi : lo) + __shfl_xor_sync(0xffffffffu, u4 ? lo : hi, 16);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) a4[j] = (u3 ? a8[4 + j] : a8[j]) + __shfl_xor_sync(0xffffffffu, u3 ? a8[j] : a8[4 + j], 8);
#pragma unroll
        for (int j = 0; j < 2; ++j) a2[j] = (u2 ? a4[2 + j] : a4[j]) + __shfl_xor_sync(0xffffffffu, u2 ? a4[j] : a4[2 + j], 4);
        e = (u1 ? a2[1] : a2[0]) + __shfl_xor_sync(0xffffffffu, u1 ? a2[0] : a2[1], 2);
        e += __shfl_xor_sync(0xffffffffu, e, 1);
    }
    const int tk = ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
    if (!(lane & 1)) asm volatile("st.shared.f32 [%0], %1;" ::"r"(nc.lpart + ((wg * 4 + quarter) * 16 + tk) * 4), "f"(e));
    tc::named_barrier(1 + wg, 128);
    const uint32_t slot = gp & 1u;
    const uint32_t rbar = nc.rbar + (slot * 4 + wg) * 8;
    if (quarter == 0 && lane < 16) {  // this CTA's sum for token `lane` of the warpgroup
        float sum = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float t;
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(t) : "r"(nc.lpart + ((wg * 4 + q) * 16 + lane) * 4));
            sum += t;
        }
        const uint32_t mine = nc.recv + ((slot * kNormMaxRanks + nc.rank) * 64 + wg * 16 + lane) * 4;
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(mine), "f"(sum));
        for (int r = 0; r < nc.cs; ++r) {
            if (r == nc.rank) continue;
            tc::st_cluster_f32(tc::mapa_shared(mine, r), sum);
            tc::mbar_arrive_cluster(tc::mapa_shared(rbar, r));
        }
    }
    tc::named_barrier(1 + wg, 128);
    if (nc.cs > 1 && !timed_out && !tc::mbar_wait_cluster(rbar, (gp >> 1) & 1u, kWaitNs)) timed_out = true;
    float tot[16];
#pragma unroll
    for (int ii = 0; ii < 16; ++ii) tot[ii] = 0.f;
    for (int r = 0; r < nc.cs; ++r) {
        const uint32_t base = nc.recv + ((slot * kNormMaxRanks + r) * 64 + wg * 16) * 4;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 t4 = tc::ld_shared_v4(base + 16 * q);
            tot[4 * q] += __uint_as_float(t4.x);
            tot[4 * q + 1] += __uint_as_float(t4.y);
            tot[4 * q + 2] += __uint_as_float(t4.z);
            tot[4 * q + 3] += __uint_as_float(t4.w);
        }
    }
    const float inv_n = 1.f / (float)(nc.cs * 2 * kP);
#pragma unroll
    for (int ii = 0; ii < 16; ++ii) v[ii] *= rsqrtf(fmaf(tot[ii], inv_n, p.norm_eps)) * wf;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        const uint32_t a0 = stage_addr(col0 + 8 * hf);
#pragma unroll
        for (int ii = 0; ii < 8; ++ii) {
            const uint32_t a = a0 + ii * 128;
            const float val = v[8 * hf + ii];
            if (IO == IO_F32) {
                asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(val));
            } else {
                uint16_t hbits;
                if (IO == IO_BF16) {
                    __nv_bfloat16 hv = __float2bfloat16_rn(val);
                    hbits = *reinterpret_cast<uint16_t *>(&hv);
                } else {
                    __half hv = __float2half_rn(val);
                    hbits = *reinterpret_cast<uint16_t *>(&hv);
                }
                asm volatile("st.shared.b16 [%0], %1;" ::"r"(a), "h"(hbits));
            }
        }
    }
    tc::fence_smem_to_async();
}

// NN = 128 (N = 128) walks segments of the sequence (SEG: unit = (batch,
// segment, group, head pair), the state entering a segment from the segment
// passes, the final state from the last segment) with the state in TMEM; it
// takes neither packed sequences nor the fused norm.
// CV (N = 64, regular layout): x, B and C arrive before their causal conv1d +
// SiLU (ops-transformer MambaV2 article, sections 1.4 and 4.1), and 4 more
// warps convolve each staged tile in place before the compute warps read it.
// A conv thread owns two channels for the whole walk of a unit, so the W-1
// tokens before a chunk (the conv's halo) stay in its registers from the
// previous chunk, and the taps too; a unit starts from zeros (no tokens before
// t = 0).  The results are rounded to the staging tile's dtype.
template <int IO, bool BF16, bool VARLEN, int ZM, int NN = 64, bool CV = false>
__global__ void __launch_bounds__(CV ? kThreadsConv : kThreads, 1)
ssd_fused_kernel(const __grid_constant__ Params p, const __grid_constant__ TmaMaps tm, int n_units,
                 unsigned int *err, int norm_cs) {
    // dtype of the tiles the operand stage reads: the staging tiles, or with the
    // conv1d the convolved tiles in POST (in the operand dtype)
    constexpr int SIO = CV ? (BF16 ? IO_BF16 : IO_F16) : IO;
    // those tiles hold the operand dtype already: x (unweighted), B and C are
    // copied chunk by chunk (or at N = 128 read in place), only the decay-weighted x
    // is converted
    constexpr bool kRaw = SIO != IO_F32 && ((SIO == IO_BF16) == BF16);
    constexpr bool DIRECT = NN == 128 && kRaw && !CV;
    using L = Smem<NN, IO, CV, DIRECT>;
    constexpr bool SEG = NN == 128;
    constexpr bool kAliasY = L::kAliasY;
    static_assert(NN == 64 || NN == 128, "state width 64 or 128");
    static_assert(NN == 64 || (!VARLEN && ZM < 2), "N = 128: no packed sequences, no fused norm");
    static_assert(!CV || (NN == 64 && !VARLEN && ZM < 2), "the in-kernel conv1d: N = 64, regular layout, no norm");
    static_assert(!kAliasY || ZM == 0, "with y staged in the C tile there is no room for a z tile");
    constexpr int kGCols = 16;      // this thread's columns of each 64-column region (G, Yoff, Yint)
    constexpr int kSCols = NN / 4;  // this thread's state columns
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bars[NBARS];
    __shared__ uint32_t tmem_slot;
    const uint32_t raw = tc::smem_addr(smem_raw);
    unsigned char *sm = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sbase = tc::smem_addr(sm);
    ChunkVec *Vbuf = reinterpret_cast<ChunkVec *>(sm + L::VEC);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Dims dm{p.L, p.H, p.G, p.hpg, p.nchunks};
    const uint32_t bar0 = tc::smem_addr(&bars[0]);
    auto bar = [bar0](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };

    if (tid == 0) {
        tc::mbar_init(bar(BAR_OPS_FULL), kComputeWarps);
        tc::mbar_init(bar(BAR_MCAT_FULL), kComputeWarps);
        tc::mbar_init(bar(BAR_S_FULL), kComputeWarps);
        tc::mbar_init(bar(BAR_G_DONE), 1);
        tc::mbar_init(bar(BAR_DS_DONE), 1);
        tc::mbar_init(bar(BAR_Y_DONE0), 1);
        tc::mbar_init(bar(BAR_Y_DONE1), 1);
        tc::mbar_init(bar(BAR_STAGE_FULL), 1);
        tc::mbar_init(bar(BAR_Y_STAGED), kComputeWarps);
        tc::mbar_init(bar(BAR_Y_FREE), 1);
        for (int i = 0; i < kVecSlots; ++i) {
            tc::mbar_init(bar(BAR_VEC_FULL0 + i), 2);
            tc::mbar_init(bar(BAR_VEC_EMPTY0 + i), kComputeWarps);
        }
        tc::mbar_init(bar(BAR_CONV_DONE), kConvWarps);
        tc::mbar_init(bar(BAR_STG_FREE), kConvWarps);
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(bar(BAR_DFULL0 + i), 1);
            tc::mbar_init(bar(BAR_DFREE0 + i), 1);
        }
        if constexpr (ZM > 0) tc::mbar_init(sbase + L::NORM + NORM_ZBAR, 1);
        if constexpr (ZM == 2) {
            if (norm_cs > 1)
                for (int i = 0; i < 8; ++i) tc::mbar_init(sbase + L::NORM + NORM_BARS + 8 * i, (norm_cs - 1) * 16);
        }
        tc::mbar_init_fence();
    }
    if (warp == kMmaWarp) {
        tc::tmem_alloc(tc::smem_addr(&tmem_slot), TM_COLS);
        tc::tmem_relinquish();
    }
    // the zero block between the two heads' x tiles (MN groups 8..15), every buffer
    for (int e = tid; e < L::kXcBufs * 8 * 8 * 8; e += blockDim.x) {
        const int buf = e >> 9, jg = (e >> 6) & 7, mg = 8 + ((e >> 3) & 7), rr = e & 7;
        st_shared_v4(sbase + L::XC + buf * XC_BYTES + (jg * 24 + mg) * 128 + rr * 16, 0u, 0u, 0u, 0u);
    }
    // Mcat starts zero: the blocks above the diagonal that no warp writes stay so
    for (int e = tid; e < 16384 / 16; e += blockDim.x) st_shared_v4(sbase + L::MC + 16 * e, 0u, 0u, 0u, 0u);
    if constexpr (DIRECT) {  // the zero box between the heads' x boxes, both buffers (no copy writes it)
        for (int e = tid; e < 2 * 8192 / 16; e += blockDim.x)
            st_shared_v4(sbase + L::STGD + (e >> 9) * DStg::BUF + DStg::DX + 8192 + 16 * (e & 511), 0u, 0u, 0u, 0u);
    }
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if constexpr (ZM == 2) {  // the partners' exchange barriers are initialised before any remote arrive
        if (norm_cs > 1) tc::cluster_sync();
    }
    const uint32_t tmem = tmem_slot;
    const int pairs = dm.hpg >> 1;
    bool timed_out = false;
    // wait on mbarrier i for the phase of the given parity; after one timeout a
    // thread stops waiting (the error word is set and the output is void)
    auto wait = [&](int i, uint32_t parity) {
        if (!timed_out && !tc::mbar_wait(bar(i), parity, kWaitNs)) timed_out = true;
    };

    if (warp == kMmaWarp) {
        // ---------------- MMA issue (one thread) ----------------
        if (lane == 0) {
            constexpr uint32_t ID_KK = tc::idesc_f16(128, 64, BF16, false, false);
            constexpr uint32_t ID_MNMN = tc::idesc_f16(128, NN, BF16, true, true);
            constexpr uint32_t ID_MNK = tc::idesc_f16(128, 64, BF16, true, false);
            uint32_t gk = 0;
            for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
                const int nch = unit_span<VARLEN, SEG>(p, dm, unit).nch;
                for (int k = 0; k < nch; ++k, ++gk) {
                    const uint32_t ph = gk & 1u;
                    const int buf = gk & 1;
                    const int xbuf = L::kXcBufs == 2 ? buf : 0;
                    if constexpr (DIRECT) {
                        // x, B and C straight from staging buffer gk % 2 (128-byte swizzle): K-major
                        // operands step 32 bytes per K = 16 inside a box row, and move to the
                        // features 64-127 box after four steps; MN-major ones step 16 token rows
                        // C B^T needs only the staged tiles, so it goes out as soon as they land (the
                        // previous chunk's Mcat has released TM_G: this thread waited for it before the
                        // previous intra product), then Yoff, and dS once the weighted x is in
                        // (gated prefill 425.5 -> 414.0 us; the same order with copied operands
                        // measured slower at N = 128 with fp32 tensors and neutral at N = 64)
                        const uint32_t sb = sbase + L::STGD + (gk & 1u) * DStg::BUF;
                        wait(BAR_DFULL0 + (gk & 1u), (gk >> 1) & 1u);
                        tc::fence_after_sync();
#pragma unroll
                        for (int ks = 0; ks < NN / 16; ++ks)  // G = C B^T, K = n: C's two copies give 128 rows
                            tc::mma_f16(tmem + TM_G,
                                        tc::desc_sw128(sb + DStg::DC + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                                        tc::desc_sw128(sb + DStg::DB + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024),
                                        ID_KK, ks > 0);
                        tc::commit(bar(BAR_G_DONE));
                        wait(BAR_S_FULL, ph);
                        tc::fence_after_sync();
#pragma unroll
                        for (int ks = 0; ks < NN / 16; ++ks)  // Yoff = S C^T, S from TMEM, K = n
                            tc::mma_f16_ts(tmem + tm_yoff<NN>(buf), tmem + TM_SBF + ks * 8,
                                           tc::desc_sw128(sb + DStg::DC + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                                           ID_KK, ks > 0);
                        wait(BAR_OPS_FULL, ph);  // the weighted x
                        tc::fence_after_sync();
#pragma unroll
                        for (int ks = 0; ks < kQ / 16; ++ks)  // S += Xw^T B onto the decayed state, K = j
                            tc::mma_f16(tmem + TM_S32, tc::desc(sbase + L::XT + ks * 4096, 2048, 128),
                                        tc::desc_sw128(sb + DStg::DB + ks * 2048, 8192, 1024), ID_MNMN, 1u);
                        tc::commit(bar(BAR_DS_DONE));
                        wait(BAR_MCAT_FULL, ph);
                        tc::fence_after_sync();
                        const uint32_t mc = sbase + L::MC;
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh)  // head hh's x box beside the zero box: its M half of Xcat
#pragma unroll
                            for (int ks = 0; ks < kQ / 16; ++ks)
                                tc::mma_f16(tmem + tm_yint<NN>(buf),
                                            tc::desc_sw128(sb + DStg::DX + hh * 8192 + ks * 2048, 8192, 1024),
                                            tc::desc(mc + hh * 8192 + ks * 2048, 1024, 128), ID_MNK, (hh | ks) != 0);
                        tc::commit(bar(buf ? BAR_Y_DONE1 : BAR_Y_DONE0));
                        tc::commit(bar(BAR_DFREE0 + (gk & 1u)));  // every product of this buffer issued
                        continue;
                    }
                    wait(BAR_OPS_FULL, ph);
                    tc::fence_after_sync();
#pragma unroll
                    for (int ks = 0; ks < NN / 16; ++ks)  // G = C B^T, K = n
                        tc::mma_f16(tmem + TM_G, tc::desc(sbase + L::CB2 + ks * 4096, 2048, 128),
                                    tc::desc(sbase + L::BB + ks * 2048, 1024, 128), ID_KK, ks > 0);
                    tc::commit(bar(BAR_G_DONE));
                    wait(BAR_S_FULL, ph);
                    tc::fence_after_sync();
                    if constexpr (NN == 64) {
#pragma unroll
                        for (int ks = 0; ks < kQ / 16; ++ks)  // dS = Xw^T B, K = j
                            tc::mma_f16(tmem + TM_DS, tc::desc(sbase + L::XT + ks * 4096, 2048, 128),
                                        tc::desc(sbase + L::BB + ks * 256, 128, 1024), ID_MNMN, ks > 0);
#pragma unroll
                        for (int ks = 0; ks < NN / 16; ++ks) {  // Yoff = S C^T, K = n
                            if constexpr (L::kStateBfTmem)
                                tc::mma_f16_ts(tmem + tm_yoff<NN>(buf), tmem + TM_SBF + ks * 8,
                                               tc::desc(sbase + L::CB2 + ks * 4096, 2048, 128), ID_KK, ks > 0);
                            else
                                tc::mma_f16(tmem + tm_yoff<NN>(buf), tc::desc(sbase + L::S + ks * 4096, 2048, 128),
                                            tc::desc(sbase + L::CB2 + ks * 4096, 2048, 128), ID_KK, ks > 0);
                        }
                    } else {
#pragma unroll
                        for (int ks = 0; ks < kQ / 16; ++ks)  // S += Xw^T B onto the decayed state, K = j
                            tc::mma_f16(tmem + TM_S32, tc::desc(sbase + L::XT + ks * 4096, 2048, 128),
                                        tc::desc(sbase + L::BB + ks * 256, 128, 1024), ID_MNMN, 1u);
#pragma unroll
                        for (int ks = 0; ks < NN / 16; ++ks)  // Yoff = S C^T, S from TMEM, K = n
                            tc::mma_f16_ts(tmem + tm_yoff<NN>(buf), tmem + TM_SBF + ks * 8,
                                           tc::desc(sbase + L::CB2 + ks * 4096, 2048, 128), ID_KK, ks > 0);
                    }
                    tc::commit(bar(BAR_DS_DONE));
                    wait(BAR_MCAT_FULL, ph);
                    tc::fence_after_sync();
                    const uint32_t xc = sbase + L::XC + xbuf * XC_BYTES, mc = sbase + L::MC;
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                        for (int ks = 0; ks < kQ / 16; ++ks)
                            tc::mma_f16(tmem + tm_yint<NN>(buf), tc::desc(xc + hh * 1024 + ks * 6144, 3072, 128),
                                        tc::desc(mc + hh * 8192 + ks * 2048, 1024, 128), ID_MNK,
                                        (hh | ks) != 0);
                    tc::commit(bar(buf ? BAR_Y_DONE1 : BAR_Y_DONE0));
                }
            }
        }
        __syncwarp();
    } else if (warp == kTmaWarp) {
        // ---------------- TMA loads and stores (one thread) ----------------
        if (lane == 0) {
            tc::prefetch_tensormap(&tm.x);
            tc::prefetch_tensormap(&tm.b);
            tc::prefetch_tensormap(&tm.c);
            tc::prefetch_tensormap(&tm.y);
            if constexpr (ZM > 0) tc::prefetch_tensormap(&tm.z);
            constexpr int bw = IO == IO_F32 ? 32 : 64;  // features per 128-byte box
            constexpr uint32_t kStageBytes = (IO == IO_F32 ? 8u : 4u) * BOX_BYTES;
            // The same loop three times: packed sequences and segmented walks take
            // per-unit spans, the regular layout keeps plain index arithmetic
            // (measured 0.8 % faster than the span version at the large training shape).
            if constexpr (VARLEN) {
                // the public x, B, C tiles of chunk k of a unit into the staging area
                // (rows past the sequence's end are read but enter with d = 0)
                auto stage = [&](const Span &u, int k) {
                    const int tok = u.t0 + k * kQ;
                    tc::mbar_arrive_expect_tx(bar(BAR_STAGE_FULL), kStageBytes);
#pragma unroll
                    for (int bx = 0; bx < 128 / bw; ++bx)
                        tc::tma_load_3d(sbase + L::STG_X + bx * BOX_BYTES, &tm.x, u.h0 * kP + bx * bw, tok, u.b,
                                        bar(BAR_STAGE_FULL));
#pragma unroll
                    for (int bx = 0; bx < NN / bw; ++bx) {
                        tc::tma_load_3d(sbase + L::STG_B + bx * BOX_BYTES, &tm.b, u.g * NN + bx * bw, tok, u.b,
                                        bar(BAR_STAGE_FULL));
                        tc::tma_load_3d(sbase + L::STG_C + bx * BOX_BYTES, &tm.c, u.g * NN + bx * bw, tok, u.b,
                                        bar(BAR_STAGE_FULL));
                    }
                };
                // the first unit at or after `unit` that has a chunk
                auto next_busy = [&](int unit) {
                    while (unit < n_units && unit_span<true>(p, dm, unit).nch == 0) unit += gridDim.x;
                    return unit;
                };
                // chunk k + ahead of this CTA's walk (skipping units without chunks) into
                // L2 only, one chunk ahead of its load
                auto prefetch_after = [&](int unit, int k, int ahead) {
                    k += ahead;
                    Span u = unit_span<true>(p, dm, unit);
                    while (k >= u.nch) {
                        k -= u.nch;
                        unit += gridDim.x;
                        if (unit >= n_units) return;
                        u = unit_span<true>(p, dm, unit);
                    }
                    const int tok = u.t0 + k * kQ;
#pragma unroll
                    for (int bx = 0; bx < 128 / bw; ++bx) tc::tma_prefetch_3d(&tm.x, u.h0 * kP + bx * bw, tok, u.b);
#pragma unroll
                    for (int bx = 0; bx < NN / bw; ++bx) {
                        tc::tma_prefetch_3d(&tm.b, u.g * NN + bx * bw, tok, u.b);
                        tc::tma_prefetch_3d(&tm.c, u.g * NN + bx * bw, tok, u.b);
                    }
                };
                uint32_t yt = 0;  // y tiles stored so far
                // the y tile of chunk k of unit u, once the compute warps staged it; the
                // last chunk of a packed sequence was written straight to y instead
                auto store_y = [&](const Span &u, int k) {
                    wait(BAR_Y_STAGED, yt & 1u);
                    if (!(VARLEN && (k + 1) * kQ > u.len)) {
#pragma unroll
                        for (int bx = 0; bx < 128 / bw; ++bx)
                            tc::tma_store_3d(&tm.y, sbase + L::STG_Y + bx * BOX_BYTES, u.h0 * kP + bx * bw,
                                             u.t0 + k * kQ, u.b);
                        tc::bulk_commit();
                        tc::bulk_wait_read();
                    }
                    tc::mbar_arrive(bar(BAR_Y_FREE));
                    ++yt;
                };
                {
                    const int first = next_busy(blockIdx.x);
                    if (first < n_units) {
                        stage(unit_span<true>(p, dm, first), 0);
                        prefetch_after(first, 0, 1);
                    }
                }
                uint32_t gk = 0;
                for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
                    const Span u = unit_span<VARLEN>(p, dm, unit);
                    for (int k = 0; k < u.nch; ++k, ++gk) {
                        wait(BAR_OPS_FULL, gk & 1u);  // the compute warps are done with the staging area
                        if (k + 1 < u.nch) {
                            stage(u, k + 1);
                        } else {
                            const int nu = next_busy(unit + gridDim.x);
                            if (nu < n_units) stage(unit_span<VARLEN>(p, dm, nu), 0);
                        }
                        prefetch_after(unit, k, 2);
                        if (k > 0) store_y(u, k - 1);
                    }
                    if (u.nch > 0) store_y(u, u.nch - 1);
                }
                tc::bulk_wait_all();
            } else if constexpr (SEG && DIRECT) {
                // chunk g of this CTA's walk into staging buffer g % 2, two chunks ahead:
                // buffer g % 2 takes chunk g + 2 once the products of chunk g have read it
                // (the MMA warp's commit after the intra product)
                auto load_chunk = [&](const Span &u, int k, uint32_t i) {
                    const int tok = u.t0 + k * kQ;
                    const uint32_t sb = sbase + L::STGD + i * DStg::BUF, fb = bar(BAR_DFULL0 + i);
                    tc::mbar_arrive_expect_tx(fb, 8 * BOX_BYTES);
#pragma unroll
                    for (int bx = 0; bx < 2; ++bx) {
                        tc::tma_load_3d(sb + DStg::DX + bx * 16384, &tm.x, u.h0 * kP + bx * 64, tok, u.b, fb);
                        tc::tma_load_3d(sb + DStg::DB + bx * 8192, &tm.b, u.g * NN + bx * 64, tok, u.b, fb);
#pragma unroll
                        for (int cp = 0; cp < 2; ++cp)  // C twice: rows 64-127 of C B^T's A operand
                            tc::tma_load_3d(sb + DStg::DC + bx * 16384 + cp * 8192, &tm.c, u.g * NN + bx * 64, tok, u.b,
                                            fb);
                    }
                    if constexpr (ZM > 0) {  // this chunk's z into L2, ahead of its load into the y tile
#pragma unroll
                        for (int bx = 0; bx < 2; ++bx) tc::tma_prefetch_3d(&tm.z, u.h0 * kP + bx * 64, tok, u.b);
                    }
                };
                // the load cursor: the next chunk of the walk to stage (lu is the span of lunit)
                int lunit = blockIdx.x, lk = 0;
                Span lu{};
                if (lunit < n_units) lu = unit_span<false, true>(p, dm, lunit);
                uint32_t gl = 0;  // chunks staged so far
                auto load_next = [&]() {
                    while (lunit < n_units && lk >= lu.nch) {
                        lk = 0;
                        lunit += gridDim.x;
                        if (lunit < n_units) lu = unit_span<false, true>(p, dm, lunit);
                    }
                    if (lunit >= n_units) return;
                    load_chunk(lu, lk, gl & 1u);
                    ++lk;
                    ++gl;
                };
                auto load_z = [&](const Span &u, int k) {
                    if constexpr (ZM > 0) {
                        const uint32_t zbar = sbase + L::NORM + NORM_ZBAR;
                        tc::mbar_arrive_expect_tx(zbar, 2 * BOX_BYTES);
#pragma unroll
                        for (int bx = 0; bx < 2; ++bx)
                            tc::tma_load_3d(sbase + L::YSTAGE + bx * BOX_BYTES, &tm.z, u.h0 * kP + bx * 64,
                                            u.t0 + k * kQ, u.b, zbar);
                    }
                };
                uint32_t yt = 0;  // y tiles stored so far
                auto store_y = [&](const Span &u, int k) {
                    wait(BAR_Y_STAGED, yt & 1u);
#pragma unroll
                    for (int bx = 0; bx < 2; ++bx)
                        tc::tma_store_3d(&tm.y, sbase + L::YSTAGE + bx * BOX_BYTES, u.h0 * kP + bx * 64,
                                         u.t0 + k * kQ, u.b);
                    tc::bulk_commit();
                    tc::bulk_wait_read();
                    tc::mbar_arrive(bar(BAR_Y_FREE));
                    ++yt;
                };
                load_next();
                load_next();
                if ((int)blockIdx.x < n_units) load_z(unit_span<false, true>(p, dm, blockIdx.x), 0);
                uint32_t gk = 0;
                for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
                    const Span u = unit_span<false, true>(p, dm, unit);
                    const bool more = unit + (int)gridDim.x < n_units;
                    for (int k = 0; k < u.nch; ++k, ++gk) {
                        if (k > 0) {
                            store_y(u, k - 1);
                            load_z(u, k);  // the next tile the compute warps stage
                        }
                        wait(BAR_DFREE0 + (gk & 1u), (gk >> 1) & 1u);  // chunk gk's products have read it
                        load_next();                                   // chunk gk + 2 into the same buffer
                    }
                    store_y(u, u.nch - 1);
                    if (more) load_z(unit_span<false, true>(p, dm, unit + gridDim.x), 0);
                }
                tc::bulk_wait_all();
            } else if constexpr (SEG) {
                // (no L2 prefetch of the next chunk here: at N = 128 it measured slower)
                // x and B of chunk k of a unit into the staging area, expecting C too
                // (its copy is issued by load_c: with y staged in the C tile it has to
                // wait until the previous y tile has left)
                constexpr uint32_t kXBytes = (128 / bw) * BOX_BYTES, kBCBytes = (NN / bw) * BOX_BYTES;
                auto load_xb = [&](const Span &u, int k) {
                    const int tok = u.t0 + k * kQ;
                    tc::mbar_arrive_expect_tx(bar(BAR_STAGE_FULL), kXBytes + 2 * kBCBytes);
#pragma unroll
                    for (int bx = 0; bx < 128 / bw; ++bx)
                        tc::tma_load_3d(sbase + L::STG_X + bx * BOX_BYTES, &tm.x, u.h0 * kP + bx * bw, tok, u.b,
                                        bar(BAR_STAGE_FULL));
#pragma unroll
                    for (int bx = 0; bx < NN / bw; ++bx) {
                        tc::tma_load_3d(sbase + L::STG_B + bx * BOX_BYTES, &tm.b, u.g * NN + bx * bw, tok, u.b,
                                        bar(BAR_STAGE_FULL));
                        if constexpr (kAliasY) tc::tma_prefetch_3d(&tm.c, u.g * NN + bx * bw, tok, u.b);
                    }
                };
                auto load_c = [&](const Span &u, int k) {
                    const int tok = u.t0 + k * kQ;
#pragma unroll
                    for (int bx = 0; bx < NN / bw; ++bx)
                        tc::tma_load_3d(sbase + L::STG_C + bx * BOX_BYTES, &tm.c, u.g * NN + bx * bw, tok, u.b,
                                        bar(BAR_STAGE_FULL));
                    if constexpr (ZM > 0) {  // this chunk's z into L2, ahead of its load into the y tile
#pragma unroll
                        for (int bx = 0; bx < 128 / bw; ++bx) tc::tma_prefetch_3d(&tm.z, u.h0 * kP + bx * bw, tok, u.b);
                    }
                };
                // gated instantiation: the z tile of chunk k into the (free) y staging tile
                auto load_z = [&](const Span &u, int k) {
                    if constexpr (ZM > 0) {
                        const uint32_t zbar = sbase + L::NORM + NORM_ZBAR;
                        tc::mbar_arrive_expect_tx(zbar, (128 / bw) * BOX_BYTES);
#pragma unroll
                        for (int bx = 0; bx < 128 / bw; ++bx)
                            tc::tma_load_3d(sbase + L::YSTAGE + bx * BOX_BYTES, &tm.z, u.h0 * kP + bx * bw,
                                            u.t0 + k * kQ, u.b, zbar);
                    }
                };
                uint32_t yt = 0;  // y tiles stored so far
                auto store_y = [&](const Span &u, int k) {
                    wait(BAR_Y_STAGED, yt & 1u);
#pragma unroll
                    for (int bx = 0; bx < 128 / bw; ++bx)
                        tc::tma_store_3d(&tm.y, sbase + L::YSTAGE + bx * BOX_BYTES, u.h0 * kP + bx * bw,
                                         u.t0 + k * kQ, u.b);
                    tc::bulk_commit();
                    tc::bulk_wait_read();
                    tc::mbar_arrive(bar(BAR_Y_FREE));
                    ++yt;
                };
                if ((int)blockIdx.x < n_units) {
                    const Span u0 = unit_span<false, true>(p, dm, blockIdx.x);
                    load_xb(u0, 0);
                    load_c(u0, 0);
                    load_z(u0, 0);
                }
                uint32_t gk = 0;
                for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
                    const Span u = unit_span<false, true>(p, dm, unit);
                    const bool more = unit + (int)gridDim.x < n_units;
                    const Span nu = unit_span<false, true>(p, dm, more ? unit + gridDim.x : unit);
                    for (int k = 0; k < u.nch; ++k, ++gk) {
                        wait(BAR_OPS_FULL, gk & 1u);  // the compute warps are done with the staging area
                        const bool next_here = k + 1 < u.nch;
                        if (next_here) load_xb(u, k + 1);
                        else if (more) load_xb(nu, 0);
                        // the C tile is free once the compute warps converted it; when y is
                        // staged there, only once y of the previous chunk has left too, and
                        // the next unit's first C then waits for this unit's last y
                        if constexpr (!kAliasY) {
                            if (next_here) load_c(u, k + 1);
                            else if (more) load_c(nu, 0);
                        }
                        if (k > 0) {
                            store_y(u, k - 1);
                            if constexpr (ZM > 0) load_z(u, k);  // the next tile the compute warps stage
                        }
                        if constexpr (kAliasY) {
                            if (next_here) load_c(u, k + 1);
                        }
                    }
                    store_y(u, u.nch - 1);
                    if (more) {
                        if constexpr (kAliasY) load_c(nu, 0);
                        load_z(nu, 0);
                    }
                }
                tc::bulk_wait_all();
            } else {
                // the public x, B, C tiles of chunk k of a unit into the staging area
                auto stage = [&](int unit, int k) {
                    const int pair = unit % pairs, bg = unit / pairs;
                    const int g = bg % dm.G, b = bg / dm.G;
                    const int h0 = g * dm.hpg + 2 * pair;
                    tc::mbar_arrive_expect_tx(bar(BAR_STAGE_FULL), kStageBytes);
#pragma unroll
                    for (int bx = 0; bx < 128 / bw; ++bx)
                        tc::tma_load_3d(sbase + L::STG_X + bx * BOX_BYTES, &tm.x, h0 * kP + bx * bw, k * kQ, b,
                                        bar(BAR_STAGE_FULL));
#pragma unroll
                    for (int bx = 0; bx < NN / bw; ++bx) {
                        tc::tma_load_3d(sbase + L::STG_B + bx * BOX_BYTES, &tm.b, g * NN + bx * bw, k * kQ, b,
                                        bar(BAR_STAGE_FULL));
                        tc::tma_load_3d(sbase + L::STG_C + bx * BOX_BYTES, &tm.c, g * NN + bx * bw, k * kQ, b,
                                        bar(BAR_STAGE_FULL));
                    }
                    if constexpr (ZM > 0) {  // this chunk's z into L2, ahead of its load into the y tile
#pragma unroll
                        for (int bx = 0; bx < 128 / bw; ++bx) tc::tma_prefetch_3d(&tm.z, h0 * kP + bx * bw, k * kQ, b);
                    }
                };
                // chunk k of a unit into L2 only, one chunk ahead of its load: the load
                // (issued when the compute warps release the staging area) then hits L2
                auto prefetch = [&](int unit, int k) {
                    const int pair = unit % pairs, bg = unit / pairs;
                    const int g = bg % dm.G, b = bg / dm.G;
                    const int h0 = g * dm.hpg + 2 * pair;
#pragma unroll
                    for (int bx = 0; bx < 128 / bw; ++bx) tc::tma_prefetch_3d(&tm.x, h0 * kP + bx * bw, k * kQ, b);
#pragma unroll
                    for (int bx = 0; bx < NN / bw; ++bx) {
                        tc::tma_prefetch_3d(&tm.b, g * NN + bx * bw, k * kQ, b);
                        tc::tma_prefetch_3d(&tm.c, g * NN + bx * bw, k * kQ, b);
                    }
                };
                // the chunk `ahead` chunks after chunk k of `unit` in this CTA's walk, if any
                auto prefetch_after = [&](int unit, int k, int ahead) {
                    k += ahead;
                    while (k >= dm.nchunks) {
                        k -= dm.nchunks;
                        unit += gridDim.x;
                    }
                    if (unit < n_units) prefetch(unit, k);
                };
                uint32_t yt = 0;  // y tiles stored so far
                // gated instantiations: the z tile of chunk k of a unit into the (free) y staging tile
                auto load_z = [&](int unit, int k) {
                    if constexpr (ZM > 0) {
                        const int pair = unit % pairs, bg = unit / pairs;
                        const int g = bg % dm.G, b = bg / dm.G;
                        const int h0 = g * dm.hpg + 2 * pair;
                        const uint32_t zbar = sbase + L::NORM + NORM_ZBAR;
                        tc::mbar_arrive_expect_tx(zbar, (IO == IO_F32 ? 4u : 2u) * BOX_BYTES);
#pragma unroll
                        for (int bx = 0; bx < 128 / bw; ++bx)
                            tc::tma_load_3d(sbase + L::STG_Y + bx * BOX_BYTES, &tm.z, h0 * kP + bx * bw, k * kQ, b,
                                            zbar);
                    }
                };
                // the y tile of chunk k of (b, head pair from h0), once the compute warps staged it
                auto store_y = [&](int b, int h0, int k) {
                    wait(BAR_Y_STAGED, yt & 1u);
#pragma unroll
                    for (int bx = 0; bx < 128 / bw; ++bx)
                        tc::tma_store_3d(&tm.y, sbase + L::STG_Y + bx * BOX_BYTES, h0 * kP + bx * bw, k * kQ, b);
                    tc::bulk_commit();
                    tc::bulk_wait_read();
                    tc::mbar_arrive(bar(BAR_Y_FREE));
                    ++yt;
                };
                if ((int)blockIdx.x < n_units) {
                    stage(blockIdx.x, 0);
                    prefetch_after(blockIdx.x, 0, 1);
                    load_z(blockIdx.x, 0);
                }
                uint32_t gk = 0;
                for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
                    const int pair = unit % pairs, bg = unit / pairs;
                    const int g = bg % dm.G, b = bg / dm.G;
                    const int h0 = g * dm.hpg + 2 * pair;
                    for (int k = 0; k < dm.nchunks; ++k, ++gk) {
                        // the staging area is free: the compute warps (or, with the conv1d,
                        // the conv warps) have read it
                        wait(CV ? BAR_STG_FREE : BAR_OPS_FULL, gk & 1u);
                        if (k + 1 < dm.nchunks) stage(unit, k + 1);
                        else if (unit + (int)gridDim.x < n_units) stage(unit + gridDim.x, 0);
                        prefetch_after(unit, k, 2);
                        if (k > 0) {
                            store_y(b, h0, k - 1);
                            load_z(unit, k);  // the next tile the compute warps stage
                        }
                    }
                    store_y(b, h0, dm.nchunks - 1);
                    if (unit + (int)gridDim.x < n_units) load_z(unit + gridDim.x, 0);
                }
                tc::bulk_wait_all();
            }
        }
        __syncwarp();
    } else if (CV && warp >= kConvWarp0) {
        // ---------------- causal conv1d + SiLU, staging tile -> POST ----------------
        // thread ct: x features 2ct, 2ct+1 of the pair (ct < 64), else B (ct < 96) or C
        // features 2 (ct % 32), 2 (ct % 32) + 1 of the group.  A chunk is convolved as
        // soon as its raw tiles land and the compute warps have read the previous
        // chunk's POST; the staging area is then released to the TMA unit.
        const int ct = (warp - kConvWarp0) * 32 + lane;
        const int kind = ct < 64 ? 0 : ct < 96 ? 1 : 2;
        const int f = kind == 0 ? 2 * ct : 2 * (ct & 31);
        const uint32_t src = sbase + (kind == 0 ? L::STG_X : kind == 1 ? L::STG_B : L::STG_C);
        const uint32_t dst = sbase + (kind == 0 ? L::POST : kind == 1 ? L::POST_B : L::POST_C);
        const float *wsrc = kind == 0 ? p.conv_wx : kind == 1 ? p.conv_wb : p.conv_wc;
        const float *bsrc = kind == 0 ? p.conv_bx : kind == 1 ? p.conv_bb : p.conv_bc;
        constexpr int esz = IO == IO_F32 ? 4 : 2, bw = 128 / esz;  // features per 128-byte staging box
        // row r's address: box + r 128 + ((c16 ^ (r % 8)) << 4) + within; rows go 8 at a
        // time from a multiple of 8, so (c16 ^ i) << 4 = (c16 << 4) ^ (i << 4) with i a constant
        const uint32_t sbox = src + (f / bw) * BOX_BYTES + (f % bw) * esz % 16;
        const uint32_t sc16 = (uint32_t)((f % bw) * esz / 16) << 4;
        const uint32_t dbox = dst + (f / 64) * BOX_BYTES + (f % 8) * 2;  // POST: 64 16-bit features per box
        const uint32_t dc16 = (uint32_t)((f % 64) / 8) << 4;
        const int W = p.conv_w;
        uint32_t gc = 0;
        for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
            const Span u = unit_span<false>(p, dm, unit);
            const int cg = kind == 0 ? u.h0 * kP + f : u.g * NN + f;  // the channel in the public tensor
            float w0[4], w1[4];  // taps right-aligned: slot 3 multiplies the current token
#pragma unroll
            for (int sl = 0; sl < 4; ++sl) {
                const int k = sl - (4 - W);
                w0[sl] = k >= 0 ? __ldg(wsrc + (size_t)cg * W + k) : 0.f;
                w1[sl] = k >= 0 ? __ldg(wsrc + (size_t)(cg + 1) * W + k) : 0.f;
            }
            const float b0 = bsrc ? __ldg(bsrc + cg) : 0.f, b1 = bsrc ? __ldg(bsrc + cg + 1) : 0.f;
            float h0[3] = {0.f, 0.f, 0.f}, h1[3] = {0.f, 0.f, 0.f};  // tokens t-3, t-2, t-1
            for (int k = 0; k < u.nch; ++k, ++gc) {
                wait(BAR_STAGE_FULL, gc & 1u);
                if (gc > 0) wait(BAR_OPS_FULL, (gc - 1) & 1u);  // the compute warps have read POST
                // 8 rows at a time: their loads first (independent), then the taps and
                // SiLU of 8 rows, then 8 stores, so the latencies overlap
                for (int r0 = 0; r0 < kQ; r0 += 8) {
                    float v0[8], v1[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t sa = sbox + (r0 + i) * 128 + (sc16 ^ (i << 4));
                        if (IO == IO_F32) {
                            asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v0[i]), "=f"(v1[i]) : "r"(sa));
                        } else {
                            uint32_t wv;
                            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(wv) : "r"(sa));
                            float2 fv;
                            if (IO == IO_BF16) fv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&wv));
                            else fv = __half22float2(*reinterpret_cast<const __half2 *>(&wv));
                            v0[i] = fv.x; v1[i] = fv.y;
                        }
                    }
                    uint32_t out[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float o0 =
                            fmaf(w0[3], v0[i], fmaf(w0[2], h0[2], fmaf(w0[1], h0[1], fmaf(w0[0], h0[0], b0))));
                        const float o1 =
                            fmaf(w1[3], v1[i], fmaf(w1[2], h1[2], fmaf(w1[1], h1[1], fmaf(w1[0], h1[0], b1))));
                        h0[0] = h0[1]; h0[1] = h0[2]; h0[2] = v0[i];
                        h1[0] = h1[1]; h1[1] = h1[2]; h1[2] = v1[i];
                        out[i] = pack2(silu_tanh(o0), silu_tanh(o1), BF16);
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t da = dbox + (r0 + i) * 128 + (dc16 ^ (i << 4));
                        asm volatile("st.shared.b32 [%0], %1;" ::"r"(da), "r"(out[i]) : "memory");
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    tc::mbar_arrive(bar(BAR_CONV_DONE));
                    tc::mbar_arrive(bar(BAR_STG_FREE));
                }
            }
        }
    } else if (warp >= kDecayWarp0) {
        // ---------------- decay vectors, one head per warp ----------------
        const int hh = warp - kDecayWarp0;
        uint32_t gd = 0;
        if constexpr (!VARLEN && !SEG) {
            // The raw dt of the walk's next chunk is loaded before the current one's
            // vectors are computed, so a chunk never waits for its own (strided) loads
            // (1.047 -> 1.023 ms at the large training shape; with packed sequences it
            // measured 1.108 -> 1.180 ms, and neutral on the segmented walks, which
            // keep the loop below).
            int unit = blockIdx.x, k = 0;
            Span u{};
            if (unit < n_units) u = unit_span<false, false>(p, dm, unit);
            // move (unit, k) to the first chunk at or after it in this CTA's walk (u is the
            // span of `unit`, computed once per unit); false past the last chunk
            auto settle = [&]() {
                while (unit < n_units && k >= u.nch) {
                    k = 0;
                    unit += gridDim.x;
                    if (unit < n_units) u = unit_span<false, false>(p, dm, unit);
                }
                return unit < n_units;
            };
            DtRegs r{};
            bool have = settle();
            if (have) load_dt(p, dm, u, u.h0 + hh, k, lane, r);
            while (have) {
                const Span cu = u;
                const int ck = k;
                const DtRegs cr = r;
                ++k;
                have = settle();
                if (have) load_dt(p, dm, u, u.h0 + hh, k, lane, r);
                const int slot = gd % kVecSlots;
                if (gd >= (uint32_t)kVecSlots) wait(BAR_VEC_EMPTY0 + slot, (gd / kVecSlots - 1) & 1u);
                decay_vectors(p, cu.h0 + hh, hh, cu.len - ck * kQ, lane, cr.dt0, cr.dt1, Vbuf[slot]);
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(bar(BAR_VEC_FULL0 + slot));
                ++gd;
            }
        } else {
            for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
                const Span u = unit_span<VARLEN, SEG>(p, dm, unit);
                const int h = u.h0 + hh;
                for (int k = 0; k < u.nch; ++k, ++gd) {
                    DtRegs r;
                    load_dt(p, dm, u, h, k, lane, r);
                    const int slot = gd % kVecSlots;
                    if (gd >= (uint32_t)kVecSlots) wait(BAR_VEC_EMPTY0 + slot, (gd / kVecSlots - 1) & 1u);
                    decay_vectors(p, h, hh, u.len - k * kQ, lane, r.dt0, r.dt1, Vbuf[slot]);
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(bar(BAR_VEC_FULL0 + slot));
                }
            }
        }
    } else {
        // ---------------- compute warps ----------------
        const int wg = warp >> 2, quarter = warp & 3;
        const int row = quarter * 32 + lane;  // TMEM lane owned by this thread
        const int my_h = row >> 6, my_p = row & 63;
        const int col0 = wg * kGCols;         // this thread's columns of each 64-column region
        const int scol0 = wg * kSCols;        // this thread's state columns
        const uint32_t tlane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        uint32_t gk = 0;
        uint32_t yt = 0;  // y tiles staged so far
        NormCtx nc{};
        float norm_wf = 0.f;  // per unit: this feature's norm weight
        if constexpr (ZM == 2) {
            nc.lpart = sbase + L::NORM + NORM_LPART;
            nc.recv = sbase + L::NORM + NORM_RECV;
            nc.rbar = sbase + L::NORM + NORM_BARS;
            nc.cs = norm_cs;
            nc.rank = norm_cs > 1 ? (int)tc::cluster_ctarank() : 0;
        }
        // epilogue of global chunk gp (chunk kk of the unit) into the y staging tile
        // (the last chunk of a packed sequence straight into y)
        auto epilogue = [&](uint32_t gp, int kk, int b, int h0, int t0, int len) {
            const int bp = gp & 1;
            const bool direct = VARLEN && (kk + 1) * kQ > len;
            if (yt > 0) wait(BAR_Y_FREE, (yt - 1) & 1u);  // the TMA unit has read the previous tile
            wait(bp ? BAR_Y_DONE1 : BAR_Y_DONE0, (gp >> 1) & 1u);
            if constexpr (ZM > 0) {  // this tile's z is in the staging tile
                if (!timed_out && !tc::mbar_wait(sbase + L::NORM + NORM_ZBAR, yt & 1u, kWaitNs)) timed_out = true;
            }
            tc::fence_after_sync();
            if constexpr (ZM == 2) {
                epilogue_norm<IO>(p, dm, Vbuf[gp % kVecSlots], tlane, bp, col0, b, h0, my_h, my_p, kk * kQ + col0,
                                  sbase + L::STG_Y, nc, gp, wg, quarter, lane, norm_wf, timed_out);
            } else if constexpr (NN == 128) {
                epilogue_tokens<IO, VARLEN, ZM, NN, SEG, 16>(p, dm, Vbuf[gp % kVecSlots], tlane, bp, col0, b, h0,
                                                             my_h, my_p, kk * kQ + col0, sbase + L::YSTAGE, t0, len,
                                                             direct);
            } else {
                epilogue_tokens<IO, VARLEN, ZM, NN, SEG, 8, false>(p, dm, Vbuf[gp % kVecSlots], tlane, bp, col0, b, h0,
                                                                   my_h, my_p, kk * kQ + col0, sbase + L::YSTAGE, t0,
                                                                   len, direct);
                epilogue_tokens<IO, VARLEN, ZM, NN, SEG, 8, true>(p, dm, Vbuf[gp % kVecSlots], tlane, bp, col0 + 8, b, h0,
                                                                  my_h, my_p, kk * kQ + col0 + 8, sbase + L::YSTAGE, t0,
                                                                  len, direct);
            }
            __syncwarp();
            if (lane == 0) {
                tc::mbar_arrive(bar(BAR_Y_STAGED));
                tc::mbar_arrive(bar(BAR_VEC_EMPTY0 + gp % kVecSlots));
            }
            ++yt;
        };
        // NN = 64: the bf16 copy of the state S (the A operand of Yoff = S C^T) into
        // shared memory, or into TMEM in the conv1d instantiation; the caller arrives
        // on S_FULL
        auto publish_bf16_state = [&](const float (&Sv)[kSCols]) {
            if constexpr (NN == 64) {
                if constexpr (L::kStateBfTmem) {
                    uint32_t r[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) r[i] = pack2(Sv[2 * i], Sv[2 * i + 1], BF16);
                    tc::tmem_st8(tlane + TM_SBF + scol0 / 2, r);
                    tc::tmem_wait_st();
                    tc::fence_before_sync();
                } else {
#pragma unroll
                    for (int q = 0; q < kSCols / 8; ++q) {
                        float v[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[e] = Sv[8 * q + e];
                        const int ng = (scol0 >> 3) + q;
                        store8(sbase + L::S + (ng * 16 + (row >> 3)) * 128 + (row & 7) * 16, v, BF16);
                    }
                    // The product that reads this copy (Yoff) is issued only after the next chunk's
                    // OPS_FULL, which these threads arrive on behind the operand stage's own proxy
                    // fence, so none is needed here (a fence here as well measured 0.999 ms against
                    // 0.986 at the large training shape; packed sequences keep it: 1.082 against
                    // 1.090 ms without)
                    if constexpr (VARLEN) tc::fence_smem_to_async();
                }
                __syncwarp();
            }
        };
        // NN = 128: the state S (this thread's kSCols columns of row (head, p))
        // goes to TMEM twice before the products of a chunk: decayed by the
        // chunk's exp(cs_last) as the fp32 accumulator that S += Xw^T B adds to,
        // and as the bf16 A operand of Yoff = S C^T
        auto publish_state = [&](const float (&Sv)[kSCols], float a) {
            if constexpr (NN == 128) {
                uint32_t r[16];
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(a * Sv[16 * hf + i]);
                    tc::tmem_st16(tlane + TM_S32 + scol0 + 16 * hf, r);
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) r[i] = pack2(Sv[2 * i], Sv[2 * i + 1], BF16);
                tc::tmem_st16(tlane + TM_SBF + scol0 / 2, r);
                tc::tmem_wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(bar(BAR_S_FULL));
            }
        };

        for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
            // b: batch row, h0: first head, sb: state index (b, or the packed
            // sequence), t0 / len: the unit's tokens in its row, nch: its chunks,
            // seg: its segment (segmented walks)
            int b, h0, sb, t0 = 0, len = 0, nch = dm.nchunks, seg = 0;
            if (VARLEN || SEG) {
                const Span u = unit_span<VARLEN, SEG>(p, dm, unit);
                b = u.b; h0 = u.h0; sb = u.sb; t0 = u.t0; len = u.len; nch = u.nch; seg = u.seg;
            } else {
                const int pairs = dm.hpg >> 1;
                const int pair = unit % pairs;
                const int bg = unit / pairs;
                const int g = bg % dm.G;
                b = bg / dm.G;
                h0 = g * dm.hpg + 2 * pair;
                sb = b;
            }
            if constexpr (ZM == 2) {
                norm_wf = __ldg(p.norm_w + (size_t)(h0 + my_h) * kP + my_p);
            }

            // state of (head my_h, row my_p), columns n = scol0 .. scol0+kSCols-1: the
            // initial state, or for a later segment the state the segment passes left
            float S[kSCols];
            {
                const float *src = nullptr;
                if (SEG && seg > 0) {
                    // launched as a programmatic dependent of the fold: its states are
                    // visible once the fold has completed (a no-op after the first time)
                    tc::pdl_wait();
                    src = p.seg_states + ((((size_t)b * p.nseg + seg) * dm.H + h0 + my_h) * kP + my_p) * NN + scol0;
                }
                else if (p.h0)
                    src = p.h0 + (((size_t)sb * dm.H + h0 + my_h) * kP + my_p) * NN + scol0;
                if (src) {
                    const float4 *s4 = reinterpret_cast<const float4 *>(src);
#pragma unroll
                    for (int q = 0; q < kSCols / 4; ++q) {
                        const float4 v = __ldg(s4 + q);
                        S[4 * q] = v.x; S[4 * q + 1] = v.y; S[4 * q + 2] = v.z; S[4 * q + 3] = v.w;
                    }
                } else {
#pragma unroll
                    for (int n = 0; n < kSCols; ++n) S[n] = 0.f;
                }
            }
            if constexpr (NN == 64) {
                publish_bf16_state(S);
                // (a packed sequence without tokens has no chunk to consume this state)
                if (lane == 0 && (!VARLEN || nch > 0)) tc::mbar_arrive(bar(BAR_S_FULL));
            }

            for (int k = 0; k < nch; ++k, ++gk) {
                const int buf = gk & 1;
                const int xbuf = L::kXcBufs == 2 ? buf : 0;
                const uint32_t ph = gk & 1u;
                ChunkVec &V = Vbuf[gk % kVecSlots];
                wait(BAR_VEC_FULL0 + gk % kVecSlots, (gk / kVecSlots) & 1u);  // decay vectors of chunk k
                if constexpr (NN == 128) {
                    if (k == 0) publish_state(S, V.a[my_h]);
                }

                // ---- A: operands of chunk k into shared memory ----
                if constexpr (DIRECT) wait(BAR_DFULL0 + (gk & 1u), (gk >> 1) & 1u);
                else wait(CV ? BAR_CONV_DONE : BAR_STAGE_FULL, ph);  // with the conv1d: once it has run
                // one Xcat buffer: the previous chunk's intra product has read it
                if (L::kXcBufs == 1 && gk > 0) wait((gk - 1) & 1 ? BAR_Y_DONE1 : BAR_Y_DONE0, ((gk - 1) >> 1) & 1u);
                {
                    float wv[2];
#pragma unroll
                    for (int it = 0; it < 2; ++it) {
                        const int e = tid + kComputeThreads * it;
                        const int jl = e & 7, c16 = (e >> 3) & 15, jg = e >> 7;
                        wv[it] = V.w[c16 >> 3][jg * 8 + jl];
                    }
                    const uint32_t xc = sbase + L::XC + xbuf * XC_BYTES;
#pragma unroll
                    for (int it = 0; it < 2; ++it) {
                        const int e = tid + kComputeThreads * it;
                        const int jl = e & 7, c16 = (e >> 3) & 15, jg = e >> 7;
                        const int h = c16 >> 3, po = c16 & 7;
                        const int mgc = h ? 16 + po : po;
                        const uint32_t xsrc = sbase + (CV ? L::POST : L::STG_X);
                        float xv[8];
                        if constexpr (DIRECT) {  // only the weighted copy: the products read x in place
                            const uint32_t xb = sbase + L::STGD + (gk & 1u) * DStg::BUF + DStg::DX + h * 16384;
                            tcstage::unpack8(tc::ld_shared_v4(tcstage::swz(xb, jg * 8 + jl, po)), BF16, xv);
                        } else if constexpr (kRaw) {  // the staged chunk is the operand already
                            const uint4 raw = stage_raw16(xsrc, jg * 8 + jl, c16);
                            st_shared_v4(xc + (jg * 24 + mgc) * 128 + jl * 16, raw.x, raw.y, raw.z, raw.w);
                            tcstage::unpack8(raw, BF16, xv);
                        } else {
                            stage_read8<SIO>(xsrc, jg * 8 + jl, c16, xv);
                            store8(xc + (jg * 24 + mgc) * 128 + jl * 16, xv, BF16);
                        }
                        float xs[8];
#pragma unroll
                        for (int q = 0; q < 8; ++q) xs[q] = xv[q] * wv[it];
                        store8(sbase + L::XT + (jg * 16 + 8 * h + po) * 128 + jl * 16, xs, BF16);
                    }
#pragma unroll
                    for (int it = 0; it < (DIRECT ? 0 : NN / 64); ++it) {  // (DIRECT: B and C are read in place)
                        const int e = tid + kComputeThreads * it;
                        const int jl = e & 7, ng = (e >> 3) & (NN / 8 - 1), jg = e / NN;
                        const uint32_t bsrc = sbase + (CV ? L::POST_B : L::STG_B);
                        const uint32_t csrc = sbase + (CV ? L::POST_C : L::STG_C);
                        const uint32_t bdst = sbase + L::BB + (ng * 8 + jg) * 128 + jl * 16;
                        const uint32_t cdst = sbase + L::CB2 + (ng * 16 + jg) * 128 + jl * 16;
                        if constexpr (kRaw) {  // B and C move as they are
                            const uint4 rb = stage_raw16(bsrc, jg * 8 + jl, ng);
                            const uint4 rc = stage_raw16(csrc, jg * 8 + jl, ng);
                            st_shared_v4(bdst, rb.x, rb.y, rb.z, rb.w);
                            st_shared_v4(cdst, rc.x, rc.y, rc.z, rc.w);
                            st_shared_v4(cdst + 8 * 128, rc.x, rc.y, rc.z, rc.w);
                        } else {
                            float bv[8], cv[8];
                            stage_read8<SIO>(bsrc, jg * 8 + jl, ng, bv);
                            stage_read8<SIO>(csrc, jg * 8 + jl, ng, cv);
                            store8(bdst, bv, BF16);
                            store8(cdst, cv, BF16);
                            store8(cdst + 8 * 128, cv, BF16);
                        }
                    }
                }
                tc::fence_smem_to_async();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(bar(BAR_OPS_FULL));
                // y staged in the C tile: every compute warp has read chunk k's C first
                if constexpr (kAliasY) tc::named_barrier(5, kComputeThreads);

                // ---- D: epilogue of the previous chunk (overlaps the G MMA) ----
                if (k > 0) epilogue(gk - 1, k - 1, b, h0, t0, len);

                // ---- B: masked, decayed C B^T -> Mcat ----
                // A warp whose rows are 0-31 and columns 32-63 holds only blocks above the
                // diagonal: they stay as zeroed at start, and the warp skips the phase.
                if (!((quarter & 1) == 0 && wg >= 2)) {
                    const int i = row & 63, h = row >> 6;
                    const float csi = V.cs2[h][i];
                    // D x_i as D on the diagonal of the intra-chunk matrix (the diagonal's decay is
                    // exp(0) = 1): on the tensor core with x's operand rounding, no x loads in the epilogue
                    const float diag_d = p.D ? __ldg(p.D + h0 + h) : 0.f;
                    wait(BAR_G_DONE, ph);
                    tc::fence_after_sync();
                    const uint32_t mc = sbase + L::MC;
                    // the thread's 16 columns with one wait, and no mask on blocks that lie wholly
                    // below the diagonal (at N = 64 two 8-column loads with the mask everywhere
                    // measured 1.024 ms against 1.012 at the large training shape)
                    float gall[kGCols];
                    tc::tmem_ld16(tlane + TM_G + col0, gall);
                    const int rows_lo = 32 * (quarter & 1);  // the warp's first row i
#pragma unroll
                    for (int q = 0; q < kGCols / 8; ++q) {
                        const int j0 = col0 + 8 * q;
                        const float4 c0 = *reinterpret_cast<const float4 *>(&V.cs2[h][j0]);
                        const float4 c1 = *reinterpret_cast<const float4 *>(&V.cs2[h][j0 + 4]);
                        const float4 d0 = *reinterpret_cast<const float4 *>(&V.d[h][j0]);
                        const float4 d1 = *reinterpret_cast<const float4 *>(&V.d[h][j0 + 4]);
                        const float cj[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                        const float dj[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
                        float m[8];
                        if (j0 + 7 < rows_lo) {  // (warp-uniform) wholly below the diagonal
#pragma unroll
                            for (int e = 0; e < 8; ++e) m[e] = gall[8 * q + e] * ex2_approx(csi - cj[e]) * dj[e];
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const float v = gall[8 * q + e] * ex2_approx(csi - cj[e]) * dj[e];
                                m[e] = (j0 + e <= i) ? v : 0.f;
                                m[e] += (j0 + e == i) ? diag_d : 0.f;
                            }
                        }
                        const int kg = 8 * h + (j0 >> 3);
                        store8(mc + (kg * 8 + (i >> 3)) * 128 + (i & 7) * 16, m, BF16);
                    }
                    tc::fence_before_sync();
                }
                tc::fence_smem_to_async();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(bar(BAR_MCAT_FULL));

                // ---- C: state update S <- exp(cs_last) S + dS ----
                if constexpr (NN == 64) {
                    const float a = V.a[my_h];
                    wait(BAR_DS_DONE, ph);
                    tc::fence_after_sync();
                    float ds[kSCols];
                    tc::tmem_ld16(tlane + TM_DS + scol0, ds);
                    tc::fence_before_sync();
#pragma unroll
                    for (int n = 0; n < kSCols; ++n) S[n] = fmaf(a, S[n], ds[n]);
                    if (k + 1 < nch) {
                        publish_bf16_state(S);
                        if (lane == 0) tc::mbar_arrive(bar(BAR_S_FULL));
                    }
                } else {
                    // the tensor core added dS onto the decayed state: read S back, and
                    // publish it for the next chunk, decayed by that chunk's exp(cs_last)
                    wait(BAR_DS_DONE, ph);
                    tc::fence_after_sync();
                    float s16[16];
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        tc::tmem_ld16(tlane + TM_S32 + scol0 + 16 * hf, s16);
#pragma unroll
                        for (int i = 0; i < 16; ++i) S[16 * hf + i] = s16[i];
                    }
                    tc::fence_before_sync();
                    if (k + 1 < nch) {
                        const uint32_t gn = gk + 1;
                        wait(BAR_VEC_FULL0 + gn % kVecSlots, (gn / kVecSlots) & 1u);
                        publish_state(S, Vbuf[gn % kVecSlots].a[my_h]);
                    }
                }
            }

            // ---- drain: epilogue of the unit's last chunk, final state ----
            if (!VARLEN || nch > 0) epilogue(gk - 1, nch - 1, b, h0, t0, len);
            if (p.final_state && (!SEG || seg == p.nseg - 1)) {
                float4 *dst = reinterpret_cast<float4 *>(
                    p.final_state + (((size_t)sb * dm.H + h0 + my_h) * kP + my_p) * NN + scol0);
#pragma unroll
                for (int q = 0; q < kSCols / 4; ++q)
                    dst[q] = make_float4(S[4 * q], S[4 * q + 1], S[4 * q + 2], S[4 * q + 3]);
            }
        }
    }

    if (timed_out) atomicOr(err, 1u);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == kMmaWarp) tc::tmem_dealloc(tmem, TM_COLS);
    if constexpr (ZM == 2) {  // no CTA leaves while a partner may still write into its shared memory
        if (norm_cs > 1) tc::cluster_sync();
    }
}

// SM count of the current device, looked up once per device index (plan
// choice and the persistent grids depend on it).
constexpr int kMaxDevices = 64;
std::mutex g_sms_mu;
int g_num_sms[kMaxDevices] = {};

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        (void)cudaGetLastError();
        dev = 0;
    }
    int n = 0;
    if (dev >= kMaxDevices) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) (void)cudaGetLastError();
        return n > 0 ? n : 1;
    }
    std::lock_guard<std::mutex> lock(g_sms_mu);
    if (g_num_sms[dev] == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) (void)cudaGetLastError();
        g_num_sms[dev] = n > 0 ? n : 1;
    }
    return g_num_sms[dev];
}

int64_t fused_units(const ssd_fwd_args *a) { return a->B * a->G * ((a->H / a->G) / 2); }

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

}  // namespace

cudaError_t encode_tile_map(CUtensorMap *m, const void *base, int io, int64_t feats, int64_t L, int64_t B,
                            bool swizzle) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    const size_t esz = io == IO_F32 ? 4 : 2;
    const CUtensorMapDataType dt = io == IO_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : io == IO_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const cuuint64_t dims[3] = {(cuuint64_t)feats, (cuuint64_t)L, (cuuint64_t)B};
    const cuuint64_t strides[2] = {(cuuint64_t)(feats * esz), (cuuint64_t)(feats * L * esz)};
    const cuuint32_t box[3] = {(cuuint32_t)(128 / esz), (cuuint32_t)kQ, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {

template <int IO, bool BF16, int NN>
cudaError_t launch_typed(const Params &p, int units, unsigned int *err, cudaStream_t s) {
    using L = Smem<NN, IO>;
    // packed variable-length sequences and the fused norm get their own
    // instantiations, so that the regular layout pays nothing for them;
    // z is staged by TMA through the y tile (ZM 1; with the norm, ZM 2),
    // except where y itself is staged in the C tile (fp32 I/O at N = 128):
    // the epilogue then loads z from global memory
    // (the in-kernel conv1d, N = 64 only, has instantiations of its own with 4 more warps)
    const bool norm = NN == 64 && p.norm_w && !p.cu;
    const bool gated = p.z && !p.cu && !L::kAliasY;
    const bool conv = NN == 64 && p.conv_w > 0 && !p.cu && !norm;
    auto kern = ssd_fused_kernel<IO, BF16, false, 0, NN>;
    if constexpr (NN == 64) {
        if (p.cu) kern = ssd_fused_kernel<IO, BF16, true, 0>;
        else if (conv) kern = gated ? ssd_fused_kernel<IO, BF16, false, 1, 64, true>
                                    : ssd_fused_kernel<IO, BF16, false, 0, 64, true>;
        else if (norm) kern = ssd_fused_kernel<IO, BF16, false, 2>;
        else if (gated) kern = ssd_fused_kernel<IO, BF16, false, 1>;
    } else if constexpr (!L::kAliasY) {
        if (gated) kern = ssd_fused_kernel<IO, BF16, false, 1, NN>;
    }
    const int threads = conv ? kThreadsConv : kThreads;
    using LC = Smem<64, IO, true>;  // (the conv1d instantiation exists at N = 64 only)
    const uint32_t smem = conv ? (gated ? LC::BYTES_NORM : LC::BYTES) : gated ? L::BYTES_NORM : L::BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    TmaMaps tm;
    if ((e = encode_tile_map(&tm.x, p.x, IO, (int64_t)p.H * kP, p.L, p.B, true)) != cudaSuccess) return e;
    if ((e = encode_tile_map(&tm.b, p.Bm, IO, (int64_t)p.G * NN, p.L, p.B, true)) != cudaSuccess) return e;
    if ((e = encode_tile_map(&tm.c, p.Cm, IO, (int64_t)p.G * NN, p.L, p.B, true)) != cudaSuccess) return e;
    if ((e = encode_tile_map(&tm.y, p.y, IO, (int64_t)p.H * kP, p.L, p.B, false)) != cudaSuccess) return e;
    if (gated && (e = encode_tile_map(&tm.z, p.z, IO, (int64_t)p.H * kP, p.L, p.B, false)) != cudaSuccess) return e;
    // one CTA per SM: its shared memory and 512 TMEM columns fill the SM
    if (!norm) {
        const int grid = units < num_sms() ? units : num_sms();
        if (p.nseg > 1) {
            // after the segment passes: a programmatic dependent launch, so that the
            // walk's CTAs set up (and walk the first segment, which needs no passed
            // state) while the fold finishes; they wait for it before reading states
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.gridDim = dim3((unsigned)grid);
            cfg.blockDim = dim3((unsigned)threads);
            cfg.dynamicSmemBytes = smem;
            cfg.stream = s;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            e = cudaLaunchKernelEx(&cfg, kern, p, tm, units, err, 1);
            if (e != cudaSuccess) return e;
            return cudaGetLastError();
        }
        kern<<<grid, threads, smem, s>>>(p, tm, units, err, 1);
        return cudaGetLastError();
    }
    // fused norm: the head pairs of a group run in one cluster of cs CTAs, in
    // step (unit u goes to the CTA of rank u % cs, and the grid is a multiple of cs)
    const int cs = p.hpg / 2;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = cs > 1 ? 1 : 0;
    int clusters = num_sms() / cs;
    if (cs > 1) {
        cfg.gridDim = dim3((unsigned)(clusters * cs));
        int active = 0;
        if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) == cudaSuccess && active > 0 && active < clusters)
            clusters = active;
        (void)cudaGetLastError();
    }
    int grid = clusters * cs;
    if (grid > units) grid = units;  // units is a multiple of cs
    cfg.gridDim = dim3((unsigned)grid);
    e = cudaLaunchKernelEx(&cfg, kern, p, tm, units, err, cs);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

// How a walk at N = 128 is cut into segments: nseg segments of seg_len tokens
// (a multiple of 64, the last one possibly shorter), chosen by a cost model
// in microseconds from measurements on GB300: rounds of (batch, group, head
// pair, segment) units over the SMs, each a segment's 64-token steps (about
// 7 us each at N = 128) plus about 3 us to start a unit; with more than one
// segment, the pre-pass re-reading x and B and writing the segment states,
// and the fold (a dependent step of about 1 us per segment, and the states
// read and written), at about 6 TB/s, plus two more launches.
struct SegPlan {
    int nseg, seg_len;
};

SegPlan seg_plan(const ssd_fwd_args *a) {
    const int64_t units0 = fused_units(a);
    const int64_t nsub = (a->L + kQ - 1) / kQ;
    const int64_t sms = num_sms();
    const double io = a->x_dtype == SSD_F32 ? 4.0 : 2.0;
    constexpr double kStepUs = 7.0, kUnitUs = 3.0, kFoldStepUs = 1.0, kLaunchUs = 6.0, kBytesPerUs = 6.0e6;
    const double reread_us = (double)a->B * a->L * (a->H * a->P + a->G * a->N) * io / kBytesPerUs;
    const double states_us = (double)a->B * a->H * a->P * a->N * 4.0 / kBytesPerUs;  // one segment boundary
    SegPlan best{1, (int)(nsub * kQ)};
    double best_cost = (double)((units0 + sms - 1) / sms) * (nsub * kStepUs + kUnitUs);
    for (int64_t want = 2; want <= nsub && want <= 256; ++want) {
        const int64_t steps = (nsub + want - 1) / want;
        const int64_t nseg = (nsub + steps - 1) / steps;
        const int seg_len = (int)(steps * kQ);
        if (nseg < 2 || !segment_smem_fits(a->x_dtype, seg_len)) continue;
        const double walk = (double)((units0 * nseg + sms - 1) / sms) * (steps * kStepUs + kUnitUs);
        const double pre = reread_us * (double)(nseg - 1) / nseg + states_us * (nseg - 1);
        const double fold = kFoldStepUs * nseg + 2.0 * states_us * (nseg - 1);
        const double cost = walk + pre + fold + kLaunchUs;
        if (cost < best_cost) {
            best_cost = cost;
            best = {(int)nseg, seg_len};
        }
    }
    return best;
}

size_t seg_states_bytes(const ssd_fwd_args *a, int nseg) {
    return up256((size_t)a->B * nseg * a->H * a->P * a->N * sizeof(float));
}

}  // namespace

const char *fused_unsupported_reason(const ssd_fwd_args *a) {
    if (a->P != kP) return "needs P = 64";
    if (a->N != 64 && a->N != 128) return "needs N = 64 or 128";
    if (a->chunk % kQ != 0) return "needs a chunk size that is a multiple of 64 (it walks each chunk in 64-token steps)";
    if ((a->H / a->G) % 2 != 0) return "needs an even number of heads per group";
    if (a->ops == SSD_OPS_F32) return "needs fp16 or bf16 operands (the fp32 path is the chunked plan)";
    if (fused_units(a) * ((a->L + kQ - 1) / kQ) > 0x7fffffffLL) return "too many (batch, group, head pair) units";
    for (const void *ptr : {static_cast<const void *>(a->x), static_cast<const void *>(a->Bm),
                            static_cast<const void *>(a->Cm), static_cast<const void *>(a->y)})
        if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return "needs 16-byte aligned x, B, C and y";
    if (a->z && reinterpret_cast<uintptr_t>(a->z) % 16 != 0) return "needs a 16-byte aligned z (its tiles come by TMA)";
    return nullptr;
}

bool fused_supported(const ssd_fwd_args *a) { return fused_unsupported_reason(a) == nullptr; }

bool fused_varlen_supported(const ssd_fwd_args *a) { return fused_supported(a) && a->N == 64; }

bool fused_conv_supported(const ssd_fwd_args *a) { return fused_supported(a) && a->N == 64; }

bool fused_norm_supported(const ssd_fwd_args *a) {
    return fused_supported(a) && a->N == 64 && a->z && (a->H / a->G) / 2 <= kNormMaxRanks;
}

// N = 64: the unit-sequential walk needs as many units as SMs; at N = 128 the
// segmented walk fills the GPU by itself.
bool fused_preferred(const ssd_fwd_args *a) { return a->N == 128 || fused_units(a) >= num_sms(); }

int fused_segments(const ssd_fwd_args *a) { return a->N == 128 ? seg_plan(a).nseg : 1; }

size_t fused_workspace_size(const ssd_fwd_args *a) {
    if (a->N != 128) return 256;
    const SegPlan sp = seg_plan(a);
    if (sp.nseg < 2) return 256;
    return 256 + seg_states_bytes(a, sp.nseg) + up256((size_t)a->B * a->H * sp.nseg * sizeof(float));
}

namespace {

Params fused_params(const ssd_fwd_args *a) {
    Params p;
    p.B = (int)a->B; p.L = (int)a->L; p.H = (int)a->H; p.P = (int)a->P; p.N = (int)a->N;
    p.G = (int)a->G; p.Q = kQ;  // every chunk is walked in 64-token steps
    p.nchunks = (int)((a->L + kQ - 1) / kQ);
    p.hpg = (int)(a->H / a->G);
    p.x = a->x; p.dt = a->dt; p.A = a->A; p.Bm = a->Bm; p.Cm = a->Cm; p.D = a->D; p.z = a->z;
    p.dt_bias = a->dt_bias; p.h0 = a->initial_state; p.y = a->y; p.final_state = a->final_state;
    p.dt_softplus = a->dt_softplus ? 1 : 0;
    p.has_limit = !(a->dt_min == 0.f && isinf(a->dt_max) && a->dt_max > 0.f);
    p.dt_min = a->dt_min; p.dt_max = a->dt_max;
    p.norm_w = a->norm_weight;
    p.norm_eps = a->norm_eps;
    p.conv_wx = a->conv_x_weight; p.conv_bx = a->conv_x_bias;
    p.conv_wb = a->conv_b_weight; p.conv_bb = a->conv_b_bias;
    p.conv_wc = a->conv_c_weight; p.conv_bc = a->conv_c_bias;
    p.conv_w = a->conv_width;
    return p;
}

// The fused kernel (the error word at err cleared by the caller).
cudaError_t launch(const ssd_fwd_args *a, const Params &p, int units, unsigned int *err, cudaStream_t s) {
    const bool bf16 = a->ops == SSD_OPS_BF16;
    if (a->N == 128) {
        switch (a->x_dtype) {
            case SSD_F32: return bf16 ? launch_typed<IO_F32, true, 128>(p, units, err, s) : launch_typed<IO_F32, false, 128>(p, units, err, s);
            case SSD_F16: return bf16 ? launch_typed<IO_F16, true, 128>(p, units, err, s) : launch_typed<IO_F16, false, 128>(p, units, err, s);
            case SSD_BF16: return bf16 ? launch_typed<IO_BF16, true, 128>(p, units, err, s) : launch_typed<IO_BF16, false, 128>(p, units, err, s);
        }
        return cudaErrorInvalidValue;
    }
    switch (a->x_dtype) {
        case SSD_F32: return bf16 ? launch_typed<IO_F32, true, 64>(p, units, err, s) : launch_typed<IO_F32, false, 64>(p, units, err, s);
        case SSD_F16: return bf16 ? launch_typed<IO_F16, true, 64>(p, units, err, s) : launch_typed<IO_F16, false, 64>(p, units, err, s);
        case SSD_BF16: return bf16 ? launch_typed<IO_BF16, true, 64>(p, units, err, s) : launch_typed<IO_BF16, false, 64>(p, units, err, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t run_fused(const ssd_fwd_args *a, cudaStream_t s) {
    unsigned int *err = static_cast<unsigned int *>(a->workspace);
    cudaError_t e = cudaMemsetAsync(err, 0, 256, s);
    if (e != cudaSuccess) return e;
    Params p = fused_params(a);
    int64_t units = fused_units(a);
    if (a->N == 128) {
        // the walk in segments: the segment passes leave the state entering
        // each later segment in the workspace
        const SegPlan sp = seg_plan(a);
        p.nseg = sp.nseg;
        p.seg_len = sp.seg_len;
        units *= sp.nseg;
        if (sp.nseg > 1) {
            char *ws = static_cast<char *>(a->workspace);
            float *states = reinterpret_cast<float *>(ws + 256);
            float *decay = reinterpret_cast<float *>(ws + 256 + seg_states_bytes(a, sp.nseg));
            p.seg_states = states;
            e = launch_segment_passes(p, a->x_dtype, a->ops == SSD_OPS_BF16, states, decay, err, num_sms(), s);
            if (e != cudaSuccess) return e;
        }
    }
    return launch(a, p, (int)units, err, s);
}

size_t fused_varlen_workspace_size(const ssd_fwd_args *a, int64_t nseq) {
    const int64_t units = nseq * a->G * ((a->H / a->G) / 2);
    return 256 + up256((size_t)(nseq + 1) * 8) + up256((size_t)units * 4);
}

cudaError_t run_fused_varlen(const ssd_fwd_args *a, const int64_t *cu, int nseq, cudaStream_t s) {
    const int pairs = (int)((a->H / a->G) / 2);
    const int units = nseq * (int)a->G * pairs;
    const int grid = units < num_sms() ? units : num_sms();
    // Longest first, dealt to the CTAs in snake order (round r goes forward
    // when r is even, back when odd): walk position i = r * grid + CTA runs the
    // unit sorted at r * grid + (r even ? CTA : m - 1 - CTA), m the round's
    // size.  Every CTA keeps the same number of units and the long ones spread
    // first.
    std::vector<int> nch(units), order(units);
    for (int u = 0; u < units; ++u) {
        const int q = (u / pairs) / (int)a->G;
        nch[u] = (int)((cu[q + 1] - cu[q] + 63) / 64);
        order[u] = u;
    }
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return nch[x] > nch[y]; });
    // workspace: error word | cu [nseq+1] int64 | schedule [units] int32
    const size_t o_cu = 256, o_sched = o_cu + up256((size_t)(nseq + 1) * 8), total = o_sched + (size_t)units * 4;
    std::vector<unsigned char> host(total - o_cu);
    memcpy(host.data(), cu, (size_t)(nseq + 1) * 8);
    int *sched = reinterpret_cast<int *>(host.data() + (o_sched - o_cu));
    for (int i = 0; i < units; ++i) {
        const int round = i / grid, c = i % grid;
        const int base = round * grid, m = std::min(grid, units - base);  // m < grid: the last round
        sched[i] = order[base + ((round & 1) ? m - 1 - c : c)];
    }
    char *ws = static_cast<char *>(a->workspace);
    cudaError_t e = cudaMemsetAsync(ws, 0, 256, s);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyAsync(ws + o_cu, host.data(), host.size(), cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    Params p = fused_params(a);
    p.cu = reinterpret_cast<const long long *>(ws + o_cu);
    p.nseq = nseq;
    p.sched_units = reinterpret_cast<const int *>(ws + o_sched);
    return launch(a, p, units, reinterpret_cast<unsigned int *>(ws), s);
}

}  // namespace ssd
