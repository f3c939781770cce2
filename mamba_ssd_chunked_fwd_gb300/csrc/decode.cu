// decode.cu -- one recurrent step of the SSD for a single new token per
// sequence, continuing from a carried state: the "final_state for the decode
// stage" use of the ops-transformer MambaV2 article (section 4.4,
// chunk_state_passing outputs).  For every (b, h), g = h / (H/G):
//
//   d      = clamp(softplus(dt[b,h] + dt_bias[h]))
//   S[p,:] = exp(d A[h]) S[p,:] + d x[b,h,p] B[b,g,:]       (in place, fp32)
//   y[p]   = (S[p,:] . C[b,g,:] + D[h] x[b,h,p]) * silu(z[b,h,p])
//
// All arithmetic is fp32 on the CUDA cores: the step reads and writes the
// [P,N] state once and does 4 flops per state element, so it is bound by HBM.
// One CTA of 128 threads per (b, h).  When N is 4, 8, ..., 128 the state is
// moved as float4: thread t owns float4 number t + 128 k of the [P,N] block
// (so a warp covers whole consecutive rows, 512 contiguous bytes per access),
// issues all its loads before any arithmetic, and a row's dot product with C
// is a shuffle reduction over the N/4 lanes holding that row.  For N = 32, 64,
// 128 a persistent streaming form of the same arithmetic walks half-blocks with
// the next one's loads in flight.  Other N take a scalar kernel (warp per row,
// lane per column).
#include "ssd_internal.cuh"

namespace ssd {

namespace {

constexpr int kDecodeThreads = 128;
constexpr int kMaxNPerLane = 4;  // N <= 128

template <int IO>
__global__ void __launch_bounds__(kDecodeThreads)
decode_step_kernel(DecodeParams p) {
    const int bh = blockIdx.x;
    const int b = bh / p.H, h = bh % p.H;
    const int g = h / (p.H / p.G);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    float u = p.dt[bh];
    if (p.dt_bias) u += __ldg(p.dt_bias + h);
    float d = p.dt_softplus ? softplus_f(u) : u;
    if (p.has_limit) d = fminf(fmaxf(d, p.dt_min), p.dt_max);
    const float a = expf(d * __ldg(p.A + h));
    const float Dh = p.D ? __ldg(p.D + h) : 0.f;

    // this lane's columns of B and C
    float Bv[kMaxNPerLane], Cv[kMaxNPerLane];
    const size_t bc0 = ((size_t)b * p.G + g) * p.N;
#pragma unroll
    for (int j = 0; j < kMaxNPerLane; ++j) {
        const int n = lane + 32 * j;
        Bv[j] = n < p.N ? ld_io<IO>(p.Bm, bc0 + n) : 0.f;
        Cv[j] = n < p.N ? ld_io<IO>(p.Cm, bc0 + n) : 0.f;
    }

    float *S = p.state + (size_t)bh * p.P * p.N;
    const size_t xr0 = (size_t)bh * p.P;
    for (int row = warp; row < p.P; row += kDecodeThreads / 32) {
        const float xv = ld_io<IO>(p.x, xr0 + row);
        const float dx = d * xv;
        float *Sr = S + (size_t)row * p.N;
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < kMaxNPerLane; ++j) {
            const int n = lane + 32 * j;
            if (n < p.N) {
                const float s = fmaf(a, Sr[n], dx * Bv[j]);
                Sr[n] = s;
                acc = fmaf(s, Cv[j], acc);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) {
            float yv = acc;
            if (p.D) yv = fmaf(Dh, xv, yv);
            if (p.z) yv *= silu_f(ld_io<IO>(p.z, xr0 + row));
            st_io<IO>(p.y, xr0 + row, yv);
        }
    }
}

// Vectorised step for N = 4 * LPR, LPR (lanes per row) a power of two <= 32.
template <int IO, int LPR>
__global__ void __launch_bounds__(kDecodeThreads)
decode_step_vec_kernel(DecodeParams p) {
    constexpr int kBatch = 8;  // float4 per thread held at once
    const int bh = blockIdx.x;
    const int b = bh / p.H, h = bh % p.H;
    const int g = h / (p.H / p.G);
    const int t = threadIdx.x;

    float u = p.dt[bh];
    if (p.dt_bias) u += __ldg(p.dt_bias + h);
    float d = p.dt_softplus ? softplus_f(u) : u;
    if (p.has_limit) d = fminf(fmaxf(d, p.dt_min), p.dt_max);
    const float a = expf(d * __ldg(p.A + h));
    const float Dh = p.D ? __ldg(p.D + h) : 0.f;

    // the thread's four columns never change: (t + 128 k) % LPR == t % LPR
    const int c4 = t % LPR;
    const size_t bc0 = ((size_t)b * p.G + g) * p.N + 4 * c4;
    float Bv[4], Cv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        Bv[e] = ld_io<IO>(p.Bm, bc0 + e);
        Cv[e] = ld_io<IO>(p.Cm, bc0 + e);
    }

    float4 *S = reinterpret_cast<float4 *>(p.state + (size_t)bh * p.P * p.N);
    const size_t xr0 = (size_t)bh * p.P;
    const int total4 = p.P * LPR;  // float4 in the [P,N] block
    for (int base = 0; base < total4; base += kDecodeThreads * kBatch) {
        float4 sv[kBatch];
        float xv[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {  // every load first
            const int f = base + t + kDecodeThreads * k;
            if (f < total4) {
                sv[k] = S[f];
                xv[k] = ld_io<IO>(p.x, xr0 + f / LPR);
            }
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int f = base + t + kDecodeThreads * k;
            const bool in = f < total4;  // uniform across a row's LPR lanes
            float acc = 0.f;
            if (in) {
                const float dx = d * xv[k];
                float4 s4 = sv[k];
                s4.x = fmaf(a, s4.x, dx * Bv[0]);
                s4.y = fmaf(a, s4.y, dx * Bv[1]);
                s4.z = fmaf(a, s4.z, dx * Bv[2]);
                s4.w = fmaf(a, s4.w, dx * Bv[3]);
                S[f] = s4;
                acc = s4.x * Cv[0];
                acc = fmaf(s4.y, Cv[1], acc);
                acc = fmaf(s4.z, Cv[2], acc);
                acc = fmaf(s4.w, Cv[3], acc);
            }
#pragma unroll
            for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (in && c4 == 0) {
                const int row = f / LPR;
                float yv = acc;
                if (p.D) yv = fmaf(Dh, xv[k], yv);
                if (p.z) yv *= silu_f(ld_io<IO>(p.z, xr0 + row));
                st_io<IO>(p.y, xr0 + row, yv);
            }
        }
    }
}

// Persistent, streaming version of the float4 step for N = 4 * LPR when a
// (b, h) state block (or half of it) is a whole number of 128-thread float4
// sweeps: a unit is that block or half, the grid is a few CTAs per SM, and each CTA walks
// units with stride gridDim.x, issuing every load of its next unit (state,
// x, B, C, dt) before it computes the current one.  The one-block-per-CTA
// kernel above pays a whole load latency per wave of CTAs; here the loads of
// unit i+1 are in flight while unit i is updated and stored.
constexpr int kStreamCtasPerSm = 6;

template <int IO, int LPR, int K>  // K = float4 per thread per unit
struct DecodeUnit {
    float4 s[K];
    float x[K];
    float B[4], C[4];
    float dt;
};

template <int IO, int LPR, int K, int UPB>  // UPB units per (b, h) block: 1 (whole) or 2 (halves)
__device__ __forceinline__ void decode_unit_load(const DecodeParams &p, int u, int t, DecodeUnit<IO, LPR, K> &v) {
    const int bh = u / UPB, part = u % UPB;
    const int b = bh / p.H, h = bh % p.H, g = h / (p.H / p.G);
    const int c4 = t % LPR;
    const size_t bc0 = ((size_t)b * p.G + g) * p.N + 4 * c4;
    if (IO == IO_F32) {  // 16-byte aligned: N is a multiple of 4 and the tensors are contiguous
        const float4 b4 = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(p.Bm) + bc0));
        const float4 cv = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(p.Cm) + bc0));
        v.B[0] = b4.x; v.B[1] = b4.y; v.B[2] = b4.z; v.B[3] = b4.w;
        v.C[0] = cv.x; v.C[1] = cv.y; v.C[2] = cv.z; v.C[3] = cv.w;
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            v.B[e] = ld_io<IO>(p.Bm, bc0 + e);
            v.C[e] = ld_io<IO>(p.Cm, bc0 + e);
        }
    }
    v.dt = __ldg(p.dt + bh);
    const float4 *S = reinterpret_cast<const float4 *>(p.state + (size_t)bh * p.P * p.N) + part * (K * kDecodeThreads);
    const size_t xr0 = (size_t)bh * p.P + part * (p.P / UPB);
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int f = t + kDecodeThreads * k;
        v.s[k] = S[f];
        v.x[k] = ld_io<IO>(p.x, xr0 + f / LPR);
    }
}

template <int IO, int LPR, int K, int UPB>
__global__ void __launch_bounds__(kDecodeThreads)
decode_step_stream_kernel(DecodeParams p, int n_units) {
    const int t = threadIdx.x;
    const int c4 = t % LPR;
    DecodeUnit<IO, LPR, K> cur, nxt;
    int u = blockIdx.x;
    if (u < n_units) decode_unit_load<IO, LPR, K, UPB>(p, u, t, cur);
    for (; u < n_units; u += gridDim.x) {
        const int un = u + gridDim.x;
        if (un < n_units) decode_unit_load<IO, LPR, K, UPB>(p, un, t, nxt);  // in flight during this unit
        const int bh = u / UPB, part = u % UPB, h = bh % p.H;
        float uu = cur.dt;
        if (p.dt_bias) uu += __ldg(p.dt_bias + h);
        float d = p.dt_softplus ? softplus_f(uu) : uu;
        if (p.has_limit) d = fminf(fmaxf(d, p.dt_min), p.dt_max);
        const float a = expf(d * __ldg(p.A + h));
        const float Dh = p.D ? __ldg(p.D + h) : 0.f;
        float4 *S = reinterpret_cast<float4 *>(p.state + (size_t)bh * p.P * p.N) + part * (K * kDecodeThreads);
        const size_t xr0 = (size_t)bh * p.P + part * (p.P / UPB);
        float prt[K];  // this thread's share of row (t / LPR + (128 / LPR) k)'s dot product with C
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int f = t + kDecodeThreads * k;
            const float dx = d * cur.x[k];
            float4 s4 = cur.s[k];
            s4.x = fmaf(a, s4.x, dx * cur.B[0]);
            s4.y = fmaf(a, s4.y, dx * cur.B[1]);
            s4.z = fmaf(a, s4.z, dx * cur.B[2]);
            s4.w = fmaf(a, s4.w, dx * cur.B[3]);
            S[f] = s4;
            float acc = s4.x * cur.C[0];
            acc = fmaf(s4.y, cur.C[1], acc);
            acc = fmaf(s4.z, cur.C[2], acc);
            prt[k] = fmaf(s4.w, cur.C[3], acc);
        }
        // Sum each row's part over its LPR lanes.  While a thread holds several rows'
        // parts, each shuffle step halves them: the lane keeps the half its lane bit
        // selects and sends the other half to its partner (K rows over LPR lanes in
        // log2(LPR) steps, K - 1 + log2(LPR / K) shuffles instead of K log2(LPR)).
        // Afterwards lane l holds the full sum of its row k(l), where k's bits are the
        // lane bits used to pick halves, highest first.
        int kk = 0;   // the row index this lane keeps
        float sum = 0.f;
        {
            constexpr int kSteps = (K >= 8) ? 3 : (K >= 4) ? 2 : (K >= 2) ? 1 : 0;
            static_assert((1 << kSteps) == K, "K is a power of two up to 8");
            static_assert(K <= LPR, "at most one row per lane after the halving");
            float v[K];
#pragma unroll
            for (int k = 0; k < K; ++k) v[k] = prt[k];
            int off = LPR / 2;
            int width = K;
#pragma unroll
            for (int st = 0; st < kSteps; ++st, off >>= 1) {
                const bool hi = (t & off) != 0;
                width >>= 1;
#pragma unroll
                for (int k = 0; k < (K >> (st + 1)); ++k) {
                    const float keep = hi ? v[k + width] : v[k];
                    const float send = hi ? v[k] : v[k + width];
                    v[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                }
                kk = 2 * kk + (hi ? 1 : 0);
            }
            sum = v[0];
#pragma unroll
            for (; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        }
        // one lane per row writes y: the lanes whose bits below the halving steps are 0
        constexpr int kLowMask = LPR / K - 1;
        if ((c4 & kLowMask) == 0) {
            const int row = t / LPR + (kDecodeThreads / LPR) * kk;
            float yv = sum;
            if (p.D) yv = fmaf(Dh, ld_io<IO>(p.x, xr0 + row), yv);
            if (p.z) yv *= silu_f(ld_io<IO>(p.z, xr0 + row));
            st_io<IO>(p.y, xr0 + row, yv);
        }
        cur = nxt;
    }
}

int g_decode_sms[64] = {};

int decode_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return 1;
    }
    if (g_decode_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) (void)cudaGetLastError();
        g_decode_sms[dev] = n > 0 ? n : 1;
    }
    return g_decode_sms[dev];
}

// The streaming kernel when a unit is K whole sweeps of 128 float4 (K <= 8):
// half a (b, h) block per unit where that works, else the whole block.  Whole
// blocks spread the per-unit work (the step's softplus and exponential, the
// index arithmetic) over twice the state, but at 128 registers only 4 CTAs fit
// on an SM; at the large training state [8,256,64,64] halves measured 11.8 us
// per launch under ncu against 12.6 us, and the same in the timed step.
template <int IO, int LPR>
bool launch_stream(const DecodeParams &p, cudaStream_t s) {
    const int block4 = p.P * LPR;  // float4 in a (b, h) block
    const bool halves = p.P % 2 == 0 && (block4 / 2) % kDecodeThreads == 0 && block4 / 2 / kDecodeThreads <= 8;
    const int upb = halves ? 2 : 1;
    if ((block4 / upb) % kDecodeThreads != 0 || block4 / upb / kDecodeThreads > 8) return false;
    const int K = block4 / upb / kDecodeThreads;
    const int units = upb * p.B * p.H;
    auto run = [&](auto kern) {
        int per_sm = 0;  // resident CTAs per SM (registers decide it), at most kStreamCtasPerSm
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDecodeThreads, 0) != cudaSuccess ||
            per_sm < 1) {
            (void)cudaGetLastError();
            per_sm = 1;
        }
        int grid = decode_sms() * (per_sm < kStreamCtasPerSm ? per_sm : kStreamCtasPerSm);
        if (grid > units) grid = units;
        kern<<<grid, kDecodeThreads, 0, s>>>(p, units);
        return true;
    };
    if (upb == 1) {
        switch (K) {
            case 1: return run(decode_step_stream_kernel<IO, LPR, 1, 1>);
            case 2: return run(decode_step_stream_kernel<IO, LPR, 2, 1>);
            case 4: return run(decode_step_stream_kernel<IO, LPR, 4, 1>);
            case 8: return run(decode_step_stream_kernel<IO, LPR, 8, 1>);
            default: return false;
        }
    }
    switch (K) {
        case 1: return run(decode_step_stream_kernel<IO, LPR, 1, 2>);
        case 2: return run(decode_step_stream_kernel<IO, LPR, 2, 2>);
        case 4: return run(decode_step_stream_kernel<IO, LPR, 4, 2>);
        case 8: return run(decode_step_stream_kernel<IO, LPR, 8, 2>);
        default: return false;
    }
}

template <int IO>
cudaError_t launch_io(const DecodeParams &p, cudaStream_t s) {
    const dim3 grid((unsigned)(p.B * p.H));
    bool done = false;
    switch (p.N) {  // the streaming kernel where its unit fits, else one block per CTA
        case 32: done = launch_stream<IO, 8>(p, s); break;
        case 64: done = launch_stream<IO, 16>(p, s); break;
        case 128: done = launch_stream<IO, 32>(p, s); break;
        default: break;
    }
    if (done) return cudaGetLastError();
    switch (p.N) {
        case 4: decode_step_vec_kernel<IO, 1><<<grid, kDecodeThreads, 0, s>>>(p); break;
        case 8: decode_step_vec_kernel<IO, 2><<<grid, kDecodeThreads, 0, s>>>(p); break;
        case 16: decode_step_vec_kernel<IO, 4><<<grid, kDecodeThreads, 0, s>>>(p); break;
        case 32: decode_step_vec_kernel<IO, 8><<<grid, kDecodeThreads, 0, s>>>(p); break;
        case 64: decode_step_vec_kernel<IO, 16><<<grid, kDecodeThreads, 0, s>>>(p); break;
        case 128: decode_step_vec_kernel<IO, 32><<<grid, kDecodeThreads, 0, s>>>(p); break;
        default: decode_step_kernel<IO><<<grid, kDecodeThreads, 0, s>>>(p); break;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_step(const DecodeParams &p, int io, cudaStream_t s) {
    // the float4 kernels need a 16-byte aligned state; any other takes the scalar kernel
    const bool vec = (reinterpret_cast<uintptr_t>(p.state) % 16) == 0;
    const dim3 grid((unsigned)(p.B * p.H));
    switch (io) {
        case IO_F32:
            if (vec) return launch_io<IO_F32>(p, s);
            decode_step_kernel<IO_F32><<<grid, kDecodeThreads, 0, s>>>(p);
            break;
        case IO_F16:
            if (vec) return launch_io<IO_F16>(p, s);
            decode_step_kernel<IO_F16><<<grid, kDecodeThreads, 0, s>>>(p);
            break;
        case IO_BF16:
            if (vec) return launch_io<IO_BF16>(p, s);
            decode_step_kernel<IO_BF16><<<grid, kDecodeThreads, 0, s>>>(p);
            break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace ssd
