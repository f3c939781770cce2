// ssd_internal.cuh -- shared device helpers and the kernel parameter block
// of the GB300 SSD forward.  Not part of the public ABI (see include/ssd.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ssd.h"

namespace ssd {

// Everything a kernel needs to know about one call, in device-friendly form.
struct Params {
    int B, L, H, P, N, G, Q, nchunks, hpg;  // hpg = heads per group = H / G
    const void *x;
    const float *dt;
    const float *A;
    const void *Bm;
    const void *Cm;
    const float *D;
    const void *z;
    const float *dt_bias;
    const float *h0;
    void *y;
    float *final_state;
    int dt_softplus;
    int has_limit;
    float dt_min, dt_max;
    // packed variable-length sequences (fused plan): B == 1 and sequence s
    // holds tokens [cu[s], cu[s+1]); states are indexed by s.  NULL otherwise.
    const long long *cu = nullptr;
    int nseq = 0;
    // packed sequences: the unit at walk position i (CTA i % grid, its
    // (i / grid)-th unit), from the host's schedule
    const int *sched_units = nullptr;
    // gated RMSNorm of the output (fused plan), NULL otherwise
    const float *norm_w = nullptr;
    float norm_eps = 0.f;
    // fused plan at N = 128: each sequence is cut into nseg segments of
    // seg_len tokens (a multiple of 64) walked in parallel; seg_states
    // [B, nseg, H, P, N] holds the state entering segment s >= 1
    int seg_len = 0, nseg = 1;
    const float *seg_states = nullptr;
    // causal conv1d + SiLU of the staged x, B, C tiles (fused plan, N = 64):
    // weights [channels, conv_w], biases [channels] or NULL; conv_w = 0: none
    const float *conv_wx = nullptr, *conv_bx = nullptr;
    const float *conv_wb = nullptr, *conv_bb = nullptr;
    const float *conv_wc = nullptr, *conv_bc = nullptr;
    int conv_w = 0;
};

enum IoType { IO_F32 = SSD_F32, IO_F16 = SSD_F16, IO_BF16 = SSD_BF16 };

template <int IO> struct IoTraits;
template <> struct IoTraits<IO_F32> {
    using T = float;
    static __device__ __forceinline__ float to_f(T v) { return v; }
    static __device__ __forceinline__ T from_f(float v) { return v; }
};
template <> struct IoTraits<IO_F16> {
    using T = __half;
    static __device__ __forceinline__ float to_f(T v) { return __half2float(v); }
    static __device__ __forceinline__ T from_f(float v) { return __float2half_rn(v); }
};
template <> struct IoTraits<IO_BF16> {
    using T = __nv_bfloat16;
    static __device__ __forceinline__ float to_f(T v) { return __bfloat162float(v); }
    static __device__ __forceinline__ T from_f(float v) { return __float2bfloat16_rn(v); }
};

template <int IO>
__device__ __forceinline__ float ld_io(const void *base, size_t i) {
    using T = typename IoTraits<IO>::T;
    return IoTraits<IO>::to_f(__ldg(reinterpret_cast<const T *>(base) + i));
}
template <>
__device__ __forceinline__ float ld_io<IO_F16>(const void *base, size_t i) {
    return __half2float(reinterpret_cast<const __half *>(base)[i]);
}
template <>
__device__ __forceinline__ float ld_io<IO_BF16>(const void *base, size_t i) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(base)[i]);
}

template <int IO>
__device__ __forceinline__ void st_io(void *base, size_t i, float v) {
    using T = typename IoTraits<IO>::T;
    reinterpret_cast<T *>(base)[i] = IoTraits<IO>::from_f(v);
}

// softplus(u) = log(1 + e^u).  Above 20 it equals u to within 2e-9 relative,
// far below fp32 resolution, so u is returned there.
__device__ __forceinline__ float softplus_f(float u) {
    return u > 20.f ? u : log1pf(expf(u));
}

// Processed step d_t: add the bias, then softplus, then clamp ("Preprocess:
// softplus / clamp / decay", README "AscendC execution path").
__device__ __forceinline__ float dt_processed(const Params &p, float raw, int h) {
    float u = raw;
    if (p.dt_bias) u += __ldg(p.dt_bias + h);
    float d = p.dt_softplus ? softplus_f(u) : u;
    if (p.has_limit) d = fminf(fmaxf(d, p.dt_min), p.dt_max);
    return d;
}

__device__ __forceinline__ float silu_f(float v) { return v / (1.f + expf(-v)); }
// The same with the fast exponential and division intrinsics (a few ulp),
// for kernels whose operands are already fp16 / bf16 (the fused kernel).
// For v < -87 the denominator is +inf and the quotient 0, the function's limit.
__device__ __forceinline__ float silu_fast(float v) { return __fdividef(v, 1.f + __expf(-v)); }
// SiLU through the hardware tanh: v sigmoid(v) = h + h tanh(h) with h = v / 2
// (sigmoid(v) = (1 + tanh(v / 2)) / 2).  PTX tanh.approx.f32 has a relative
// error of about 2^-11, so this is for values rounded to a 16-bit type next
// (the convolved operands of the fused kernel, 16-bit conv1d outputs): one
// MUFU operation instead of two.
__device__ __forceinline__ float silu_tanh(float v) {
    const float h = 0.5f * v;
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
    return fmaf(h, t, h);
}

// One decode step (decode.cu): the shape of ssd_decode_args in device form.
struct DecodeParams {
    int B, H, P, N, G;
    const void *x;
    const float *dt;
    const float *A;
    const void *Bm;
    const void *Cm;
    const float *D;
    const void *z;
    const float *dt_bias;
    float *state;
    void *y;
    int dt_softplus;
    int has_limit;
    float dt_min, dt_max;
};
cudaError_t launch_decode_step(const DecodeParams &p, int io, cudaStream_t s);

// The backward (bwd.cu): buffers of one call (device pointers).
struct BwdBuffers {
    const float *dtp, *cs;      // [B,H,c,Q] from the forward's chunk_cumsum
    const float *states;        // [B,c,H,P,N] states entering each chunk
    float *adj;                 // [B,c,H,P,N] scratch: adjoint at each chunk's end
    const void *dy;             // [B,L,H,P] public dtype
    const void *ypre;           // [B,L,H,P] y before the gate (only with z)
    float *dyp;                 // [B,L,H,P] scratch: dy after the gate
    const float *dfinal;        // [B,H,P,N] or NULL
    void *dx, *dz, *dB, *dC;    // outputs in the public dtype (dz only with z)
    float *ddt, *dA, *dD, *dbias, *dh0;  // outputs (dD, dbias, dh0 may be NULL)
    float *dBh, *dCh;           // [B,L,H,N] scratch: per-head dB, dC
    float *partA, *partD, *partBias;     // [B,c,H] scratch
};
size_t bwd_chunk_smem_bytes();
cudaError_t launch_bwd(const Params &p, int io, const BwdBuffers &w, cudaStream_t s);

// The SSD's neighbours (neighbors.cu).
cudaError_t launch_causal_conv1d(int B, int D, int S, int W, int io, const void *x, const float *w,
                                 const float *bias, int silu, void *out, cudaStream_t s);
cudaError_t launch_conv_tokens(int B, int S, int C, int W, int io, const void *x, const float *w, const float *bias,
                               int silu, void *out, cudaStream_t s);
cudaError_t launch_gated_rmsnorm(long long rows, int D, int groups, float eps, int io, const void *x, const void *z,
                                 const float *w, void *out, cudaStream_t s);

// The sequence-parallel exchange (seqpar.cu).
cudaError_t launch_segment_log_decay(const Params &p, float *out, cudaStream_t s);
cudaError_t launch_state_fold(int nseg, long long bh_count, int pn, const float *log_decay, const float *states,
                              float *out, cudaStream_t s);

// Launchers of the chunked plan (CUDA-core fp32 kernels).
cudaError_t launch_chunk_cumsum(const Params &p, float *dtp, float *cs, cudaStream_t s);
cudaError_t launch_chunk_state(const Params &p, int io, const float *dtp, const float *cs,
                               float *states, cudaStream_t s);
cudaError_t launch_state_passing(const Params &p, const float *cs, float *states,
                                 cudaStream_t s);
cudaError_t launch_chunk_scan(const Params &p, int io, const float *dtp, const float *cs,
                              const float *states, cudaStream_t s);

// Tensor-core (tcgen05) versions of steps 2 and 4 for fp16 / bf16 operands.
// `err` (may be NULL) receives bit 2 if a bounded wait gave up.
bool chunk_tc_state_supported(const Params &p, int ops);
bool chunk_tc_scan_supported(const Params &p, int ops);
cudaError_t launch_chunk_state_tc(const Params &p, int io, int ops, const float *dtp, const float *cs,
                                  float *states, unsigned int *err, cudaStream_t s);
cudaError_t launch_chunk_scan_tc(const Params &p, int io, int ops, const float *dtp, const float *cs,
                                 const float *states, unsigned int *err, cudaStream_t s);

// Record `msg` as this thread's ssd_last_error_detail() and return `st`.
ssd_status report_error(ssd_status st, const char *msg);

}  // namespace ssd
