// seqpar.cu -- the two kernels of the sequence-parallel exchange.  A
// sequence split into consecutive token segments has, per (b, h), the affine
// state map of each segment, S_out = exp(a) S_in + S_seg (a = the segment's
// total d*A, S_seg = its final state from a zero start): the same composition
// rule the chunk_state_passing step applies between chunks (ops-transformer
// MambaV2 article, section 4.4), applied between segments held by different
// ranks.
//
//   segment_log_decay: a[b,h] = sum_t d_t A[h] over the segment's L tokens,
//                      accumulated in fp64 in token order (deterministic).
//   state_fold:        S = 0; for q in 0..nseg-1: S = exp(a[q]) S + S_q,
//                      the state entering the segment after the nseg given.
#include "ssd_internal.cuh"

namespace ssd {

namespace {

__global__ void segment_log_decay_kernel(Params p, float *out) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;  // (b, h)
    if (i >= p.B * p.H) return;
    const int b = i / p.H, h = i % p.H;
    const float A = __ldg(p.A + h);
    const float *dt = p.dt + (size_t)b * p.L * p.H + h;
    double acc = 0.0;
    for (int t = 0; t < p.L; ++t) acc += (double)(dt_processed(p, __ldg(dt + (size_t)t * p.H), h) * A);
    out[i] = (float)acc;
}

__global__ void state_fold_kernel(int nseg, long long bh_count, int pn, const float *log_decay,
                                  const float *states, float *out) {
    const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // element of [B,H,P,N]
    const long long total = bh_count * pn;
    if (e >= total) return;
    const long long bh = e / pn;
    float s = 0.f;
    for (int q = 0; q < nseg; ++q)
        s = fmaf(expf(__ldg(log_decay + (long long)q * bh_count + bh)), s, __ldg(states + (long long)q * total + e));
    out[e] = s;
}

}  // namespace

cudaError_t launch_segment_log_decay(const Params &p, float *out, cudaStream_t s) {
    const int n = p.B * p.H;
    segment_log_decay_kernel<<<(n + 127) / 128, 128, 0, s>>>(p, out);
    return cudaGetLastError();
}

cudaError_t launch_state_fold(int nseg, long long bh_count, int pn, const float *log_decay, const float *states,
                              float *out, cudaStream_t s) {
    const long long total = bh_count * pn;
    const long long blocks = (total + 255) / 256;
    state_fold_kernel<<<(unsigned)blocks, 256, 0, s>>>(nseg, bh_count, pn, log_decay, states, out);
    return cudaGetLastError();
}

}  // namespace ssd
