// state_passing.cu -- step 3 of the chunked SSD forward (ops-transformer
// MambaV2 article, section 4.4 "mamba2_chunk_state_passing"): the sequential
// inter-chunk recurrence, per (b,h), vectorised over the P x N state:
//     S_0 = h0 (or 0),   S_{k+1} = exp(cs[k,Q-1]) * S_k + states[k],
// done in place so that states[k] ends up holding S_k, the state ENTERING
// chunk k; S_c goes to final_state.
//
// Each thread owns four consecutive state elements (one float4) and walks
// the chunks in order; the next chunk's float4 is loaded before the current
// one is stored, so loads stay one step ahead of the dependent FMA chain.
// Grid: x = batch*head, y = state slices of 1024 elements.
#include "ssd_internal.cuh"

namespace ssd {

namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
state_passing_kernel(Params p, const float *__restrict__ cs, float *__restrict__ states) {
    const int bh = blockIdx.x;
    const int b = bh / p.H, h = bh % p.H;
    const int PN = p.P * p.N;
    const int e = (blockIdx.y * kThreads + threadIdx.x) * 4;
    if (e >= PN) return;
    const int c = p.nchunks;
    const size_t crow = ((size_t)b * p.H + h) * c;
    const size_t kstride = (size_t)p.H * PN;  // distance between chunks in states
    float *base = states + (((size_t)b * c) * p.H + h) * PN + e;

    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    if (p.h0) s = __ldg(reinterpret_cast<const float4 *>(p.h0 + ((size_t)b * p.H + h) * PN + e));
    float4 nxt = *reinterpret_cast<const float4 *>(base);
    for (int k = 0; k < c; ++k) {
        const float4 loc = nxt;
        if (k + 1 < c) nxt = *reinterpret_cast<const float4 *>(base + (size_t)(k + 1) * kstride);
        *reinterpret_cast<float4 *>(base + (size_t)k * kstride) = s;
        const float a = expf(__ldg(cs + (crow + k) * p.Q + p.Q - 1));
        s.x = fmaf(a, s.x, loc.x);
        s.y = fmaf(a, s.y, loc.y);
        s.z = fmaf(a, s.z, loc.z);
        s.w = fmaf(a, s.w, loc.w);
    }
    if (p.final_state)
        *reinterpret_cast<float4 *>(p.final_state + ((size_t)b * p.H + h) * PN + e) = s;
}

}  // namespace

cudaError_t launch_state_passing(const Params &p, const float *cs, float *states, cudaStream_t s) {
    const int PN = p.P * p.N;
    if (PN % 4) return cudaErrorInvalidValue;
    dim3 grid(p.B * p.H, (PN / 4 + kThreads - 1) / kThreads);
    state_passing_kernel<<<grid, kThreads, 0, s>>>(p, cs, states);
    return cudaGetLastError();
}

}  // namespace ssd
