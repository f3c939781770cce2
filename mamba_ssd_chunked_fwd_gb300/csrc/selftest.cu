// selftest.cu -- ssd_selftest_wait_timeout: runs the library's bounded
// mbarrier wait (tc::mbar_wait, the wait every tensor-core kernel uses for its
// handoffs) on a barrier that nothing arrives on, so that the give-up path
// can be exercised without a hang: the wait returns after the limit, the
// kernel records the timeout in the workspace error word and exits, and
// ssd_check_device_error maps the word to SSD_ERR_TIMEOUT.  No TMA copy,
// tensor-core operation or TMEM allocation is in flight when the wait gives up.
//
// ssd_selftest_fma_rate: a plain fp32 FMA-chain kernel whose CUDA-event time
// gives this GPU's fp32 CUDA-core throughput (the denominator of the
// backward's roofline, which runs on the CUDA cores).
#include "ssd_internal.cuh"
#include "tc_ptx.cuh"

namespace {

// One thread waits on phase 0 of a fresh mbarrier (expected count 1).  With
// `arrive` set it arrives first, so the wait completes at once and the error
// word stays clear (the control case).
__global__ void selftest_wait_kernel(unsigned int *err, uint64_t timeout_ns, int arrive) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = ssd::tc::smem_addr(&bar);
    if (threadIdx.x == 0) {
        ssd::tc::mbar_init(b, 1);
        ssd::tc::mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (arrive) ssd::tc::mbar_arrive(b);
        if (!ssd::tc::mbar_wait(b, 0u, timeout_ns)) atomicOr(err, 1u);
    }
}

constexpr int kFmaThreads = 256;
constexpr int kFmaChains = 8;  // independent chains per thread: enough to cover the FMA latency

// Every thread advances kFmaChains independent chains a <- a*m + c, `iters`
// times each (m < 1 keeps them bounded), then stores their sum so that none
// of the work is dead.  2 * kFmaChains * iters flops per thread.
__global__ void __launch_bounds__(kFmaThreads) selftest_fma_kernel(float *out, int iters, float m, float c) {
    float a[kFmaChains];
#pragma unroll
    for (int k = 0; k < kFmaChains; ++k) a[k] = 1e-3f * static_cast<float>(threadIdx.x) + static_cast<float>(k);
#pragma unroll 8
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int k = 0; k < kFmaChains; ++k) a[k] = fmaf(a[k], m, c);
    }
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < kFmaChains; ++k) sum += a[k];
    out[static_cast<size_t>(blockIdx.x) * kFmaThreads + threadIdx.x] = sum;
}

}  // namespace

extern "C" ssd_status ssd_selftest_fma_rate(float *out, int64_t out_count, int32_t iters, int32_t grid,
                                            void *stream) {
    if (!out) return ssd::report_error(SSD_ERR_INVALID_ARG, "ssd_selftest_fma_rate: out is null");
    if (iters < 8 || iters > (1 << 22) || iters % 8 != 0)
        return ssd::report_error(SSD_ERR_INVALID_ARG, "ssd_selftest_fma_rate: iters must be a multiple of 8 in [8, 2^22]");
    if (grid < 1 || grid > (1 << 16))
        return ssd::report_error(SSD_ERR_INVALID_ARG, "ssd_selftest_fma_rate: grid must be in [1, 65536]");
    if (out_count < static_cast<int64_t>(grid) * kFmaThreads)
        return ssd::report_error(SSD_ERR_INVALID_ARG, "ssd_selftest_fma_rate: out must hold grid * 256 floats");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    selftest_fma_kernel<<<grid, kFmaThreads, 0, s>>>(out, iters, 0.9999f, 1e-4f);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return ssd::report_error(SSD_ERR_CUDA, cudaGetErrorString(e));
    return ssd::report_error(SSD_OK, "");
}

extern "C" ssd_status ssd_selftest_wait_timeout(void *workspace, uint32_t timeout_us, int32_t arrive,
                                                void *stream) {
    if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
        return ssd::report_error(SSD_ERR_INVALID_ARG, "ssd_selftest_wait_timeout: workspace must be 256-byte aligned");
    if (timeout_us < 1 || timeout_us > 1000000)
        return ssd::report_error(SSD_ERR_INVALID_ARG, "ssd_selftest_wait_timeout: timeout_us must be in [1, 1e6]");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int *err = static_cast<unsigned int *>(workspace);
    cudaError_t e = cudaMemsetAsync(err, 0, 256, s);
    if (e == cudaSuccess) {
        selftest_wait_kernel<<<1, 32, 0, s>>>(err, static_cast<uint64_t>(timeout_us) * 1000ull, arrive ? 1 : 0);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return ssd::report_error(SSD_ERR_CUDA, cudaGetErrorString(e));
    return ssd::report_error(SSD_OK, "");
}
