// noalloc.cu -- ssd_fwd_noalloc: the SSD forward for callers that cannot
// allocate device memory themselves.
//
// ssd_fwd needs a scratch workspace (the chunked plan keeps the processed
// steps, the cumulative decays and every chunk state there; the fused plan
// keeps its error word there), and it leaves allocating that workspace to the
// caller.  Some callers have no allocator at hand: code running under an
// allocator they do not own, plugins that may not call cudaMalloc, or
// real-time paths where an allocation could stall.  This entry point takes
// the scratch from a fixed buffer compiled into the library instead, so the
// caller only passes inputs and outputs.
//
// The buffer is a file-scope __device__ array of kScratchBytes; every GPU
// that loads the library holds it until the process exits.  Host code may not
// use the array's name as a pointer (on the host it is only a stand-in), so
// the device address is looked up with cudaGetSymbolAddress, once per device,
// on the first call made while that device is current.
#include <mutex>
#include <stdio.h>

#include "ssd_internal.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;  // 64 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once per device).
cudaError_t scratch_address(int dev, void **out) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" ssd_status ssd_fwd_noalloc(const ssd_fwd_args *args, void *stream) {
    size_t need = 0;
    ssd_status st = ssd_fwd_workspace_size(args, &need);
    if (st != SSD_OK) return st;
    if (need > kScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "ssd_fwd_noalloc: this call needs %zu bytes of scratch, the built-in buffer holds %zu; "
                 "use ssd_fwd with a caller-owned workspace",
                 need, kScratchBytes);
        return ssd::report_error(SSD_ERR_WORKSPACE, msg);
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return ssd::report_error(SSD_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return ssd::report_error(SSD_ERR_UNSUPPORTED, "ssd_fwd_noalloc: device index out of range");
    void *scratch = nullptr;
    if ((e = scratch_address(dev, &scratch)) != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof(msg), "ssd_fwd_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
        return ssd::report_error(SSD_ERR_CUDA, msg);
    }
    ssd_fwd_args a = *args;
    a.workspace = scratch;
    a.workspace_bytes = kScratchBytes;
    return ssd_fwd(&a, stream);
}
