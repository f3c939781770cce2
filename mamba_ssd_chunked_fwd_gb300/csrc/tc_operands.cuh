// tc_operands.cuh -- writing 16-bit MMA operands into shared memory, shared
// by the tensor-core kernels (fused plan and chunked plan).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "ssd_internal.cuh"
#include "tc_ptx.cuh"

namespace ssd {
namespace tcop {

// 2^x on the MUFU unit (PTX ex2.approx, relative error ~2^-22, flushes below
// 2^-126 to 0): used where the result is rounded to a 16-bit operand.
__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool bf16) {
    if (bf16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&v);
    }
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// 16-byte shared store of an MMA operand.  No "memory" clobber: operand
// memory is only read by the tensor core, and the fences / barriers that
// publish it carry the ordering.
__device__ __forceinline__ void st_shared_v4(uint32_t saddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(a), "r"(b), "r"(c), "r"(d));
}

// 8 floats rounded to one 16-byte row of an operand block.
__device__ __forceinline__ void store8(uint32_t saddr, const float (&v)[8], bool bf16) {
    st_shared_v4(saddr, pack2(v[0], v[1], bf16), pack2(v[2], v[3], bf16), pack2(v[4], v[5], bf16),
                 pack2(v[6], v[7], bf16));
}

// 8 consecutive elements of a public tensor as floats (zeros when !valid).
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
            float2 f;
            if (IO == IO_BF16) f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
            else f = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
            v[2 * i] = f.x; v[2 * i + 1] = f.y;
        }
    }
}

}  // namespace tcop
}  // namespace ssd
