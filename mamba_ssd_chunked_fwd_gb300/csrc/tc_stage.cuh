// tc_stage.cuh -- reading the TMA staging tiles of the tensor-core kernels
// (the fused plan and the segment pre-pass): boxes of 64 token rows x 128
// bytes, written by TMA with the 128-byte swizzle (16-byte chunk index XOR
// row % 8), so that reading one column of chunks touches distinct banks.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "ssd_internal.cuh"
#include "tc_ptx.cuh"

namespace ssd {
namespace tcstage {

constexpr uint32_t BOX_BYTES = 8192;  // 64 token rows x 128 bytes

// 16-byte chunk c of row r in a 128-byte-swizzled TMA box (chunk index XOR row % 8)
__device__ __forceinline__ uint32_t swz(uint32_t box, int r, int c) {
    return box + r * 128 + ((c ^ (r & 7)) << 4);
}

__device__ __forceinline__ void unpack8(uint4 u, bool bf16, float (&v)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f;
        if (bf16) f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
        else f = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
        v[2 * i] = f.x; v[2 * i + 1] = f.y;
    }
}

// 8 consecutive features [8c8, 8c8+8) of token row r from a staged tile whose
// rows are split over consecutive boxes of 128 bytes (32 fp32 or 64 16-bit
// features per box).
template <int IO>
__device__ __forceinline__ void stage_read8(uint32_t base, int r, int c8, float (&v)[8]) {
    if (IO == IO_F32) {  // 32 features per box, 8 floats = 2 chunks
        const uint32_t box = base + (c8 >> 2) * BOX_BYTES;
        const int c = 2 * (c8 & 3);
        const uint4 a = tc::ld_shared_v4(swz(box, r, c)), b = tc::ld_shared_v4(swz(box, r, c + 1));
        v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y); v[2] = __uint_as_float(a.z);
        v[3] = __uint_as_float(a.w); v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y);
        v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
    } else {  // 64 features per box, 8 values = 1 chunk
        const uint32_t box = base + (c8 >> 3) * BOX_BYTES;
        unpack8(tc::ld_shared_v4(swz(box, r, c8 & 7)), IO == IO_BF16, v);
    }
}

// The 16-byte chunk of 8 consecutive 16-bit features [8c8, 8c8+8) of token row
// r, as stored (64 features per box).
__device__ __forceinline__ uint4 stage_raw16(uint32_t base, int r, int c8) {
    return tc::ld_shared_v4(swz(base + (c8 >> 3) * BOX_BYTES, r, c8 & 7));
}

}  // namespace tcstage
}  // namespace ssd
