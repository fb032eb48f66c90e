// Helpers shared by the kernels: element loads and stores in the I/O type,
// the silu gate, and the constants of the bounded waits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"

namespace vssm {

constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s: limit of every device-side wait
constexpr unsigned kErrTimeout = 1u;                // device error word: a wait expired

__device__ __forceinline__ float ld_as_f32(const float *p) { return *p; }
__device__ __forceinline__ float ld_as_f32(const __nv_bfloat16 *p)
{
    return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const unsigned short *>(p)) << 16);
}
__device__ __forceinline__ void st_from_f32(float *p, float v) { *p = v; }
__device__ __forceinline__ void st_from_f32(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

// 16 consecutive elements from shared memory to fp32 (16-byte aligned source).
__device__ __forceinline__ void load16_f32(const float *src, float *dst)
{
    const float4 *s = reinterpret_cast<const float4 *>(src);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 v = s[q];
        dst[4 * q + 0] = v.x;
        dst[4 * q + 1] = v.y;
        dst[4 * q + 2] = v.z;
        dst[4 * q + 3] = v.w;
    }
}
__device__ __forceinline__ void load16_f32(const __nv_bfloat16 *src, float *dst)
{
    const uint4 *s = reinterpret_cast<const uint4 *>(src);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const uint4 v = s[q];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            dst[8 * q + 2 * k + 0] = __uint_as_float(w[k] << 16);
            dst[8 * q + 2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        }
    }
}

// silu(z) = z * sigmoid(z). For fp32 outputs: z / (1 + 2^(-z*log2e)). For
// 16-bit outputs the identity z*sigmoid(z) = h + h*tanh(h), h = z/2, needs one
// MUFU operation instead of two; tanh.approx's error (about 2^-11 relative)
// stays below the output's own rounding (2^-9).
template <typename T>
__device__ __forceinline__ float silu_f32(float z)
{
    if (sizeof(T) == 2) {
        const float hz = 0.5f * z;
        return fmaf(hz, tanh_mufu(hz), hz);
    }
    return __fdividef(z, 1.0f + ex2_mufu(-1.4426950408889634f * z));
}

}  // namespace vssm
