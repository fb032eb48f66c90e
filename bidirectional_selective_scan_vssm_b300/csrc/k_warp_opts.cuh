// Launchers of the warp-per-channel-group scan (scan_warp.cuh) for one
// combination of the step options (SP: softplus step; CONV: directional
// convolution). Each combination is compiled in its own translation unit
// (k_warp_*.cu) so that the library builds in parallel.
#pragma once

#include "launch.h"

namespace vssm {

template <typename K>
cudaError_t warp_set_smem(K kern, size_t smem)
{
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)   // all of the unified L1/shared array as shared memory: residency is smem-bound
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
    return e;
}

template <typename T, int DIRS, bool SP, bool CONV>
cudaError_t warp_launch_dirs(const WarpScanParams &p, bool carry, long long ctas, long long summ_ctas, cudaStream_t s)
{
    constexpr int G = 1;
    constexpr int W = warps_per_cta(G);
    cudaError_t e;
    if (carry) {
        constexpr int WC = kCarryW;
        const size_t smem = (size_t)WC * WarpLayout<T, 1, false>::kWarpBytes;
        auto sk = warp_carry_kernel<T, DIRS, WC, SP, CONV>;
        if ((e = warp_set_smem(sk, smem)) != cudaSuccess) return e;
        sk<<<(unsigned)summ_ctas, WC * 32, smem, s>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if constexpr (DIRS == 3) {
        if (!carry && p.L <= kOneStageMaxL) {   // short rows: a one-deep copy ring
            const size_t smem1 = (size_t)W * WarpLayout<T, G, true, 1>::kWarpBytes;
            auto k1 = warp_scan_kernel<T, G, DIRS, W, false, SP, CONV, 1>;
            if ((e = warp_set_smem(k1, smem1)) != cudaSuccess) return e;
            k1<<<(unsigned)ctas, W * 32, smem1, s>>>(p);
            return cudaGetLastError();
        }
    }
    const size_t smem = (size_t)W * WarpLayout<T, G, DIRS == 3>::kWarpBytes;
    if constexpr (!(CONV && DIRS == 3)) {
        if (!carry && p.L > kOneStageMaxL && p.ckpt == nullptr) {   // long uncut rows: wider unroll
            auto k4 = warp_scan_kernel<T, G, DIRS, W, false, SP, CONV, kStages, kLongRowUnroll>;
            if ((e = warp_set_smem(k4, smem)) != cudaSuccess) return e;
            k4<<<(unsigned)ctas, W * 32, smem, s>>>(p);
            return cudaGetLastError();
        }
    }
    auto kern = carry ? warp_scan_kernel<T, G, DIRS, W, true, SP, CONV> : warp_scan_kernel<T, G, DIRS, W, false, SP, CONV>;
    if ((e = warp_set_smem(kern, smem)) != cudaSuccess) return e;
    kern<<<(unsigned)ctas, W * 32, smem, s>>>(p);
    return cudaGetLastError();
}

template <bool SP, bool CONV>
cudaError_t launch_warp_opts(const WarpScanParams &p, int dirs, bool f32, bool carry, long long ctas,
                             long long summ_ctas, cudaStream_t s);

#define VSSM_WARP_OPTS_DEFINE(SP, CONV)                                                                      \
    template <>                                                                                              \
    cudaError_t launch_warp_opts<SP, CONV>(const WarpScanParams &p, int dirs, bool f32, bool carry,         \
                                           long long ctas, long long summ_ctas, cudaStream_t s)             \
    {                                                                                                        \
        if (f32) {                                                                                           \
            switch (dirs) {                                                                                  \
            case 1: return warp_launch_dirs<float, 1, SP, CONV>(p, carry, ctas, summ_ctas, s);              \
            case 2: return warp_launch_dirs<float, 2, SP, CONV>(p, carry, ctas, summ_ctas, s);              \
            default: return warp_launch_dirs<float, 3, SP, CONV>(p, carry, ctas, summ_ctas, s);             \
            }                                                                                                \
        }                                                                                                    \
        switch (dirs) {                                                                                      \
        case 1: return warp_launch_dirs<__nv_bfloat16, 1, SP, CONV>(p, carry, ctas, summ_ctas, s);          \
        case 2: return warp_launch_dirs<__nv_bfloat16, 2, SP, CONV>(p, carry, ctas, summ_ctas, s);          \
        default: return warp_launch_dirs<__nv_bfloat16, 3, SP, CONV>(p, carry, ctas, summ_ctas, s);         \
        }                                                                                                    \
    }

}  // namespace vssm
