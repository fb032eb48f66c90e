// Launchers of the general scan (scan_kernel.cuh, dstate 1..15).
#include "launch.h"

namespace vssm {

namespace {

constexpr int kBidirR = 32, kBidirG = 2;     // 128 threads: 64 forward, 64 backward
constexpr int kOneDirR = 64, kOneDirG = 2;   // 128 threads

template <typename T, int DIRS, int R, int G, bool YSMEM>
cudaError_t launch_variant(const ScanParams &p, long long ctas, cudaStream_t s)
{
    constexpr int NDIR = DIRS == 3 ? 2 : 1;
    const size_t smem = sizeof(float) * ((size_t)NDIR * DirBlock<R>::kFloats + (YSMEM ? (size_t)R * p.ypitch : 0));
    auto kern = scan_kernel<T, DIRS, R, G, YSMEM>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)ctas, NDIR * R * G, smem, s>>>(p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const ScanParams &p, int dirs, bool ysmem, long long ctas, cudaStream_t s)
{
    switch (dirs) {
    case 1: return launch_variant<T, 1, kOneDirR, kOneDirG, false>(p, ctas, s);
    case 2: return launch_variant<T, 2, kOneDirR, kOneDirG, false>(p, ctas, s);
    default:
        return ysmem ? launch_variant<T, 3, kBidirR, kBidirG, true>(p, ctas, s)
                     : launch_variant<T, 3, kBidirR, kBidirG, false>(p, ctas, s);
    }
}

}  // namespace

cudaError_t launch_general(const ScanParams &p, int dirs, bool ysmem, bool f32, long long ctas, cudaStream_t s)
{
    return f32 ? launch_typed<float>(p, dirs, ysmem, ctas, s) : launch_typed<__nv_bfloat16>(p, dirs, ysmem, ctas, s);
}

}  // namespace vssm
