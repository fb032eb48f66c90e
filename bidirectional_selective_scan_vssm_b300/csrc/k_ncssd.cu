// Launchers of the NC-SSD kernels (ncssd.cuh).
#include "launch.h"

namespace vssm {

namespace {

template <typename T, int Q, bool GATE, bool SKIP>
void launch_k(const NcssdParams &p, dim3 grid, cudaStream_t s)
{
    const dim3 block(kNcW * 32);
    if (sizeof(T) == 2) ncssd_mma_kernel<Q, GATE, SKIP><<<grid, block, 0, s>>>(p);
    else ncssd_kernel<float, Q, GATE, SKIP><<<grid, block, 0, s>>>(p);
}

template <typename T, int Q>
void launch_q(const NcssdParams &p, bool gate, bool skip, dim3 grid, cudaStream_t s)
{
    if (gate && skip) launch_k<T, Q, true, true>(p, grid, s);
    else if (gate) launch_k<T, Q, true, false>(p, grid, s);
    else if (skip) launch_k<T, Q, false, true>(p, grid, s);
    else launch_k<T, Q, false, false>(p, grid, s);
}

template <typename T>
void launch_tiled(const NcssdParams &p, int q, bool gate, bool skip, dim3 grid, cudaStream_t s)
{
    switch (q) {
    case 1: launch_q<T, 1>(p, gate, skip, grid, s); break;
    case 2: launch_q<T, 2>(p, gate, skip, grid, s); break;
    case 4: launch_q<T, 4>(p, gate, skip, grid, s); break;
    default: launch_q<T, 8>(p, gate, skip, grid, s); break;
    }
}

template <bool GATE, bool SKIP>
cudaError_t launch_rows(const NcssdParams &p, dim3 grid, cudaStream_t s)
{
    const NcRowsLayout lay(p.L, GATE);
    auto kern = ncssd_rows_kernel<GATE, SKIP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, lay.total);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    kern<<<grid, kNcW * 32, lay.total, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ncssd(const NcssdParams &p, bool rows, int q, bool gate, bool skip, bool f32, dim3 grid,
                         cudaStream_t s)
{
    if (rows)
        return gate ? (skip ? launch_rows<true, true>(p, grid, s) : launch_rows<true, false>(p, grid, s))
                    : (skip ? launch_rows<false, true>(p, grid, s) : launch_rows<false, false>(p, grid, s));
    if (f32) launch_tiled<float>(p, q, gate, skip, grid, s);
    else launch_tiled<__nv_bfloat16>(p, q, gate, skip, grid, s);
    return cudaGetLastError();
}

}  // namespace vssm
