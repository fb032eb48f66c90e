// Launchers of the gradient kernels (scan_grad.cuh, grad_ext.cuh).
#include <algorithm>

#include "grad_ext.cuh"
#include "launch.h"

namespace vssm {

namespace {

// Test of the bounded-wait path: one warp waits on a pair barrier whose
// second arrival never comes, gives up after limit_ns and records a timeout
// in the device error word as the kernels with bounded waits do.
__global__ void selftest_wait_kernel(unsigned *err, uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 2);
        fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) mbar_arrive(&bar);
    const bool met = mbar_wait(&bar, 0, limit_ns);
    if (!__all_sync(0xffffffffu, met) && threadIdx.x == 0) atomicOr(err, kErrTimeout);
}

__global__ void zero_f32_kernel(float *p, long long n)
{
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x)
        p[i] = 0.f;
}


template <typename T, int DIRS>
cudaError_t launch_dirs(const GradParams &p, long long ngroups, int nrange, bool have_ckpt, cudaStream_t s)
{
    constexpr int NDIR = DIRS == 3 ? 2 : 1;
    const long long units = (long long)NDIR * ngroups;
    cudaError_t e = cudaSuccess;
    if (!have_ckpt) {     // (else the training forward stored them)
        const long long walks = units * (p.summ ? 1 : nrange);   // independent ranges walk apart
        const size_t csmem = 4 * SummLayout<T>::kWarpBytes;
        auto ckern = grad_ckpt_kernel<T, DIRS>;
        if ((e = cudaFuncSetAttribute(ckern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)csmem)) != cudaSuccess)
            return e;
        ckern<<<(unsigned)((walks + 3) / 4), 128, csmem, s>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (nrange > 1 && p.summ) {     // (ranges at folded segment starts need no summaries)
        const long long su = units * nrange;
        const size_t ssmem = 4 * SummLayout<T>::kWarpBytes;
        auto skern = grad_adj_summary_kernel<T, DIRS>;
        if ((e = cudaFuncSetAttribute(skern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssmem)) != cudaSuccess)
            return e;
        skern<<<(unsigned)((su + 3) / 4), 128, ssmem, s>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const size_t smem = (size_t)NDIR * GradLayout<T, DIRS>::kWarpBytes;
    auto kern = grad_adjoint_kernel<T, DIRS>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
    kern<<<(unsigned)(ngroups * nrange), NDIR * 32, smem, s>>>(p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const GradParams &p, int dirs, long long ngroups, int nrange, bool have_ckpt,
                         cudaStream_t s)
{
    switch (dirs) {
    case 1: return launch_dirs<T, 1>(p, ngroups, nrange, have_ckpt, s);
    case 2: return launch_dirs<T, 2>(p, ngroups, nrange, have_ckpt, s);
    default: return launch_dirs<T, 3>(p, ngroups, nrange, have_ckpt, s);
    }
}

}  // namespace

cudaError_t launch_grad(const GradParams &p, int dirs, bool f32, long long ngroups, int nrange, bool have_ckpt,
                        cudaStream_t s)
{
    return f32 ? launch_typed<float>(p, dirs, ngroups, nrange, have_ckpt, s)
               : launch_typed<__nv_bfloat16>(p, dirs, ngroups, nrange, have_ckpt, s);
}

cudaError_t launch_zero_f32(float *p, size_t n, cudaStream_t s)
{
    if (!p || n == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)std::min<size_t>((n + 255) / 256, (size_t)sm_count() * 8);
    zero_f32_kernel<<<blocks, 256, 0, s>>>(p, (long long)n);
    return cudaGetLastError();
}

unsigned stride_blocks(long long n)
{
    return (unsigned)std::min<long long>((n + 255) / 256, 16LL * sm_count());
}

// One block per (row, tile of 256 TPT tokens); 4 tokens per thread on rows of
// 1024 tokens or more; the tap count and whether rows are folded as template
// parameters.
template <template <typename, int, int, bool> class KL, typename T, int TPT>
void ext_launch_k(unsigned blocks, const GradExtParams &p, cudaStream_t s)
{
    const bool fold = p.seg_len > 0;
    switch (p.K) {
    case 0: KL<T, TPT, 0, false>::run(blocks, p, s); break;
    case 1: fold ? KL<T, TPT, 1, true>::run(blocks, p, s) : KL<T, TPT, 1, false>::run(blocks, p, s); break;
    case 2: fold ? KL<T, TPT, 2, true>::run(blocks, p, s) : KL<T, TPT, 2, false>::run(blocks, p, s); break;
    case 3: fold ? KL<T, TPT, 3, true>::run(blocks, p, s) : KL<T, TPT, 3, false>::run(blocks, p, s); break;
    default: fold ? KL<T, TPT, 4, true>::run(blocks, p, s) : KL<T, TPT, 4, false>::run(blocks, p, s); break;
    }
}

template <template <typename, int, int, bool> class KL>
void ext_launch(const GradExtParams &p, bool f32, cudaStream_t s)
{
    const long long rows = (long long)p.batch * p.dim;
    if (p.L >= kExtThreads * kExtLongTPT) {
        constexpr int tile = kExtThreads * kExtLongTPT;
        const unsigned blocks = (unsigned)(rows * ((p.L + tile - 1) / tile));
        if (f32) ext_launch_k<KL, float, kExtLongTPT>(blocks, p, s);
        else ext_launch_k<KL, __nv_bfloat16, kExtLongTPT>(blocks, p, s);
    } else {
        const unsigned blocks = (unsigned)(rows * ((p.L + kExtThreads - 1) / kExtThreads));
        if (f32) ext_launch_k<KL, float, 1>(blocks, p, s);
        else ext_launch_k<KL, __nv_bfloat16, 1>(blocks, p, s);
    }
}

template <typename T, int TPT, int K, bool FOLD>
struct PrepLaunch {
    static void run(unsigned blocks, const GradExtParams &p, cudaStream_t s)
    {
        grad_prep_kernel<T, TPT, K, FOLD><<<blocks, kExtThreads, 0, s>>>(p);
    }
};

template <typename T, int TPT, int K, bool FOLD>
struct PostLaunch {
    static void run(unsigned blocks, const GradExtParams &p, cudaStream_t s)
    {
        grad_post_kernel<T, TPT, K, FOLD><<<blocks, kExtThreads, 0, s>>>(p);
    }
};

cudaError_t launch_grad_ext_prep(const GradExtParams &p, bool f32, cudaStream_t s)
{
    if ((long long)p.batch * p.dim * p.L == 0) return cudaSuccess;
    ext_launch<PrepLaunch>(p, f32, s);
    return cudaGetLastError();
}

cudaError_t launch_widen_bf16(const void *src, float *dst, long long n, cudaStream_t s)
{
    if (n == 0) return cudaSuccess;
    widen_f32_kernel<__nv_bfloat16><<<stride_blocks(n), 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(src), dst, n);
    return cudaGetLastError();
}

cudaError_t launch_grad_ext_post(const GradExtParams &p, bool f32, cudaStream_t s)
{
    if ((long long)p.batch * p.dim * p.L == 0) return cudaSuccess;
    ext_launch<PostLaunch>(p, f32, s);
    return cudaGetLastError();
}

cudaError_t launch_selftest_wait(unsigned *err, uint64_t limit_ns, cudaStream_t s)
{
    selftest_wait_kernel<<<1, 32, 0, s>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace vssm
