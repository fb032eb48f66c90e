// Launchers of the kernel families, one translation unit each, called by the
// C ABI layer (vssm_api.cu). Each returns the CUDA error of its launches.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "grad_ext.cuh"
#include "ncssd.cuh"
#include "scan_grad.cuh"
#include "scan_kernel.cuh"
#include "scan_warp.cuh"

namespace vssm {

// Warp-per-channel-group scan (dstate 16): dirs 1, 2 or 3; carry: a summary
// pass (summ_ctas CTAs) runs first; sp / conv: the step options.
cudaError_t launch_warp(const WarpScanParams &p, int dirs, bool f32, bool carry, bool sp, bool conv,
                        long long ctas, long long summ_ctas, cudaStream_t s);

// Warps per CTA of the scan kernel and of the summary kernel.
constexpr int warps_per_cta(int G) { return G == 4 ? 8 : (G == 2 ? 4 : 2); }
#ifndef VSSM_CARRY_WARPS
#define VSSM_CARRY_WARPS 1
#endif
constexpr int kCarryW = VSSM_CARRY_WARPS;

// General scan (dstate 1..15): dirs 1, 2 or 3; ysmem: shared y-buffer.
cudaError_t launch_general(const ScanParams &p, int dirs, bool ysmem, bool f32, long long ctas,
                           cudaStream_t s);

// Gradient: checkpoints (unless have_ckpt: stored by the training forward),
// optional adjoint summaries (nrange > 1), adjoint.
cudaError_t launch_grad(const GradParams &p, int dirs, bool f32, long long ngroups, int nrange, bool have_ckpt,
                        cudaStream_t s);
// Multiprocessors of the current device (queried once per device).
int sm_count();

cudaError_t launch_zero_f32(float *p, size_t n, cudaStream_t s);
// Gradient with the step options and the convolution: the float32 inputs of
// each direction, a bfloat16 -> float32 copy, and the chain rule to the raw
// tensors.
cudaError_t launch_grad_ext_prep(const GradExtParams &p, bool f32, cudaStream_t s);
cudaError_t launch_widen_bf16(const void *src, float *dst, long long n, cudaStream_t s);
cudaError_t launch_grad_ext_post(const GradExtParams &p, bool f32, cudaStream_t s);
cudaError_t launch_selftest_wait(unsigned *err, uint64_t limit_ns, cudaStream_t s);

// NC-SSD: rows kernel (bf16, whole rows in shared memory), else the tiled
// kernel with q CTAs per cluster.
cudaError_t launch_ncssd(const NcssdParams &p, bool rows, int q, bool gate, bool skip, bool f32, dim3 grid,
                         cudaStream_t s);

}  // namespace vssm
