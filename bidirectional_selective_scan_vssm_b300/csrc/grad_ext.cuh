// Gradient of the scan with the fused step and the directional convolution
// (vssm_scan_grad with delta_softplus, delta_bwd or conv_k > 0), sm_103a.
//
// What it computes is stated in include/vssm.h. The gradient is composed
// around the plain scan's gradient kernels (scan_grad.cuh), which run once
// per direction on float32 copies of that direction's step and input:
//
//  * grad_prep_kernel: per direction k, the step s_k = softplus(v_k + b_k)
//    (or the raw step v_k) and the input u_k = silu(pre_k), pre_k = the
//    direction's depthwise convolution of x (or u_k = x), in float32 -- the
//    values the forward kernel computes in registers -- plus float32 copies
//    of z and dout.
//  * the plain gradient, direction by direction, gives d s_k and d u_k per
//    token (and dB, dC, dA, dD, and each direction's share of dz).
//  * grad_post_kernel: the chain rule back to the raw tensors (VSSD page
//    §4.2.1.3 for the recurrence; the step map and the convolution as the
//    forward applies them): d v_k = d s_k * sigmoid(v_k + b_k) (softplus' =
//    sigmoid), d b_k = sum_t d v_k; d pre_k = d u_k * silu'(pre_k) with
//    silu'(p) = sigmoid(p) (1 + p (1 - sigmoid(p))); dx gathers d pre_k of
//    the output tokens whose taps read it (the transposed convolution), and
//    the taps' and biases' gradients sum d pre_k * x and d pre_k. One warp per
//    (batch, channel) row; the per-channel sums are reduced over the warp and
//    added atomically.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace vssm {

struct GradExtParams {
    const void *x, *delta[2], *z, *dout;   // raw inputs; delta[k]: direction k's raw step
    const float *bias[2];                  // step bias per direction (softplus only), or null
    const float *conv_w[2], *conv_b[2];    // taps [dim][K] and bias per direction (K > 0)
    int softplus, K;
    int batch, dim, L, seg_len, dirs;
    // float32 intermediates (workspace); null for a direction that is not run
    float *u[2];                           // input of each direction (may alias x when x is float32)
    float *pre[2];                         // convolution argument of each direction (K > 0)
    float *st[2];                          // step of each direction (may alias the raw step)
    float *z32, *dout32;                   // float32 copies (bfloat16 I/O), else null
    const float *du[2], *dst[2], *dz[2];   // the plain gradient's outputs per direction
    // outputs
    void *dx, *ddelta, *ddelta_bwd, *dzo;  // in the I/O type; ddelta_bwd null = shared step
    float *dbias[2];                       // [dim]; [1] == [0] when the bias is shared, null = none
    float *dconv_w[2], *dconv_b[2];        // [dim][K], [dim]; [1] == [0] when shared, null = none
};

__device__ __forceinline__ float sigmoid_acc(float v) { return 1.f / (1.f + expf(-v)); }

__device__ __forceinline__ float softplus_acc(float v)
{
    return v > 20.f ? v : log1pf(expf(v));
}

// Source token of convolution tap j for output token t, or -1 when the tap
// reads zero (outside the row or, folded, outside t's segment).
__device__ __forceinline__ int conv_src(int t, int j, int K, int L, int seg_len, int rev)
{
    const int s = rev ? t + (K - 1) - j : t - (K - 1) + j;
    if (s < 0 || s >= L) return -1;
    if (seg_len > 0 && s / seg_len != t / seg_len) return -1;
    return s;
}

template <typename T>
__global__ void __launch_bounds__(256) grad_prep_kernel(const GradExtParams p)
{
    const long long n = (long long)p.batch * p.dim * p.L;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (long long)gridDim.x * blockDim.x) {
        const long long row = e / p.L;
        const int t = (int)(e - row * p.L);
        const int d = (int)(row % p.dim);
        const T *xr = static_cast<const T *>(p.x) + row * p.L;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            if (!(p.dirs & (1 << k))) continue;
            if ((p.softplus || sizeof(T) == 2) && (k == 0 || p.st[1] != p.st[0])) {
                float v = ld_as_f32(static_cast<const T *>(p.delta[k]) + e);
                if (p.softplus) v = softplus_acc(v + (p.bias[k] ? p.bias[k][d] : 0.f));
                p.st[k][e] = v;
            }
            if (p.K > 0) {
                float a = p.conv_b[k] ? p.conv_b[k][d] : 0.f;
                for (int j = 0; j < p.K; ++j) {
                    const int s = conv_src(t, j, p.K, p.L, p.seg_len, k);
                    if (s >= 0) a = fmaf(p.conv_w[k][(long long)d * p.K + j], ld_as_f32(xr + s), a);
                }
                p.pre[k][e] = a;
                p.u[k][e] = a * sigmoid_acc(a);
            } else if (sizeof(T) == 2 && (k == 0 || p.u[1] != p.u[0])) {
                p.u[k][e] = ld_as_f32(xr + t);
            }
        }
        if (p.z32) p.z32[e] = ld_as_f32(static_cast<const T *>(p.z) + e);
        if (p.dout32) p.dout32[e] = ld_as_f32(static_cast<const T *>(p.dout) + e);
    }
}

template <typename T>
__global__ void __launch_bounds__(256) widen_f32_kernel(const T *src, float *dst, long long n)
{
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x)
        dst[i] = ld_as_f32(src + i);
}

template <typename T>
__global__ void __launch_bounds__(128) grad_post_kernel(const GradExtParams p)
{
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (row >= (long long)p.batch * p.dim) return;
    const int d = (int)(row % p.dim);
    const long long base = row * p.L;
    const T *xr = static_cast<const T *>(p.x) + base;
    const int K = p.K;
    float accb[2] = {0.f, 0.f}, acccb[2] = {0.f, 0.f};
    float accw[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    float bias[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) bias[k] = (p.softplus && p.bias[k]) ? p.bias[k][d] : 0.f;
    for (int t = lane; t < p.L; t += 32) {
        const long long e = base + t;
        float dv[2] = {0.f, 0.f}, dxv = 0.f;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            if (!(p.dirs & (1 << k))) continue;
            float g = p.dst[k][e];
            if (p.softplus) g *= sigmoid_acc(ld_as_f32(static_cast<const T *>(p.delta[k]) + e) + bias[k]);
            dv[k] = g;
            accb[k] += g;
            if (K > 0) {
                // taps of this token's own output (the weights' and bias's sums)
                const float pr = p.pre[k][e];
                const float sg = sigmoid_acc(pr);
                const float dp = p.du[k][e] * (sg + pr * sg * (1.f - sg));
                acccb[k] += dp;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (j >= K) break;
                    const int s = conv_src(t, j, K, p.L, p.seg_len, k);
                    if (s >= 0) accw[k][j] = fmaf(dp, ld_as_f32(xr + s), accw[k][j]);
                }
                // the output tokens whose taps read x_t (the transposed convolution)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (j >= K) break;
                    const int to = k ? t - (K - 1) + j : t + (K - 1) - j;
                    if (to < 0 || to >= p.L) continue;
                    if (p.seg_len > 0 && to / p.seg_len != t / p.seg_len) continue;
                    const long long eo = base + to;
                    const float po = p.pre[k][eo];
                    const float so = sigmoid_acc(po);
                    dxv = fmaf(p.conv_w[k][(long long)d * K + j], p.du[k][eo] * (so + po * so * (1.f - so)), dxv);
                }
            } else {
                dxv += p.du[k][e];
            }
        }
        st_from_f32(static_cast<T *>(p.dx) + e, dxv);
        if (p.ddelta_bwd) {     // (a direction that is not run has a zero gradient)
            st_from_f32(static_cast<T *>(p.ddelta) + e, dv[0]);
            st_from_f32(static_cast<T *>(p.ddelta_bwd) + e, dv[1]);
        } else {
            st_from_f32(static_cast<T *>(p.ddelta) + e, dv[0] + dv[1]);
        }
        if (p.dzo) {
            float s = 0.f;
            if (p.dirs & 1) s += p.dz[0][e];
            if (p.dirs & 2) s += p.dz[1][e];
            st_from_f32(static_cast<T *>(p.dzo) + e, s);
        }
    }
    // per-channel sums: over the warp, then one atomic add per row
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        if (!(p.dirs & (1 << k))) continue;
        float vb = accb[k], vc = acccb[k];
        float vw[4] = {accw[k][0], accw[k][1], accw[k][2], accw[k][3]};
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            vb += __shfl_xor_sync(0xffffffffu, vb, o);
            vc += __shfl_xor_sync(0xffffffffu, vc, o);
#pragma unroll
            for (int j = 0; j < 4; ++j) vw[j] += __shfl_xor_sync(0xffffffffu, vw[j], o);
        }
        if (lane == 0) {
            if (p.softplus && p.dbias[k]) atomicAdd(p.dbias[k] + d, vb);
            if (K > 0) {
                if (p.dconv_b[k]) atomicAdd(p.dconv_b[k] + d, vc);
                for (int j = 0; j < K; ++j) atomicAdd(p.dconv_w[k] + (long long)d * K + j, vw[j]);
            }
        }
    }
}

}  // namespace vssm
