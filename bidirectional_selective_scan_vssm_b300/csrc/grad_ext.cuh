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
//    the taps' and biases' gradients sum d pre_k * x and d pre_k. pre_k is
//    recomputed from x rather than stored.
//
// Both kernels take one (batch, channel) row and a tile of 256 TPT tokens per
// block, TPT tokens per thread (strided by the block, so that loads coalesce;
// TPT = 4 for rows of 1024 tokens or more, else 1). The tile's x and its halo
// of up to 2 (K - 1) tokens are staged in shared memory, and so are the
// neighbours' d pre_k, both zero outside the row: a tap then needs no row
// test, and on folded rows only a segment test (a select, not a branch). The
// tap count K and the folding are template parameters. The step, softplus
// and silu are the forward kernel's own functions, the taps summed in its
// order, so that s_k and u_k are the values the forward used. Each thread
// issues its loads before its stores. The per-channel sums are reduced over
// the block (a warp reduce-scatter, then shared memory) and added with one
// atomic per sum and block.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "ptx.cuh"

namespace vssm {

struct GradExtParams {
    const void *x, *delta[2], *z, *dout;   // raw inputs; delta[k]: direction k's raw step
    const float *bias[2];                  // step bias per direction (softplus only), or null
    const float *conv_w[2], *conv_b[2];    // taps [dim][K] and bias per direction (K > 0)
    int softplus, K;
    int batch, dim, L, seg_len, dirs;
    // float32 intermediates (workspace); null for a direction that is not run
    float *u[2];                           // input of each direction (may alias x when x is float32)
    float *st[2];                          // step of each direction (may alias the raw step)
    float *z32, *dout32;                   // float32 copies (bfloat16 I/O), else null
    const float *du[2], *dst[2], *dz[2];   // the plain gradient's outputs per direction
    // outputs
    void *dx, *ddelta, *ddelta_bwd, *dzo;  // in the I/O type; ddelta_bwd null = shared step
    float *dbias[2];                       // [dim]; [1] == [0] when the bias is shared, null = none
    float *dconv_w[2], *dconv_b[2];        // [dim][K], [dim]; [1] == [0] when shared, null = none
};

// sigmoid(v) = 1 / (1 + 2^(-v log2 e)); tends to 0 and 1 at the ends.
__device__ __forceinline__ float sigmoid_f32(float v)
{
    return __fdividef(1.0f, 1.0f + ex2_mufu(-1.4426950408889634f * v));
}

// silu'(p) = sigmoid(p) (1 + p (1 - sigmoid(p))).
__device__ __forceinline__ float silu_grad(float p)
{
    const float sg = sigmoid_f32(p);
    return fmaf(p * sg, 1.f - sg, sg);
}

// Threads per block of the preparation and chain-rule kernels, the tokens per
// thread of long rows, and the largest halo the chain rule stages
// (2 (K - 1) for K <= 4).
constexpr int kExtThreads = 256;
constexpr int kExtLongTPT = 4;
constexpr int kExtHalo = 6;

// Block -> (row, first token of the tile, tokens of the tile).
template <int TILE>
__device__ __forceinline__ void ext_tile(int L, long long &row, int &t0, int &tl)
{
    const int ntile = (L + TILE - 1) / TILE;
    row = (long long)blockIdx.x / ntile;
    t0 = (int)((long long)blockIdx.x - row * ntile) * TILE;
    tl = min(TILE, L - t0);
}

// Place in its segment of token t, then of t + kExtThreads, ... : one modulo
// (t mod seg_len in [0, seg_len), also for the halo before the row, t < 0),
// then a step of kExtThreads mod seg_len with one wrap (not folded: t itself,
// with a segment longer than any row).
struct SegPos {
    int pos, step, seg;
    __device__ __forceinline__ SegPos(int t, int seg_len)
        : pos(t), step(kExtThreads), seg(0x7fffffff)
    {
        if (seg_len > 0) {
            pos = t % seg_len;
            if (pos < 0) pos += seg_len;
            step = kExtThreads % seg_len;
            seg = seg_len;
        }
    }
    __device__ __forceinline__ void next()
    {
        pos += step;
        if (pos >= seg) pos -= seg;
    }
};

// Stage x[t0 - h, t0 + tl + h) of row xr as float32, zero outside the row
// (at most R passes of the block).
template <int R, typename T>
__device__ __forceinline__ void stage_x(float *xs, const T *xr, int t0, int tl, int h, int L)
{
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int i = threadIdx.x + r * kExtThreads, t = t0 - h + i;
        if (i < tl + 2 * h) xs[i] = (t >= 0 && t < L) ? ld_as_f32(xr + t) : 0.f;
    }
}

// The convolution argument of a token in direction k: bias + sum over the K
// taps of w_j x_s, s = t - m (k = 0) or t + m (k = 1), m = K - 1 - j, summed
// from the token's own tap outwards as the forward kernel does. xc points at
// x_t in the staged tile, which reads zero outside the row; a tap outside
// the token's segment (pos: its place in it) gets weight zero (FOLD: folded
// rows; otherwise the staged zeros are the only bound).
template <int K, bool FOLD>
__device__ __forceinline__ float conv_arg(const float *xc, const float (&w)[4], float b, int k, int pos,
                                          int seg)
{
    float a = b;
#pragma unroll
    for (int m = 0; m < K; ++m) {
        const bool ok = !FOLD || (k ? (pos + m < seg) : (pos >= m));
        a = fmaf(ok ? w[K - 1 - m] : 0.f, xc[k ? m : -m], a);
    }
    return a;
}

// Taps and biases of channel d for the directions that run.
template <int K>
__device__ __forceinline__ void ext_weights(const GradExtParams &p, int d, float (&w)[2][4], float (&cb)[2],
                                            float (&sb)[2])
{
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        w[k][0] = w[k][1] = w[k][2] = w[k][3] = 0.f;
        cb[k] = sb[k] = 0.f;
        if (!(p.dirs & (1 << k))) continue;
#pragma unroll
        for (int j = 0; j < K; ++j) w[k][j] = p.conv_w[k][(long long)d * K + j];
        if (K > 0 && p.conv_b[k]) cb[k] = p.conv_b[k][d];
        if (p.softplus && p.bias[k]) sb[k] = p.bias[k][d];
    }
}

template <typename T, int TPT, int K, bool FOLD>
__global__ void __launch_bounds__(kExtThreads) grad_prep_kernel(const GradExtParams p)
{
    constexpr int kTile = kExtThreads * TPT;
    constexpr int H = K > 0 ? K - 1 : 0;
    __shared__ float xs[kTile + 2 * H + 1];
    long long row;
    int t0, tl;
    ext_tile<kTile>(p.L, row, t0, tl);
    const int d = (int)(row % p.dim);
    const long long base = row * p.L;
    const T *xr = static_cast<const T *>(p.x) + base;
    float w[2][4], cb[2], sb[2];
    ext_weights<K>(p, d, w, cb, sb);
    // this thread's tokens: loads first (the stores below may alias them for
    // all the compiler knows), then x staged, then the step and input maps
    const bool own_st1 = p.st[1] != p.st[0], own_u1 = p.u[1] != p.u[0];
    // (the thread's r-th token is eb + r kExtThreads: constant offsets)
    const long long eb = base + t0 + threadIdx.x;
    float gv[2][TPT], gz[TPT], go[TPT], gx[TPT];
#pragma unroll
    for (int r = 0; r < TPT; ++r) {
        const int o = r * kExtThreads;
        const bool in = (int)threadIdx.x + o < tl;
        gz[r] = go[r] = gx[r] = 0.f;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            gv[k][r] = 0.f;
            if (in && (p.dirs & (1 << k)) && (p.softplus || sizeof(T) == 2) && (k == 0 || own_st1))
                gv[k][r] = ld_as_f32(static_cast<const T *>(p.delta[k]) + eb + o);
        }
        if (in && p.z32) gz[r] = ld_as_f32(static_cast<const T *>(p.z) + eb + o);
        if (in && p.dout32) go[r] = ld_as_f32(static_cast<const T *>(p.dout) + eb + o);
        if (in && K == 0 && sizeof(T) == 2) gx[r] = ld_as_f32(static_cast<const T *>(p.x) + eb + o);
    }
    if (K > 0) {
        stage_x<TPT + 1>(xs, xr, t0, tl, H, p.L);
        __syncthreads();
    }
    SegPos sp(t0 + (int)threadIdx.x, FOLD ? p.seg_len : 0);
#pragma unroll
    for (int r = 0; r < TPT; ++r, sp.next()) {
        const int o = r * kExtThreads, i = (int)threadIdx.x + o;
        if (i >= tl) break;
        const long long e = eb + o;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            if (!(p.dirs & (1 << k))) continue;
            if ((p.softplus || sizeof(T) == 2) && (k == 0 || own_st1))
                p.st[k][e] = p.softplus ? softplus_f32(gv[k][r] + sb[k]) : gv[k][r];
            if (K > 0)
                p.u[k][e] = silu_f32<T>(conv_arg<K, FOLD>(xs + H + i, w[k], cb[k], k, sp.pos, sp.seg));
            else if (sizeof(T) == 2 && (k == 0 || own_u1))
                p.u[k][e] = gx[r];
        }
        if (p.z32) p.z32[e] = gz[r];
        if (p.dout32) p.dout32[e] = go[r];
    }
}

template <typename T>
__global__ void __launch_bounds__(256) widen_f32_kernel(const T *src, float *dst, long long n)
{
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x)
        dst[i] = ld_as_f32(src + i);
}

// Per-channel sums of a direction: the step bias, the convolution bias and the
// K <= 4 taps (slots 6, 7 unused).
constexpr int kExtSums = 8;

// Reduce-scatter of 16 values over the warp: on return lane l's v[0] holds the
// warp's total of value l / 2 (each halving step sends one half of the values
// to the partner lane and keeps the other; a last step adds the lane pair).
__device__ __forceinline__ float warp_reduce_scatter16(float (&v)[16], int lane)
{
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const int half = 8 >> s, o = 16 >> s;
        const bool up = lane & o;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i >= half) break;
            const float send = up ? v[i] : v[i + half];
            const float keep = up ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

template <typename T, int TPT, int K, bool FOLD>
__global__ void __launch_bounds__(kExtThreads) grad_post_kernel(const GradExtParams p)
{
    constexpr int kTile = kExtThreads * TPT;
    constexpr int H = K > 0 ? K - 1 : 0;
    __shared__ float xs[kTile + 4 * H + 1];
    __shared__ float dps[2][kTile + 2 * H + 1];   // d pre_k of tokens t0 - H ...
    __shared__ float red[kExtThreads / 32][2 * kExtSums];
    long long row;
    int t0, tl;
    ext_tile<kTile>(p.L, row, t0, tl);
    const int d = (int)(row % p.dim);
    const int tid = threadIdx.x, lane = tid & 31;
    const long long base = row * p.L;
    const T *xr = static_cast<const T *>(p.x) + base;
    float w[2][4], cb[2], sb[2];
    ext_weights<K>(p, d, w, cb, sb);
    // this thread's tokens: loads first (before the staging, to overlap it)
    // (the thread's r-th token is eb + r kExtThreads: constant offsets)
    const long long eb = base + t0 + tid;
    float gs[2][TPT], gv[2][TPT], gz[TPT], gu[TPT];
#pragma unroll
    for (int r = 0; r < TPT; ++r) {
        const int o = r * kExtThreads;
        const bool in = tid + o < tl;
        gz[r] = gu[r] = 0.f;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            gs[k][r] = gv[k][r] = 0.f;
            if (!(p.dirs & (1 << k)) || !in) continue;
            gs[k][r] = p.dst[k][eb + o];
            if (p.softplus) gv[k][r] = ld_as_f32(static_cast<const T *>(p.delta[k]) + eb + o);
            if (p.dzo) gz[r] += p.dz[k][eb + o];
            if (K == 0) gu[r] += p.du[k][eb + o];
        }
    }
    if (K > 0) {
        // x over [t0 - 2H, t0 + tl + 2H), then d pre_k over [t0 - H, t0 + tl + H)
        // (zero outside the row, where the direction's gradient d u_k is read as zero)
        stage_x<TPT + 1>(xs, xr, t0, tl, 2 * H, p.L);
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            if (!(p.dirs & (1 << k))) continue;
            const float *dur = p.du[k] + base;
            float duv[TPT + 1];
#pragma unroll
            for (int r = 0; r <= TPT; ++r) {
                const int i = tid + r * kExtThreads, tt = t0 - H + i;
                duv[r] = (i < tl + 2 * H && tt >= 0 && tt < p.L) ? dur[tt] : 0.f;
            }
            SegPos sp(t0 - H + tid, FOLD ? p.seg_len : 0);
#pragma unroll
            for (int r = 0; r <= TPT; ++r, sp.next()) {
                const int i = tid + r * kExtThreads;
                if (i < tl + 2 * H)
                    dps[k][i] = duv[r] * silu_grad(conv_arg<K, FOLD>(xs + H + i, w[k], cb[k], k, sp.pos, sp.seg));
            }
        }
        __syncthreads();
    }
    float sums[2][kExtSums] = {};
    SegPos sp(t0 + tid, FOLD ? p.seg_len : 0);
#pragma unroll
    for (int r = 0; r < TPT; ++r, sp.next()) {
        const int o = r * kExtThreads, i = tid + o;
        if (i >= tl) break;
        const long long e = eb + o;
        const int pos = sp.pos;
        float dv[2] = {0.f, 0.f}, dxv = gu[r];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            if (!(p.dirs & (1 << k))) continue;
            float g = gs[k][r];
            if (p.softplus) g *= sigmoid_f32(gv[k][r] + sb[k]);
            dv[k] = g;
            sums[k][0] += g;
            if (K > 0) {
                const float dp = dps[k][H + i];
                const float *xc = xs + 2 * H + i;   // x_t
                sums[k][1] += dp;
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    const int m = K - 1 - j;
                    // tap j of token t reads x at t -/+ m (zero outside the row)
                    const bool tap = !FOLD || (k ? (pos + m < sp.seg) : (pos >= m));
                    sums[k][2 + j] = fmaf(tap ? dp : 0.f, xc[k ? m : -m], sums[k][2 + j]);
                    // output token t +/- m reads x_t with tap j (transposed
                    // convolution; its d pre is zero outside the row)
                    const bool out = !FOLD || (k ? (pos >= m) : (pos + m < sp.seg));
                    dxv = fmaf(out ? w[k][j] : 0.f, dps[k][H + i + (k ? -m : m)], dxv);
                }
            }
        }
        st_from_f32(static_cast<T *>(p.dx) + e, dxv);
        if (p.ddelta_bwd) {     // (a direction that is not run has a zero gradient)
            st_from_f32(static_cast<T *>(p.ddelta) + e, dv[0]);
            st_from_f32(static_cast<T *>(p.ddelta_bwd) + e, dv[1]);
        } else {
            st_from_f32(static_cast<T *>(p.ddelta) + e, dv[0] + dv[1]);
        }
        if (p.dzo) st_from_f32(static_cast<T *>(p.dzo) + e, gz[r]);
    }
    // per-channel sums: over the warp, then over the block, one atomic each
    if (!p.softplus && K == 0) return;
    float v[16];
#pragma unroll
    for (int q = 0; q < kExtSums; ++q) {
        v[q] = sums[0][q];
        v[kExtSums + q] = sums[1][q];
    }
    const float tot = warp_reduce_scatter16(v, lane);
    if (!(lane & 1)) red[tid >> 5][lane >> 1] = tot;
    __syncthreads();
    if (tid < 2 * kExtSums) {
        const int k = tid / kExtSums, q = tid % kExtSums;
        if (!(p.dirs & (1 << k))) return;
        float s = 0.f;
#pragma unroll
        for (int wi = 0; wi < kExtThreads / 32; ++wi) s += red[wi][tid];
        float *dst = nullptr;
        if (q == 0) dst = (p.softplus && p.dbias[k]) ? p.dbias[k] + d : nullptr;
        else if (q == 1) dst = (K > 0 && p.dconv_b[k]) ? p.dconv_b[k] + d : nullptr;
        else if (q - 2 < K) dst = p.dconv_w[k] + (long long)d * K + (q - 2);
        if (dst) atomicAdd(dst, s);
    }
}

}  // namespace vssm
