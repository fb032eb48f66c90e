// NC-SSD, the non-causal global-state variant of the VSSD page (§4.2.4,
// §4.2.5: Y = C (B^T (X m))), for sm_103a (B300), N = 16.
//
// What it computes is stated in include/vssm.h (vssm_ncssd): per batch entry
// one hidden state H[n][d] = sum_j m_j B_j[n] x[d][j] shared by all tokens,
// then out[d][t] = (sum_n C_t[n] H[n][d] + D[d] x[d][t]) silu(z[d][t]).
// There is no recurrence: two small contractions, bound by the bytes of x, z
// and out. Two kernels:
//
//  * ncssd_state_kernel: a CTA owns 128 channels of one batch entry over a
//    range of tokens. It stages 32-token tiles of x (warps read rows along
//    tokens, coalesced) and of m_j B_j into shared memory; each thread then
//    accumulates 2 channels x 4 states with packed f32x2 FMAs and adds its
//    partial state to H atomically (H is zeroed first; long rows are split
//    over several CTAs).
//  * ncssd_out_kernel: a CTA owns 64 channels x 128 tokens. H's columns and
//    the tokens' C rows go to shared memory (fp32); a thread owns one token
//    and walks 32 channels (four at a time, so that their loads are in flight
//    together), reading x, z and writing out along tokens (coalesced across
//    the warp).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"
#include "scan_warp.cuh"

namespace vssm {

struct NcssdParams {
    const void *x, *z, *B, *C;
    const float *m, *D;
    void *out;
    float *H;                  // [batch][dim][16] fp32, accumulated
    int batch, dim, L, tok_per_cta;
};

constexpr int kNcChS = 128;    // channels per CTA (state kernel)
constexpr int kNcCh = 64;      // channels per CTA (output kernel)
constexpr int kNcTile = 32;    // tokens per staged tile (state kernel)
constexpr int kNcTok = 128;    // tokens per CTA (output kernel)

template <typename T>
__global__ void __launch_bounds__(256) ncssd_state_kernel(const NcssdParams p)
{
    __shared__ float xs[kNcChS][kNcTile + 1];            // x tile [channel][token]
    __shared__ __align__(16) float mb[kNcTile][16];      // m_j B_j[n]
    const int tid = threadIdx.x;
    const int b = blockIdx.z, d0 = blockIdx.y * kNcChS;
    const int ta = blockIdx.x * p.tok_per_cta, tb = min(p.L, ta + p.tok_per_cta);
    const int dl = (tid >> 2) * 2, q = tid & 3;          // channels dl, dl+1; states 4q..4q+3
    f2 h[2][2];
#pragma unroll
    for (int c = 0; c < 2; ++c) h[c][0] = h[c][1] = pack2(0.f, 0.f);
    const long long xrow0 = ((long long)b * p.dim + d0) * p.L;
    for (int t0 = ta; t0 < tb; t0 += kNcTile) {
        const int len = min(kNcTile, tb - t0);
        __syncthreads();
        // x tile: warp w reads rows 16w .. 16w+15, lane = token
        {
            const int lane = tid & 31, w = tid >> 5;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const int r = w * 16 + k;
                float v = 0.f;
                if (lane < len && d0 + r < p.dim)
                    v = ld_as_f32(static_cast<const T *>(p.x) + xrow0 + (long long)r * p.L + t0 + lane);
                xs[r][lane] = v;
            }
        }
        // m_j B_j: 32 tokens x 16 states, 2 per thread
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int e = tid + 256 * k, j = e >> 4, n = e & 15;
            float v = 0.f;
            if (j < len) {
                const long long bi = ((long long)b * p.L + t0 + j) * 16 + n;
                v = p.m[(long long)b * p.L + t0 + j] * ld_as_f32(static_cast<const T *>(p.B) + bi);
            }
            mb[j][n] = v;
        }
        __syncthreads();
#pragma unroll 4
        for (int j = 0; j < kNcTile; ++j) {
            f2 w0, w1;
            lds_2xf2(&mb[j][4 * q], w0, w1);
            const float x0 = xs[dl][j], x1 = xs[dl + 1][j];
            const f2 xx0 = pack2(x0, x0), xx1 = pack2(x1, x1);
            h[0][0] = fma2(xx0, w0, h[0][0]);
            h[0][1] = fma2(xx0, w1, h[0][1]);
            h[1][0] = fma2(xx1, w0, h[1][0]);
            h[1][1] = fma2(xx1, w1, h[1][1]);
        }
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int d = d0 + dl + c;
        if (d >= p.dim) continue;
        float *dst = p.H + ((long long)b * p.dim + d) * 16 + 4 * q;
        const float2 a0 = unpack2(h[c][0]), a1 = unpack2(h[c][1]);
        atomicAdd(dst + 0, a0.x);
        atomicAdd(dst + 1, a0.y);
        atomicAdd(dst + 2, a1.x);
        atomicAdd(dst + 3, a1.y);
    }
}

template <typename T>
__global__ void __launch_bounds__(256) ncssd_out_kernel(const NcssdParams p)
{
    __shared__ __align__(16) float hs[kNcCh][16];        // H columns of the tile's channels
    __shared__ __align__(16) float cs[kNcTok][16];       // C rows of the tile's tokens
    const int tid = threadIdx.x;
    const int b = blockIdx.z, d0 = blockIdx.y * kNcCh, t0 = blockIdx.x * kNcTok;
    for (int e = tid; e < kNcCh * 16; e += 256) {
        const int dd = e >> 4;
        hs[dd][e & 15] = d0 + dd < p.dim ? p.H[((long long)b * p.dim + d0) * 16 + e] : 0.f;
    }
    for (int e = tid; e < kNcTok * 16; e += 256) {
        const int tt = e >> 4;
        cs[tt][e & 15] = t0 + tt < p.L
            ? ld_as_f32(static_cast<const T *>(p.C) + ((long long)b * p.L + t0) * 16 + e) : 0.f;
    }
    __syncthreads();
    const int tt = tid & (kNcTok - 1), cg = tid >> 7;      // token; channel half
    const int t = t0 + tt;
    if (t >= p.L) return;
    f2 c[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) lds_2xf2(&cs[tt][4 * k], c[2 * k], c[2 * k + 1]);
    const bool hasZ = p.z != nullptr, hasD = p.D != nullptr;
    const int nd = min(kNcCh / 2, p.dim - d0 - cg * (kNcCh / 2));   // this half's channels
#pragma unroll 4
    for (int k = 0; k < kNcCh / 2; ++k) {
        if (k < nd) {
            const int dd = cg * (kNcCh / 2) + k, d = d0 + dd;
            const long long e = ((long long)b * p.dim + d) * p.L + t;
            const float xv = hasD ? ld_as_f32(static_cast<const T *>(p.x) + e) : 0.f;
            const float zv = hasZ ? ld_as_f32(static_cast<const T *>(p.z) + e) : 0.f;
            f2 acc = pack2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                f2 h0, h1;
                lds_2xf2(&hs[dd][4 * q], h0, h1);
                acc = fma2(c[2 * q], h0, acc);
                acc = fma2(c[2 * q + 1], h1, acc);
            }
            const float2 a = unpack2(acc);
            float y = a.x + a.y;
            if (hasD) y = fmaf(p.D[d], xv, y);
            if (hasZ) y *= silu_f32<T>(zv);
            st_from_f32(static_cast<T *>(p.out) + e, y);
        }
    }
}

}  // namespace vssm
