// Selective-scan kernels for sm_103a (B300).
//
// What one launch computes is stated in include/vssm.h. This file holds the
// device code; vssm_api.cu validates arguments and picks the variant.
//
// Decomposition. A CTA owns R consecutive channels d0..d0+R-1 of one batch
// entry b and one token range [ta, tb) -- the whole sequence, or, for a
// folded sequence, a piece that starts and ends on segment boundaries (the
// reset makes pieces independent; SF-Mamba page, "周期性状态重置"). Every
// thread runs one direction of one channel over the range, holding 16/G of
// the N <= 16 states in fp32 registers; G threads (adjacent lanes) share a
// channel and add their partial C.h with one shuffle.
//
// Both directions in one CTA ("meet in the middle"): in phase 0 the forward
// threads walk the first half upward while the backward threads walk the
// second half downward; each stores its y (with its own D-skip) for every
// token it passes into a y-buffer. In phase 1 each direction walks the other
// half, adds the partner's buffered y, applies the silu(z) gate and emits the
// output. The y-buffer is shared memory for short rows and a global
// workspace otherwise. Inputs are read from HBM once; the state never leaves
// registers.
//
// Staging. Tokens are processed in chunks of kChunk per direction. All
// threads of the CTA cooperatively load the chunk's delta, x (and z / partner
// y in the output phase) for R channels plus B_t, C_t into shared memory as
// fp32, then each thread scans its chunk reading delta/x at its own row and
// B/C broadcast (all lanes of a warp are at the same token).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"

namespace vssm {

constexpr int kMaxState = 16;       // N <= 16
constexpr int kMaxConv = 4;         // taps of the directional convolution
constexpr int kChunk = 32;          // tokens per direction per staging step
constexpr int kPitch = kChunk + 1;  // padded row pitch (floats): rows hit distinct banks

struct ScanParams {
    const void *x, *delta[2], *z;   // delta: [0] forward, [1] backward step
    const float *dbias[2];          // step bias per direction (softplus only), or null
    int softplus;                   // 1: step = softplus(delta + bias)
    const float *conv_w[2], *conv_b[2];   // directional convolution per direction
    int conv_k;                     // 0: none; else taps (input = silu(conv(x)))
    const void *B[2], *C[2];        // [0] forward, [1] backward
    const float *A[2], *D[2];
    void *out;
    float *ybuf;                    // global y-buffer, [rows][L] floats, or null
    int batch, dim, L, N;
    int seg_len;                    // 0: no reset
    int pieces, piece_len;          // token ranges per (b, d): 1 and L unless folded
    int ypitch;                     // floats per channel in the shared y-buffer
};

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ void store_as(float *p, float v) { *p = v; }
__device__ __forceinline__ void store_as(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

// 2^x on the MUFU unit (PTX ex2.approx.ftz.f32).
__device__ __forceinline__ float mufu_ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float silu(float z) {
    return __fdividef(z, 1.0f + __expf(-z));
}

template <int R>
struct DirBlock {
    static constexpr int kRowArr = R * kPitch;                       // one [R][kPitch] array
    static constexpr int kFloats = 4 * kRowArr + 2 * kChunk * kMaxState;
};

// dirs: 1 forward only, 2 backward only, 3 both (meet in the middle).
template <typename T, int DIRS, int R, int G, bool YSMEM>
__global__ void __launch_bounds__((DIRS == 3 ? 2 : 1) * R * G)
scan_kernel(const ScanParams p)
{
    constexpr int NDIR = (DIRS == 3) ? 2 : 1;
    constexpr int NS = kMaxState / G;
    constexpr int NT = NDIR * R * G;
    constexpr int RA = DirBlock<R>::kRowArr;
    constexpr int DB = DirBlock<R>::kFloats;
    static_assert(NS % 4 == 0, "states per thread must be a multiple of 4");
    static_assert(G == 1 || G == 2, "G in {1, 2}");

    extern __shared__ __align__(16) float smem[];
    const int tid = threadIdx.x;

    // CTA -> (batch b, piece, channel block)
    const int dblocks = (p.dim + R - 1) / R;
    int cta = blockIdx.x;
    const int db = cta % dblocks;
    cta /= dblocks;
    const int piece = cta % p.pieces;
    const int b = cta / p.pieces;
    const int d0 = db * R;
    const int ta = piece * p.piece_len;
    const int tb = min(p.L, ta + p.piece_len);
    const int Lv = tb - ta;
    if (Lv <= 0) return;                                  // uniform over the CTA
    const int H = (DIRS == 3) ? (Lv + 1) / 2 : Lv;

    const int slot = (DIRS == 3) ? tid / (R * G) : 0;     // warp-uniform
    const int dir = (DIRS == 2) ? 1 : slot;               // 0 forward, 1 backward
    const int rg = tid % (R * G);
    const int r = rg / G;
    const int g = rg % G;
    const int d = d0 + r;
    const bool active = d < p.dim;

    const T *X = static_cast<const T *>(p.x);
    const T *Z = static_cast<const T *>(p.z);
    T *OUT = static_cast<T *>(p.out);
    const bool hasZ = Z != nullptr;
    const size_t row0 = ((size_t)b * p.dim + d0) * (size_t)p.L;   // element of (b, d0, t=0)
    float *ybig = smem + NDIR * DB;

    // Per-thread parameters: A pre-scaled by log2(e) so that exp(dt*A) = 2^(dt*A').
    const float kLog2e = 1.4426950408889634f;
    float Al2[NS], h[NS];
#pragma unroll
    for (int n = 0; n < NS; ++n) {
        const int nn = g * NS + n;
        Al2[n] = (active && nn < p.N) ? p.A[dir][(size_t)d * p.N + nn] * kLog2e : 0.0f;
        h[n] = 0.0f;
    }
    const float Dd = (active && p.D[dir] != nullptr) ? p.D[dir][d] : 0.0f;

    const int nphase = (DIRS == 3) ? 2 : 1;
    for (int phase = 0; phase < nphase; ++phase) {
        const bool fin = (phase == nphase - 1);
        // Token range of each staging slot in this phase.
        int lo[NDIR], hi[NDIR], nsteps = 0;
#pragma unroll
        for (int s = 0; s < NDIR; ++s) {
            const int ds = (DIRS == 2) ? 1 : s;
            if (DIRS == 3) {
                const bool first_half = ((ds == 0) == (phase == 0));
                lo[s] = first_half ? ta : ta + H;
                hi[s] = first_half ? ta + H : tb;
            } else {
                lo[s] = ta;
                hi[s] = tb;
            }
            nsteps = max(nsteps, (hi[s] - lo[s] + kChunk - 1) / kChunk);
        }

        for (int step = 0; step < nsteps; ++step) {
            int c0[NDIR], c1[NDIR];
#pragma unroll
            for (int s = 0; s < NDIR; ++s) {
                const int ds = (DIRS == 2) ? 1 : s;
                if (ds == 0) {                       // forward: chunks ascend
                    c0[s] = min(hi[s], lo[s] + step * kChunk);
                    c1[s] = min(hi[s], c0[s] + kChunk);
                } else {                             // backward: chunks descend
                    c1[s] = max(lo[s], hi[s] - step * kChunk);
                    c0[s] = max(lo[s], c1[s] - kChunk);
                }
            }

            __syncthreads();   // the previous step's readers of the staging buffers are done
            // ---- stage inputs of every slot (all threads cooperate)
#pragma unroll
            for (int s = 0; s < NDIR; ++s) {
                const int ds = (DIRS == 2) ? 1 : s;
                float *blk = smem + s * DB;
                const int len = c1[s] - c0[s];
                const T *DT = static_cast<const T *>(p.delta[ds]);
                const float *dbias = p.dbias[ds];
                for (int idx = tid; idx < R * kChunk; idx += NT) {
                    const int rr = idx / kChunk, i = idx % kChunk;
                    float dtv = 0.f, xv = 0.f, zv = 0.f, yv = 0.f;
                    if (i < len && d0 + rr < p.dim) {
                        const size_t gi = row0 + (size_t)rr * p.L + c0[s] + i;
                        dtv = to_f32(DT[gi]);
                        if (p.softplus) dtv = softplus_f32(dtv + (dbias ? dbias[d0 + rr] : 0.f));
                        if (p.conv_k > 0) {
                            // silu of the direction's convolution at token t: taps
                            // t-(K-1)+k forward, t+(K-1)-k backward; zero outside the
                            // row and, folded, outside t's segment
                            const int K = p.conv_k, t = c0[s] + i;
                            const float *w = p.conv_w[ds] + (size_t)(d0 + rr) * K;
                            float acc = p.conv_b[ds] ? p.conv_b[ds][d0 + rr] : 0.f;
                            for (int k = 0; k < K; ++k) {
                                const int ts = ds == 0 ? t - (K - 1) + k : t + (K - 1) - k;
                                if (ts < 0 || ts >= p.L) continue;
                                if (p.seg_len > 0 && ts / p.seg_len != t / p.seg_len) continue;
                                acc = fmaf(w[k], to_f32(X[gi - t + ts]), acc);
                            }
                            xv = silu(acc);
                        } else {
                            xv = to_f32(X[gi]);
                        }
                        if (fin && hasZ) zv = to_f32(Z[gi]);
                        if (DIRS == 3 && fin)
                            yv = YSMEM ? ybig[rr * p.ypitch + (c0[s] - ta) + i] : p.ybuf[gi];
                    }
                    const int o = rr * kPitch + i;
                    blk[o] = dtv;
                    blk[RA + o] = xv;
                    blk[2 * RA + o] = zv;
                    blk[3 * RA + o] = yv;
                }
                const T *Bp = static_cast<const T *>(p.B[ds]);
                const T *Cp = static_cast<const T *>(p.C[ds]);
                float *sB = blk + 4 * RA;
                float *sC = sB + kChunk * kMaxState;
                for (int idx = tid; idx < kChunk * kMaxState; idx += NT) {
                    const int i = idx / kMaxState, n = idx % kMaxState;
                    float bv = 0.f, cv = 0.f;
                    if (i < len && n < p.N) {
                        const size_t gi = ((size_t)b * p.L + c0[s] + i) * p.N + n;
                        bv = to_f32(Bp[gi]);
                        cv = to_f32(Cp[gi]);
                    }
                    sB[idx] = bv;
                    sC[idx] = cv;
                }
            }
            __syncthreads();

            // ---- scan this thread's chunk
            {
                float *blk = smem + slot * DB;
                const float *rDt = blk + r * kPitch;
                const float *rX = blk + RA + r * kPitch;
                const float *rZ = blk + 2 * RA + r * kPitch;
                float *rY = blk + 3 * RA + r * kPitch;
                const float *sB = blk + 4 * RA + g * NS;
                const float *sC = blk + 4 * RA + kChunk * kMaxState + g * NS;
                const int len = c1[slot] - c0[slot];
                const int seg = p.seg_len;
                // position inside the current segment (only used when folded)
                int pos = 0;
                if (seg > 0) pos = (dir == 0 ? c0[slot] : c1[slot] - 1) % seg;

                for (int k = 0; k < len; ++k) {
                    const int i = (dir == 0) ? k : len - 1 - k;
                    const float dtv = rDt[i];
                    const float xv = rX[i];
                    const float dx = dtv * xv;
                    if (seg > 0) {
                        const bool reset = (dir == 0) ? (pos == 0) : (pos == seg - 1);
                        if (reset) {
#pragma unroll
                            for (int n = 0; n < NS; ++n) h[n] = 0.0f;
                        }
                        pos = (dir == 0) ? (pos + 1 == seg ? 0 : pos + 1) : (pos == 0 ? seg - 1 : pos - 1);
                    }
                    const float4 *Bq = reinterpret_cast<const float4 *>(sB + i * kMaxState);
                    const float4 *Cq = reinterpret_cast<const float4 *>(sC + i * kMaxState);
                    float ya = 0.f, yb = 0.f;
#pragma unroll
                    for (int q = 0; q < NS / 4; ++q) {
                        const float4 bb = Bq[q];
                        const float4 cc = Cq[q];
                        h[4 * q + 0] = fmaf(mufu_ex2(dtv * Al2[4 * q + 0]), h[4 * q + 0], dx * bb.x);
                        h[4 * q + 1] = fmaf(mufu_ex2(dtv * Al2[4 * q + 1]), h[4 * q + 1], dx * bb.y);
                        h[4 * q + 2] = fmaf(mufu_ex2(dtv * Al2[4 * q + 2]), h[4 * q + 2], dx * bb.z);
                        h[4 * q + 3] = fmaf(mufu_ex2(dtv * Al2[4 * q + 3]), h[4 * q + 3], dx * bb.w);
                        ya = fmaf(cc.x, h[4 * q + 0], ya);
                        yb = fmaf(cc.y, h[4 * q + 1], yb);
                        ya = fmaf(cc.z, h[4 * q + 2], ya);
                        yb = fmaf(cc.w, h[4 * q + 3], yb);
                    }
                    float y = ya + yb;
                    if (G == 2) y += __shfl_xor_sync(0xffffffffu, y, 1);
                    y = fmaf(Dd, xv, y);
                    if (fin) {
                        float tot = (DIRS == 3) ? y + rY[i] : y;
                        if (hasZ) tot *= silu(rZ[i]);
                        y = tot;
                    }
                    if (g == 0) rY[i] = y;
                }
            }
            __syncthreads();

            // ---- drain: partial y to the y-buffer (phase 0) or output (last phase)
#pragma unroll
            for (int s = 0; s < NDIR; ++s) {
                const float *sY = smem + s * DB + 3 * RA;
                const int len = c1[s] - c0[s];
                for (int idx = tid; idx < R * kChunk; idx += NT) {
                    const int rr = idx / kChunk, i = idx % kChunk;
                    if (i < len && d0 + rr < p.dim) {
                        const float v = sY[rr * kPitch + i];
                        const size_t gi = row0 + (size_t)rr * p.L + c0[s] + i;
                        if (fin) {
                            store_as(OUT + gi, v);
                        } else if (YSMEM) {
                            ybig[rr * p.ypitch + (c0[s] - ta) + i] = v;
                        } else {
                            p.ybuf[gi] = v;
                        }
                    }
                }
            }
        }
    }
}

}  // namespace vssm
