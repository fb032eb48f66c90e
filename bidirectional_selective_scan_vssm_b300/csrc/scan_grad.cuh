// Gradient of the bidirectional selective scan (N = 16) for sm_103a (B300).
//
// What it computes is stated in include/vssm.h (vssm_scan_grad): the exact
// reverse-mode derivative of L = sum(dout * out) for a call of the forward
// scan. Per direction, against its scan order, with the adjoint
// lambda_t = dL/dh_t carried in registers:
//
//     lambda_t = ds_t * C_t + abar_next * lambda_next,   ds_t = dout_t * silu(z_t)
//     dC_t += ds_t * h_t,   dB_t += lambda_t * delta_t * x_t
//     dx_t += ds_t * D + delta_t * sum_n lambda_t[n] B_t[n]
//     ddelta_t += x_t * sum_n lambda_t[n] B_t[n] + sum_n A[n] abar_t[n] h_prev[n] lambda_t[n]
//     dA[n] += delta_t * abar_t[n] h_prev[n] lambda_t[n],   dD += ds_t * x_t
//     dz_t = dout_t * silu'(z_t) * (y_fwd_t + y_bwd_t)
//
// Work decomposition (one lane per channel, 32 channels per warp, like the
// forward kernel):
//
//  * grad_ckpt_kernel: one warp per (direction, channel group) runs the
//    forward recurrence over the row and stores the state entering every
//    8-token chunk (in that direction's scan order) to a checkpoint buffer.
//  * grad_adjoint_kernel: the two directions of a channel group are a warp
//    pair that meets in the middle, as in the forward kernel but walking
//    against the scan orders: the forward direction's adjoint walks the
//    chunks downward, the backward one upward. Per chunk a warp recomputes
//    the chunk's states from its checkpoint into shared memory (fp32, one
//    slot per token), then walks the chunk backward through the adjoint.
//    In phase 0 each warp leaves its fp32 partial dx, ddelta, dz for its half
//    in the workspace; after a bounded rendezvous, phase 1 adds the
//    partner's partials and writes the gradients. dB and dC are reduced
//    over the warp's 32 channels by a butterfly reduce-scatter (each lane
//    ends with one of the 32 sums) and added to global memory atomically;
//    dA and dD accumulate in registers over the row and are added at the end.
//
// The only wait on another warp is the pair rendezvous (bounded, as in the
// forward kernel).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"
#include "scan_warp.cuh"

namespace vssm {

constexpr int kTG = 8;                  // tokens per gradient chunk

struct GradParams {
    const void *x, *delta, *z, *dout;
    const void *B[2], *C[2];
    const float *A[2], *D[2];
    void *dx, *ddelta, *dz;
    float *dB[2], *dC[2];               // [1] == [0] when the directions share B / C
    float *dA[2], *dD[2];
    float *ckpt;                        // [slot][ngroups][nch][16][32]
    float *part;                        // [ngroups][L][3][32] (both directions only)
    unsigned *err;
    int batch, dim, L, seg_len, rgroups, nch;
    long long ngroups;                  // batch * rgroups
};

template <typename T>
__device__ __forceinline__ float gload(const void *base, long long i)
{
    return ld_as_f32(static_cast<const T *>(base) + i);
}

__device__ __forceinline__ bool reset_at(int t, int seg_len, int dir)
{
    if (seg_len <= 0) return false;
    const int ph = t % seg_len;
    return dir == 0 ? ph == 0 : ph == seg_len - 1;
}

// Checkpoints: the state entering each 8-token chunk in this direction's
// scan order.
template <typename T, int DIRS>
__global__ void __launch_bounds__(128) grad_ckpt_kernel(const GradParams p)
{
    constexpr int NDIR = (DIRS == 3) ? 2 : 1;
    const int lane = threadIdx.x & 31;
    const long long u = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (u >= NDIR * p.ngroups) return;
    const int slot = (int)(u / p.ngroups);
    const long long grp = u % p.ngroups;
    const int dir = (DIRS == 3) ? slot : (DIRS == 1 ? 0 : 1);
    const int b = (int)(grp / p.rgroups), d0 = (int)(grp % p.rgroups) * 32;
    const int d = d0 + lane;
    const bool act = d < p.dim;
    constexpr float kLog2e = 1.4426950408889634f;
    float Al2[16], h[16];
#pragma unroll
    for (int n = 0; n < 16; ++n) {
        Al2[n] = act ? p.A[dir][(long long)d * 16 + n] * kLog2e : 0.f;
        h[n] = 0.f;
    }
    const long long row = ((long long)b * p.dim + (act ? d : d0)) * p.L;
    const char *Bb = static_cast<const char *>(p.B[dir]) + (long long)b * p.L * 16 * sizeof(T);
    float *ck = p.ckpt + ((long long)slot * p.ngroups + grp) * p.nch * 512;
    for (int s = 0; s < p.nch; ++s) {
        const int j = dir == 0 ? s : p.nch - 1 - s;          // chunk in scan order
        float *cj = ck + (long long)j * 512;
#pragma unroll
        for (int n = 0; n < 16; ++n) cj[n * 32 + lane] = h[n];
        const int t0 = j * kTG, t1 = min(p.L, t0 + kTG);
        for (int k = 0; k < t1 - t0; ++k) {
            const int t = dir == 0 ? t0 + k : t1 - 1 - k;
            const float dt = act ? gload<T>(p.delta, row + t) : 0.f;
            const float xv = act ? gload<T>(p.x, row + t) : 0.f;
            const bool rs = reset_at(t, p.seg_len, dir);
            const T *Bt = reinterpret_cast<const T *>(Bb) + (long long)t * 16;
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                const float a = rs ? 0.f : ex2_mufu(dt * Al2[n]);
                h[n] = fmaf(a, h[n], dt * xv * ld_as_f32(Bt + n));
            }
        }
    }
}

// One butterfly stage over the 2W live values v[0..2W): the lane keeps the
// half selected by its bit W, sends the other half to lane ^ W and adds what
// comes back.
template <int W>
__device__ __forceinline__ void reduce_scatter_stage(float (&v)[32], bool upper)
{
#pragma unroll
    for (int i = 0; i < W; ++i) {
        const float send = upper ? v[i] : v[i + W];
        const float keep = upper ? v[i + W] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, W);
    }
}

// Butterfly reduce-scatter of 32 values over the warp: on return lane l holds
// the warp's sum of v[l] in v[0] (31 shuffles and 31 adds per lane).
__device__ __forceinline__ void reduce_scatter32(float (&v)[32], int lane)
{
    reduce_scatter_stage<16>(v, (lane & 16) != 0);
    reduce_scatter_stage<8>(v, (lane & 8) != 0);
    reduce_scatter_stage<4>(v, (lane & 4) != 0);
    reduce_scatter_stage<2>(v, (lane & 2) != 0);
    reduce_scatter_stage<1>(v, (lane & 1) != 0);
}

template <typename T, int DIRS>
struct GradLayout {
    // per warp: states [kTG + 1][16][32] fp32, then B and C of the chunk [kTG][32] fp32
    static constexpr int kH = (kTG + 1) * 16 * 32 * 4;
    static constexpr int kBC = kTG * 32 * 4;
    static constexpr int kWarpBytes = kH + kBC + 16;      // + pair barrier
};

template <typename T, int DIRS>
__global__ void __launch_bounds__((DIRS == 3 ? 2 : 1) * 32, 1)
grad_adjoint_kernel(const GradParams p)
{
    constexpr int NDIR = (DIRS == 3) ? 2 : 1;
    using Lay = GradLayout<T, DIRS>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long grp = blockIdx.x;
    const int slot = warp;
    const int dir = (DIRS == 3) ? warp : (DIRS == 1 ? 0 : 1);
    unsigned char *wsm = smem_raw + warp * Lay::kWarpBytes;
    float *hb = reinterpret_cast<float *>(wsm);                 // [kTG + 1][16][32]
    float *bc = reinterpret_cast<float *>(wsm + Lay::kH);       // [kTG][32]: B[16], C[16]
    uint64_t *pairbar = reinterpret_cast<uint64_t *>(smem_raw + Lay::kWarpBytes - 16);
    if (DIRS == 3 && threadIdx.x == 0) {
        mbar_init(pairbar, 2);
        fence_mbar_init();
    }
    __syncthreads();
    if (grp >= p.ngroups) return;

    const int b = (int)(grp / p.rgroups), d0 = (int)(grp % p.rgroups) * 32;
    const int d = d0 + lane;
    const bool act = d < p.dim;
    constexpr float kLog2e = 1.4426950408889634f;
    float Al2[16], Aa[16], lam[16], dA[16];
#pragma unroll
    for (int n = 0; n < 16; ++n) {
        Aa[n] = act ? p.A[dir][(long long)d * 16 + n] : 0.f;
        Al2[n] = Aa[n] * kLog2e;
        lam[n] = 0.f;
        dA[n] = 0.f;
    }
    const float Dk = (act && p.D[dir]) ? p.D[dir][d] : 0.f;
    float dD = 0.f;
    const long long row = ((long long)b * p.dim + (act ? d : d0)) * p.L;
    const long long bcrow = (long long)b * p.L * 16;
    const float *ck = p.ckpt + ((long long)slot * p.ngroups + grp) * p.nch * 512;
    const bool hasZ = p.z != nullptr;
    float *dBk = p.dB[dir], *dCk = p.dC[dir];

    // chunks of each phase, walked against the scan order
    const int Hc = (p.nch + 1) / 2;
    const int nphase = (DIRS == 3) ? 2 : 1;
    bool ok = true;
    for (int phase = 0; phase < nphase && ok; ++phase) {
        const bool fin = phase == nphase - 1;
        int clo, chi;                                  // chunk range [clo, chi)
        if (DIRS == 3) {
            const bool upper = (dir == 0) == (phase == 0);
            clo = upper ? Hc : 0;
            chi = upper ? p.nch : Hc;
        } else {
            clo = 0;
            chi = p.nch;
        }
        for (int s = 0; s < chi - clo; ++s) {
            const int j = dir == 0 ? chi - 1 - s : clo + s;
            const int t0 = j * kTG, t1 = min(p.L, t0 + kTG), len = t1 - t0;
            // B and C of the chunk (lane = (token, part))
            {
                const int tk = lane >> 2, q = lane & 3;   // 8 tokens x 4 quarters of 8 values
                if (tk < len) {
                    const void *src = q < 2 ? p.B[dir] : p.C[dir];
                    const long long o = bcrow + (long long)(t0 + tk) * 16 + (q & 1) * 8;
#pragma unroll
                    for (int i = 0; i < 8; ++i) bc[tk * 32 + (q >> 1) * 16 + (q & 1) * 8 + i] = gload<T>(src, o + i);
                }
            }
            // this lane's inputs of the chunk, indexed by scan position k
            // (token t0 + k going forward, t1 - 1 - k going backward)
            float dtv[kTG], xv[kTG], zv[kTG], go[kTG];
#pragma unroll
            for (int k = 0; k < kTG; ++k) {
                const bool in = act && k < len;
                const long long e = row + (dir == 0 ? t0 + k : t1 - 1 - k);
                dtv[k] = in ? gload<T>(p.delta, e) : 0.f;
                xv[k] = in ? gload<T>(p.x, e) : 0.f;
                zv[k] = (in && hasZ) ? gload<T>(p.z, e) : 0.f;
                go[k] = in ? gload<T>(p.dout, e) : 0.f;
            }
            // recompute the chunk's states in scan order: slot 0 = entering
            // state, slot k + 1 = state after the k-th token in scan order
            {
                const float *cj = ck + (long long)j * 512;
                float h[16];
#pragma unroll
                for (int n = 0; n < 16; ++n) {
                    h[n] = cj[n * 32 + lane];
                    hb[n * 32 + lane] = h[n];
                }
                __syncwarp();
#pragma unroll
                for (int k = 0; k < kTG; ++k) {
                    if (k < len) {
                        const int i = dir == 0 ? k : len - 1 - k;
                        const bool rs = reset_at(t0 + i, p.seg_len, dir);
                        const float ux = dtv[k] * xv[k];
#pragma unroll
                        for (int n = 0; n < 16; ++n) {
                            const float a = rs ? 0.f : ex2_mufu(dtv[k] * Al2[n]);
                            h[n] = fmaf(a, h[n], ux * bc[i * 32 + n]);
                            hb[((k + 1) * 16 + n) * 32 + lane] = h[n];
                        }
                    }
                }
            }
            __syncwarp();
            // adjoint, against the scan order
            float hn[16];                               // state after the current token
#pragma unroll
            for (int n = 0; n < 16; ++n) hn[n] = hb[(len * 16 + n) * 32 + lane];
#pragma unroll
            for (int k = kTG - 1; k >= 0; --k) {
                if (k >= len) continue;
                const int i = dir == 0 ? k : len - 1 - k;
                const int t = t0 + i;
                const bool rs = reset_at(t, p.seg_len, dir);
                float g = 1.f, gp = 0.f;
                if (hasZ) {
                    const float sg = __frcp_rn(1.f + ex2_mufu(-kLog2e * zv[k]));
                    g = zv[k] * sg;
                    gp = sg * fmaf(zv[k], 1.f - sg, 1.f);
                }
                const float ds = go[k] * g;
                const float *Bt = bc + i * 32, *Ct = Bt + 16;
                float v[32];                            // dB[16], dC[16] contributions
                float yk = Dk * xv[k], sB = 0.f, sw = 0.f;
                const float ux = dtv[k] * xv[k];
#pragma unroll
                for (int n = 0; n < 16; ++n) {
                    const float hp = hb[(k * 16 + n) * 32 + lane];
                    const float a = rs ? 0.f : ex2_mufu(dtv[k] * Al2[n]);
                    yk = fmaf(Ct[n], hn[n], yk);
                    const float l = fmaf(ds, Ct[n], lam[n]);
                    v[16 + n] = ds * hn[n];
                    v[n] = l * ux;
                    sB = fmaf(l, Bt[n], sB);
                    const float w = l * a * hp;
                    sw = fmaf(w, Aa[n], sw);
                    dA[n] = fmaf(w, dtv[k], dA[n]);
                    lam[n] = a * l;
                    hn[n] = hp;
                }
                dD = fmaf(ds, xv[k], dD);
                float gx = fmaf(ds, Dk, dtv[k] * sB);
                float gdt = fmaf(xv[k], sB, sw);
                float gz = go[k] * gp * yk;
                // dB, dC: sum over the warp's channels, then one atomic per lane
                if (!act) {
#pragma unroll
                    for (int n = 0; n < 32; ++n) v[n] = 0.f;
                }
                reduce_scatter32(v, lane);
                float *dst = lane < 16 ? dBk + bcrow + (long long)t * 16 + lane
                                       : dCk + bcrow + (long long)t * 16 + (lane - 16);
                atomicAdd(dst, v[0]);
                // per-token gradients of x, delta, z
                float *pp = (DIRS == 3) ? p.part + ((grp * p.L + t) * 3) * 32 + lane : nullptr;
                if (!fin) {
                    pp[0] = gx;
                    pp[32] = gdt;
                    pp[64] = gz;
                } else if (act) {
                    if (DIRS == 3) {
                        gx += __ldcg(pp);
                        gdt += __ldcg(pp + 32);
                        gz += __ldcg(pp + 64);
                    }
                    st_from_f32(static_cast<T *>(p.dx) + row + t, gx);
                    st_from_f32(static_cast<T *>(p.ddelta) + row + t, gdt);
                    if (hasZ) st_from_f32(static_cast<T *>(p.dz) + row + t, gz);
                }
            }
            __syncwarp();
        }
        if (DIRS == 3 && phase == 0) {
            __threadfence();
            __syncwarp();
            if (lane == 0) mbar_arrive(pairbar);
            const bool met = mbar_wait(pairbar, 0, kWaitLimitNs);
            if (!__all_sync(0xffffffffu, met)) {
                if (lane == 0) atomicOr(p.err, kErrTimeout);
                ok = false;
            }
        }
    }
    if (act && ok) {
#pragma unroll
        for (int n = 0; n < 16; ++n) atomicAdd(p.dA[dir] + (long long)d * 16 + n, dA[n]);
        atomicAdd(p.dD[dir] + d, dD);
    }
}

__global__ void zero_f32_kernel(float *p, long long n)
{
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x)
        p[i] = 0.f;
}

}  // namespace vssm
