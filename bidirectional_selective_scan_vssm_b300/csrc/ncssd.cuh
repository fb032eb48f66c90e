// NC-SSD, the non-causal global-state variant of the VSSD page (§4.2.4,
// §4.2.5: Y = C (B^T (X m))), for sm_103a (B300), N = 16.
//
// What it computes is stated in include/vssm.h (vssm_ncssd): per batch entry
// one hidden state H[n][d] = sum_j m_j B_j[n] x[d][j] shared by all tokens,
// then out[d][t] = (sum_n C_t[n] H[n][d] + D[d] x[d][t]) silu(z[d][t]).
// There is no recurrence: two contractions of depth 16 per element, bound by
// the bytes of x, z and out and by the FMA pipe about equally.
//
// One kernel, ncssd_kernel. A CTA of four warps owns 32 channels of one batch
// entry over a token range; a thread-block cluster of Q CTAs (Q = 1, 2, 4 or
// 8) covers the whole row, so that rows that are few and long still fill the
// GPU.
//
//  1. State. Warps take 32-token tiles in turn. A tile of x is read along
//     tokens (lane = token, coalesced), scaled by m_j and written transposed
//     to shared memory; B_j goes to shared memory as fp32. Then lane = channel:
//     for each token the lane adds x m_j B_j[0..15] (B broadcast) to its 16
//     fp32 sums in packed f32x2 FMAs.
//  2. Join. The four warps' sums are added in shared memory in warp order;
//     with Q > 1 every CTA then adds the Q CTA sums of its cluster in rank
//     order through distributed shared memory. The order is fixed, so H is
//     the same on every run.
//  3. Output. Lane = token again: the lane holds C_t (16 fp32) and walks the
//     32 channels, H[:, d] and D[d] broadcast from shared memory, reading x,
//     z and writing out along tokens. x was read moments before by the same
//     CTA, so its second read comes from L2.
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
    int batch, dim, L, rng;     // rng: tokens per CTA of a cluster
};

constexpr int kNcW = 4;         // warps per CTA
constexpr int kNcT = 32;        // tokens per tile
constexpr int kNcBP = 20;       // fp32 pitch of a staged B row (80 bytes: 16-byte aligned,
                                // and eight consecutive rows cover all 32 banks)
constexpr int kNcMaxQ = 8;      // CTAs per cluster at most (the portable limit)
constexpr int kNcU = 8;         // channels whose loads are in flight together (output)

// 16 values of a B or C row (16-byte aligned) as fp32 pairs.
__device__ __forceinline__ void load_row16(const float *src, f2 (&v)[8])
{
    const float4 *s = reinterpret_cast<const float4 *>(src);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 a = __ldg(s + q);
        v[2 * q] = pack2(a.x, a.y);
        v[2 * q + 1] = pack2(a.z, a.w);
    }
}
__device__ __forceinline__ void load_row16(const __nv_bfloat16 *src, f2 (&v)[8])
{
    const uint4 *s = reinterpret_cast<const uint4 *>(src);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const uint4 a = __ldg(s + q);
        v[4 * q + 0] = pack2(__uint_as_float(a.x << 16), __uint_as_float(a.x & 0xffff0000u));
        v[4 * q + 1] = pack2(__uint_as_float(a.y << 16), __uint_as_float(a.y & 0xffff0000u));
        v[4 * q + 2] = pack2(__uint_as_float(a.z << 16), __uint_as_float(a.z & 0xffff0000u));
        v[4 * q + 3] = pack2(__uint_as_float(a.w << 16), __uint_as_float(a.w & 0xffff0000u));
    }
}

__device__ __forceinline__ void cluster_arrive()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// fp32 at shared address `a` of cluster CTA `rank`.
__device__ __forceinline__ float ld_cluster_f32(uint32_t a, uint32_t rank)
{
    uint32_t ra;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
    return v;
}

// Output of one token (this lane's) for the CTA's channels: C_t in c, H and
// D in shared memory, x, z, out along the rows at px, pz, po (stride L).
// FULL: all 32 channels exist, so no channel checks.
template <typename T, bool GATE, bool SKIP, bool FULL>
__device__ __forceinline__ void ncssd_token_out(const f2 (&c)[8], const T *px, const T *pz, T *po,
                                                int L, int nch, const float (&hall)[32][16],
                                                const float (&ds)[32])
{
#pragma unroll 1
    for (int r0 = 0; r0 < (FULL ? 32 : nch); r0 += kNcU) {
        float xv[kNcU], zv[kNcU];
#pragma unroll
        for (int k = 0; k < kNcU; ++k) {
            const bool ok = FULL || r0 + k < nch;
            xv[k] = (SKIP && ok) ? ld_as_f32(px + k * L) : 0.f;
            zv[k] = (GATE && ok) ? ld_as_f32(pz + k * L) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < kNcU; ++k) {
            const int r = r0 + k;
            if (FULL || r < nch) {
                f2 acc = pack2(0.f, 0.f), acc2 = pack2(0.f, 0.f);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    f2 h0, h1;
                    lds_2xf2(&hall[r][4 * q], h0, h1);
                    acc = fma2(c[2 * q], h0, acc);
                    acc2 = fma2(c[2 * q + 1], h1, acc2);
                }
                const float2 a = unpack2(add2(acc, acc2));
                float y = a.x + a.y;
                if (SKIP) y = fmaf(ds[r], xv[k], y);
                if (GATE) y *= silu_f32<T>(zv[k]);
                st_from_f32(po + k * L, y);
            }
        }
        px += kNcU * L;
        pz += kNcU * L;
        po += kNcU * L;
    }
}

// Q: CTAs per cluster, fixed at compile time so that a launch cannot run the
// cluster code without its cluster. GATE: z is given; SKIP: D is given.
template <typename T, int Q, bool GATE, bool SKIP>
__global__ void __cluster_dims__(Q, 1, 1) __launch_bounds__(kNcW * 32, 5) ncssd_kernel(const NcssdParams p)
{
    __shared__ float xs[kNcW][kNcT][33];                     // m_j x[c][j]: [token][channel]
    __shared__ __align__(16) float bs[kNcW][kNcT][kNcBP];    // B_j fp32; later the warps' sums
    __shared__ __align__(16) float hcta[32][16];             // this CTA's sum
    __shared__ __align__(16) float hall[32][16];             // the row's H
    __shared__ float ds[32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, d0 = blockIdx.y * 32;
    const int ta = min(p.L, (int)blockIdx.x * p.rng), tb = min(p.L, ta + p.rng);
    const int nch = min(32, p.dim - d0), L = p.L;
    const long long row0 = ((long long)b * p.dim + d0) * L;     // the CTA's first row
    const T *xg = static_cast<const T *>(p.x) + row0;
    const T *Bg = static_cast<const T *>(p.B) + (long long)b * L * 16;
    const float *mg = p.m + (long long)b * L;

    // ---- 1. state sums, lane = channel
    f2 h[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) h[q] = pack2(0.f, 0.f);
    for (int t0 = ta + warp * kNcT; t0 < tb; t0 += kNcW * kNcT) {
        const int t = t0 + lane, len = min(kNcT, tb - t0);
        const bool tv = lane < len;
        {   // B_t as fp32 (zeros past the range, so that whole groups of 8 tokens can run)
            f2 v[8];
            if (tv) load_row16(Bg + (long long)t * 16, v);
            float4 *dst = reinterpret_cast<float4 *>(&bs[warp][lane][0]);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 a = tv ? unpack2(v[2 * q]) : make_float2(0.f, 0.f);
                const float2 c = tv ? unpack2(v[2 * q + 1]) : make_float2(0.f, 0.f);
                dst[q] = make_float4(a.x, a.y, c.x, c.y);
            }
        }
        const float mj = tv ? __ldg(mg + t) : 0.f;
        float xv[32];
        const T *px = xg + t;
        if (nch == 32) {
#pragma unroll
            for (int r = 0; r < 32; ++r) xv[r] = tv ? ld_as_f32(px + r * L) : 0.f;
        } else {
#pragma unroll
            for (int r = 0; r < 32; ++r) xv[r] = (tv && r < nch) ? ld_as_f32(px + r * L) : 0.f;
        }
#pragma unroll
        for (int r = 0; r < 32; ++r) xs[warp][lane][r] = mj * xv[r];
        __syncwarp();
        for (int j0 = 0; j0 < len; j0 += 8) {
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int j = j0 + jj;
                const float u = xs[warp][j][lane];
                const f2 uu = pack2(u, u);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    f2 b0, b1;
                    lds_2xf2(&bs[warp][j][4 * q], b0, b1);
                    h[2 * q] = fma2(uu, b0, h[2 * q]);
                    h[2 * q + 1] = fma2(uu, b1, h[2 * q + 1]);
                }
            }
        }
        __syncwarp();
    }

    // ---- 2. join: warps in order, then the cluster's CTAs in rank order
    __syncthreads();                                  // every warp is done with bs
    float *part = &bs[0][0][0];                       // [kNcW][32][16] fits in bs
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float2 a = unpack2(h[q]);
        part[(warp * 32 + lane) * 16 + 2 * q] = a.x;
        part[(warp * 32 + lane) * 16 + 2 * q + 1] = a.y;
    }
    if (threadIdx.x < 32) ds[threadIdx.x] = (SKIP && (int)threadIdx.x < nch) ? p.D[d0 + threadIdx.x] : 0.f;
    __syncthreads();
    for (int e = threadIdx.x; e < 32 * 16; e += kNcW * 32) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kNcW; ++w) s += part[w * 32 * 16 + e];
        (Q > 1 ? &hcta[0][0] : &hall[0][0])[e] = s;
    }
    if (Q > 1) {
        cluster_arrive();                             // hcta of every CTA is written
        cluster_wait();
        const uint32_t a0 = smem_addr(&hcta[0][0]);
        for (int e = threadIdx.x; e < 32 * 16; e += kNcW * 32) {
            float s = 0.f;
#pragma unroll
            for (int r = 0; r < Q; ++r) s += ld_cluster_f32(a0 + 4u * e, (uint32_t)r);
            (&hall[0][0])[e] = s;
        }
        cluster_arrive();                             // done reading the others' hcta
    }
    __syncthreads();

    // ---- 3. output, lane = token
    const T *zg = static_cast<const T *>(p.z) + row0;
    T *og = static_cast<T *>(p.out) + row0;
    const T *Cg = static_cast<const T *>(p.C) + (long long)b * L * 16;
    for (int t0 = ta + warp * kNcT; t0 < tb; t0 += kNcW * kNcT) {
        const int t = t0 + lane;
        if (t < tb) {
            f2 c[8];
            load_row16(Cg + (long long)t * 16, c);
            if (nch == 32)
                ncssd_token_out<T, GATE, SKIP, true>(c, xg + t, zg + t, og + t, L, nch, hall, ds);
            else
                ncssd_token_out<T, GATE, SKIP, false>(c, xg + t, zg + t, og + t, L, nch, hall, ds);
        }
    }
    __syncwarp();
    if (Q > 1) cluster_wait();                        // no CTA leaves while its hcta is read
}

}  // namespace vssm
