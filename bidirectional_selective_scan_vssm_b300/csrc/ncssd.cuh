// NC-SSD, the non-causal global-state variant of the VSSD page (§4.2.4,
// §4.2.5: Y = C (B^T (X m))), for sm_103a (B300), N = 16.
//
// What it computes is stated in include/vssm.h (vssm_ncssd): per batch entry
// one hidden state H[n][d] = sum_j m_j B_j[n] x[d][j] shared by all tokens,
// then out[d][t] = (sum_n C_t[n] H[n][d] + D[d] x[d][t]) silu(z[d][t]).
// There is no recurrence: two contractions of depth 16 per element, bound by
// the bytes of x, z and out (6 bytes per element at bf16) once the
// contractions are off the FMA pipe.
//
// Every kernel here is one launch per call: a CTA owns 32 channels of one
// batch entry, sums their part of H, joins the partial sums on chip (warps
// in order, then, with a cluster, its CTAs in rank order through distributed
// shared memory) and writes the outputs. No workspace, no atomics; the sums
// are added in a fixed order, so the result is the same on every run.
//
//  * ncssd_rows_kernel (bf16, 32 whole rows per CTA, L <= 256, dim a
//    multiple of 8): the rows' x, z and out are contiguous spans moved by
//    single bulk copies; both contractions on bf16 tensor-core MMAs.
//  * ncssd_mma_kernel (bf16, any shape): 32 x 32 tiles staged by lanes
//    along tokens; a cluster of Q = 1, 2, 4 or 8 CTAs covers a long row.
//  * ncssd_kernel (fp32 I/O): the same structure on the FMA pipe:
//     1. State. Warps take 32-token tiles in turn. A tile of x is read along
//        tokens (lane = token, coalesced), scaled by m_j and written
//        transposed to shared memory; B_j goes to shared memory as fp32. Then
//        lane = channel: for each token the lane adds x m_j B_j[0..15] (B
//        broadcast) to its 16 fp32 sums in packed f32x2 FMAs.
//     2. Join, as above.
//     3. Output. Lane = token again: the lane holds C_t (16 fp32) and walks
//        the 32 channels, H[:, d] and D[d] broadcast from shared memory,
//        reading x, z and writing out along tokens. x was read moments
//        before by the same CTA, so its second read comes from L2.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"
#include "common.cuh"

namespace vssm {

struct NcssdParams {
    const void *x, *z, *B, *C;
    const float *m, *D;
    void *out;
    unsigned *err;              // device error word (row-resident kernel's bounded wait)
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

// The join: hall = the sum of the kNcW warps' partial sums (part, [kNcW][32][16]
// fp32, written before a __syncthreads) in warp order; with Q > 1 every CTA
// then adds its cluster's CTA sums in rank order through distributed shared
// memory. Ends with __syncthreads. With Q > 1 the caller must pass one more
// cluster_wait() before it exits (the other CTAs may still read its hcta).
template <int Q>
__device__ __forceinline__ void ncssd_join(const float *part, float (&hcta)[32][16],
                                           float (&hall)[32][16])
{
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
    ncssd_join<Q>(part, hcta, hall);

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

// ---- bf16 I/O: both contractions on the tensor cores (warp-level
// mma.m16n8k16, bf16 operands, fp32 accumulators).
//
// The contractions are small (16 states) and sit inside a bandwidth-bound
// kernel; on the FMA pipe they cost 32 fp32 operations per element, which
// binds before the bytes do. Warp-level MMAs take them off the FMA pipe and
// keep every operand where the warp already has it: x tiles in shared memory
// feed ldmatrix directly, C rows feed the B fragments straight from global
// memory, and the accumulator layout (channel pairs x token pairs) is what
// the gate epilogue needs.
//
// Accuracy: x, B and C are bf16 already (exact operands). The two products
// that are not, m_j B_j and H, are split into bf16 hi + lo parts (hi =
// bf16(v), lo = bf16(v - hi)) and each contraction runs once per part, so
// the operands carry about 16 significant bits and the sums are fp32.
//
// Shared-memory tiles are [32 rows][40] bf16 (80-byte pitch: the 8 rows that
// one 8x8 ldmatrix matrix reads fall on distinct banks, and lane-along-row
// 2-byte writes are conflict-free).

constexpr int kNcXP = 40;       // bf16 pitch of an x / z / out tile row (tokens)
constexpr int kNcMP = 24;       // bf16 pitch of an m B row (16 states + 8)

__device__ __forceinline__ void ldsm_x4(const void *p, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_addr(p)));
}
__device__ __forceinline__ void ldsm_x4_t(const void *p, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_addr(p)));
}
// d += a b (16x8x16, bf16 operands, fp32 accumulators)
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w)
{
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
// v as hi + lo, both bf16
__device__ __forceinline__ void split_bf16(float v, unsigned short &hi, unsigned short &lo)
{
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    const __nv_bfloat16 l = __float2bfloat16_rn(v - __bfloat162float(h));
    hi = *reinterpret_cast<const unsigned short *>(&h);
    lo = *reinterpret_cast<const unsigned short *>(&l);
}

template <int Q, bool GATE, bool SKIP>
__global__ void __cluster_dims__(Q, 1, 1) __launch_bounds__(kNcW * 32, 6)
ncssd_mma_kernel(const NcssdParams p)
{
    // per warp: an x tile (then the out tile, in place) and a union of the
    // m B hi/lo tiles (state pass) and the z tile (output pass)
    __shared__ __align__(16) unsigned short xt[kNcW][32][kNcXP];
    __shared__ __align__(16) unsigned short uz[kNcW][2 * 32 * kNcMP];
    __shared__ __align__(16) float hcta[32][16];
    __shared__ __align__(16) float hall[32][16];
    __shared__ __align__(16) unsigned short hb[2][32][kNcMP];        // H hi / lo, [channel][state]
    __shared__ float ds[32];
    static_assert(sizeof(uz) >= kNcW * 32 * 16 * sizeof(float), "the warps' partial sums fit in uz");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int b = blockIdx.z, d0 = blockIdx.y * 32;
    const int ta = min(p.L, (int)blockIdx.x * p.rng), tb = min(p.L, ta + p.rng);
    const int nch = min(32, p.dim - d0), L = p.L;
    const long long row0 = ((long long)b * p.dim + d0) * L;
    const unsigned short *xg = static_cast<const unsigned short *>(p.x) + row0;
    const __nv_bfloat16 *Bg = static_cast<const __nv_bfloat16 *>(p.B) + (long long)b * L * 16;
    const float *mg = p.m + (long long)b * L;
    unsigned short (*xw)[kNcXP] = xt[warp];
    unsigned short (*mw)[kNcMP] = reinterpret_cast<unsigned short (*)[kNcMP]>(uz[warp]);  // [hi 32 | lo 32]
    unsigned short (*zw)[kNcXP] = reinterpret_cast<unsigned short (*)[kNcXP]>(uz[warp]);

    // x tile rows (channels) along tokens t0 .. t0+31, zeros outside
    auto stage = [&](unsigned short (*dst)[kNcXP], const unsigned short *src, int t0, bool tv) {
        const unsigned short *ps = src + t0 + lane;
        if (nch == 32) {
#pragma unroll
            for (int r = 0; r < 32; ++r) dst[r][lane] = tv ? ps[r * L] : (unsigned short)0;
        } else {
#pragma unroll
            for (int r = 0; r < 32; ++r) dst[r][lane] = (tv && r < nch) ? ps[r * L] : (unsigned short)0;
        }
    };

    // ---- 1. state sums: H^T[channel][state] += X[channel][token] (m B)[token][state]
    float acc[2][2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[i][j][k] = 0.f;
    for (int t0 = ta + warp * kNcT; t0 < tb; t0 += kNcW * kNcT) {
        const int t = t0 + lane, len = min(kNcT, tb - t0);
        const bool tv = lane < len;
        {   // this lane's token: m_t B_t as hi / lo rows
            f2 v[8];
            if (tv) load_row16(Bg + (long long)t * 16, v);
            const float mj = tv ? __ldg(mg + t) : 0.f;
            uint32_t hw[8], lw[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float2 a = tv ? unpack2(v[q]) : make_float2(0.f, 0.f);
                unsigned short h0, l0, h1, l1;
                split_bf16(mj * a.x, h0, l0);
                split_bf16(mj * a.y, h1, l1);
                hw[q] = (uint32_t)h0 | ((uint32_t)h1 << 16);
                lw[q] = (uint32_t)l0 | ((uint32_t)l1 << 16);
            }
            uint4 *dh = reinterpret_cast<uint4 *>(&mw[lane][0]);
            uint4 *dl = reinterpret_cast<uint4 *>(&mw[32 + lane][0]);
            dh[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            dh[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
            dl[0] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            dl[1] = make_uint4(lw[4], lw[5], lw[6], lw[7]);
        }
        stage(xw, xg, t0, tv);
        __syncwarp();
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            if (ks * 16 >= len) break;
            uint32_t a[2][4], bh[4], bl[4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) ldsm_x4(&xw[mt * 16 + (lane & 15)][ks * 16 + (lane >> 4) * 8], a[mt]);
            const int kr = ks * 16 + ((lane >> 3) & 1) * 8 + (lane & 7), nc = (lane >> 4) * 8;
            ldsm_x4_t(&mw[kr][nc], bh);
            ldsm_x4_t(&mw[32 + kr][nc], bl);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    mma_bf16(acc[mt][nt], a[mt], bh[2 * nt], bh[2 * nt + 1]);
                    mma_bf16(acc[mt][nt], a[mt], bl[2 * nt], bl[2 * nt + 1]);
                }
        }
        __syncwarp();
    }

    // ---- 2. join
    __syncthreads();                                  // every warp is done with uz
    float *part = reinterpret_cast<float *>(&uz[0][0]);
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            float *q = part + (warp * 32 + mt * 16 + g) * 16 + nt * 8 + 2 * t4;
            *reinterpret_cast<float2 *>(q) = make_float2(acc[mt][nt][0], acc[mt][nt][1]);
            *reinterpret_cast<float2 *>(q + 8 * 16) = make_float2(acc[mt][nt][2], acc[mt][nt][3]);
        }
    if (threadIdx.x < 32) ds[threadIdx.x] = (SKIP && (int)threadIdx.x < nch) ? p.D[d0 + threadIdx.x] : 0.f;
    __syncthreads();
    ncssd_join<Q>(part, hcta, hall);
    for (int e = threadIdx.x; e < 32 * 16; e += kNcW * 32) {
        unsigned short hi, lo;
        split_bf16((&hall[0][0])[e], hi, lo);
        hb[0][e >> 4][e & 15] = hi;
        hb[1][e >> 4][e & 15] = lo;
    }
    __syncthreads();

    // ---- 3. output: Y[channel][token] = H^T[channel][state] C^T[state][token]
    uint32_t ah[2][4], al[2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
        ldsm_x4(&hb[0][mt * 16 + (lane & 15)][(lane >> 4) * 8], ah[mt]);
        ldsm_x4(&hb[1][mt * 16 + (lane & 15)][(lane >> 4) * 8], al[mt]);
    }
    const unsigned short *zg = static_cast<const unsigned short *>(p.z) + row0;
    __nv_bfloat16 *og = static_cast<__nv_bfloat16 *>(p.out) + row0;
    const uint32_t *Cg = reinterpret_cast<const uint32_t *>(static_cast<const __nv_bfloat16 *>(p.C) +
                                                            (long long)b * L * 16);
    float dv[2][2];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
        dv[mt][0] = ds[mt * 16 + g];
        dv[mt][1] = ds[mt * 16 + g + 8];
    }
    for (int t0 = ta + warp * kNcT; t0 < tb; t0 += kNcW * kNcT) {
        const int len = min(kNcT, tb - t0);
        const bool tv = lane < len;
        if (SKIP) stage(xw, xg, t0, tv);
        if (GATE) stage(zw, zg, t0, tv);
        __syncwarp();
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            if (nt * 8 >= len) break;
            const int tok = t0 + nt * 8 + g;
            const bool ok = tok < tb;
            const uint32_t b0 = ok ? __ldg(Cg + (long long)tok * 8 + t4) : 0u;
            const uint32_t b1 = ok ? __ldg(Cg + (long long)tok * 8 + 4 + t4) : 0u;
            const int col = nt * 8 + 2 * t4;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                float d[4] = {0.f, 0.f, 0.f, 0.f};
                mma_bf16(d, ah[mt], b0, b1);
                mma_bf16(d, al[mt], b0, b1);
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {              // rows g and g + 8
                    const int r = mt * 16 + g + 8 * hr;
                    float y0 = d[2 * hr], y1 = d[2 * hr + 1];
                    if (SKIP) {
                        const float2 xv = bf16x2_to_f2(*reinterpret_cast<const uint32_t *>(&xw[r][col]));
                        y0 = fmaf(dv[mt][hr], xv.x, y0);
                        y1 = fmaf(dv[mt][hr], xv.y, y1);
                    }
                    if (GATE) {
                        const float2 zv = bf16x2_to_f2(*reinterpret_cast<const uint32_t *>(&zw[r][col]));
                        y0 *= silu_f32<__nv_bfloat16>(zv.x);
                        y1 *= silu_f32<__nv_bfloat16>(zv.y);
                    }
                    *reinterpret_cast<uint32_t *>(&xw[r][col]) = bf16x2_bits(y0, y1);
                }
            }
        }
        __syncwarp();
        {   // the out tile leaves along tokens
            unsigned short *po = reinterpret_cast<unsigned short *>(og) + t0 + lane;
            if (tv) {
                if (nch == 32) {
#pragma unroll
                    for (int r = 0; r < 32; ++r) po[r * L] = xw[r][lane];
                } else {
                    for (int r = 0; r < nch; ++r) po[r * L] = xw[r][lane];
                }
            }
        }
        __syncwarp();
    }
    __syncwarp();
    if (Q > 1) cluster_wait();                        // no CTA leaves while its hcta is read
}

// ---- bf16 I/O, short rows: whole rows resident in shared memory.
//
// A CTA owns 32 whole rows (channels) of one batch entry. Their x, z and out
// are then three contiguous spans of 32 L elements, 16-byte aligned when dim
// is a multiple of 8, so each span moves as ONE bulk copy (cp.async.bulk,
// completion on an mbarrier; the out span leaves the same way). x is read
// from HBM once for both contractions and no thread spends instructions on
// staging. While the spans are in flight every lane already loads what it
// will need from global memory (B, m and the C fragments of its tiles, at
// most two 32-token tiles per warp), so that no load latency remains on the
// path once the spans have landed.
//
// The spans keep the global layout (row c at element c L, misaligned for odd
// L), so the MMA fragments and the epilogue gather token pairs with 16-bit
// shared loads. The output is written over x in place (each element by the
// thread that read it), then the x span is stored as the out span.

constexpr int kNcRowsTiles = 2;                       // 32-token tiles per warp at most
constexpr int kNcRowsMaxL = kNcW * kNcT * kNcRowsTiles;
constexpr int kNcPad = 64;            // bf16 elements after the last row (read, masked, never written)

struct NcRowsLayout {
    int sx, oZ, oM, oHB, oD, oBar, total;
    __host__ __device__ NcRowsLayout(int L, bool gate)
    {
        sx = ((32 * L + kNcPad) * 2 + 15) / 16 * 16;      // one span buffer
        oZ = sx;
        oM = oZ + (gate ? sx : 0);
        oHB = oM + kNcW * 2 * 16 * kNcMP * 2;            // m B rows of one 16-token step per warp
        oD = oHB + 2 * 32 * kNcMP * 2;
        oBar = oD + 32 * 4;
        total = oBar + 16;                                 // two mbarriers: x, z
    }
};

// bf16 pair (row-relative element i, i + 1) of a span in shared memory
__device__ __forceinline__ uint32_t lds_pair(const unsigned short *s, int i)
{
    return (uint32_t)s[i] | ((uint32_t)s[i + 1] << 16);
}

template <bool GATE, bool SKIP>
__global__ void __launch_bounds__(kNcW * 32, 6) ncssd_rows_kernel(const NcssdParams p)
{
    extern __shared__ __align__(128) unsigned char nsm[];
    const int L = p.L;
    const NcRowsLayout lay(L, GATE);
    unsigned short *xr = reinterpret_cast<unsigned short *>(nsm);
    const unsigned short *zr = reinterpret_cast<const unsigned short *>(nsm + lay.oZ);
    unsigned short (*hb)[32][kNcMP] = reinterpret_cast<unsigned short (*)[32][kNcMP]>(nsm + lay.oHB);
    float *ds = reinterpret_cast<float *>(nsm + lay.oD);
    uint64_t *bar = reinterpret_cast<uint64_t *>(nsm + lay.oBar);
    // the warps' partial sums, [kNcW][32][16] fp32, over the m B rows and hb
    float *part = reinterpret_cast<float *>(nsm + lay.oM);
    static_assert(kNcW * 2 * 16 * kNcMP * 2 + 2 * 32 * kNcMP * 2 >= kNcW * 32 * 16 * 4, "part fits");
    __shared__ int s_ok;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int b = blockIdx.z, d0 = blockIdx.y * 32;
    const int nch = min(32, p.dim - d0);
    const long long row0 = ((long long)b * p.dim + d0) * L;
    const uint32_t span = (uint32_t)nch * L * 2;                 // bytes, a multiple of 16
    unsigned short (*mw)[kNcMP] =
        reinterpret_cast<unsigned short (*)[kNcMP]>(nsm + lay.oM + warp * 2 * 16 * kNcMP * 2);

    if (threadIdx.x == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {                            // x on bar[0] (state pass), z on bar[1] (output)
        mbar_expect_tx(&bar[0], span);
        bulk_g2s(xr, static_cast<const __nv_bfloat16 *>(p.x) + row0, span, &bar[0]);
        mbar_arrive(&bar[0]);
        if (GATE) {
            mbar_expect_tx(&bar[1], span);
            bulk_g2s(nsm + lay.oZ, static_cast<const __nv_bfloat16 *>(p.z) + row0, span, &bar[1]);
            mbar_arrive(&bar[1]);
        }
    }

    // while the spans fly: B_t, m_t of this lane's tokens, and the C fragments
    const __nv_bfloat16 *Bg = static_cast<const __nv_bfloat16 *>(p.B) + (long long)b * L * 16;
    const uint32_t *Cg = reinterpret_cast<const uint32_t *>(static_cast<const __nv_bfloat16 *>(p.C) +
                                                            (long long)b * L * 16);
    uint4 braw[kNcRowsTiles][2];
    float mj[kNcRowsTiles];
    uint32_t cf[kNcRowsTiles][4][2];
#pragma unroll
    for (int k = 0; k < kNcRowsTiles; ++k) {
        const int t0 = warp * kNcT + k * kNcW * kNcT, t = t0 + lane;
        const bool tv = t < L;
        const uint4 *src = reinterpret_cast<const uint4 *>(Bg + (long long)t * 16);
        braw[k][0] = tv ? __ldg(src) : make_uint4(0u, 0u, 0u, 0u);
        braw[k][1] = tv ? __ldg(src + 1) : make_uint4(0u, 0u, 0u, 0u);
        mj[k] = tv ? __ldg(p.m + (long long)b * L + t) : 0.f;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const int tok = t0 + nt * 8 + g;
            const bool ok = tok < L;
            cf[k][nt][0] = ok ? __ldg(Cg + (long long)tok * 8 + t4) : 0u;
            cf[k][nt][1] = ok ? __ldg(Cg + (long long)tok * 8 + 4 + t4) : 0u;
        }
    }
    if (threadIdx.x < 32) ds[threadIdx.x] = (SKIP && (int)threadIdx.x < nch) ? p.D[d0 + threadIdx.x] : 0.f;
    // thread 0 waits (bounded) for barrier i; on expiry the CTA stops after
    // waiting once more for each copy still in flight
    auto landed = [&](int i) {
        if (threadIdx.x == 0) {
            const bool met = mbar_wait(&bar[i], 0, kWaitLimitNs);
            if (!met) {
                atomicOr(p.err, kErrTimeout);
                for (int j = i; j < (GATE ? 2 : 1); ++j) mbar_wait(&bar[j], 0, kWaitLimitNs);
            }
            s_ok = met ? 1 : 0;
        }
        __syncthreads();
        return s_ok != 0;                              // CTA-uniform
    };
    if (!landed(0)) return;

    // ---- 1. state sums: H^T[channel][state] += X[channel][token] (m B)[token][state]
    float acc[2][2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[i][j][q] = 0.f;
#pragma unroll
    for (int k = 0; k < kNcRowsTiles; ++k) {
        const int t0 = warp * kNcT + k * kNcW * kNcT;
        if (t0 >= L) break;
        const int len = min(kNcT, L - t0);
        // this lane's token: m_t B_t as hi / lo rows (zeros past the row)
        const uint32_t w[8] = {braw[k][0].x, braw[k][0].y, braw[k][0].z, braw[k][0].w,
                               braw[k][1].x, braw[k][1].y, braw[k][1].z, braw[k][1].w};
        uint32_t hw[8], lw[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float2 a = bf16x2_to_f2(w[q]);
            unsigned short h0, l0, h1, l1;
            split_bf16(mj[k] * a.x, h0, l0);
            split_bf16(mj[k] * a.y, h1, l1);
            hw[q] = (uint32_t)h0 | ((uint32_t)h1 << 16);
            lw[q] = (uint32_t)l0 | ((uint32_t)l1 << 16);
        }
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            if (ks * 16 >= len) break;
            if ((lane >> 4) == ks) {                   // the step's 16 tokens: rows hi 0..15, lo 16..31
                uint4 *dh = reinterpret_cast<uint4 *>(&mw[lane & 15][0]);
                uint4 *dl = reinterpret_cast<uint4 *>(&mw[16 + (lane & 15)][0]);
                dh[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                dh[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
                dl[0] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                dl[1] = make_uint4(lw[4], lw[5], lw[6], lw[7]);
            }
            __syncwarp();
            uint32_t a[2][4], bh[4], bl[4];
            const int c0 = t0 + ks * 16 + 2 * t4;
            // a token pair at or past the row's end reads the next row: keep
            // only the row's own tokens (so that a non-finite value there
            // cannot meet a zero weight)
            const uint32_t m0 = c0 + 1 < L ? 0xffffffffu : (c0 < L ? 0xffffu : 0u);
            const uint32_t m8 = c0 + 9 < L ? 0xffffffffu : (c0 + 8 < L ? 0xffffu : 0u);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const int e = (mt * 16 + g) * L + c0;
                a[mt][0] = lds_pair(xr, e) & m0;
                a[mt][1] = lds_pair(xr, e + 8 * L) & m0;
                a[mt][2] = lds_pair(xr, e + 8) & m8;
                a[mt][3] = lds_pair(xr, e + 8 * L + 8) & m8;
            }
            const int kr = ((lane >> 3) & 1) * 8 + (lane & 7), nc = (lane >> 4) * 8;
            ldsm_x4_t(&mw[kr][nc], bh);
            ldsm_x4_t(&mw[16 + kr][nc], bl);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    mma_bf16(acc[mt][nt], a[mt], bh[2 * nt], bh[2 * nt + 1]);
                    mma_bf16(acc[mt][nt], a[mt], bl[2 * nt], bl[2 * nt + 1]);
                }
            __syncwarp();                              // the rows are read before the next step's
        }
    }

    // ---- 2. join: the warps' sums in warp order, as bf16 hi / lo
    __syncthreads();                                   // every warp is done with its m B tiles
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            float *q = part + (warp * 32 + mt * 16 + g) * 16 + nt * 8 + 2 * t4;
            *reinterpret_cast<float2 *>(q) = make_float2(acc[mt][nt][0], acc[mt][nt][1]);
            *reinterpret_cast<float2 *>(q + 8 * 16) = make_float2(acc[mt][nt][2], acc[mt][nt][3]);
        }
    __syncthreads();
    constexpr int kPer = 32 * 16 / (kNcW * 32);
    float hs[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int e = threadIdx.x + i * kNcW * 32;
        hs[i] = 0.f;
#pragma unroll
        for (int w = 0; w < kNcW; ++w) hs[i] += part[w * 32 * 16 + e];
    }
    __syncthreads();                                   // hb overlaps part
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int e = threadIdx.x + i * kNcW * 32;
        unsigned short hi, lo;
        split_bf16(hs[i], hi, lo);
        hb[0][e >> 4][e & 15] = hi;
        hb[1][e >> 4][e & 15] = lo;
    }
    __syncthreads();

    // ---- 3. output: Y[channel][token] = H^T[channel][state] C^T[state][token], over x in place
    if (GATE && !landed(1)) return;
    uint32_t ah[2][4], al[2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
        ldsm_x4(&hb[0][mt * 16 + (lane & 15)][(lane >> 4) * 8], ah[mt]);
        ldsm_x4(&hb[1][mt * 16 + (lane & 15)][(lane >> 4) * 8], al[mt]);
    }
    f2 dv[2][2];                                       // (D, D) of rows g, g + 8 of each m tile
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
        dv[mt][0] = pack2(ds[mt * 16 + g], ds[mt * 16 + g]);
        dv[mt][1] = pack2(ds[mt * 16 + g + 8], ds[mt * 16 + g + 8]);
    }
    const f2 half2 = pack2(0.5f, 0.5f);
    auto f32_of = [](unsigned short v) { return __uint_as_float((uint32_t)v << 16); };
#pragma unroll
    for (int k = 0; k < kNcRowsTiles; ++k) {
        const int t0 = warp * kNcT + k * kNcW * kNcT;
        if (t0 >= L) break;
        const int len = min(kNcT, L - t0);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            if (nt * 8 >= len) break;
            const int col = t0 + nt * 8 + 2 * t4;     // this thread's token pair
            const bool w0 = col < L, w1 = col + 1 < L;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                float d[4] = {0.f, 0.f, 0.f, 0.f};
                mma_bf16(d, ah[mt], cf[k][nt][0], cf[k][nt][1]);
                mma_bf16(d, al[mt], cf[k][nt][0], cf[k][nt][1]);
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int r = mt * 16 + g + 8 * hr;
                    const int e = r * L + col;
                    // the pair in packed f32x2: y + D x, then y silu(z) with
                    // silu(z) = h + h tanh(h), h = z / 2 (as silu_f32 for bf16)
                    f2 y = pack2(d[2 * hr], d[2 * hr + 1]);
                    if (SKIP) y = fma2(dv[mt][hr], pack2(f32_of(xr[e]), f32_of(xr[e + 1])), y);
                    if (GATE) {
                        const f2 h = mul2(pack2(f32_of(zr[e]), f32_of(zr[e + 1])), half2);
                        const float2 hv = unpack2(h);
                        y = mul2(y, fma2(h, pack2(tanh_mufu(hv.x), tanh_mufu(hv.y)), h));
                    }
                    const float2 yv = unpack2(y);
                    const uint32_t o = bf16x2_bits(yv.x, yv.y);
                    if (w0) xr[e] = (unsigned short)(o & 0xffffu);
                    if (w1) xr[e + 1] = (unsigned short)(o >> 16);
                }
            }
        }
    }
    fence_proxy_async_smem();                          // the in-place output, before the bulk read
    __syncthreads();
    if (threadIdx.x == 0) {
        bulk_s2g(static_cast<__nv_bfloat16 *>(p.out) + row0, xr, span);
        bulk_commit();
        bulk_wait_read();                              // the span is read before the CTA leaves
    }
}

}  // namespace vssm
