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
//    chunk of kTG tokens (in that direction's scan order) to a checkpoint
//    buffer.
//  * grad_adjoint_kernel: the two directions of a channel group are a warp
//    pair that meets in the middle, as in the forward kernel but walking
//    against the scan orders: the forward direction's adjoint walks the
//    chunks downward, the backward one upward. Per chunk a warp recomputes
//    the chunk's states from its checkpoint into shared memory (fp32, one
//    slot per token), then walks the chunk backward through the adjoint.
//    In phase 0 each warp leaves its fp32 partial dx, ddelta, dz for its half
//    in the workspace; after a bounded rendezvous, phase 1 adds the
//    partner's partials and writes the gradients. dB and dC are reduced
//    over the warp's 32 channels through shared memory (each lane writes its
//    32 contributions as a row, then sums one column) and added to global
//    memory atomically, one value per lane and token; dA and dD accumulate
//    in registers over the row and are added at the end. The state and B/C
//    arithmetic runs on packed f32x2 instructions.
//
// The only wait on another warp is the pair rendezvous (bounded, as in the
// forward kernel).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"
#include "common.cuh"

namespace vssm {

#ifndef VSSM_GRAD_CHUNK
#define VSSM_GRAD_CHUNK 4
#endif
constexpr int kTG = VSSM_GRAD_CHUNK;     // tokens per gradient chunk

struct GradParams {
    const void *x, *delta, *z, *dout;
    const void *B[2], *C[2];
    const float *A[2], *D[2];
    void *dx, *ddelta, *dz;
    float *dB[2], *dC[2];               // [1] == [0] when the directions share B / C
    float *dA[2], *dD[2];
    float *ckpt;                        // [slot][ngroups][nch][16][32]
    float *part;                        // [ngroups][L][3][32] (both directions only)
    float *summ;                        // [slot][ngroups][nrange][P 16 | q 16][32] when ranges are
                                        // joined by summaries; null when uncut or independent
    unsigned *err;
    int batch, dim, L, seg_len, rgroups, nch;
    int nrange, rch;                    // token ranges per row, chunks per range
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

// Staging of the checkpoint pass and of the adjoint summaries: per warp a
// two-stage ring of kSC-token chunks; each lane copies the 16-byte blocks that
// cover its own row's span of the inputs it walks (delta and x, or delta,
// dout and z) into row slots, and the chunk's B or C rows are copied one block
// per lane, so that no load in the walk touches more than one line per lane
// and token.
template <typename T>
struct SummLayout {
    static constexpr int kSC = 16;                                  // tokens per chunk
    static constexpr int ES = (int)sizeof(T);
    static constexpr int SLOT = ((16 - ES) + kSC * ES + 15) / 16 * 16;
    static constexpr int ROWS = 32 * SLOT + 16 * 3;                // one array's 32 rows
    __device__ static constexpr int row_off(int a, int r) { return a * ROWS + r * SLOT + 16 * (r >> 3); }
    static constexpr int sC = 3 * ROWS;
    static constexpr int kStage = (sC + kSC * 16 * ES + 15) / 16 * 16;
    static constexpr int kWarpBytes = 2 * kStage;
};

// Checkpoints: the state entering each kTG-token chunk in this direction's
// scan order. One warp per (direction, group) walks the whole row; when the
// ranges are independent (folded rows cut at segment starts, no summaries)
// one warp per (direction, group, range) walks its range from zero, which is
// exact because the range starts on a reset in either direction.
template <typename T, int DIRS>
__global__ void __launch_bounds__(128) grad_ckpt_kernel(const GradParams p)
{
    constexpr int NDIR = (DIRS == 3) ? 2 : 1;
    const int lane = threadIdx.x & 31;
    const int nr = p.summ ? 1 : p.nrange;             // walks per row
    const long long uu = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (uu >= (long long)NDIR * p.ngroups * nr) return;
    const int rr = (int)(uu % nr);
    const long long u = uu / nr;
    const int clo = nr > 1 ? rr * p.rch : 0, chi = nr > 1 ? min(p.nch, clo + p.rch) : p.nch;
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
    float *ck = p.ckpt + ((long long)slot * p.ngroups + grp) * p.nch * 512 + lane;
    // the walk over tokens [T0, T1) in scan order, in staged chunks of kSC
    // tokens (the inputs' row spans as 16-byte blocks into a two-stage ring,
    // as in grad_adj_summary_kernel); the state is stored before the first
    // token, in scan order, of every kTG-token chunk
    using Lay = SummLayout<T>;
    constexpr int kSC = Lay::kSC, ES = Lay::ES;
    extern __shared__ __align__(128) unsigned char csm[];
    unsigned char *wsm = csm + (threadIdx.x >> 5) * Lay::kWarpBytes;
    const long long total = (long long)p.batch * p.dim * p.L;
    const long long erow = ((long long)b * p.dim + (act ? d : d0)) * p.L;
    const T *Bg = static_cast<const T *>(p.B[dir]) + (long long)b * p.L * 16;
    const void *arr[2] = {p.delta, p.x};
    if (!act) {   // an idle lane's row slots are never copied into: zero them once
        for (int st = 0; st < 2; ++st)
            for (int a = 0; a < 2; ++a) {
                uint4 *r = reinterpret_cast<uint4 *>(wsm + st * Lay::kStage + Lay::row_off(a, lane));
                for (int k = 0; k < Lay::SLOT / 16; ++k) r[k] = make_uint4(0u, 0u, 0u, 0u);
            }
    }
    const int T0 = clo * kTG, T1 = min(p.L, chi * kTG);
    const int nc = (T1 - T0 + kSC - 1) / kSC;
    auto span = [&](int c, int &c0, int &c1) {
        if (dir == 0) {
            c0 = T0 + c * kSC;
            c1 = min(T1, c0 + kSC);
        } else {
            c1 = T1 - c * kSC;
            c0 = max(T0, c1 - kSC);
        }
    };
    auto issue = [&](int st, int c) {
        unsigned char *sg = wsm + st * Lay::kStage;
        int c0, c1;
        span(c, c0, c1);
        const int len = c1 - c0;
        if (act) {
            const uint32_t lead = (uint32_t)(((erow + c0) * ES) & 15);
            const int nblk = (int)((lead + (uint32_t)(len * ES) + 15u) >> 4);
            const long long avail = (total - erow - c0) * ES + lead;
            const long long off = (long long)c0 * ES - lead;
            for (int a = 0; a < 2; ++a) {
                const char *src = static_cast<const char *>(arr[a]) + erow * ES + off;
                unsigned char *dst = sg + Lay::row_off(a, lane);
                for (int k = 0; k < nblk; ++k) {
                    const long long rem = avail - 16 * k;
                    cp_async16(dst + 16 * k, src + 16 * k, rem >= 16 ? 16u : (uint32_t)rem);
                }
            }
        }
        const int nb = len * ES;                                    // 16-byte blocks of B rows
        const char *srcB = reinterpret_cast<const char *>(Bg + (long long)c0 * 16);
#pragma unroll
        for (int m = 0; m < (kSC * ES + 31) / 32; ++m) {
            const int jj = lane + 32 * m;
            cp_async16_if(sg + Lay::sC + 16 * jj, srcB + 16 * jj, jj < nb);
        }
        cp_async_commit();
    };
    for (int c = 0; c < 2; ++c) {
        if (c < nc) issue(c, c);
        else cp_async_commit();
    }
    for (int c = 0; c < nc; ++c) {
        const int st = c & 1;
        const unsigned char *sg = wsm + st * Lay::kStage;
        int c0, c1;
        span(c, c0, c1);
        const int len = c1 - c0;
        cp_async_wait<1>();
        __syncwarp();
        const uint32_t lead = (uint32_t)(((erow + c0) * ES) & 15);
        const T *rdt = reinterpret_cast<const T *>(sg + Lay::row_off(0, lane) + lead);
        const T *rx = reinterpret_cast<const T *>(sg + Lay::row_off(1, lane) + lead);
        const T *bs = reinterpret_cast<const T *>(sg + Lay::sC);
#pragma unroll 2
        for (int k = 0; k < len; ++k) {
            const int i = dir == 0 ? k : len - 1 - k;               // scan order
            const int t = c0 + i;
            const bool first = dir == 0 ? (t % kTG) == 0 : ((t % kTG) == kTG - 1 || t == p.L - 1);
            if (first) {
                float *cj = ck + (long long)(t / kTG) * 512;
#pragma unroll
                for (int n = 0; n < 16; ++n) cj[n * 32] = h[n];
            }
            const bool rs = reset_at(t, p.seg_len, dir);
            const float dt = ld_as_f32(rdt + i);
            const float ux = dt * ld_as_f32(rx + i);
            float Bv[16];
            load16_f32(bs + i * 16, Bv);
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                const float a = rs ? 0.f : ex2_mufu(dt * Al2[n]);
                h[n] = fmaf(a, h[n], ux * Bv[n]);
            }
        }
        __syncwarp();                                               // the stage is read
        if (c + 2 < nc) issue(st, c + 2);
        else cp_async_commit();
    }
    cp_async_wait<0>();
}


// Adjoint range summaries, for rows cut into nrange ranges of rch chunks. The
// adjoint of a direction runs against its scan order, l_t = ds_t C_t + lam
// and then lam = a_t l_t (a_t = exp(delta_t A), 0 at a folded reset), so a
// range walked from an incoming lam hands lam_out = P lam + q to the next
// range in walk order, with P = prod(a_t) over the range (exp(A sum(delta)),
// or 0 across a reset) and q the hand-over of the walk from lam = 0. These
// maps compose associatively, exactly as the forward range summaries; one
// warp per (direction, group, range) stores (P, q) for the adjoint kernel's
// start-up fold.
template <typename T, int DIRS>
__global__ void __launch_bounds__(128) grad_adj_summary_kernel(const GradParams p)
{
    using Lay = SummLayout<T>;
    constexpr int NDIR = (DIRS == 3) ? 2 : 1;
    constexpr int kSC = Lay::kSC, ES = Lay::ES;
    constexpr float kLog2e = 1.4426950408889634f;
    extern __shared__ __align__(128) unsigned char ssm[];
    const int lane = threadIdx.x & 31;
    unsigned char *wsm = ssm + (threadIdx.x >> 5) * Lay::kWarpBytes;
    const long long u = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (u >= (long long)NDIR * p.ngroups * p.nrange) return;
    const int rr = (int)(u % p.nrange);
    const long long gu = u / p.nrange;
    const int slot = (int)(gu / p.ngroups);
    const long long grp = gu % p.ngroups;
    const int dir = (DIRS == 3) ? slot : (DIRS == 1 ? 0 : 1);
    const int b = (int)(grp / p.rgroups), d0 = (int)(grp % p.rgroups) * 32;
    const int d = d0 + lane;
    const bool act = d < p.dim;
    const int ta = min(p.L, rr * p.rch * kTG), tb = min(p.L, (rr + 1) * p.rch * kTG);
    float Al2[16], lam[16];
#pragma unroll
    for (int n = 0; n < 16; ++n) {
        Al2[n] = act ? p.A[dir][(long long)d * 16 + n] * kLog2e : 0.f;
        lam[n] = 0.f;
    }
    const long long total = (long long)p.batch * p.dim * p.L;
    const long long erow = ((long long)b * p.dim + (act ? d : d0)) * p.L;   // element of (b, d, 0)
    const T *Cb = static_cast<const T *>(p.C[dir]) + (long long)b * p.L * 16;
    const bool hasZ = p.z != nullptr;
    const void *arr[3] = {p.delta, p.dout, hasZ ? p.z : p.delta};
    if (!act) {   // an idle lane's row slots are never copied into: zero them once
        for (int st = 0; st < 2; ++st)
            for (int a = 0; a < 3; ++a) {
                uint4 *r = reinterpret_cast<uint4 *>(wsm + st * Lay::kStage + Lay::row_off(a, lane));
                for (int k = 0; k < Lay::SLOT / 16; ++k) r[k] = make_uint4(0u, 0u, 0u, 0u);
            }
    }
    // chunk c of the walk (against the scan order) covers tokens [c0, c1)
    const int n = tb - ta, nc = (n + kSC - 1) / kSC;
    auto span = [&](int c, int &c0, int &c1) {
        if (dir == 0) {
            c1 = tb - c * kSC;
            c0 = max(ta, c1 - kSC);
        } else {
            c0 = ta + c * kSC;
            c1 = min(tb, c0 + kSC);
        }
    };
    auto issue = [&](int st, int c) {
        unsigned char *sg = wsm + st * Lay::kStage;
        int c0, c1;
        span(c, c0, c1);
        const int len = c1 - c0;
        if (act) {
            const uint32_t lead = (uint32_t)(((erow + c0) * ES) & 15);
            const int nblk = (int)((lead + (uint32_t)(len * ES) + 15u) >> 4);
            const long long avail = (total - erow - c0) * ES + lead;
            const long long off = (long long)c0 * ES - lead;
            for (int a = 0; a < (hasZ ? 3 : 2); ++a) {
                const char *src = static_cast<const char *>(arr[a]) + erow * ES + off;
                unsigned char *dst = sg + Lay::row_off(a, lane);
                for (int k = 0; k < nblk; ++k) {
                    const long long rem = avail - 16 * k;
                    cp_async16(dst + 16 * k, src + 16 * k, rem >= 16 ? 16u : (uint32_t)rem);
                }
            }
        }
        const int nb = len * ES;                                    // 16-byte blocks of C rows
        const char *srcC = reinterpret_cast<const char *>(Cb + (long long)c0 * 16);
#pragma unroll
        for (int m = 0; m < (kSC * ES + 31) / 32; ++m) {
            const int jj = lane + 32 * m;
            cp_async16_if(sg + Lay::sC + 16 * jj, srcC + 16 * jj, jj < nb);
        }
        cp_async_commit();
    };
    float sdt = 0.f;
    bool cut = false;
    for (int c = 0; c < 2; ++c) {
        if (c < nc) issue(c, c);
        else cp_async_commit();
    }
    for (int c = 0; c < nc; ++c) {
        const int st = c & 1;
        const unsigned char *sg = wsm + st * Lay::kStage;
        int c0, c1;
        span(c, c0, c1);
        const int len = c1 - c0;
        cp_async_wait<1>();
        __syncwarp();
        const uint32_t lead = (uint32_t)(((erow + c0) * ES) & 15);
        const T *rdt = reinterpret_cast<const T *>(sg + Lay::row_off(0, lane) + lead);
        const T *rgo = reinterpret_cast<const T *>(sg + Lay::row_off(1, lane) + lead);
        const T *rz = reinterpret_cast<const T *>(sg + Lay::row_off(2, lane) + lead);
        const T *cs = reinterpret_cast<const T *>(sg + Lay::sC);
#pragma unroll 2
        for (int k = 0; k < len; ++k) {
            const int i = dir == 0 ? len - 1 - k : k;                // against the scan order
            const int t = c0 + i;
            const float dt = ld_as_f32(rdt + i);
            float ds = ld_as_f32(rgo + i);
            if (hasZ) {
                const float zv = ld_as_f32(rz + i);
                ds = ds * (zv * __frcp_rn(1.f + ex2_mufu(-kLog2e * zv)));
            }
            float Cv[16];
            load16_f32(cs + i * 16, Cv);
            const bool rs = reset_at(t, p.seg_len, dir);
            cut = cut || rs;
            sdt += dt;
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const float l = fmaf(ds, Cv[q], lam[q]);
                lam[q] = (rs ? 0.f : ex2_mufu(dt * Al2[q])) * l;
            }
        }
        __syncwarp();                                               // the stage is read
        if (c + 2 < nc) issue(st, c + 2);
        else cp_async_commit();
    }
    cp_async_wait<0>();
    float *sm = p.summ + (((long long)slot * p.ngroups + grp) * p.nrange + rr) * 1024;
#pragma unroll
    for (int q = 0; q < 16; ++q) {
        sm[q * 32 + lane] = cut ? 0.f : ex2_mufu(sdt * Al2[q]);
        sm[(16 + q) * 32 + lane] = lam[q];
    }
}

// 16 bytes of shared memory as two fp32 pairs, and back (ordered against the
// warp's other shared-memory accesses by the memory clobber).
__device__ __forceinline__ void lds2(const float *p, f2 &a, f2 &b)
{
    asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];" : "=l"(a.v), "=l"(b.v) : "r"(smem_addr(p)) : "memory");
}
__device__ __forceinline__ void sts2(float *p, f2 a, f2 b)
{
    asm volatile("st.shared.v2.b64 [%0], {%1, %2};" :: "r"(smem_addr(p)), "l"(a.v), "l"(b.v) : "memory");
}

template <typename T, int DIRS>
struct GradLayout {
    static constexpr int ES = (int)sizeof(T);
    static constexpr bool BIDIR = DIRS == 3;
    // one ring stage: this lane's 16-byte blocks of delta, x, z, dout over the
    // chunk (row slots of SLOT bytes), B and C of the chunk (raw). The chunk's
    // checkpoint and the partner's partial gradients go to registers instead
    // (prefetched), which keeps a warp's shared memory small enough for four
    // two-warp CTAs per SM.
    static constexpr int SLOT = ((16 - ES) + kTG * ES + 15) / 16 * 16;
    // rows staggered by 16 bytes every 8 rows so that lanes r and r + 8 read
    // different banks
    static constexpr int ROWS = 32 * SLOT + 16 * 3;           // one array's 32 rows
    __device__ static constexpr int row_off(int a, int r) { return a * ROWS + r * SLOT + 16 * (r >> 3); }
    static constexpr int sROW = 0;
    static constexpr int sB = sROW + 4 * ROWS;
    static constexpr int sC = sB + kTG * 16 * ES;
    static constexpr int kStage = (sC + kTG * 16 * ES + 15) / 16 * 16;
    // per warp: 2 stages, then
    //   hb  [kTG][4][32 lanes][4] states entering each token of the chunk
    //                                 (quarter q of a lane's 16 states;
    //                                 a warp's access to one quarter is 512
    //                                 contiguous bytes)
    //   bc  [kTG][32]                 B[16], C[16] of each token, fp32
    //   tr  [32 lanes][kTP]           dB, dC contributions of two consecutive
    //                                 tokens of the walk ([token][B 16 | C 16]
    //                                 per lane), reduced over the lanes together
    static constexpr int kTP = 68;
    static constexpr int oHB = 2 * kStage;
    static constexpr int oBC = oHB + kTG * 4 * 32 * 16;
    static constexpr int oTR = oBC + kTG * 32 * 4;              // two buffers
    static constexpr int kWarpBytes = oTR + 32 * kTP * 4 + 16;   // + pair barrier
    static_assert(kStage % 16 == 0 && oHB % 16 == 0 && oTR % 16 == 0, "alignment");
    // CTAs per SM that shared memory allows (228 KB, 1 KB reserved per CTA)
    static constexpr int kPerSm = (228 * 1024) / ((BIDIR ? 2 : 1) * kWarpBytes + 1024);
    static constexpr int kMinBlocks = kPerSm < 1 ? 1 : (kPerSm > 8 ? 8 : kPerSm);
};

// The dB, dC contributions of two tokens summed over the warp's 32 channels:
// row r of the [32][TP] buffer holds channel r's values for token slot 0
// (columns 0..31: B 16, C 16) and slot 1 (columns 32..63). Lane l sums the
// column pair 2(l mod 16), +1 of slot l / 16 over the rows (one 8-byte load
// and one packed add per row) and adds it to dB / dC of that slot's token,
// t[slot]; a slot whose token is -1 (the walk's last, unpaired token) is
// skipped.
template <int TP>
__device__ __forceinline__ void column_pair_sum_add(const float *buf, int lane, float *dB, float *dC,
                                                    long long bcrow, int t0, int t1)
{
    const int slot = lane >> 4, c = 2 * (lane & 15);
    const float *col = buf + slot * 32 + c;
    f2 acc[4] = {pack2(0.f, 0.f), pack2(0.f, 0.f), pack2(0.f, 0.f), pack2(0.f, 0.f)};
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        const float2 v = *reinterpret_cast<const float2 *>(col + r * TP);
        acc[r & 3] = add2(acc[r & 3], pack2(v.x, v.y));
    }
    const float2 sum = unpack2(add2(add2(acc[0], acc[1]), add2(acc[2], acc[3])));
    const int t = slot ? t1 : t0;
    if (t >= 0) {
        float *dst = c < 16 ? dB + bcrow + (long long)t * 16 + c : dC + bcrow + (long long)t * 16 + (c - 16);
        atomicAdd(reinterpret_cast<float2 *>(dst), sum);
    }
}

template <typename T, int DIRS>
__global__ void __launch_bounds__((DIRS == 3 ? 2 : 1) * 32, (GradLayout<T, DIRS>::kMinBlocks))
grad_adjoint_kernel(const GradParams p)
{
    using Lay = GradLayout<T, DIRS>;
    constexpr int TP = Lay::kTP, ES = Lay::ES;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long grp = blockIdx.x / p.nrange;          // CTA = (group, token range)
    const int rr = (int)(blockIdx.x % p.nrange);
    const int slot = warp;
    const int dir = (DIRS == 3) ? warp : (DIRS == 1 ? 0 : 1);
    unsigned char *wsm = smem_raw + warp * Lay::kWarpBytes;
    float *hb = reinterpret_cast<float *>(wsm + Lay::oHB);
    float *bc = reinterpret_cast<float *>(wsm + Lay::oBC);
    float *tr = reinterpret_cast<float *>(wsm + Lay::oTR);
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
    f2 Ap[8], Aa[8], lam[8], dA[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float a0 = act ? p.A[dir][(long long)d * 16 + 2 * q] : 0.f;
        const float a1 = act ? p.A[dir][(long long)d * 16 + 2 * q + 1] : 0.f;
        Aa[q] = pack2(a0, a1);
        Ap[q] = pack2(a0 * kLog2e, a1 * kLog2e);
        lam[q] = pack2(0.f, 0.f);
        dA[q] = pack2(0.f, 0.f);
    }
    const float Dk = (act && p.D[dir]) ? p.D[dir][d] : 0.f;
    float dD = 0.f;
    const long long total = (long long)p.batch * p.dim * p.L;
    const long long erow = ((long long)b * p.dim + (act ? d : d0)) * p.L;   // element of (b, d, 0)
    const long long bcrow = (long long)b * p.L * 16;
    const float *ck = p.ckpt + ((long long)slot * p.ngroups + grp) * p.nch * 512;
    const bool hasZ = p.z != nullptr;
    float *dBk = p.dB[dir], *dCk = p.dC[dir];
    float *my_h = hb + lane * 4;              // quarter q of slot s: my_h + (s * 4 + q) * 128
    const void *arr[4] = {p.delta, p.x, hasZ ? p.z : p.x, p.dout};

    // this CTA's chunks [rlo, rhi); the two directions meet in its middle
    const int rlo = rr * p.rch, rhi = min(p.nch, rlo + p.rch);
    const int Hc = rlo + (rhi - rlo + 1) / 2;
    const int nphase = (DIRS == 3) ? 2 : 1;
    // chunk list: phase 0 then phase 1, each against the scan order
    auto chunk_of = [&](int phase, int s, int &j) -> bool {
        int clo, chi;
        if (DIRS == 3) {
            const bool upper = (dir == 0) == (phase == 0);
            clo = upper ? Hc : rlo;
            chi = upper ? rhi : Hc;
        } else {
            clo = rlo;
            chi = rhi;
        }
        if (s >= chi - clo) return false;
        j = dir == 0 ? chi - 1 - s : clo + s;
        return true;
    };
    auto nchunks = [&](int phase) {
        if (DIRS != 3) return rhi - rlo;
        const bool upper = (dir == 0) == (phase == 0);
        return upper ? rhi - Hc : Hc - rlo;
    };
    // the lam entering this range, from the summaries of the ranges before it
    // in walk order (the forward direction walks right to left, the backward
    // one left to right), nearest last
    if (p.summ && act) {
        const float *sg = p.summ + ((long long)slot * p.ngroups + grp) * p.nrange * 1024 + lane;
        const int n_before = dir == 0 ? p.nrange - 1 - rr : rr;
        for (int k = 0; k < n_before; ++k) {
            const int r2 = dir == 0 ? p.nrange - 1 - k : k;
            const float *sm = sg + (long long)r2 * 1024;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const f2 P = pack2(__ldcg(sm + (2 * q) * 32), __ldcg(sm + (2 * q + 1) * 32));
                const f2 Q = pack2(__ldcg(sm + (16 + 2 * q) * 32), __ldcg(sm + (17 + 2 * q) * 32));
                lam[q] = fma2(P, lam[q], Q);
            }
        }
    }
    // copy chunk j (phase ph) into ring stage st and commit it as one group
    auto issue = [&](int st, int j, bool fin) {
        unsigned char *sg = wsm + st * Lay::kStage;
        const int t0 = j * kTG, len = min(p.L, t0 + kTG) - t0;
        if (act) {
            const uint32_t lead = (uint32_t)(((erow + t0) * ES) & 15);
            const int nblk = (int)((lead + (uint32_t)(len * ES) + 15u) >> 4);
            const long long avail = (total - erow - t0) * ES + lead;
            const long long off = (long long)t0 * ES - lead;
            for (int a = 0; a < 4; ++a) {
                if (a == 2 && !hasZ) continue;
                const char *src = static_cast<const char *>(arr[a]) + erow * ES + off;
                unsigned char *dst = sg + Lay::sROW + Lay::row_off(a, lane);
                for (int k = 0; k < nblk; ++k) {
                    const long long rem = avail - 16 * k;
                    cp_async16(dst + 16 * k, src + 16 * k, rem >= 16 ? 16u : (uint32_t)rem);
                }
            }
        }
        {   // B and C: len * 16 * ES bytes each, contiguous
            const int nb = len * ES;                  // 16-byte blocks per tensor
            const char *srcB = static_cast<const char *>(p.B[dir]) + (bcrow + (long long)t0 * 16) * ES;
            const char *srcC = static_cast<const char *>(p.C[dir]) + (bcrow + (long long)t0 * 16) * ES;
#pragma unroll
            for (int m = 0; m < (kTG * ES + 31) / 32; ++m) {
                const int jj = lane + 32 * m;
                cp_async16_if(sg + Lay::sB + 16 * jj, srcB + 16 * jj, jj < nb);
                cp_async16_if(sg + Lay::sC + 16 * jj, srcC + 16 * jj, jj < nb);
            }
        }
        cp_async_commit();
    };
    // the checkpoint entering chunk j, this lane's 16 states
    auto load_ckpt = [&](int j, f2 (&c)[8]) {
        const float *src = ck + (long long)j * 512 + lane;
#pragma unroll
        for (int q = 0; q < 8; ++q) c[q] = pack2(__ldcg(src + (2 * q) * 32), __ldcg(src + (2 * q + 1) * 32));
    };

    if (!act) {   // an idle lane's row slots are never copied into: zero them once
#pragma unroll 1
        for (int st = 0; st < 2; ++st)
            for (int a = 0; a < 4; ++a) {
                uint4 *r = reinterpret_cast<uint4 *>(wsm + st * Lay::kStage + Lay::sROW + Lay::row_off(a, lane));
                for (int k = 0; k < Lay::SLOT / 16; ++k) r[k] = make_uint4(0u, 0u, 0u, 0u);
            }
    }
    bool ok = true;
    int ring = 0;
    for (int phase = 0; phase < nphase && ok; ++phase) {
        const bool fin = phase == nphase - 1;
        const int nk = nchunks(phase);
        for (int s = 0; s < 2; ++s) {
            int j;
            if (chunk_of(phase, s, j)) issue((ring + s) & 1, j, fin);
            else cp_async_commit();
        }
        f2 ckn[8];                                // the next chunk's checkpoint
        {
            int j0;
            if (chunk_of(phase, 0, j0)) load_ckpt(j0, ckn);
        }
        for (int s = 0; s < nk; ++s, ++ring) {
            const int st = ring & 1;
            unsigned char *sg = wsm + st * Lay::kStage;
            int j;
            chunk_of(phase, s, j);
            const int t0 = j * kTG, t1 = min(p.L, t0 + kTG), len = t1 - t0;
            // this chunk's checkpoint; the next one's is fetched during this chunk
            f2 h[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) h[q] = ckn[q];
            {
                int jn1;
                if (chunk_of(phase, s + 1, jn1)) load_ckpt(jn1, ckn);
            }
            // the partner's partials of the chunk's tokens (last phase), in walk order
            float ppx[kTG], ppd[kTG], ppz[kTG];
#pragma unroll
            for (int m = 0; m < kTG; ++m) {
                ppx[m] = ppd[m] = ppz[m] = 0.f;
                if (DIRS == 3 && fin && m < len) {
                    const int i = dir == 0 ? len - 1 - m : m;
                    const float *pp = p.part + ((grp * p.L + t0 + i) * 3) * 32 + lane;
                    ppx[m] = __ldcg(pp);
                    ppd[m] = __ldcg(pp + 32);
                    ppz[m] = __ldcg(pp + 64);
                }
            }
            cp_async_wait<1>();
            __syncwarp();
            const uint32_t lead = (uint32_t)(((erow + t0) * ES) & 15);
            const T *rowv[4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
                rowv[a] = reinterpret_cast<const T *>(sg + Lay::sROW + Lay::row_off(a, lane) + lead);
            // B and C to fp32 (lane = (token, quarter of 8 values))
            {
                const int tk = lane >> 2, q = lane & 3;
                if (tk < len) {
                    const T *src = reinterpret_cast<const T *>(sg + (q < 2 ? Lay::sB : Lay::sC)) + tk * 16 + (q & 1) * 8;
                    float *dst = bc + tk * 32 + (q >> 1) * 16 + (q & 1) * 8;
#pragma unroll
                    for (int i = 0; i < 8; ++i) dst[i] = ld_as_f32(src + i);
                }
            }
            // recompute the chunk's states: slot k = state entering the token
            // at scan position k (slot 0 the checkpoint); the state after the
            // last token stays in registers
#pragma unroll
            for (int q = 0; q < 4; ++q) sts2(my_h + q * 128, h[2 * q], h[2 * q + 1]);
            __syncwarp();
            // (rows of idle lanes hold zeros: every per-token value below is 0 there)
            auto rec_step = [&](int k, bool store) {
                const int i = dir == 0 ? k : len - 1 - k;
                const float dt = ld_as_f32(rowv[0] + i);
                const float ux = dt * ld_as_f32(rowv[1] + i);
                const bool rs = reset_at(t0 + i, p.seg_len, dir);
                const f2 dd = pack2(dt, dt), uu = pack2(ux, ux);
                const f2 lmd = rs ? pack2(-INFINITY, -INFINITY) : pack2(0.f, 0.f);
                const float *Bt = bc + i * 32;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    f2 B0, B1;
                    lds2(Bt + 4 * q, B0, B1);
                    h[2 * q] = fma2(ex2_fma2(dd, Ap[2 * q], lmd), h[2 * q], mul2(uu, B0));
                    h[2 * q + 1] = fma2(ex2_fma2(dd, Ap[2 * q + 1], lmd), h[2 * q + 1], mul2(uu, B1));
                    if (store) sts2(my_h + ((k + 1) * 4 + q) * 128, h[2 * q], h[2 * q + 1]);
                }
            };
            // adjoint, against the scan order (walk step m at scan position
            // k = len - 1 - m); hn = state after the current token
            f2 hn[8];
            int t_prev = -1;                      // the previous token of the walk (its pair's slot 0)
            auto adj_step = [&](int m, float px, float pdt, float pz) {
                const int k = len - 1 - m;
                const int i = dir == 0 ? k : len - 1 - k;
                const int t = t0 + i;
                const bool rs = reset_at(t, p.seg_len, dir);
                const float dt = ld_as_f32(rowv[0] + i);
                const float xv = ld_as_f32(rowv[1] + i);
                const float zv = hasZ ? ld_as_f32(rowv[2] + i) : 0.f;
                const float go = ld_as_f32(rowv[3] + i);
                float g = 1.f, gp = 0.f;
                if (hasZ) {
                    const float sgm = __frcp_rn(1.f + ex2_mufu(-kLog2e * zv));
                    g = zv * sgm;
                    gp = sgm * fmaf(zv, 1.f - sgm, 1.f);
                }
                const float ds = go * g;
                const float ux = dt * xv;
                const f2 dsv = pack2(ds, ds), uxv = pack2(ux, ux), dd = pack2(dt, dt);
                const f2 lmd = rs ? pack2(-INFINITY, -INFINITY) : pack2(0.f, 0.f);
                const float *Bt = bc + i * 32;
                f2 yk2 = pack2(0.f, 0.f), sB2 = pack2(0.f, 0.f), sw2 = pack2(0.f, 0.f);
                const int pslot = m & 1;                 // slot of this token in its pair
                float *trow = tr + lane * TP + pslot * 32;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    f2 B0, B1, C0, C1, hp0, hp1;
                    lds2(Bt + 4 * q, B0, B1);
                    lds2(Bt + 16 + 4 * q, C0, C1);
                    lds2(my_h + (k * 4 + q) * 128, hp0, hp1);
                    const f2 e0 = ex2_fma2(dd, Ap[2 * q], lmd), e1 = ex2_fma2(dd, Ap[2 * q + 1], lmd);
                    const f2 l0 = fma2(dsv, C0, lam[2 * q]), l1 = fma2(dsv, C1, lam[2 * q + 1]);
                    yk2 = fma2(C0, hn[2 * q], yk2);
                    yk2 = fma2(C1, hn[2 * q + 1], yk2);
                    sts2(trow + 16 + 4 * q, mul2(dsv, hn[2 * q]), mul2(dsv, hn[2 * q + 1]));   // dC
                    sts2(trow + 4 * q, mul2(l0, uxv), mul2(l1, uxv));                         // dB
                    sB2 = fma2(l0, B0, sB2);
                    sB2 = fma2(l1, B1, sB2);
                    const f2 w0 = mul2(mul2(l0, e0), hp0), w1 = mul2(mul2(l1, e1), hp1);
                    sw2 = fma2(w0, Aa[2 * q], sw2);
                    sw2 = fma2(w1, Aa[2 * q + 1], sw2);
                    dA[2 * q] = fma2(w0, dd, dA[2 * q]);
                    dA[2 * q + 1] = fma2(w1, dd, dA[2 * q + 1]);
                    lam[2 * q] = mul2(e0, l0);
                    lam[2 * q + 1] = mul2(e1, l1);
                    hn[2 * q] = hp0;
                    hn[2 * q + 1] = hp1;
                }
                const float2 yv = unpack2(yk2), sBv = unpack2(sB2), swv = unpack2(sw2);
                const float yk = fmaf(Dk, xv, yv.x + yv.y), sB = sBv.x + sBv.y, sw = swv.x + swv.y;
                dD = fmaf(ds, xv, dD);
                float gx = fmaf(ds, Dk, dt * sB);
                float gdt = fmaf(xv, sB, sw);
                float gz = go * gp * yk;
                // dB, dC of the pair's tokens once both are written (or the
                // chunk's last token): sums over the warp's channels (rows of
                // idle lanes hold zeros)
                if (pslot == 1 || k == 0) {
                    __syncwarp();
                    column_pair_sum_add<TP>(tr, lane, dBk, dCk, bcrow, pslot ? t_prev : t, pslot ? t : -1);
                    __syncwarp();                 // the buffer is written again by the next pair
                }
                t_prev = t;
                // per-token gradients of x, delta, z
                if (!fin) {
                    float *pp = p.part + ((grp * p.L + t) * 3) * 32 + lane;
                    pp[0] = gx;
                    pp[32] = gdt;
                    pp[64] = gz;
                } else if (act) {
                    gx += px;
                    gdt += pdt;
                    gz += pz;
                    const long long e = erow + t;
                    st_from_f32(static_cast<T *>(p.dx) + e, gx);
                    st_from_f32(static_cast<T *>(p.ddelta) + e, gdt);
                    if (hasZ) st_from_f32(static_cast<T *>(p.dz) + e, gz);
                }
            };
            if (len == kTG) {                     // a whole chunk: straight-line code
#pragma unroll
                for (int k = 0; k < kTG; ++k) rec_step(k, k + 1 < kTG);
                __syncwarp();
#pragma unroll
                for (int q = 0; q < 8; ++q) hn[q] = h[q];
#pragma unroll
                for (int m = 0; m < kTG; ++m) adj_step(m, ppx[m], ppd[m], ppz[m]);
            } else {                              // the row's last, partial chunk
#pragma unroll 1
                for (int k = 0; k < len; ++k) rec_step(k, k + 1 < len);
                __syncwarp();
#pragma unroll
                for (int q = 0; q < 8; ++q) hn[q] = h[q];
#pragma unroll 1
                for (int m = 0; m < len; ++m) {
                    float px = ppx[0], pdt = ppd[0], pz = ppz[0];
#pragma unroll
                    for (int u = 1; u < kTG; ++u)
                        if (m == u) {
                            px = ppx[u];
                            pdt = ppd[u];
                            pz = ppz[u];
                        }
                    adj_step(m, px, pdt, pz);
                }
            }
            __syncwarp();
            {
                int jn;
                if (chunk_of(phase, s + 2, jn)) issue(st, jn, fin);
                else cp_async_commit();
            }

        }
        cp_async_wait<0>();
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
    cp_async_wait<0>();
    if (act && ok) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float2 v = unpack2(dA[q]);
            atomicAdd(p.dA[dir] + (long long)d * 16 + 2 * q, v.x);
            atomicAdd(p.dA[dir] + (long long)d * 16 + 2 * q + 1, v.y);
        }
        atomicAdd(p.dD[dir] + d, dD);
    }
}

}  // namespace vssm
