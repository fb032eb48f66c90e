// Warp-per-channel-group selective scan for sm_103a (B300), N = 16 states.
//
// What it computes is stated in include/vssm.h. Work decomposition:
//
//  * A "group" is RPW = 32/G consecutive channels d0..d0+RPW-1 of one batch
//    entry over one token range [ta, tb): the whole sequence, or, for a folded
//    sequence, a piece that starts and ends on segment boundaries (the reset
//    makes pieces independent; SF-Mamba page, "周期性状态重置").
//  * One warp scans one direction of one group. Lane (r, g) = (lane/G, lane%G)
//    holds states g*NS .. g*NS+NS-1 (NS = 16/G) of channel d0+r in fp32
//    registers and walks the tokens one at a time (Vim page §2.2: forward in
//    spatial order, backward in reverse). The recurrence per state and token
//    (VSSD page §4.1.2, §4.2.1.3) is
//        h = 2^(delta*A*log2e + lambda) * h + (delta*x) * B,   y += C*h
//    where lambda = -inf at a folded segment start (decay forced to 0) and 0
//    elsewhere. Two states share each packed f32x2 instruction.
//  * Both directions: the two warps of a pair own the same group and meet in
//    the middle. Phase 0: forward walks the first half up, backward the second
//    half down, each writing its y (no skip) to the workspace y-buffer with
//    bulk stores. Phase 1: each walks the other half, bulk-loads the partner's
//    y, adds the skip (D_fwd + D_bwd) * x, applies silu(z) and stores out.
//
// Data movement per warp and chunk of kTC tokens: the warp's lanes issue 1-D
// bulk async copies (TMA engine) of each channel's delta, x (and z) span and
// of B_t, C_t into a kStages-deep shared-memory ring, completion tracked by
// one mbarrier per stage. The warp then converts the chunk with lane = token
// (reads along a channel, conflict-free) into a [token][channel] float4
// (delta, delta*x, x, z) table and an fp32 B/C/lambda table, so that the scan
// with lane = channel reads one float4 per token and broadcast B/C. Inputs are
// read from HBM once and the state never leaves registers.
//
// Every wait is bounded (kWaitLimitNs); on expiry the kernel sets a bit in the
// device error word and the warp stops.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"

namespace vssm {

constexpr int kTC = 16;          // tokens per chunk
constexpr int kStages = 2;       // depth of the bulk-copy ring
constexpr int kBCPitch = 36;     // floats per token: B[16], C[16], lambda, pad
constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s
constexpr unsigned kErrTimeout = 1u;

struct WarpScanParams {
    const void *x, *delta, *z;
    const void *B[2], *C[2];     // [0] forward, [1] backward
    const float *A[2], *D[2];
    void *out;
    float *ybuf;                 // [ngroups][piece_len][RPW] floats (both directions only)
    unsigned *err;               // device error word
    long long total;             // batch * dim * L elements
    int batch, dim, L, seg_len, pieces, piece_len;
    int rgroups;                 // ceil(dim / RPW)
    long long ngroups;           // batch * pieces * rgroups
};

template <typename T, int G>
struct WarpLayout {
    static constexpr int RPW = 32 / G;            // channels per warp
    static constexpr int NS = 16 / G;             // states per lane
    static constexpr int ES = (int)sizeof(T);
    // bytes per channel span: kTC elements plus up to 16-ES bytes of lead-in
    // to the 16-byte aligned copy start
    static constexpr int BOXB = ((16 - ES) + kTC * ES + 15) / 16 * 16;
    // one ring stage (bytes)
    static constexpr int oD = 0;
    static constexpr int oX = oD + RPW * BOXB;
    static constexpr int oZ = oX + RPW * BOXB;
    static constexpr int oB = oZ + RPW * BOXB;
    static constexpr int oC = oB + kTC * 16 * ES;
    static constexpr int oPY = oC + kTC * 16 * ES;
    static constexpr int kStageBytes = oPY + kTC * RPW * 4;
    // one warp's region (bytes)
    static constexpr int CP = RPW + 1;            // float4 pitch of the converted table
    static constexpr int oConv = kStages * kStageBytes;
    static constexpr int oBC = oConv + kTC * CP * 16;
    static constexpr int oYS = oBC + kTC * kBCPitch * 4;
    static constexpr int oBar = oYS + kTC * RPW * 4;
    static constexpr int kWarpBytes = (oBar + 8 * (kStages + 1) + 127) / 128 * 128;
    static_assert(BOXB % 16 == 0 && kStageBytes % 16 == 0 && oBar % 16 == 0, "alignment");
};

__device__ __forceinline__ float ld_as_f32(const float *p) { return *p; }
__device__ __forceinline__ float ld_as_f32(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_from_f32(float *p, float v) { *p = v; }
__device__ __forceinline__ void st_from_f32(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

// 16 consecutive elements from shared memory to fp32 (16-byte aligned source).
__device__ __forceinline__ void load16_f32(const float *src, float *dst)
{
    const float4 *s = reinterpret_cast<const float4 *>(src);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 v = s[q];
        dst[4 * q + 0] = v.x;
        dst[4 * q + 1] = v.y;
        dst[4 * q + 2] = v.z;
        dst[4 * q + 3] = v.w;
    }
}
__device__ __forceinline__ void load16_f32(const __nv_bfloat16 *src, float *dst)
{
    const uint4 *s = reinterpret_cast<const uint4 *>(src);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const uint4 v = s[q];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            dst[8 * q + 2 * k + 0] = __uint_as_float(w[k] << 16);
            dst[8 * q + 2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        }
    }
}

__device__ __forceinline__ float silu_f32(float z)
{
    return __fdividef(z, 1.0f + ex2_mufu(-1.4426950408889634f * z));
}

template <typename T, int G, int DIRS, int W>
struct WarpScan {
    using Lay = WarpLayout<T, G>;
    static constexpr int RPW = Lay::RPW, NS = Lay::NS, CP = Lay::CP;
    static constexpr int NDIR = (DIRS == 3) ? 2 : 1;

    const WarpScanParams &p;
    unsigned char *wsm;          // this warp's shared region
    uint64_t *full;              // kStages mbarriers
    uint64_t *pairbar;           // pair rendezvous (both directions)
    int lane, dir;
    long long grp;
    int b, d0, ta, tb;
    bool ok;                     // false once a wait has timed out
    uint32_t inflight;           // bit s: stage s has copies issued and not yet waited for
    uint32_t parity;             // bit s: parity of stage s's next completion

    __device__ WarpScan(const WarpScanParams &p_) : p(p_) {}

    __device__ __forceinline__ unsigned char *stage(int s) const { return wsm + s * Lay::kStageBytes; }

    __device__ __forceinline__ const T *arr(int a) const
    {
        return static_cast<const T *>(a == 0 ? p.delta : (a == 1 ? p.x : p.z));
    }

    // Bytes of a channel span copied by bulk copy: a full box unless the box
    // would run past the end of the tensor (then whole 16-byte blocks only).
    __device__ __forceinline__ uint32_t box_bytes(const T *base, const char *a0) const
    {
        const char *tend = reinterpret_cast<const char *>(base + p.total);
        if (a0 + Lay::BOXB <= tend) return Lay::BOXB;
        return (uint32_t)((tend - a0) & ~(ptrdiff_t)15);
    }

    // Issue the bulk copies of chunk [c0, c1) into ring stage s.
    __device__ void issue(int s, int c0, int c1, bool fin)
    {
        unsigned char *st = stage(s);
        const int len = c1 - c0;
        const bool hasZ = fin && p.z != nullptr;
        const int narr = hasZ ? 3 : 2;
        for (int j = lane; j < narr * RPW; j += 32) {
            const int a = j / RPW, rr = j % RPW;
            const int d = d0 + rr;
            if (d >= p.dim) continue;
            const T *base = arr(a);
            const char *src = reinterpret_cast<const char *>(base + ((long long)b * p.dim + d) * p.L + c0);
            const char *a0 = reinterpret_cast<const char *>(reinterpret_cast<uintptr_t>(src) & ~(uintptr_t)15);
            const uint32_t bytes = box_bytes(base, a0);
            if (bytes) {
                mbar_expect_tx(&full[s], bytes);
                bulk_g2s(st + (a == 0 ? Lay::oD : a == 1 ? Lay::oX : Lay::oZ) + rr * Lay::BOXB, a0, bytes,
                         &full[s]);
            }
        }
        if (lane == 0 || lane == 1) {
            const T *src = static_cast<const T *>(lane == 0 ? p.B[dir] : p.C[dir]) + ((long long)b * p.L + c0) * 16;
            const uint32_t bytes = (uint32_t)(len * 16 * Lay::ES);
            mbar_expect_tx(&full[s], bytes);
            bulk_g2s(st + (lane == 0 ? Lay::oB : Lay::oC), src, bytes, &full[s]);
        }
        if (DIRS == 3 && fin && lane == 2) {
            const float *src = p.ybuf + (grp * p.piece_len + (c0 - ta)) * RPW;
            const uint32_t bytes = (uint32_t)(len * RPW * 4);
            mbar_expect_tx(&full[s], bytes);
            bulk_g2s(st + Lay::oPY, src, bytes, &full[s]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
        inflight |= 1u << s;
    }

    // Wait for stage s (bounded). Records a timeout in the error word.
    __device__ bool wait_stage(int s)
    {
        const bool done = mbar_wait(&full[s], (parity >> s) & 1u, kWaitLimitNs);
        const bool all = __all_sync(0xffffffffu, done);
        if (all) {
            parity ^= 1u << s;
            inflight &= ~(1u << s);
        } else if (lane == 0) {
            atomicOr(p.err, kErrTimeout);
        }
        return all;
    }

    // Convert ring stage s (chunk [c0, c1)) into the float4 table and the B/C table.
    __device__ void convert(int s, int c0, int c1, bool fin)
    {
        const unsigned char *st = stage(s);
        const int len = c1 - c0;
        float4 *conv = reinterpret_cast<float4 *>(wsm + Lay::oConv);
        float *bc = reinterpret_cast<float *>(wsm + Lay::oBC);
        const bool hasZ = fin && p.z != nullptr;
        const int i = lane & 15;
        const int hsel = lane >> 4;
#pragma unroll 4
        for (int rr0 = 0; rr0 < RPW; rr0 += 2) {
            const int rr = rr0 + hsel;
            const int d = d0 + rr;
            float dv = 0.f, xv = 0.f, zv = 0.f;
            if (i < len && d < p.dim) {
                const long long e = ((long long)b * p.dim + d) * p.L + c0 + i;
                const uintptr_t s0 = reinterpret_cast<uintptr_t>(static_cast<const T *>(p.delta) +
                                                                 (e - i));
                const uint32_t o = (uint32_t)(s0 & 15u) + (uint32_t)(i * Lay::ES);   // byte in box
                const T *dbase = static_cast<const T *>(p.delta);
                const char *a0 = reinterpret_cast<const char *>(s0 & ~(uintptr_t)15);
                // all activation tensors share the element offset and 16-byte alignment
                if (o + Lay::ES <= box_bytes(dbase, a0)) {
                    const int ro = rr * Lay::BOXB + (int)o;
                    dv = ld_as_f32(reinterpret_cast<const T *>(st + Lay::oD + ro));
                    xv = ld_as_f32(reinterpret_cast<const T *>(st + Lay::oX + ro));
                    if (hasZ) zv = ld_as_f32(reinterpret_cast<const T *>(st + Lay::oZ + ro));
                } else {   // tail of the tensor not covered by whole 16-byte blocks
                    dv = ld_as_f32(static_cast<const T *>(p.delta) + e);
                    xv = ld_as_f32(static_cast<const T *>(p.x) + e);
                    if (hasZ) zv = ld_as_f32(static_cast<const T *>(p.z) + e);
                }
            }
            conv[i * CP + rr] = make_float4(dv, dv * xv, xv, zv);
        }
        {
            const int t2 = lane >> 1, part = lane & 1;     // token, 0: B / 1: C
            float v[16];
            if (t2 < len) {
                load16_f32(reinterpret_cast<const T *>(st + (part ? Lay::oC : Lay::oB)) + t2 * 16, v);
            } else {
#pragma unroll
                for (int n = 0; n < 16; ++n) v[n] = 0.f;
            }
            float4 *dst = reinterpret_cast<float4 *>(bc + t2 * kBCPitch + part * 16);
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            if (part == 0) {
                float lam = 0.f;
                if (p.seg_len > 0 && t2 < len) {
                    const int ph = (c0 + t2) % p.seg_len;
                    if (ph == (dir == 0 ? 0 : p.seg_len - 1)) lam = -__int_as_float(0x7f800000);
                }
                bc[t2 * kBCPitch + 32] = lam;
            }
        }
        __syncwarp();
    }

    // Scan the converted chunk. FIN: last phase (emit output), else partial y.
    template <int DIR, bool FIN>
    __device__ __forceinline__ void scan_chunk(f2 (&h)[NS / 2], const f2 (&Ap)[NS / 2], float Dsum,
                                               bool hasZ, int s)
    {
        const float4 *conv = reinterpret_cast<const float4 *>(wsm + Lay::oConv);
        float4 *convw = reinterpret_cast<float4 *>(wsm + Lay::oConv);
        const float *bc = reinterpret_cast<const float *>(wsm + Lay::oBC);
        float *ys = reinterpret_cast<float *>(wsm + Lay::oYS);
        const float *py = reinterpret_cast<const float *>(stage(s) + Lay::oPY);
        const int r = lane / G, g = lane % G;
#pragma unroll
        for (int k = 0; k < kTC; ++k) {
            const int i = (DIR == 0) ? k : (kTC - 1 - k);
            const float4 v = conv[i * CP + r];
            const float *bcp = bc + i * kBCPitch;
            const float lam = bcp[32];
            const f2 dd = pack2(v.x, v.x), ll = pack2(lam, lam), uu = pack2(v.y, v.y);
            f2 ya = pack2(0.f, 0.f), yb = pack2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < NS / 4; ++q) {
                const float4 Bq = *reinterpret_cast<const float4 *>(bcp + g * NS + 4 * q);
                const float4 Cq = *reinterpret_cast<const float4 *>(bcp + 16 + g * NS + 4 * q);
                const float2 a0 = unpack2(fma2(dd, Ap[2 * q], ll));
                const float2 a1 = unpack2(fma2(dd, Ap[2 * q + 1], ll));
                const f2 e0 = pack2(ex2_mufu(a0.x), ex2_mufu(a0.y));
                const f2 e1 = pack2(ex2_mufu(a1.x), ex2_mufu(a1.y));
                h[2 * q] = fma2(e0, h[2 * q], mul2(uu, pack2(Bq.x, Bq.y)));
                h[2 * q + 1] = fma2(e1, h[2 * q + 1], mul2(uu, pack2(Bq.z, Bq.w)));
                ya = fma2(pack2(Cq.x, Cq.y), h[2 * q], ya);
                yb = fma2(pack2(Cq.z, Cq.w), h[2 * q + 1], yb);
            }
            const float2 y2a = unpack2(ya), y2b = unpack2(yb);
            float y = (y2a.x + y2a.y) + (y2b.x + y2b.y);
            if (G >= 2) y += __shfl_xor_sync(0xffffffffu, y, 1);
            if (G >= 4) y += __shfl_xor_sync(0xffffffffu, y, 2);
            if (!FIN) {
                if (g == 0) ys[i * RPW + r] = y;
            } else {
                float tot = y + fmaf(Dsum, v.z, (DIRS == 3) ? py[i * RPW + r] : 0.f);
                if (hasZ) tot *= silu_f32(v.w);
                if (g == 0) convw[i * CP + r].x = tot;
            }
        }
        __syncwarp();
    }

    // Store the chunk's outputs (lane = token, two channels per instruction).
    __device__ void store_out(int c0, int c1)
    {
        const float4 *conv = reinterpret_cast<const float4 *>(wsm + Lay::oConv);
        T *out = static_cast<T *>(p.out);
        const int len = c1 - c0;
        const int i = lane & 15, hsel = lane >> 4;
#pragma unroll 4
        for (int rr0 = 0; rr0 < RPW; rr0 += 2) {
            const int rr = rr0 + hsel;
            const int d = d0 + rr;
            if (i < len && d < p.dim)
                st_from_f32(out + ((long long)b * p.dim + d) * p.L + c0 + i, conv[i * CP + rr].x);
        }
    }

    // Bulk-store the chunk's partial y to the y-buffer.
    __device__ void store_partial(int c0, int c1)
    {
        float *ys = reinterpret_cast<float *>(wsm + Lay::oYS);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            bulk_s2g(p.ybuf + (grp * p.piece_len + (c0 - ta)) * RPW, ys, (uint32_t)((c1 - c0) * RPW * 4));
            bulk_commit();
        }
    }

    __device__ void chunk_range(int k, int lo, int hi, int &c0, int &c1) const
    {
        if (dir == 0) {
            c0 = lo + k * kTC;
            c1 = min(hi, c0 + kTC);
        } else {
            c1 = hi - k * kTC;
            c0 = max(lo, c1 - kTC);
        }
    }

    __device__ void run()
    {
        // ---- per-lane parameters
        const int r = lane / G, g = lane % G;
        const int d = d0 + r;
        const bool active = d < p.dim;
        constexpr float kLog2e = 1.4426950408889634f;
        f2 Ap[NS / 2], h[NS / 2];
#pragma unroll
        for (int j = 0; j < NS / 2; ++j) {
            const int n = g * NS + 2 * j;
            const float a0 = active ? p.A[dir][(long long)d * 16 + n] * kLog2e : 0.f;
            const float a1 = active ? p.A[dir][(long long)d * 16 + n + 1] * kLog2e : 0.f;
            Ap[j] = pack2(a0, a1);
            h[j] = pack2(0.f, 0.f);
        }
        float Dsum = 0.f;
        if (active) {
            if (DIRS == 3) {
                Dsum = (p.D[0] ? p.D[0][d] : 0.f) + (p.D[1] ? p.D[1][d] : 0.f);
            } else {
                Dsum = p.D[dir] ? p.D[dir][d] : 0.f;
            }
        }
        const bool hasZ = p.z != nullptr;

        const int Lv = tb - ta;
        const int H = (DIRS == 3) ? (Lv + 1) / 2 : Lv;
        const int nphase = (DIRS == 3) ? 2 : 1;
        uint32_t kk = 0;   // chunks consumed so far (ring position)
        for (int phase = 0; phase < nphase && ok; ++phase) {
            const bool fin = (phase == nphase - 1);
            int lo, hi;
            if (DIRS == 3) {
                const bool first_half = ((dir == 0) == (phase == 0));
                lo = first_half ? ta : ta + H;
                hi = first_half ? ta + H : tb;
            } else {
                lo = ta;
                hi = tb;
            }
            const int nk = (hi - lo + kTC - 1) / kTC;
            for (int k = 0; k < kStages && k < nk; ++k) {
                int c0, c1;
                chunk_range(k, lo, hi, c0, c1);
                issue((kk + k) % kStages, c0, c1, fin);
            }
            for (int k = 0; k < nk; ++k, ++kk) {
                const int s = kk % kStages;
                int c0, c1;
                chunk_range(k, lo, hi, c0, c1);
                if (!wait_stage(s)) {
                    ok = false;
                    break;
                }
                convert(s, c0, c1, fin);
                if (!fin) {                      // the staging buffer of the previous bulk store
                    if (lane == 0) bulk_wait_read();
                    __syncwarp();
                }
                if (dir == 0) {
                    if (fin) scan_chunk<0, true>(h, Ap, Dsum, hasZ, s);
                    else scan_chunk<0, false>(h, Ap, Dsum, hasZ, s);
                } else {
                    if (fin) scan_chunk<1, true>(h, Ap, Dsum, hasZ, s);
                    else scan_chunk<1, false>(h, Ap, Dsum, hasZ, s);
                }
                if (k + kStages < nk) {
                    int n0, n1;
                    chunk_range(k + kStages, lo, hi, n0, n1);
                    issue(s, n0, n1, fin);
                }
                if (fin) store_out(c0, c1);
                else store_partial(c0, c1);
                __syncwarp();
            }
            if (DIRS == 3 && phase == 0) {
                // Partial y fully written before the partner reads it.
                if (lane == 0) {
                    bulk_wait_all();
                    __threadfence();
                    mbar_arrive(pairbar);
                }
                __syncwarp();
                bool met = mbar_wait(pairbar, 0, kWaitLimitNs);
                if (!__all_sync(0xffffffffu, met)) {
                    if (lane == 0) atomicOr(p.err, kErrTimeout);
                    ok = false;
                }
            }
        }
        if (!ok) {
            // Let copies already issued land before the warp's shared memory
            // goes away (each wait again bounded).
            for (int s = 0; s < kStages; ++s)
                if (inflight & (1u << s)) (void)mbar_wait(&full[s], (parity >> s) & 1u, kWaitLimitNs);
        }
        if (lane == 0) bulk_wait_all();
    }
};

template <typename T, int G, int DIRS, int W>
__global__ void __launch_bounds__(W * 32) warp_scan_kernel(const WarpScanParams p)
{
    using Lay = WarpLayout<T, G>;
    constexpr int NDIR = (DIRS == 3) ? 2 : 1;
    static_assert(W % NDIR == 0, "whole pairs per CTA");
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int warp = threadIdx.x >> 5;
    WarpScan<T, G, DIRS, W> ws(p);
    ws.lane = threadIdx.x & 31;
    ws.wsm = smem_raw + warp * Lay::kWarpBytes;
    ws.full = reinterpret_cast<uint64_t *>(ws.wsm + Lay::oBar);
    ws.pairbar = reinterpret_cast<uint64_t *>(smem_raw + (warp - warp % NDIR) * Lay::kWarpBytes + Lay::oBar) +
                 kStages;
    ws.dir = (DIRS == 3) ? (warp % 2) : (DIRS == 1 ? 0 : 1);
    ws.ok = true;
    ws.inflight = 0;
    ws.parity = 0;
    if (ws.lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&ws.full[s], 1);
        if (DIRS == 3 && warp % 2 == 0) mbar_init(ws.pairbar, 2);
        fence_mbar_init();
    }
    __syncthreads();
    ws.grp = (long long)blockIdx.x * (W / NDIR) + warp / NDIR;
    if (ws.grp >= p.ngroups) return;             // both warps of a pair leave together
    long long t = ws.grp;
    const int rg = (int)(t % p.rgroups);
    t /= p.rgroups;
    const int piece = (int)(t % p.pieces);
    ws.b = (int)(t / p.pieces);
    ws.d0 = rg * Lay::RPW;
    ws.ta = piece * p.piece_len;
    ws.tb = min(p.L, ws.ta + p.piece_len);
    ws.run();
}

}  // namespace vssm
