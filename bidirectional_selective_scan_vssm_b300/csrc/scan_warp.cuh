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
//    spatial order, backward in reverse). Per state and token (VSSD page
//    §4.1.2, §4.2.1.3):
//        h = 2^(delta*A*log2e + lambda) * h + (delta*x) * B,   y += C*h
//    with lambda = -inf at a folded segment start (decay forced to 0) and 0
//    elsewhere. Two states share each packed f32x2 instruction.
//  * Both directions: the two warps of a pair own the same group and meet in
//    the middle. Phase 0: forward walks the first half up, backward the second
//    half down, each storing its y (no skip) to the workspace y-buffer.
//    Phase 1: each walks the other half, adds the partner's y and the skip
//    (D_fwd + D_bwd) * x, applies silu(z) and writes the output.
//
// Data movement per warp and chunk of kTC tokens: every lane copies the
// 16-byte blocks that cover its own channel's delta, x (and z) span into a
// row slot of an NST-deep shared-memory ring (two chunks; one on short rows,
// where the smaller footprint buys more warps) with per-thread async copies
// (the tensor's final partial block is zero-filled past its end); B_t, C_t and
// the partner's y are copied the same way, one block per lane. The scan lanes
// read delta/x/z straight from their row slots (rows staggered across banks);
// B/C are widened once per chunk into an fp32 table read by broadcast.
// Outputs go to a small tile and leave with row-contiguous stores; partial y
// leaves directly, one coalesced row of RPW values per token. Inputs are read
// from HBM once and the state never leaves registers.
//
// The only wait on another warp (the pair rendezvous) is bounded
// (kWaitLimitNs); on expiry the kernel sets a bit in the device error word
// and the warp stops.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "ptx.cuh"

namespace vssm {

constexpr int kTC = 16;          // tokens per chunk
#ifndef VSSM_SCAN_STAGES
#define VSSM_SCAN_STAGES 2
#endif
constexpr int kStages = VSSM_SCAN_STAGES;   // depth of the copy ring (default)
// Uncut rows of both directions and at most this many tokens use a one-deep
// ring: their chunks are few, and the smaller footprint fits 16 warps per SM
// instead of 12, which hides more of the per-token latency than the lost
// copy/compute overlap costs (measured on Vim-S 224^2; longer rows lose).
constexpr int kOneStageMaxL = 256;
#ifndef VSSM_SCAN_UNROLL
#define VSSM_SCAN_UNROLL 2
#endif
constexpr int kUnroll = VSSM_SCAN_UNROLL;   // tokens per unrolled scan step
// Uncut rows longer than kOneStageMaxL unroll more tokens: each warp walks
// many chunks, and the extra independent work per step hides more latency.
// Not taken with the convolution in both directions, nor when the training
// forward writes checkpoints: there it measured slower (register pressure).
constexpr int kLongRowUnroll = 4;

struct WarpScanParams {
    const void *x, *delta[2], *z;  // delta: [0] forward, [1] backward step
    const float *dbias[2];         // step bias per direction (SP kernels), or null
    const float *conv_w[2], *conv_b[2];   // directional convolution (CONV kernels)
    int conv_k;                    // its taps, 1..4
    const void *B[2], *C[2];     // [0] forward, [1] backward
    const float *A[2], *D[2];
    void *out;
    float *ybuf;                 // [ngroups][piece_len][RPW] floats (both directions only)
    int discard_y;               // ybuf is 128-byte aligned: its rows are dropped from L2 once read
    float *summ;                 // carry summaries [slot][srows][pieces][kSummFloats], or null
    float *ckpt;                 // training forward: [slot][srows][nch][16][32], the state
                                 // entering every 4-token chunk in each direction's scan
                                 // order (the gradient's checkpoints), or null
    int nch;                     // 4-token chunks per row (ckpt)
                                 // when every piece starts from a zero state
    unsigned *err;               // device error word
    long long total;             // batch * dim * L elements
    int batch, dim, L, seg_len, pieces, piece_len;
    int rgroups;                 // ceil(dim / RPW)
    long long ngroups;           // batch * pieces * rgroups
    long long srows;             // batch * rgroups
};

// One piece's summary for 32 channels: the state reached by scanning the
// piece from zero, h[n][lane] (n < 16), then the piece's delta sum [16][lane],
// or kCutBits there when a folded reset inside the piece cuts the carry.
constexpr int kSummFloats = 17 * 32;
constexpr uint32_t kCutBits = 0xffffffffu;

template <typename T, int G, bool BIDIR, int NST = kStages>
struct WarpLayout {
    static constexpr int RPW = 32 / G;            // channels per warp
    static constexpr int NS = 16 / G;             // states per lane
    static constexpr int ES = (int)sizeof(T);
    // bytes per row slot: kTC elements plus up to 16-ES bytes of lead-in to
    // the 16-byte aligned copy start
    static constexpr int SLOT = ((16 - ES) + kTC * ES + 15) / 16 * 16;
    // rows are staggered by 16 bytes every 8 rows so that rows r and r+8 fall
    // on different bank groups
    static constexpr int ROWB = RPW * SLOT + 16 * ((RPW - 1) >> 3);
    // one ring stage (bytes)
    static constexpr int oD = 0;
    static constexpr int oX = oD + ROWB;
    static constexpr int oZ = oX + ROWB;
    static constexpr int oB = oZ + ROWB;
    static constexpr int oC = oB + kTC * 16 * ES;
    static constexpr int oPY = oC + kTC * 16 * ES;
    static constexpr int kStageBytes = (oPY + (BIDIR ? kTC * RPW * 4 : 0) + 15) / 16 * 16;
    // one warp's region (bytes)
    static constexpr int oBC = NST * kStageBytes;       // fp32 [kTC][32]: B[16], C[16]
    // output tile [RPW][OTP] in the output type; the pitch makes the scan's
    // column writes (one row per lane) land on distinct banks
    static constexpr int OTP = ES == 2 ? kTC + 2 : kTC + 1;
    static constexpr int oOT = oBC + kTC * 32 * 4;
    static constexpr int oBar = (oOT + RPW * OTP * ES + 15) / 16 * 16;
    static constexpr int kWarpBytes = oBar + 16;
    static_assert(SLOT % 16 == 0 && ROWB % 16 == 0 && kStageBytes % 16 == 0 && oBar % 16 == 0,
                  "alignment");

    __device__ static constexpr int row_off(int r) { return r * SLOT + 16 * (r >> 3); }
};

// CARRY: ranges start from a carried-in state. SP: the step is
// softplus(delta + bias[d]) of the direction's own delta and bias. CONV: the
// input is silu of the direction's depthwise convolution of x, computed from
// a three-token history of x that each lane carries in registers.
template <typename T, int G, int DIRS, int W, bool CARRY = false, bool SP = false,
          bool CONV = false, int NST = kStages, int UNR = kUnroll>
struct WarpScan {
    using Lay = WarpLayout<T, G, DIRS == 3, NST>;
    static constexpr int RPW = Lay::RPW, NS = Lay::NS, ES = Lay::ES;
    static constexpr int NDIR = (DIRS == 3) ? 2 : 1;

    const WarpScanParams &p;
    unsigned char *wsm;          // this warp's shared region
    uint64_t *pairbar;           // pair rendezvous (both directions)
    int lane, dir, r, g;
    int slot;                    // direction slot of the carry summaries
    int piece, rg;               // token range and channel group of this warp
    float dbias_l;               // this lane's step bias (SP)
    float cw[4], cb;             // this lane's convolution taps, right-aligned, and bias (CONV)
    long long grp;
    int b, d0, ta, tb;
    bool ok;                     // false once the pair rendezvous has timed out
    uint32_t lane_emod;          // (element index of (b, d0+r, 0)) mod 16
    long long lane_erow;         // element index of (b, d0+r, 0)
    const char *rowp[3];         // this lane's row (b, d0+r, 0) of delta, x, z
    T *out_row0;                 // output row (b, d0, 0)
    float *ck_row;               // this warp's checkpoint row (b, d0 .. d0+31, slot), or null

    __device__ WarpScan(const WarpScanParams &p_) : p(p_) {}

    // Token range, channel rows and row pointers from (b, rg, piece).
    __device__ void place()
    {
        d0 = rg * RPW;
        ta = piece * p.piece_len;
        tb = min(p.L, ta + p.piece_len);
        const long long e0 = ((long long)b * p.dim + d0) * p.L;
        lane_erow = e0 + (long long)r * p.L;
        lane_emod = (uint32_t)(lane_erow & 15);
        rowp[0] = static_cast<const char *>(p.delta[dir]) + lane_erow * ES;
        dbias_l = (SP && d0 + r < p.dim && p.dbias[dir]) ? p.dbias[dir][d0 + r] : 0.f;
        if (CONV) {
            // taps right-aligned: cw[3] multiplies x_t, cw[3-j] the token j
            // steps back along this direction
            const bool act = d0 + r < p.dim;
            const int K = p.conv_k;
            const float *w = p.conv_w[dir] + (long long)(d0 + r) * K;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int k = j - (4 - K);
                cw[j] = (act && k >= 0) ? w[k] : 0.f;
            }
            cb = (act && p.conv_b[dir]) ? p.conv_b[dir][d0 + r] : 0.f;
        }
        rowp[1] = static_cast<const char *>(p.x) + lane_erow * ES;
        rowp[2] = p.z ? static_cast<const char *>(p.z) + lane_erow * ES : rowp[1];
        out_row0 = static_cast<T *>(p.out) + e0;
        ck_row = p.ckpt ? p.ckpt + (((long long)slot * p.srows + (long long)b * p.rgroups + rg) * p.nch) * 512 + lane
                        : nullptr;
    }

    __device__ __forceinline__ unsigned char *stage(int s) const { return wsm + s * Lay::kStageBytes; }

    // Byte offset of token c0 inside its 16-byte block (tensor bases are
    // 16-byte aligned).
    __device__ __forceinline__ uint32_t lead_of(uint32_t emod, int c0) const
    {
        return ((emod + (uint32_t)c0) * ES) & 15u;
    }

    // Copy chunk [c0, c1) into ring stage s and commit it as one group. Each
    // row span is copied from the 16-byte boundary at or before token c0 in
    // whole blocks; a block that would run past the end of the tensor (only
    // on its final row) is zero-filled past the end instead of read.
    __device__ void issue(int s, int c0, int c1, bool fin)
    {
        unsigned char *st = stage(s);
        const int len = c1 - c0;
        if ((G == 1 || g == 0) && d0 + r < p.dim) {
            const uint32_t lead = lead_of(lane_emod, c0);
            const int nblk = (int)((lead + (uint32_t)(len * ES) + 15u) >> 4);
            const long long avail = (p.total - lane_erow - c0) * ES + lead;   // bytes to tensor end
            const int narr = (fin && p.z != nullptr) ? 3 : 2;
            const long long off = (long long)c0 * ES - lead;
            unsigned char *dst = st + Lay::row_off(r);
            if (avail >= 16 * nblk) {             // every block lies inside the tensor
                const char *s0 = rowp[0] + off, *s1 = rowp[1] + off, *s2 = rowp[2] + off;
#pragma unroll
                for (int k = 0; k < Lay::SLOT / 16; ++k) {
                    const bool in = k < nblk;
                    cp_async16_if(dst + 16 * k, s0 + 16 * k, in);
                    cp_async16_if(dst + Lay::ROWB + 16 * k, s1 + 16 * k, in);
                    if (narr == 3) cp_async16_if(dst + 2 * Lay::ROWB + 16 * k, s2 + 16 * k, in);
                }
            } else {                              // the tensor's final row: clip the last block
                for (int a = 0; a < narr; ++a)
                    for (int k = 0; k < nblk; ++k) {
                        const long long rem = avail - 16 * k;
                        cp_async16(dst + a * Lay::ROWB + 16 * k, rowp[a] + off + 16 * k,
                                   rem >= 16 ? 16u : (uint32_t)rem);
                    }
            }
        }
        {   // B and C: len*ES blocks each, contiguous
            const int nb = len * ES;
            const long long boff = ((long long)b * p.L + c0) * 16 * ES;
            const char *srcB = static_cast<const char *>(p.B[dir]) + boff;
            const char *srcC = static_cast<const char *>(p.C[dir]) + boff;
#pragma unroll
            for (int m = 0; m < kTC * ES / 32; ++m) {
                const int j = lane + 32 * m;
                cp_async16_if(st + Lay::oB + 16 * j, srcB + 16 * j, j < nb);
                cp_async16_if(st + Lay::oC + 16 * j, srcC + 16 * j, j < nb);
            }
        }
        if (DIRS == 3 && fin) {   // partner's partial y, len rows of RPW floats
            const int nb = len * RPW / 4;
            const char *src = reinterpret_cast<const char *>(p.ybuf + (grp * p.piece_len + (c0 - ta)) * RPW);
#pragma unroll
            for (int m = 0; m < kTC * RPW / 128; ++m) {
                const int j = lane + 32 * m;
                cp_async16_if(st + Lay::oPY + 16 * j, src + 16 * j, j < nb);
            }
        }
        cp_async_commit();
    }

    // Widen the chunk's B_t, C_t into the fp32 table (lane = token x {B, C}).
    __device__ void widen_bc(int s, int len)
    {
        const unsigned char *st = stage(s);
        float *bc = reinterpret_cast<float *>(wsm + Lay::oBC);
        const int t2 = lane >> 1, part = lane & 1;
        float v[16];
        if (t2 < len) {
            load16_f32(reinterpret_cast<const T *>(st + (part ? Lay::oC : Lay::oB)) + t2 * 16, v);
        } else {
#pragma unroll
            for (int n = 0; n < 16; ++n) v[n] = 0.f;
        }
        float4 *dst = reinterpret_cast<float4 *>(bc + t2 * 32 + part * 16);
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        __syncwarp();
    }

    // Bit i set: token c0+i starts a folded segment in this warp's direction.
    __device__ __forceinline__ uint32_t reset_mask(int c0, int len) const
    {
        if (p.seg_len <= 0) return 0u;
        uint32_t m = 0;
        const int start = dir == 0 ? 0 : p.seg_len - 1;
        int ph = c0 % p.seg_len;
        for (int i = 0; i < len; ++i) {
            if (ph == start) m |= 1u << i;
            ph = (ph + 1 == p.seg_len) ? 0 : ph + 1;
        }
        return m;
    }

    // Scan the staged chunk. FIN: last phase (emit output), else partial y.
    // SEG: folded sequence (segment-start decay forced to 0). Tokens past len
    // up to the unroll multiple read delta = x = 0 (zero_tail), which leaves
    // h unchanged.
    // CK: store the state entering every 4-token chunk of the row, in this
    // direction's scan order, before the chunk's first token in that order
    // (the gradient's checkpoints; G == 1).
    template <int DIR, bool FIN, bool SEG, bool GATE, bool CK>
    __device__ __forceinline__ void scan_chunk(f2 (&h)[NS / 2], const f2 (&Ap)[NS / 2], float Dsum,
                                               float (&xh)[3], int s, int c0, int len,
                                               uint32_t rmask)
    {
        const unsigned char *st = stage(s);
        const float *bc = reinterpret_cast<const float *>(wsm + Lay::oBC);
        T *ot = reinterpret_cast<T *>(wsm + Lay::oOT) + r * Lay::OTP;
        const float *py = reinterpret_cast<const float *>(st + Lay::oPY);
        float *yrow = (DIRS == 3 && !FIN) ? p.ybuf + (grp * p.piece_len + (c0 - ta)) * RPW + r : nullptr;
        const uint32_t lead = lead_of(lane_emod, c0);
        const T *rd = reinterpret_cast<const T *>(st + Lay::oD + Lay::row_off(r) + lead);
        const T *rx = reinterpret_cast<const T *>(st + Lay::oX + Lay::row_off(r) + lead);
        const T *rz = reinterpret_cast<const T *>(st + Lay::oZ + Lay::row_off(r) + lead);
        const int n4 = (len + UNR - 1) / UNR * UNR;   // len rounded up to the unroll
#pragma unroll 1
        for (int k0 = 0; k0 < n4; k0 += UNR) {
#pragma unroll
            for (int j = 0; j < UNR; ++j) {
                const int i = (DIR == 0) ? (k0 + j) : (n4 - 1 - k0 - j);
                if (CK) {
                    static_assert(!CK || G == 1, "checkpoints hold one channel per lane");
                    const int t = c0 + i;
                    const bool first = DIR == 0 ? (t & 3) == 0 : ((t & 3) == 3 || t == p.L - 1);
                    if (i < len && first) {
                        // (lanes past the last channel hold zeros: their staged
                        // rows are not copied, so their states are undefined)
                        const bool act = d0 + r < p.dim;
                        float *dst = ck_row + (long long)(t >> 2) * 512;
#pragma unroll
                        for (int q = 0; q < NS / 2; ++q) {
                            const float2 v = unpack2(h[q]);
                            // (streaming stores: the adjoint reads them after this
                            // kernel, long after they would have left L2 anyway)
                            __stcs(dst + (2 * q) * 32, act ? v.x : 0.f);
                            __stcs(dst + (2 * q + 1) * 32, act ? v.y : 0.f);
                        }
                    }
                }
                float dtv = ld_as_f32(rd + i);
                if (SP) dtv = softplus_f32(dtv + dbias_l);
                const float xv = conv_input<SEG>(ld_as_f32(rx + i), xh, i, len, rmask);
                const float dx = dtv * xv;
                const f2 dd = pack2(dtv, dtv), uu = pack2(dx, dx);
                const float *bcp = bc + i * 32;
                f2 ya = pack2(0.f, 0.f), yb = pack2(0.f, 0.f);
                f2 ll = pack2(0.f, 0.f);
                if (SEG) {                        // -inf at a segment start, else 0
                    const float lam = __uint_as_float(0xff800000u & (0u - ((rmask >> i) & 1u)));
                    ll = pack2(lam, lam);
                }
#pragma unroll
                for (int q = 0; q < NS / 4; ++q) {
                    f2 B0, B1, C0, C1;
                    lds_2xf2(bcp + g * NS + 4 * q, B0, B1);
                    lds_2xf2(bcp + 16 + g * NS + 4 * q, C0, C1);
                    const f2 e0 = SEG ? ex2_fma2(dd, Ap[2 * q], ll) : ex2_mul2(dd, Ap[2 * q]);
                    const f2 e1 = SEG ? ex2_fma2(dd, Ap[2 * q + 1], ll) : ex2_mul2(dd, Ap[2 * q + 1]);
                    h[2 * q] = fma2(e0, h[2 * q], mul2(uu, B0));
                    h[2 * q + 1] = fma2(e1, h[2 * q + 1], mul2(uu, B1));
                    ya = fma2(C0, h[2 * q], ya);
                    yb = fma2(C1, h[2 * q + 1], yb);
                }
                const float2 y2 = unpack2(add2(ya, yb));
                float y = y2.x + y2.y;
                if (G >= 2) y += __shfl_xor_sync(0xffffffffu, y, 1);
                if (G >= 4) y += __shfl_xor_sync(0xffffffffu, y, 2);
                // (all G lanes of a channel hold the same y and store it alike)
                if (!FIN) {
                    // with CONV each direction adds its own skip D * u here
                    if (CONV) y = fmaf(Dsum, xv, y);
                    if (DIRS == 3) st_global_if(yrow + i * RPW, y, i < len);
                } else {
                    float tot = y + fmaf(Dsum, xv, (DIRS == 3) ? py[i * RPW + r] : 0.f);
                    if (GATE) tot *= silu_f32<T>(ld_as_f32(rz + i));
                    st_from_f32(ot + i, tot);
                }
            }
        }
        __syncwarp();
    }

    // Zero delta and x of the tokens between len and the unroll multiple in
    // this lane's row slot (only for a partial chunk). With SP the padded
    // delta is -inf, whose softplus is exactly 0.
    __device__ void zero_tail(int s, int c0, int len)
    {
        const int n4 = (len + UNR - 1) / UNR * UNR;
        if (n4 != len && (G == 1 || g == 0)) {
            unsigned char *st = stage(s);
            const uint32_t lead = lead_of(lane_emod, c0);
            T *rd = reinterpret_cast<T *>(st + Lay::oD + Lay::row_off(r) + lead);
            T *rx = reinterpret_cast<T *>(st + Lay::oX + Lay::row_off(r) + lead);
            for (int i = len; i < n4; ++i) {
                rd[i] = T(SP ? -INFINITY : 0.f);
                rx[i] = T(0.f);
            }
        }
        __syncwarp();
    }

    // Write the chunk's outputs from the output tile with row-contiguous
    // stores: lane = token within the chunk, 32/kTC rows per pass.
    __device__ void store_out(int c0, int c1)
    {
        const T *ot = reinterpret_cast<const T *>(wsm + Lay::oOT);
        constexpr int RPI = 32 / kTC;                 // rows per pass
        const int len = c1 - c0;
        const int i = lane % kTC, sub = lane / kTC;
        const int rows = min(RPW, p.dim - d0);
        T *op = out_row0 + (long long)sub * p.L + c0 + i;
        const long long step = (long long)RPI * p.L;
        const bool in = i < len;
#pragma unroll 4
        for (int rr = sub; rr < rows; rr += RPI, op += step) st_global_if(op, ot[rr * Lay::OTP + i], in);
        __syncwarp();
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

    template <bool FIN, bool SEG, bool GATE, bool CK>
    __device__ __forceinline__ void scan_dir(f2 (&h)[NS / 2], const f2 (&Ap)[NS / 2], float Dsum,
                                             float (&xh)[3], int s, int c0, int len, uint32_t rmask)
    {
        if (dir == 0) scan_chunk<0, FIN, SEG, GATE, CK>(h, Ap, Dsum, xh, s, c0, len, rmask);
        else scan_chunk<1, FIN, SEG, GATE, CK>(h, Ap, Dsum, xh, s, c0, len, rmask);
    }

    // The scan_chunk instance for this chunk: last phase or not, folded,
    // gate, checkpoints (the gate only matters in the last phase).
    __device__ __forceinline__ void scan_dispatch(bool fin, bool seg, bool gate, bool ck, f2 (&h)[NS / 2],
                                                  const f2 (&Ap)[NS / 2], float Dsum, float (&xh)[3], int s,
                                                  int c0, int len, uint32_t rmask)
    {
#define VSSM_SCAN_CASE(F, S, Z)                                                          \
        if (ck) scan_dir<F, S, Z, (G == 1)>(h, Ap, Dsum, xh, s, c0, len, rmask);        \
        else scan_dir<F, S, Z, false>(h, Ap, Dsum, xh, s, c0, len, rmask);
        if (fin) {
            if (seg) {
                if (gate) { VSSM_SCAN_CASE(true, true, true) } else { VSSM_SCAN_CASE(true, true, false) }
            } else {
                if (gate) { VSSM_SCAN_CASE(true, false, true) } else { VSSM_SCAN_CASE(true, false, false) }
            }
        } else {
            if (seg) { VSSM_SCAN_CASE(false, true, false) } else { VSSM_SCAN_CASE(false, false, false) }
        }
#undef VSSM_SCAN_CASE
    }

    // History of the convolution at the first token t0 this warp visits in
    // its direction: x at t0 -/+ 1, 2, 3, zero outside the row and, folded,
    // outside t0's segment.
    __device__ __forceinline__ void conv_history(float (&xh)[3], int t0) const
    {
        const T *xr = reinterpret_cast<const T *>(rowp[1]);
        const bool act = d0 + r < p.dim;
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const int ts = dir == 0 ? t0 - 1 - j : t0 + 1 + j;
            const bool in = act && ts >= 0 && ts < p.L &&
                            (p.seg_len <= 0 || ts / p.seg_len == t0 / p.seg_len);
            xh[j] = in ? ld_as_f32(xr + ts) : 0.f;
        }
    }

    // Input of token i of the chunk: x itself, or silu of the convolution
    // (CONV), which then shifts x into the history (not for the padding past
    // len, which must leave it as it is). A segment start clears the history.
    template <bool SEG>
    __device__ __forceinline__ float conv_input(float xraw, float (&xh)[3], int i, int len,
                                                uint32_t rmask) const
    {
        if (!CONV) return xraw;
        if (SEG) {
            const float keep = ((rmask >> i) & 1u) ? 0.f : 1.f;
            xh[0] *= keep;
            xh[1] *= keep;
            xh[2] *= keep;
        }
        float pre = fmaf(cw[3], xraw, cb);
        pre = fmaf(cw[2], xh[0], pre);
        pre = fmaf(cw[1], xh[1], pre);
        pre = fmaf(cw[0], xh[2], pre);
        const bool in = i < len;
        xh[2] = in ? xh[1] : xh[2];
        xh[1] = in ? xh[0] : xh[1];
        xh[0] = in ? xraw : xh[0];
        return silu_f32<T>(pre);
    }

    // A * log2(e) for this lane's states, and a zero state.
    __device__ __forceinline__ void init_state(f2 (&Ap)[NS / 2], f2 (&h)[NS / 2]) const
    {
        const int d = d0 + r;
        const bool active = d < p.dim;
        constexpr float kLog2e = 1.4426950408889634f;
#pragma unroll
        for (int j = 0; j < NS / 2; ++j) {
            const int n = g * NS + 2 * j;
            const float a0 = active ? p.A[dir][(long long)d * 16 + n] * kLog2e : 0.f;
            const float a1 = active ? p.A[dir][(long long)d * 16 + n + 1] * kLog2e : 0.f;
            Ap[j] = pack2(a0, a1);
            h[j] = pack2(0.f, 0.f);
        }
    }

    __device__ __forceinline__ float *summary_ptr(int j) const
    {
        return p.summ + (((long long)slot * p.srows + (long long)b * p.rgroups + rg) * p.pieces + j) * kSummFloats;
    }

    // State entering this warp's piece, from the summaries of the pieces that
    // precede it in this warp's direction (Vim page §3.1, parallel scan). A
    // piece maps a state h to P*h + hp, with P = 2^(A*log2e * its delta sum)
    // per state (0 when a folded reset lies inside it) and hp its state from
    // zero. Composing the maps, (P1, h1) then (P2, h2) = (P1*P2, P2*h1 + h2),
    // is associative, and the exclusive prefix applied to h = 0 reduces to
    // h <- P*h + hp over the preceding pieces in order.
    __device__ void carry_in(f2 (&h)[NS / 2], const f2 (&Ap)[NS / 2]) const
    {
        static_assert(G == 1, "summaries hold one channel per lane");
        const int n = dir == 0 ? piece : p.pieces - 1 - piece;
        constexpr int kBatch = 4;        // summaries loaded together (L2 latency)
        for (int s0 = 0; s0 < n; s0 += kBatch) {
            float v[kBatch][17];
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                if (s0 + k < n) {
                    const float *u = summary_ptr(dir == 0 ? s0 + k : p.pieces - 1 - s0 - k);
#pragma unroll
                    for (int m = 0; m < 17; ++m) v[k][m] = __ldcg(u + m * 32 + lane);
                }
            }
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                if (s0 + k < n) {
                    const float S = v[k][16];
                    const bool cut = __float_as_uint(S) == kCutBits;
                    const f2 SS = pack2(S, S);
#pragma unroll
                    for (int q = 0; q < NS / 2; ++q) {
                        const f2 e = cut ? pack2(0.f, 0.f) : ex2_mul2(SS, Ap[q]);
                        h[q] = fma2(e, h[q], pack2(v[k][2 * q], v[k][2 * q + 1]));
                    }
                }
            }
        }
    }

    // Scan the staged chunk for the piece summary: the state recurrence and
    // the delta sum only (no C, no output).
    template <int DIR, bool SEG>
    __device__ __forceinline__ void summary_chunk(f2 (&h)[NS / 2], const f2 (&Ap)[NS / 2], float &S,
                                                  float (&xh)[3], int s, int c0, int len,
                                                  uint32_t rmask)
    {
        const unsigned char *st = stage(s);
        const float *bc = reinterpret_cast<const float *>(wsm + Lay::oBC);
        const uint32_t lead = lead_of(lane_emod, c0);
        const T *rd = reinterpret_cast<const T *>(st + Lay::oD + Lay::row_off(r) + lead);
        const T *rx = reinterpret_cast<const T *>(st + Lay::oX + Lay::row_off(r) + lead);
        const int n4 = (len + UNR - 1) / UNR * UNR;
#pragma unroll 1
        for (int k0 = 0; k0 < n4; k0 += UNR) {
#pragma unroll
            for (int j = 0; j < UNR; ++j) {
                const int i = (DIR == 0) ? (k0 + j) : (n4 - 1 - k0 - j);
                float dtv = ld_as_f32(rd + i);
                if (SP) dtv = softplus_f32(dtv + dbias_l);
                const float xv = conv_input<SEG>(ld_as_f32(rx + i), xh, i, len, rmask);
                S += dtv;
                const float dx = dtv * xv;
                const f2 dd = pack2(dtv, dtv), uu = pack2(dx, dx);
                const float *bcp = bc + i * 32;
                f2 ll = pack2(0.f, 0.f);
                if (SEG) {
                    const float lam = __uint_as_float(0xff800000u & (0u - ((rmask >> i) & 1u)));
                    ll = pack2(lam, lam);
                }
#pragma unroll
                for (int q = 0; q < NS / 4; ++q) {
                    f2 B0, B1;
                    lds_2xf2(bcp + g * NS + 4 * q, B0, B1);
                    const f2 e0 = SEG ? ex2_fma2(dd, Ap[2 * q], ll) : ex2_mul2(dd, Ap[2 * q]);
                    const f2 e1 = SEG ? ex2_fma2(dd, Ap[2 * q + 1], ll) : ex2_mul2(dd, Ap[2 * q + 1]);
                    h[2 * q] = fma2(e0, h[2 * q], mul2(uu, B0));
                    h[2 * q + 1] = fma2(e1, h[2 * q + 1], mul2(uu, B1));
                }
            }
        }
        __syncwarp();
    }

    // Summary of this warp's piece in its direction (see carry_in).
    __device__ void run_summary()
    {
        static_assert(G == 1, "summaries hold one channel per lane");
        f2 Ap[NS / 2], h[NS / 2];
        init_state(Ap, h);
        float xh[3] = {0.f, 0.f, 0.f};
        if (CONV) conv_history(xh, dir == 0 ? ta : tb - 1);
        float S = 0.f;
        bool cut = false;
        const bool seg = p.seg_len > 0;
        const int nk = (tb - ta + kTC - 1) / kTC;
        for (int k = 0; k < NST; ++k) {
            if (k < nk) {
                int c0, c1;
                chunk_range(k, ta, tb, c0, c1);
                issue(k, c0, c1, false);
            } else {
                cp_async_commit();
            }
        }
        for (int k = 0; k < nk; ++k) {
            const int s = k % NST;
            int c0, c1;
            chunk_range(k, ta, tb, c0, c1);
            cp_async_wait<NST - 1>();
            __syncwarp();
            const int len = c1 - c0;
            zero_tail(s, c0, len);
            widen_bc(s, len);
            const uint32_t rmask = reset_mask(c0, len);
            cut = cut || rmask != 0u;
            if (dir == 0) {
                if (seg) summary_chunk<0, true>(h, Ap, S, xh, s, c0, len, rmask);
                else summary_chunk<0, false>(h, Ap, S, xh, s, c0, len, rmask);
            } else {
                if (seg) summary_chunk<1, true>(h, Ap, S, xh, s, c0, len, rmask);
                else summary_chunk<1, false>(h, Ap, S, xh, s, c0, len, rmask);
            }
            if (k + NST < nk) {
                int n0, n1;
                chunk_range(k + NST, ta, tb, n0, n1);
                issue(s, n0, n1, false);
            } else {
                cp_async_commit();
            }
        }
        cp_async_wait<0>();
        float *u = summary_ptr(piece);
#pragma unroll
        for (int q = 0; q < NS / 2; ++q) {
            const float2 v = unpack2(h[q]);
            u[(2 * q) * 32 + lane] = v.x;
            u[(2 * q + 1) * 32 + lane] = v.y;
        }
        u[16 * 32 + lane] = cut ? __uint_as_float(kCutBits) : S;
    }

    __device__ void run()
    {
        // ---- per-lane parameters
        const int d = d0 + r;
        const bool active = d < p.dim;
        f2 Ap[NS / 2], h[NS / 2];
        init_state(Ap, h);
        if constexpr (CARRY) carry_in(h, Ap);
        float xh[3] = {0.f, 0.f, 0.f};
        if (CONV) conv_history(xh, dir == 0 ? ta : tb - 1);
        float Dsum = 0.f;   // skip weight applied to the input: both directions' (x
                            // shared) or this direction's own (CONV: inputs differ)
        if (active) {
            if (DIRS == 3 && !CONV) {
                Dsum = (p.D[0] ? p.D[0][d] : 0.f) + (p.D[1] ? p.D[1][d] : 0.f);
            } else {
                Dsum = p.D[dir] ? p.D[dir][d] : 0.f;
            }
        }
        const bool hasZ = p.z != nullptr;
        const bool seg = p.seg_len > 0;
        const bool ck = ck_row != nullptr;

        const int Lv = tb - ta;
        const int H = (DIRS == 3) ? (Lv + 1) / 2 : Lv;
        const int nphase = (DIRS == 3) ? 2 : 1;
        uint32_t kk = 0;   // ring position
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
            // One copy group per ring slot in flight (empty groups past the end
            // keep the group count uniform).
            for (int k = 0; k < NST; ++k) {
                if (k < nk) {
                    int c0, c1;
                    chunk_range(k, lo, hi, c0, c1);
                    issue((kk + k) % NST, c0, c1, fin);
                } else {
                    cp_async_commit();
                }
            }
            for (int k = 0; k < nk; ++k, ++kk) {
                const int s = kk % NST;
                int c0, c1;
                chunk_range(k, lo, hi, c0, c1);
                cp_async_wait<NST - 1>();
                __syncwarp();
                const int len = c1 - c0;
                if (DIRS == 3 && fin && p.discard_y && lane < len) {
                    // the partner's partial y of these tokens has been read for
                    // the last time: drop its lines from L2 without a write-back
                    discard_l2(p.ybuf + (grp * p.piece_len + (c0 - ta) + lane) * RPW);
                }
                zero_tail(s, c0, len);
                widen_bc(s, len);
                const uint32_t rmask = reset_mask(c0, len);
                scan_dispatch(fin, seg, hasZ, ck, h, Ap, Dsum, xh, s, c0, len, rmask);
                if (fin) store_out(c0, c1);
                if (k + NST < nk) {
                    int n0, n1;
                    chunk_range(k + NST, lo, hi, n0, n1);
                    issue(s, n0, n1, fin);
                } else {
                    cp_async_commit();
                }
            }
            cp_async_wait<0>();
            if (DIRS == 3 && phase == 0) {
                // Partial y fully written before the partner reads it.
                __threadfence();
                __syncwarp();
                if (lane == 0) mbar_arrive(pairbar);
                bool met = mbar_wait(pairbar, 0, kWaitLimitNs);
                if (!__all_sync(0xffffffffu, met)) {
                    if (lane == 0) atomicOr(p.err, kErrTimeout);
                    ok = false;
                }
            }
        }
        cp_async_wait<0>();
    }
};

// CTAs per SM that the shared-memory footprint allows; used as the register
// budget hint so that registers never limit residency below it.
template <typename T, int G, int DIRS, int W, int NST = kStages>
constexpr int warp_scan_min_blocks()
{
    // 228 KB of shared memory per SM, 1 KB of it reserved per CTA
    constexpr int kb = W * WarpLayout<T, G, DIRS == 3, NST>::kWarpBytes + 1024;
    return (228 * 1024) / kb < 1 ? 1 : ((228 * 1024) / kb > 8 ? 8 : (228 * 1024) / kb);
}

// CARRY: the row is cut into ranges that start from the state carried in by
// warp_carry_kernel's summaries (else every range starts from zero). NST:
// depth of the copy ring.
template <typename T, int G, int DIRS, int W, bool CARRY, bool SP, bool CONV, int NST = kStages,
          int UNR = kUnroll>
__global__ void __launch_bounds__(W * 32, (warp_scan_min_blocks<T, G, DIRS, W, NST>()))
warp_scan_kernel(const WarpScanParams p)
{
    using Lay = WarpLayout<T, G, DIRS == 3, NST>;
    constexpr int NDIR = (DIRS == 3) ? 2 : 1;
    static_assert(W % NDIR == 0, "whole pairs per CTA");
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int warp = threadIdx.x >> 5;
    WarpScan<T, G, DIRS, W, CARRY, SP, CONV, NST, UNR> ws(p);
    ws.lane = threadIdx.x & 31;
    ws.r = ws.lane / G;
    ws.g = ws.lane % G;
    ws.wsm = smem_raw + warp * Lay::kWarpBytes;
    ws.pairbar = reinterpret_cast<uint64_t *>(smem_raw + (warp - warp % NDIR) * Lay::kWarpBytes + Lay::oBar);
    ws.dir = (DIRS == 3) ? (warp % 2) : (DIRS == 1 ? 0 : 1);
    ws.ok = true;
    if (DIRS == 3 && ws.lane == 0 && warp % 2 == 0) {
        mbar_init(ws.pairbar, 2);
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
    ws.rg = rg;
    ws.piece = piece;
    ws.slot = (DIRS == 3) ? ws.dir : 0;
    ws.place();
    ws.run();
}

// Piece summaries for the carry between token ranges of a row: one warp per
// (direction slot, channel group, piece that has a successor in that
// direction). Runs before warp_scan_kernel on the same stream.
template <typename T, int DIRS, int W, bool SP, bool CONV>
__global__ void __launch_bounds__(W * 32, (warp_scan_min_blocks<T, 1, 1, W>()))
warp_carry_kernel(const WarpScanParams p)
{
    using Lay = WarpLayout<T, 1, false>;
    constexpr int NDIR = (DIRS == 3) ? 2 : 1;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int warp = threadIdx.x >> 5;
    const long long per_slot = p.srows * (p.pieces - 1);
    const long long u = (long long)blockIdx.x * W + warp;
    if (u >= NDIR * per_slot) return;
    WarpScan<T, 1, 1, W, false, SP, CONV> ws(p);  // single-direction staging layout
    ws.slot = (int)(u / per_slot);
    const long long rem = u % per_slot;
    const int jj = (int)(rem % (p.pieces - 1));
    const long long row = rem / (p.pieces - 1);
    ws.dir = (DIRS == 3) ? ws.slot : (DIRS == 1 ? 0 : 1);
    ws.lane = threadIdx.x & 31;
    ws.r = ws.lane;
    ws.g = 0;
    ws.wsm = smem_raw + warp * Lay::kWarpBytes;
    ws.pairbar = nullptr;
    ws.ok = true;
    ws.rg = (int)(row % p.rgroups);
    ws.b = (int)(row / p.rgroups);
    ws.piece = ws.dir == 0 ? jj : jj + 1;
    ws.grp = ((long long)ws.b * p.pieces + ws.piece) * p.rgroups + ws.rg;
    ws.place();
    ws.run_summary();
}

}  // namespace vssm
