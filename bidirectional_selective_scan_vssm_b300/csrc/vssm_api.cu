// C ABI of the selective-scan library (declared in include/vssm.h):
// argument validation, planning and launch on the caller's stream.
#include <algorithm>
#include <numeric>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "launch.h"
#include "vssm.h"

// Device error word written by kernels whose bounded waits expire (one per
// device that loads the library).
__device__ unsigned g_vssm_device_error;

// Built-in scratch of vssm_scan_bidir_noalloc: stands in for the caller's
// workspace. Every device that loads the library holds it until the process
// exits; host code reaches it only through noalloc_scratch() below.
static __device__ __align__(256) unsigned char g_vssm_noalloc_scratch[VSSM_NOALLOC_SCRATCH_BYTES];

namespace vssm {

// Multiprocessors of the current device, queried once per device (148 on a
// B300; the same figure when no device is visible, so that sizes reported
// without a GPU match a B300).
int sm_count()
{
    static std::mutex mu;
    static int cnt[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return 148;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!cnt[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
            cudaGetLastError();
            v = 148;
        }
        cnt[dev] = v;
    }
    return cnt[dev];
}

}  // namespace vssm

namespace {

thread_local std::string g_last_error;

int fail(int status, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int status, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return status;
}

int cuda_fail(cudaError_t e, const char *what)
{
    return fail(VSSM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

size_t al256(size_t n) { return (n + 255) / 256 * 256; }

using vssm::sm_count;

// Launch plan for one call.
struct Plan {
    bool warp = false;     // warp-per-channel-group kernel (N = 16) vs general kernel
    int G = 1;             // lanes per channel (warp kernel)
    int W = 4;             // warps per CTA (warp kernel)
    int rgroups = 0;       // channel groups per (batch, piece) (warp kernel)
    long long ngroups = 0; // channel groups x pieces x batch (warp kernel)
    int dirs = 0;          // 1, 2 or 3
    int pieces = 1;        // token ranges per (b, d)
    int piece_len = 0;     // tokens per range
    bool ysmem = false;    // y-buffer in shared memory
    int ypitch = 0;        // floats per channel of the shared y-buffer
    size_t workspace = 0;  // bytes of workspace needed (y-buffer, then carry summaries)
    long long ctas = 0;
    bool carry = false;    // pieces joined by the carry (summary kernel first)
    size_t summ_off = 0;   // byte offset of the summaries in the workspace
    long long srows = 0;   // batch x channel groups
    long long summ_ctas = 0;
};

constexpr int kBidirR = 32, kBidirG = 2;     // 128 threads: 64 forward, 64 backward
constexpr int kOneDirR = 64, kOneDirG = 2;   // 128 threads
constexpr int kYSmemMaxBytes = 48 * 1024;    // shared y-buffer budget per CTA

// Folded sequences are cut into independent pieces (each starts on a reset):
// as many as fill kFoldWaves waves of the warps resident at once, rounded
// down so that no extra, mostly idle wave starts. On the SF-Mamba shape
// (1024 segments of 51 tokens, 32 channel groups) this gives 128 pieces;
// 64 to 1024 pieces measured 3-16 % slower, the 205 of a three-wave target
// 8 % slower.
constexpr int kFoldWaves = 2;

using vssm::kCarryW;
using vssm::warps_per_cta;


// Cost model of one call with each row cut into P ranges of lp tokens, in
// microseconds. It is a least-squares fit to B300 timings of each kernel
// (ncu launch lists over 34 cuts of six shapes, batch 1 x 384 channels x
// 197 tokens to batch 16 x 768 x 1025 and batch 8 x 768 x 4097; 3.4 % rms
// error for the scan, 5.9 % for the summary pass). A kernel's warps run in
// rounds of its residency (warps that fit on the GPU at once); in a round
// each scheduler holds k of them, and a warp costs c(k) cycles per token plus
// a start-up cost. The scan also pays for gathering up to P - 1 summaries.
struct KernelCost {
    double c1, c2, c3;   // cycles per token per warp with 1, 2, >= 3 warps per scheduler
    double start;        // cycles per warp outside the token loop
    double launch_us;    // per launch
};
constexpr KernelCost kScanCost{268.8, 189.2, 173.4, 5717.0, 3.7};
constexpr KernelCost kSummaryCost{170.9, 130.3, 113.4, 620.0, 4.3};
constexpr double kFoldUsPerRange = 0.2;
constexpr double kClockMHz = 2032.0;   // B300 maximum SM clock (the fit's cycle counts are per clock)

double kernel_us(const KernelCost &m, long long warps, long long lp, long long resident)
{
    auto per_token = [&](double k) { return k <= 1.0 ? m.c1 : (k <= 2.0 ? m.c2 : m.c3); };
    const long long kSubParts = 4LL * sm_count();   // schedulers of the GPU
    const long long full = warps / resident, rem = warps - full * resident;
    const double kf = (double)resident / kSubParts;
    double cyc = (double)full * kf * ((double)lp * per_token(kf) + m.start);
    if (rem > 0) {
        const double kr = (double)((rem + kSubParts - 1) / kSubParts);
        cyc += kr * ((double)lp * per_token(kr) + m.start);
    }
    return cyc / kClockMHz + m.launch_us;
}

// Warps of a kernel resident on the GPU at once: shared memory per SM
// (228 KB, 1 KB reserved per CTA) over the CTA footprint.
long long resident_warps(size_t warp_bytes, int warps_per_cta)
{
    const long long per_sm = (228 * 1024) / ((long long)warps_per_cta * warp_bytes + 1024);
    return (long long)sm_count() * std::max(1LL, std::min(32LL, per_sm)) * warps_per_cta;
}

struct CarryShape {
    long long row_warps;         // batch x channel groups x directions
    long long res_scan, res_summary;
};

double carry_us(const CarryShape &c, long long lp, int P)
{
    double t = kernel_us(kScanCost, c.row_warps * P, lp, c.res_scan);
    if (P > 1)
        t += kernel_us(kSummaryCost, c.row_warps * (P - 1), lp, c.res_summary) +
             kFoldUsPerRange * (P - 1);
    return t;
}

// Ranges per row (cut on the 16-token chunk grid, at most 32, at least 32
// tokens each) that minimise carry_us; 1 unless cutting saves 5 % or more.
// Returns the range length in *lp_out.
int auto_carry_pieces(const CarryShape &c, int L, long long *lp_out)
{
    *lp_out = L;
    if (c.row_warps <= 0 || c.row_warps >= c.res_scan || L < 64) return 1;
    const double one = carry_us(c, L, 1);
    double best = 0.0;
    int bestP = 1;
    long long bestLp = L;
    for (int P = 2; P <= 32; ++P) {
        const long long lp = ((long long)L + P - 1) / P;
        if (lp < 32) break;
        const long long lp16 = (lp + 15) / 16 * 16;
        const int pieces = (int)(((long long)L + lp16 - 1) / lp16);
        if (pieces < 2) continue;
        const double t = carry_us(c, lp16, pieces);
        if (bestP == 1 || t < best) {
            best = t;
            bestP = pieces;
            bestLp = lp16;
        }
    }
    if (bestP == 1 || best >= 0.95 * one) return 1;
    *lp_out = bestLp;
    return bestP;
}

template <typename T>
CarryShape carry_shape(long long row_warps, unsigned dirs)
{
    CarryShape c;
    c.row_warps = row_warps;
    const size_t scan_bytes = dirs == 3 ? vssm::WarpLayout<T, 1, true>::kWarpBytes
                                        : vssm::WarpLayout<T, 1, false>::kWarpBytes;
    c.res_scan = resident_warps(scan_bytes, warps_per_cta(1));
    c.res_summary = resident_warps(vssm::WarpLayout<T, 1, false>::kWarpBytes, kCarryW);
    return c;
}

// Plan for the warp kernel (dstate == 16). pieces_req: 0 lets the plan
// choose; otherwise each row is cut into about that many token ranges
// joined by the carry.
void make_warp_plan(const vssm_scan_args *a, int seg_len, int pieces_req, Plan *pl)
{
    const unsigned dirs = a->dir_flags;
    const int ndir = dirs == 3 ? 2 : 1;
    pl->warp = true;
    pl->dirs = (int)dirs;
    const long long nseg = seg_len > 0 ? (a->seqlen + seg_len - 1) / seg_len : 1;
    // One lane per channel, all 16 states in its registers. Measured on
    // B300, the variants that split a channel's states over 2 or 4 lanes
    // (more warps, a shuffle per token) were slower on every workload, long
    // rows with few channels included.
    const int G = 1;
    pl->G = G;
    pl->W = warps_per_cta(G);
    const int rpw = 32 / G;
    pl->rgroups = (a->dim + rpw - 1) / rpw;
    pl->pieces = 1;
    pl->piece_len = a->seqlen;
    pl->srows = (long long)a->batch * pl->rgroups;
    long long lp = a->seqlen;
    int carry_p = pieces_req;
    if (carry_p > 1) {                     // ceil(L / ceil(L / P)) ranges
        lp = std::max(1LL, ((long long)a->seqlen + carry_p - 1) / carry_p);
        carry_p = (int)(((long long)a->seqlen + lp - 1) / lp);
    } else if (carry_p == 0 && seg_len == 0) {
        const CarryShape cs = a->dtype == VSSM_F32 ? carry_shape<float>(pl->srows * ndir, dirs)
                                                   : carry_shape<__nv_bfloat16>(pl->srows * ndir, dirs);
        carry_p = auto_carry_pieces(cs, a->seqlen, &lp);
    }
    if (carry_p > 1) {
        pl->piece_len = (int)lp;
        pl->pieces = carry_p;
        pl->carry = true;
    } else if (seg_len > 0 && a->seqlen > 0) {
        const long long per_piece_warps = (long long)a->batch * pl->rgroups * ndir;
        const size_t wb = a->dtype == VSSM_F32
                              ? (dirs == 3 ? vssm::WarpLayout<float, 1, true>::kWarpBytes
                                           : vssm::WarpLayout<float, 1, false>::kWarpBytes)
                              : (dirs == 3 ? vssm::WarpLayout<__nv_bfloat16, 1, true>::kWarpBytes
                                           : vssm::WarpLayout<__nv_bfloat16, 1, false>::kWarpBytes);
        const long long target = kFoldWaves * resident_warps(wb, pl->W);
        long long want = target / std::max<long long>(1, per_piece_warps);
        want = std::max<long long>(1, std::min<long long>(want, nseg));
        const long long per = (nseg + want - 1) / want;        // segments per piece
        pl->pieces = (int)((nseg + per - 1) / per);
        pl->piece_len = (int)(per * seg_len);
    }
    pl->ngroups = (long long)a->batch * pl->pieces * pl->rgroups;
    const int gpc = pl->W / ndir;
    pl->ctas = (pl->ngroups + gpc - 1) / gpc;
    pl->workspace = dirs == 3 ? (size_t)pl->ngroups * pl->piece_len * rpw * sizeof(float) : 0;
    if (pl->carry) {
        pl->summ_off = (pl->workspace + 255) / 256 * 256;
        pl->workspace = pl->summ_off + (size_t)ndir * pl->srows * pl->pieces * vssm::kSummFloats * sizeof(float);
        const long long units = (long long)ndir * pl->srows * (pl->pieces - 1);
        pl->summ_ctas = (units + kCarryW - 1) / kCarryW;
    }
}

// pieces_req as in make_warp_plan; only the dstate-16 kernel joins pieces by
// the carry, and the caller rejects pieces_req > 1 for other state sizes.
int make_plan(const vssm_scan_args *a, int seg_len, int pieces_req, Plan *pl)
{
    if (a->dstate == vssm::kMaxState) {
        make_warp_plan(a, seg_len, pieces_req, pl);
        return VSSM_OK;
    }
    const unsigned dirs = a->dir_flags;
    pl->dirs = (int)dirs;
    const int R = (dirs == 3) ? kBidirR : kOneDirR;
    const long long dblocks = (a->dim + R - 1) / R;
    pl->pieces = 1;
    pl->piece_len = a->seqlen;
    if (seg_len > 0 && a->seqlen > 0) {
        // Split each folded row at segment boundaries so that the grid has
        // enough CTAs; every piece starts on a reset, so pieces are independent.
        const long long nseg = (a->seqlen + seg_len - 1) / seg_len;
        const long long target = 8LL * sm_count();
        long long want = (target + (long long)a->batch * dblocks - 1) /
                         std::max<long long>(1, (long long)a->batch * dblocks);
        want = std::max<long long>(1, std::min<long long>(want, nseg));
        const long long per = (nseg + want - 1) / want;        // segments per piece
        pl->pieces = (int)((nseg + per - 1) / per);
        pl->piece_len = (int)(per * seg_len);
    }
    pl->ctas = (long long)a->batch * pl->pieces * dblocks;
    pl->ysmem = false;
    pl->workspace = 0;
    if (dirs == 3) {
        const int lv = std::min(a->seqlen, pl->piece_len);
        const int pitch = lv | 1;                              // odd: rows hit distinct banks
        if ((long long)R * pitch * 4 <= kYSmemMaxBytes) {
            pl->ysmem = true;
            pl->ypitch = pitch;
        } else {
            pl->workspace = (size_t)a->batch * a->dim * a->seqlen * sizeof(float);
        }
    }
    return VSSM_OK;
}

// need_out: the call writes a->out (the gradient does not read it).
int validate(const vssm_scan_args *a, int seg_len, bool folded, bool need_out = true)
{
    if (!a) return fail(VSSM_ERR_INVALID_ARG, "args is NULL");
    if (a->batch < 0 || a->dim < 0 || a->seqlen < 0)
        return fail(VSSM_ERR_INVALID_ARG, "negative size (batch=%d dim=%d seqlen=%d)",
                    a->batch, a->dim, a->seqlen);
    if (a->dstate < 1 || a->dstate > vssm::kMaxState)
        return fail(VSSM_ERR_UNSUPPORTED, "dstate=%d outside 1..%d", a->dstate, vssm::kMaxState);
    if (a->dtype != VSSM_F32 && a->dtype != VSSM_BF16)
        return fail(VSSM_ERR_UNSUPPORTED, "unknown dtype %d", a->dtype);
    if (a->dir_flags < 1 || a->dir_flags > 3)
        return fail(VSSM_ERR_INVALID_ARG, "dir_flags=%u: need VSSM_DIR_FWD and/or VSSM_DIR_BWD",
                    a->dir_flags);
    if (folded) {
        if (seg_len < 1) return fail(VSSM_ERR_INVALID_ARG, "seg_len=%d must be >= 1", seg_len);
        if ((a->dir_flags & VSSM_DIR_BWD) && a->seqlen % seg_len != 0)
            return fail(VSSM_ERR_INVALID_ARG,
                        "backward folded scan needs seqlen (%d) to be a multiple of seg_len (%d)",
                        a->seqlen, seg_len);
    }
    const long long tok = (long long)a->batch * a->dim * a->seqlen;
    if (tok == 0) return VSSM_OK;
    if (!a->x || !a->delta || !a->B || !a->C || (need_out && !a->out))
        return fail(VSSM_ERR_INVALID_ARG, "x, delta, B, C and out are required");
    if ((a->dir_flags & VSSM_DIR_FWD) && !a->A_fwd)
        return fail(VSSM_ERR_INVALID_ARG, "A_fwd is required for the forward direction");
    if ((a->dir_flags & VSSM_DIR_BWD) && !a->A_bwd)
        return fail(VSSM_ERR_INVALID_ARG, "A_bwd is required for the backward direction");
    if (a->delta_softplus != 0 && a->delta_softplus != 1)
        return fail(VSSM_ERR_INVALID_ARG, "delta_softplus=%d must be 0 or 1", a->delta_softplus);
    if (a->conv_k < 0 || a->conv_k > vssm::kMaxConv)
        return fail(VSSM_ERR_UNSUPPORTED, "conv_k=%d outside 0..%d", a->conv_k, vssm::kMaxConv);
    if (a->conv_k > 0 && !a->conv_w)
        return fail(VSSM_ERR_INVALID_ARG, "conv_w is required when conv_k > 0");
    const void *ptrs[] = {a->x, a->delta, a->z, a->B, a->C, a->B_bwd, a->C_bwd, a->A_fwd,
                          a->A_bwd, a->D_fwd, a->D_bwd, a->out, a->workspace,
                          a->delta_bwd, a->delta_bias, a->delta_bias_bwd,
                          a->conv_w, a->conv_b, a->conv_w_bwd, a->conv_b_bwd};
    const char *names[] = {"x", "delta", "z", "B", "C", "B_bwd", "C_bwd", "A_fwd",
                           "A_bwd", "D_fwd", "D_bwd", "out", "workspace",
                           "delta_bwd", "delta_bias", "delta_bias_bwd",
                           "conv_w", "conv_b", "conv_w_bwd", "conv_b_bwd"};
    for (int i = 0; i < 20; ++i)
        if (ptrs[i] && !aligned16(ptrs[i]))
            return fail(VSSM_ERR_MISALIGNED, "%s=%p is not 16-byte aligned", names[i], ptrs[i]);
    const size_t es = a->dtype == VSSM_F32 ? 4 : 2;
    const size_t nact = (size_t)tok * es;
    const size_t nbc = (size_t)a->batch * a->seqlen * a->dstate * es;
    const size_t npar = (size_t)a->dim * a->dstate * 4;
    const struct { const void *p; size_t n; const char *name; } ins[] = {
        {a->x, nact, "x"}, {a->delta, nact, "delta"}, {a->z, nact, "z"},
        {a->B, nbc, "B"}, {a->C, nbc, "C"}, {a->B_bwd, nbc, "B_bwd"}, {a->C_bwd, nbc, "C_bwd"},
        {a->A_fwd, npar, "A_fwd"}, {a->A_bwd, npar, "A_bwd"},
        {a->D_fwd, (size_t)a->dim * 4, "D_fwd"}, {a->D_bwd, (size_t)a->dim * 4, "D_bwd"},
        {a->workspace, a->workspace_bytes, "workspace"}, {a->delta_bwd, nact, "delta_bwd"},
        {a->delta_bias, (size_t)a->dim * 4, "delta_bias"},
        {a->delta_bias_bwd, (size_t)a->dim * 4, "delta_bias_bwd"},
        {a->conv_w, (size_t)a->dim * a->conv_k * 4, "conv_w"},
        {a->conv_b, (size_t)a->dim * 4, "conv_b"},
        {a->conv_w_bwd, (size_t)a->dim * a->conv_k * 4, "conv_w_bwd"},
        {a->conv_b_bwd, (size_t)a->dim * 4, "conv_b_bwd"}};
    for (const auto &in : ins)
        if (overlaps(a->out, nact, in.p, in.n))
            return fail(VSSM_ERR_INVALID_ARG, "out overlaps %s", in.name);
    if (a->workspace && overlaps(a->workspace, a->workspace_bytes, a->x, nact))
        return fail(VSSM_ERR_INVALID_ARG, "workspace overlaps x");
    return VSSM_OK;
}

// Address of this device's error word (looked up once per device).
unsigned *device_error_word()
{
    static std::mutex mu;
    static unsigned *addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_vssm_device_error) != cudaSuccess) return nullptr;
        addr[dev] = static_cast<unsigned *>(ptr);
    }
    return addr[dev];
}

// Device address of this device's built-in scratch, looked up once per
// device with that device current. In host code the array's name is only a
// host-side handle, so kernels are given this address instead.
void *noalloc_scratch()
{
    static std::mutex mu;
    static void *addr[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        fail(VSSM_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_vssm_noalloc_scratch);
        if (e != cudaSuccess) {
            fail(VSSM_ERR_CUDA, "cudaGetSymbolAddress(built-in scratch): %s", cudaGetErrorString(e));
            return nullptr;
        }
        addr[dev] = ptr;
    }
    return addr[dev];
}

// Bytes of the gradient's state checkpoints for this call: 16 fp32 per
// 4-token chunk, channel (in groups of 32) and direction.
size_t ckpt_bytes(const vssm_scan_args *a)
{
    const size_t ndir = a->dir_flags == 3 ? 2 : 1;
    const size_t rgroups = ((size_t)a->dim + 31) / 32, nch = ((size_t)a->seqlen + 3) / 4;
    return ndir * (size_t)a->batch * rgroups * nch * 512 * sizeof(float);
}

// ckpt: the training forward also stores the gradient's checkpoints there
// (dstate 16 only).
int run(const vssm_scan_args *a, int seg_len, bool folded, int pieces_req, void *stream,
        float *ckpt = nullptr, size_t ckpt_size = 0)
{
    int st = validate(a, seg_len, folded);
    if (st != VSSM_OK) return st;
    if (ckpt) {
        if (a->dstate != vssm::kMaxState)
            return fail(VSSM_ERR_UNSUPPORTED, "checkpoints need dstate %d (got %d)", vssm::kMaxState, a->dstate);
        if (!aligned16(ckpt)) return fail(VSSM_ERR_MISALIGNED, "ckpt is not 16-byte aligned");
        const size_t need = ckpt_bytes(a);
        if (ckpt_size < need)
            return fail(VSSM_ERR_INVALID_ARG, "ckpt of %zu bytes required, %zu given", need, ckpt_size);
        const size_t es = a->dtype == VSSM_F32 ? 4 : 2;
        const size_t nact = (size_t)a->batch * a->dim * a->seqlen * es;
        const size_t nbc = (size_t)a->batch * a->seqlen * a->dstate * es;
        const void *bufs[] = {a->x, a->delta, a->z, a->out, a->delta_bwd, a->B, a->C, a->B_bwd, a->C_bwd,
                              a->workspace};
        const size_t sz[] = {nact, nact, nact, nact, nact, nbc, nbc, nbc, nbc, a->workspace_bytes};
        for (size_t i = 0; i < sizeof(bufs) / sizeof(bufs[0]); ++i)
            if (overlaps(ckpt, need, bufs[i], sz[i]))
                return fail(VSSM_ERR_INVALID_ARG, "ckpt overlaps an input, the output or the workspace");
    }
    if (pieces_req < 0) return fail(VSSM_ERR_INVALID_ARG, "pieces=%d must be >= 0", pieces_req);
    if (pieces_req > 1 && a->dstate != vssm::kMaxState)
        return fail(VSSM_ERR_UNSUPPORTED, "pieces joined by the carry need dstate %d (got %d)",
                    vssm::kMaxState, a->dstate);
    if ((long long)a->batch * a->dim * a->seqlen == 0) return VSSM_OK;
    Plan pl;
    make_plan(a, folded ? seg_len : 0, pieces_req, &pl);
    if (pl.ctas > 0x7fffffffLL || pl.summ_ctas > 0x7fffffffLL)
        return fail(VSSM_ERR_UNSUPPORTED, "problem too large for one grid");
    if (pl.workspace > 0 && (!a->workspace || a->workspace_bytes < pl.workspace))
        return fail(VSSM_ERR_WORKSPACE, "workspace of %zu bytes required, %zu given", pl.workspace,
                    a->workspace ? a->workspace_bytes : (size_t)0);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool f32 = a->dtype == VSSM_F32;
    if (pl.warp) {
        vssm::WarpScanParams w{};
        w.x = a->x;
        w.delta[0] = a->delta;
        w.delta[1] = a->delta_bwd ? a->delta_bwd : a->delta;
        w.dbias[0] = a->delta_bias;
        w.dbias[1] = a->delta_bias_bwd ? a->delta_bias_bwd : a->delta_bias;
        w.conv_w[0] = a->conv_w;
        w.conv_w[1] = a->conv_w_bwd ? a->conv_w_bwd : a->conv_w;
        w.conv_b[0] = a->conv_b;
        w.conv_b[1] = a->conv_b_bwd ? a->conv_b_bwd : a->conv_b;
        w.conv_k = a->conv_k;
        w.z = a->z;
        w.B[0] = a->B;
        w.C[0] = a->C;
        w.B[1] = a->B_bwd ? a->B_bwd : a->B;
        w.C[1] = a->C_bwd ? a->C_bwd : a->C;
        w.A[0] = a->A_fwd;
        w.A[1] = a->A_bwd;
        w.D[0] = a->D_fwd;
        w.D[1] = a->D_bwd;
        w.out = a->out;
        w.ybuf = pl.dirs == 3 ? static_cast<float *>(a->workspace) : nullptr;
        w.discard_y = (reinterpret_cast<uintptr_t>(w.ybuf) & 127u) == 0 && vssm::WarpLayout<float, 1, true>::RPW == 32;
        w.summ = pl.carry ? reinterpret_cast<float *>(static_cast<char *>(a->workspace) + pl.summ_off)
                          : nullptr;
        w.err = device_error_word();
        if (!w.err) return fail(VSSM_ERR_CUDA, "cannot locate the device error word");
        w.total = (long long)a->batch * a->dim * a->seqlen;
        w.batch = a->batch;
        w.dim = a->dim;
        w.L = a->seqlen;
        w.seg_len = folded ? seg_len : 0;
        w.pieces = pl.pieces;
        w.piece_len = pl.piece_len;
        w.rgroups = pl.rgroups;
        w.ngroups = pl.ngroups;
        w.srows = pl.srows;
        w.ckpt = ckpt;
        w.nch = (a->seqlen + 3) / 4;
        const cudaError_t e = vssm::launch_warp(w, pl.dirs, a->dtype == VSSM_F32, pl.carry,
                                                a->delta_softplus != 0, a->conv_k > 0, pl.ctas,
                                                pl.summ_ctas, s);
        return e == cudaSuccess ? VSSM_OK : cuda_fail(e, "launch");
    }
    vssm::ScanParams p{};
    p.x = a->x;
    p.delta[0] = a->delta;
    p.delta[1] = a->delta_bwd ? a->delta_bwd : a->delta;
    p.dbias[0] = a->delta_bias;
    p.dbias[1] = a->delta_bias_bwd ? a->delta_bias_bwd : a->delta_bias;
    p.softplus = a->delta_softplus;
    p.conv_w[0] = a->conv_w;
    p.conv_w[1] = a->conv_w_bwd ? a->conv_w_bwd : a->conv_w;
    p.conv_b[0] = a->conv_b;
    p.conv_b[1] = a->conv_b_bwd ? a->conv_b_bwd : a->conv_b;
    p.conv_k = a->conv_k;
    p.z = a->z;
    p.B[0] = a->B;
    p.C[0] = a->C;
    p.B[1] = a->B_bwd ? a->B_bwd : a->B;
    p.C[1] = a->C_bwd ? a->C_bwd : a->C;
    p.A[0] = a->A_fwd;
    p.A[1] = a->A_bwd;
    p.D[0] = a->D_fwd;
    p.D[1] = a->D_bwd;
    p.out = a->out;
    p.ybuf = pl.workspace ? static_cast<float *>(a->workspace) : nullptr;
    p.batch = a->batch;
    p.dim = a->dim;
    p.L = a->seqlen;
    p.N = a->dstate;
    p.seg_len = folded ? seg_len : 0;
    p.pieces = pl.pieces;
    p.piece_len = pl.piece_len;
    p.ypitch = pl.ypitch;
    const cudaError_t e = vssm::launch_general(p, pl.dirs, pl.ysmem, f32, pl.ctas, s);
    return e == cudaSuccess ? VSSM_OK : cuda_fail(e, "launch");
}

struct GradPlan {
    int ndir = 1, rgroups = 0, nch = 0;
    int nrange = 1, rch = 0;          // token ranges per row for the adjoint, chunks per range
    bool summaries = false;           // ranges joined by the adjoint summaries (else independent)
    long long ngroups = 0;
    size_t ckpt_bytes = 0, part_off = 0, summ_off = 0, workspace = 0;
};

// Rows are cut into ranges for the adjoint when there are too few of them
// to fill the GPU (about two waves of the adjoint's two-warp CTAs at four
// per SM), keeping at least 16 chunks (64 tokens) per range; the ranges are
// joined by the adjoint summaries (grad_adj_summary_kernel). Folded rows are
// cut at segment starts instead, where the reset cuts the adjoint in both
// directions (the decay that would carry lambda across is 0), so their
// ranges are independent: no summaries, and as many as fill the GPU.
constexpr int kGradMaxRanges = 16, kGradMinRangeChunks = 16, kGradMaxIndepRanges = 4096;

GradPlan make_grad_plan(const vssm_scan_args *a, int seg_len)
{
    const long long kGradTargetCtas = 8LL * sm_count();
    GradPlan g;
    g.ndir = a->dir_flags == 3 ? 2 : 1;
    g.rgroups = (a->dim + 31) / 32;
    g.ngroups = (long long)a->batch * g.rgroups;
    g.nch = (a->seqlen + vssm::kTG - 1) / vssm::kTG;
    g.rch = g.nch;
    // chunks per step of segment-aligned ranges: seg_len / gcd(seg_len, kTG)
    const int unit = seg_len > 0 ? seg_len / std::gcd(seg_len, vssm::kTG) : 0;
    if (unit > 0 && unit < g.nch && g.ngroups > 0 && g.ngroups < 2 * kGradTargetCtas) {
        const long long want = std::min<long long>(kGradMaxIndepRanges,
                                                   (2 * kGradTargetCtas + g.ngroups - 1) / g.ngroups);
        long long rch = (g.nch + want - 1) / want;
        rch = std::max<long long>(unit, (rch + unit - 1) / unit * unit);
        const int r = (int)((g.nch + rch - 1) / rch);
        if (r > 1) {
            g.rch = (int)rch;
            g.nrange = r;
        }
    } else if (g.ngroups > 0 && g.ngroups < kGradTargetCtas) {
        const long long want = std::min<long long>(kGradMaxRanges, (kGradTargetCtas + g.ngroups - 1) / g.ngroups);
        const int r = (int)std::min<long long>(want, g.nch / kGradMinRangeChunks);
        if (r > 1) {
            g.rch = (g.nch + r - 1) / r;
            g.nrange = (g.nch + g.rch - 1) / g.rch;
            g.summaries = true;
        }
    }
    g.ckpt_bytes = (size_t)g.ndir * g.ngroups * g.nch * 512 * sizeof(float);
    g.part_off = (g.ckpt_bytes + 255) / 256 * 256;
    const size_t part_end = a->dir_flags == 3 ? g.part_off + (size_t)g.ngroups * a->seqlen * 96 * sizeof(float)
                                              : g.ckpt_bytes;
    g.summ_off = (part_end + 255) / 256 * 256;
    g.workspace = g.summaries ? g.summ_off + (size_t)g.ndir * g.ngroups * g.nrange * 1024 * sizeof(float)
                              : part_end;
    return g;
}


// ---- host-buffer pipeline (vssm_scan_host)

// Streams and events of the pipeline, created once per device and kept for
// the life of the process; calls on one device take the mutex while they
// enqueue, so that two calls never interleave their use of the events.
constexpr int kHostRing = 3;           // device slots in flight
struct HostPipe {
    std::mutex mu;
    bool ready = false;
    cudaStream_t copy = nullptr, comp = nullptr, back = nullptr;
    cudaEvent_t fork = nullptr, params = nullptr, join = nullptr;
    cudaEvent_t in[kHostRing] = {}, done[kHostRing] = {}, out[kHostRing] = {};
};

HostPipe *host_pipe(int *status)
{
    static std::mutex mu;
    static HostPipe *pipes[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        *status = fail(VSSM_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!pipes[dev]) {
        HostPipe *hp = new HostPipe;
        const unsigned sf = cudaStreamNonBlocking, ef = cudaEventDisableTiming;
        e = cudaStreamCreateWithFlags(&hp->copy, sf);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp->comp, sf);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp->back, sf);
        cudaEvent_t *evs[] = {&hp->fork, &hp->params, &hp->join};
        for (cudaEvent_t *ev : evs)
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, ef);
        for (int i = 0; i < kHostRing && e == cudaSuccess; ++i) {
            e = cudaEventCreateWithFlags(&hp->in[i], ef);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp->done[i], ef);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp->out[i], ef);
        }
        if (e != cudaSuccess) {
            *status = fail(VSSM_ERR_CUDA, "creating the pipeline's streams: %s", cudaGetErrorString(e));
            return nullptr;      // (the partial objects are kept; nothing else uses them)
        }
        hp->ready = true;
        pipes[dev] = hp;
    }
    return pipes[dev];
}

// How a host-pipeline call is cut: whole batch entries per slice when there
// are at least as many entries as slices, else channel ranges (multiples of
// 32) of one batch entry each.
struct HostCut {
    bool by_batch = true;
    int per_b = 1;           // batch entries per slice (by_batch)
    int per_d = 0;           // channels per slice (!by_batch)
    int nslices = 0;
    size_t slot_bytes = 0;   // one ring slot
    size_t ws_off = 0;       // scan workspace within a slot
    size_t up_bytes = 0;     // B, C and per-channel parameters
    size_t total = 0;
};


int host_cut(const vssm_scan_args *a, int seg_len, int slices, HostCut *c)
{
    if (slices < 0) return fail(VSSM_ERR_INVALID_ARG, "slices=%d must be >= 0", slices);
    const int S = slices == 0 ? 8 : slices;
    const size_t es = a->dtype == VSSM_F32 ? 4 : 2;
    const size_t L = (size_t)a->seqlen, N = (size_t)a->dstate, D = (size_t)a->dim;
    c->by_batch = a->batch >= S;
    int rows_b = 1, rows_d = a->dim;
    if (c->by_batch) {
        c->per_b = (a->batch + S - 1) / S;
        c->nslices = (a->batch + c->per_b - 1) / c->per_b;
        rows_b = c->per_b;
    } else {
        const int per_entry = std::max(1, (S + a->batch - 1) / std::max(1, a->batch));
        c->per_d = std::max(32, ((a->dim + per_entry - 1) / per_entry + 31) / 32 * 32);
        const int nd = (a->dim + c->per_d - 1) / c->per_d;
        c->nslices = a->batch * nd;
        rows_d = c->per_d;
    }
    // a slot: x, delta, z, delta_bwd, out of one slice, then its scan workspace
    const size_t act = al256((size_t)rows_b * rows_d * L * es);
    // the scan workspace of the largest slice and of the last (smaller) one:
    // a smaller slice may be planned differently
    vssm_scan_args sub = *a;
    sub.batch = rows_b;
    sub.dim = std::min(rows_d, a->dim);
    Plan pl;
    make_plan(&sub, seg_len, 0, &pl);
    size_t ws = pl.workspace;
    if (c->by_batch) {
        sub.batch = a->batch - (c->nslices - 1) * c->per_b;
    } else {
        const int last = a->dim % c->per_d;
        sub.dim = last ? last : c->per_d;
    }
    Plan pl2;
    make_plan(&sub, seg_len, 0, &pl2);
    ws = std::max(ws, pl2.workspace);
    c->ws_off = 5 * act;
    c->slot_bytes = al256(c->ws_off + ws);
    // up front: B, C (and the backward ones), A, D, biases, convolution
    const size_t bc = al256((size_t)a->batch * L * N * es);
    const size_t par = al256(D * N * 4), vec = al256(D * 4), cw = al256(D * (size_t)std::max(1, a->conv_k) * 4);
    c->up_bytes = 4 * bc + 2 * par + 4 * vec + 2 * vec + 2 * cw;
    c->total = c->up_bytes + (size_t)kHostRing * c->slot_bytes;
    return VSSM_OK;
}

int host_scan(const vssm_scan_args *a, int seg_len, int slices, void *stream)
{
    const bool folded = seg_len > 0;
    int st = validate(a, seg_len, folded);
    if (st != VSSM_OK) return st;
    if ((long long)a->batch * a->dim * a->seqlen == 0) return VSSM_OK;
    HostCut c;
    if ((st = host_cut(a, seg_len, slices, &c)) != VSSM_OK) return st;
    if (!a->workspace || a->workspace_bytes < c.total)
        return fail(VSSM_ERR_WORKSPACE, "device workspace of %zu bytes required, %zu given", c.total,
                    a->workspace ? a->workspace_bytes : (size_t)0);
    HostPipe *hp = host_pipe(&st);
    if (!hp) return st;
    std::lock_guard<std::mutex> lock(hp->mu);
    cudaStream_t user = static_cast<cudaStream_t>(stream);
    const size_t es = a->dtype == VSSM_F32 ? 4 : 2;
    const size_t L = (size_t)a->seqlen, N = (size_t)a->dstate, D = (size_t)a->dim;
    char *w = static_cast<char *>(a->workspace);
    cudaError_t e = cudaSuccess;
    auto h2d = [&](void *dst, const void *src, size_t n) {
        if (e == cudaSuccess && src && n) e = cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, hp->copy);
    };
    // up-front copies
    const size_t bc = al256((size_t)a->batch * L * N * es);
    const size_t par = al256(D * N * 4), vec = al256(D * 4), cw = al256(D * (size_t)std::max(1, a->conv_k) * 4);
    char *up = w;
    char *dB = up, *dC = up + bc, *dBb = up + 2 * bc, *dCb = up + 3 * bc;
    char *dAf = up + 4 * bc, *dAb = dAf + par, *dDf = dAb + par, *dDb = dDf + vec;
    char *dbf = dDb + vec, *dbb = dbf + vec, *dcwf = dbb + vec, *dcwb = dcwf + cw, *dcbf = dcwb + cw,
         *dcbb = dcbf + vec;
    e = cudaEventRecord(hp->fork, user);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->copy, hp->fork, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->comp, hp->fork, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->back, hp->fork, 0);
    const size_t nbc = (size_t)a->batch * L * N * es;
    h2d(dB, a->B, nbc);
    h2d(dC, a->C, nbc);
    h2d(dBb, a->B_bwd, nbc);
    h2d(dCb, a->C_bwd, nbc);
    h2d(dAf, a->A_fwd, D * N * 4);
    h2d(dAb, a->A_bwd, D * N * 4);
    h2d(dDf, a->D_fwd, D * 4);
    h2d(dDb, a->D_bwd, D * 4);
    h2d(dbf, a->delta_bias, D * 4);
    h2d(dbb, a->delta_bias_bwd, D * 4);
    h2d(dcwf, a->conv_w, D * a->conv_k * 4);
    h2d(dcwb, a->conv_w_bwd, D * a->conv_k * 4);
    h2d(dcbf, a->conv_b, D * 4);
    h2d(dcbb, a->conv_b_bwd, D * 4);
    if (e == cudaSuccess) e = cudaEventRecord(hp->params, hp->copy);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->comp, hp->params, 0);
    if (e != cudaSuccess) return fail(VSSM_ERR_CUDA, "pipeline set-up: %s", cudaGetErrorString(e));
    const size_t act = c.ws_off / 5;
    const int nd_per_b = c.by_batch ? 1 : (a->dim + c.per_d - 1) / c.per_d;
    for (int k = 0; k < c.nslices; ++k) {
        const int sl = k % kHostRing;
        char *slot = w + c.up_bytes + (size_t)sl * c.slot_bytes;
        int b0, nb, d0, nd;
        if (c.by_batch) {
            b0 = k * c.per_b;
            nb = std::min(c.per_b, a->batch - b0);
            d0 = 0;
            nd = a->dim;
        } else {
            b0 = k / nd_per_b;
            nb = 1;
            d0 = (k % nd_per_b) * c.per_d;
            nd = std::min(c.per_d, a->dim - d0);
        }
        const size_t off = ((size_t)b0 * D + d0) * L * es;           // first element of the slice
        const size_t n = (size_t)nb * nd * L * es;                     // contiguous bytes
        char *sx = slot, *sdt = slot + act, *sz = slot + 2 * act, *sdb = slot + 3 * act, *so = slot + 4 * act;
        if (k >= kHostRing && e == cudaSuccess) e = cudaStreamWaitEvent(hp->copy, hp->out[sl], 0);
        h2d(sx, static_cast<const char *>(a->x) + off, n);
        h2d(sdt, static_cast<const char *>(a->delta) + off, n);
        if (a->z) h2d(sz, static_cast<const char *>(a->z) + off, n);
        if (a->delta_bwd) h2d(sdb, static_cast<const char *>(a->delta_bwd) + off, n);
        if (e == cudaSuccess) e = cudaEventRecord(hp->in[sl], hp->copy);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->comp, hp->in[sl], 0);
        if (e != cudaSuccess) return fail(VSSM_ERR_CUDA, "pipeline copy: %s", cudaGetErrorString(e));
        vssm_scan_args sub = *a;
        const size_t bo = (size_t)b0 * L * N * es;
        sub.x = sx;
        sub.delta = sdt;
        sub.z = a->z ? sz : nullptr;
        sub.delta_bwd = a->delta_bwd ? sdb : nullptr;
        sub.B = dB + bo;
        sub.C = dC + bo;
        sub.B_bwd = a->B_bwd ? dBb + bo : nullptr;
        sub.C_bwd = a->C_bwd ? dCb + bo : nullptr;
        sub.A_fwd = a->A_fwd ? reinterpret_cast<const float *>(dAf) + (size_t)d0 * N : nullptr;
        sub.A_bwd = a->A_bwd ? reinterpret_cast<const float *>(dAb) + (size_t)d0 * N : nullptr;
        sub.D_fwd = a->D_fwd ? reinterpret_cast<const float *>(dDf) + d0 : nullptr;
        sub.D_bwd = a->D_bwd ? reinterpret_cast<const float *>(dDb) + d0 : nullptr;
        sub.delta_bias = a->delta_bias ? reinterpret_cast<const float *>(dbf) + d0 : nullptr;
        sub.delta_bias_bwd = a->delta_bias_bwd ? reinterpret_cast<const float *>(dbb) + d0 : nullptr;
        sub.conv_w = a->conv_w ? reinterpret_cast<const float *>(dcwf) + (size_t)d0 * a->conv_k : nullptr;
        sub.conv_w_bwd = a->conv_w_bwd ? reinterpret_cast<const float *>(dcwb) + (size_t)d0 * a->conv_k : nullptr;
        sub.conv_b = a->conv_b ? reinterpret_cast<const float *>(dcbf) + d0 : nullptr;
        sub.conv_b_bwd = a->conv_b_bwd ? reinterpret_cast<const float *>(dcbb) + d0 : nullptr;
        sub.out = so;
        sub.workspace = slot + c.ws_off;
        sub.workspace_bytes = c.slot_bytes - c.ws_off;
        sub.batch = nb;
        sub.dim = nd;
        st = run(&sub, seg_len, folded, 0, hp->comp);
        if (st != VSSM_OK) return st;
        e = cudaEventRecord(hp->done[sl], hp->comp);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->back, hp->done[sl], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(static_cast<char *>(a->out) + off, so, n, cudaMemcpyDeviceToHost, hp->back);
        if (e == cudaSuccess) e = cudaEventRecord(hp->out[sl], hp->back);
        if (e != cudaSuccess) return fail(VSSM_ERR_CUDA, "pipeline step: %s", cudaGetErrorString(e));
    }
    e = cudaEventRecord(hp->join, hp->back);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(user, hp->join, 0);
    if (e != cudaSuccess) return fail(VSSM_ERR_CUDA, "pipeline join: %s", cudaGetErrorString(e));
    return VSSM_OK;
}

// ---- gradient

bool grad_composed(const vssm_scan_args *a)
{
    return a->delta_softplus || a->delta_bwd || a->conv_k > 0;
}

// Workspace of the composed gradient (step options or convolution): float32
// intermediates of each direction that runs, then the plain gradient's
// workspace for one direction (the directions run one after the other and
// reuse it). kNone marks an array that is not allocated: u then reads x, st
// the raw step (float32 I/O without convolution / softplus).
struct GradExtLayout {
    static constexpr size_t kNone = ~(size_t)0;
    size_t u[2] = {kNone, kNone}, st[2] = {kNone, kNone};
    size_t du[2] = {kNone, kNone}, dst[2] = {kNone, kNone}, dz[2] = {kNone, kNone};
    size_t B32[2] = {kNone, kNone}, C32[2] = {kNone, kNone};
    size_t z32 = kNone, dout32 = kNone, core = 0, total = 0;
    GradPlan gl;
};

GradExtLayout grad_ext_layout(const vssm_scan_args *a, int seg_len)
{
    GradExtLayout w;
    const bool bf16 = a->dtype != VSSM_F32;
    const size_t nf = (size_t)a->batch * a->dim * a->seqlen * sizeof(float);
    const size_t nbc = (size_t)a->batch * a->seqlen * a->dstate * sizeof(float);
    size_t cur = 0;
    auto take = [&cur](size_t n) {
        const size_t o = cur;
        cur = al256(cur + n);
        return o;
    };
    // both directions read the same step when neither the step nor its bias differ
    const bool st_shared = !a->delta_bwd && !(a->delta_softplus && a->delta_bias_bwd);
    for (int k = 0; k < 2; ++k) {
        if (!(a->dir_flags & (1 << k))) continue;
        const bool second = k == 1 && (a->dir_flags & 1);
        if (a->conv_k > 0) {
            w.u[k] = take(nf);
        } else if (bf16) {
            w.u[k] = second ? w.u[0] : take(nf);
        }
        if (a->delta_softplus || bf16) w.st[k] = (second && st_shared) ? w.st[0] : take(nf);
        w.du[k] = take(nf);
        w.dst[k] = take(nf);
        if (a->z) w.dz[k] = take(nf);
        if (bf16) {
            w.B32[k] = (second && !a->B_bwd) ? w.B32[0] : take(nbc);
            w.C32[k] = (second && !a->C_bwd) ? w.C32[0] : take(nbc);
        }
    }
    if (bf16) {
        if (a->z) w.z32 = take(nf);
        w.dout32 = take(nf);
    }
    vssm_scan_args one = *a;
    one.dir_flags = 1;
    w.gl = make_grad_plan(&one, seg_len);
    w.core = take(w.gl.workspace);
    w.total = cur;
    return w;
}

size_t grad_workspace(const vssm_scan_args *a, int seg_len)
{
    if ((long long)a->batch * a->dim * a->seqlen == 0) return 0;
    return grad_composed(a) ? grad_ext_layout(a, seg_len).total : make_grad_plan(a, seg_len).workspace;
}

// The plain gradient's parameters common to both paths.
void grad_fill_sizes(vssm::GradParams &p, const vssm_scan_args *a, const GradPlan &gl, int seg_len)
{
    p.batch = a->batch;
    p.dim = a->dim;
    p.L = a->seqlen;
    p.seg_len = seg_len;
    p.rgroups = gl.rgroups;
    p.nch = gl.nch;
    p.nrange = gl.nrange;
    p.rch = gl.rch;
    p.ngroups = gl.ngroups;
}

// Composed gradient: float32 step and input of each direction (prep), the
// plain gradient once per direction in float32, then the chain rule back to
// the raw tensors (post). The accumulated outputs are zeroed by the caller.
cudaError_t grad_composed_launch(const vssm_scan_args *a, const vssm_grad_args *g, int seg_len,
                                 unsigned *err, cudaStream_t s)
{
    const GradExtLayout w = grad_ext_layout(a, seg_len);
    char *ws = static_cast<char *>(a->workspace);
    auto at = [ws](size_t off) -> float * {
        return off == GradExtLayout::kNone ? nullptr : reinterpret_cast<float *>(ws + off);
    };
    const bool f32 = a->dtype == VSSM_F32;
    const unsigned dirs = a->dir_flags;
    vssm::GradExtParams q{};
    q.x = a->x;
    q.delta[0] = a->delta;
    q.delta[1] = a->delta_bwd ? a->delta_bwd : a->delta;
    q.z = a->z;
    q.dout = g->dout;
    q.bias[0] = a->delta_bias;
    q.bias[1] = a->delta_bias_bwd ? a->delta_bias_bwd : a->delta_bias;
    q.conv_w[0] = a->conv_w;
    q.conv_w[1] = a->conv_w_bwd ? a->conv_w_bwd : a->conv_w;
    q.conv_b[0] = a->conv_b;
    q.conv_b[1] = a->conv_b_bwd ? a->conv_b_bwd : a->conv_b;
    q.softplus = a->delta_softplus != 0;
    q.K = a->conv_k;
    q.batch = a->batch;
    q.dim = a->dim;
    q.L = a->seqlen;
    q.seg_len = seg_len;
    q.dirs = (int)dirs;
    for (int k = 0; k < 2; ++k) {
        if (!(dirs & (1u << k))) continue;
        q.u[k] = w.u[k] != GradExtLayout::kNone ? at(w.u[k]) : const_cast<float *>(static_cast<const float *>(a->x));
        q.st[k] = w.st[k] != GradExtLayout::kNone ? at(w.st[k])
                                                   : const_cast<float *>(static_cast<const float *>(q.delta[k]));
        q.du[k] = at(w.du[k]);
        q.dst[k] = at(w.dst[k]);
        q.dz[k] = at(w.dz[k]);
    }
    q.z32 = at(w.z32);
    q.dout32 = at(w.dout32);
    q.dx = g->dx;
    q.ddelta = g->ddelta;
    q.ddelta_bwd = g->ddelta_bwd;
    q.dzo = g->dz;
    q.dbias[0] = g->ddelta_bias;
    q.dbias[1] = a->delta_bias_bwd ? g->ddelta_bias_bwd : g->ddelta_bias;
    q.dconv_w[0] = g->dconv_w;
    q.dconv_w[1] = a->conv_w_bwd ? g->dconv_w_bwd : g->dconv_w;
    q.dconv_b[0] = g->dconv_b;
    q.dconv_b[1] = a->conv_b_bwd ? g->dconv_b_bwd : g->dconv_b;

    cudaError_t e = vssm::launch_grad_ext_prep(q, f32, s);
    const long long nbc = (long long)a->batch * a->seqlen * a->dstate;
    for (int k = 0; k < 2 && e == cudaSuccess; ++k) {
        if (!(dirs & (1u << k)) || w.B32[k] == GradExtLayout::kNone) continue;
        const bool own_b = k == 0 || !(dirs & 1) || w.B32[1] != w.B32[0];
        const bool own_c = k == 0 || !(dirs & 1) || w.C32[1] != w.C32[0];
        if (own_b) e = vssm::launch_widen_bf16(k && a->B_bwd ? a->B_bwd : a->B, at(w.B32[k]), nbc, s);
        if (own_c && e == cudaSuccess)
            e = vssm::launch_widen_bf16(k && a->C_bwd ? a->C_bwd : a->C, at(w.C32[k]), nbc, s);
    }
    for (int k = 0; k < 2 && e == cudaSuccess; ++k) {
        if (!(dirs & (1u << k))) continue;
        vssm::GradParams p{};
        p.x = q.u[k];
        p.delta = q.st[k];
        p.z = f32 ? a->z : q.z32;
        p.dout = f32 ? g->dout : q.dout32;
        const void *Bk = f32 ? (k && a->B_bwd ? a->B_bwd : a->B) : at(w.B32[k]);
        const void *Ck = f32 ? (k && a->C_bwd ? a->C_bwd : a->C) : at(w.C32[k]);
        p.B[0] = p.B[1] = Bk;
        p.C[0] = p.C[1] = Ck;
        p.A[0] = a->A_fwd;
        p.A[1] = a->A_bwd;
        p.D[0] = a->D_fwd;
        p.D[1] = a->D_bwd;
        p.dx = at(w.du[k]);
        p.ddelta = at(w.dst[k]);
        p.dz = at(w.dz[k]);
        p.dB[0] = p.dB[1] = k && g->dB_bwd ? g->dB_bwd : g->dB;
        p.dC[0] = p.dC[1] = k && g->dC_bwd ? g->dC_bwd : g->dC;
        p.dA[0] = g->dA_fwd;
        p.dA[1] = g->dA_bwd;
        p.dD[0] = g->dD_fwd;
        p.dD[1] = g->dD_bwd;
        p.ckpt = g->ckpt ? const_cast<float *>(g->ckpt) + (dirs == 3 ? (size_t)k : 0) * (size_t)w.gl.ngroups *
                                                         w.gl.nch * 512
                         : at(w.core);
        p.part = nullptr;
        p.summ = w.gl.summaries ? reinterpret_cast<float *>(ws + w.core + w.gl.summ_off) : nullptr;
        p.err = err;
        grad_fill_sizes(p, a, w.gl, seg_len);
        e = vssm::launch_grad(p, 1 << k, true, w.gl.ngroups, w.gl.nrange, g->ckpt != nullptr, s);
    }
    if (e == cudaSuccess) e = vssm::launch_grad_ext_post(q, f32, s);
    return e;
}

}  // namespace

extern "C" {

int vssm_scan_workspace_size(const vssm_scan_args *a, int seg_len, size_t *bytes)
{
    if (!a || !bytes) return fail(VSSM_ERR_INVALID_ARG, "args or bytes is NULL");
    if (a->batch < 0 || a->dim < 0 || a->seqlen < 0 || a->dir_flags < 1 || a->dir_flags > 3 ||
        seg_len < 0)
        return fail(VSSM_ERR_INVALID_ARG, "invalid sizes or dir_flags");
    Plan pl;
    make_plan(a, seg_len, 0, &pl);
    *bytes = pl.workspace;
    return VSSM_OK;
}

int vssm_scan_chunked_workspace_size(const vssm_scan_args *a, int seg_len, int pieces, size_t *bytes)
{
    if (!a || !bytes) return fail(VSSM_ERR_INVALID_ARG, "args or bytes is NULL");
    if (a->batch < 0 || a->dim < 0 || a->seqlen < 0 || a->dir_flags < 1 || a->dir_flags > 3 ||
        seg_len < 0 || pieces < 0)
        return fail(VSSM_ERR_INVALID_ARG, "invalid sizes, dir_flags or pieces");
    Plan pl;
    make_plan(a, seg_len, pieces, &pl);
    *bytes = pl.workspace;
    return VSSM_OK;
}

int vssm_scan_plan_query(const vssm_scan_args *a, int seg_len, int pieces, int *ranges_per_row,
                         int *launches)
{
    if (!a || !ranges_per_row || !launches) return fail(VSSM_ERR_INVALID_ARG, "NULL argument");
    if (a->batch < 0 || a->dim < 0 || a->seqlen < 0 || a->dir_flags < 1 || a->dir_flags > 3 ||
        seg_len < 0 || pieces < 0)
        return fail(VSSM_ERR_INVALID_ARG, "invalid sizes, dir_flags or pieces");
    if (a->dstate < 1 || a->dstate > vssm::kMaxState)
        return fail(VSSM_ERR_UNSUPPORTED, "dstate=%d outside 1..%d", a->dstate, vssm::kMaxState);
    if (pieces > 1 && a->dstate != vssm::kMaxState)
        return fail(VSSM_ERR_UNSUPPORTED, "pieces joined by the carry need dstate %d (got %d)",
                    vssm::kMaxState, a->dstate);
    if ((long long)a->batch * a->dim * a->seqlen == 0) {
        *ranges_per_row = 0;
        *launches = 0;
        return VSSM_OK;
    }
    Plan pl;
    make_plan(a, seg_len, pieces, &pl);
    *ranges_per_row = pl.pieces;
    *launches = pl.carry ? 2 : 1;
    return VSSM_OK;
}

int vssm_scan_bidir(const vssm_scan_args *a, void *stream) { return run(a, 0, false, 0, stream); }

int vssm_scan_ckpt_size(const vssm_scan_args *a, size_t *bytes)
{
    if (!a || !bytes) return fail(VSSM_ERR_INVALID_ARG, "args or bytes is NULL");
    if (a->batch < 0 || a->dim < 0 || a->seqlen < 0 || a->dir_flags < 1 || a->dir_flags > 3)
        return fail(VSSM_ERR_INVALID_ARG, "invalid sizes or dir_flags");
    *bytes = ckpt_bytes(a);
    return VSSM_OK;
}

int vssm_scan_train(const vssm_scan_args *a, int seg_len, float *ckpt, size_t ckpt_size, void *stream)
{
    if (seg_len < 0) return fail(VSSM_ERR_INVALID_ARG, "seg_len=%d must be >= 0", seg_len);
    if (!ckpt && a && (long long)a->batch * a->dim * a->seqlen > 0)
        return fail(VSSM_ERR_INVALID_ARG, "ckpt is NULL");
    return run(a, seg_len, seg_len > 0, 0, stream, ckpt, ckpt_size);
}

int vssm_scan_host_workspace_size(const vssm_scan_args *a, int seg_len, int slices, size_t *bytes)
{
    if (!a || !bytes) return fail(VSSM_ERR_INVALID_ARG, "args or bytes is NULL");
    if (a->batch < 0 || a->dim < 0 || a->seqlen < 0 || a->dir_flags < 1 || a->dir_flags > 3 ||
        seg_len < 0 || a->conv_k < 0 || a->conv_k > vssm::kMaxConv)
        return fail(VSSM_ERR_INVALID_ARG, "invalid sizes, dir_flags or conv_k");
    if ((long long)a->batch * a->dim * a->seqlen == 0) {
        *bytes = 0;
        return VSSM_OK;
    }
    HostCut c;
    const int st = host_cut(a, seg_len, slices, &c);
    if (st != VSSM_OK) return st;
    *bytes = c.total;
    return VSSM_OK;
}

int vssm_scan_host(const vssm_scan_args *a, int seg_len, int slices, void *stream)
{
    return host_scan(a, seg_len, slices, stream);
}

int vssm_ncssd_workspace_size(const vssm_ncssd_args *a, size_t *bytes)
{
    if (!a || !bytes) return fail(VSSM_ERR_INVALID_ARG, "args or bytes is NULL");
    if (a->batch < 0 || a->dim < 0 || a->seqlen < 0)
        return fail(VSSM_ERR_INVALID_ARG, "negative size");
    *bytes = 0;
    return VSSM_OK;
}

int vssm_ncssd(const vssm_ncssd_args *a, void *stream)
{
    if (!a) return fail(VSSM_ERR_INVALID_ARG, "args is NULL");
    if (a->batch < 0 || a->dim < 0 || a->seqlen < 0)
        return fail(VSSM_ERR_INVALID_ARG, "negative size (batch=%d dim=%d seqlen=%d)", a->batch,
                    a->dim, a->seqlen);
    if (a->dstate != 16) return fail(VSSM_ERR_UNSUPPORTED, "NC-SSD needs dstate 16 (got %d)", a->dstate);
    if (a->dtype != VSSM_F32 && a->dtype != VSSM_BF16)
        return fail(VSSM_ERR_UNSUPPORTED, "unknown dtype %d", a->dtype);
    if (a->batch > 65535) return fail(VSSM_ERR_UNSUPPORTED, "batch=%d above 65535", a->batch);
    const long long tok = (long long)a->batch * a->dim * a->seqlen;
    if (tok == 0) return VSSM_OK;
    if (!a->x || !a->B || !a->C || !a->m || !a->out)
        return fail(VSSM_ERR_INVALID_ARG, "x, B, C, m and out are required");
    const void *ptrs[] = {a->x, a->z, a->B, a->C, a->m, a->D, a->out};
    for (const void *q : ptrs)
        if (q && !aligned16(q)) return fail(VSSM_ERR_MISALIGNED, "pointer %p is not 16-byte aligned", q);
    const size_t es = a->dtype == VSSM_F32 ? 4 : 2;
    const size_t nact = (size_t)tok * es, nbc = (size_t)a->batch * a->seqlen * 16 * es;
    const struct { const void *p; size_t n; } ins[] = {
        {a->x, nact}, {a->z, nact}, {a->B, nbc}, {a->C, nbc},
        {a->m, (size_t)a->batch * a->seqlen * 4}, {a->D, (size_t)a->dim * 4}};
    for (const auto &in : ins)
        if (overlaps(a->out, nact, in.p, in.n)) return fail(VSSM_ERR_INVALID_ARG, "out overlaps an input");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    vssm::NcssdParams p{};
    p.x = a->x;
    p.z = a->z;
    p.B = a->B;
    p.C = a->C;
    p.m = a->m;
    p.D = a->D;
    p.out = a->out;
    p.batch = a->batch;
    p.dim = a->dim;
    p.L = a->seqlen;
    // CTAs per cluster: split the rows until about seven CTAs per SM are
    // busy, keeping at least 64 tokens per CTA
    const int dtiles = (a->dim + 31) / 32;
    if (dtiles > 65535) return fail(VSSM_ERR_UNSUPPORTED, "dim=%d above 65535 x 32", a->dim);
    const long long base = (long long)a->batch * dtiles;
    int q = 1;
    while (q < vssm::kNcMaxQ && base * q < 7LL * sm_count() && a->seqlen >= 2 * q * 64) q *= 2;
    p.rng = (a->seqlen + q - 1) / q;
    const dim3 grid((unsigned)q, (unsigned)dtiles, (unsigned)a->batch);
    const bool gate = a->z != nullptr, skip = a->D != nullptr;
    // whole rows resident in shared memory, spans moved by bulk copies
    const bool rows = a->dtype == VSSM_BF16 && q == 1 && a->dim % 8 == 0 && a->seqlen <= vssm::kNcRowsMaxL;
    if (rows) {
        p.err = device_error_word();
        if (!p.err) return fail(VSSM_ERR_CUDA, "device error word unavailable");
    }
    const cudaError_t e = vssm::launch_ncssd(p, rows, q, gate, skip, a->dtype == VSSM_F32, grid, s);
    return e == cudaSuccess ? VSSM_OK : cuda_fail(e, "launch");
}

int vssm_selftest_wait_timeout(unsigned limit_us, void *stream)
{
    if (limit_us < 1 || limit_us > 1000000)
        return fail(VSSM_ERR_INVALID_ARG, "limit_us=%u outside 1..1000000", limit_us);
    unsigned *err = device_error_word();
    if (!err) return fail(VSSM_ERR_CUDA, "cannot locate the device error word");
    const cudaError_t e = vssm::launch_selftest_wait(err, (uint64_t)limit_us * 1000ull,
                                                     static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? VSSM_OK : cuda_fail(e, "launch");
}

int vssm_scan_grad_workspace_size(const vssm_scan_args *a, int seg_len, size_t *bytes)
{
    if (!a || !bytes) return fail(VSSM_ERR_INVALID_ARG, "args or bytes is NULL");
    if (a->batch < 0 || a->dim < 0 || a->seqlen < 0 || a->dir_flags < 1 || a->dir_flags > 3 ||
        seg_len < 0 || a->conv_k < 0 || a->conv_k > vssm::kMaxConv)
        return fail(VSSM_ERR_INVALID_ARG, "invalid sizes, dir_flags or conv_k");
    *bytes = grad_workspace(a, seg_len);
    return VSSM_OK;
}

int vssm_scan_grad(const vssm_scan_args *a, const vssm_grad_args *g, int seg_len, void *stream)
{
    const bool folded = seg_len > 0;
    if (seg_len < 0) return fail(VSSM_ERR_INVALID_ARG, "seg_len=%d must be >= 0", seg_len);
    if (!g) return fail(VSSM_ERR_INVALID_ARG, "grad args is NULL");
    int st = validate(a, seg_len, folded, false);
    if (st != VSSM_OK) return st;
    if (a->dstate != vssm::kMaxState)
        return fail(VSSM_ERR_UNSUPPORTED, "the gradient needs dstate %d (got %d)", vssm::kMaxState,
                    a->dstate);
    const bool sp = a->delta_softplus != 0, conv = a->conv_k > 0;
    struct { const void *out; bool want; const char *what; } pairs[] = {
        {g->ddelta_bwd, a->delta_bwd != nullptr, "ddelta_bwd goes with delta_bwd"},
        {g->ddelta_bias, sp && a->delta_bias, "ddelta_bias goes with delta_softplus and delta_bias"},
        {g->ddelta_bias_bwd, sp && a->delta_bias_bwd, "ddelta_bias_bwd goes with delta_softplus and delta_bias_bwd"},
        {g->dconv_w, conv, "dconv_w goes with conv_k > 0"},
        {g->dconv_b, conv && a->conv_b, "dconv_b goes with conv_k > 0 and conv_b"},
        {g->dconv_w_bwd, conv && a->conv_w_bwd, "dconv_w_bwd goes with conv_k > 0 and conv_w_bwd"},
        {g->dconv_b_bwd, conv && a->conv_b_bwd, "dconv_b_bwd goes with conv_k > 0 and conv_b_bwd"}};
    for (const auto &pr : pairs)
        if ((pr.out != nullptr) != pr.want) return fail(VSSM_ERR_INVALID_ARG, "%s", pr.what);
    if ((long long)a->batch * a->dim * a->seqlen == 0) return VSSM_OK;
    const unsigned dirs = a->dir_flags;
    if (!g->dout || !g->dx || !g->ddelta || !g->dB || !g->dC)
        return fail(VSSM_ERR_INVALID_ARG, "dout, dx, ddelta, dB and dC are required");
    if (a->z && !g->dz) return fail(VSSM_ERR_INVALID_ARG, "dz is required when z is given");
    if ((a->B_bwd != nullptr) != (g->dB_bwd != nullptr) || (a->C_bwd != nullptr) != (g->dC_bwd != nullptr))
        return fail(VSSM_ERR_INVALID_ARG, "dB_bwd / dC_bwd go with B_bwd / C_bwd");
    if ((dirs & 1) && (!g->dA_fwd || !g->dD_fwd))
        return fail(VSSM_ERR_INVALID_ARG, "dA_fwd and dD_fwd are required for the forward direction");
    if ((dirs & 2) && (!g->dA_bwd || !g->dD_bwd))
        return fail(VSSM_ERR_INVALID_ARG, "dA_bwd and dD_bwd are required for the backward direction");
    const void *gp[] = {g->dout, g->dx, g->ddelta, g->dz, g->dB, g->dC, g->dB_bwd, g->dC_bwd,
                        g->dA_fwd, g->dA_bwd, g->dD_fwd, g->dD_bwd, g->ddelta_bwd, g->ddelta_bias,
                        g->ddelta_bias_bwd, g->dconv_w, g->dconv_b, g->dconv_w_bwd, g->dconv_b_bwd};
    for (const void *q : gp)
        if (q && !aligned16(q)) return fail(VSSM_ERR_MISALIGNED, "gradient pointer %p is not 16-byte aligned", q);
    if (g->ckpt) {
        if (!aligned16(g->ckpt)) return fail(VSSM_ERR_MISALIGNED, "ckpt is not 16-byte aligned");
        if (g->ckpt_bytes < ckpt_bytes(a))
            return fail(VSSM_ERR_INVALID_ARG, "ckpt of %zu bytes required, %zu given", ckpt_bytes(a), g->ckpt_bytes);
    }
    const bool composed = grad_composed(a);
    const GradPlan gl = composed ? grad_ext_layout(a, seg_len).gl : make_grad_plan(a, seg_len);
    const size_t need = grad_workspace(a, seg_len);
    if (!a->workspace || a->workspace_bytes < need)
        return fail(VSSM_ERR_WORKSPACE, "workspace of %zu bytes required, %zu given", need,
                    a->workspace ? a->workspace_bytes : (size_t)0);
    if (gl.ngroups * gl.nrange > 0x7fffffffLL) return fail(VSSM_ERR_UNSUPPORTED, "problem too large for one grid");
    const size_t es = a->dtype == VSSM_F32 ? 4 : 2;
    const size_t nact = (size_t)a->batch * a->dim * a->seqlen * es;
    const size_t nbc = (size_t)a->batch * a->seqlen * a->dstate * 4;
    const size_t npar = (size_t)a->dim * a->dstate * 4, nd = (size_t)a->dim * 4;
    const size_t ncw = (size_t)a->dim * std::max(a->conv_k, 0) * 4;
    const struct { const void *p; size_t n; } outs[] = {
        {g->dx, nact}, {g->ddelta, nact}, {g->dz, nact}, {g->dB, nbc}, {g->dC, nbc},
        {g->dB_bwd, nbc}, {g->dC_bwd, nbc}, {g->dA_fwd, npar}, {g->dA_bwd, npar},
        {g->dD_fwd, nd}, {g->dD_bwd, nd}, {g->ddelta_bwd, nact}, {g->ddelta_bias, nd},
        {g->ddelta_bias_bwd, nd}, {g->dconv_w, ncw}, {g->dconv_b, nd}, {g->dconv_w_bwd, ncw},
        {g->dconv_b_bwd, nd}};
    const void *ins[] = {a->x, a->delta, a->z, a->B, a->C, a->B_bwd, a->C_bwd, a->A_fwd, a->A_bwd,
                         a->D_fwd, a->D_bwd, g->dout, a->delta_bwd, a->delta_bias, a->delta_bias_bwd,
                         a->conv_w, a->conv_b, a->conv_w_bwd, a->conv_b_bwd, g->ckpt};
    const size_t insz[] = {nact, nact, nact, nbc / 4 * es, nbc / 4 * es, nbc / 4 * es, nbc / 4 * es,
                           npar, npar, nd, nd, nact, nact, nd, nd, ncw, nd, ncw, nd,
                           g->ckpt ? ckpt_bytes(a) : 0};
    for (size_t i = 0; i < sizeof(outs) / sizeof(outs[0]); ++i) {
        if (!outs[i].p) continue;
        if (overlaps(outs[i].p, outs[i].n, a->workspace, a->workspace_bytes))
            return fail(VSSM_ERR_INVALID_ARG, "a gradient output overlaps the workspace");
        for (size_t k = 0; k < sizeof(ins) / sizeof(ins[0]); ++k)
            if (overlaps(outs[i].p, outs[i].n, ins[k], insz[k]))
                return fail(VSSM_ERR_INVALID_ARG, "a gradient output overlaps an input");
        for (size_t k = i + 1; k < sizeof(outs) / sizeof(outs[0]); ++k)
            if (overlaps(outs[i].p, outs[i].n, outs[k].p, outs[k].n))
                return fail(VSSM_ERR_INVALID_ARG, "two gradient outputs overlap");
    }
    for (size_t k = 0; k < sizeof(ins) / sizeof(ins[0]); ++k)
        if (overlaps(a->workspace, a->workspace_bytes, ins[k], insz[k]))
            return fail(VSSM_ERR_INVALID_ARG, "the workspace overlaps an input");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned *err = device_error_word();
    if (!err) return fail(VSSM_ERR_CUDA, "cannot locate the device error word");
    // the reductions accumulate atomically: start them at zero
    const size_t nbcf = (size_t)a->batch * a->seqlen * a->dstate;
    const struct { float *p; size_t n; } zs[] = {
        {g->dB, nbcf}, {g->dC, nbcf}, {g->dB_bwd, nbcf}, {g->dC_bwd, nbcf},
        {(dirs & 1) ? g->dA_fwd : nullptr, npar / 4}, {(dirs & 1) ? g->dD_fwd : nullptr, nd / 4},
        {(dirs & 2) ? g->dA_bwd : nullptr, npar / 4}, {(dirs & 2) ? g->dD_bwd : nullptr, nd / 4},
        {g->ddelta_bias, nd / 4}, {g->ddelta_bias_bwd, nd / 4}, {g->dconv_w, ncw / 4},
        {g->dconv_b, nd / 4}, {g->dconv_w_bwd, ncw / 4}, {g->dconv_b_bwd, nd / 4}};
    cudaError_t e = cudaSuccess;
    for (const auto &z : zs)
        if (e == cudaSuccess) e = vssm::launch_zero_f32(z.p, z.n, s);
    if (e == cudaSuccess && composed) e = grad_composed_launch(a, g, seg_len, err, s);
    if (e == cudaSuccess && !composed) {
        vssm::GradParams p{};
        p.x = a->x;
        p.delta = a->delta;
        p.z = a->z;
        p.dout = g->dout;
        p.B[0] = a->B;
        p.C[0] = a->C;
        p.B[1] = a->B_bwd ? a->B_bwd : a->B;
        p.C[1] = a->C_bwd ? a->C_bwd : a->C;
        p.A[0] = a->A_fwd;
        p.A[1] = a->A_bwd;
        p.D[0] = a->D_fwd;
        p.D[1] = a->D_bwd;
        p.dx = g->dx;
        p.ddelta = g->ddelta;
        p.dz = g->dz;
        p.dB[0] = g->dB;
        p.dC[0] = g->dC;
        p.dB[1] = g->dB_bwd ? g->dB_bwd : g->dB;
        p.dC[1] = g->dC_bwd ? g->dC_bwd : g->dC;
        p.dA[0] = g->dA_fwd;
        p.dA[1] = g->dA_bwd;
        p.dD[0] = g->dD_fwd;
        p.dD[1] = g->dD_bwd;
        p.ckpt = g->ckpt ? const_cast<float *>(g->ckpt) : static_cast<float *>(a->workspace);
        p.part = dirs == 3 ? reinterpret_cast<float *>(static_cast<char *>(a->workspace) + gl.part_off)
                           : nullptr;
        p.summ = gl.summaries ? reinterpret_cast<float *>(static_cast<char *>(a->workspace) + gl.summ_off)
                               : nullptr;
        p.err = err;
        grad_fill_sizes(p, a, gl, seg_len);
        e = vssm::launch_grad(p, (int)dirs, a->dtype == VSSM_F32, gl.ngroups, gl.nrange, g->ckpt != nullptr, s);
    }
    return e == cudaSuccess ? VSSM_OK : cuda_fail(e, "launch");
}

int vssm_scan_grad_plan_query(const vssm_scan_args *a, const vssm_grad_args *g, int seg_len,
                              int *ranges_per_row, int *launches)
{
    if (!a || !g || !ranges_per_row || !launches) return fail(VSSM_ERR_INVALID_ARG, "NULL argument");
    if (a->batch < 0 || a->dim < 0 || a->seqlen < 0 || a->dir_flags < 1 || a->dir_flags > 3 ||
        seg_len < 0 || a->conv_k < 0 || a->conv_k > vssm::kMaxConv)
        return fail(VSSM_ERR_INVALID_ARG, "invalid sizes, dir_flags or conv_k");
    if (a->dstate != vssm::kMaxState)
        return fail(VSSM_ERR_UNSUPPORTED, "the gradient needs dstate %d (got %d)", vssm::kMaxState, a->dstate);
    *ranges_per_row = 0;
    *launches = 0;
    if ((long long)a->batch * a->dim * a->seqlen == 0) return VSSM_OK;
    const unsigned dirs = a->dir_flags;
    // zero-fills of the accumulated outputs (as vssm_scan_grad)
    const void *zs[] = {g->dB, g->dC, g->dB_bwd, g->dC_bwd, (dirs & 1) ? g->dA_fwd : nullptr,
                        (dirs & 1) ? g->dD_fwd : nullptr, (dirs & 2) ? g->dA_bwd : nullptr,
                        (dirs & 2) ? g->dD_bwd : nullptr, g->ddelta_bias, g->ddelta_bias_bwd,
                        g->dconv_w, g->dconv_b, g->dconv_w_bwd, g->dconv_b_bwd};
    int n = 0;
    for (const void *z : zs) n += z != nullptr;
    const int per_dir_extra = g->ckpt ? 0 : 1;   // the checkpoint pass
    if (grad_composed(a)) {
        const GradExtLayout w = grad_ext_layout(a, seg_len);
        n += 2;                                  // prep, post
        for (int k = 0; k < 2; ++k) {
            if (!(dirs & (1u << k))) continue;
            if (w.B32[k] != GradExtLayout::kNone) {
                n += (k == 0 || !(dirs & 1) || w.B32[1] != w.B32[0]) ? 1 : 0;
                n += (k == 0 || !(dirs & 1) || w.C32[1] != w.C32[0]) ? 1 : 0;
            }
            n += per_dir_extra + (w.gl.summaries ? 1 : 0) + 1;
        }
        *ranges_per_row = w.gl.nrange;
    } else {
        const GradPlan gl = make_grad_plan(a, seg_len);
        n += per_dir_extra + (gl.summaries ? 1 : 0) + 1;
        *ranges_per_row = gl.nrange;
    }
    *launches = n;
    return VSSM_OK;
}

int vssm_scan_chunked(const vssm_scan_args *a, int seg_len, int pieces, void *stream)
{
    return run(a, seg_len, seg_len > 0, pieces, stream);
}

int vssm_scan_bidir_noalloc(const vssm_scan_args *a, void *stream)
{
    if (!a) return fail(VSSM_ERR_INVALID_ARG, "args is NULL");
    vssm_scan_args b = *a;                 // the caller's workspace fields are ignored
    b.workspace = nullptr;
    b.workspace_bytes = 0;
    size_t need = 0;
    int pieces = 0;
    int st = vssm_scan_workspace_size(&b, 0, &need);
    if (st != VSSM_OK) return st;
    if (need > VSSM_NOALLOC_SCRATCH_BYTES) {   // rows not cut for the carry need less
        pieces = 1;
        st = vssm_scan_chunked_workspace_size(&b, 0, pieces, &need);
        if (st != VSSM_OK) return st;
    }
    if (need > VSSM_NOALLOC_SCRATCH_BYTES)
        return fail(VSSM_ERR_UNSUPPORTED,
                    "vssm_scan_bidir_noalloc: this call needs %zu bytes of scratch but the built-in "
                    "scratch holds %zu (VSSM_NOALLOC_SCRATCH_BYTES); use vssm_scan_bidir with a workspace",
                    need, (size_t)VSSM_NOALLOC_SCRATCH_BYTES);
    if (need > 0) {
        b.workspace = noalloc_scratch();
        if (!b.workspace) return VSSM_ERR_CUDA;
        b.workspace_bytes = VSSM_NOALLOC_SCRATCH_BYTES;
    }
    return run(&b, 0, false, pieces, stream);
}

int vssm_scan_folded(const vssm_scan_args *a, int seg_len, void *stream)
{
    return run(a, seg_len, true, 0, stream);
}

int vssm_device_error(void *stream)
{
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(VSSM_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
    unsigned word = 0, zero = 0;
    e = cudaMemcpyFromSymbol(&word, g_vssm_device_error, sizeof word);
    if (e == cudaSuccess && word) e = cudaMemcpyToSymbol(g_vssm_device_error, &zero, sizeof zero);
    if (e != cudaSuccess) return fail(VSSM_ERR_CUDA, "error word: %s", cudaGetErrorString(e));
    if (word & vssm::kErrTimeout)
        return fail(VSSM_ERR_TIMEOUT, "a device-side wait exceeded its limit; results are invalid");
    return VSSM_OK;
}

const char *vssm_status_string(int status)
{
    switch (status) {
    case VSSM_OK: return "ok";
    case VSSM_ERR_INVALID_ARG: return "invalid argument";
    case VSSM_ERR_UNSUPPORTED: return "unsupported configuration";
    case VSSM_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case VSSM_ERR_CUDA: return "CUDA runtime error";
    case VSSM_ERR_TIMEOUT: return "device-side wait timed out";
    case VSSM_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
    }
}

const char *vssm_last_error(void) { return g_last_error.c_str(); }

int vssm_version(void) { return VSSM_VERSION; }

}  // extern "C"
