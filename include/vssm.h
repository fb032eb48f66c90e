/*
 * vssm.h -- C ABI of the bidirectional selective-scan (S6) library for
 * NVIDIA B300 (sm_103a).
 *
 * The operation (for every batch b and channel d, states n = 0..N-1):
 *
 *   decay      Abar_t[n] = exp(delta_t * A[d][n])         VSSD page, §4.1.2
 *   recurrence h_t[n] = Abar_t[n] * h_{t-1}[n] + delta_t * B_t[n] * x_t
 *              y_t    = sum_n C_t[n] * h_t[n] + D[d] * x_t  VSSD page, §4.2.1.3
 *   backward   the same recurrence over t = L-1 .. 0 with its own A and D
 *                                                           Vim page, §2.2
 *   output     out_t = (y_fwd_t + y_bwd_t) * silu(z_t),  silu(z) = z * sigmoid(z)
 *   folded     with seg_len > 0 the decay is 0 at every segment start
 *              (t mod seg_len == 0 forward, == seg_len-1 backward), so
 *              segments concatenated along t never exchange state
 *                                  SF-Mamba page, "批量折叠与周期性状态重置"
 *
 * The first-order input term delta*B (the pages' "≈ΔB") is used; the state
 * starts at zero in each direction and is never returned.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller. The library
 *    allocates nothing and keeps no pointer after the call returns.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL = the legacy default stream). A return of VSSM_OK means the kernel
 *    was enqueued; execution errors surface at the caller's next
 *    synchronisation, as for any CUDA launch.
 *  - Arguments are validated on the host BEFORE anything is launched; an
 *    invalid call launches nothing and returns a negative vssm_status. The
 *    text of the last error on the calling thread is vssm_last_error().
 *  - Layouts (row-major, last index fastest):
 *      x, delta, z, out : [batch][dim][seqlen]
 *      B, C, B_bwd, C_bwd: [batch][seqlen][dstate]
 *      A_fwd, A_bwd     : [dim][dstate]   float32
 *      D_fwd, D_bwd     : [dim]           float32
 *    x, delta, z, B, C, B_bwd, C_bwd and out all have the element type
 *    `dtype`; arithmetic and the state are float32 in both cases, and out is
 *    rounded once (round to nearest even) when stored.
 *  - Every pointer must be 16-byte aligned (torch allocations are).
 *  - `out` must not overlap any input or the workspace.
 */
#ifndef VSSM_H
#define VSSM_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define VSSM_VERSION 180 /* 1.8.0 */

typedef enum {
    VSSM_OK = 0,
    VSSM_ERR_INVALID_ARG = -1,   /* null/negative/inconsistent argument        */
    VSSM_ERR_UNSUPPORTED = -2,   /* e.g. dstate > 16, unknown dtype            */
    VSSM_ERR_MISALIGNED = -3,    /* a pointer is not 16-byte aligned           */
    VSSM_ERR_CUDA = -4,          /* the CUDA runtime refused the launch        */
    VSSM_ERR_TIMEOUT = -5,       /* a bounded device-side wait expired         */
    VSSM_ERR_WORKSPACE = -6      /* workspace missing or smaller than required */
} vssm_status;

typedef enum { VSSM_F32 = 0, VSSM_BF16 = 1 } vssm_dtype;

enum { VSSM_DIR_FWD = 1, VSSM_DIR_BWD = 2, VSSM_DIR_BOTH = 3 };

typedef struct {
    const void *x;          /* [batch][dim][seqlen]                      required */
    const void *delta;      /* [batch][dim][seqlen], the step Δ (already
                               positive, e.g. after softplus)            required */
    const void *z;          /* [batch][dim][seqlen] gate input; NULL = no gate    */
    const void *B;          /* [batch][seqlen][dstate]                   required */
    const void *C;          /* [batch][seqlen][dstate]                   required */
    const void *B_bwd;      /* backward B; NULL = use B                           */
    const void *C_bwd;      /* backward C; NULL = use C                           */
    const float *A_fwd;     /* [dim][dstate]; required if the FWD bit is set      */
    const float *A_bwd;     /* [dim][dstate]; required if the BWD bit is set      */
    const float *D_fwd;     /* [dim] skip weight; NULL = 0                        */
    const float *D_bwd;     /* [dim] skip weight; NULL = 0                        */
    void *out;              /* [batch][dim][seqlen] output               required */
    void *workspace;        /* device scratch, see vssm_scan_workspace_size()     */
    size_t workspace_bytes; /* size of `workspace` in bytes                       */
    int batch, dim, seqlen; /* >= 0; an empty problem is a no-op                  */
    int dstate;             /* 1..16                                              */
    int dtype;              /* vssm_dtype                                         */
    unsigned dir_flags;     /* VSSM_DIR_FWD | VSSM_DIR_BWD (at least one)         */
    /* Step options (zero-initialise the struct to leave them off). Each
     * direction is its own SSM module (Vim page §2.2, forward_ssm /
     * backward_ssm), so the backward direction may take its own step; and the
     * step may be passed before its positivity map, as the output of a step
     * projection with bias (Mamba2D page, "Mamba2D Block结构", dt_proj with
     * bias=True). With delta_softplus = 1 the step of each direction is
     * softplus(its delta + its bias[d]), softplus(v) = log(1 + exp(v)),
     * evaluated in fp32 (absolute error about 1e-7). */
    const void *delta_bwd;        /* backward step [batch][dim][seqlen]; NULL = delta */
    const float *delta_bias;      /* [dim] forward step bias; NULL = 0 (softplus only) */
    const float *delta_bias_bwd;  /* [dim] backward step bias; NULL = delta_bias      */
    int delta_softplus;           /* 0: steps used as given; 1: softplus(step + bias)  */
    /* Directional depthwise convolution + SiLU in front of the scan (off when
     * conv_k = 0). The forward and backward paths use 1D convolutions of
     * opposite directions (Vim page §2.3), and the SSM reads SiLU of the
     * convolution (SF-Mamba page, "MambaVision Mixer", X1 = SSM(σ(Conv(...)))).
     * Per channel d, K = conv_k taps w[d][0..K-1] and bias b[d]:
     *   forward:  u[t] = silu(b + sum_k w[k] * x[t - (K-1) + k])   (causal)
     *   backward: u[t] = silu(b + sum_k w[k] * x[t + (K-1) - k])   (reversed)
     * Taps outside the row read 0; on a folded row (vssm_scan_folded) also
     * outside the current segment (SF-Mamba page, "1D深度可分离卷积适配": the
     * convolution never crosses sequences). Each direction then reads its own
     * u in place of x, for the input term and its skip D*u alike. */
    const float *conv_w;          /* [dim][conv_k] forward taps; required if conv_k > 0 */
    const float *conv_b;          /* [dim] forward bias; NULL = 0                     */
    const float *conv_w_bwd;      /* [dim][conv_k] backward taps; NULL = conv_w       */
    const float *conv_b_bwd;      /* [dim] backward bias; NULL = conv_b               */
    int conv_k;                   /* 0 = no convolution; 1..4 taps                    */
} vssm_scan_args;

/*
 * Bytes of device workspace the call with these arguments needs (0 when it
 * needs none). With both directions, the direction that reaches a token first
 * leaves its partial output (fp32, one per token and channel) there until the
 * other direction arrives; a single direction needs no workspace, and with
 * dstate != 16 short rows keep that buffer in shared memory. The workspace
 * holds nothing between calls, and two calls in flight at the same time must
 * not share one. seg_len as in vssm_scan_folded
 * (0 for vssm_scan_bidir). Only `batch`, `dim`, `seqlen`, `dstate`, `dtype`
 * and `dir_flags` of `a` are read.
 */
int vssm_scan_workspace_size(const vssm_scan_args *a, int seg_len, size_t *bytes);

/*
 * Bidirectional (or single-direction, by dir_flags) selective scan over
 * independent sequences of seqlen tokens. Vim page §2.2 and §3.1; VSSD page
 * §4.1.2 and §4.2.1.3. When the rows are too few to occupy the GPU (small
 * batch x dim), each row is cut into token ranges joined by the carry, as in
 * vssm_scan_chunked; the result is the same up to fp32 rounding order.
 */
int vssm_scan_bidir(const vssm_scan_args *a, void *stream);

/*
 * The scan of vssm_scan_bidir (seg_len == 0) or vssm_scan_folded
 * (seg_len >= 1) with each row cut into a chosen number of contiguous token
 * ranges that are scanned in parallel and joined exactly (Vim page §3.1,
 * parallel scan; SF-Mamba page, the warp-scan remark):
 *
 *   1. every range except the last one in a direction is scanned from a zero
 *      state, giving its end state hp[n] and its decay
 *      P[n] = exp(A[d][n] * sum of delta over the range), or P = 0 when a
 *      folded reset lies inside it;
 *   2. the range maps an incoming state h to P*h + hp; these maps compose
 *      associatively, (P1, h1) then (P2, h2) = (P1*P2, P2*h1 + h2), and the
 *      exclusive prefix of the ranges before a range, applied to h = 0, is
 *      that range's incoming state;
 *   3. every range is scanned from its incoming state and writes its output.
 *
 * In exact arithmetic the result equals the unsplit scan; in fp32 it differs
 * only in rounding order. Step 1 repeats the recurrence's exponentials on the
 * ranges it summarises, so splitting pays only when the rows alone leave the
 * GPU idle; vssm_scan_bidir chooses the count itself.
 *
 * pieces: 0 = the library's choice (what vssm_scan_bidir / vssm_scan_folded
 * do; a folded call is split at segment starts into as many independent
 * ranges of whole segments as fill two waves of the warps resident at once);
 * 1 = rows are not cut for the carry (a folded call may still be split at
 * segment starts, which needs no carry); P > 1 = rows are cut into
 * ceil(seqlen / ceil(seqlen / P)) ranges of ceil(seqlen / P) tokens (the last
 * one shorter). P > 1 needs dstate == 16, else VSSM_ERR_UNSUPPORTED. The
 * workspace must hold vssm_scan_chunked_workspace_size bytes: the partial
 * outputs of bidirectional calls plus 2176 bytes per 32-channel group, range
 * and direction for the range summaries. Other arguments and errors as in
 * vssm_scan_bidir and vssm_scan_folded; seg_len < 0 or pieces < 0 give
 * VSSM_ERR_INVALID_ARG.
 */
int vssm_scan_chunked(const vssm_scan_args *a, int seg_len, int pieces, void *stream);

/* Workspace bytes for vssm_scan_chunked with these seg_len and pieces. */
int vssm_scan_chunked_workspace_size(const vssm_scan_args *a, int seg_len, int pieces, size_t *bytes);

/*
 * How the call vssm_scan_chunked(a, seg_len, pieces, ...) would run (pieces
 * = 0: also vssm_scan_bidir for seg_len == 0 and vssm_scan_folded for
 * seg_len >= 1): *ranges_per_row receives the number of token ranges each
 * row is scanned in (independent ranges at folded segment starts, or ranges
 * joined by the carry), *launches the number of kernel launches (2 when a
 * summary pass runs first, else 1; 0 for an empty problem). Reads only the
 * sizes, dstate, dtype and dir_flags of `a`; touches no device. Errors:
 * VSSM_ERR_INVALID_ARG for NULL pointers or invalid sizes, dir_flags,
 * seg_len or pieces; VSSM_ERR_UNSUPPORTED as in vssm_scan_chunked.
 */
int vssm_scan_plan_query(const vssm_scan_args *a, int seg_len, int pieces, int *ranges_per_row,
                         int *launches);

/*
 * Bytes of the built-in scratch that vssm_scan_bidir_noalloc uses (16 MiB).
 * A call needs as much scratch as vssm_scan_workspace_size reports for it;
 * when that is more than the built-in scratch, the call runs without cutting
 * rows for the carry, which for bidirectional calls with dstate 16 needs 4
 * bytes per token and channel (rounded up to whole 32-channel groups), so up
 * to about 4.19 million token-channels fit.
 */
#define VSSM_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/*
 * vssm_scan_bidir for callers that cannot allocate device memory. (The pages
 * have no counterpart to this: it only changes where the scratch lives.)
 *
 * vssm_scan_bidir needs a device workspace from its caller for bidirectional
 * calls. Some callers cannot provide one: a plain C or embedded host program
 * with no device allocator of its own, or a serving loop that must not call
 * cudaMalloc once it is running (an allocation can synchronise the device or
 * fail under memory pressure). This entry point computes exactly what
 * vssm_scan_bidir computes, with the same arguments and layouts, but takes
 * its scratch from an array of VSSM_NOALLOC_SCRATCH_BYTES that the library
 * holds in device memory on every device that loads it, until the process
 * exits. It allocates nothing, and a->workspace and a->workspace_bytes are
 * ignored. The caller still owns all inputs and the output.
 *
 *  - A call that would need more than VSSM_NOALLOC_SCRATCH_BYTES of scratch
 *    is rejected with VSSM_ERR_UNSUPPORTED before anything is launched (see
 *    vssm_last_error()); pass a workspace to vssm_scan_bidir instead.
 *  - The first call on a device looks up the scratch's device address
 *    (cudaGetSymbolAddress, with that device current). Make that first call
 *    before any stream capture on that device.
 *  - All calls share the one array, and it keeps the last call's contents.
 *    Nothing in it has to start at zero: a call writes every scratch value
 *    before it reads it. Calls that overlap on the GPU (on different streams,
 *    or issued from different host threads without ordering) race on the
 *    scratch and give wrong results; order them on one stream.
 */
int vssm_scan_bidir_noalloc(const vssm_scan_args *a, void *stream);

/*
 * Batch-folded scan: each row of seqlen tokens is a concatenation of
 * segments of seg_len tokens with the state reset at every segment start
 * (SF-Mamba page, "批量折叠与周期性状态重置"; folded tensor Z' of shape
 * B1 x D x (B2*T)). The caller folds (B2 sequences of T tokens become one row
 * of B2*T tokens) and unfolds; the kernel receives the folded tensors.
 * seg_len >= 1. Forward-only calls accept a partial last segment; when the
 * BWD bit is set, seqlen must be a multiple of seg_len (else
 * VSSM_ERR_INVALID_ARG).
 */
int vssm_scan_folded(const vssm_scan_args *a, int seg_len, void *stream);

/*
 * Gradient of the scan (training). Arguments of the forward call plus the
 * gradient of a loss with respect to its output; all device pointers,
 * caller-owned.
 */
typedef struct {
    const void *dout;        /* [batch][dim][seqlen] dL/d out, dtype of x      required */
    void *dx, *ddelta, *dz;  /* [batch][dim][seqlen], dtype of x, written; dz
                                required iff the forward call has z           */
    float *dB, *dC;          /* [batch][seqlen][dstate] fp32, written         required */
    float *dB_bwd, *dC_bwd;  /* required iff B_bwd / C_bwd are given (the
                                backward direction's own); else NULL          */
    float *dA_fwd, *dA_bwd;  /* [dim][dstate] fp32, written; required for each
                                direction the call runs                       */
    float *dD_fwd, *dD_bwd;  /* [dim] fp32, written; as dA                     */
    /* Gradients of the step options and of the convolution (zero-initialise
     * the struct to leave them unset; each is required exactly when the
     * forward call has the corresponding input): */
    void *ddelta_bwd;        /* [batch][dim][seqlen], dtype of x: d/d delta_bwd;
                                iff delta_bwd is given (ddelta is then the
                                forward direction's step only)                */
    float *ddelta_bias;      /* [dim] fp32; iff delta_softplus and delta_bias
                                (with a shared bias it holds both directions') */
    float *ddelta_bias_bwd;  /* [dim] fp32; iff delta_softplus and delta_bias_bwd */
    float *dconv_w, *dconv_b;          /* [dim][conv_k], [dim] fp32; dconv_w iff
                                          conv_k > 0, dconv_b iff conv_b      */
    float *dconv_w_bwd, *dconv_b_bwd;  /* iff conv_w_bwd / conv_b_bwd (else the
                                          backward taps' gradients are added
                                          to dconv_w / dconv_b)               */
    /* State checkpoints stored by vssm_scan_train for this same forward call
     * (NULL = recompute them: one more pass over the inputs). Read only. */
    const float *ckpt;
    size_t ckpt_bytes;       /* bytes available at ckpt (>= vssm_scan_ckpt_size) */
} vssm_grad_args;

/*
 * Reverse-mode gradient of L = sum(dout * out) for the forward call
 * vssm_scan_bidir(a) (seg_len == 0) or vssm_scan_folded(a, seg_len): the
 * exact derivative with respect to x, delta, z, B, C (and B_bwd, C_bwd), A
 * and D of each direction (the adjoint recurrence of the scan: each
 * direction's adjoint walks against its own scan order; VSSD page §4.2.1.3
 * for the recurrence, Vim page §2.2 for the two directions). a->out is not
 * read. dx, ddelta, dz are rounded once to the I/O dtype; dB, dC, dA, dD are
 * fp32 sums over batch, channels and tokens, computed with atomic additions
 * (their summation order, and so their last bits, can vary from run to run).
 *
 * With the step options and the convolution (delta_softplus, delta_bwd,
 * conv_k > 0) the derivatives reach the raw tensors through the chain rule:
 * the step of direction k is s_k = softplus(v_k + bias_k) (or v_k), so
 * d v_k = d s_k * sigmoid(v_k + bias_k) and d bias_k = sum over batch and
 * tokens of d v_k; its input is u_k = silu(pre_k), pre_k the direction's
 * depthwise convolution of x (causal forward, reversed backward, segment
 * bounded when folded), so x, the taps and the bias get the transposed
 * convolution of d pre_k = d u_k * silu'(pre_k). The call then runs the
 * scan's gradient once per direction on float32 copies of that direction's
 * step and input (the values the forward computes), and needs the larger
 * workspace that vssm_scan_grad_workspace_size reports for it.
 *
 * Supported: dstate == 16; anything else is VSSM_ERR_UNSUPPORTED.
 * a->workspace must hold vssm_scan_grad_workspace_size bytes and must not
 * overlap any input or output. Asynchronous on `stream`; the
 * pair rendezvous of the two directions is bounded as in the forward kernel
 * (vssm_device_error). When that wait expires (vssm_device_error then
 * returns VSSM_ERR_TIMEOUT), every gradient output of the call is undefined:
 * the warps that gave up stop before their second half, so part of dB/dC was
 * accumulated and part of dx/ddelta/dz, dA, dD was never written.
 */
int vssm_scan_grad(const vssm_scan_args *a, const vssm_grad_args *g, int seg_len, void *stream);

/* Workspace bytes of vssm_scan_grad: 16 bytes per token, channel and
 * direction for the state checkpoints (16 fp32 every 4 tokens), plus 12 bytes
 * per token and channel for the partial gradients exchanged between the two
 * directions (both directions only), channels rounded up to groups of 32.
 * When there are too few 32-channel groups to fill the GPU, the rows are cut
 * into token ranges for the adjoint, and 128 bytes per range, channel and
 * direction hold the ranges' adjoint summaries; folded rows (seg_len > 0) are
 * cut at segment starts instead, into ranges the reset makes independent,
 * which need no summaries.
 * With the step options or the convolution the directions run one after the
 * other and share one direction's workspace of the above, after float32
 * intermediates of 4 bytes per token and channel each, per direction run:
 * the gradients of its step and input and, with z, its share of dz; with the
 * convolution its input; with softplus or
 * bfloat16 I/O its step (one for both directions when they share step and
 * bias); with bfloat16 I/O and no convolution one input copy; with bfloat16
 * I/O float32 copies of z, dout and (per distinct tensor) B and C. Arrays
 * start on 256-byte boundaries. */
int vssm_scan_grad_workspace_size(const vssm_scan_args *a, int seg_len, size_t *bytes);

/*
 * Training forward: the scan of vssm_scan_bidir (seg_len == 0) or
 * vssm_scan_folded (seg_len >= 1), with the same output, that also stores
 * the states vssm_scan_grad needs as checkpoints: per direction run, channel
 * and 4-token chunk of the row, the state h (16 fp32) entering the chunk in
 * that direction's scan order (VSSD page §4.2.1.3: the recurrence the
 * gradient walks back through), zero when the chunk's first token in that
 * order starts a folded segment (the recurrence restarts there). Layout [direction slot][batch][channel group
 * of 32][chunk][16][32] fp32 (slot 0 = forward, 1 = backward when both run;
 * slot 0 alone for one direction). Passing the buffer to vssm_scan_grad
 * (vssm_grad_args.ckpt) saves the gradient its checkpoint pass, a full
 * recurrence over the inputs, for 64 bytes per 4 tokens, channel and
 * direction written here. ckpt is caller-owned device memory of at least
 * vssm_scan_ckpt_size bytes, 16-byte aligned, overlapping no other tensor
 * of the call. dstate must be 16 (else VSSM_ERR_UNSUPPORTED); other errors
 * as the plain calls, VSSM_ERR_INVALID_ARG for a NULL or short ckpt.
 */
int vssm_scan_train(const vssm_scan_args *a, int seg_len, float *ckpt, size_t ckpt_bytes, void *stream);

/*
 * How vssm_scan_grad(a, g, seg_len, ...) would run: *ranges_per_row receives
 * the token ranges each row's adjoint is cut into (joined by the adjoint
 * summaries when more than 1), *launches the number of kernel launches of
 * the call (zero-fills of the accumulated outputs, the checkpoint pass unless
 * g->ckpt is given, the summaries, the adjoint; with the step options or the
 * convolution also the float32 preparation, bfloat16 widening of B and C and
 * the chain rule, and the passes once per direction). Reads only sizes,
 * dstate, dir_flags, the option fields of `a` and which pointers of `g` are
 * set; touches no device. 0 and 0 for an empty problem.
 */
int vssm_scan_grad_plan_query(const vssm_scan_args *a, const vssm_grad_args *g, int seg_len,
                              int *ranges_per_row, int *launches);

/* Bytes of the checkpoints of vssm_scan_train:
 * 64 * directions * batch * ceil(dim / 32) * 32 * ceil(seqlen / 4). */
int vssm_scan_ckpt_size(const vssm_scan_args *a, size_t *bytes);

/*
 * Synchronises `stream`, then reads and clears this device's error word.
 * Returns VSSM_ERR_TIMEOUT if a kernel launched by this library since the
 * last check stopped because its bounded wait for its partner warp (limit
 * 1 s) expired -- its output is then invalid -- and VSSM_OK otherwise. The
 * kernels never trap and never spin without a limit.
 */
int vssm_device_error(void *stream);

/*
 * The scan of vssm_scan_bidir (seg_len == 0) or vssm_scan_folded (seg_len >=
 * 1) with every tensor of `a` in HOST memory (page-locked host memory lets
 * the copies overlap; pageable memory works but serialises them) and the
 * output written back to host memory. The library has no counterpart on the
 * pages: it moves the data for callers whose inputs live on the host.
 *
 * The call is cut into `slices` parts (0 = 8): whole batch entries per slice
 * when batch >= slices, else channel ranges (multiples of 32) of one batch
 * entry. B, C and the per-channel parameters are copied first; then, through
 * a ring of three device slots, each slice's x, delta (z, delta_bwd) are
 * copied in on one stream, scanned on a second and its output copied back on
 * a third, so that the copies in both directions overlap the scans of other
 * slices. a->workspace is DEVICE memory of vssm_scan_host_workspace_size
 * bytes (it holds the slots and the scans' own workspaces); the other
 * pointers of `a` are host pointers, 16-byte aligned. Asynchronous on
 * `stream` (the internal streams fork from it and join back); the output is
 * complete when `stream` reaches the point after the call. Calls on one
 * device serialise their enqueueing. Errors as vssm_scan_bidir; slices < 0
 * gives VSSM_ERR_INVALID_ARG.
 */
int vssm_scan_host(const vssm_scan_args *a, int seg_len, int slices, void *stream);

/* Device workspace bytes of vssm_scan_host with these seg_len and slices. */
int vssm_scan_host_workspace_size(const vssm_scan_args *a, int seg_len, int slices, size_t *bytes);

/*
 * NC-SSD, the non-causal global-state variant (VSSD page, §4.2.4 and §4.2.5:
 * Y = C (B^T (X m))): one hidden state per batch entry, shared by all tokens,
 *
 *   H[n][d]   = sum_j m[j] * B_j[n] * x[d][j]
 *   out[d][t] = (sum_n C_t[n] * H[n][d] + D[d] * x[d][t]) * silu(z[d][t])
 *
 * with per-token weights m (the page's m_j = 1/A_j, computed by the caller),
 * D optional (NULL = 0) and z optional (NULL = no gate). Accumulation in
 * fp32; out is rounded once to the I/O dtype. Tensors as in vssm_scan_args:
 * x, z, out [batch][dim][seqlen], B, C [batch][seqlen][dstate] in `dtype`;
 * m [batch][seqlen] and D [dim] fp32. dstate must be 16 (else
 * VSSM_ERR_UNSUPPORTED); batch <= 65535. H stays on chip: no workspace is
 * needed (vssm_ncssd_workspace_size reports 0 and `workspace` is ignored).
 * The sums over tokens are added in a fixed order, so the result is the same
 * on every run. Device pointers, 16-byte aligned, caller-owned; asynchronous
 * on `stream`. Errors: VSSM_ERR_INVALID_ARG (NULL x, B, C, m or out;
 * negative sizes; out overlapping an input), VSSM_ERR_MISALIGNED,
 * VSSM_ERR_UNSUPPORTED, VSSM_ERR_CUDA (launch failure).
 */
typedef struct {
    const void *x, *z, *B, *C;
    const float *m, *D;
    void *out;
    void *workspace;
    size_t workspace_bytes;
    int batch, dim, seqlen, dstate, dtype;
} vssm_ncssd_args;

int vssm_ncssd(const vssm_ncssd_args *a, void *stream);
int vssm_ncssd_workspace_size(const vssm_ncssd_args *a, size_t *bytes);

/*
 * Test of the timeout path, for callers' own failure-handling tests: runs one
 * warp that waits on a pair barrier whose second arrival never comes. The
 * wait gives up after limit_us microseconds (1..1000000, else
 * VSSM_ERR_INVALID_ARG) and records a timeout in the device error word
 * exactly as the scan kernels do, so that the next vssm_device_error on that
 * stream returns VSSM_ERR_TIMEOUT. Nothing traps, faults or hangs; the device
 * stays usable. Asynchronous on `stream`.
 */
int vssm_selftest_wait_timeout(unsigned limit_us, void *stream);

/* Static text for a vssm_status value. */
const char *vssm_status_string(int status);

/* Text of the last failed call on this thread ("" if none). */
const char *vssm_last_error(void);

/* VSSM_VERSION of the loaded library. */
int vssm_version(void);

#ifdef __cplusplus
}
#endif
#endif /* VSSM_H */
