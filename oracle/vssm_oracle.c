/*
 * fp64 CPU oracle for the bidirectional selective scan (S6) -- TEST
 * INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this. It shares no code with the CUDA path.
 *
 * What it computes, for every batch b and channel d (one "row"), written as
 * the plain definition with no blocking, fusion or reordering:
 *
 *   Discretisation (VSSD page, §4.1.2 "连续→离散化"): the decay is
 *     Abar_t = exp(delta_t * A[d][n]) and the input matrix is taken in its
 *     first-order form Bbar_t ≈ delta_t * B_t (the page's "≈ΔB").
 *   Recurrence (VSSD page, §4.2.1.3 "SSD的线性形式"):
 *     h_t = Abar_t * h_{t-1} + delta_t * B_t * x_t,   h_{-1} = 0
 *     y_t = sum_n C_t[n] * h_t[n] + D[d] * x_t
 *   Backward direction (Vim page, §2.2 "双向状态空间建模": the backward path
 *     runs along the reversed order): the same recurrence walked from
 *     t = L-1 down to 0 with its own A and D, h_L = 0.
 *   Combination: y = y_fwd + y_bwd (each direction adds its own D-skip),
 *     then gated: out_t = y_t * silu(z_t), silu(z) = z / (1 + exp(-z)).
 *   Batch folding with periodic state reset (SF-Mamba page, "批量折叠与周期性
 *     状态重置"): on a folded sequence of segments of seg_len tokens the
 *     discrete decay is set to 0 at every segment start, i.e. at
 *     t mod seg_len == 0 going forward; going backward the segment start is
 *     t mod seg_len == seg_len - 1. There h_t = delta_t * B_t * x_t.
 *
 * No hidden state is returned (SF-Mamba page, "实现优化": hidden-state output
 * suppressed at inference).
 *
 * Per-direction step and fused step transform (oracle_scan_ex): each
 * direction is its own SSM module (Vim page §2.2, the forward_ssm /
 * backward_ssm sketch), so the backward direction may take its own delta.
 * The step may also be given before its positivity map: with `softplus` set,
 * the step of direction k is softplus(delta_k[t] + bias_k[d]), the bias being
 * the step projection's bias (Mamba2D page, "Mamba2D Block结构": dt_proj has
 * bias=True) and softplus(v) = log(1 + exp(v)) the map the Mamba family uses
 * to keep the step positive (the pages name no map; this is a reading).
 *
 * Directional convolution in front of the scan (oracle_conv_silu): "the
 * forward and backward paths use 1D convolutions of different directions"
 * (Vim page §2.3), and the SSM branch takes SiLU of a 1D depthwise
 * convolution (SF-Mamba page, "MambaVision Mixer": X1 = SSM(σ(Conv(...))),
 * σ = SiLU). Per channel d with K taps w[d][0..K-1] and bias b[d]:
 *   forward (causal):   u[t] = silu(b + sum_k w[k] * x[t - (K-1) + k])
 *   backward (reverse): u[t] = silu(b + sum_k w[k] * x[t + (K-1) - k])
 * i.e. the backward one is the causal convolution of the flipped sequence.
 * Taps outside the row are zero; on a folded row they are also zero outside
 * the current segment ("1D深度可分离卷积适配": implicit padding at every
 * segment boundary, the convolution never crosses sequences). The scan then
 * reads each direction's u in place of x (input term and skip alike).
 *
 * Layouts (row-major, last index fastest): x, delta, z, out: [batch][dim][L];
 * B, C (and B_bwd, C_bwd): [batch][L][N]; A: [dim][N]; D: [dim].
 */
#include <math.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_ENOMEM (-2)

int oracle_version(void) { return 2; }

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Folded segment start in a direction's scan order: t mod seg_len == 0
 * going forward, t mod seg_len == seg_len - 1 going backward (never when
 * seg_len == 0). */
static int reset_at(long t, long seg_len, int rev)
{
    if (seg_len <= 0) return 0;
    return rev ? (t % seg_len == seg_len - 1) : (t % seg_len == 0);
}

/* One direction over one row. `rev` = 0 walks t upward, 1 walks downward.
 * Adds y_t into acc[t]. */
static void scan_row_direction(const double *xr, const double *dtr,
                               const double *Bb, const double *Cb,
                               const double *Ad, double Dd,
                               long L, long N, int rev, long seg_len,
                               double *h, double *acc)
{
    for (long n = 0; n < N; ++n) h[n] = 0.0;
    for (long k = 0; k < L; ++k) {
        const long t = rev ? (L - 1 - k) : k;
        const double dt = dtr[t];
        const double xt = xr[t];
        const double *Bt = Bb + t * N;
        const double *Ct = Cb + t * N;
        const int reset = reset_at(t, seg_len, rev);
        double y = 0.0;
        for (long n = 0; n < N; ++n) {
            const double abar = reset ? 0.0 : exp(dt * Ad[n]);
            h[n] = abar * h[n] + dt * Bt[n] * xt;
            y += Ct[n] * h[n];
        }
        acc[t] += y + Dd * xt;
    }
}

/* silu(v) = v / (1 + exp(-v)). */
static double silu(double v) { return v / (1.0 + exp(-v)); }

/*
 * Directional depthwise convolution + SiLU over [batch][dim][L] rows (see the
 * header): reverse = 0 is the causal (forward) one, 1 the backward one. w is
 * [dim][K], b is [dim] (NULL = 0). seg_len > 0 zeroes the taps that fall in
 * another segment. out has x's shape.
 */
int oracle_conv_silu(const double *x, const double *w, const double *b, double *out,
                     long batch, long dim, long L, long K, int reverse, long seg_len)
{
    if (!x || !w || !out || batch < 0 || dim < 0 || L < 0 || K < 1 || seg_len < 0)
        return -1;
    for (long r = 0; r < batch * dim; ++r) {
        const long d = r % dim;
        const double *xr = x + r * L;
        for (long t = 0; t < L; ++t) {
            double acc = b ? b[d] : 0.0;
            for (long k = 0; k < K; ++k) {
                const long s = reverse ? t + (K - 1) - k : t - (K - 1) + k;
                if (s < 0 || s >= L) continue;
                if (seg_len > 0 && s / seg_len != t / seg_len) continue;
                acc += w[d * K + k] * xr[s];
            }
            out[r * L + t] = silu(acc);
        }
    }
    return 0;
}

/* softplus(v) = log(1 + exp(v)), evaluated as max(v, 0) + log(1 + exp(-|v|))
 * so that exp never overflows (the two forms are equal). */
static double softplus(double v)
{
    return (v > 0.0 ? v : 0.0) + log1p(exp(-fabs(v)));
}

/* The step of one direction over one row: the raw values, or, with
 * softplus set, softplus(raw + bias). */
static const double *direction_step(const double *raw, long L, int use_softplus, double bias,
                                    double *buf)
{
    if (!use_softplus) return raw;
    for (long t = 0; t < L; ++t) buf[t] = softplus(raw[t] + bias);
    return buf;
}

/*
 * dirs: bit 0 = forward, bit 1 = backward (at least one set).
 * seg_len: 0 = plain sequences; > 0 = folded with reset every seg_len tokens
 *          (with the backward bit set, L must be a multiple of seg_len).
 * z, D_fwd, D_bwd may be NULL (no gate / zero skip). B_bwd, C_bwd may be NULL
 * (backward shares B, C). nthreads <= 0 uses the OpenMP default.
 */
int oracle_scan_ex(const double *x, const double *delta, const double *z,
                   const double *B, const double *C,
                   const double *B_bwd, const double *C_bwd,
                   const double *A_fwd, const double *A_bwd,
                   const double *D_fwd, const double *D_bwd,
                   const double *delta_bwd, const double *bias_fwd, const double *bias_bwd,
                   int use_softplus, const double *x_bwd, double *out,
                   long batch, long dim, long L, long N,
                   int dirs, long seg_len, int nthreads);

/* The scan with one step tensor for both directions, used as given. */
int oracle_scan(const double *x, const double *delta, const double *z,
                const double *B, const double *C,
                const double *B_bwd, const double *C_bwd,
                const double *A_fwd, const double *A_bwd,
                const double *D_fwd, const double *D_bwd,
                double *out,
                long batch, long dim, long L, long N,
                int dirs, long seg_len, int nthreads)
{
    return oracle_scan_ex(x, delta, z, B, C, B_bwd, C_bwd, A_fwd, A_bwd, D_fwd, D_bwd,
                          NULL, NULL, NULL, 0, NULL, out, batch, dim, L, N, dirs, seg_len,
                          nthreads);
}

/*
 * As oracle_scan, plus: delta_bwd ([batch][dim][L]) is the backward step
 * (NULL = delta); with use_softplus set each direction's step is
 * softplus(its delta + its bias[d]), bias_fwd / bias_bwd ([dim]; NULL = 0 for
 * the forward bias, = bias_fwd for the backward one); x_bwd is the backward
 * direction's input (NULL = x), e.g. its own convolution output.
 */
int oracle_scan_ex(const double *x, const double *delta, const double *z,
                   const double *B, const double *C,
                   const double *B_bwd, const double *C_bwd,
                   const double *A_fwd, const double *A_bwd,
                   const double *D_fwd, const double *D_bwd,
                   const double *delta_bwd, const double *bias_fwd, const double *bias_bwd,
                   int use_softplus, const double *x_bwd, double *out,
                   long batch, long dim, long L, long N,
                   int dirs, long seg_len, int nthreads)
{
    if (!x || !delta || !B || !C || !out) return ORACLE_EINVAL;
    if (batch < 0 || dim < 0 || L < 0 || N <= 0) return ORACLE_EINVAL;
    if (dirs < 1 || dirs > 3) return ORACLE_EINVAL;
    if ((dirs & 1) && !A_fwd) return ORACLE_EINVAL;
    if ((dirs & 2) && !A_bwd) return ORACLE_EINVAL;
    if (seg_len < 0) return ORACLE_EINVAL;
    if (seg_len > 0 && (dirs & 2) && L % seg_len != 0) return ORACLE_EINVAL;
    if (!B_bwd) B_bwd = B;
    if (!C_bwd) C_bwd = C;
    if (!delta_bwd) delta_bwd = delta;
    if (!x_bwd) x_bwd = x;
    if (!bias_bwd) bias_bwd = bias_fwd;

    const long rows = batch * dim;
    int err = ORACLE_OK;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double *h = (double *)malloc(sizeof(double) * (size_t)N);
        double *acc = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        double *step = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        if (!h || !acc || !step) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            err = ORACLE_ENOMEM;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
            for (long r = 0; r < rows; ++r) {
                const long b = r / dim, d = r % dim;
                const double *xr = x + r * L;
                for (long t = 0; t < L; ++t) acc[t] = 0.0;
                if (dirs & 1) {
                    const double *dtr = direction_step(delta + r * L, L, use_softplus,
                                                       bias_fwd ? bias_fwd[d] : 0.0, step);
                    scan_row_direction(xr, dtr, B + b * L * N, C + b * L * N,
                                       A_fwd + d * N, D_fwd ? D_fwd[d] : 0.0,
                                       L, N, 0, seg_len, h, acc);
                }
                if (dirs & 2) {
                    const double *dtr = direction_step(delta_bwd + r * L, L, use_softplus,
                                                       bias_bwd ? bias_bwd[d] : 0.0, step);
                    scan_row_direction(x_bwd + r * L, dtr, B_bwd + b * L * N, C_bwd + b * L * N,
                                       A_bwd + d * N, D_bwd ? D_bwd[d] : 0.0,
                                       L, N, 1, seg_len, h, acc);
                }
                double *outr = out + r * L;
                for (long t = 0; t < L; ++t) {
                    double g = 1.0;
                    if (z) g = silu(z[r * L + t]);
                    outr[t] = acc[t] * g;
                }
            }
        }
        free(h);
        free(acc);
        free(step);
    }
    return err;
}

/*
 * Gradient of the scan (reverse-mode, the plain adjoint of the recurrence
 * above). Given dout = dL/d out, every output gradient below is the exact
 * derivative of L = sum(dout * out) with respect to that input:
 *
 *   s_t = y_fwd_t + y_bwd_t, out_t = s_t * g(z_t), g = silu,
 *   g'(z) = sigma(z) * (1 + z * (1 - sigma(z)));
 *   ds_t = dout_t * g(z_t);   dz_t = dout_t * s_t * g'(z_t);
 *   per direction, walking the tokens against its scan order with the
 *   adjoint lambda_t = dL/dh_t (an N-vector), where x_t and delta_t are that
 *   direction's input and step:
 *     lambda_t = ds_t * C_t + abar_next * lambda_next      (0 past the end)
 *     dC_t    += ds_t * h_t;           dB_t += lambda_t * delta_t * x_t
 *     dx_t    += ds_t * D + sum_n lambda_t[n] * delta_t * B_t[n]
 *     ddelta_t += sum_n lambda_t[n] * (x_t * B_t[n] + A[n] * abar_t[n] * h_prev[n])
 *     dA[n]   += lambda_t[n] * abar_t[n] * h_prev[n] * delta_t
 *     dD      += ds_t * x_t
 *   where h_prev is the state before token t in scan order and abar_t =
 *   exp(delta_t * A); at a folded reset abar_t is the constant 0, so neither
 *   ddelta nor dA gets a decay term there and lambda is not carried past it.
 *
 * With the step options and the convolution of oracle_scan_ex (the inputs
 * below), each direction k's step and input are functions of the raw
 * tensors, and the chain rule carries the per-direction gradients of the
 * step (d step_k) and of the input (d u_k) back to them:
 *   step_k = softplus(v_k + bias_k)  (use_softplus; v_k = delta or delta_bwd)
 *            d v_k = d step_k * sigma(v_k + bias_k),  d bias_k = sum_t d v_k
 *            (softplus'(v) = sigma(v)); otherwise step_k = v_k, d v_k = d step_k
 *   u_k = silu(pre_k), pre_k[t] = cb_k + sum_j w_k[j] * x[tap_k(t, j)]  (K > 0)
 *            d pre_k = d u_k * silu'(pre_k),  silu'(p) = sigma(p) + p sigma(p) (1 - sigma(p))
 *            dx[tap] += w_k[j] * d pre_k,  d w_k[j] += d pre_k * x[tap],  d cb_k += d pre_k
 *            with tap_k(t, j) = t - (K-1) + j forward, t + (K-1) - j backward
 *            (taps outside the row or, folded, the segment read zero)
 *   u_k = x otherwise, dx += d u_k.
 * A backward parameter that is NULL is the forward one, and its gradient is
 * added to the forward one's.
 *
 * Inputs as oracle_scan_ex (delta_bwd, bias_fwd, bias_bwd, use_softplus) plus
 * the convolution (conv_w [dim][K], conv_b [dim], conv_w_bwd, conv_b_bwd;
 * K = 0: none). z, D_fwd, D_bwd, B_bwd, C_bwd, delta_bwd, biases and conv_b*
 * may be NULL. Gradients are written (not accumulated): dx, ddelta, dz
 * [batch][dim][L] (dz ignored if z is NULL); ddelta_bwd (required iff
 * delta_bwd is given); dB, dC [batch][L][N]; when B_bwd / C_bwd are given,
 * the backward direction's go to dB_bwd / dC_bwd (else into dB / dC); dA_fwd,
 * dA_bwd [dim][N]; dD_fwd, dD_bwd [dim] (each required iff its direction
 * runs); dbias_fwd [dim] (required iff use_softplus), dbias_bwd (iff
 * bias_bwd is given with use_softplus); dconv_w [dim][K] (iff K > 0),
 * dconv_b (iff conv_b), dconv_w_bwd (iff conv_w_bwd), dconv_b_bwd (iff
 * conv_b_bwd). Single-threaded.
 */
static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

/* silu'(p) = sigma(p) + p * sigma(p) * (1 - sigma(p)). */
static double dsilu(double p)
{
    const double q = sigmoid(p);
    return q + p * q * (1.0 - q);
}

/* Source token of convolution tap j for output token t (-1 when the tap
 * reads zero: outside the row or, folded, outside t's segment). */
static long conv_tap(long t, long j, long K, long L, long seg_len, int reverse)
{
    const long s = reverse ? t + (K - 1) - j : t - (K - 1) + j;
    if (s < 0 || s >= L) return -1;
    if (seg_len > 0 && s / seg_len != t / seg_len) return -1;
    return s;
}

int oracle_scan_grad_ex(const double *x, const double *delta, const double *z,
                        const double *B, const double *C,
                        const double *B_bwd, const double *C_bwd,
                        const double *A_fwd, const double *A_bwd,
                        const double *D_fwd, const double *D_bwd,
                        const double *delta_bwd, const double *bias_fwd, const double *bias_bwd,
                        int use_softplus,
                        const double *conv_w, const double *conv_b,
                        const double *conv_w_bwd, const double *conv_b_bwd, long K,
                        const double *dout,
                        double *dx, double *ddelta, double *dz,
                        double *dB, double *dC, double *dB_bwd, double *dC_bwd,
                        double *dA_fwd, double *dA_bwd, double *dD_fwd, double *dD_bwd,
                        double *ddelta_bwd, double *dbias_fwd, double *dbias_bwd,
                        double *dconv_w, double *dconv_b, double *dconv_w_bwd, double *dconv_b_bwd,
                        long batch, long dim, long L, long N, int dirs, long seg_len)
{
    if (!x || !delta || !B || !C || !dout || !dx || !ddelta || !dB || !dC) return ORACLE_EINVAL;
    if (batch < 0 || dim < 0 || L < 0 || N <= 0 || dirs < 1 || dirs > 3 || seg_len < 0 || K < 0)
        return ORACLE_EINVAL;
    if ((dirs & 1) && (!A_fwd || !dA_fwd || !dD_fwd)) return ORACLE_EINVAL;
    if ((dirs & 2) && (!A_bwd || !dA_bwd || !dD_bwd)) return ORACLE_EINVAL;
    if (seg_len > 0 && (dirs & 2) && L % seg_len != 0) return ORACLE_EINVAL;
    if ((B_bwd && !dB_bwd) || (C_bwd && !dC_bwd)) return ORACLE_EINVAL;
    if (delta_bwd && !ddelta_bwd) return ORACLE_EINVAL;
    if (use_softplus && (!dbias_fwd || (bias_bwd && !dbias_bwd))) return ORACLE_EINVAL;
    if (K > 0 && (!conv_w || !dconv_w || (conv_b && !dconv_b) || (conv_w_bwd && !dconv_w_bwd) ||
                  (conv_b_bwd && !dconv_b_bwd)))
        return ORACLE_EINVAL;
    const long rows = batch * dim;
    for (long i = 0; i < rows * L; ++i) {
        dx[i] = 0.0;
        ddelta[i] = 0.0;
        if (delta_bwd) ddelta_bwd[i] = 0.0;
        if (z && dz) dz[i] = 0.0;
    }
    for (long i = 0; i < batch * L * N; ++i) {
        dB[i] = 0.0;
        dC[i] = 0.0;
        if (B_bwd) dB_bwd[i] = 0.0;
        if (C_bwd) dC_bwd[i] = 0.0;
    }
    for (long i = 0; i < dim * N; ++i) {
        if (dirs & 1) dA_fwd[i] = 0.0;
        if (dirs & 2) dA_bwd[i] = 0.0;
    }
    for (long i = 0; i < dim; ++i) {
        if (dirs & 1) dD_fwd[i] = 0.0;
        if (dirs & 2) dD_bwd[i] = 0.0;
        if (use_softplus) dbias_fwd[i] = 0.0;
        if (use_softplus && bias_bwd) dbias_bwd[i] = 0.0;
        if (K > 0 && conv_b) dconv_b[i] = 0.0;
        if (K > 0 && conv_b_bwd) dconv_b_bwd[i] = 0.0;
    }
    for (long i = 0; i < dim * K; ++i) {
        dconv_w[i] = 0.0;
        if (conv_w_bwd) dconv_w_bwd[i] = 0.0;
    }
    const size_t LL = (size_t)(L > 0 ? L : 1);
    double *H = (double *)malloc(sizeof(double) * LL * (size_t)N * 2);
    double *Ab = (double *)malloc(sizeof(double) * LL * (size_t)N * 2);
    double *y = (double *)malloc(sizeof(double) * LL * 2);
    double *lam = (double *)malloc(sizeof(double) * (size_t)N);
    double *u = (double *)malloc(sizeof(double) * LL * 2);      /* each direction's input   */
    double *pre = (double *)malloc(sizeof(double) * LL * 2);    /* ... its conv argument    */
    double *st = (double *)malloc(sizeof(double) * LL * 2);     /* ... its step             */
    double *du = (double *)malloc(sizeof(double) * LL * 2);     /* d input, per direction   */
    double *dst = (double *)malloc(sizeof(double) * LL * 2);    /* d step, per direction    */
    if (!H || !Ab || !y || !lam || !u || !pre || !st || !du || !dst) {
        free(H); free(Ab); free(y); free(lam); free(u); free(pre); free(st); free(du); free(dst);
        return ORACLE_ENOMEM;
    }
    for (long r = 0; r < rows; ++r) {
        const long b = r / dim, d = r % dim;
        const double *xraw = x + r * L;
        /* each direction's step and input */
        for (int k = 0; k < 2; ++k) {
            if (!(dirs & (1 << k))) continue;
            const double *v = (k && delta_bwd ? delta_bwd : delta) + r * L;
            const double *bk = k && bias_bwd ? bias_bwd : bias_fwd;
            const double bias = bk ? bk[d] : 0.0;
            const double *wk = k && conv_w_bwd ? conv_w_bwd : conv_w;
            const double *cbk = k && conv_b_bwd ? conv_b_bwd : conv_b;
            for (long t = 0; t < L; ++t) {
                st[k * L + t] = use_softplus ? softplus(v[t] + bias) : v[t];
                if (K > 0) {
                    double a = cbk ? cbk[d] : 0.0;
                    for (long j = 0; j < K; ++j) {
                        const long sidx = conv_tap(t, j, K, L, seg_len, k);
                        if (sidx >= 0) a += wk[d * K + j] * xraw[sidx];
                    }
                    pre[k * L + t] = a;
                    u[k * L + t] = silu(a);
                } else {
                    u[k * L + t] = xraw[t];
                }
                du[k * L + t] = 0.0;
                dst[k * L + t] = 0.0;
            }
        }
        /* forward states and outputs of each direction (k = 0 fwd, 1 bwd) */
        for (int k = 0; k < 2; ++k) {
            if (!(dirs & (1 << k))) continue;
            const double *xr = u + k * L, *dtr = st + k * L;
            const double *Bk = (k && B_bwd ? B_bwd : B) + b * L * N;
            const double *Ck = (k && C_bwd ? C_bwd : C) + b * L * N;
            const double *Ak = (k ? A_bwd : A_fwd) + d * N;
            const double Dk = k ? (D_bwd ? D_bwd[d] : 0.0) : (D_fwd ? D_fwd[d] : 0.0);
            double *Hk = H + (size_t)k * L * N, *Abk = Ab + (size_t)k * L * N;
            for (long s = 0; s < L; ++s) {
                const long t = k ? L - 1 - s : s;
                const int reset = reset_at(t, seg_len, k);
                const long tp = k ? t + 1 : t - 1;           /* previous token in scan order */
                double yy = 0.0;
                for (long n = 0; n < N; ++n) {
                    const double a = reset ? 0.0 : exp(dtr[t] * Ak[n]);
                    const double hp = (s == 0) ? 0.0 : Hk[tp * N + n];
                    Abk[t * N + n] = a;
                    Hk[t * N + n] = a * hp + dtr[t] * Bk[t * N + n] * xr[t];
                    yy += Ck[t * N + n] * Hk[t * N + n];
                }
                y[k * L + t] = yy + Dk * xr[t];
            }
        }
        for (int k = 0; k < 2; ++k) {
            if (!(dirs & (1 << k))) continue;
            const double *xr = u + k * L, *dtr = st + k * L;
            double *dur = du + k * L, *dstr = dst + k * L;
            const double *Bk = (k && B_bwd ? B_bwd : B) + b * L * N;
            const double *Ck = (k && C_bwd ? C_bwd : C) + b * L * N;
            double *dBk = (k && B_bwd ? dB_bwd : dB) + b * L * N;
            double *dCk = (k && C_bwd ? dC_bwd : dC) + b * L * N;
            const double *Ak = (k ? A_bwd : A_fwd) + d * N;
            double *dAk = (k ? dA_bwd : dA_fwd) + d * N;
            const double Dk = k ? (D_bwd ? D_bwd[d] : 0.0) : (D_fwd ? D_fwd[d] : 0.0);
            double *dDk = (k ? dD_bwd : dD_fwd) + d;
            const double *Hk = H + (size_t)k * L * N, *Abk = Ab + (size_t)k * L * N;
            for (long n = 0; n < N; ++n) lam[n] = 0.0;
            /* against the scan order: forward walks down, backward walks up */
            for (long s = L - 1; s >= 0; --s) {
                const long t = k ? L - 1 - s : s;
                const long tp = k ? t + 1 : t - 1;
                const double g = z ? silu(z[r * L + t]) : 1.0;
                const double ds = dout[r * L + t] * g;
                *dDk += ds * xr[t];
                double dxx = ds * Dk, ddt = 0.0;
                for (long n = 0; n < N; ++n) {
                    lam[n] = ds * Ck[t * N + n] + lam[n];
                    dCk[t * N + n] += ds * Hk[t * N + n];
                    dBk[t * N + n] += lam[n] * dtr[t] * xr[t];
                    dxx += lam[n] * dtr[t] * Bk[t * N + n];
                    const double hp = (s == 0) ? 0.0 : Hk[tp * N + n];
                    const double a = Abk[t * N + n];
                    ddt += lam[n] * (xr[t] * Bk[t * N + n] + Ak[n] * a * hp);
                    dAk[n] += lam[n] * a * hp * dtr[t];
                    lam[n] = a * lam[n];
                }
                dur[t] += dxx;
                dstr[t] += ddt;
            }
        }
        if (z && dz) {
            for (long t = 0; t < L; ++t) {
                const double zt = z[r * L + t];
                const double sg = 1.0 / (1.0 + exp(-zt));
                double s = 0.0;
                if (dirs & 1) s += y[t];
                if (dirs & 2) s += y[L + t];
                dz[r * L + t] = dout[r * L + t] * s * sg * (1.0 + zt * (1.0 - sg));
            }
        }
        /* chain rule back to the raw step, its bias, x and the taps */
        for (int k = 0; k < 2; ++k) {
            if (!(dirs & (1 << k))) continue;
            const double *v = (k && delta_bwd ? delta_bwd : delta) + r * L;
            double *dv = (k && delta_bwd ? ddelta_bwd : ddelta) + r * L;
            const double *bk = k && bias_bwd ? bias_bwd : bias_fwd;
            double *dbk = k && bias_bwd ? dbias_bwd : dbias_fwd;
            const double bias = bk ? bk[d] : 0.0;
            const double *wk = k && conv_w_bwd ? conv_w_bwd : conv_w;
            double *dwk = k && conv_w_bwd ? dconv_w_bwd : dconv_w;
            double *dcbk = k && conv_b_bwd ? dconv_b_bwd : (conv_b ? dconv_b : NULL);
            for (long t = 0; t < L; ++t) {
                const double g_step = dst[k * L + t] * (use_softplus ? sigmoid(v[t] + bias) : 1.0);
                dv[t] += g_step;
                if (use_softplus) dbk[d] += g_step;
                if (K > 0) {
                    const double dp = du[k * L + t] * dsilu(pre[k * L + t]);
                    for (long j = 0; j < K; ++j) {
                        const long sidx = conv_tap(t, j, K, L, seg_len, k);
                        if (sidx < 0) continue;
                        dx[r * L + sidx] += wk[d * K + j] * dp;
                        dwk[d * K + j] += dp * xraw[sidx];
                    }
                    if (dcbk) dcbk[d] += dp;
                } else {
                    dx[r * L + t] += du[k * L + t];
                }
            }
        }
    }
    free(H); free(Ab); free(y); free(lam); free(u); free(pre); free(st); free(du); free(dst);
    return ORACLE_OK;
}

/* The gradient with the steps used as given, shared by both directions, and
 * no convolution (the inputs and outputs of oracle_scan). */
int oracle_scan_grad(const double *x, const double *delta, const double *z,
                     const double *B, const double *C,
                     const double *B_bwd, const double *C_bwd,
                     const double *A_fwd, const double *A_bwd,
                     const double *D_fwd, const double *D_bwd,
                     const double *dout,
                     double *dx, double *ddelta, double *dz,
                     double *dB, double *dC, double *dB_bwd, double *dC_bwd,
                     double *dA_fwd, double *dA_bwd, double *dD_fwd, double *dD_bwd,
                     long batch, long dim, long L, long N, int dirs, long seg_len)
{
    return oracle_scan_grad_ex(x, delta, z, B, C, B_bwd, C_bwd, A_fwd, A_bwd, D_fwd, D_bwd,
                               NULL, NULL, NULL, 0, NULL, NULL, NULL, NULL, 0, dout,
                               dx, ddelta, dz, dB, dC, dB_bwd, dC_bwd, dA_fwd, dA_bwd, dD_fwd, dD_bwd,
                               NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                               batch, dim, L, N, dirs, seg_len);
}

/*
 * NC-SSD, the non-causal global-state variant (VSSD page, §4.2.4 and
 * §4.2.5): every token contributes m_j * B_j x_j^T to one hidden state per
 * batch entry, shared by all tokens, and each token reads it through C:
 *
 *   H[n][d]  = sum_j m[j] * B_j[n] * x[d][j]                (§4.2.4, H = sum_j (1/A_j) Z_j)
 *   out[d][t] = (sum_n C_t[n] * H[n][d] + D[d] * x[d][t]) * g(z[d][t])
 *
 * with m the per-token weights (the page's m_j = 1/A_j, passed in), D the
 * optional skip (NULL = 0) and g = silu of the optional gate (NULL = 1), as
 * in the scan. Layouts as oracle_scan; m is [batch][L].
 */
int oracle_ncssd(const double *x, const double *z, const double *B, const double *C,
                 const double *m, const double *D, double *out,
                 long batch, long dim, long L, long N)
{
    if (!x || !B || !C || !m || !out || batch < 0 || dim < 0 || L < 0 || N <= 0)
        return ORACLE_EINVAL;
    double *H = (double *)malloc(sizeof(double) * (size_t)N * (size_t)(dim > 0 ? dim : 1));
    if (!H) return ORACLE_ENOMEM;
    for (long b = 0; b < batch; ++b) {
        const double *xb = x + b * dim * L, *Bb = B + b * L * N, *Cb = C + b * L * N;
        const double *mb = m + b * L;
        for (long n = 0; n < N; ++n)
            for (long d = 0; d < dim; ++d) {
                double h = 0.0;
                for (long j = 0; j < L; ++j) h += mb[j] * Bb[j * N + n] * xb[d * L + j];
                H[n * dim + d] = h;
            }
        for (long d = 0; d < dim; ++d)
            for (long t = 0; t < L; ++t) {
                double y = D ? D[d] * xb[d * L + t] : 0.0;
                for (long n = 0; n < N; ++n) y += Cb[t * N + n] * H[n * dim + d];
                const double g = z ? silu(z[(b * dim + d) * L + t]) : 1.0;
                out[(b * dim + d) * L + t] = y * g;
            }
    }
    free(H);
    return ORACLE_OK;
}
