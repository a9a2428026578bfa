/*
 * CPU oracle for the Mamba-3 layer recurrence -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, sequential fp64 code that states the recurrence literally, with
 * a complex-valued state.  It exists so that the CUDA path has something
 * independent to be compared against.  Only tests/, __graft_entry__.smoke()
 * and bench.py's cpu_baseline / reference legs may load it; the product
 * library never links or calls it, and it shares no code with the CUDA path.
 *
 * Sources (the Mamba-3 pages; page title or address, then section):
 *  - linkstar.cloud/article/869, section "第一刀：指数梯形离散化 / Mamba-3的升级":
 *      h_t = alpha_t h_{t-1} + beta_t B_{t-1} x_{t-1} + gamma_t B_t x_t,
 *      alpha_t = exp(dt_t A_t), beta_t = (1 - lambda_t) dt_t alpha_t,
 *      gamma_t = lambda_t dt_t.
 *  - same page, section "第二刀：复值状态空间 / Mamba-3的解法": the state is
 *      complex; its transition is exp(dt_t (A_t + i theta_t)), which on a real
 *      (re, im) pair is a scaling by exp(dt_t A_t) times the 2x2 rotation
 *      R(dt_t theta_t) = [[cos, -sin], [sin, cos]]; C carries a minus sign
 *      on its imaginary half so that the complex and the real forms agree.
 *  - "Mamba-3：基于状态空间原理改进序列建模" (papers.ananclaw.com explainer),
 *      section "关键公式与伪代码": y_t = Re(C_t h_t).
 *  - linkstar.cloud/article/869, section "第三刀：多输入多输出 / MIMO的思路":
 *      B_t is N x R and x_t is P x R, so B_t x_t^T is a rank-R matrix product.
 *
 * Readings taken where the pages are silent:
 *  - complex pairs are adjacent real entries: S_k = h[2k] + i h[2k+1];
 *  - the left-endpoint (beta) term is propagated by the full complex
 *    transition, i.e. beta_t = (1 - lambda_t) dt_t exp(dt_t (A_t + i theta_k));
 *  - complex C_k = C[2k] - i C[2k+1], so y = Re(sum_k C_k S_k) equals the real
 *    dot product C^T h;
 *  - before the first token, B_{-1} x_{-1} is the carry passed in (0 if none).
 *
 * Layouts (row-major, contiguous, all double):
 *   x      [batch][L][H][R][P]        B, C   [batch][L][H][R][N]
 *   dt, A, lam [batch][L][H]          theta  [batch][L][H][N/2]
 *   h0, h_out  [batch][H][N][P]       Bprev  [batch][H][R][N]   xprev [batch][H][R][P]
 *   y      [batch][L][H][R][P]
 * h0, Bprev, xprev may be NULL (zero state, zero carry).  h_out, Bprev_out and
 * xprev_out may be NULL (not written).  The decode step is this function
 * with L = 1.
 */
#include <complex.h>
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int batch, L, H, P, N, R;
    const double *x, *B, *C, *dt, *A, *lam, *theta;
    const double *h0, *Bprev, *xprev;
    double *y, *h_out, *Bprev_out, *xprev_out;
} oracle_problem;

/* One (b, h) sequence, token by token. Returns 0, or -1 when out of memory. */
static int scan_sequence(const oracle_problem *pr, int b, int h)
{
    const int L = pr->L, H = pr->H, P = pr->P, N = pr->N, R = pr->R, K = N / 2;
    double complex *S = calloc((size_t)K * P, sizeof(double complex));
    double complex *Bp = calloc((size_t)R * K, sizeof(double complex));   /* previous B, complex pairs */
    double *xp = calloc((size_t)R * P, sizeof(double));                   /* previous x */
    double complex *z = calloc((size_t)K, sizeof(double complex));
    if (!S || !Bp || !xp || !z) {
        free(S); free(Bp); free(xp); free(z);
        return -1;
    }
    const size_t bh = (size_t)b * H + h;

    /* initial state (true frame) and carry */
    if (pr->h0) {
        const double *h0 = pr->h0 + bh * N * P;
        for (int k = 0; k < K; ++k)
            for (int p = 0; p < P; ++p)
                S[k * P + p] = h0[(2 * k) * P + p] + I * h0[(2 * k + 1) * P + p];
    }
    if (pr->Bprev && pr->xprev) {
        const double *bq = pr->Bprev + bh * R * N;
        const double *xq = pr->xprev + bh * R * P;
        for (int r = 0; r < R; ++r) {
            for (int k = 0; k < K; ++k)
                Bp[r * K + k] = bq[r * N + 2 * k] + I * bq[r * N + 2 * k + 1];
            for (int p = 0; p < P; ++p)
                xp[r * P + p] = xq[r * P + p];
        }
    }

    for (int t = 0; t < L; ++t) {
        const size_t tok = ((size_t)b * L + t) * H + h;        /* index into [batch][L][H] */
        const double dt = pr->dt[tok], A = pr->A[tok], lam = pr->lam[tok];
        const double *th = pr->theta + tok * K;
        const double *xt = pr->x + tok * R * P;
        const double *Bt = pr->B + tok * R * N;
        const double *Ct = pr->C + tok * R * N;

        /* complex transition z_k = exp(dt (A + i theta_k)) */
        for (int k = 0; k < K; ++k)
            z[k] = cexp(dt * A + I * (dt * th[k]));
        const double left = (1.0 - lam) * dt;   /* beta_t / transition */
        const double right = lam * dt;          /* gamma_t */

        for (int k = 0; k < K; ++k) {
            for (int p = 0; p < P; ++p) {
                double complex u = 0.0, v = 0.0;   /* B_{t-1} x_{t-1}^T and B_t x_t^T, entry (k, p) */
                for (int r = 0; r < R; ++r) {
                    u += Bp[r * K + k] * xp[r * P + p];
                    v += (Bt[r * N + 2 * k] + I * Bt[r * N + 2 * k + 1]) * xt[r * P + p];
                }
                S[k * P + p] = z[k] * (S[k * P + p] + left * u) + right * v;
            }
        }

        /* y_t = Re(C_t h_t), complex C_k = C[2k] - i C[2k+1] */
        double *yt = pr->y + tok * R * P;
        for (int r = 0; r < R; ++r) {
            for (int p = 0; p < P; ++p) {
                double acc = 0.0;
                for (int k = 0; k < K; ++k) {
                    const double complex ck = Ct[r * N + 2 * k] - I * Ct[r * N + 2 * k + 1];
                    acc += creal(ck * S[k * P + p]);
                }
                yt[r * P + p] = acc;
            }
        }

        /* this token becomes the previous one */
        for (int r = 0; r < R; ++r) {
            for (int k = 0; k < K; ++k)
                Bp[r * K + k] = Bt[r * N + 2 * k] + I * Bt[r * N + 2 * k + 1];
            for (int p = 0; p < P; ++p)
                xp[r * P + p] = xt[r * P + p];
        }
    }

    if (pr->h_out) {
        double *ho = pr->h_out + bh * N * P;
        for (int k = 0; k < K; ++k)
            for (int p = 0; p < P; ++p) {
                ho[(2 * k) * P + p] = creal(S[k * P + p]);
                ho[(2 * k + 1) * P + p] = cimag(S[k * P + p]);
            }
    }
    if (pr->Bprev_out && pr->xprev_out) {
        double *bo = pr->Bprev_out + bh * R * N;
        double *xo = pr->xprev_out + bh * R * P;
        for (int r = 0; r < R; ++r) {
            for (int k = 0; k < K; ++k) {
                bo[r * N + 2 * k] = creal(Bp[r * K + k]);
                bo[r * N + 2 * k + 1] = cimag(Bp[r * K + k]);
            }
            for (int p = 0; p < P; ++p)
                xo[r * P + p] = xp[r * P + p];
        }
    }
    free(S); free(Bp); free(xp); free(z);
    return 0;
}

/*
 * Reverse mode (the backward pass used for training; linkstar.cloud/article/869, section
 * "训练怎么办": the recurrence is trained through its chunked form) of one (b, h) sequence,
 * written as the adjoint of the sequential recurrence above, step by step backwards.  For a real
 * loss and a complex state S, G = dLoss/dRe(S) + i dLoss/dIm(S).  Per token t, with
 * W = S_{t-1} + left u (pre-transition), S_t = z W + right v, y_t = Re(sum_k Cc_k S_t):
 *   G += sum_r dy_t[r] (C[2k] + i C[2k+1]);  dC[2k] = sum_p dy Re S, dC[2k+1] = sum_p dy Im S;
 *   G_W = conj(z) G;  d(dt A) = sum Re(conj(z W) G);  d(dt theta_k) = sum_p Im(conj(z W) G);
 *   d right = sum Re(conj(v) G);  d left = sum Re(conj(u) G_W);
 *   v = sum_r Bc_r x_r:  dBc_r += right sum_p G x_r,   dx_r += right sum_k Re(conj(Bc_r) G);
 *   u likewise with the previous token's B, x and left G_W;   then G <- G_W.
 * Gradients in, all double and of the forward layouts: dy [L][H][R][P] (of the whole problem),
 * dh_out [H][N][P], dBprev_out [H][R][N], dxprev_out [H][R][P] (NULL = 0).  Out: dx, dB, dC, ddt,
 * dA, dlam, dtheta, dh0, dBprev, dxprev (NULL = not written).
 */
typedef struct {
    const double *dy, *dh_out, *dBprev_out, *dxprev_out;
    double *dx, *dB, *dC, *ddt, *dA, *dlam, *dtheta, *dh0, *dBprev, *dxprev;
} oracle_grads;

static int scan_sequence_bwd(const oracle_problem *pr, const oracle_grads *gr, int b, int h)
{
    const int L = pr->L, H = pr->H, P = pr->P, N = pr->N, R = pr->R, K = N / 2;
    const size_t bh = (size_t)b * H + h;
    double complex *S = calloc((size_t)(L + 1) * K * P, sizeof(double complex));   /* S_{t-1} at t */
    double complex *G = calloc((size_t)K * P, sizeof(double complex));
    double complex *GW = calloc((size_t)K * P, sizeof(double complex));
    double *dBcur = calloc((size_t)R * N, sizeof(double));    /* gradient of the current token's B, x */
    double *dxcur = calloc((size_t)R * P, sizeof(double));
    if (!S || !G || !GW || !dBcur || !dxcur) {
        free(S); free(G); free(GW); free(dBcur); free(dxcur);
        return -1;
    }
    /* forward, keeping every state */
    const double *bq = pr->Bprev ? pr->Bprev + bh * R * N : NULL;
    const double *xq = pr->xprev ? pr->xprev + bh * R * P : NULL;
    if (pr->h0)
        for (int k = 0; k < K; ++k)
            for (int p = 0; p < P; ++p)
                S[k * P + p] = pr->h0[(bh * N + 2 * k) * P + p] + I * pr->h0[(bh * N + 2 * k + 1) * P + p];
    for (int t = 0; t < L; ++t) {
        const size_t tok = ((size_t)b * L + t) * H + h;
        const double dt = pr->dt[tok], A = pr->A[tok], lam = pr->lam[tok];
        const double *Bp = t > 0 ? pr->B + (tok - H) * R * N : bq;
        const double *xp = t > 0 ? pr->x + (tok - H) * R * P : xq;
        const double *Bt = pr->B + tok * R * N, *xt = pr->x + tok * R * P;
        const double complex *Sp = S + (size_t)t * K * P;
        double complex *Sn = S + (size_t)(t + 1) * K * P;
        for (int k = 0; k < K; ++k) {
            const double complex z = cexp(dt * A + I * (dt * pr->theta[tok * K + k]));
            for (int p = 0; p < P; ++p) {
                double complex u = 0.0, v = 0.0;
                for (int r = 0; r < R; ++r) {
                    if (Bp) u += (Bp[r * N + 2 * k] + I * Bp[r * N + 2 * k + 1]) * xp[r * P + p];
                    v += (Bt[r * N + 2 * k] + I * Bt[r * N + 2 * k + 1]) * xt[r * P + p];
                }
                Sn[k * P + p] = z * (Sp[k * P + p] + (1.0 - lam) * dt * u) + lam * dt * v;
            }
        }
    }
    /* backward */
    if (gr->dh_out)
        for (int k = 0; k < K; ++k)
            for (int p = 0; p < P; ++p)
                G[k * P + p] = gr->dh_out[(bh * N + 2 * k) * P + p] + I * gr->dh_out[(bh * N + 2 * k + 1) * P + p];
    /* the carry out is the last token's (B, x) */
    for (int i = 0; i < R * N; ++i) dBcur[i] = gr->dBprev_out ? gr->dBprev_out[bh * R * N + i] : 0.0;
    for (int i = 0; i < R * P; ++i) dxcur[i] = gr->dxprev_out ? gr->dxprev_out[bh * R * P + i] : 0.0;
    for (int t = L - 1; t >= 0; --t) {
        const size_t tok = ((size_t)b * L + t) * H + h;
        const double dt = pr->dt[tok], A = pr->A[tok], lam = pr->lam[tok];
        const double left = (1.0 - lam) * dt, right = lam * dt;
        const double *Bp = t > 0 ? pr->B + (tok - H) * R * N : bq;
        const double *xp = t > 0 ? pr->x + (tok - H) * R * P : xq;
        const double *Bt = pr->B + tok * R * N, *xt = pr->x + tok * R * P, *Ct = pr->C + tok * R * N;
        const double *dyt = gr->dy + tok * R * P;
        const double complex *Sp = S + (size_t)t * K * P, *St = S + (size_t)(t + 1) * K * P;
        /* readout y_t = Re(Cc S_t) */
        for (int r = 0; r < R; ++r)
            for (int k = 0; k < K; ++k) {
                double c0 = 0.0, c1 = 0.0;
                for (int p = 0; p < P; ++p) {
                    c0 += dyt[r * P + p] * creal(St[k * P + p]);
                    c1 += dyt[r * P + p] * cimag(St[k * P + p]);
                    G[k * P + p] += dyt[r * P + p] * (Ct[r * N + 2 * k] + I * Ct[r * N + 2 * k + 1]);
                }
                if (gr->dC) {
                    gr->dC[tok * R * N + r * N + 2 * k] = c0;
                    gr->dC[tok * R * N + r * N + 2 * k + 1] = c1;
                }
            }
        double da = 0.0, dleft = 0.0, dright = 0.0, dth_sum = 0.0;
        double *dBprev_t = calloc((size_t)R * N, sizeof(double)), *dxprev_t = calloc((size_t)R * P, sizeof(double));
        if (!dBprev_t || !dxprev_t) {
            free(dBprev_t); free(dxprev_t); free(S); free(G); free(GW); free(dBcur); free(dxcur);
            return -1;
        }
        for (int k = 0; k < K; ++k) {
            const double th = pr->theta[tok * K + k];
            const double complex z = cexp(dt * A + I * (dt * th));
            double dom = 0.0;
            for (int p = 0; p < P; ++p) {
                double complex u = 0.0, v = 0.0;
                for (int r = 0; r < R; ++r) {
                    if (Bp) u += (Bp[r * N + 2 * k] + I * Bp[r * N + 2 * k + 1]) * xp[r * P + p];
                    v += (Bt[r * N + 2 * k] + I * Bt[r * N + 2 * k + 1]) * xt[r * P + p];
                }
                const double complex g = G[k * P + p];
                const double complex W = Sp[k * P + p] + left * u;
                const double complex gw = conj(z) * g;
                const double complex q = conj(z * W) * g;
                da += creal(q);
                dom += cimag(q);
                dright += creal(conj(v) * g);
                dleft += creal(conj(u) * gw);
                GW[k * P + p] = gw;
                /* v = sum_r Bc_r x_r (this token), u = sum_r Bp_r xp_r (previous token) */
                for (int r = 0; r < R; ++r) {
                    const double complex bc = Bt[r * N + 2 * k] + I * Bt[r * N + 2 * k + 1];
                    const double complex dv = right * g, du = left * gw;
                    dBcur[r * N + 2 * k] += creal(dv) * xt[r * P + p];
                    dBcur[r * N + 2 * k + 1] += cimag(dv) * xt[r * P + p];
                    dxcur[r * P + p] += creal(conj(bc) * dv);
                    if (Bp) {
                        const double complex bpc = Bp[r * N + 2 * k] + I * Bp[r * N + 2 * k + 1];
                        dBprev_t[r * N + 2 * k] += creal(du) * xp[r * P + p];
                        dBprev_t[r * N + 2 * k + 1] += cimag(du) * xp[r * P + p];
                        dxprev_t[r * P + p] += creal(conj(bpc) * du);
                    }
                }
            }
            if (gr->dtheta) gr->dtheta[tok * K + k] = dt * dom;
            dth_sum += th * dom;
        }
        if (gr->dA) gr->dA[tok] = dt * da;
        if (gr->ddt) gr->ddt[tok] = A * da + dth_sum + (1.0 - lam) * dleft + lam * dright;
        if (gr->dlam) gr->dlam[tok] = dt * (dright - dleft);
        /* this token's B, x are complete; the previous token's start with what u gave them */
        if (gr->dB) memcpy(gr->dB + tok * R * N, dBcur, sizeof(double) * R * N);
        if (gr->dx) memcpy(gr->dx + tok * R * P, dxcur, sizeof(double) * R * P);
        memcpy(dBcur, dBprev_t, sizeof(double) * R * N);
        memcpy(dxcur, dxprev_t, sizeof(double) * R * P);
        free(dBprev_t); free(dxprev_t);
        memcpy(G, GW, sizeof(double complex) * K * P);
    }
    if (gr->dh0)
        for (int k = 0; k < K; ++k)
            for (int p = 0; p < P; ++p) {
                gr->dh0[(bh * N + 2 * k) * P + p] = creal(G[k * P + p]);
                gr->dh0[(bh * N + 2 * k + 1) * P + p] = cimag(G[k * P + p]);
            }
    if (gr->dBprev) memcpy(gr->dBprev + bh * R * N, dBcur, sizeof(double) * R * N);
    if (gr->dxprev) memcpy(gr->dxprev + bh * R * P, dxcur, sizeof(double) * R * P);
    free(S); free(G); free(GW); free(dBcur); free(dxcur);
    return 0;
}

/* The backward pass of every (b, h) sequence, one after another.  Returns 0, or -1 on bad arguments
 * or out of memory.  L = 0: the gradients of the state and carry pass through. */
int oracle_scan_bwd(int batch, int L, int H, int P, int N, int R,
                    const double *x, const double *B, const double *C,
                    const double *dt, const double *A, const double *lam, const double *theta,
                    const double *h0, const double *Bprev, const double *xprev,
                    const double *dy, const double *dh_out, const double *dBprev_out, const double *dxprev_out,
                    double *dx, double *dB, double *dC, double *ddt, double *dA, double *dlam, double *dtheta,
                    double *dh0, double *dBprev, double *dxprev)
{
    if (batch < 0 || L < 1 || H <= 0 || P <= 0 || N <= 0 || (N % 2) != 0 || R <= 0)
        return -1;
    if (!x || !B || !C || !dt || !A || !lam || !theta || !dy || (!Bprev) != (!xprev))
        return -1;
    oracle_problem pr = {batch, L, H, P, N, R, x, B, C, dt, A, lam, theta,
                         h0, Bprev, xprev, NULL, NULL, NULL, NULL};
    oracle_grads gr = {dy, dh_out, dBprev_out, dxprev_out, dx, dB, dC, ddt, dA, dlam, dtheta, dh0, dBprev, dxprev};
    for (int b = 0; b < batch; ++b)
        for (int h = 0; h < H; ++h)
            if (scan_sequence_bwd(&pr, &gr, b, h) != 0)
                return -1;
    return 0;
}

typedef struct {
    const oracle_problem *pr;
    int64_t next, stop;        /* sequences [next, stop) handled by this worker */
    int stride;
    int status;
} worker_arg;

static void *worker(void *p)
{
    worker_arg *w = (worker_arg *)p;
    for (int64_t s = w->next; s < w->stop; s += w->stride) {
        const int b = (int)(s / w->pr->H), h = (int)(s % w->pr->H);
        if (scan_sequence(w->pr, b, h) != 0)
            w->status = -1;
    }
    return NULL;
}

/*
 * BC normalisation and bias (linkstar.cloud/article/869, section
 * "架构上的其他改动": "BC归一化" and "BC偏置"): every row of B (or C) -- the N
 * entries of one (token, head, rank) -- is RMS-normalised as in a QK-norm, scaled
 * by a per-head gain and shifted by a per-head, per-rank bias:
 *     v'[n] = v[n] / sqrt(mean_m v[m]^2 + eps) * weight[h][n] + bias[h][r][n].
 * The page gives no formula; this is the plain reading (RMSNorm over the state
 * dimension, then the learnable, data-independent bias).  rows = number of
 * (token, head, rank) rows laid out [...][H][R][N]; weight [H][N] or NULL (1);
 * bias [H][R][N] or NULL (0).  out may equal v.  Returns 0, or -1 on bad
 * arguments.
 */
int oracle_bc_prep(int64_t rows, int H, int R, int N, const double *v, const double *weight,
                   const double *bias, double eps, double *out)
{
    if (rows < 0 || H <= 0 || R <= 0 || N <= 0 || !v || !out)
        return -1;
    for (int64_t i = 0; i < rows; ++i) {
        const int r = (int)(i % R), h = (int)((i / R) % H);
        const double *row = v + i * N;
        double ms = 0.0;
        for (int n = 0; n < N; ++n)
            ms += row[n] * row[n];
        ms /= N;
        const double inv = 1.0 / sqrt(ms + eps);
        double *o = out + i * N;
        for (int n = 0; n < N; ++n) {
            const double g = weight ? weight[(size_t)h * N + n] : 1.0;
            const double c = bias ? bias[((size_t)h * R + r) * N + n] : 0.0;
            o[n] = row[n] * inv * g + c;
        }
    }
    return 0;
}

/*
 * Runs the recurrence for every (b, h) sequence.  Sequences are independent;
 * with nthreads > 1 they are spread over POSIX threads (sequence s goes to
 * thread s mod nthreads).  Returns 0 on success, -1 on bad arguments or out of
 * memory.
 */
int oracle_scan(int batch, int L, int H, int P, int N, int R,
                const double *x, const double *B, const double *C,
                const double *dt, const double *A, const double *lam, const double *theta,
                const double *h0, const double *Bprev, const double *xprev,
                double *y, double *h_out, double *Bprev_out, double *xprev_out,
                int nthreads)
{
    if (batch < 0 || L < 0 || H <= 0 || P <= 0 || N <= 0 || (N % 2) != 0 || R <= 0)
        return -1;
    if (L > 0 && (!x || !B || !C || !dt || !A || !lam || !theta || !y))
        return -1;
    oracle_problem pr = {batch, L, H, P, N, R, x, B, C, dt, A, lam, theta,
                         h0, Bprev, xprev, y, h_out, Bprev_out, xprev_out};
    const int64_t nseq = (int64_t)batch * H;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nseq) nthreads = (int)(nseq > 0 ? nseq : 1);

    worker_arg *args = calloc((size_t)nthreads, sizeof(worker_arg));
    pthread_t *tids = calloc((size_t)nthreads, sizeof(pthread_t));
    if (!args || !tids) { free(args); free(tids); return -1; }
    int status = 0;
    for (int i = 0; i < nthreads; ++i) {
        args[i] = (worker_arg){&pr, i, nseq, nthreads, 0};
    }
    if (nthreads == 1) {
        worker(&args[0]);
    } else {
        int started = 0;
        for (; started < nthreads; ++started)
            if (pthread_create(&tids[started], NULL, worker, &args[started]) != 0)
                break;
        for (int i = 0; i < started; ++i)
            pthread_join(tids[i], NULL);
        for (int i = started; i < nthreads; ++i)   /* threads that could not start: run here */
            worker(&args[i]);
    }
    for (int i = 0; i < nthreads; ++i)
        if (args[i].status) status = -1;
    free(args); free(tids);
    return status;
}
