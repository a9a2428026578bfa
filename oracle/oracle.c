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
