// One-token recurrent step of the Mamba-3 recurrence, state updated in place.
//
// For every (b, h) and complex pair k = (2k, 2k+1) of the N x P fp32 state
// (linkstar.cloud/article/869, sections "第一刀" and "第二刀"):
//   h   <- rho R(dt theta_k) [h + (1 - lambda) dt B_prev x_prev^T] + lambda dt B x^T,
//   rho  = exp(dt A),   R(a) = [[cos a, -sin a], [sin a, cos a]],
//   y    = C^T h   (R x P, fp32),   carry <- (B, x).
// B x^T is the rank-R product of B (N x R) and x^T (R x P) ("第三刀").
//
// The state streams through once (read + write, 8 N P bytes per head); it is
// the whole cost.  One CTA owns one head: 128 threads, each a 4-column slice of
// P (one float4 per state row) and a strided set of pairs, with all of its
// state loads issued before any arithmetic so that many bytes are in flight.
// The per-token inputs (B, C, carry, x) are staged in shared memory as fp32.
// y is reduced over N inside the thread, then across threads in shared memory.
#include "m3_internal.cuh"

namespace m3 {
namespace {

constexpr int kThreads = 128;

template <typename T>
__device__ __forceinline__ void load_f(float *dst, const T *src, int n, int tid) {
    for (int i = tid; i < n; i += kThreads) dst[i] = to_f(src[i]);
}

// PPT = pairs held in registers per pass.
template <typename T, int PPT>
__global__ void __launch_bounds__(kThreads)
decode_kernel(int H, int P, int N, int R, const T *__restrict__ x, const T *__restrict__ Bm,
              const T *__restrict__ Cm, const T *__restrict__ dtp, const T *__restrict__ Ap,
              const T *__restrict__ lp, const T *__restrict__ thp, float *__restrict__ hs,
              T *__restrict__ Bprev, T *__restrict__ xprev, float *__restrict__ y) {
    extern __shared__ float sm[];
    const int K = N / 2, RN = R * N, RP = R * P;
    float *sB = sm, *sC = sB + RN, *sBp = sC + RN, *sx = sBp + RN, *sxp = sx + RP;
    float *sc = sxp + RP, *ss = sc + K, *red = ss + K;   // red: [KG][R][P]

    const int tid = threadIdx.x;
    const size_t bh = blockIdx.x;
    const int NCG = P / 4;               // float4 column groups
    const int KG = kThreads / NCG;       // pair groups
    const int cg = tid % NCG, kg = tid / NCG;
    const bool active = kg < KG;

    // ---- stage the token's inputs (the carry is read before it is overwritten)
    load_f(sB, Bm + bh * RN, RN, tid);
    load_f(sC, Cm + bh * RN, RN, tid);
    load_f(sBp, Bprev + bh * RN, RN, tid);
    load_f(sx, x + bh * RP, RP, tid);
    load_f(sxp, xprev + bh * RP, RP, tid);
    const float d = to_f(dtp[bh]), rho = expf(d * to_f(Ap[bh])), l = to_f(lp[bh]);
    for (int k = tid; k < K; k += kThreads) {
        float s, c;
        sincosf(d * to_f(thp[bh * K + k]), &s, &c);
        sc[k] = c;
        ss[k] = s;
    }
    __syncthreads();
    // new carry = this token's (B, x); every read of the old carry is above
    for (int i = tid; i < RN; i += kThreads) Bprev[bh * RN + i] = Bm[bh * RN + i];
    for (int i = tid; i < RP; i += kThreads) xprev[bh * RP + i] = x[bh * RP + i];

    const float left = (1.f - l) * d, right = l * d;
    float yacc[8][4];   // R <= 8
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) yacc[r][c] = 0.f;

    if (active) {
        const int p0 = cg * 4;
        float4 *h4 = reinterpret_cast<float4 *>(hs + bh * (size_t)N * P);
        const int P4 = P / 4;
        for (int kb = kg; kb < K; kb += KG * PPT) {
            float4 h0[PPT], h1[PPT];
#pragma unroll
            for (int j = 0; j < PPT; ++j) {
                const int k = kb + j * KG;
                if (k < K) {
                    h0[j] = __ldcs(h4 + (size_t)(2 * k) * P4 + cg);
                    h1[j] = __ldcs(h4 + (size_t)(2 * k + 1) * P4 + cg);
                }
            }
#pragma unroll
            for (int j = 0; j < PPT; ++j) {
                const int k = kb + j * KG;
                if (k >= K) break;
                float a0[4] = {h0[j].x, h0[j].y, h0[j].z, h0[j].w};
                float a1[4] = {h1[j].x, h1[j].y, h1[j].z, h1[j].w};
                float u0[4] = {0, 0, 0, 0}, u1[4] = {0, 0, 0, 0}, v0[4] = {0, 0, 0, 0}, v1[4] = {0, 0, 0, 0};
                for (int r = 0; r < R; ++r) {
                    const float bp0 = sBp[r * N + 2 * k], bp1 = sBp[r * N + 2 * k + 1];
                    const float b0 = sB[r * N + 2 * k], b1 = sB[r * N + 2 * k + 1];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const float xp = sxp[r * P + p0 + c], xc = sx[r * P + p0 + c];
                        u0[c] += bp0 * xp;
                        u1[c] += bp1 * xp;
                        v0[c] += b0 * xc;
                        v1[c] += b1 * xc;
                    }
                }
                const float cr = rho * sc[k], sr = rho * ss[k];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float s0 = a0[c] + left * u0[c], s1 = a1[c] + left * u1[c];
                    a0[c] = cr * s0 - sr * s1 + right * v0[c];
                    a1[c] = sr * s0 + cr * s1 + right * v1[c];
                }
                __stcs(h4 + (size_t)(2 * k) * P4 + cg, make_float4(a0[0], a0[1], a0[2], a0[3]));
                __stcs(h4 + (size_t)(2 * k + 1) * P4 + cg, make_float4(a1[0], a1[1], a1[2], a1[3]));
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    if (r < R) {
                        const float c0 = sC[r * N + 2 * k], c1 = sC[r * N + 2 * k + 1];
#pragma unroll
                        for (int c = 0; c < 4; ++c) yacc[r][c] += c0 * a0[c] + c1 * a1[c];
                    }
                }
            }
        }
        // ---- reduce y over pair groups
#pragma unroll
        for (int r = 0; r < 8; ++r)
            if (r < R)
#pragma unroll
                for (int c = 0; c < 4; ++c) red[(kg * R + r) * P + p0 + c] = yacc[r][c];
    }
    __syncthreads();
    for (int i = tid; i < RP; i += kThreads) {
        float v = 0.f;
        for (int g = 0; g < KG; ++g) v += red[g * RP + i];
        y[bh * RP + i] = v;
    }
}

template <typename T>
cudaError_t launch_decode(int batch, int H, int P, int N, int R, const void *x, const void *B,
                          const void *C, const void *dt, const void *A, const void *lam,
                          const void *theta, float *h, void *Bprev, void *xprev, void *y,
                          cudaStream_t s) {
    const int NCG = P / 4, KG = kThreads / NCG, K = N / 2;
    const size_t smem = sizeof(float) * (3 * (size_t)R * N + 2 * (size_t)R * P + 2 * (size_t)K +
                                         (size_t)KG * R * P);
    const int pairs_per_thread = (K + KG - 1) / KG;
    const dim3 grid((unsigned)((size_t)batch * H));
    if (grid.x == 0) return cudaSuccess;
#define M3_DECODE_LAUNCH(PPT)                                                                     \
    do {                                                                                          \
        auto kern = decode_kernel<T, PPT>;                                                        \
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,   \
                                             (int)smem);                                          \
        if (e != cudaSuccess) return e;                                                           \
        kern<<<grid, kThreads, smem, s>>>(H, P, N, R, (const T *)x, (const T *)B, (const T *)C,  \
                                          (const T *)dt, (const T *)A, (const T *)lam,            \
                                          (const T *)theta, h, (T *)Bprev, (T *)xprev, (float *)y);   \
    } while (0)
    trace_mark(M3_KERNEL_DECODE, s, 0);
    if (pairs_per_thread <= 4)
        M3_DECODE_LAUNCH(4);
    else
        M3_DECODE_LAUNCH(8);
#undef M3_DECODE_LAUNCH
    trace_mark(M3_KERNEL_DECODE, s, 1);
    count_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t decode_step(int dtype, int batch, int H, int P, int N, int R, const void *x,
                        const void *B, const void *C, const void *dt, const void *A,
                        const void *lam, const void *theta, float *h, void *Bprev, void *xprev,
                        void *y, cudaStream_t s) {
    if (dtype == M3_F32)
        return launch_decode<float>(batch, H, P, N, R, x, B, C, dt, A, lam, theta, h, Bprev, xprev, y, s);
    return launch_decode<__nv_bfloat16>(batch, H, P, N, R, x, B, C, dt, A, lam, theta, h, Bprev,
                                        xprev, y, s);
}

}  // namespace m3
