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
//
// That generic kernel takes any shape.  Two persistent kernels below take the
// common ones and stage whole heads in shared memory with asynchronous bulk
// copies: a streaming FMA kernel (fp32 or bf16 inputs, P in {32, 64, 128}) and
// a tensor-core kernel (bf16 inputs, P = 64, N in {64, 128}) that runs the
// rank-R products and the readout on warp-level MMAs.  The tensor-core kernel
// also serves the pooled step, whose states live in a caller-owned pool
// indexed by a per-row slot table.
#include "m3_internal.cuh"
#include "m3_tc.cuh"

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
              T *__restrict__ Bprev, T *__restrict__ xprev, void *__restrict__ y, int yd, BcNorm bc) {
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
    if (bc.on) {
        // BC normalisation and bias of the staged rows, in place: B, C and the carried B_prev
        // (one warp per row: inverse RMS over the N entries, then gain and bias)
        const int lane = tid & 31, h = (int)(bh % H);
        for (int q = tid >> 5; q < 3 * R; q += kThreads / 32) {
            float *row = (q < R ? sB : (q < 2 * R ? sC : sBp)) + (q % R) * N;
            const float *w = q >= R && q < 2 * R ? bc.wC : bc.wB, *bias = q >= R && q < 2 * R ? bc.bC : bc.bB;
            float ssq = 0.f;
            for (int n = lane; n < N; n += 32) ssq = fmaf(row[n], row[n], ssq);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
            const float inv = 1.f / sqrtf(ssq / (float)N + bc.eps);
            for (int n = lane; n < N; n += 32) row[n] = bc_apply(row[n], inv, w, bias, h, q % R, R, N, n);
        }
        __syncthreads();
    }
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
        store_y(y, bh * RP + i, v, yd);
    }
}

// ---------------------------------------------------------------- streaming kernel
// Persistent variant for the common shapes (P in {32, 64, 128}, N a multiple
// of 16).  Each CTA walks heads blockIdx.x, blockIdx.x + gridDim.x, ... and
// keeps several in flight: one elected thread moves a head's state and token
// inputs into a shared-memory stage with bulk asynchronous copies (completion
// on the stage's mbarrier), the CTA updates the state in place there, and the
// same thread writes the state and the new carry back with bulk copies.  Bytes
// in flight therefore do not depend on registers or occupancy, and two CTAs
// per SM overlap one's barrier with the other's arithmetic.  Thread (kg, cg)
// owns the four columns 4cg..4cg+3 (128-bit shared-memory accesses) of the
// pairs k = kg, kg + NPG, ..., computes their rotation factors itself, and
// reads B, B_prev and C as bf16 pairs shared by its four columns; y is summed
// over the NPG pair groups in shared memory.
constexpr int kStreamThreads = 256;
constexpr uint64_t kStreamWaitNs = 2000000000ull;   // 2 s per mbarrier wait; far above any legal wait

struct StreamLayout {
    uint32_t st, B, C, Bp, x, xp, th, stage;   // byte offsets inside a stage, stage size
    uint32_t red, bar, flag, inv, total;       // offsets after the stages, total bytes
    __host__ __device__ StreamLayout(int N, int P, int R, int e, int nst) {
        auto up = [](uint32_t v) { return (v + 127u) & ~127u; };
        const uint32_t bn = (uint32_t)(R * N * e), xn = (uint32_t)(R * P * e);
        st = 0;
        B = up(st + (uint32_t)(N * P * 4));
        C = up(B + bn);
        Bp = up(C + bn);
        x = up(Bp + bn);
        xp = up(x + xn);
        th = up(xp + xn);
        stage = up(th + (uint32_t)(N / 2 * e));
        red = stage * nst;                                     // y partial sums [NPG][R][P]
        bar = up(red + (uint32_t)(kStreamThreads * 4 * R * 4));
        flag = bar + 8u * nst;
        inv = flag + 16;                                       // BC norm: inverse RMS of 3 R rows
        total = inv + 3u * 8u * 4u;
    }
};

__device__ __forceinline__ void pair_f(const float *q, float &a, float &b) {
    const float2 v = *reinterpret_cast<const float2 *>(q);
    a = v.x;
    b = v.y;
}
__device__ __forceinline__ void pair_f(const __nv_bfloat16 *q, float &a, float &b) {
    const uint32_t v = *reinterpret_cast<const uint32_t *>(q);
    a = __uint_as_float(v << 16);
    b = __uint_as_float(v & 0xFFFF0000u);
}
__device__ __forceinline__ void quad_f(const float *q, float (&o)[4]) {
    const float4 v = *reinterpret_cast<const float4 *>(q);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
}
__device__ __forceinline__ void quad_f(const __nv_bfloat16 *q, float (&o)[4]) {
    const uint2 v = *reinterpret_cast<const uint2 *>(q);
    o[0] = __uint_as_float(v.x << 16); o[1] = __uint_as_float(v.x & 0xFFFF0000u);
    o[2] = __uint_as_float(v.y << 16); o[3] = __uint_as_float(v.y & 0xFFFF0000u);
}
// sin / cos: Cody-Waite reduction by 2 pi (two-constant split) to [-pi, pi],
// then the hardware approximations there
__device__ __forceinline__ void sincos_reduced(float a, float *s, float *c) {
    const float n = rintf(a * 0.15915494309189535f);
    float r = fmaf(-n, 6.28318548202514648f, a);
    r = fmaf(-n, -1.7484555314695172e-7f, r);
    __sincosf(r, s, c);
}

template <typename T, int R>
__global__ void __launch_bounds__(kStreamThreads, 2)
decode_stream_kernel(int nbh, int H, int P, int N, int nst, BcNorm bc, const T *__restrict__ x, const T *__restrict__ Bm,
                     const T *__restrict__ Cm, const T *__restrict__ dtp, const T *__restrict__ Ap,
                     const T *__restrict__ lp, const T *__restrict__ thp, float *__restrict__ hs,
                     T *__restrict__ Bprev, T *__restrict__ xprev, void *__restrict__ y, int yd, unsigned *status) {
    using namespace tc;
    extern __shared__ __align__(128) unsigned char smem_s[];
    unsigned char *sm = smem_s;
    const StreamLayout Lo(N, P, R, (int)sizeof(T), nst);
    const int K = N / 2, tid = threadIdx.x;
    const int NCG = P / 4, NPG = kStreamThreads / NCG, cg = tid % NCG, kg = tid / NCG;
    float *red = reinterpret_cast<float *>(sm + Lo.red);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + Lo.bar);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(sm + Lo.flag);

    const int first = blockIdx.x, step = gridDim.x;
    const int mine = first < nbh ? (nbh - first + step - 1) / step : 0;
    const uint32_t bn = (uint32_t)(R * N * sizeof(T)), xn = (uint32_t)(R * P * sizeof(T));
    const uint32_t hn = (uint32_t)(N * P * 4), tn = (uint32_t)(K * sizeof(T));

    auto issue = [&](int j) {   // head j of this CTA -> stage j % nst (elected thread)
        const size_t bh = (size_t)first + (size_t)j * step;
        unsigned char *sg = sm + (size_t)(j % nst) * Lo.stage;
        uint64_t *bar = full + (j % nst);
        mbar_expect_tx(bar, hn + 3 * bn + 2 * xn + tn);
        bulk_load(sg + Lo.st, hs + bh * N * P, hn, bar);
        bulk_load(sg + Lo.B, Bm + bh * R * N, bn, bar);
        bulk_load(sg + Lo.C, Cm + bh * R * N, bn, bar);
        bulk_load(sg + Lo.Bp, Bprev + bh * R * N, bn, bar);
        bulk_load(sg + Lo.x, x + bh * R * P, xn, bar);
        bulk_load(sg + Lo.xp, xprev + bh * R * P, xn, bar);
        bulk_load(sg + Lo.th, thp + bh * K, tn, bar);
    };

    if (tid == 0) {
        for (int i = 0; i < nst; ++i) mbar_init(full + i, 1);
        mbar_init_fence();
        *abort_flag = 0;
    }
    __syncthreads();
    int issued = 0;
    if (tid == 0)
        for (; issued < nst - 1 && issued < mine; ++issued) issue(issued);

    // per-head scalars one head ahead, in registers (every thread loads the same address)
    float d_n = 0.f, a_n = 0.f, l_n = 0.f;
    if (mine > 0) {
        d_n = to_f(dtp[first]);
        a_n = to_f(Ap[first]);
        l_n = to_f(lp[first]);
    }
    int j = 0;
    for (; j < mine; ++j) {
        const size_t bh = (size_t)first + (size_t)j * step;
        const float d = d_n, av = a_n, l = l_n;
        if (j + 1 < mine) {
            const size_t nb = bh + step;
            d_n = to_f(dtp[nb]);
            a_n = to_f(Ap[nb]);
            l_n = to_f(lp[nb]);
        }
        unsigned char *sg = sm + (size_t)(j % nst) * Lo.stage;
        const bool ok = mbar_wait(full + (j % nst), (uint32_t)((j / nst) & 1), kStreamWaitNs);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) atomicOr(status, kStatusTimeout);
            *abort_flag = 1;
            break;
        }
        const T *sB = reinterpret_cast<const T *>(sg + Lo.B), *sC = reinterpret_cast<const T *>(sg + Lo.C);
        const T *sBp = reinterpret_cast<const T *>(sg + Lo.Bp), *sx = reinterpret_cast<const T *>(sg + Lo.x);
        const T *sxp = reinterpret_cast<const T *>(sg + Lo.xp), *sth = reinterpret_cast<const T *>(sg + Lo.th);
        float *st = reinterpret_cast<float *>(sg + Lo.st);
        float *binv = reinterpret_cast<float *>(sm + Lo.inv);   // [3][R]: B, C, B_prev rows
        const int hh = (int)(bh % H);
        if (bc.on) {
            // inverse RMS of the staged B, C and B_prev rows (one warp per row); the staged rows
            // stay raw (B is stored back as the carry) and are normalised as they are read
            const int lane = tid & 31;
            for (int q = tid >> 5; q < 3 * R; q += kStreamThreads / 32) {
                const T *row = (q < R ? sB : (q < 2 * R ? sC : sBp)) + (q % R) * N;
                float ssq = 0.f;
                for (int n = lane; n < N; n += 32) {
                    const float v = to_f(row[n]);
                    ssq = fmaf(v, v, ssq);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
                if (lane == 0) binv[q] = 1.f / sqrtf(ssq / (float)N + bc.eps);
            }
            __syncthreads();
        }

        const float rho = expf(d * av), left = (1.f - l) * d, right = l * d;
        float xr[R][4], xq[R][4];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            quad_f(sx + r * P + 4 * cg, xr[r]);
            quad_f(sxp + r * P + 4 * cg, xq[r]);
        }
        float yacc[R][4];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) yacc[r][c] = 0.f;
        for (int k = kg; k < K; k += NPG) {
            float sa, ca;
            sincos_reduced(d * to_f(sth[k]), &sa, &ca);
            const float cr = rho * ca, sr = rho * sa;
            float4 *r0 = reinterpret_cast<float4 *>(st + (size_t)(2 * k) * P + 4 * cg);
            float4 *r1 = reinterpret_cast<float4 *>(st + (size_t)(2 * k + 1) * P + 4 * cg);
            const float4 e0 = *r0, e1 = *r1;
            float a0[4] = {e0.x, e0.y, e0.z, e0.w}, a1[4] = {e1.x, e1.y, e1.z, e1.w};
            float u0[4] = {0.f, 0.f, 0.f, 0.f}, u1[4] = {0.f, 0.f, 0.f, 0.f};
            float v0[4] = {0.f, 0.f, 0.f, 0.f}, v1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float b0, b1, q0, q1;
                pair_f(sB + r * N + 2 * k, b0, b1);
                pair_f(sBp + r * N + 2 * k, q0, q1);
                if (bc.on) {
                    b0 = bc_apply(b0, binv[r], bc.wB, bc.bB, hh, r, R, N, 2 * k);
                    b1 = bc_apply(b1, binv[r], bc.wB, bc.bB, hh, r, R, N, 2 * k + 1);
                    q0 = bc_apply(q0, binv[2 * R + r], bc.wB, bc.bB, hh, r, R, N, 2 * k);
                    q1 = bc_apply(q1, binv[2 * R + r], bc.wB, bc.bB, hh, r, R, N, 2 * k + 1);
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    u0[c] = fmaf(q0, xq[r][c], u0[c]);
                    u1[c] = fmaf(q1, xq[r][c], u1[c]);
                    v0[c] = fmaf(b0, xr[r][c], v0[c]);
                    v1[c] = fmaf(b1, xr[r][c], v1[c]);
                }
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float s0 = fmaf(left, u0[c], a0[c]), s1 = fmaf(left, u1[c], a1[c]);
                a0[c] = fmaf(cr, s0, fmaf(-sr, s1, right * v0[c]));
                a1[c] = fmaf(sr, s0, fmaf(cr, s1, right * v1[c]));
            }
            *r0 = make_float4(a0[0], a0[1], a0[2], a0[3]);
            *r1 = make_float4(a1[0], a1[1], a1[2], a1[3]);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float c0, c1;
                pair_f(sC + r * N + 2 * k, c0, c1);
                if (bc.on) {
                    c0 = bc_apply(c0, binv[R + r], bc.wC, bc.bC, hh, r, R, N, 2 * k);
                    c1 = bc_apply(c1, binv[R + r], bc.wC, bc.bC, hh, r, R, N, 2 * k + 1);
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) yacc[r][c] = fmaf(c0, a0[c], fmaf(c1, a1[c], yacc[r][c]));
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
            *reinterpret_cast<float4 *>(red + (kg * R + r) * P + 4 * cg) =
                make_float4(yacc[r][0], yacc[r][1], yacc[r][2], yacc[r][3]);
        fence_proxy_async();   // the state writes above feed the bulk store below
        __syncthreads();
        if (tid == 0) {
            bulk_store(hs + bh * N * P, st, hn);
            bulk_store(Bprev + bh * R * N, sB, bn);     // new carry = this token's (B, x)
            bulk_store(xprev + bh * R * P, sx, xn);
            bulk_commit();
            if (issued < mine) {
                bulk_wait_read<1>();   // the stage about to be refilled has been written out
                issue(issued);
                ++issued;
            }
        }
        for (int i = tid; i < R * P; i += kStreamThreads) {
            float v = 0.f;
            for (int q = 0; q < NPG; ++q) v += red[q * R * P + i];
            store_y(y, bh * R * P + i, v, yd);
        }
    }
    if (tid == 0) {
        if (*abort_flag) {
            // let the copies already issued land before the CTA's shared memory goes away
            for (int i = j; i < issued; ++i) mbar_wait(full + (i % nst), (uint32_t)((i / nst) & 1), kStreamWaitNs);
        }
        bulk_wait<0>();
    }
}

template <typename T>
cudaError_t launch_decode(int batch, int H, int P, int N, int R, const void *x, const void *B,
                          const void *C, const void *dt, const void *A, const void *lam,
                          const void *theta, float *h, void *Bprev, void *xprev, void *y, int yd, const BcNorm &bc,
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
        cudaError_t e = allow_dynamic_smem<decode_kernel<T, PPT>>(smem);                          \
        if (e != cudaSuccess) return e;                                                           \
        kern<<<grid, kThreads, smem, s>>>(H, P, N, R, (const T *)x, (const T *)B, (const T *)C,  \
                                          (const T *)dt, (const T *)A, (const T *)lam,            \
                                          (const T *)theta, h, (T *)Bprev, (T *)xprev, y, yd, bc);   \
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


template <typename T, int R>
cudaError_t launch_stream(int nbh, int H, int P, int N, const void *x, const void *B, const void *C, const void *dt,
                          const void *A, const void *lam, const void *theta, float *h, void *Bprev, void *xprev,
                          void *y, int yd, const BcNorm &bc, cudaStream_t s) {
    const int e = (int)sizeof(T);
    // two CTAs per SM with as many stages as fit (2..6), else one CTA per SM
    int per_sm = 2, nst = 6;
    while (nst > 2 && StreamLayout(N, P, R, e, nst).total > 113u * 1024u) --nst;
    if (StreamLayout(N, P, R, e, nst).total > 113u * 1024u) {
        per_sm = 1;
        nst = 6;
        while (nst > 2 && StreamLayout(N, P, R, e, nst).total > 224u * 1024u) --nst;
    }
    const StreamLayout Lo(N, P, R, e, nst);
    if (Lo.total > 224u * 1024u) return cudaErrorInvalidValue;
    unsigned *status = device_status_word();
    if (!status) return cudaErrorUnknown;
    auto kern = decode_stream_kernel<T, R>;
    cudaError_t err = allow_dynamic_smem<decode_stream_kernel<T, R>>(Lo.total);
    if (err != cudaSuccess) return err;
    const int grid = nbh < per_sm * sm_count() ? nbh : per_sm * sm_count();
    trace_mark(M3_KERNEL_DECODE, s, 0);
    kern<<<grid, kStreamThreads, Lo.total, s>>>(nbh, H, P, N, nst, bc, (const T *)x, (const T *)B, (const T *)C,
                                                (const T *)dt, (const T *)A, (const T *)lam, (const T *)theta, h,
                                                (T *)Bprev, (T *)xprev, y, yd, status);
    trace_mark(M3_KERNEL_DECODE, s, 1);
    count_launch();
    return cudaGetLastError();
}

// Shapes the streaming kernel takes: every per-head block a multiple of 16 bytes
// at 16-byte aligned addresses, and a whole number of state columns per warp.
bool stream_ok(int e, int P, int N, int R, const void *const *ptrs, int nptr) {
    if (P != 32 && P != 64 && P != 128) return false;
    if ((N * e / 2) % 16 != 0 || (R * N * e) % 16 != 0 || (R * P * e) % 16 != 0) return false;
    if (R != 1 && R != 2 && R != 4 && R != 8) return false;
    for (int i = 0; i < nptr; ++i)
        if (reinterpret_cast<uintptr_t>(ptrs[i]) & 15u) return false;
    return true;
}

template <typename T>
cudaError_t stream_dispatch(int nbh, int H, int P, int N, int R, const void *x, const void *B, const void *C,
                            const void *dt, const void *A, const void *lam, const void *theta, float *h,
                            void *Bprev, void *xprev, void *y, int yd, const BcNorm &bc, cudaStream_t s) {
    switch (R) {
        case 1: return launch_stream<T, 1>(nbh, H, P, N, x, B, C, dt, A, lam, theta, h, Bprev, xprev, y, yd, bc, s);
        case 2: return launch_stream<T, 2>(nbh, H, P, N, x, B, C, dt, A, lam, theta, h, Bprev, xprev, y, yd, bc, s);
        case 4: return launch_stream<T, 4>(nbh, H, P, N, x, B, C, dt, A, lam, theta, h, Bprev, xprev, y, yd, bc, s);
        default: return launch_stream<T, 8>(nbh, H, P, N, x, B, C, dt, A, lam, theta, h, Bprev, xprev, y, yd, bc, s);
    }
}


// ---------------------------------------------------------------- tensor-core variant (bf16 inputs, P = 64)
// The same streaming pipeline, with the rank-R products B_prev x_prev^T and B x^T
// and the readout y = C^T h on warp-level bf16 MMAs (fp32 accumulation) instead
// of per-thread FMAs; the rotation factors are computed once per pair into a
// shared table.  A pipeline unit is HPU adjacent heads (their state rows, token
// inputs and carries are contiguous).  Warp w owns the 16 state columns
// p0 = 16 (w % 4) ... p0 + 15 and, with HPU = 2, all N rows of head w / 4 of the
// unit; with HPU = 1, rows (w / 4) N / 2 ... of the one head, the two halves' y
// summed through shared memory.  Per 8-row tile at n0:
//   U = x_prev^T B_prev, V = x^T B    (m16n8k8: M = p, N = n, K = r padded to 8)
// lands in the MMA accumulator layout, in which lane (g, t) holds the columns
// p0 + g, p0 + g + 8 of the rows n0 + 2t, n0 + 2t + 1: exactly one complex pair,
// so the update needs no data exchange.  The new state, split into bf16
// hi + lo parts (error below 2^-16 of |h|), is the A operand of
//   Y^T += h^T C^T     (m16n8k16: M = p, N = r padded to 8, K = n).
// The state is staged by 2-d TMA with the 128-byte swizzle (boxes of 32 columns
// x HPU N rows): the MMA layout's accesses are then free of bank conflicts.  When
// a unit has a multiple of 8 rank rows (HPU R), B, C and B_prev are staged the
// same way (boxes of 64 columns x HPU R rows, no padding needed); otherwise by
// bulk copies in their linear layout, where rank rows N * 2 bytes apart share
// banks.
constexpr int kMmaThreads = 256;
constexpr int kMmaP = 64;

struct MmaLayout {
    uint32_t B, C, Bp, x, xp, stage;     // byte offsets inside a stage (the state at 0), stage size
    uint32_t half;                       // swizzled B, C, B_prev: bytes per 64-column half tile
    uint32_t rot, red, bar, flag, total;
    __host__ __device__ MmaLayout(int N, int R, int hpu, int nst) {
        auto up = [](uint32_t v, uint32_t a) { return (v + a - 1u) & ~(a - 1u); };
        const uint32_t xn = (uint32_t)(hpu * R * kMmaP * 2);
        half = (uint32_t)(hpu * R * 128);   // a multiple of 1024 when the tiles are swizzled
        const uint32_t tile = up(half * (uint32_t)(N / 64), 128u);
        B = (uint32_t)(hpu * N * kMmaP * 4);
        C = B + tile;
        Bp = C + tile;
        x = Bp + tile;
        xp = up(x + xn, 128u);
        stage = up(xp + xn, 1024u);
        rot = stage * nst;                                   // (rho cos, rho sin) per pair of the unit
        red = up(rot + (uint32_t)(hpu * N / 2 * 8), 128u);   // HPU = 1: row group 0's y partials,
        bar = red + (hpu == 1 ? 4u * 32u * 16u : 0u);        //   [4 p-tiles][32 lanes] float4
        flag = bar + 8u * nst;
        total = flag + 16u + 1024u;                          // slack to put the stages on a 1024-byte boundary
    }
};

// Byte offset of (row, col) in a B / C / B_prev tile: 64-column halves of `half` bytes, each
// rows of 128 bytes with the 16-byte chunks of row r XOR-ed by r mod 8 (the TMA 128-byte swizzle)
// (linear layout: row-major [rows][N] bf16)
template <bool SWZ, int N>
__device__ __forceinline__ uint32_t rank_off(uint32_t half, int row, int col) {
    if (!SWZ) return (uint32_t)(row * N + col) * 2u;
    const uint32_t c = (uint32_t)col & 63u, r = (uint32_t)row;
    return ((uint32_t)col >> 6) * half + r * 128u + ((((c >> 3) ^ r) & 7u) << 4) + ((c & 7u) << 1);
}

// POOL: the state rows come from a slot table (pooled decode); otherwise row bh is state bh.
// SWZ: B, C, B_prev through swizzled TMA tiles (a unit of 8k rank rows, one B / C per head).
template <int R, int N, int HPU, bool POOL, bool SWZ>
__global__ void __launch_bounds__(kMmaThreads, 2)
decode_mma_kernel(const __grid_constant__ CUtensorMap hmap, const __grid_constant__ CUtensorMap bmap,
                  const __grid_constant__ CUtensorMap cmap, const __grid_constant__ CUtensorMap bpmap, int nunit,
                  int nst, const int *__restrict__ slot, int pool, int H, int G,
                  const __nv_bfloat16 *__restrict__ x,
                  const __nv_bfloat16 *__restrict__ Bm, const __nv_bfloat16 *__restrict__ Cm,
                  const __nv_bfloat16 *__restrict__ dtp, const __nv_bfloat16 *__restrict__ Ap,
                  const __nv_bfloat16 *__restrict__ lp, const __nv_bfloat16 *__restrict__ thp,
                  __nv_bfloat16 *__restrict__ Bprev, __nv_bfloat16 *__restrict__ xprev, void *__restrict__ y, int yd,
                  unsigned *status) {
    using namespace tc;
    constexpr int P = kMmaP, K = N / 2, NW = HPU == 2 ? N : N / 2, NKS = NW / 16;
    constexpr int NR = HPU * N, KU = HPU * K, KT = kMmaThreads - KU;   // rows, pairs per unit; table threads
    static_assert((HPU == 1 || HPU == 2) && N % 32 == 0 && NR <= 256 && KU <= kMmaThreads && R >= 1 && R <= 8,
                  "shape outside the tensor-core decode");
    static_assert(!SWZ || (HPU * R) % 8 == 0, "swizzled rank tiles need 8k rows");
    extern __shared__ __align__(1024) unsigned char smem_m[];
    unsigned char *sm = smem_m + ((1024u - (smem_u32(smem_m) & 1023u)) & 1023u);
    const MmaLayout Lo(N, R, HPU, nst);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3, pt = warp & 3, grp = warp >> 2;
    const int p0 = 16 * pt, hh = HPU == 2 ? grp : 0, nb0 = HPU == 2 ? 0 : grp * NW;   // head in unit, first row
    const int ti = tid - KT, th_head = ti / K;                           // rotation-table entry of this thread
    float2 *rot = reinterpret_cast<float2 *>(sm + Lo.rot);
    float4 *red = reinterpret_cast<float4 *>(sm + Lo.red);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + Lo.bar);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(sm + Lo.flag);

    const int first = blockIdx.x, step = gridDim.x;
    const int mine = first < nunit ? (nunit - first + step - 1) / step : 0;
    constexpr uint32_t bn = HPU * R * N * 2, xn = HPU * R * P * 2, hn = NR * P * 4;

    // Head of the state (pool) holding token head bh0 of a unit: bh0 itself, or with a slot
    // table (pooled decode), slot[b] * H + h; -1 for an inactive or out-of-range row.  The
    // heads of a unit share b (H is even whenever a unit holds two heads).
    auto state_head = [&](int bh0) -> int {
        if (!POOL) return bh0;
        const int b = bh0 / H, sl = slot[b];
        return sl >= 0 && sl < pool ? sl * H + (bh0 - b * H) : -1;
    };
    auto issue = [&](int j) {   // unit j of this CTA -> stage j % nst (elected thread)
        const int bh0 = (first + j * step) * HPU, sh0 = state_head(bh0);
        unsigned char *sg = sm + (size_t)(j % nst) * Lo.stage;
        uint64_t *bar = full + (j % nst);
        if (sh0 < 0) {   // inactive row: the stage's phase completes with no bytes
            mbar_expect_tx(bar, 0);
            return;
        }
        mbar_expect_tx(bar, hn + 3 * bn + 2 * xn);
        tma_load_2d(sg, &hmap, 0, sh0 * N, bar);
        tma_load_2d(sg + NR * 128, &hmap, 32, sh0 * N, bar);
        if (SWZ) {
#pragma unroll
            for (int hf = 0; hf < N / 64; ++hf) {
                tma_load_2d(sg + Lo.B + hf * Lo.half, &bmap, 64 * hf, bh0 * R, bar);
                tma_load_2d(sg + Lo.C + hf * Lo.half, &cmap, 64 * hf, bh0 * R, bar);
                tma_load_2d(sg + Lo.Bp + hf * Lo.half, &bpmap, 64 * hf, sh0 * R, bar);
            }
        } else {
            if (G == H) {
                bulk_load(sg + Lo.B, Bm + (size_t)bh0 * R * N, bn, bar);
                bulk_load(sg + Lo.C, Cm + (size_t)bh0 * R * N, bn, bar);
            } else {   // grouped B / C: each head's rank rows from its group (head h: group h / (H / G))
#pragma unroll
                for (int hh = 0; hh < HPU; ++hh) {
                    const int bh = bh0 + hh, gi = (bh / H) * G + (bh % H) / (H / G);
                    bulk_load(sg + Lo.B + hh * R * N * 2, Bm + (size_t)gi * R * N, R * N * 2, bar);
                    bulk_load(sg + Lo.C + hh * R * N * 2, Cm + (size_t)gi * R * N, R * N * 2, bar);
                }
            }
            bulk_load(sg + Lo.Bp, Bprev + (size_t)sh0 * R * N, bn, bar);
        }
        bulk_load(sg + Lo.x, x + (size_t)bh0 * R * P, xn, bar);
        bulk_load(sg + Lo.xp, xprev + (size_t)sh0 * R * P, xn, bar);
    };

    // Programmatic dependent launch: the next step's grid may be scheduled now (its CTAs take SMs as
    // these leave and set up while the last units drain); this grid touches no global memory before
    // the grid it depends on has completed and its writes are visible
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (tid == 0) {
        tma_prefetch_desc(&hmap);
        if (SWZ) {
            tma_prefetch_desc(&bmap);
            tma_prefetch_desc(&cmap);
            tma_prefetch_desc(&bpmap);
        }
        for (int i = 0; i < nst; ++i) mbar_init(full + i, 1);
        mbar_init_fence();
        *abort_flag = 0;
    }
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    int issued = 0;
    if (tid == 0)
        for (; issued < nst - 1 && issued < mine; ++issued) issue(issued);

    // swizzled byte offsets of this lane's four state elements, relative to unit row
    // hh N + n0 + 2t (n0 a multiple of 8): columns p0 + g, p0 + g + 8 of that row and the next
    const uint32_t lb = (uint32_t)(pt >> 1) * NR * 128u + ((uint32_t)(g & 3) << 2);
    const uint32_t c0 = 4u * (uint32_t)(pt & 1) + (uint32_t)(g >> 2), c1 = c0 + 2u;
    const uint32_t o00 = lb + ((c0 ^ (2u * t)) << 4), o01 = lb + 128u + ((c0 ^ (2u * t + 1u)) << 4);
    const uint32_t o10 = lb + ((c1 ^ (2u * t)) << 4), o11 = lb + 128u + ((c1 ^ (2u * t + 1u)) << 4);
    const bool rlane = 2 * t < R;   // lanes holding rank rows 2t (and 2t + 1 when R > 1)

    // per-head scalars of this warp's head and of this thread's table entry, one unit ahead
    float d_n = 0.f, l_n = 0.f, dq_n = 0.f, aq_n = 0.f, th_n = 0.f;
    auto prefetch = [&](int unit) {
        const int bh0 = unit * HPU;
        d_n = to_f(dtp[bh0 + hh]);
        l_n = to_f(lp[bh0 + hh]);
        if (ti >= 0) {
            dq_n = to_f(dtp[bh0 + th_head]);
            aq_n = to_f(Ap[bh0 + th_head]);
            th_n = to_f(thp[(size_t)bh0 * K + ti]);
        }
    };
    if (mine > 0) prefetch(first);
    int j = 0;
    for (; j < mine; ++j) {
        const int bh0 = (first + j * step) * HPU;
        const float d = d_n, l = l_n, dq = dq_n, aq = aq_n, th = th_n;
        if (j + 1 < mine) prefetch(first + (j + 1) * step);
        // the last warps fill the rotation table (warp 0 also issues the copies); it is read after
        // the barrier below, and its last reads came before the previous one
        if (ti >= 0) {
            const float rho = expf(dq * aq);
            float sa, ca;
            sincos_reduced(dq * th, &sa, &ca);
            rot[ti] = make_float2(rho * ca, rho * sa);
        }
        unsigned char *sg = sm + (size_t)(j % nst) * Lo.stage;
        const bool ok = mbar_wait(full + (j % nst), (uint32_t)((j / nst) & 1), kStreamWaitNs);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) atomicOr(status, kStatusTimeout);
            *abort_flag = 1;
            break;
        }
        const int sh0 = state_head(bh0);   // < 0: inactive row, nothing to read or write
        if (POOL && tid == 0 && sh0 < 0 && slot[bh0 / H] >= pool) atomicOr(status, kStatusBadIndex);
        float yacc[4] = {0.f, 0.f, 0.f, 0.f};
        // y[r][p] for r = 2t, 2t + 1 and p = p0 + g, p0 + g + 8
        const size_t yo = (size_t)(bh0 + hh) * R * P + 2 * t * P + p0 + g;
        if (sh0 >= 0) {
            const unsigned char *sB = sg + Lo.B, *sBp = sg + Lo.Bp, *sC = sg + Lo.C;
            const unsigned short *sx = reinterpret_cast<const unsigned short *>(sg + Lo.x) + hh * R * P;
            const unsigned short *sxp = reinterpret_cast<const unsigned short *>(sg + Lo.xp) + hh * R * P;
            const float2 *hrot = rot + hh * K;
            unsigned char *hst = sg + (uint32_t)(hh * N) * 128u;
            const float left = (1.f - l) * d, right = l * d;

            // A operands of the rank-R products: x^T rows p0 + g, p0 + g + 8, rank columns 2t, 2t + 1
            uint32_t ax0 = 0, ax1 = 0, aq0 = 0, aq1 = 0;
            if (rlane) {
                const int r0 = 2 * t * P + p0 + g;
                ax0 = sx[r0];
                ax1 = sx[r0 + 8];
                aq0 = sxp[r0];
                aq1 = sxp[r0 + 8];
                if (R > 1) {
                    ax0 |= (uint32_t)sx[r0 + P] << 16;
                    ax1 |= (uint32_t)sx[r0 + P + 8] << 16;
                    aq0 |= (uint32_t)sxp[r0 + P] << 16;
                    aq1 |= (uint32_t)sxp[r0 + P + 8] << 16;
                }
            }
#pragma unroll
            for (int ks = 0; ks < NKS; ++ks) {
                uint32_t ahi[4], alo[4];
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int n0 = nb0 + 16 * ks + 8 * hf;
                    uint32_t bb = 0, bq = 0;   // B operands: rank rows 2t, 2t + 1 of state row n0 + g
                    if (rlane) {
                        const int row = hh * R + 2 * t;
                        const uint32_t o0 = rank_off<SWZ, N>(Lo.half, row, n0 + g), o1 = rank_off<SWZ, N>(Lo.half, row + 1, n0 + g);
                        bb = *reinterpret_cast<const unsigned short *>(sB + o0);
                        bq = *reinterpret_cast<const unsigned short *>(sBp + o0);
                        if (R > 1) {
                            bb |= (uint32_t)*reinterpret_cast<const unsigned short *>(sB + o1) << 16;
                            bq |= (uint32_t)*reinterpret_cast<const unsigned short *>(sBp + o1) << 16;
                        }
                    }
                    float u[4] = {0.f, 0.f, 0.f, 0.f}, v[4] = {0.f, 0.f, 0.f, 0.f};
                    mma_m16n8k8(u, aq0, aq1, bq);
                    mma_m16n8k8(v, ax0, ax1, bb);
                    const float2 rt = hrot[n0 / 2 + t];
                    unsigned char *rb = hst + (uint32_t)(n0 + 2 * t) * 128u;
                    float *q00 = reinterpret_cast<float *>(rb + o00), *q01 = reinterpret_cast<float *>(rb + o01);
                    float *q10 = reinterpret_cast<float *>(rb + o10), *q11 = reinterpret_cast<float *>(rb + o11);
                    float s0 = fmaf(left, u[0], *q00), s1 = fmaf(left, u[1], *q01);
                    const float n00 = fmaf(rt.x, s0, fmaf(-rt.y, s1, right * v[0]));
                    const float n01 = fmaf(rt.y, s0, fmaf(rt.x, s1, right * v[1]));
                    s0 = fmaf(left, u[2], *q10);
                    s1 = fmaf(left, u[3], *q11);
                    const float n10 = fmaf(rt.x, s0, fmaf(-rt.y, s1, right * v[2]));
                    const float n11 = fmaf(rt.y, s0, fmaf(rt.x, s1, right * v[3]));
                    *q00 = n00;
                    *q01 = n01;
                    *q10 = n10;
                    *q11 = n11;
                    split2(n00, n01, ahi[2 * hf], alo[2 * hf]);           // row p0 + g
                    split2(n10, n11, ahi[2 * hf + 1], alo[2 * hf + 1]);   // row p0 + g + 8
                }
                uint32_t b0 = 0, b1 = 0;   // C^T: state rows 2t, 2t + 1 (+ 8) of this K step, rank column g
                if (g < R) {
                    const int row = hh * R + g, c0 = nb0 + 16 * ks + 2 * t;
                    b0 = *reinterpret_cast<const uint32_t *>(sC + rank_off<SWZ, N>(Lo.half, row, c0));
                    b1 = *reinterpret_cast<const uint32_t *>(sC + rank_off<SWZ, N>(Lo.half, row, c0 + 8));
                }
                mma_m16n8k16(yacc, ahi, b0, b1);
                mma_m16n8k16(yacc, alo, b0, b1);
            }
            if (HPU == 2 && rlane) {
                store_y(y, yo, yacc[0], yd);
                store_y(y, yo + 8, yacc[2], yd);
                if (R > 1) {
                    store_y(y, yo + P, yacc[1], yd);
                    store_y(y, yo + P + 8, yacc[3], yd);
                }
            }
            if (HPU == 1 && grp == 0) red[pt * 32 + lane] = make_float4(yacc[0], yacc[1], yacc[2], yacc[3]);
        }
        fence_proxy_async();   // the state writes above feed the tensor stores below
        __syncthreads();
        if (tid == 0) {
            if (sh0 >= 0) {
                tma_store_2d(&hmap, sg, 0, sh0 * N);
                tma_store_2d(&hmap, sg + NR * 128, 32, sh0 * N);
                if (SWZ) {   // new carry = this token's (B, x)
#pragma unroll
                    for (int hf = 0; hf < N / 64; ++hf)
                        tma_store_2d(&bpmap, sg + Lo.B + hf * Lo.half, 64 * hf, sh0 * R);
                } else {
                    bulk_store(Bprev + (size_t)sh0 * R * N, sg + Lo.B, bn);
                }
                bulk_store(xprev + (size_t)sh0 * R * P, sg + Lo.x, xn);
            }
            bulk_commit();
            if (issued < mine) {
                bulk_wait_read<1>();   // the stage about to be refilled has been written out
                issue(issued);
                ++issued;
            }
        }
        if (sh0 >= 0 && HPU == 1 && grp == 1 && rlane) {
            const float4 o = red[pt * 32 + lane];
            store_y(y, yo, yacc[0] + o.x, yd);
            store_y(y, yo + 8, yacc[2] + o.z, yd);
            if (R > 1) {
                store_y(y, yo + P, yacc[1] + o.y, yd);
                store_y(y, yo + P + 8, yacc[3] + o.w, yd);
            }
        }
    }
    if (tid == 0) {
        if (*abort_flag) {
            for (int i = j; i < issued; ++i) mbar_wait(full + (i % nst), (uint32_t)((i / nst) & 1), kStreamWaitNs);
        }
        bulk_wait<0>();
    }
}

// 2-d map over a [rows][cols] bf16 array (B, C or B_prev as [nbh * R][N]); box = 64 columns x
// box_rows, 128-byte swizzle
bool map_rank(CUtensorMap *m, const void *base, long long rows, int cols, int box_rows) {
    tc::EncodeFn enc = tc::encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-d map over the fp32 state viewed as [nbh * N rows][64 columns]; box = 32 columns x box_rows,
// 128-byte swizzle
bool map_state(CUtensorMap *m, float *h, long long rows, int box_rows) {
    tc::EncodeFn enc = tc::encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)kMmaP, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kMmaP * 4};
    const cuuint32_t box[2] = {32, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, h, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// nbh: token heads (batch * H); with a slot table the state arrays hold pool_heads heads; B and C
// hold G groups of heads
template <int R, int N, int HPU, bool kSwz>
cudaError_t launch_mma_t(int nbh, int H, int G, const int *slot, int pool, const void *x, const void *B,
                         const void *C, const void *dt, const void *A, const void *lam, const void *theta, float *h,
                         void *Bprev, void *xprev, void *y, int yd, cudaStream_t s) {
    const long long pool_heads = slot ? (long long)pool * H : (long long)nbh;
    // the state and carry maps depend only on (h, B_prev, shape); a decode loop reuses one state
    struct MapCache {
        const float *h = nullptr;
        const void *bp = nullptr;
        long long rows = 0;
        int n = 0, r = 0, hpu = 0;
        CUtensorMap hmap, bpmap;
    };
    thread_local MapCache cache;
    const long long rows = pool_heads * N;
    if (cache.h != h || cache.bp != Bprev || cache.rows != rows || cache.n != N || cache.r != R || cache.hpu != HPU) {
        cache.h = nullptr;
        if (!map_state(&cache.hmap, h, rows, HPU * N)) return cudaErrorInvalidValue;
        if (kSwz && !map_rank(&cache.bpmap, Bprev, pool_heads * R, N, HPU * R)) return cudaErrorInvalidValue;
        cache.h = h;
        cache.bp = Bprev;
        cache.rows = rows;
        cache.n = N;
        cache.r = R;
        cache.hpu = HPU;
    }
    CUtensorMap bmap = cache.hmap, cmap = cache.hmap;   // unused unless swizzled
    if (kSwz && (!map_rank(&bmap, B, (long long)nbh * R, N, HPU * R) ||
                 !map_rank(&cmap, C, (long long)nbh * R, N, HPU * R)))
        return cudaErrorInvalidValue;
    if (!kSwz) cache.bpmap = cache.hmap;
    // two CTAs per SM with as many stages as fit (2..6), else one CTA per SM
    int per_sm = 2, nst = 6;
    while (nst > 2 && MmaLayout(N, R, HPU, nst).total > 113u * 1024u) --nst;
    if (MmaLayout(N, R, HPU, nst).total > 113u * 1024u) {
        per_sm = 1;
        nst = 6;
        while (nst > 2 && MmaLayout(N, R, HPU, nst).total > 224u * 1024u) --nst;
    }
    const MmaLayout Lo(N, R, HPU, nst);
    if (Lo.total > 224u * 1024u) return cudaErrorInvalidValue;
    unsigned *status = device_status_word();
    if (!status) return cudaErrorUnknown;
    auto kern = slot ? decode_mma_kernel<R, N, HPU, true, kSwz> : decode_mma_kernel<R, N, HPU, false, kSwz>;
    cudaError_t err = slot ? allow_dynamic_smem<decode_mma_kernel<R, N, HPU, true, kSwz>>(Lo.total)
                           : allow_dynamic_smem<decode_mma_kernel<R, N, HPU, false, kSwz>>(Lo.total);
    if (err != cudaSuccess) return err;
    const int nunit = nbh / HPU;
    const int grid = nunit < per_sm * sm_count() ? nunit : per_sm * sm_count();
    using bf = __nv_bfloat16;
    // launched as a programmatic dependent of the kernel before it in the stream (consecutive decode
    // steps overlap one's launch and set-up with the other's tail; see the kernel's entry)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kMmaThreads);
    cfg.dynamicSmemBytes = Lo.total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    trace_mark(M3_KERNEL_DECODE, s, 0);
    err = cudaLaunchKernelEx(&cfg, kern, cache.hmap, bmap, cmap, cache.bpmap, nunit, nst, slot, pool, H, G,
                             (const bf *)x, (const bf *)B, (const bf *)C, (const bf *)dt, (const bf *)A,
                             (const bf *)lam, (const bf *)theta, (bf *)Bprev, (bf *)xprev, y, yd, status);
    trace_mark(M3_KERNEL_DECODE, s, 1);
    if (err != cudaSuccess) return err;
    count_launch();
    return cudaGetLastError();
}

template <int R, int N, int HPU>
cudaError_t launch_mma(int nbh, int H, int G, const int *slot, int pool, const void *x, const void *B, const void *C,
                       const void *dt, const void *A, const void *lam, const void *theta, float *h, void *Bprev,
                       void *xprev, void *y, int yd, cudaStream_t s) {
    if constexpr ((HPU * R) % 8 == 0) {
        if (G == H)
            return launch_mma_t<R, N, HPU, true>(nbh, H, G, slot, pool, x, B, C, dt, A, lam, theta, h, Bprev, xprev,
                                                 y, yd, s);
    }
    return launch_mma_t<R, N, HPU, false>(nbh, H, G, slot, pool, x, B, C, dt, A, lam, theta, h, Bprev, xprev, y, yd, s);
}

// The tensor-core variant takes bf16 inputs with P = 64, N in {64, 128}, R in {1, 2, 4, 8},
// the streaming kernel's alignment, and state row indices within int range.  (For R = 1 the
// padded rank products waste tensor work, but that work is far from binding and the per-pair
// FMAs it replaces are not.)
bool mma_ok(int dtype, int P, int N, int R, long long nbh) {
    return dtype == M3_BF16 && P == kMmaP && (N == 64 || N == 128) && (R == 1 || R == 2 || R == 4 || R == 8) &&
           nbh * N < (1ll << 31);
}

// N = 64 pairs adjacent heads into one unit when the head count is even (with a slot table:
// when H is even, so that the two heads share a batch row and thus a pool slot).
cudaError_t mma_dispatch(int nbh, int H, int G, const int *slot, int pool, int N, int R, const void *x,
                         const void *B, const void *C, const void *dt, const void *A, const void *lam,
                         const void *theta, float *h, void *Bprev, void *xprev, void *y, int yd, cudaStream_t s) {
    const bool pair = N == 64 && (slot || G != H ? H % 2 == 0 : nbh % 2 == 0);
#define M3_MMA(RR, NN, HH)                                                                                         \
    if (R == RR && N == NN && (HH == 2) == pair)                                                                 \
    return launch_mma<RR, NN, HH>(nbh, H, G, slot, pool, x, B, C, dt, A, lam, theta, h, Bprev, xprev, y, yd, s)
    M3_MMA(1, 64, 2);
    M3_MMA(2, 64, 2);
    M3_MMA(4, 64, 2);
    M3_MMA(8, 64, 2);
    M3_MMA(1, 64, 1);
    M3_MMA(2, 64, 1);
    M3_MMA(4, 64, 1);
    M3_MMA(8, 64, 1);
    M3_MMA(1, 128, 1);
    M3_MMA(2, 128, 1);
    M3_MMA(4, 128, 1);
    M3_MMA(8, 128, 1);
#undef M3_MMA
    return cudaErrorInvalidValue;
}

}  // namespace

std::atomic<int> g_last_decode_variant{-1};

cudaError_t decode_step(int dtype, int yd, int batch, int H, int G, int P, int N, int R, const void *x,
                        const void *B, const void *C, const void *dt, const void *A,
                        const void *lam, const void *theta, float *h, void *Bprev, void *xprev,
                        void *y, cudaStream_t s, const BcNorm *bcp) {
    const int e = dtype == M3_F32 ? 4 : 2;
    const void *ptrs[] = {x, B, C, theta, h, Bprev, xprev};
    const int nbh = batch * H;
    const BcNorm bc = bcp ? *bcp : BcNorm{};
    if (G != H) {   // grouped B / C: tensor-core kernel only (the caller checked decode_tc_ok, and bc is off)
        if (nbh == 0) return cudaSuccess;
        g_last_decode_variant.store(M3_DECODE_TENSOR, std::memory_order_relaxed);
        return mma_dispatch(nbh, H, G, nullptr, batch, N, R, x, B, C, dt, A, lam, theta, h, Bprev, xprev, y, yd, s);
    }
    if (nbh > 0 && stream_ok(e, P, N, R, ptrs, 7)) {
        if (!bc.on && mma_ok(dtype, P, N, R, nbh)) {
            g_last_decode_variant.store(M3_DECODE_TENSOR, std::memory_order_relaxed);
            return mma_dispatch(nbh, H, H, nullptr, batch, N, R, x, B, C, dt, A, lam, theta, h, Bprev, xprev, y, yd, s);
        }
        g_last_decode_variant.store(M3_DECODE_STREAM, std::memory_order_relaxed);
        if (dtype == M3_F32)
            return stream_dispatch<float>(nbh, H, P, N, R, x, B, C, dt, A, lam, theta, h, Bprev, xprev, y, yd, bc, s);
        return stream_dispatch<__nv_bfloat16>(nbh, H, P, N, R, x, B, C, dt, A, lam, theta, h, Bprev, xprev, y, yd, bc,
                                              s);
    }
    g_last_decode_variant.store(M3_DECODE_GENERIC, std::memory_order_relaxed);
    if (dtype == M3_F32)
        return launch_decode<float>(batch, H, P, N, R, x, B, C, dt, A, lam, theta, h, Bprev, xprev, y, yd, bc, s);
    return launch_decode<__nv_bfloat16>(batch, H, P, N, R, x, B, C, dt, A, lam, theta, h, Bprev,
                                        xprev, y, yd, bc, s);
}

bool decode_tc_ok(int dtype, int P, int N, int R, long long heads, const void *const *ptrs, int nptr) {
    return mma_ok(dtype, P, N, R, heads) && stream_ok(2, P, N, R, ptrs, nptr);
}

cudaError_t decode_step_pooled(int yd, int batch, int H, int G, int P, int N, int R, const int *slot, int pool,
                               const void *x, const void *B, const void *C, const void *dt, const void *A,
                               const void *lam, const void *theta, float *h, void *Bprev, void *xprev, void *y,
                               cudaStream_t s) {
    (void)P;
    if (batch == 0) return cudaSuccess;
    g_last_decode_variant.store(M3_DECODE_TENSOR, std::memory_order_relaxed);
    return mma_dispatch(batch * H, H, G, slot, pool, N, R, x, B, C, dt, A, lam, theta, h, Bprev, xprev, y, yd, s);
}

}  // namespace m3

extern "C" int mamba3_decode_last_variant(void) {
    return m3::g_last_decode_variant.load(std::memory_order_relaxed);
}
