// Backward pass of the chunked Mamba-3 recurrence (reverse mode, for training; linkstar.cloud
// article 869, section "训练怎么办": the model is trained through the chunked, matrix form of the
// recurrence, and its gradients follow that form).
//
// One CTA per (b, h) sequence, fp32 arithmetic on CUDA cores.
//   Pass 1 walks the chunks forward and stores the state H'_c entering every chunk (the checkpoints;
//   H'_0 includes the carry's left-endpoint term).
//   Pass 2 walks them backward carrying D = dLoss/dH' (true frame).  Per chunk, in its rotated frame
//   (B~ = R(-phi) B, C~ = R(-phi) C, chunk-local cumulative sums cA and phi):
//     forward:  y_t = sum_{j<=t} M_tj (C~_t . B~_j) x_j + e^{cA_t} C~_t H'_c
//               H'_{c+1} = R(phi_e) [e^{cA_e} H'_c + sum_j s_j B~_j x_j^T],  s_j = e^{cA_e - cA_j} w_j
//               M_tj = e^{cA_t - cA_j} w_j (j < t), g_t = lambda_t dt_t (j = t)
//     backward, with D~ = R(-phi_e) D, S = C~ B~^T, Z = dY X^T (rows (t, r)):
//               dX  = (M o S)^T dY + diag(s) B~ D~
//               dB~ = (M o Z)^T C~ + diag(s) X D~^T
//               dC~ = (M o Z) B~ + diag(e^{cA}) dY H'_c^T
//               dM  = S o Z (summed over rank pairs);  ds_j = x_j . (B~_j D~)
//               dcA_t, dw_j, dg_t from dM, ds and the inter-chunk terms; dphi from dB~, dC~ and the
//               turn R(phi_e) of the state; then reverse cumulative sums give d(dt A), d(dt theta)
//               D <- e^{cA_e} D~ + C~^T diag(e^{cA}) dY
//   and finally dh0 = D, with the carry's gradients from H'_0's left-endpoint term.
// w_j carries the next token's left-endpoint weight (1 - lambda_{j+1}) dt_{j+1}; the gradient of
// that term reaches token j + 1's lambda and dt, which for the chunk's last token lies in the chunk
// processed just before (a read-modify-write of its two gradients).
//
// Layout.  The contractions run as register tiles: a thread forms a 1 x 4 or 2 x 4 block of the
// output from one broadcast scalar of the left operand and one float4 of the right one per step, so
// every right operand is stored with the output's column index contiguous (B~ and its transpose, x
// and its transpose, D~ and its transpose; the checkpoints are kept transposed, [P][N]).  Tiles are
// zero-padded to whole float4 columns, and their rows padded by 4 floats against bank conflicts.
// The raw rows of the next chunk (B, C, x, theta, dy, as stored) are copied into a staging area by
// asynchronous 16-byte copies while the current chunk is processed, and its per-token scalars are
// fetched into registers; the state checkpoint of a chunk is copied in while its inputs are turned.
#include "m3_internal.cuh"

namespace m3 {
namespace {

constexpr int kBwdThreads = 512;
constexpr int kBwdWarps = kBwdThreads / 32;

__host__ __device__ constexpr int rup4(int v) { return (v + 3) & ~3; }

// Shared-memory carve-up (floats).  Tiles first (each a multiple of 4 floats, so every one starts on
// a 16-byte boundary), then the per-token vectors.
struct BwdSmem {
    int Q, R, N, P, K, QR, NP, PP, QRP, N4, P4, QR4, QS, QP1;
    size_t rowB, rowX, rowT, rowY;   // bytes per token of the raw B (and C), x, theta, dy rows
    size_t oD, oDtT, oH, oB, oC, oBT, oX, oXT, oY, oYe, oS, oZ, oT1, oT2, odM;
    size_t oStB, oStC, oStX, oStT, oStY;   // staging (byte offsets from the start of the area)
    size_t odt, oA, olam, olamn, odtn, ocA, ow, og, os, oe, odcA, odw, odg, ods;
    size_t oStg, ocs, osn, odph, oth, ored, total;
    // hn2: a second state tile, so that H'_{c+1} (the checkpoint loaded for the chunk after) stays
    // in shared memory for chunk c
    __host__ __device__ BwdSmem(int Q_, int R_, int N_, int P_, int esz, bool hn2) {
        Q = Q_; R = R_; N = N_; P = P_; K = N / 2; QR = Q * R;
        NP = rup4(N); PP = rup4(P); QRP = rup4(QR);
        N4 = NP + 4; P4 = PP + 4; QR4 = QRP + 4; QS = QRP + 4; QP1 = Q + 1;
        rowB = (size_t)R * N * esz; rowX = (size_t)R * P * esz; rowT = (size_t)K * esz; rowY = (size_t)R * P * 4;
        size_t o = 0;
        oD = o;   o += (size_t)N * P4;      // D (true frame); during a chunk D~ = R(-phi_e) D   [N][P4]
        oDtT = o; o += (size_t)PP * N4;     // D~^T                    [PP][N4]
        oH = o;   o += (size_t)PP * N4 * (hn2 ? 2 : 1);   // H'_c^T [2]; in pass 1 the running state H'^T
        oB = o;   o += (size_t)QR * N4;     // B~                      [QR][N4]
        oC = o;   o += (size_t)QR * N4;     // C~
        oBT = o;  o += (size_t)NP * QR4;    // B~^T                    [NP][QR4]
        oX = o;   o += (size_t)QR * P4;     // x; in pass 1 X^ = s x   [QR][P4]
        oXT = o;  o += (size_t)PP * QR4;    // x^T                     [PP][QR4]
        oY = o;   o += (size_t)QR * P4;     // dy
        oYe = o;  o += (size_t)QR * P4;     // e^{cA_t} dy
        oS = o;   o += (size_t)QRP * QS;    // S, then M o S           [QRP][QS]
        oZ = o;   o += (size_t)QRP * QS;    // Z, then M o Z
        oT1 = o;  o += (size_t)QR * P4;     // B~ D~
        oT2 = o;  o += (size_t)QR * N4;     // dY H'^T
        // staging of the raw rows of one chunk (16-byte aligned parts)
        {
            size_t sb = 0;
            auto part = [&](size_t bytes) { const size_t at = sb; sb += (bytes + 15) / 16 * 16; return at; };
            oStB = part(Q * rowB); oStC = part(Q * rowB); oStX = part(Q * rowX); oStT = part(Q * rowT);
            oStY = part(Q * rowY);
            oStg = o; o += sb / 4;
        }
        odM = o;  o += (size_t)Q * Q;       // dM per token pair
        odt = o; o += Q; oA = o; o += Q; olam = o; o += Q; olamn = o; o += Q; odtn = o; o += Q;
        ocA = o; o += Q; ow = o; o += Q; og = o; o += Q; os = o; o += Q; oe = o; o += Q;
        odcA = o; o += Q; odw = o; o += Q; odg = o; o += Q; ods = o; o += Q;
        ocs = o; o += (size_t)K * QP1; osn = o; o += (size_t)K * QP1;   // cos / sin, [K][Q + 1]
        odph = o; o += (size_t)Q * K;
        oth = o; o += (size_t)K * QP1;     // theta of the chunk, [K][Q + 1]
        ored = o; o += kBwdWarps;           // per-warp partial sums
        total = o;
    }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((unsigned)__cvta_generic_to_shared(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// sin and cos of x: reduced by 2 pi with a two-constant Cody-Waite split to [-pi, pi] (n = round(x / 2 pi)
// by the 1.5 * 2^23 addition, exact for |x / 2 pi| < 2^22), then the hardware approximations
__device__ __forceinline__ void sincos_red(float x, float *s, float *c) {
    const float n = (fmaf(x, 0.15915494309189535f, 12582912.f) - 12582912.f);
    float r = fmaf(n, -6.28318548202514648f, x);
    r = fmaf(n, 1.7484555314695172e-7f, r);
    __sincosf(r, s, c);
}

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void fma4(float a, float4 b, float4 &c) {
    c.x = fmaf(a, b.x, c.x);
    c.y = fmaf(a, b.y, c.y);
    c.z = fmaf(a, b.z, c.z);
    c.w = fmaf(a, b.w, c.w);
}
__device__ __forceinline__ float4 axpy4(float a, float4 x, float4 y) {   // a x + y
    return make_float4(fmaf(a, x.x, y.x), fmaf(a, x.y, y.y), fmaf(a, x.z, y.z), fmaf(a, x.w, y.w));
}

// c0 += sum_k A0[k as] B[k bs .. + 3] for k in [k0, k1) (one output row, four columns); four steps
// at a time, so that with constant strides every load takes an immediate offset, in a loop kept
// rolled (with constant bounds a full unroll of every call site crowds the instruction cache)
__device__ __forceinline__ void mm1(const float *A0, int as, const float *B, int bs, int k0, int k1, float4 &c0) {
    int k = k0;
#pragma unroll 1
    for (; k + 4 <= k1; k += 4) {
        const float *a = A0 + k * as, *bp = B + k * bs;
#pragma unroll
        for (int u = 0; u < 4; ++u) fma4(a[u * as], ld4(bp + u * bs), c0);
    }
    for (; k < k1; ++k) fma4(A0[k * as], ld4(B + k * bs), c0);
}
// c0, c1 += the same for two output rows sharing the right operand
__device__ __forceinline__ void mm2(const float *A0, const float *A1, int as, const float *B, int bs, int k0, int k1,
                                    float4 &c0, float4 &c1) {
    int k = k0;
#pragma unroll 1
    for (; k + 4 <= k1; k += 4) {
        const float *a0 = A0 + k * as, *a1 = A1 + k * as, *bp = B + k * bs;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float4 b = ld4(bp + u * bs);
            fma4(a0[u * as], b, c0);
            fma4(a1[u * as], b, c1);
        }
    }
    for (; k < k1; ++k) {
        const float4 b = ld4(B + k * bs);
        fma4(A0[k * as], b, c0);
        fma4(A1[k * as], b, c1);
    }
}

// NT, PT, QRT: the state size, head dim and rows per chunk when fixed at compile time (0: at run
// time), so that the tile strides and most loop bounds are constants
template <typename T, int NT, int PT, int QRT>
__global__ void __launch_bounds__(kBwdThreads, 1)
scan_bwd_kernel(BwdArgs a, int Q, int cp16, int hn2) {   // cp16: the raw rows and checkpoints copy in 16-byte
                                                        // pieces; hn2: two state tiles (BwdSmem)
    extern __shared__ __align__(16) float sm[];
    const BwdSmem Lo(Q, a.R, a.N, a.P, (int)sizeof(T), hn2 != 0);
    const int N = NT ? NT : a.N, P = PT ? PT : a.P, R = a.R, K = N / 2, H = a.H, L = a.L;
    // the same values as Lo's, as constants where the shape is fixed
    const int NP = NT ? rup4(NT) : Lo.NP, PP = PT ? rup4(PT) : Lo.PP;
    const int N4 = NP + 4, P4 = PP + 4, QR4 = QRT ? rup4(QRT) + 4 : Lo.QR4, QS = QR4;
    const int NC4 = NP / 4, PC4 = PP / 4;   // float4 columns of the N- and P-wide tiles
    float *Dm = sm + Lo.oD, *DtT = sm + Lo.oDtT, *Hs = sm + Lo.oH;   // Hs: pass 1's running state, buffer 0
    float *Bt = sm + Lo.oB, *Ct = sm + Lo.oC, *BtT = sm + Lo.oBT, *Xs = sm + Lo.oX, *XsT = sm + Lo.oXT;
    float *Ys = sm + Lo.oY, *Ye = sm + Lo.oYe;
    float *Sm = sm + Lo.oS, *Zm = sm + Lo.oZ, *T1 = sm + Lo.oT1, *T2 = sm + Lo.oT2, *dMt = sm + Lo.odM;
    float *vdt = sm + Lo.odt, *vA = sm + Lo.oA, *vl = sm + Lo.olam, *vln = sm + Lo.olamn, *vdtn = sm + Lo.odtn;
    float *cA = sm + Lo.ocA, *wv = sm + Lo.ow, *gv = sm + Lo.og, *sv = sm + Lo.os, *ev = sm + Lo.oe;
    float *dcA = sm + Lo.odcA, *dwv = sm + Lo.odw, *dgv = sm + Lo.odg, *dsv = sm + Lo.ods;
    float *cs = sm + Lo.ocs, *sn = sm + Lo.osn, *dph = sm + Lo.odph, *thv = sm + Lo.oth, *red = sm + Lo.ored;
    unsigned char *stg = reinterpret_cast<unsigned char *>(sm + Lo.oStg);
    const T *stB = reinterpret_cast<const T *>(stg + Lo.oStB), *stC = reinterpret_cast<const T *>(stg + Lo.oStC);
    const T *stX = reinterpret_cast<const T *>(stg + Lo.oStX), *stT = reinterpret_cast<const T *>(stg + Lo.oStT);
    const float *stY = reinterpret_cast<const float *>(stg + Lo.oStY);
    const int QP1 = Lo.QP1;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int bh = blockIdx.x, b = bh / H, h = bh % H;
    const int nc = (L + Q - 1) / Q;
    const T *xg = static_cast<const T *>(a.x), *Bg = static_cast<const T *>(a.B), *Cg = static_cast<const T *>(a.C);
    const T *dtg = static_cast<const T *>(a.dt), *Ag = static_cast<const T *>(a.A), *lg = static_cast<const T *>(a.lam);
    const T *thg = static_cast<const T *>(a.theta);
    auto tok = [&](int t) { return ((size_t)b * L + t) * H + h; };
    float *ckpt = a.ws + (size_t)bh * (nc + 1) * N * P;   // H'_c^T ([P][N]), c = 0..nc

    // every pad column and row starts (and stays) zero
    for (size_t i = tid; i < Lo.total; i += kBwdThreads) sm[i] = 0.f;
    __syncthreads();

    // The raw rows of the Qn tokens at s0n (B; with C also C and dy) into the staging area: 16-byte
    // asynchronous copies (one commit group), or plain copies where the rows do not split into them
    auto stage = [&](int s0n, int Qn, bool withC) {
        const size_t tok0 = ((size_t)b * L + s0n) * H + h;   // token rows are H rows apart
        if (cp16) {
            const int pB = (int)(Lo.rowB / 16), pX = (int)(Lo.rowX / 16), pT = (int)(Lo.rowT / 16);
            const int pY = (int)(Lo.rowY / 16);
            const int nB = Qn * pB, nC = withC ? nB : 0, nX = Qn * pX, nT = Qn * pT, nY = withC ? Qn * pY : 0;
            for (int i = tid; i < nB + nC + nX + nT + nY; i += kBwdThreads) {
                int j = i, pp;
                size_t row, dst;
                const char *base;
                if (j < nB) {
                    pp = pB; base = static_cast<const char *>(a.B); row = Lo.rowB; dst = Lo.oStB;
                } else if ((j -= nB) < nC) {
                    pp = pB; base = static_cast<const char *>(a.C); row = Lo.rowB; dst = Lo.oStC;
                } else if ((j -= nC) < nX) {
                    pp = pX; base = static_cast<const char *>(a.x); row = Lo.rowX; dst = Lo.oStX;
                } else if ((j -= nX) < nT) {
                    pp = pT; base = static_cast<const char *>(a.theta); row = Lo.rowT; dst = Lo.oStT;
                } else {
                    j -= nT; pp = pY; base = reinterpret_cast<const char *>(a.dy); row = Lo.rowY; dst = Lo.oStY;
                }
                const int t = j / pp, q = j % pp;
                cp_async16(stg + dst + t * row + 16 * q, base + (tok0 + (size_t)t * H) * row + 16 * q);
            }
        } else {
            T *sB = reinterpret_cast<T *>(stg + Lo.oStB), *sC = reinterpret_cast<T *>(stg + Lo.oStC);
            T *sX = reinterpret_cast<T *>(stg + Lo.oStX), *sT = reinterpret_cast<T *>(stg + Lo.oStT);
            float *sY = reinterpret_cast<float *>(stg + Lo.oStY);
            for (int i = tid; i < Qn * R * N; i += kBwdThreads) {
                const size_t g = (tok0 + (size_t)(i / (R * N)) * H) * R * N + i % (R * N);
                sB[i] = Bg[g];
                if (withC) sC[i] = Cg[g];
            }
            for (int i = tid; i < Qn * R * P; i += kBwdThreads) {
                const size_t g = (tok0 + (size_t)(i / (R * P)) * H) * R * P + i % (R * P);
                sX[i] = xg[g];
                if (withC) sY[i] = a.dy[g];
            }
            for (int i = tid; i < Qn * K; i += kBwdThreads) sT[i] = thg[(tok0 + (size_t)(i / K) * H) * K + i % K];
        }
        cp_async_commit();   // (an empty group on the plain path)
    };
    // per-token scalars of the Qn tokens at s0n, one token per thread (threads < Q), into registers
    float r_dt = 0.f, r_A = 0.f, r_l = 0.f, r_ln = 1.f, r_dtn = 0.f;
    auto fetch = [&](int s0n, int Qn) {
        r_dt = r_A = r_l = r_dtn = 0.f;
        r_ln = 1.f;
        if (tid < Qn) {
            const size_t ti = tok(s0n + tid);
            r_dt = to_f(dtg[ti]);
            r_A = to_f(Ag[ti]);
            r_l = to_f(lg[ti]);
            if (s0n + tid + 1 < L) {
                r_ln = to_f(lg[tok(s0n + tid + 1)]);
                r_dtn = to_f(dtg[tok(s0n + tid + 1)]);
            }
        }
    };

    // The chunk at s0 (Qc tokens, staged and fetched): its scalars, angles (cos / sin of the
    // chunk-local phi), rotated B (with pass2 also C and the transposes) and x (pass 1: X^ = s x)
    // into their tiles.  Entered with the staging copies complete (this thread's); its first
    // barrier makes every thread's visible.
    auto load_chunk = [&](int Qc, bool pass2) {
        for (int i = tid; i < Q; i += kBwdThreads) {
            vdt[i] = r_dt; vA[i] = r_A; vl[i] = r_l; vln[i] = r_ln; vdtn[i] = r_dtn;
            cA[i] = r_dt * r_A;
        }
        __syncthreads();
        for (int i = tid; i < Q * K; i += kBwdThreads) {
            const int t = i / K, k = i % K;
            thv[k * QP1 + t] = t < Qc ? to_f(stT[i]) : 0.f;
        }
        if (warp == 0) {   // inclusive cumsum of dt A (chunk-local), 32 tokens at a time
            float carry = 0.f;
            for (int base = 0; base < Q; base += 32) {
                float v = base + lane < Q ? cA[base + lane] : 0.f;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float t = __shfl_up_sync(0xffffffffu, v, o);
                    if (lane >= o) v += t;
                }
                v += carry;
                if (base + lane < Q) cA[base + lane] = v;
                carry = __shfl_sync(0xffffffffu, v, 31);
            }
        }
        __syncthreads();
        // chunk-local angle of token t (a lane), pair k: an inclusive scan over the tokens (Q <= 32)
        for (int k = warp; k < K; k += kBwdWarps) {
            float phi = lane < Q ? vdt[lane] * thv[k * QP1 + lane] : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float t = __shfl_up_sync(0xffffffffu, phi, o);
                if (lane >= o) phi += t;
            }
            if (lane < Q) {
                float s, c;
                sincos_red(phi, &s, &c);
                cs[k * QP1 + lane] = c;
                sn[k * QP1 + lane] = s;
            }
        }
        const int e = Qc - 1;
        for (int i = tid; i < Q; i += kBwdThreads) {
            const float w = vl[i] * vdt[i] + (1.f - vln[i]) * vdtn[i];
            wv[i] = i < Qc ? w : 0.f;
            gv[i] = i < Qc ? vl[i] * vdt[i] : 0.f;
            sv[i] = i < Qc ? expf(cA[e] - cA[i]) * w : 0.f;
            ev[i] = i < Qc ? expf(cA[i]) : 0.f;
        }
        __syncthreads();
        for (int i = tid; i < Q * R * K; i += kBwdThreads) {
            const int row = i / K, k = i % K, t = row / R;
            float b0 = 0.f, b1 = 0.f, c0 = 0.f, c1 = 0.f;
            if (t < Qc) {
                const int q = row * N + 2 * k;
                b0 = to_f(stB[q]);
                b1 = to_f(stB[q + 1]);
                if (pass2) {
                    c0 = to_f(stC[q]);
                    c1 = to_f(stC[q + 1]);
                }
            }
            const float c = cs[k * QP1 + t], s = sn[k * QP1 + t];
            const float bt0 = c * b0 + s * b1, bt1 = -s * b0 + c * b1;   // R(-phi) applied to the pair
            Bt[row * N4 + 2 * k] = bt0;
            Bt[row * N4 + 2 * k + 1] = bt1;
            if (pass2) {
                BtT[(2 * k) * QR4 + row] = bt0;
                BtT[(2 * k + 1) * QR4 + row] = bt1;
                Ct[row * N4 + 2 * k] = c * c0 + s * c1;
                Ct[row * N4 + 2 * k + 1] = -s * c0 + c * c1;
            }
        }
        for (int i = tid; i < Q * R * P; i += kBwdThreads) {
            const int row = i / P, p = i % P, t = row / R;
            float v = t < Qc ? to_f(stX[i]) : 0.f;
            if (pass2) {
                Xs[row * P4 + p] = v;
                XsT[p * QR4 + row] = v;
            } else {
                Xs[row * P4 + p] = sv[t] * v;
            }
        }
        __syncthreads();
    };

    // ================================================================ pass 1: checkpoints
    {
        const float *h0 = a.h0 ? a.h0 + (size_t)bh * N * P : nullptr;
        const T *bq = static_cast<const T *>(a.Bprev), *xq = static_cast<const T *>(a.xprev);
        const float left0 = L > 0 ? (1.f - to_f(lg[tok(0)])) * to_f(dtg[tok(0)]) : 0.f;
        for (int i = tid; i < N * P; i += kBwdThreads) {   // i = p N + n: the transposed layout
            const int p = i / N, n = i % N;
            float v = h0 ? h0[(size_t)n * P + p] : 0.f;
            if (bq && xq) {
                float u = 0.f;
                for (int r = 0; r < R; ++r)
                    u += to_f(bq[((size_t)bh * R + r) * N + n]) * to_f(xq[((size_t)bh * R + r) * P + p]);
                v += left0 * u;
            }
            Hs[p * N4 + n] = v;
            ckpt[i] = v;
        }
        stage(0, min(Q, L), false);
        fetch(0, min(Q, L));
        __syncthreads();
        for (int c = 0; c < nc; ++c) {
            const int s0 = c * Q, Qc = min(Q, L - s0), e = Qc - 1, QRc = Qc * R;
            cp_async_wait<0>();
            load_chunk(Qc, false);
            if (c + 1 < nc) {   // the next chunk's rows come in while this one is folded into the state
                stage(s0 + Q, min(Q, L - s0 - Q), false);
                fetch(s0 + Q, min(Q, L - s0 - Q));
            }
            const float de = expf(cA[e]);
            float *dst = ckpt + (size_t)(c + 1) * N * P;
            // H'^T <- R(phi_e) [e^{cA_e} H'^T + X^^T B~], rows p in pairs, four columns n (two pairs)
            for (int i = tid; i < ((P + 1) / 2) * NC4; i += kBwdThreads) {
                const int p = 2 * (i / NC4), n4 = i % NC4, p1 = min(p + 1, P - 1);
                float4 u0 = make_float4(0.f, 0.f, 0.f, 0.f), u1 = u0;
                mm2(Xs + p, Xs + p1, P4, Bt + 4 * n4, N4, 0, QRc, u0, u1);
                const int k0 = 2 * n4, k1 = min(2 * n4 + 1, K - 1);
                const float c0 = cs[k0 * QP1 + e], s0_ = sn[k0 * QP1 + e], c1 = cs[k1 * QP1 + e], s1 = sn[k1 * QP1 + e];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int pp = q ? p1 : p;
                    if (q && p1 == p) continue;
                    float *hrow = Hs + pp * N4 + 4 * n4;
                    const float4 hv = ld4(hrow), u = q ? u1 : u0;
                    const float4 v = axpy4(de, hv, u);
                    const float4 nv = make_float4(c0 * v.x - s0_ * v.y, s0_ * v.x + c0 * v.y,
                                                  c1 * v.z - s1 * v.w, s1 * v.z + c1 * v.w);
                    st4(hrow, nv);
                    const int n = 4 * n4;
                    float *drow = dst + (size_t)pp * N + n;
                    drow[0] = nv.x;
                    drow[1] = nv.y;
                    if (n + 2 < N) {
                        drow[2] = nv.z;
                        drow[3] = nv.w;
                    }
                }
            }
            __syncthreads();
        }
    }

    // ================================================================ pass 2: gradients
    for (int i = tid; i < N * P; i += kBwdThreads)
        Dm[(i / P) * P4 + i % P] = a.dh_out ? a.dh_out[(size_t)bh * N * P + i] : 0.f;
    stage((nc - 1) * Q, L - (nc - 1) * Q, true);
    fetch((nc - 1) * Q, L - (nc - 1) * Q);
    for (int c = nc - 1; c >= 0; --c) {
        const int s0 = c * Q, Qc = min(Q, L - s0), e = Qc - 1, QRc = Qc * R;
        for (int i = tid; i < Q; i += kBwdThreads) {
            dcA[i] = 0.f;
            dwv[i] = 0.f;
            dgv[i] = 0.f;
            dsv[i] = 0.f;
        }
        for (int i = tid; i < Q * K; i += kBwdThreads) dph[i] = 0.f;
        // H'_c^T copied in while the chunk's inputs are turned (a second commit group).  With two
        // tiles, chunk c's goes to tile (c ^ nc) & 1: the other one holds H'_{c+1}, which for the
        // last chunk is pass 1's final state, left in tile 0
        const float *Hc = ckpt + (size_t)c * N * P;
        float *Hs = sm + Lo.oH + (hn2 ? (size_t)((c ^ nc) & 1) * Lo.PP * N4 : 0);
        const float *Hn_s = sm + Lo.oH + (size_t)((c ^ nc ^ 1) & 1) * Lo.PP * N4;   // (hn2 only)
        if (cp16) {
            const int pr = N / 4;
            for (int i = tid; i < P * pr; i += kBwdThreads)
                cp_async16(Hs + (i / pr) * N4 + 4 * (i % pr), Hc + (size_t)(i / pr) * N + 4 * (i % pr));
        } else {
            for (int i = tid; i < N * P; i += kBwdThreads) Hs[(i / N) * N4 + i % N] = Hc[i];
        }
        cp_async_commit();
        cp_async_wait<1>();         // the staged rows (the group before)
        load_chunk(Qc, true);       // its barriers also order the zeroing above
        const float *Hn = ckpt + (size_t)(c + 1) * N * P;
        for (int i = tid; i < QRc * P; i += kBwdThreads) {
            const int row = i / P, p = i % P, t = row / R;
            const float v = stY[i];
            Ys[row * P4 + p] = v;
            Ye[row * P4 + p] = ev[t] * v;
        }
        for (int i = QRc * P + tid; i < Q * R * P; i += kBwdThreads) {   // rows past the sequence end
            const int row = i / P, p = i % P;
            Ys[row * P4 + p] = 0.f;
            Ye[row * P4 + p] = 0.f;
        }
        // D~ = R(-phi_e) D in place (and its transpose), and the angle gradient of the turn R(phi_e):
        // <D, J H'_{c+1}> per pair, over four columns p per thread
        for (int i = tid; i < K * PC4; i += kBwdThreads) {   // consecutive threads: consecutive pairs
            const int k = i % K, p = 4 * (i / K);
            const float cc = cs[k * QP1 + e], ss = sn[k * QP1 + e];
            const float4 d0 = ld4(Dm + (2 * k) * P4 + p), d1 = ld4(Dm + (2 * k + 1) * P4 + p);
            const float4 t0 = make_float4(cc * d0.x + ss * d1.x, cc * d0.y + ss * d1.y, cc * d0.z + ss * d1.z,
                                          cc * d0.w + ss * d1.w);
            const float4 t1 = make_float4(-ss * d0.x + cc * d1.x, -ss * d0.y + cc * d1.y, -ss * d0.z + cc * d1.z,
                                          -ss * d0.w + cc * d1.w);
            st4(Dm + (2 * k) * P4 + p, t0);
            st4(Dm + (2 * k + 1) * P4 + p, t1);
            const float a0[4] = {t0.x, t0.y, t0.z, t0.w}, a1[4] = {t1.x, t1.y, t1.z, t1.w};
            const float e0[4] = {d0.x, d0.y, d0.z, d0.w}, e1[4] = {d1.x, d1.y, d1.z, d1.w};
            float v = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                *reinterpret_cast<float2 *>(DtT + (p + q) * N4 + 2 * k) = make_float2(a0[q], a1[q]);
                if (p + q < P) {
                    const float2 hn = hn2 ? *reinterpret_cast<const float2 *>(Hn_s + (p + q) * N4 + 2 * k)
                                          : *reinterpret_cast<const float2 *>(Hn + (size_t)(p + q) * N + 2 * k);
                    v += e1[q] * hn.x - e0[q] * hn.y;
                }
            }
            atomicAdd(&dph[e * K + k], v);
        }
        cp_async_wait<0>();         // H'_c^T
        __syncthreads();
        if (c > 0) {   // the chunk before: its rows come in while this one is processed
            stage(s0 - Q, Q, true);
            fetch(s0 - Q, Q);
        }
        // S = C~ B~^T, Z = dY X^T (1 x 4 tiles), B~ D~ (rows x P) and dY H'^T (rows x N) (2 x 4 tiles)
        {
            const int QC4 = (QRc + 3) / 4, R2 = (QRc + 1) / 2;
            const int nS = QRc * QC4, nT1 = R2 * PC4, nT2 = R2 * NC4;
            for (int i = tid; i < 2 * nS + nT1 + nT2; i += kBwdThreads) {
                float4 c0 = make_float4(0.f, 0.f, 0.f, 0.f), c1 = c0;
                if (i < 2 * nS) {
                    const bool isZ = i >= nS;
                    const int q = isZ ? i - nS : i, rt = q / QC4, j4 = q % QC4;
                    if ((4 * j4) / R <= rt / R) {   // otherwise every column lies past the token
                        if (isZ) mm1(Ys + rt * P4, 1, XsT + 4 * j4, QR4, 0, P, c0);
                        else mm1(Ct + rt * N4, 1, BtT + 4 * j4, QR4, 0, N, c0);
                    }
                    st4((isZ ? Zm : Sm) + rt * QS + 4 * j4, c0);
                } else if (i < 2 * nS + nT1) {
                    const int q = i - 2 * nS, r0 = 2 * (q / PC4), p4 = q % PC4, r1 = min(r0 + 1, QRc - 1);
                    mm2(Bt + r0 * N4, Bt + r1 * N4, 1, Dm + 4 * p4, P4, 0, N, c0, c1);
                    st4(T1 + r0 * P4 + 4 * p4, c0);
                    if (r1 != r0) st4(T1 + r1 * P4 + 4 * p4, c1);
                } else {
                    const int q = i - 2 * nS - nT1, r0 = 2 * (q / NC4), n4 = q % NC4, r1 = min(r0 + 1, QRc - 1);
                    mm2(Ys + r0 * P4, Ys + r1 * P4, 1, Hs + 4 * n4, N4, 0, P, c0, c1);
                    st4(T2 + r0 * N4 + 4 * n4, c0);
                    if (r1 != r0) st4(T2 + r1 * N4 + 4 * n4, c1);
                }
            }
        }
        __syncthreads();
        // dM per token pair (sum over rank pairs), then M o S and M o Z in place
        for (int i = tid; i < Qc * Qc; i += kBwdThreads) {
            const int t = i / Qc, j = i % Qc;
            float v = 0.f;
            if (j <= t)
                for (int r = 0; r < R; ++r)
                    for (int r2 = 0; r2 < R; ++r2)
                        v = fmaf(Sm[(t * R + r) * QS + j * R + r2], Zm[(t * R + r) * QS + j * R + r2], v);
            dMt[t * Q + j] = v;
        }
        __syncthreads();
        for (int i = tid; i < QRc * QRc; i += kBwdThreads) {
            const int rt = i / QRc, rj = i % QRc, t = rt / R, j = rj / R;
            const float m = j < t ? __expf(cA[t] - cA[j]) * wv[j] : (j == t ? gv[t] : 0.f);
            Sm[rt * QS + rj] *= m;
            Zm[rt * QS + rj] *= m;
        }
        // token scalars: mask terms (dcA, dw, dg) and the inter-chunk and state terms
        for (int t = warp; t < Qc; t += kBwdWarps) {
            float rowv = 0.f, colv = 0.f, dwj = 0.f;
            for (int j = lane; j < Qc; j += 32) {
                if (j < t) rowv += dMt[t * Q + j] * __expf(cA[t] - cA[j]) * wv[j];   // d cA_t
                if (j > t) {
                    const float f = __expf(cA[j] - cA[t]);
                    colv += dMt[j * Q + t] * f * wv[t];                              // -d cA_t (as column)
                    dwj += dMt[j * Q + t] * f;                                       // d w_t
                }
            }
            rowv = warp_sum(rowv);
            colv = warp_sum(colv);
            dwj = warp_sum(dwj);
            // inter-chunk readout: e^{cA_t} C~_t . (dY H'^T)_t, summed over ranks; state term ds_t
            float yi = 0.f, dsum = 0.f;
            for (int r = 0; r < R; ++r) {
                const int row = t * R + r;
                for (int n = lane; n < N; n += 32) yi += Ct[row * N4 + n] * T2[row * N4 + n];
                for (int p = lane; p < P; p += 32) dsum += Xs[row * P4 + p] * T1[row * P4 + p];
            }
            yi = warp_sum(yi);
            dsum = warp_sum(dsum);
            if (lane == 0) {
                dcA[t] += rowv - colv + ev[t] * yi;
                dwv[t] += dwj;
                dgv[t] = dMt[t * Q + t];
                dsv[t] = dsum;
            }
        }
        // <D~, H'_c> (the transport e^{cA_e} H'_c into the chunk end), per-warp partial sums
        {
            float v = 0.f;
            for (int i = tid; i < P * NC4; i += kBwdThreads) {
                const int q = (i / NC4) * N4 + 4 * (i % NC4);
                const float4 d = ld4(DtT + q), hv = ld4(Hs + q);
                v += d.x * hv.x + d.y * hv.y + d.z * hv.z + d.w * hv.w;
            }
            v = warp_sum(v);
            if (lane == 0) red[warp] = v;
        }
        __syncthreads();
        if (warp == 0) {
            // s_j = e^{cA_e - cA_j} w_j, and the transport (one lane per token; Qc <= 32)
            float dh = lane < kBwdWarps ? red[lane] : 0.f, v = 0.f;
            if (lane < Qc) {
                v = sv[lane] * dsv[lane];
                dcA[lane] -= v;
                dwv[lane] += expf(cA[e] - cA[lane]) * dsv[lane];
            }
            dh = warp_sum(dh);
            v = warp_sum(v);
            __syncwarp();
            if (lane == 0) dcA[e] += v + expf(cA[e]) * dh;
        }
        __syncthreads();
        // dX = (M o S)^T dY + diag(s) B~ D~  (the carry out adds to the sequence's last token);
        // dB~ = (M o Z)^T C~ + diag(s) X D~^T and dC~ = (M o Z) B~ + diag(e^{cA}) dY H'^T, un-rotated
        // as they are formed, with the angle gradients dphi_{t,k} += dv0 v1 - dv1 v0 over the B~ and
        // C~ rows of token t
        {
            const int R2 = (QRc + 1) / 2, nX = R2 * PC4, nB = R2 * NC4;
            for (int i = tid; i < nX + 2 * nB; i += kBwdThreads) {
                float4 c0 = make_float4(0.f, 0.f, 0.f, 0.f), c1 = c0;
                if (i < nX) {
                    const int r0 = 2 * (i / PC4), p4 = i % PC4, r1 = min(r0 + 1, QRc - 1), p = 4 * p4;
                    // rows of earlier tokens hold M o S = 0: start at the first row of r0's token
                    mm2(Sm + r0, Sm + r1, QS, Ys + p, P4, (r0 / R) * R, QRc, c0, c1);
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const int rj = q ? r1 : r0;
                        if (q && r1 == r0) continue;
                        const int j = rj / R, r = rj % R;
                        float4 v = axpy4(sv[j], ld4(T1 + rj * P4 + p), q ? c1 : c0);
                        const float vv[4] = {v.x, v.y, v.z, v.w};
                        const bool last = s0 + j == L - 1 && a.dxprev_out;
                        float *dxr = a.dx + (tok(s0 + j) * R + r) * P;
#pragma unroll
                        for (int z = 0; z < 4; ++z)
                            if (p + z < P)
                                dxr[p + z] = vv[z] + (last ? a.dxprev_out[((size_t)bh * R + r) * P + p + z] : 0.f);
                    }
                } else {
                    const bool isC = i >= nX + nB;
                    const int q = isC ? i - nX - nB : i - nX;
                    const int r0 = 2 * (q / NC4), n4 = q % NC4, r1 = min(r0 + 1, QRc - 1), n = 4 * n4;
                    if (!isC) {
                        mm2(Zm + r0, Zm + r1, QS, Ct + n, N4, (r0 / R) * R, QRc, c0, c1);
                        float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
                        mm2(Xs + r0 * P4, Xs + r1 * P4, 1, DtT + n, N4, 0, P, x0, x1);
                        c0 = axpy4(sv[r0 / R], x0, c0);
                        c1 = axpy4(sv[r1 / R], x1, c1);
                    } else {
                        // row r1's token ends the range of columns rj with M o Z != 0
                        mm2(Zm + r0 * QS, Zm + r1 * QS, 1, Bt + n, N4, 0, min(QRc, (r1 / R + 1) * R), c0, c1);
                        c0 = axpy4(ev[r0 / R], ld4(T2 + r0 * N4 + n), c0);
                        c1 = axpy4(ev[r1 / R], ld4(T2 + r1 * N4 + n), c1);
                    }
                    const float *Vt = isC ? Ct : Bt;   // the rotated operand itself
                    float *dst = isC ? a.dC : a.dB;
#pragma unroll
                    for (int qq = 0; qq < 2; ++qq) {
                        const int row = qq ? r1 : r0;
                        if (qq && r1 == r0) continue;
                        const int j = row / R, r = row % R;
                        const float4 g = qq ? c1 : c0, vt = ld4(Vt + row * N4 + n);
                        const float gg[4] = {g.x, g.y, g.z, g.w}, tv[4] = {vt.x, vt.y, vt.z, vt.w};
                        const size_t base = (tok(s0 + j) * R + r) * N;
                        const bool last = !isC && s0 + j == L - 1 && a.dBprev_out;
#pragma unroll
                        for (int pr = 0; pr < 2; ++pr) {
                            const int k = 2 * n4 + pr;
                            if (k >= K) continue;
                            const float g0 = gg[2 * pr], g1 = gg[2 * pr + 1];
                            atomicAdd(&dph[j * K + k], g0 * tv[2 * pr + 1] - g1 * tv[2 * pr]);
                            // un-rotate: dB = R(phi) dB~
                            const float cc = cs[k * QP1 + j], ss = sn[k * QP1 + j];
                            float o0 = cc * g0 - ss * g1, o1 = ss * g0 + cc * g1;
                            if (last) {
                                o0 += a.dBprev_out[((size_t)bh * R + r) * N + 2 * k];
                                o1 += a.dBprev_out[((size_t)bh * R + r) * N + 2 * k + 1];
                            }
                            dst[base + 2 * k] = o0;
                            dst[base + 2 * k + 1] = o1;
                        }
                    }
                }
            }
        }
        __syncthreads();
        // reverse cumulative sums: d(dt A)_u = sum_{t >= u} dcA_t, d(dt theta)_u = sum_{t >= u} dphi_t
        if (warp == 0) {
            float carry = 0.f;
            for (int base = ((Qc - 1) / 32) * 32; base >= 0; base -= 32) {
                const int u = base + 31 - lane;   // lanes walk the tokens from the top
                float v = (u < Qc) ? dcA[u] : 0.f;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float t = __shfl_up_sync(0xffffffffu, v, o);
                    if (lane >= o) v += t;
                }
                v += carry;
                if (u < Qc) dcA[u] = v;
                carry = __shfl_sync(0xffffffffu, v, 31);
            }
        }
        for (int k = tid; k < K; k += kBwdThreads) {
            float acc = 0.f;
            for (int u = Qc - 1; u >= 0; --u) {
                acc += dph[u * K + k];
                dph[u * K + k] = acc;
            }
        }
        __syncthreads();
        // parameter gradients of the chunk's tokens; the left-endpoint part of w_{u-1} belongs to
        // token u: for the chunk's first token it is added when the chunk before is processed
        for (int i = tid; i < Qc * K; i += kBwdThreads) {
            const int u = i / K, k = i % K;
            a.dtheta[tok(s0 + u) * K + k] = vdt[u] * dph[i];
        }
        for (int u = warp; u < Qc; u += kBwdWarps) {   // one warp per token: sum_k theta_k d(dt theta)_k
            const size_t ti = tok(s0 + u);
            float thsum = 0.f;
            for (int k = lane; k < K; k += 32) thsum = fmaf(thv[k * QP1 + u], dph[u * K + k], thsum);
            thsum = warp_sum(thsum);
            if (lane == 0) {
                const float d = vdt[u], av = vA[u], l = vl[u];
                const float dwp = u > 0 ? dwv[u - 1] : 0.f;
                const float ddt = av * dcA[u] + thsum + l * (dwv[u] + dgv[u]) + (1.f - l) * dwp;
                const float dl = d * (dwv[u] + dgv[u]) - d * dwp;
                if (u == Qc - 1 && s0 + Qc < L) {   // this token's w also feeds the next chunk's first token
                    const size_t tn = tok(s0 + Qc);
                    a.ddt[tn] += (1.f - vln[u]) * dwv[u];
                    a.dlam[tn] -= vdtn[u] * dwv[u];
                }
                a.dA[ti] = d * dcA[u];
                a.ddt[ti] = ddt;
                a.dlam[ti] = dl;
            }
        }
        // D <- e^{cA_e} D~ + C~^T diag(e^{cA}) dY in place (rows n in pairs, four columns p)
        {
            const float de = expf(cA[e]);
            for (int i = tid; i < (N / 2) * PC4; i += kBwdThreads) {
                const int n0 = 2 * (i / PC4), p = 4 * (i % PC4);
                float4 c0 = make_float4(0.f, 0.f, 0.f, 0.f), c1 = c0;
                mm2(Ct + n0, Ct + n0 + 1, N4, Ye + p, P4, 0, QRc, c0, c1);
                st4(Dm + n0 * P4 + p, axpy4(de, ld4(Dm + n0 * P4 + p), c0));
                st4(Dm + (n0 + 1) * P4 + p, axpy4(de, ld4(Dm + (n0 + 1) * P4 + p), c1));
            }
        }
        __syncthreads();
    }

    // ================================================================ initial state and carry
    // H'_0 = h0 + left_0 B_{-1} x_{-1}^T: dh0 = D; d left_0 = <D, B_{-1} x_{-1}^T>
    if (a.dh0)
        for (int i = tid; i < N * P; i += kBwdThreads) a.dh0[(size_t)bh * N * P + i] = Dm[(i / P) * P4 + i % P];
    const T *bq = static_cast<const T *>(a.Bprev), *xq = static_cast<const T *>(a.xprev);
    if (bq && xq) {
        const float d0 = to_f(dtg[tok(0)]), l0 = to_f(lg[tok(0)]), left0 = (1.f - l0) * d0;
        float dl = 0.f;
        for (int i = tid; i < N * P; i += kBwdThreads) {
            const int n = i / P, p = i % P;
            float u = 0.f;
            for (int r = 0; r < R; ++r)
                u += to_f(bq[((size_t)bh * R + r) * N + n]) * to_f(xq[((size_t)bh * R + r) * P + p]);
            dl = fmaf(Dm[n * P4 + p], u, dl);
        }
        dl = warp_sum(dl);
        if (lane == 0) red[warp] = dl;
        __syncthreads();
        if (tid == 0) {
            float tot = 0.f;
            for (int q = 0; q < kBwdWarps; ++q) tot += red[q];
            a.ddt[tok(0)] += (1.f - l0) * tot;
            a.dlam[tok(0)] -= d0 * tot;
        }
        if (a.dBprev)
            for (int i = tid; i < R * N; i += kBwdThreads) {
                const int r = i / N, n = i % N;
                float v = 0.f;
                for (int p = 0; p < P; ++p) v = fmaf(Dm[n * P4 + p], to_f(xq[((size_t)bh * R + r) * P + p]), v);
                a.dBprev[(size_t)bh * R * N + i] = left0 * v;
            }
        if (a.dxprev)
            for (int i = tid; i < R * P; i += kBwdThreads) {
                const int r = i / P, p = i % P;
                float v = 0.f;
                for (int n = 0; n < N; ++n) v = fmaf(Dm[n * P4 + p], to_f(bq[((size_t)bh * R + r) * N + n]), v);
                a.dxprev[(size_t)bh * R * P + i] = left0 * v;
            }
    } else {
        if (a.dBprev)
            for (int i = tid; i < R * N; i += kBwdThreads) a.dBprev[(size_t)bh * R * N + i] = 0.f;
        if (a.dxprev)
            for (int i = tid; i < R * P; i += kBwdThreads) a.dxprev[(size_t)bh * R * P + i] = 0.f;
    }
}

}  // namespace

// Tokens per chunk: the most rows (t, r) per chunk, up to 32, whose tiles fit one CTA's 227 KB of
// shared memory.
int bwd_chunk(int N, int P, int R, int esz) {
    int Q = 1;
    for (int rows = 32; rows >= 1; rows /= 2) {
        Q = rows / R > 0 ? rows / R : 1;
        if (BwdSmem(Q, R, N, P, esz, false).total * sizeof(float) <= 227u * 1024u) break;
    }
    return Q;
}

size_t bwd_smem_bytes(int N, int P, int R, int esz) {
    return BwdSmem(bwd_chunk(N, P, R, esz), R, N, P, esz, false).total * sizeof(float);
}

size_t bwd_workspace_bytes(int batch, int H, int L, int N, int P, int R, int esz) {
    const int Q = bwd_chunk(N, P, R, esz);
    const size_t nc = (size_t)(L + Q - 1) / Q;
    return (size_t)batch * H * (nc + 1) * N * P * sizeof(float);
}

template <auto Kern>
cudaError_t launch_bwd(const BwdArgs &a, int Q, int cp16, int hn2, size_t smem, unsigned grid, cudaStream_t s) {
    const cudaError_t e = allow_dynamic_smem<Kern>(smem);
    if (e != cudaSuccess) return e;
    Kern<<<grid, kBwdThreads, smem, s>>>(a, Q, cp16, hn2);
    return cudaSuccess;
}

cudaError_t scan_bwd(const BwdArgs &a, cudaStream_t s) {
    const int esz = a.dtype == M3_F32 ? 4 : 2;
    const int Q = bwd_chunk(a.N, a.P, a.R, esz);
    // a second state tile where it fits
    const size_t smem2 = BwdSmem(Q, a.R, a.N, a.P, esz, true).total * sizeof(float);
    const int hn2 = smem2 <= 227u * 1024u;
    const size_t smem = hn2 ? smem2 : bwd_smem_bytes(a.N, a.P, a.R, esz);
    // 16-byte asynchronous copies: every raw row a whole number of 16-byte pieces, every base
    // pointer on a 16-byte boundary (the workspace is), the checkpoint rows too
    auto al16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const int cp16 = ((size_t)a.R * a.N * esz) % 16 == 0 && ((size_t)a.R * a.P * esz) % 16 == 0 &&
                     ((size_t)(a.N / 2) * esz) % 16 == 0 && ((size_t)a.R * a.P * 4) % 16 == 0 && a.N % 4 == 0 &&
                     al16(a.B) && al16(a.C) && al16(a.x) && al16(a.theta) && al16(a.dy) && al16(a.ws);
    const unsigned grid = (unsigned)((long long)a.batch * a.H);
    if (grid == 0 || a.L == 0) return cudaSuccess;
    cudaError_t e;
    trace_mark(M3_KERNEL_BACKWARD, s, 0);
    // the shapes of the pages' models have their own constant-stride builds (bf16 inputs)
    const int QR = Q * a.R;
    if (a.dtype == M3_F32) e = launch_bwd<scan_bwd_kernel<float, 0, 0, 0>>(a, Q, cp16, hn2, smem, grid, s);
    else if (a.N == 64 && a.P == 64 && QR == 32)
        e = launch_bwd<scan_bwd_kernel<__nv_bfloat16, 64, 64, 32>>(a, Q, cp16, hn2, smem, grid, s);
    else if (a.N == 128 && a.P == 64 && QR == 16)
        e = launch_bwd<scan_bwd_kernel<__nv_bfloat16, 128, 64, 16>>(a, Q, cp16, hn2, smem, grid, s);
    else e = launch_bwd<scan_bwd_kernel<__nv_bfloat16, 0, 0, 0>>(a, Q, cp16, hn2, smem, grid, s);
    if (e != cudaSuccess) return e;
    trace_mark(M3_KERNEL_BACKWARD, s, 1);
    count_launch();
    return cudaGetLastError();
}

}  // namespace m3
