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
#include "m3_internal.cuh"

namespace m3 {
namespace {

constexpr int kBwdThreads = 512;
constexpr int kBwdWarps = kBwdThreads / 32;

// Shared-memory carve-up (floats); row-major tiles padded by one column against bank conflicts
// (the N x P tiles too: several contractions walk their rows n across the threads of a warp).
struct BwdSmem {
    int Q, R, N, P, K, QR, NS, PS, QS;
    size_t oD, oDt, oH, oH2, oB, oC, oX, oY, oS, oZ, oT1, oT2, odM;
    size_t odt, oA, olam, olamn, odtn, ocA, ow, og, os, oe, odcA, odw, odg, ods;
    size_t ocs, osn, odph, oth, ored, total;
    __host__ __device__ BwdSmem(int Q_, int R_, int N_, int P_) {
        Q = Q_; R = R_; N = N_; P = P_; K = N / 2; QR = Q * R; NS = N + 1; PS = P + 1; QS = QR + 1;
        size_t o = 0;
        oD = o;  o += (size_t)N * PS;       // D (true frame); in pass 1 the running state
        oDt = o; o += (size_t)N * PS;       // D~ = R(-phi_e) D
        oH = o;  o += (size_t)N * PS;       // H'_c
        oH2 = o; o += (size_t)N * PS;       // H'_{c+1}
        oB = o;  o += (size_t)QR * NS;      // B~
        oC = o;  o += (size_t)QR * NS;      // C~
        oX = o;  o += (size_t)QR * PS;      // x
        oY = o;  o += (size_t)QR * PS;      // dy
        oS = o;  o += (size_t)QR * QS;      // S, then M o S
        oZ = o;  o += (size_t)QR * QS;      // Z, then M o Z
        oT1 = o; o += (size_t)QR * PS;      // B~ D~
        oT2 = o; o += (size_t)QR * NS;      // dY H'^T
        odM = o; o += (size_t)Q * Q;        // dM per token pair
        odt = o; o += Q; oA = o; o += Q; olam = o; o += Q; olamn = o; o += Q; odtn = o; o += Q;
        ocA = o; o += Q; ow = o; o += Q; og = o; o += Q; os = o; o += Q; oe = o; o += Q;
        odcA = o; o += Q; odw = o; o += Q; odg = o; o += Q; ods = o; o += Q;
        ocs = o; o += (size_t)Q * K; osn = o; o += (size_t)Q * K; odph = o; o += (size_t)Q * K;
        oth = o; o += (size_t)Q * K;
        ored = o; o += kBwdWarps;           // per-warp partial sums
        total = o;
    }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <typename T>
__global__ void __launch_bounds__(kBwdThreads, 1)
scan_bwd_kernel(BwdArgs a, int Q) {
    extern __shared__ float sm[];
    const BwdSmem Lo(Q, a.R, a.N, a.P);
    const int N = a.N, P = a.P, R = a.R, K = N / 2, H = a.H, L = a.L, NS = Lo.NS, PS = Lo.PS, QS = Lo.QS;
    float *Dm = sm + Lo.oD, *Dt = sm + Lo.oDt, *Hc = sm + Lo.oH, *Hn = sm + Lo.oH2;
    float *Bt = sm + Lo.oB, *Ct = sm + Lo.oC, *Xs = sm + Lo.oX, *Ys = sm + Lo.oY;
    float *Sm = sm + Lo.oS, *Zm = sm + Lo.oZ, *T1 = sm + Lo.oT1, *T2 = sm + Lo.oT2, *dMt = sm + Lo.odM;
    float *vdt = sm + Lo.odt, *vA = sm + Lo.oA, *vl = sm + Lo.olam, *vln = sm + Lo.olamn, *vdtn = sm + Lo.odtn;
    float *cA = sm + Lo.ocA, *wv = sm + Lo.ow, *gv = sm + Lo.og, *sv = sm + Lo.os, *ev = sm + Lo.oe;
    float *dcA = sm + Lo.odcA, *dwv = sm + Lo.odw, *dgv = sm + Lo.odg, *dsv = sm + Lo.ods;
    float *cs = sm + Lo.ocs, *sn = sm + Lo.osn, *dph = sm + Lo.odph, *thv = sm + Lo.oth, *red = sm + Lo.ored;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int bh = blockIdx.x, b = bh / H, h = bh % H;
    const int nc = (L + Q - 1) / Q;
    const T *xg = static_cast<const T *>(a.x), *Bg = static_cast<const T *>(a.B), *Cg = static_cast<const T *>(a.C);
    const T *dtg = static_cast<const T *>(a.dt), *Ag = static_cast<const T *>(a.A), *lg = static_cast<const T *>(a.lam);
    const T *thg = static_cast<const T *>(a.theta);
    auto tok = [&](int t) { return ((size_t)b * L + t) * H + h; };
    float *ckpt = a.ws + (size_t)bh * (nc + 1) * N * P;   // H'_c, c = 0..nc

    // Loads the scalars, angles (cos / sin of the chunk-local phi) and rotated B (and C), x of the
    // chunk at s0 into shared memory; Qc tokens.
    auto load_chunk = [&](int s0, int Qc, bool withC) {
        for (int i = tid; i < Q; i += kBwdThreads) {
            float d = 0.f, av = 0.f, l = 0.f, ln = 1.f, dn = 0.f;
            if (i < Qc) {
                const size_t ti = tok(s0 + i);
                d = to_f(dtg[ti]);
                av = to_f(Ag[ti]);
                l = to_f(lg[ti]);
                if (s0 + i + 1 < L) {
                    ln = to_f(lg[tok(s0 + i + 1)]);
                    dn = to_f(dtg[tok(s0 + i + 1)]);
                }
            }
            vdt[i] = d; vA[i] = av; vl[i] = l; vln[i] = ln; vdtn[i] = dn;
            cA[i] = d * av;
        }
        for (int i = tid; i < Q * K; i += kBwdThreads) {
            const int t = i / K, k = i % K;
            thv[i] = t < Qc ? to_f(thg[tok(s0 + t) * K + k]) : 0.f;
        }
        __syncthreads();
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
        for (int i = tid; i < Q * K; i += kBwdThreads) {   // chunk-local angle of token t, pair k
            const int t = i / K, k = i % K;
            float phi = 0.f;
            for (int u = 0; u <= t; ++u) phi = fmaf(vdt[u], thv[u * K + k], phi);
            float s, c;
            sincosf(phi, &s, &c);
            cs[i] = c;
            sn[i] = s;
        }
        __syncthreads();
        const int e = Qc - 1;
        for (int i = tid; i < Q; i += kBwdThreads) {
            const float w = vl[i] * vdt[i] + (1.f - vln[i]) * vdtn[i];
            wv[i] = i < Qc ? w : 0.f;
            gv[i] = i < Qc ? vl[i] * vdt[i] : 0.f;
            sv[i] = i < Qc ? expf(cA[e] - cA[i]) * w : 0.f;
            ev[i] = i < Qc ? expf(cA[i]) : 0.f;
        }
        for (int i = tid; i < Q * R * K; i += kBwdThreads) {
            const int row = i / K, k = i % K, t = row / R, r = row % R;
            float b0 = 0.f, b1 = 0.f, c0 = 0.f, c1 = 0.f;
            if (t < Qc) {
                const size_t base = (tok(s0 + t) * R + r) * N + 2 * k;
                b0 = to_f(Bg[base]);
                b1 = to_f(Bg[base + 1]);
                if (withC) {
                    c0 = to_f(Cg[base]);
                    c1 = to_f(Cg[base + 1]);
                }
            }
            const float c = cs[t * K + k], s = sn[t * K + k];
            Bt[row * NS + 2 * k] = c * b0 + s * b1;       // R(-phi) applied to the pair
            Bt[row * NS + 2 * k + 1] = -s * b0 + c * b1;
            Ct[row * NS + 2 * k] = c * c0 + s * c1;
            Ct[row * NS + 2 * k + 1] = -s * c0 + c * c1;
        }
        for (int i = tid; i < Q * R * P; i += kBwdThreads) {
            const int row = i / P, p = i % P, t = row / R, r = row % R;
            Xs[row * PS + p] = t < Qc ? to_f(xg[(tok(s0 + t) * R + r) * P + p]) : 0.f;
        }
        __syncthreads();
    };

    // ================================================================ pass 1: checkpoints
    {
        const float *h0 = a.h0 ? a.h0 + (size_t)bh * N * P : nullptr;
        const T *bq = static_cast<const T *>(a.Bprev), *xq = static_cast<const T *>(a.xprev);
        const float left0 = L > 0 ? (1.f - to_f(lg[tok(0)])) * to_f(dtg[tok(0)]) : 0.f;
        for (int i = tid; i < N * P; i += kBwdThreads) {
            const int n = i / P, p = i % P;
            float v = h0 ? h0[i] : 0.f;
            if (bq && xq) {
                float u = 0.f;
                for (int r = 0; r < R; ++r)
                    u += to_f(bq[((size_t)bh * R + r) * N + n]) * to_f(xq[((size_t)bh * R + r) * P + p]);
                v += left0 * u;
            }
            Dm[n * PS + p] = v;
            ckpt[i] = v;
        }
        __syncthreads();
        for (int c = 0; c < nc; ++c) {
            const int s0 = c * Q, Qc = min(Q, L - s0), e = Qc - 1;
            load_chunk(s0, Qc, false);
            const float de = expf(cA[e]);
            float *dst = ckpt + (size_t)(c + 1) * N * P;
            for (int i = tid; i < K * P; i += kBwdThreads) {
                const int k = i / P, p = i % P;
                float v0 = de * Dm[(2 * k) * PS + p], v1 = de * Dm[(2 * k + 1) * PS + p];
                for (int row = 0; row < Qc * R; ++row) {
                    const float wx = sv[row / R] * Xs[row * PS + p];
                    v0 = fmaf(Bt[row * NS + 2 * k], wx, v0);
                    v1 = fmaf(Bt[row * NS + 2 * k + 1], wx, v1);
                }
                const float cc = cs[e * K + k], ss = sn[e * K + k];
                const float n0 = cc * v0 - ss * v1, n1 = ss * v0 + cc * v1;
                Dm[(2 * k) * PS + p] = n0;
                Dm[(2 * k + 1) * PS + p] = n1;
                dst[(2 * k) * P + p] = n0;
                dst[(2 * k + 1) * P + p] = n1;
            }
            __syncthreads();
        }
    }

    // ================================================================ pass 2: gradients
    for (int i = tid; i < N * P; i += kBwdThreads)
        Dm[(i / P) * PS + i % P] = a.dh_out ? a.dh_out[(size_t)bh * N * P + i] : 0.f;
    __syncthreads();
    for (int c = nc - 1; c >= 0; --c) {
        const int s0 = c * Q, Qc = min(Q, L - s0), e = Qc - 1, QRc = Qc * R;
        load_chunk(s0, Qc, true);
        for (int i = tid; i < N * P; i += kBwdThreads) {
            Hc[(i / P) * PS + i % P] = ckpt[(size_t)c * N * P + i];
            Hn[(i / P) * PS + i % P] = ckpt[(size_t)(c + 1) * N * P + i];
        }
        for (int i = tid; i < Q * R * P; i += kBwdThreads) {
            const int row = i / P, p = i % P, t = row / R, r = row % R;
            Ys[row * PS + p] = t < Qc ? a.dy[(tok(s0 + t) * R + r) * P + p] : 0.f;
        }
        for (int i = tid; i < Q; i += kBwdThreads) {
            dcA[i] = 0.f;
            dwv[i] = 0.f;
            dgv[i] = 0.f;
            dsv[i] = 0.f;
        }
        // D~ = R(-phi_e) D, and the angle gradient of the turn R(phi_e): <D, J H'_{c+1}> per pair
        for (int i = tid; i < K * P; i += kBwdThreads) {
            const int k = i / P, p = i % P;
            const float cc = cs[e * K + k], ss = sn[e * K + k];
            const float d0 = Dm[(2 * k) * PS + p], d1 = Dm[(2 * k + 1) * PS + p];
            Dt[(2 * k) * PS + p] = cc * d0 + ss * d1;
            Dt[(2 * k + 1) * PS + p] = -ss * d0 + cc * d1;
        }
        for (int i = tid; i < Q * K; i += kBwdThreads) dph[i] = 0.f;
        __syncthreads();
        for (int k = warp; k < K; k += kBwdWarps) {
            float v = 0.f;
            for (int p = lane; p < P; p += 32)
                v += Dm[(2 * k + 1) * PS + p] * Hn[(2 * k) * PS + p] - Dm[(2 * k) * PS + p] * Hn[(2 * k + 1) * PS + p];
            v = warp_sum(v);
            if (lane == 0) dph[e * K + k] += v;
        }
        // S = C~ B~^T and Z = dY X^T over the chunk's rows
        for (int i = tid; i < QRc * QRc; i += kBwdThreads) {
            const int rt = i / QRc, rj = i % QRc;
            float s = 0.f, z = 0.f;
            if (rj / R <= rt / R) {
                for (int n = 0; n < N; ++n) s = fmaf(Ct[rt * NS + n], Bt[rj * NS + n], s);
                for (int p = 0; p < P; ++p) z = fmaf(Ys[rt * PS + p], Xs[rj * PS + p], z);
            }
            Sm[rt * QS + rj] = s;
            Zm[rt * QS + rj] = z;
        }
        // B~ D~ (rows x P) and dY H'^T (rows x N)
        for (int i = tid; i < QRc * P; i += kBwdThreads) {
            const int row = i / P, p = i % P;
            float v = 0.f;
            for (int n = 0; n < N; ++n) v = fmaf(Bt[row * NS + n], Dt[n * PS + p], v);
            T1[row * PS + p] = v;
        }
        for (int i = tid; i < QRc * N; i += kBwdThreads) {
            const int row = i / N, n = i % N;
            float v = 0.f;
            for (int p = 0; p < P; ++p) v = fmaf(Ys[row * PS + p], Hc[n * PS + p], v);
            T2[row * NS + n] = v;
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
            const float m = j < t ? expf(cA[t] - cA[j]) * wv[j] : (j == t ? gv[t] : 0.f);
            Sm[rt * QS + rj] *= m;
            Zm[rt * QS + rj] *= m;
        }
        // token scalars: mask terms (dcA, dw, dg) and the inter-chunk and state terms
        for (int t = warp; t < Qc; t += kBwdWarps) {
            float rowv = 0.f, colv = 0.f, dwj = 0.f;
            for (int j = lane; j < Qc; j += 32) {
                if (j < t) rowv += dMt[t * Q + j] * expf(cA[t] - cA[j]) * wv[j];   // d cA_t
                if (j > t) {
                    const float f = expf(cA[j] - cA[t]);
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
                for (int n = lane; n < N; n += 32) yi += Ct[row * NS + n] * T2[row * NS + n];
                for (int p = lane; p < P; p += 32) dsum += Xs[row * PS + p] * T1[row * PS + p];
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
            for (int i = tid; i < N * P; i += kBwdThreads) {
                const int q = (i / P) * PS + i % P;
                v += Dt[q] * Hc[q];
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
        // dX = (M o S)^T dY + diag(s) B~ D~  (the carry out adds to the sequence's last token)
        for (int i = tid; i < QRc * P; i += kBwdThreads) {
            const int rj = i / P, p = i % P, j = rj / R, r = rj % R;
            float v = sv[j] * T1[rj * PS + p];
            for (int rt = rj - r; rt < QRc; ++rt) v = fmaf(Sm[rt * QS + rj], Ys[rt * PS + p], v);
            if (s0 + j == L - 1 && a.dxprev_out) v += a.dxprev_out[((size_t)bh * R + r) * P + p];
            a.dx[(tok(s0 + j) * R + r) * P + p] = v;
        }
        // dB~ = (M o Z)^T C~ + diag(s) X D~^T and dC~ = (M o Z) B~ + diag(e^{cA}) dY H'^T, pair by pair;
        // they are un-rotated as they are formed, and the angle gradients gather
        // dphi_{t,k} += dv0 v1 - dv1 v0 over the B~ and C~ rows of token t
        for (int i = tid; i < QRc * K; i += kBwdThreads) {
            const int rj = i / K, k = i % K, j = rj / R, r = rj % R;
            // dB~ entries 2k, 2k + 1 of row rj
            float b0 = 0.f, b1 = 0.f, xd0 = 0.f, xd1 = 0.f;
            for (int rt = rj - r; rt < QRc; ++rt) {
                const float m = Zm[rt * QS + rj];
                b0 = fmaf(m, Ct[rt * NS + 2 * k], b0);
                b1 = fmaf(m, Ct[rt * NS + 2 * k + 1], b1);
            }
            for (int p = 0; p < P; ++p) {
                xd0 = fmaf(Xs[rj * PS + p], Dt[(2 * k) * PS + p], xd0);
                xd1 = fmaf(Xs[rj * PS + p], Dt[(2 * k + 1) * PS + p], xd1);
            }
            b0 = fmaf(sv[j], xd0, b0);
            b1 = fmaf(sv[j], xd1, b1);
            // dC~ entries 2k, 2k + 1 of row rj (as the row index t)
            float c0 = 0.f, c1 = 0.f;
            for (int rr = 0; rr < (j + 1) * R; ++rr) {
                const float m = Zm[rj * QS + rr];
                c0 = fmaf(m, Bt[rr * NS + 2 * k], c0);
                c1 = fmaf(m, Bt[rr * NS + 2 * k + 1], c1);
            }
            c0 = fmaf(ev[j], T2[rj * NS + 2 * k], c0);
            c1 = fmaf(ev[j], T2[rj * NS + 2 * k + 1], c1);
            // angle gradient of the rotations R(-phi_j) of B~ and C~
            const float bt0 = Bt[rj * NS + 2 * k], bt1 = Bt[rj * NS + 2 * k + 1];
            const float ct0 = Ct[rj * NS + 2 * k], ct1 = Ct[rj * NS + 2 * k + 1];
            atomicAdd(&dph[j * K + k], b0 * bt1 - b1 * bt0 + c0 * ct1 - c1 * ct0);
            // un-rotate: dB = R(phi) dB~
            const float cc = cs[j * K + k], ss = sn[j * K + k];
            float db0 = cc * b0 - ss * b1, db1 = ss * b0 + cc * b1;
            const float dc0 = cc * c0 - ss * c1, dc1 = ss * c0 + cc * c1;
            if (s0 + j == L - 1 && a.dBprev_out) {
                db0 += a.dBprev_out[((size_t)bh * R + r) * N + 2 * k];
                db1 += a.dBprev_out[((size_t)bh * R + r) * N + 2 * k + 1];
            }
            const size_t base = (tok(s0 + j) * R + r) * N + 2 * k;
            a.dB[base] = db0;
            a.dB[base + 1] = db1;
            a.dC[base] = dc0;
            a.dC[base + 1] = dc1;
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
            for (int k = lane; k < K; k += 32) thsum = fmaf(thv[u * K + k], dph[u * K + k], thsum);
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
        // D <- e^{cA_e} D~ + C~^T diag(e^{cA}) dY
        const float de = expf(cA[e]);
        for (int i = tid; i < N * P; i += kBwdThreads) {
            const int n = i / P, p = i % P;
            float v = de * Dt[n * PS + p];
            for (int row = 0; row < QRc; ++row) v = fmaf(Ct[row * NS + n] * ev[row / R], Ys[row * PS + p], v);
            Dm[n * PS + p] = v;
        }
        __syncthreads();
    }

    // ================================================================ initial state and carry
    // H'_0 = h0 + left_0 B_{-1} x_{-1}^T: dh0 = D; d left_0 = <D, B_{-1} x_{-1}^T>
    if (a.dh0)
        for (int i = tid; i < N * P; i += kBwdThreads) a.dh0[(size_t)bh * N * P + i] = Dm[(i / P) * PS + i % P];
    const T *bq = static_cast<const T *>(a.Bprev), *xq = static_cast<const T *>(a.xprev);
    if (bq && xq) {
        const float d0 = to_f(dtg[tok(0)]), l0 = to_f(lg[tok(0)]), left0 = (1.f - l0) * d0;
        float dl = 0.f;
        for (int i = tid; i < N * P; i += kBwdThreads) {
            const int n = i / P, p = i % P;
            float u = 0.f;
            for (int r = 0; r < R; ++r)
                u += to_f(bq[((size_t)bh * R + r) * N + n]) * to_f(xq[((size_t)bh * R + r) * P + p]);
            dl = fmaf(Dm[n * PS + p], u, dl);
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
                for (int p = 0; p < P; ++p) v = fmaf(Dm[n * PS + p], to_f(xq[((size_t)bh * R + r) * P + p]), v);
                a.dBprev[(size_t)bh * R * N + i] = left0 * v;
            }
        if (a.dxprev)
            for (int i = tid; i < R * P; i += kBwdThreads) {
                const int r = i / P, p = i % P;
                float v = 0.f;
                for (int n = 0; n < N; ++n) v = fmaf(Dm[n * PS + p], to_f(bq[((size_t)bh * R + r) * N + n]), v);
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

// Tokens per chunk: 32 rows (t, r) per chunk, 16 when the four N x P state tiles are large (so that
// the shared memory stays within one CTA's 227 KB).
int bwd_chunk(int N, int P, int R) {
    const int rows = N * P > 4096 ? 16 : 32;
    return rows / R > 0 ? rows / R : 1;
}

size_t bwd_smem_bytes(int N, int P, int R) { return BwdSmem(bwd_chunk(N, P, R), R, N, P).total * sizeof(float); }

size_t bwd_workspace_bytes(int batch, int H, int L, int N, int P, int R) {
    const int Q = bwd_chunk(N, P, R);
    const size_t nc = (size_t)(L + Q - 1) / Q;
    return (size_t)batch * H * (nc + 1) * N * P * sizeof(float);
}

cudaError_t scan_bwd(const BwdArgs &a, cudaStream_t s) {
    const int Q = bwd_chunk(a.N, a.P, a.R);
    const size_t smem = bwd_smem_bytes(a.N, a.P, a.R);
    const unsigned grid = (unsigned)((long long)a.batch * a.H);
    if (grid == 0 || a.L == 0) return cudaSuccess;
    cudaError_t e;
    trace_mark(M3_KERNEL_BACKWARD, s, 0);
    if (a.dtype == M3_F32) {
        if ((e = allow_dynamic_smem<scan_bwd_kernel<float>>(smem)) != cudaSuccess) return e;
        scan_bwd_kernel<float><<<grid, kBwdThreads, smem, s>>>(a, Q);
    } else {
        if ((e = allow_dynamic_smem<scan_bwd_kernel<__nv_bfloat16>>(smem)) != cudaSuccess) return e;
        scan_bwd_kernel<__nv_bfloat16><<<grid, kBwdThreads, smem, s>>>(a, Q);
    }
    trace_mark(M3_KERNEL_BACKWARD, s, 1);
    count_launch();
    return cudaGetLastError();
}

}  // namespace m3
