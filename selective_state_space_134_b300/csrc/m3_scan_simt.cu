// Chunked prefill of the Mamba-3 recurrence on plain CUDA cores (fp32 FMA).
//
// This is the generic path: every supported shape and both dtypes, and the
// only path for fp32 inputs (whose 1e-4 tolerance rules out bf16/tf32 tensor
// cores).  One CTA walks the chunks of one segment of one (b, h) sequence in
// order and keeps the N x P fp32 state in shared memory.
//
// Per chunk (tokens s0..e, chunk-local cumulative sums; linkstar.cloud
// article, sections "第一刀" (parallel form) and "RoPE技巧"):
//   cA_t  = sum_{s0<=u<=t} dt_u A_u,        phi_{t,k} = sum_{s0<=u<=t} dt_u theta_{u,k}
//   B~_t  = R(-phi_t) B_t,  C~_t = R(-phi_t) C_t           (2x2 block rotations)
//   y_t   = sum_{j<=t} M_tj (C~_t . B~_j) x_j + exp(cA_t) C~_t^T H
//   M_tj  = exp(cA_t - cA_j) w_j  (j < t),   M_tt = lambda_t dt_t
//   w_j   = lambda_j dt_j + (1 - lambda_{j+1}) dt_{j+1}   (second term 0 at the sequence end)
//   H    <- R(phi_e) [exp(cA_e) H + sum_j exp(cA_e - cA_j) w_j B~_j x_j^T]
// H is the true-frame state entering the chunk, including the left-endpoint
// (beta) term of the chunk's first token.
#include "m3_internal.cuh"

namespace m3 {
namespace {

constexpr int kThreads = 256;

// Shared-memory carve-up, in floats.  Rows of B~ / C~ are padded to N + 1 so
// that threads reading consecutive rows hit different banks.
struct SimtSmem {
    int N, P, Q, R, K, QR, NS;
    size_t oH, oB, oC, oX, oG, ocA, og, ow, odt, ocs, osn, oacc, oiB, oiC, total;
    __host__ __device__ SimtSmem(int Q_, int R_, int N_, int P_, bool out) {
        Q = Q_; R = R_; N = N_; P = P_; K = N / 2; QR = Q * R; NS = N + 1;
        size_t o = 0;
        oH = o;  o += (size_t)N * P;
        oB = o;  o += (size_t)QR * NS;
        oC = o;  o += out ? (size_t)QR * NS : 0;
        oX = o;  o += (size_t)QR * P;
        oG = o;  o += out ? (size_t)QR * QR : 0;
        ocA = o; o += Q;
        og = o;  o += Q;
        ow = o;  o += Q;
        odt = o; o += Q;
        ocs = o; o += (size_t)Q * K;
        osn = o; o += (size_t)Q * K;
        oacc = o; o += 1 + K;        // segment totals (pass 1)
        oiB = o; o += QR;            // BC norm: inverse RMS of the chunk's B rows (carry rows first)
        oiC = o; o += QR;            // ... and of its C rows
        total = o;
    }
};

// Inclusive prefix sum of arr[0..n) by one warp (shuffle scan, 32 at a time).
__device__ void warp_cumsum(float *arr, int n, int lane) {
    float carry = 0.f;
    for (int base = 0; base < n; base += 32) {
        float v = (base + lane < n) ? arr[base + lane] : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            float t = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t;
        }
        v += carry;
        if (base + lane < n) arr[base + lane] = v;
        carry = __shfl_sync(0xffffffffu, v, 31);
    }
}

// OUT = true: pass 3 (outputs).  OUT = false: pass 1 (segment-end state only).
template <typename T, bool OUT>
__global__ void __launch_bounds__(kThreads)
simt_segment_kernel(ScanArgs a, int Q, int seglen, int nseg, int nlaunch) {
    extern __shared__ float sm[];
    const SimtSmem L(Q, a.R, a.N, a.P, OUT);
    float *Hs = sm + L.oH, *Bb = sm + L.oB, *Cb = sm + L.oC, *Xs = sm + L.oX, *G = sm + L.oG;
    float *cA = sm + L.ocA, *gv = sm + L.og, *wv = sm + L.ow, *dts = sm + L.odt;
    float *cs = sm + L.ocs, *sn = sm + L.osn, *acc = sm + L.oacc, *iB = sm + L.oiB, *iC = sm + L.oiC;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int N = a.N, P = a.P, R = a.R, K = N / 2, H = a.H, Lq = a.L, NS = L.NS;
    // blockIdx.x = bh * nlaunch + g  (nlaunch = segments launched per sequence)
    const int g = blockIdx.x % nlaunch, bh = blockIdx.x / nlaunch, b = bh / H, h = bh % H;
    const int t_begin = g * seglen;
    const int t_end = min(Lq, t_begin + seglen);
    const T *x = (const T *)a.x, *Bm = (const T *)a.B, *Cm = (const T *)a.C;
    const T *dtp = (const T *)a.dt, *Ap = (const T *)a.A, *lp = (const T *)a.lam;
    const T *thp = (const T *)a.theta;
    auto tok = [&](int t) { return ((size_t)b * Lq + t) * H + h; };   // index into [b][L][H]

    // ---- state entering the segment
    if (!OUT) {
        for (int i = tid; i < N * P; i += kThreads) Hs[i] = 0.f;
        for (int i = tid; i < 1 + K; i += kThreads) acc[i] = 0.f;
    } else if (nseg == 1) {
        const float left0 = (1.f - to_f(lp[tok(0)])) * to_f(dtp[tok(0)]);
        const T *bq = (const T *)a.Bprev, *xq = (const T *)a.xprev;
        if (a.bc.on && bq && xq) {
            // inverse RMS of the carried B rows (BC normalisation; one warp per row)
            for (int r = warp; r < R; r += kThreads / 32) {
                float ssq = 0.f;
                for (int n = lane; n < N; n += 32) {
                    const float v = to_f(bq[((size_t)bh * R + r) * N + n]);
                    ssq = fmaf(v, v, ssq);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
                if (lane == 0) iB[r] = 1.f / sqrtf(ssq / (float)N + a.bc.eps);
            }
            __syncthreads();
        }
        for (int i = tid; i < N * P; i += kThreads) {
            const int n = i / P, p = i % P;
            float v = a.h0 ? a.h0[(size_t)bh * N * P + i] : 0.f;
            if (bq && xq) {
                float u = 0.f;
                for (int r = 0; r < R; ++r) {
                    float bv = to_f(bq[((size_t)bh * R + r) * N + n]);
                    if (a.bc.on) bv = bc_apply(bv, iB[r], a.bc.wB, a.bc.bB, h, r, R, N, n);
                    u += bv * to_f(xq[((size_t)bh * R + r) * P + p]);
                }
                v += left0 * u;
            }
            Hs[i] = v;
        }
    } else {
        const float *src = a.ws_state + ((size_t)bh * nseg + g) * N * P;
        for (int i = tid; i < N * P; i += kThreads) Hs[i] = src[i];
    }
    __syncthreads();

    for (int s0 = t_begin; s0 < t_end; s0 += Q) {
        const int Qc = min(Q, t_end - s0), QRc = Qc * R, e = Qc - 1;

        // ---- per-token scalars: log-decay, weights
        for (int i = tid; i < Qc; i += kThreads) {
            const size_t ti = tok(s0 + i);
            const float d = to_f(dtp[ti]), l = to_f(lp[ti]);
            dts[i] = d;
            cA[i] = d * to_f(Ap[ti]);
            gv[i] = l * d;
            float nxt = 0.f;
            if (s0 + i + 1 < Lq) {
                const size_t tn = tok(s0 + i + 1);
                nxt = (1.f - to_f(lp[tn])) * to_f(dtp[tn]);
            }
            wv[i] = l * d + nxt;
        }
        __syncthreads();
        if (warp == 0) warp_cumsum(cA, Qc, lane);
        if (a.bc.on) {
            // BC normalisation: inverse RMS of every B (and C) row of the chunk (one warp per row)
            for (int row = warp; row < QRc * (OUT ? 2 : 1); row += kThreads / 32) {
                const bool isC = row >= QRc;
                const int rr = isC ? row - QRc : row, ti = rr / R, r = rr % R;
                const T *src = (isC ? Cm : Bm) + (tok(s0 + ti) * R + r) * N;
                float ssq = 0.f;
                for (int n = lane; n < N; n += 32) {
                    const float v = to_f(src[n]);
                    ssq = fmaf(v, v, ssq);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
                if (lane == 0) (isC ? iC : iB)[rr] = 1.f / sqrtf(ssq / (float)N + a.bc.eps);
            }
        }
        // ---- chunk-local angles, their cos / sin
        for (int k = tid; k < K; k += kThreads) {
            float phi = 0.f;
            for (int i = 0; i < Qc; ++i) {
                phi += dts[i] * to_f(thp[tok(s0 + i) * K + k]);
                float sv, cv;
                sincosf(phi, &sv, &cv);
                cs[i * K + k] = cv;
                sn[i * K + k] = sv;
            }
        }
        __syncthreads();

        // ---- rotate B (and C) by R(-phi_t); stage x
        for (int i = tid; i < QRc * K; i += kThreads) {
            const int row = i / K, k = i % K, ti = row / R, r = row % R;
            const float c = cs[ti * K + k], s = sn[ti * K + k];
            const size_t base = (tok(s0 + ti) * R + r) * N + 2 * k;
            float b0 = to_f(Bm[base]), b1 = to_f(Bm[base + 1]);
            if (a.bc.on) {
                b0 = bc_apply(b0, iB[row], a.bc.wB, a.bc.bB, h, r, R, N, 2 * k);
                b1 = bc_apply(b1, iB[row], a.bc.wB, a.bc.bB, h, r, R, N, 2 * k + 1);
            }
            Bb[row * NS + 2 * k] = c * b0 + s * b1;
            Bb[row * NS + 2 * k + 1] = -s * b0 + c * b1;
            if (OUT) {
                float c0 = to_f(Cm[base]), c1 = to_f(Cm[base + 1]);
                if (a.bc.on) {
                    c0 = bc_apply(c0, iC[row], a.bc.wC, a.bc.bC, h, r, R, N, 2 * k);
                    c1 = bc_apply(c1, iC[row], a.bc.wC, a.bc.bC, h, r, R, N, 2 * k + 1);
                }
                Cb[row * NS + 2 * k] = c * c0 + s * c1;
                Cb[row * NS + 2 * k + 1] = -s * c0 + c * c1;
            }
        }
        for (int i = tid; i < QRc * P; i += kThreads) {
            const int row = i / P, p = i % P, ti = row / R, r = row % R;
            Xs[i] = to_f(x[(tok(s0 + ti) * R + r) * P + p]);
        }
        __syncthreads();

        if (OUT) {
            // ---- masked score G[(t,r),(j,r')] = M_tj (C~_{t,r} . B~_{j,r'})
            for (int i = tid; i < QRc * QRc; i += kThreads) {
                const int rt = i / QRc, rj = i % QRc, ti = rt / R, tj = rj / R;
                float v = 0.f;
                if (tj <= ti) {
                    const float *cr = Cb + rt * NS, *br = Bb + rj * NS;
                    for (int n = 0; n < N; ++n) v += cr[n] * br[n];
                    v *= (tj < ti) ? expf(cA[ti] - cA[tj]) * wv[tj] : gv[ti];
                }
                G[rt * QRc + rj] = v;
            }
            __syncthreads();
            // ---- y = G X + exp(cA_t) C~ H
            for (int i = tid; i < QRc * P; i += kThreads) {
                const int rt = i / P, p = i % P, ti = rt / R, r = rt % R;
                float v = 0.f;
                const int jend = (ti + 1) * R;
                for (int rj = 0; rj < jend; ++rj) v += G[rt * QRc + rj] * Xs[rj * P + p];
                float u = 0.f;
                const float *cr = Cb + rt * NS;
                for (int n = 0; n < N; ++n) u += cr[n] * Hs[n * P + p];
                v += expf(cA[ti]) * u;
                store_y(a.y, (tok(s0 + ti) * R + r) * P + p, v, a.ydtype);
            }
            __syncthreads();   // every read of H above precedes the update below
        }
        // ---- state update (in the chunk-local frame), then turn by phi_e
        const float decay_e = expf(cA[e]);
        for (int i = tid; i < K * P; i += kThreads) {
            const int k = i / P, p = i % P;
            float v0 = decay_e * Hs[(2 * k) * P + p], v1 = decay_e * Hs[(2 * k + 1) * P + p];
            for (int rj = 0; rj < QRc; ++rj) {
                const int tj = rj / R;
                const float wx = expf(cA[e] - cA[tj]) * wv[tj] * Xs[rj * P + p];
                v0 += Bb[rj * NS + 2 * k] * wx;
                v1 += Bb[rj * NS + 2 * k + 1] * wx;
            }
            const float c = cs[e * K + k], s = sn[e * K + k];
            // all reads of Hs for this (k, p) happened above in this thread
            Hs[(2 * k) * P + p] = c * v0 - s * v1;
            Hs[(2 * k + 1) * P + p] = s * v0 + c * v1;
        }
        if (!OUT) {
            if (tid == 0) acc[0] += cA[e];
            for (int k = tid; k < K; k += kThreads) {
                // phi_e = atan2 would lose range; accumulate the plain angle sum instead
                float phi = 0.f;
                for (int i = 0; i < Qc; ++i) phi += dts[i] * to_f(thp[tok(s0 + i) * K + k]);
                acc[1 + k] += phi;
            }
        }
        __syncthreads();
    }

    if (!OUT) {
        float *dst = a.ws_state + ((size_t)bh * nseg + g + 1) * N * P;
        for (int i = tid; i < N * P; i += kThreads) dst[i] = Hs[i];
        float *tot = a.ws_tot + ((size_t)bh * (nseg - 1) + g) * (1 + K);
        for (int i = tid; i < 1 + K; i += kThreads) tot[i] = acc[i];
        return;
    }
    if (g == nseg - 1) {
        if (a.h_out) {
            float *dst = a.h_out + (size_t)bh * N * P;
            for (int i = tid; i < N * P; i += kThreads) dst[i] = Hs[i];
        }
        if (a.Bprev_out && a.xprev_out && Lq > 0) {
            const size_t tl = tok(Lq - 1);
            T *bo = (T *)a.Bprev_out, *xo = (T *)a.xprev_out;
            for (int i = tid; i < R * N; i += kThreads) bo[(size_t)bh * R * N + i] = Bm[tl * R * N + i];
            for (int i = tid; i < R * P; i += kThreads) xo[(size_t)bh * R * P + i] = x[tl * R * P + i];
        }
    }
}

// Pass 2: H'_0 = h0 + (1 - lambda_0) dt_0 B_{-1} x_{-1}^T;
//         H'_{g+1} = exp(cA_g) R(phi_g) H'_g + S_g  (S_g stored in slot g + 1).
template <typename T>
__global__ void segment_pass_kernel(ScanArgs a, int nseg) {
    const int N = a.N, P = a.P, R = a.R, K = N / 2;
    const long long gi = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (gi >= (long long)a.batch * a.H * K * P) return;
    const int bh = (int)(gi / (K * P)), i = (int)(gi % (K * P)), b = bh / a.H, h = bh % a.H;
    const int k = i / P, p = i % P;
    const T *dtp = (const T *)a.dt, *lp = (const T *)a.lam;
    const size_t t0 = ((size_t)b * a.L) * a.H + h;
    float h0v = 0.f, h1v = 0.f;
    if (a.h0) {
        h0v = a.h0[((size_t)bh * N + 2 * k) * P + p];
        h1v = a.h0[((size_t)bh * N + 2 * k + 1) * P + p];
    }
    if (a.Bprev && a.xprev) {
        const float left0 = (1.f - to_f(lp[t0])) * to_f(dtp[t0]);
        const T *bq = (const T *)a.Bprev, *xq = (const T *)a.xprev;
        float u0 = 0.f, u1 = 0.f;
        for (int r = 0; r < R; ++r) {
            const float xv = to_f(xq[((size_t)bh * R + r) * P + p]);
            const T *row = bq + ((size_t)bh * R + r) * N;
            float q0 = to_f(row[2 * k]), q1 = to_f(row[2 * k + 1]);
            if (a.bc.on) {   // BC normalisation of the carried B row (this thread sums it itself)
                float ssq = 0.f;
                for (int n = 0; n < N; ++n) ssq = fmaf(to_f(row[n]), to_f(row[n]), ssq);
                const float inv = 1.f / sqrtf(ssq / (float)N + a.bc.eps);
                q0 = bc_apply(q0, inv, a.bc.wB, a.bc.bB, bh % a.H, r, R, N, 2 * k);
                q1 = bc_apply(q1, inv, a.bc.wB, a.bc.bB, bh % a.H, r, R, N, 2 * k + 1);
            }
            u0 += q0 * xv;
            u1 += q1 * xv;
        }
        h0v += left0 * u0;
        h1v += left0 * u1;
    }
    float *st = a.ws_state + (size_t)bh * nseg * N * P;
    st[(2 * k) * P + p] = h0v;
    st[(2 * k + 1) * P + p] = h1v;
    for (int g = 0; g + 1 < nseg; ++g) {
        const float *tot = a.ws_tot + ((size_t)bh * (nseg - 1) + g) * (1 + K);
        const float rho = expf(tot[0]);
        float s, c;
        sincosf(tot[1 + k], &s, &c);
        float *slot = st + (size_t)(g + 1) * N * P;
        const float n0 = rho * (c * h0v - s * h1v) + slot[(2 * k) * P + p];
        const float n1 = rho * (s * h0v + c * h1v) + slot[(2 * k + 1) * P + p];
        slot[(2 * k) * P + p] = n0;
        slot[(2 * k + 1) * P + p] = n1;
        h0v = n0;
        h1v = n1;
    }
}

template <typename T>
cudaError_t launch_simt(const ScanArgs &a, const ScanPlan &pl, cudaStream_t s) {
    const long long bh = (long long)a.batch * a.H;
    if (pl.nseg > 1) {
        const SimtSmem l1(pl.Q, a.R, a.N, a.P, false);
        const size_t bytes1 = l1.total * sizeof(float);
        auto k1 = simt_segment_kernel<T, false>;
        cudaError_t err = allow_dynamic_smem<simt_segment_kernel<T, false>>(bytes1);
        if (err != cudaSuccess) return err;
        trace_mark(M3_KERNEL_PREFILL_STATE, s, 0);
        k1<<<(unsigned)(bh * (pl.nseg - 1)), kThreads, bytes1, s>>>(a, pl.Q, pl.seglen, pl.nseg, pl.nseg - 1);
        trace_mark(M3_KERNEL_PREFILL_STATE, s, 1);
        count_launch();
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
        if ((err = segment_pass(a, pl, s)) != cudaSuccess) return err;
    }
    const SimtSmem l3(pl.Q, a.R, a.N, a.P, true);
    const size_t bytes3 = l3.total * sizeof(float);
    auto k3 = simt_segment_kernel<T, true>;
    cudaError_t err = allow_dynamic_smem<simt_segment_kernel<T, true>>(bytes3);
    if (err != cudaSuccess) return err;
    trace_mark(M3_KERNEL_PREFILL_OUTPUT, s, 0);
    k3<<<(unsigned)(bh * pl.nseg), kThreads, bytes3, s>>>(a, pl.Q, pl.seglen, pl.nseg, pl.nseg);
    trace_mark(M3_KERNEL_PREFILL_OUTPUT, s, 1);
    count_launch();
    return cudaGetLastError();
}

}  // namespace

size_t scan_workspace_bytes(int batch, int H, int N, int P, int nseg) {
    if (nseg <= 1) return 0;
    const size_t bh = (size_t)batch * H;
    const size_t state = bh * nseg * N * P * sizeof(float);
    const size_t tot = bh * (nseg - 1) * (1 + N / 2) * sizeof(float);
    return ((state + 255) / 256) * 256 + tot;
}

bool simt_plan(const m3_dims &d, int sms, ScanPlan *pl) {
    pl->bal = 0;
    if (d.ngroups > 0 && d.ngroups != d.nheads) return false;   // grouped B / C: tensor-core path only
    const int R = d.rank, N = d.dstate, P = d.headdim;
    const size_t smem_cap = 200 * 1024;
    int Q = d.chunk;
    if (Q > 0) {
        if (Q * R > 128 || SimtSmem(Q, R, N, P, true).total * 4 > smem_cap) return false;
    } else {
        Q = 64 / R > 0 ? 64 / R : 1;
        while (Q > 1 && SimtSmem(Q, R, N, P, true).total * 4 > smem_cap) Q /= 2;
        if (SimtSmem(Q, R, N, P, true).total * 4 > smem_cap) return false;
    }
    const long long seqs = (long long)d.batch * d.nheads;
    const int L = d.seqlen;
    int nseg = 1;
    if (seqs > 0 && L > 0) {
        const long long target = 2LL * (sms > 0 ? sms : 148);
        const int max_seg = (L + 4 * Q - 1) / (4 * Q);        // segments of at least 4 chunks
        long long want = (target + seqs - 1) / seqs;
        nseg = (int)(want < max_seg ? want : max_seg);
        if (nseg < 1) nseg = 1;
    }
    int seglen = L > 0 ? (L + nseg - 1) / nseg : Q;
    seglen = ((seglen + Q - 1) / Q) * Q;
    nseg = L > 0 ? (L + seglen - 1) / seglen : 1;
    pl->Q = Q;
    pl->nseg = nseg;
    pl->nsub = 1;
    pl->seglen = seglen;
    pl->path = kPathSimt;
    pl->ws_bytes = scan_workspace_bytes(d.batch, d.nheads, N, P, nseg);
    return true;
}

cudaError_t simt_scan(const ScanArgs &a, const ScanPlan &pl, cudaStream_t s) {
    return a.dtype == M3_F32 ? launch_simt<float>(a, pl, s) : launch_simt<__nv_bfloat16>(a, pl, s);
}

cudaError_t segment_pass(const ScanArgs &a, const ScanPlan &pl, cudaStream_t s) {
    const long long total = (long long)a.batch * a.H * (a.N / 2) * a.P;
    const unsigned grid = (unsigned)((total + 127) / 128);
    trace_mark(M3_KERNEL_SEGMENT_PASS, s, 0);
    if (a.dtype == M3_F32)
        segment_pass_kernel<float><<<grid, 128, 0, s>>>(a, pl.nseg);
    else
        segment_pass_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(a, pl.nseg);
    trace_mark(M3_KERNEL_SEGMENT_PASS, s, 1);
    count_launch();
    return cudaGetLastError();
}

}  // namespace m3
