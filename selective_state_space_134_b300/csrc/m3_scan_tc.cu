// Chunked prefill of the Mamba-3 recurrence on the sm_100-family tensor cores
// (tcgen05 MMA, accumulators in TMEM, inputs brought in by TMA).
//
// One CTA walks the chunks of one segment of one (b, h) sequence, in order,
// with the N x P fp32 state in registers.  Per chunk of Q tokens (QR = Q R
// rows (t, r); linkstar.cloud/article/869, sections "第一刀" (parallel form),
// "RoPE技巧" and "第三刀" (MIMO)):
//   prologue   chunk-local cumsums cA_t (warp shuffle scan) and phi_t, rotation
//              of B and C by R(-phi_t) into bf16 hi + lo tiles; X^_j = s_j x_j
//              with s_j = exp(cA_e - cA_j) w_j (hi + lo);
//   MMA  S   = C~ B~^T                 (QR x QR, K = N)      score
//   MMA  Yi  = C~ H                    (QR x P,  K = N)      state -> output
//   MMA  Sn  = B~^T X^                 (N x P,   K = QR)     chunk's state contribution
//   epi  Pm  = S o M, M_tj = exp(cA_t - cA_j) w_j (j < t), lambda_t dt_t (j = t)  -> TMEM (bf16 hi+lo)
//   epi  H  <- R(phi_e) [exp(cA_e) H + Sn]                   (fp32 registers)
//   MMA  Ya  = Pm X                    (QR x P, K = QR, A operand read from TMEM)
//   epi  y   = Ya + exp(cA_t) Yi       (fp32 out)
// Every product whose operands are not exact in bf16 (rotated B and C, masked
// scores, the state, scaled x) is formed from bf16 hi + lo parts as
// hi*hi + hi*lo + lo*hi, accumulated in fp32: the outputs are heavy-tailed
// (max |y| ~ 16 rms(y) on these inputs), so one plain bf16 rounding of an
// operand would by itself cost ~3e-2 of rms(y).
//
// Tiles: B~ and C~ are K-major with the 128-byte swizzle (64-column slabs);
// the same B~ bytes serve as the MN-major A operand of the Sn MMA.  X comes
// straight from TMA in the MN-major 128-byte-swizzle layout.  N = 64 uses
// QR = 128 row chunks (M = 128 MMAs); N = 128 uses QR = 64 (M = 64) so that
// tiles, TMA staging and double-buffered X fit in shared memory.
#include "m3_internal.cuh"
#include "m3_tc.cuh"

#include <mutex>

namespace m3 {
namespace {

using namespace tc;

constexpr int kThreads = 256;
constexpr int kP = 64;
constexpr uint32_t kWaitPolls = 1u << 22;   // per mbarrier wait; far above any legal wait
constexpr float kLog2e = 1.4426950408889634f;

template <int N, int R>
struct Cfg {
    static constexpr int QR = (N == 64) ? 128 : 64;    // rows per chunk
    static constexpr int Q = QR / R;                   // tokens per chunk
    static constexpr int K = N / 2;                    // complex pairs
    static constexpr int NSLAB = N / 64;               // 64-column slabs of B~ / C~
    static constexpr int NSEG = 8 / NSLAB;             // token segments of the angle scan
    static constexpr int TPS = Q / NSEG;               // tokens per segment
    static constexpr uint32_t TILE = QR * N * 2;       // one B~ or C~ part
    static constexpr uint32_t XT = QR * kP * 2;        // one X tile
    static constexpr uint32_t HT = N * kP * 2;         // one state tile part
    static constexpr uint32_t RAWB = QR * N * 2;       // TMA staging of B or C
    static constexpr uint32_t RAWT = Q * K * 2;        // TMA staging of theta
    static_assert(Q % NSEG == 0, "token segments must tile the chunk");
    static_assert(K == 32 * NSLAB, "one lane per pair within a slab");
};

// Shared-memory map (byte offsets from a 1024-aligned base).
template <int N, int R, bool OUT>
struct Smem {
    using C = Cfg<N, R>;
    static constexpr uint32_t oBh = 0;
    static constexpr uint32_t oBl = oBh + C::TILE;
    static constexpr uint32_t oCh = oBl + C::TILE;
    static constexpr uint32_t oCl = oCh + (OUT ? C::TILE : 0);
    static constexpr uint32_t oX = oCl + (OUT ? C::TILE : 0);       // 2 buffers
    static constexpr uint32_t oXh = oX + 2 * C::XT;
    static constexpr uint32_t oXl = oXh + C::XT;
    static constexpr uint32_t oHh = oXl + C::XT;
    static constexpr uint32_t oHl = oHh + (OUT ? C::HT : 0);
    static constexpr uint32_t oRawB = oHl + (OUT ? C::HT : 0);
    static constexpr uint32_t oRawC = oRawB + C::RAWB;
    static constexpr uint32_t oRawT = oRawC + (OUT ? C::RAWB : 0);
    static constexpr uint32_t oSmall = ((oRawT + C::RAWT + 127) / 128) * 128;
    // small arrays (floats unless noted)
    static constexpr uint32_t oCA = oSmall;                 // cA in log2 units [Q]
    static constexpr uint32_t oG = oCA + 4 * C::Q;          // lambda dt [Q]
    static constexpr uint32_t oW = oG + 4 * C::Q;           // w [Q]
    static constexpr uint32_t oDT = oW + 4 * C::Q;          // dt [Q]
    static constexpr uint32_t oPart = oDT + 4 * C::Q;       // [NSEG][K]
    static constexpr uint32_t oCos = oPart + 4 * C::NSEG * C::K;
    static constexpr uint32_t oSin = oCos + 4 * C::K;
    static constexpr uint32_t oTot = oSin + 4 * C::K;       // [1 + K] segment totals (pass 1)
    static constexpr uint32_t oBar = ((oTot + 4 * (1 + C::K) + 7) / 8) * 8;   // 3 mbarriers
    static constexpr uint32_t oTmem = oBar + 24;
    static constexpr uint32_t oFlag = oTmem + 4;
    static constexpr uint32_t kBytes = oFlag + 4;
    static constexpr uint32_t kAlloc = kBytes + 1024;       // slack for the 1024-byte alignment
};

// Byte offset of element (row, col) in a 128-byte-swizzled tile of 128-byte rows
// (K-major tiles: col < 64 within a slab; MN-major tiles: col = the MN index).
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t col) {
    return row * 128u + ((((col >> 3) ^ row) & 7u) << 4) + ((col & 7u) << 1);
}

__device__ __forceinline__ void fast_sincos(float x, float *s, float *c) {
    // Cody-Waite reduction by 2 pi (two-constant split), then the hardware sin/cos on [-pi, pi]
    const float n = rintf(x * 0.15915494309189535f);
    float r = fmaf(-n, 6.28318548202514648f, x);
    r = fmaf(-n, -1.7484555314695172e-7f, r);
    __sincosf(r, s, c);
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

struct TcMaps {
    CUtensorMap B, C, X, T;
};

template <int N, int R, bool OUT>
__global__ void __launch_bounds__(kThreads, 1)
tc_segment_kernel(const __grid_constant__ TcMaps maps, ScanArgs a, int seglen, int nseg, int nlaunch,
                  unsigned *status) {
    using Cf = Cfg<N, R>;
    using S = Smem<N, R, OUT>;
    constexpr int QR = Cf::QR, Q = Cf::Q, K = Cf::K, NSLAB = Cf::NSLAB, TPS = Cf::TPS;
    constexpr bool kM64Rows = (QR == 64);   // rows of S / Y use the M = 64 TMEM lane layout
    constexpr bool kM64State = (N == 64);   // rows of Sn use the M = 64 TMEM lane layout
    constexpr uint32_t kTmemCols = OUT ? 512 : 64;
    // TMEM columns
    constexpr uint32_t cS = 0, cYa = 128, cYi = 192, cSn = OUT ? 256 : 0, cPh = 320, cPl = 384;

    extern __shared__ __align__(16) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float *cA2 = reinterpret_cast<float *>(sm + S::oCA);
    float *gv = reinterpret_cast<float *>(sm + S::oG);
    float *wv = reinterpret_cast<float *>(sm + S::oW);
    float *dts = reinterpret_cast<float *>(sm + S::oDT);
    float *part = reinterpret_cast<float *>(sm + S::oPart);
    float *cosE = reinterpret_cast<float *>(sm + S::oCos);
    float *sinE = reinterpret_cast<float *>(sm + S::oSin);
    float *tot = reinterpret_cast<float *>(sm + S::oTot);
    uint64_t *bar_ld = reinterpret_cast<uint64_t *>(sm + S::oBar);
    uint64_t *bar_mma1 = bar_ld + 1;
    uint64_t *bar_mma2 = bar_ld + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + S::oTmem);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(sm + S::oFlag);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int quad = warp & 3, half = warp >> 2;
    const int H = a.H, L = a.L;
    const int g = blockIdx.x % nlaunch, bh = blockIdx.x / nlaunch, b = bh / H, h = bh % H;
    const int t_begin = g * seglen, t_end = min(L, t_begin + seglen);
    const __nv_bfloat16 *dtp = static_cast<const __nv_bfloat16 *>(a.dt);
    const __nv_bfloat16 *Ap = static_cast<const __nv_bfloat16 *>(a.A);
    const __nv_bfloat16 *lp = static_cast<const __nv_bfloat16 *>(a.lam);
    auto tok = [&](int t) { return ((size_t)b * L + t) * H + h; };

    // ---- set-up: barriers, TMEM, state
    if (tid == 0) {
        mbar_init(bar_ld, 1);
        mbar_init(bar_mma1, 1);
        mbar_init(bar_mma2, 1);
        mbar_init_fence();
        *abort_flag = 0;
        tma_prefetch_desc(&maps.B);
        tma_prefetch_desc(&maps.X);
        tma_prefetch_desc(&maps.T);
        if (OUT) tma_prefetch_desc(&maps.C);
    }
    for (int i = tid; i < 1 + K; i += kThreads) tot[i] = 0.f;
    if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;

    auto issue_loads = [&](int s0, int buf) {
        constexpr uint32_t bytes = Cf::RAWB * (OUT ? 2 : 1) + Cf::XT + Cf::RAWT;
        mbar_expect_tx(bar_ld, bytes);
        const int row0 = b * L + s0;
        tma_load_4d(sm + S::oRawB, &maps.B, 0, 0, h, row0, bar_ld);
        if (OUT) tma_load_4d(sm + S::oRawC, &maps.C, 0, 0, h, row0, bar_ld);
        tma_load_4d(sm + S::oX + buf * Cf::XT, &maps.X, 0, 0, h, row0, bar_ld);
        tma_load_3d(sm + S::oRawT, &maps.T, 0, h, row0, bar_ld);
    };
    if (tid == 0 && t_begin < t_end) issue_loads(t_begin, 0);

    // State rows owned by this thread: row n of the N x P state, 32 columns [32 half, +32).
    const bool st_owner = kM64State ? (lane < 16) : true;
    const int st_row = kM64State ? quad * 16 + lane : quad * 32 + lane;
    float hreg[32];
    {
        const int n = st_row;
        if (!OUT || !st_owner) {
#pragma unroll
            for (int j = 0; j < 32; ++j) hreg[j] = 0.f;
        } else if (nseg == 1) {
            const float left0 = (1.f - to_f(lp[tok(0)])) * to_f(dtp[tok(0)]);
            const __nv_bfloat16 *bq = static_cast<const __nv_bfloat16 *>(a.Bprev);
            const __nv_bfloat16 *xq = static_cast<const __nv_bfloat16 *>(a.xprev);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int p = 32 * half + j;
                float v = a.h0 ? a.h0[((size_t)bh * N + n) * kP + p] : 0.f;
                if (bq && xq) {
                    float u = 0.f;
                    for (int r = 0; r < R; ++r)
                        u += to_f(bq[((size_t)bh * R + r) * N + n]) * to_f(xq[((size_t)bh * R + r) * kP + p]);
                    v += left0 * u;
                }
                hreg[j] = v;
            }
        } else {
            const float *src = a.ws_state + (((size_t)bh * nseg + g) * N + n) * kP + 32 * half;
#pragma unroll
            for (int j = 0; j < 32; ++j) hreg[j] = src[j];
        }
    }
    // bf16 hi / lo copy of the state for the C~ H MMA (MN-major, 128-byte swizzle, rows n)
    auto write_state_tile = [&]() {
        if (!OUT || !st_owner) return;
        const int n = st_row;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) split2(hreg[8 * q4 + 2 * e], hreg[8 * q4 + 2 * e + 1], hi[e], lo[e]);
            const uint32_t off = sw128(n, 32 * half + 8 * q4);
            *reinterpret_cast<uint4 *>(sm + S::oHh + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4 *>(sm + S::oHl + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
    };
    write_state_tile();

    auto fail = [&]() {
        *abort_flag = 1;
        atomicOr(status, kStatusTimeout);
    };

    int it = 0;
    for (int s0 = t_begin; s0 < t_end; s0 += Q, ++it) {
        const int Qc = min(Q, t_end - s0), e = Qc - 1, buf = it & 1;
        const bool last_chunk = s0 + Q >= t_end;

        // ---------------- prologue: per-token scalars (plain loads overlap the TMA wait)
        if (tid < Q) {
            float d = 0.f, av = 0.f, gg = 0.f, ww = 0.f;
            if (tid < Qc) {
                const size_t ti = tok(s0 + tid);
                d = to_f(dtp[ti]);
                av = d * to_f(Ap[ti]) * kLog2e;
                const float l = to_f(lp[ti]);
                gg = l * d;
                float nxt = 0.f;
                if (s0 + tid + 1 < L) {
                    const size_t tn = tok(s0 + tid + 1);
                    nxt = (1.f - to_f(lp[tn])) * to_f(dtp[tn]);
                }
                ww = gg + nxt;
            }
            dts[tid] = d;
            cA2[tid] = av;
            gv[tid] = gg;
            wv[tid] = ww;
        }
        if (!mbar_wait(bar_ld, it & 1, kWaitPolls)) fail();
        __syncthreads();
        if (*abort_flag) break;

        const __nv_bfloat16 *rawT = reinterpret_cast<const __nv_bfloat16 *>(sm + S::oRawT);
        const int slab = warp % NSLAB, seg = warp / NSLAB, k = 32 * slab + lane;
        // chunk-local prefix of dt A (one warp, shuffle scan); per-segment angle sums (all warps)
        if (warp == 0) {
            float carry = 0.f;
            for (int base = 0; base < Q; base += 32) {
                float v = (base + lane < Q) ? cA2[base + lane] : 0.f;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float t = __shfl_up_sync(0xffffffffu, v, o);
                    if (lane >= o) v += t;
                }
                v += carry;
                if (base + lane < Q) cA2[base + lane] = v;
                carry = __shfl_sync(0xffffffffu, v, 31);
            }
        }
        {
            float ps = 0.f;
#pragma unroll
            for (int i = 0; i < TPS; ++i) {
                const int t = seg * TPS + i;
                if (t < Qc) ps += dts[t] * __bfloat162float(rawT[t * K + k]);
            }
            part[seg * K + k] = ps;
        }
        __syncthreads();
        if (!OUT && tid < K) {
            float s = 0.f;
            for (int sg = 0; sg < Cf::NSEG; ++sg) s += part[sg * K + tid];
            tot[1 + tid] += s;
        }
        if (!OUT && tid == 0) tot[0] += cA2[e];

        // ---------------- rotation of B (and C) by R(-phi_t), split into bf16 hi + lo
        {
            float phi = 0.f;
            for (int sg = 0; sg < seg; ++sg) phi += part[sg * K + k];
            const uint32_t *rawB = reinterpret_cast<const uint32_t *>(sm + S::oRawB);
            const uint32_t *rawC = reinterpret_cast<const uint32_t *>(sm + S::oRawC);
            const uint32_t slab_off = slab * (QR * 128);
            const uint32_t col = 2 * (lane);   // column within the slab (n % 64), even
#pragma unroll
            for (int i = 0; i < TPS; ++i) {
                const int t = seg * TPS + i;
                float c = 1.f, s = 0.f;
                const bool valid = t < Qc;
                if (valid) {
                    phi += dts[t] * __bfloat162float(rawT[t * K + k]);
                    fast_sincos(phi, &s, &c);
                    if (t == e) {
                        cosE[k] = c;
                        sinE[k] = s;
                    }
                }
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int row = t * R + r;
                    const uint32_t off = slab_off + sw128(row, col);
                    uint32_t hi = 0, lo = 0;
                    if (valid) {
                        const uint32_t v = rawB[(row * N) / 2 + k];
                        const float b0 = bf16_lo_f(v), b1 = bf16_hi_f(v);
                        split2(c * b0 + s * b1, c * b1 - s * b0, hi, lo);
                    }
                    *reinterpret_cast<uint32_t *>(sm + S::oBh + off) = hi;
                    *reinterpret_cast<uint32_t *>(sm + S::oBl + off) = lo;
                    if (OUT) {
                        uint32_t chi = 0, clo = 0;
                        if (valid) {
                            const uint32_t v = rawC[(row * N) / 2 + k];
                            const float c0 = bf16_lo_f(v), c1 = bf16_hi_f(v);
                            split2(c * c0 + s * c1, c * c1 - s * c0, chi, clo);
                        }
                        *reinterpret_cast<uint32_t *>(sm + S::oCh + off) = chi;
                        *reinterpret_cast<uint32_t *>(sm + S::oCl + off) = clo;
                    }
                }
            }
        }
        // ---------------- X^ = s_j x_j (hi + lo); zero the rows past the chunk end in X
        {
            unsigned char *xb = sm + S::oX + buf * Cf::XT;
            const float ce = cA2[e];
            for (int item = tid; item < QR * 8; item += kThreads) {
                const int row = item >> 3, c8 = item & 7, t = row / R;
                const uint32_t off = sw128(row, 8 * c8);
                uint4 hi = make_uint4(0, 0, 0, 0), lo = hi;
                if (t < Qc) {
                    const float sj = fast_exp2(ce - cA2[t]) * wv[t];
                    const uint4 v = *reinterpret_cast<const uint4 *>(xb + off);
                    split2(sj * bf16_lo_f(v.x), sj * bf16_hi_f(v.x), hi.x, lo.x);
                    split2(sj * bf16_lo_f(v.y), sj * bf16_hi_f(v.y), hi.y, lo.y);
                    split2(sj * bf16_lo_f(v.z), sj * bf16_hi_f(v.z), hi.z, lo.z);
                    split2(sj * bf16_lo_f(v.w), sj * bf16_hi_f(v.w), hi.w, lo.w);
                } else if (OUT) {
                    *reinterpret_cast<uint4 *>(xb + off) = make_uint4(0, 0, 0, 0);
                }
                *reinterpret_cast<uint4 *>(sm + S::oXh + off) = hi;
                *reinterpret_cast<uint4 *>(sm + S::oXl + off) = lo;
            }
        }
        fence_proxy_async();
        fence_before();
        __syncthreads();
        fence_after();

        // ---------------- MMAs of this chunk; then prefetch the next chunk's inputs
        if (tid == 0) {
            const uint32_t bh_ = smem_u32(sm + S::oBh), bl_ = smem_u32(sm + S::oBl);
            if (OUT) {
                const uint32_t ch_ = smem_u32(sm + S::oCh), cl_ = smem_u32(sm + S::oCl);
                const uint32_t hh_ = smem_u32(sm + S::oHh), hl_ = smem_u32(sm + S::oHl);
                constexpr uint32_t idS = idesc_bf16(QR, QR, 0, 0);
                constexpr uint32_t idYi = idesc_bf16(QR, kP, 0, 1);
#pragma unroll
                for (int ks = 0; ks < N / 16; ++ks) {
                    // K-major, 128-byte swizzle: slab (ks / 4), 32 bytes per 16-column step inside it
                    const uint32_t ko = (ks / 4) * (QR * 128) + (ks % 4) * 32;
                    const uint64_t dCh = make_desc(ch_ + ko, 16, 1024, kSwizzle128B);
                    const uint64_t dCl = make_desc(cl_ + ko, 16, 1024, kSwizzle128B);
                    const uint64_t dBh = make_desc(bh_ + ko, 16, 1024, kSwizzle128B);
                    const uint64_t dBl = make_desc(bl_ + ko, 16, 1024, kSwizzle128B);
                    mma_ss(tmem + cS, dCh, dBh, idS, ks > 0);
                    mma_ss(tmem + cS, dCh, dBl, idS, 1);
                    mma_ss(tmem + cS, dCl, dBh, idS, 1);
                    // state operand: MN-major (p), K = n rows in 8-row groups of 1024 bytes
                    const uint64_t dHh = make_desc(hh_ + ks * 2048, 0, 1024, kSwizzle128B);
                    const uint64_t dHl = make_desc(hl_ + ks * 2048, 0, 1024, kSwizzle128B);
                    mma_ss(tmem + cYi, dCh, dHh, idYi, ks > 0);
                    mma_ss(tmem + cYi, dCh, dHl, idYi, 1);
                    mma_ss(tmem + cYi, dCl, dHh, idYi, 1);
                }
            }
            {
                const uint32_t xh_ = smem_u32(sm + S::oXh), xl_ = smem_u32(sm + S::oXl);
                constexpr uint32_t idSn = idesc_bf16(N, kP, 1, 1);
#pragma unroll
                for (int ks = 0; ks < QR / 16; ++ks) {
                    // B~ read as the MN-major A operand (M = n in 64-wide slabs, K = rows j)
                    const uint64_t dAh = make_desc(bh_ + ks * 2048, QR * 128, 1024, kSwizzle128B);
                    const uint64_t dAl = make_desc(bl_ + ks * 2048, QR * 128, 1024, kSwizzle128B);
                    const uint64_t dXh = make_desc(xh_ + ks * 2048, 0, 1024, kSwizzle128B);
                    const uint64_t dXl = make_desc(xl_ + ks * 2048, 0, 1024, kSwizzle128B);
                    mma_ss(tmem + cSn, dAh, dXh, idSn, ks > 0);
                    mma_ss(tmem + cSn, dAh, dXl, idSn, 1);
                    mma_ss(tmem + cSn, dAl, dXh, idSn, 1);
                }
            }
            mma_commit(bar_mma1);
            if (!last_chunk) issue_loads(s0 + Q, buf ^ 1);
        }
        if (!mbar_wait(bar_mma1, it & 1, kWaitPolls)) fail();
        fence_after();

        // ---------------- epilogue 1: masked score -> TMEM (bf16 hi + lo); state update
        if (OUT) {
            constexpr int COLS = QR / 2;                      // score columns per thread
            const bool rvalid = kM64Rows ? (lane < 16) : true;
            const int row = kM64Rows ? quad * 16 + lane : quad * 32 + lane;
            const int ti = row / R;
            const float cai = cA2[min(ti, Q - 1)];
            const float gi = gv[min(ti, Q - 1)];
            const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
#pragma unroll
            for (int cc = 0; cc < COLS; cc += 32) {
                uint32_t sv[32];
                tmem_ld32(tmem + lane_base + cS + half * COLS + cc, sv);
                uint32_t ph[16], pl[16];
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    float pm[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int col = half * COLS + cc + j + u, tj = col / R;
                        float m = 0.f;
                        if (tj < ti) m = fast_exp2(cai - cA2[tj]) * wv[tj];
                        else if (tj == ti) m = gi;
                        pm[u] = rvalid ? __uint_as_float(sv[j + u]) * m : 0.f;
                    }
                    split2(pm[0], pm[1], ph[j / 2], pl[j / 2]);
                }
                const uint32_t pcol = (half * COLS + cc) / 2;
                tmem_st16(tmem + lane_base + cPh + pcol, ph);
                tmem_st16(tmem + lane_base + cPl + pcol, pl);
            }
        }
        {
            uint32_t sn[32];
            const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
            tmem_ld32(tmem + lane_base + cSn + 32 * half, sn);
            const float rho = fast_exp2(cA2[e]);
            const int n = st_row, kk = n >> 1;
            const float c = st_owner ? cosE[kk] : 1.f, s = st_owner ? sinE[kk] : 0.f;
            const bool odd = n & 1;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float v = rho * hreg[j] + __uint_as_float(sn[j]);
                const float pv = __shfl_xor_sync(0xffffffffu, v, 1);
                hreg[j] = odd ? fmaf(s, pv, c * v) : fmaf(-s, pv, c * v);
            }
            write_state_tile();
            if (last_chunk && st_owner) {
                float *dst = nullptr;
                if (!OUT) dst = a.ws_state + (((size_t)bh * nseg + g + 1) * N + n) * kP;
                else if (g == nseg - 1 && a.h_out) dst = a.h_out + ((size_t)bh * N + n) * kP;
                if (dst) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4 *>(dst + 32 * half + j) =
                            make_float4(hreg[j], hreg[j + 1], hreg[j + 2], hreg[j + 3]);
                }
            }
        }
        fence_proxy_async();
        fence_before();
        __syncthreads();
        fence_after();

        if (OUT) {
            // ---------------- Ya = Pm X (A operand from TMEM), then y = Ya + exp(cA_t) Yi
            if (tid == 0) {
                const uint32_t xb_ = smem_u32(sm + S::oX + buf * Cf::XT);
                constexpr uint32_t idYa = idesc_bf16(QR, kP, 0, 1);
#pragma unroll
                for (int ks = 0; ks < QR / 16; ++ks) {
                    const uint64_t dX = make_desc(xb_ + ks * 2048, 0, 1024, kSwizzle128B);
                    mma_ts(tmem + cYa, tmem + cPh + ks * 8, dX, idYa, ks > 0);
                    mma_ts(tmem + cYa, tmem + cPl + ks * 8, dX, idYa, 1);
                }
                mma_commit(bar_mma2);
            }
            if (!mbar_wait(bar_mma2, it & 1, kWaitPolls)) fail();
            fence_after();
            {
                const bool rvalid = kM64Rows ? (lane < 16) : true;
                const int row = kM64Rows ? quad * 16 + lane : quad * 32 + lane;
                const int ti = row / R, r = row % R;
                const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
                uint32_t ya[32], yi[32];
                tmem_ld32(tmem + lane_base + cYa + 32 * half, ya);
                tmem_ld32(tmem + lane_base + cYi + 32 * half, yi);
                if (rvalid && ti < Qc) {
                    const float sc = fast_exp2(cA2[ti]);
                    float *yp = static_cast<float *>(a.y) + (tok(s0 + ti) * R + r) * kP + 32 * half;
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4 *>(yp + j) = make_float4(
                            fmaf(sc, __uint_as_float(yi[j]), __uint_as_float(ya[j])),
                            fmaf(sc, __uint_as_float(yi[j + 1]), __uint_as_float(ya[j + 1])),
                            fmaf(sc, __uint_as_float(yi[j + 2]), __uint_as_float(ya[j + 2])),
                            fmaf(sc, __uint_as_float(yi[j + 3]), __uint_as_float(ya[j + 3])));
                }
            }
            fence_before();
            __syncthreads();
            fence_after();
        }
        if (*abort_flag) break;
    }

    // ---------------- segment outputs
    if (!*abort_flag) {
        if (!OUT) {
            float *dst = a.ws_tot + ((size_t)bh * (nseg - 1) + g) * (1 + K);
            for (int i = tid; i < 1 + K; i += kThreads) dst[i] = (i == 0) ? tot[0] / kLog2e : tot[i];
        } else if (g == nseg - 1 && a.Bprev_out && a.xprev_out && L > 0) {
            const size_t tl = tok(L - 1);
            const __nv_bfloat16 *Bm = static_cast<const __nv_bfloat16 *>(a.B);
            const __nv_bfloat16 *xm = static_cast<const __nv_bfloat16 *>(a.x);
            __nv_bfloat16 *bo = static_cast<__nv_bfloat16 *>(a.Bprev_out);
            __nv_bfloat16 *xo = static_cast<__nv_bfloat16 *>(a.xprev_out);
            for (int i = tid; i < R * N; i += kThreads) bo[(size_t)bh * R * N + i] = Bm[tl * R * N + i];
            for (int i = tid; i < R * kP; i += kThreads) xo[(size_t)bh * R * kP + i] = xm[tl * R * kP + i];
        }
    } else if (tid == 0) {
        // a wait gave up: let any outstanding bulk copy land before the CTA's shared memory goes away
        mbar_wait(bar_ld, it & 1, kWaitPolls);
    }
    fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- host side
using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
    static std::once_flag once;
    static EncodeFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(p);
    });
    return fn;
}

// 4-d map over a [b*L][H][R][inner] bf16 tensor, box = {inner, R, 1, Q}
bool map4(CUtensorMap *m, const void *base, int inner, int R, int H, long long rows, int Q, bool swz) {
    EncodeFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)R, (cuuint64_t)H, (cuuint64_t)rows};
    const cuuint64_t strides[3] = {(cuuint64_t)inner * 2, (cuuint64_t)inner * 2 * R, (cuuint64_t)inner * 2 * R * H};
    const cuuint32_t box[4] = {(cuuint32_t)inner, (cuuint32_t)R, 1, (cuuint32_t)Q};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// 3-d map over a [b*L][H][inner] bf16 tensor, box = {inner, 1, Q}
bool map3(CUtensorMap *m, const void *base, int inner, int H, long long rows, int Q) {
    EncodeFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)H, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)inner * 2, (cuuint64_t)inner * 2 * H};
    const cuuint32_t box[3] = {(cuuint32_t)inner, 1, (cuuint32_t)Q};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int N, int R, bool OUT>
cudaError_t launch_pass(const TcMaps &maps, const ScanArgs &a, const ScanPlan &pl, int nlaunch, cudaStream_t s) {
    using Sm = Smem<N, R, OUT>;
    auto kern = tc_segment_kernel<N, R, OUT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Sm::kAlloc);
    if (e != cudaSuccess) return e;
    unsigned *status = device_status_word();
    if (!status) return cudaErrorUnknown;
    const long long grid = (long long)a.batch * a.H * nlaunch;
    const int kid = OUT ? M3_KERNEL_PREFILL_OUTPUT : M3_KERNEL_PREFILL_STATE;
    trace_mark(kid, s, 0);
    kern<<<(unsigned)grid, kThreads, Sm::kAlloc, s>>>(maps, a, pl.seglen, pl.nseg, nlaunch, status);
    trace_mark(kid, s, 1);
    count_launch();
    return cudaGetLastError();
}

template <int N, int R>
cudaError_t run_tc(const ScanArgs &a, const ScanPlan &pl, cudaStream_t s) {
    using Cf = Cfg<N, R>;
    const long long rows = (long long)a.batch * a.L;
    TcMaps maps;
    if (!map4(&maps.B, a.B, N, R, a.H, rows, Cf::Q, false) || !map4(&maps.C, a.C, N, R, a.H, rows, Cf::Q, false) ||
        !map4(&maps.X, a.x, kP, R, a.H, rows, Cf::Q, true) || !map3(&maps.T, a.theta, N / 2, a.H, rows, Cf::Q))
        return cudaErrorInvalidValue;
    cudaError_t e;
    if (pl.nseg > 1) {
        if ((e = launch_pass<N, R, false>(maps, a, pl, pl.nseg - 1, s)) != cudaSuccess) return e;
        if ((e = segment_pass(a, pl, s)) != cudaSuccess) return e;
    }
    return launch_pass<N, R, true>(maps, a, pl, pl.nseg, s);
}

int tc_chunk(int N, int R) { return (N == 64 ? 128 : 64) / R; }

}  // namespace

bool tc_supported(const m3_dims &d) {
    if (d.dtype != M3_BF16 || d.headdim != 64) return false;
    if (d.dstate != 64 && d.dstate != 128) return false;
    if (d.rank != 1 && d.rank != 2 && d.rank != 4 && d.rank != 8) return false;
    if (d.chunk != 0 && d.chunk != tc_chunk(d.dstate, d.rank)) return false;
    if ((long long)d.batch * d.seqlen >= (1LL << 31)) return false;   // TMA row coordinates are int32
    return true;
}

bool tc_plan(const m3_dims &d, int sms, ScanPlan *pl) {
    if (!tc_supported(d)) return false;
    const int Q = tc_chunk(d.dstate, d.rank);
    const long long seqs = (long long)d.batch * d.nheads;
    const int L = d.seqlen;
    int nseg = 1;
    if (seqs > 0 && L > 0 && seqs < (long long)(0.8 * sms)) {
        // fill the SMs (one CTA each); segments of at least 8 chunks
        const int max_seg = (L + 8 * Q - 1) / (8 * Q);
        long long want = (sms + seqs - 1) / seqs;
        nseg = (int)(want < max_seg ? want : max_seg);
        if (nseg < 1) nseg = 1;
    }
    int seglen = L > 0 ? (L + nseg - 1) / nseg : Q;
    seglen = ((seglen + Q - 1) / Q) * Q;
    nseg = L > 0 ? (L + seglen - 1) / seglen : 1;
    pl->Q = Q;
    pl->nseg = nseg;
    pl->seglen = seglen;
    pl->path = kPathTc;
    pl->ws_bytes = scan_workspace_bytes(d.batch, d.nheads, d.dstate, d.headdim, nseg);
    return true;
}

cudaError_t tc_scan(const ScanArgs &a, const ScanPlan &pl, cudaStream_t s) {
#define M3_TC_CASE(NN, RR) \
    if (a.N == NN && a.R == RR) return run_tc<NN, RR>(a, pl, s);
    M3_TC_CASE(64, 1) M3_TC_CASE(64, 2) M3_TC_CASE(64, 4) M3_TC_CASE(64, 8)
    M3_TC_CASE(128, 1) M3_TC_CASE(128, 2) M3_TC_CASE(128, 4) M3_TC_CASE(128, 8)
#undef M3_TC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace m3
