// Kernel and launch templates of the tensor-core prefill, included by the translation units that
// instantiate them (one per state size N and BC variant, so that they compile in parallel).
#pragma once
// Chunked prefill of the Mamba-3 recurrence on the sm_100-family tensor cores
// (tcgen05 MMA with TMEM accumulators, operands brought in by TMA), as a
// warp-specialised pipeline.
//
// One CTA walks the chunks of one segment of one (b, h) sequence in order.
// Per chunk of Q tokens (QR = Q R rows (t, r); linkstar.cloud/article/869,
// sections "第一刀" (parallel form), "RoPE技巧" and "第三刀" (MIMO)):
//   prologue  chunk-local cumsums cA_t (warp shuffle scan) and phi_t; B and C
//             turned by R(-phi_t) in place into fp16 tiles; X^_j = s_j x_j with
//             s_j = exp(cA_e - cA_j) w_j; mask column factors
//   MMA 1     S  = C~ B~^T        (QR x QR, K = N)    score
//             Yi = C~ H           (QR x P,  K = N)    state -> output
//             Sn = B~^T X^        (N x P,   K = QR)   the chunk's state contribution
//   epilogue  P = S o M, M_tj = exp(cA_t - cA_j) w_j (j < t), lambda_t dt_t (j = t),
//             into TMEM as fp16;  H <- R(phi_e) [exp(cA_e) H + Sn]
//   MMA 2     Ya = P X            (QR x P,  K = QR, A operand read from TMEM)
//   epilogue  y = Ya + exp(cA_t) Yi   (fp32)
//
// Roles: warp 0 issues the TMA loads (two raw slots), warp 1 allocates TMEM and
// issues the MMAs, warps 2-9 run the prologue of chunk c+1 while warps 10-17
// run the epilogues of chunk c; they hand chunks over through mbarriers.  The
// fp32 state H stays in TMEM next to the accumulators.
//
// Precision.  Every MMA operand (B~, C~, X^, H, P and x) is fp16 (11-bit
// significand, fp32 accumulation) scaled by a per-chunk power of two that
// puts a bound of the tile just under 2^14, so the result does not depend on
// the magnitude of the inputs (x itself converts exactly); the scales are
// undone exactly in the fp32 epilogues.
// The decay is always formed as exp2 of a difference of chunk-local
// cumulative sums (exponent <= 0) and factored per 32-column block, so no
// partial product overflows.
#include "m3_internal.cuh"
#include "m3_tc.cuh"

#include <atomic>
#include <chrono>
#include <mutex>
#include <type_traits>

namespace m3 {
namespace {

using namespace tc;

constexpr int kP = 64;
constexpr int kWarps = 18;
constexpr int kThreads = kWarps * 32;
constexpr int kProW0 = 2, kProWarps = 8, kEpiW0 = 10, kEpiWarps = 8;
constexpr int kProThreads = kProWarps * 32, kEpiThreads = kEpiWarps * 32;
constexpr int kBarPro = 1, kBarEpi = 2;          // named barriers of the two groups
constexpr uint64_t kWaitNs = 2000000000ull;      // 2 s per mbarrier wait; far above any legal wait
constexpr float kLog2e = 1.4426950408889634f;

// QRT: rows (t, r) per chunk; by default 128 for N = 64 and 64 for N = 128 (what shared memory
// holds); 64 for N = 64 is the chunk rule Q = N / R of the pages
template <int N, int R, int QRT = (N == 64 ? 128 : 64)>
struct Cfg {
    static constexpr int QR = QRT;                    // rows (t, r) per chunk
    static constexpr int Q = QR / R;                  // tokens per chunk
    static constexpr int K = N / 2;                   // complex pairs
    static constexpr int NSLAB = N / 64;              // 64-column (128-byte) slabs of B and C
    static constexpr int NSEG = kProWarps / NSLAB;    // token segments of the prologue
    static constexpr int TPS = Q / NSEG;              // tokens per segment
    static constexpr int TB = 32 / R;                 // tokens per 32-column block of the score
    static constexpr uint32_t BT = QR * N * 2;        // B or C tile
    static constexpr uint32_t XT = QR * kP * 2;       // X or X^ tile
    static constexpr uint32_t TT = Q * K * 2;         // theta tile
    static constexpr uint32_t HT = N * kP * 2;        // fp16 state tile
    static_assert(Q % NSEG == 0 && TPS >= 1, "token segments must tile the chunk");
    static_assert(K == 32 * NSLAB, "one lane per pair within a slab");
    static_assert(Q <= kProThreads, "one prologue thread per token");
};

// Shared-memory map (byte offsets from a 1024-aligned base).
// YB: bytes per element of y (4: fp32, 2: fp16 / bf16); BCN: BC normalisation and bias
template <int N, int R, bool OUT, int YB = 4, bool BCN = false, int QRT = (N == 64 ? 128 : 64)>
struct Smem {
    using C = Cfg<N, R, QRT>;
    // raw slot: B, C (turned into fp16 B~, C~ in place), X (bf16), theta
    static constexpr uint32_t sB = 0;
    static constexpr uint32_t sC = sB + C::BT;
    static constexpr uint32_t sX = sC + (OUT ? C::BT : 0);
    static constexpr uint32_t sT = sX + C::XT;
    static constexpr uint32_t SLOT = ((sT + C::TT + 1023) / 1024) * 1024;
    static constexpr uint32_t oXh = 2 * SLOT;                  // X^ [2] (fp16)
    static constexpr uint32_t oXp = oXh + 2 * C::XT;           // X' [2] (fp16), OUT only
    static constexpr uint32_t oH = oXp + (OUT ? 2 * C::XT : 0); // H (fp16), OUT only
    // y staging, OUT only: fp32 y as 2 halves [QR][32]; 16-bit y as one [QR][64] tile
    static constexpr uint32_t oYs = oH + (OUT ? C::HT : 0);
    static constexpr uint32_t oVec = oYs + (OUT ? C::QR * kP * YB : 0);   // per-parity vectors
    // per parity (floats): cA2[Q] g[Q] w[Q] vj[Q] dt[Q] cosE[K] sinE[K] sig[8]
    static constexpr uint32_t VF = 5 * C::Q + 2 * C::K + 8;
    static constexpr uint32_t oPart = oVec + 2 * 4 * VF;       // angle partials [8][K]
    static constexpr uint32_t oMx = oPart + 4 * kProWarps * C::K;   // prologue maxima [8][4]
    static constexpr uint32_t oMxH = oMx + 4 * kProWarps * 4;       // epilogue maxima [2][8]
    static constexpr uint32_t oSigH = oMxH + 4 * 2 * kEpiWarps;     // H scale [2] and inverse [2]
    static constexpr uint32_t oTot = oSigH + 16;                    // segment totals [1 + K]
    static constexpr uint32_t oWtot = oTot + 4 * (1 + C::K);                    // per-warp dt A totals [4]
    // BC normalisation (BCN only): row inverse RMS [B, C][QR] (room for [B, C][slab][QR]), gains [B, C][N],
    // biases [B, C][R][N], static bounds of |B'|, |C'| [2]
    static constexpr uint32_t oSS = ((oWtot + 16 + 15) / 16) * 16;   // float2 reads of gains and biases
    static constexpr uint32_t oBW = oSS + (BCN ? 4 * 2 * C::NSLAB * C::QR : 0);
    static constexpr uint32_t oBB = oBW + (BCN ? 4 * 2 * N : 0);
    static constexpr uint32_t oBnd = oBB + (BCN ? 4 * 2 * R * N : 0);
    static constexpr uint32_t oBar = ((oBnd + (BCN ? 8 : 0) + 7) / 8) * 8;
    static_assert(oBW % 8 == 0 && oBB % 8 == 0, "8-byte aligned float2 gains and biases");
    static constexpr int kNumBars = 16;
    static constexpr uint32_t oTmem = oBar + 8 * kNumBars;
    static constexpr uint32_t oFlag = oTmem + 4;
    static constexpr uint32_t kBytes = oFlag + 4;
    static constexpr uint32_t kAlloc = kBytes + 1024;          // slack for the 1024-byte alignment
};

// Byte offset of element (row, col) in a 128-byte-swizzled tile of 128-byte rows
// (16-bit elements; sw128f: 32-bit elements).
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t col) {
    return row * 128u + ((((col >> 3) ^ row) & 7u) << 4) + ((col & 7u) << 1);
}
__device__ __forceinline__ uint32_t sw128f(uint32_t row, uint32_t col) {
    return row * 128u + ((((col >> 2) ^ row) & 7u) << 4) + ((col & 3u) << 2);
}

// packed fp32 pairs (one instruction for two lanes of arithmetic)
__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 f2u(uint32_t a, uint32_t b) { return make_float2(__uint_as_float(a), __uint_as_float(b)); }

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 2^(13 - floor(log2 m)): maps m to [2^13, 2^14).  1 for m = 0 or non-finite m.
__device__ __forceinline__ float pow2_scale(float m) {
    if (!(m > 0.f) || !(m <= 3.0e38f)) return 1.f;
    const int e = (int)((__float_as_uint(m) >> 23) & 0xFFu) - 127;
    int s = 13 - e;
    s = s < -126 ? -126 : (s > 127 ? 127 : s);
    return __uint_as_float((uint32_t)(s + 127) << 23);
}
__device__ __forceinline__ float pow2_inv(float s) {   // exact inverse of a power of two
    return __uint_as_float((uint32_t)(254 - (int)(__float_as_uint(s) >> 23)) << 23);
}

// fp16 pair (lo element in the low half), round to nearest even
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// fp16 x fp16 -> fp32, dense; a_mn / b_mn: 1 = MN-major operand.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *m) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(m)) : "memory");
}
__device__ __forceinline__ float warp_max(float v) {   // v >= 0
    return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(v)));
}

struct TcMaps {
    CUtensorMap B, C, X, T, Y;
};

// hand-off flags of the balanced plan (a CTA's end state of a sequence head, to the CTA holding its tail)
__device__ __forceinline__ void flag_release(unsigned long long *f, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(f), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long flag_acquire(const unsigned long long *f) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(f) : "memory");
    return v;
}

enum Bar {
    kRawFull = 0,      // [2] TMA -> prologue (transaction bytes)
    kRawEmpty = 2,     // [2] MMAs done with a raw slot -> producer
    kTilesFull = 4,    // [2] prologue -> MMA
    kStateReady = 6,   // [2] epilogue wrote H (and read S, Sn) -> MMA
    kMma1 = 8,         // [2] first MMAs done -> epilogue
    kPReady = 10,      // [2] epilogue wrote P -> MMA
    kMma2 = 12,        // [2] Ya done -> epilogue
    kEpiDone = 14      // [2] epilogue done with a chunk's vectors and x' -> prologue
};

// YT: element type of y (an m3_dtype; OUT only).  BCN: B and C go through the BC normalisation
// and bias (a.bc) before the rotation.  BAL: the balanced plan for more sequences than CTAs (OUT, one
// segment): the sequences' chunk lists, laid end to end, are cut into nbal equal ranges, one per CTA
// (a cooperative launch, so all of them run at once).  A range holds the tail of one sequence, whole
// sequences and the head of another; the CTA runs the head first and hands its end state to the CTA
// holding that sequence's tail (a state slot of the workspace and a flag set to `epoch`), then the
// whole sequences, then its own tail, whose start state it takes from the CTA before.  With more
// sequences than CTAs every range is at least one sequence long, so no hand-off waits on another.
template <int N, int R, bool OUT, int YT = M3_F32, bool BCN = false, int QRT = (N == 64 ? 128 : 64), bool BAL = false>
__global__ void __launch_bounds__(kThreads, 1)
tc_segment_kernel(const __grid_constant__ TcMaps maps, ScanArgs a, int seglen, int nseg, int nlaunch, int ws_stride,
                  int ws_step, unsigned *status, unsigned long long epoch, int nbal) {
    using Cf = Cfg<N, R, QRT>;
    constexpr int YB = YT == M3_F32 ? 4 : 2;
    using S = Smem<N, R, OUT, YB, BCN, QRT>;
    constexpr int QR = Cf::QR, Q = Cf::Q, K = Cf::K, NSLAB = Cf::NSLAB, TPS = Cf::TPS, TB = Cf::TB;
    constexpr uint32_t kTmemCols = OUT ? 512 : 128;
    // TMEM columns: score, state contribution, Yi (two buffers), Ya, P (fp16 pairs), fp32 state
    constexpr uint32_t cS = 0, cSn = OUT ? 128 : 0, cYi0 = 192, cYa = 320, cP = 384, cH = OUT ? 448 : 64;
    constexpr bool kRowsM64 = (QR == 64);    // S / Yi / Ya use the M = 64 lane layout
    constexpr bool kStateM64 = (N == 64);    // Sn uses the M = 64 lane layout

    extern __shared__ __align__(16) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + S::oBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + S::oTmem);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(sm + S::oFlag);
    float *part = reinterpret_cast<float *>(sm + S::oPart);
    float *mx = reinterpret_cast<float *>(sm + S::oMx);
    float *mxH = reinterpret_cast<float *>(sm + S::oMxH);
    float *sigH = reinterpret_cast<float *>(sm + S::oSigH);   // [0..1] scale, [2..3] inverse
    float *tot = reinterpret_cast<float *>(sm + S::oTot);
    float *wtot = reinterpret_cast<float *>(sm + S::oWtot);
    auto vec = [&](int p) { return reinterpret_cast<float *>(sm + S::oVec) + p * S::VF; };
    // per-parity vector fields
    auto v_cA = [&](int p) { return vec(p); };
    auto v_g = [&](int p) { return vec(p) + Q; };
    auto v_w = [&](int p) { return vec(p) + 2 * Q; };
    auto v_vj = [&](int p) { return vec(p) + 3 * Q; };
    auto v_dt = [&](int p) { return vec(p) + 4 * Q; };
    auto v_cos = [&](int p) { return vec(p) + 5 * Q; };
    auto v_sin = [&](int p) { return vec(p) + 5 * Q + K; };
    // scales: sB, sC, sX, tauP / (sB sC), 1 / (sB sX), 1 / sC, 1 / (tauP sX')
    auto v_sig = [&](int p) { return vec(p) + 5 * Q + 2 * K; };

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = a.H, L = a.L;
    // sequence of this CTA: its index scrambled by s -> m s mod (batch H), m = 41 or 43 (primes, so that one
    // of them is coprime to the count and the map a permutation), spreading each wave over batches and heads
    const int nseq_ = a.batch * a.H, smul = nseq_ % 41 ? 41 : (nseq_ % 43 ? 43 : 1);
    const int g = blockIdx.x % nlaunch, bh = (int)(((long long)(blockIdx.x / nlaunch) * smul) % nseq_), b = bh / H, h = bh % H;
    const int t_begin = g * seglen, t_end = min(L, t_begin + seglen);
    int nchunks = t_end > t_begin ? (t_end - t_begin + Q - 1) / Q : 0;
    static_assert(!BAL || (OUT && !BCN), "the balanced plan runs the output pass without BC normalisation");
    // The chunks this CTA walks, in order, as pieces (sequence, chunks [cb, ce)).  Without BAL one piece:
    // this CTA's segment of sequence bh.  With BAL: the range [c0, c1) of the concatenated chunk lists
    // (ncs chunks per sequence), sequence sA from chunk a0 on to sequence sB up to chunk bE.
    const int ncs = (L + Q - 1) / Q;
    int sA = bh, a0 = t_begin / Q, sB = bh, bE = a0 + nchunks, npc = 1;
    if constexpr (BAL) {
        const long long T = (long long)a.batch * H * ncs;
        const long long c0 = T * blockIdx.x / nbal, c1 = T * (blockIdx.x + 1) / nbal;
        nchunks = (int)(c1 - c0);
        if (nchunks > 0) {
            sA = (int)(c0 / ncs);
            a0 = (int)(c0 % ncs);
            sB = (int)((c1 - 1) / ncs);
            bE = (int)((c1 - 1) % ncs) + 1;
            npc = sA == sB ? 1 : sB - sA + 1;
        }
    }
    // piece p: sequence seq (batch qb, head qh), chunks [cb, ce); current chunk c.  The plain plan's one
    // piece is the CTA's segment: only c varies, the rest are the CTA's constants (the accessors below)
    struct PosB { int p, seq, qb, qh, cb, ce, c; };
    struct PosP { int c; };
    using Pos = std::conditional_t<BAL, PosB, PosP>;
    auto piece_at = [&](int pi) -> Pos {
        if constexpr (BAL) {
            int sq = sA, cb = a0, ce = bE;
            if (sA != sB) {
                if (pi == 0) { sq = sB; cb = 0; ce = bE; }                       // head of the last sequence
                else if (pi < npc - 1) { sq = sA + pi; cb = 0; ce = ncs; }       // whole sequences
                else { sq = sA; cb = a0; ce = ncs; }                              // tail of the first
            }
            return Pos{pi, sq, sq / H, sq % H, cb, ce, cb};
        } else {
            return Pos{a0};
        }
    };
    auto pos_next = [&](Pos u) {
        ++u.c;
        if constexpr (BAL) {
            if (u.c >= u.ce && u.p + 1 < npc) u = piece_at(u.p + 1);
        }
        return u;
    };
    auto p_seq = [&](const Pos &u) { if constexpr (BAL) return u.seq; else return bh; };
    auto p_qb = [&](const Pos &u) { if constexpr (BAL) return u.qb; else return b; };
    auto p_qh = [&](const Pos &u) { if constexpr (BAL) return u.qh; else return h; };
    auto p_cb = [&](const Pos &u) { if constexpr (BAL) return u.cb; else return a0; };
    auto p_ce = [&](const Pos &u) { if constexpr (BAL) return u.ce; else return bE; };
    const int t_stop = BAL ? L : t_end;   // y, and the chunk's tokens, end here
    // state slots and flags of the hand-offs (BAL): slot i carries CTA i's head state to CTA i + 1
    unsigned long long *hflags = BAL ? reinterpret_cast<unsigned long long *>(a.ws_state + (size_t)nbal * N * kP)
                                     : nullptr;
    const __nv_bfloat16 *dtp = static_cast<const __nv_bfloat16 *>(a.dt);
    const __nv_bfloat16 *Ap = static_cast<const __nv_bfloat16 *>(a.A);
    const __nv_bfloat16 *lp = static_cast<const __nv_bfloat16 *>(a.lam);
    auto tok = [&](int t) { return ((size_t)b * L + t) * H + h; };
    auto tokq = [&](const Pos &u, int t) { return ((size_t)p_qb(u) * L + t) * H + p_qh(u); };   // token t of u's sequence

    // bounded wait; after any timeout every later wait returns at once
    // (backoff: single-thread roles nap between polls so that they do not take
    // issue slots from the warps doing arithmetic)
    auto wait = [&](int i, uint32_t parity, bool backoff = false) {
        uint64_t *m = bars + i;
        const uint64_t t0 = global_ns();
        for (uint32_t n = 0;; ++n) {
            if (mbar_try_wait(m, parity)) return;
            if (backoff) __nanosleep(64);
            if ((n & 7u) == 7u) {
                if (*abort_flag) return;
                if (global_ns() - t0 > kWaitNs) break;
            }
        }
        *abort_flag = 1;
        atomicOr(status, kStatusTimeout);
    };

    // ---- set-up
    // Programmatic dependent launch: the next kernel in the stream may be scheduled from now on (its CTAs
    // take SMs as these leave); nothing below touches global memory or TMEM before the grid this one
    // depends on has completed and its writes are visible
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (tid == 0) {
        for (int p = 0; p < 2; ++p) {
            mbar_init(bars + kRawFull + p, 1);
            mbar_init(bars + kRawEmpty + p, 1);
            mbar_init(bars + kTilesFull + p, kProThreads);
            mbar_init(bars + kStateReady + p, kEpiThreads);
            mbar_init(bars + kMma1 + p, 1);
            mbar_init(bars + kPReady + p, kEpiThreads);
            mbar_init(bars + kMma2 + p, 1);
            mbar_init(bars + kEpiDone + p, kEpiThreads);
        }
        mbar_init_fence();
        *abort_flag = 0;
        tma_prefetch_desc(&maps.B);
        tma_prefetch_desc(&maps.X);
        tma_prefetch_desc(&maps.T);
        if (OUT) {
            tma_prefetch_desc(&maps.C);
            tma_prefetch_desc(&maps.Y);
        }
    }
    for (int i = tid; i < 1 + K; i += kThreads) tot[i] = 0.f;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ================================================================ producer
        if (lane == 0) {
            int issued = 0;
            Pos u = piece_at(0);
            for (int it = 0; it < nchunks; ++it, u = pos_next(u)) {
                const int p = it & 1;
                if (it >= 2) wait(kRawEmpty + p, ((it - 2) >> 1) & 1, true);
                // after a timeout nothing more is issued: a refill could land on a slot whose
                // previous copy is still in flight
                if (*abort_flag) break;
                unsigned char *slot = sm + p * S::SLOT;
                constexpr uint32_t bytes = Cf::BT * (OUT ? 2 : 1) + Cf::XT + Cf::TT;
                mbar_expect_tx(bars + kRawFull + p, bytes);
                const int qh = p_qh(u);
                const int t0 = u.c * Q, b0 = p_qb(u);   // rows past the sequence end arrive as zeros
                const int hg = qh / (H / a.G);   // B / C group of this head
#pragma unroll
                for (int sl = 0; sl < NSLAB; ++sl) {
                    tma_load_5d(slot + S::sB + sl * QR * 128, &maps.B, 64 * sl, 0, hg, t0, b0, bars + kRawFull + p);
                    if (OUT)
                        tma_load_5d(slot + S::sC + sl * QR * 128, &maps.C, 64 * sl, 0, hg, t0, b0, bars + kRawFull + p);
                }
                tma_load_5d(slot + S::sX, &maps.X, 0, 0, qh, t0, b0, bars + kRawFull + p);
                tma_load_4d(slot + S::sT, &maps.T, 0, qh, t0, b0, bars + kRawFull + p);
                ++issued;
            }
            if (*abort_flag) {
                // let the copies issued land before the CTA's shared memory goes away: a slot is
                // refilled only after its previous chunk was consumed, so at most the last two
                // issued copies are outstanding, each the only one on its barrier phase
                for (int it = issued - 2 < 0 ? 0 : issued - 2; it < issued; ++it)
                    mbar_wait(bars + kRawFull + (it & 1), (it >> 1) & 1, kWaitNs);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = idesc_f16(QR, QR, 0, 0);
            constexpr uint32_t idYi = idesc_f16(QR, kP, 0, 1);
            constexpr uint32_t idSn = idesc_f16(N, kP, 1, 1);
            constexpr uint32_t idYa = idesc_f16(QR, kP, 0, 1);
            for (int it = 0; it < nchunks; ++it) {
                const int p = it & 1;
                const uint32_t ph = (it >> 1) & 1;
                wait(kTilesFull + p, ph, true);
                wait(kStateReady + p, ph, true);
                fence_after();
                unsigned char *slot = sm + p * S::SLOT;
                const uint32_t bA = smem_u32(slot + S::sB), xh = smem_u32(sm + S::oXh + p * Cf::XT);
                if (OUT) {
                    const uint32_t cA = smem_u32(slot + S::sC), hA = smem_u32(sm + S::oH);
                    const uint32_t cYi = cYi0 + 64 * p;
#pragma unroll
                    for (int ks = 0; ks < N / 16; ++ks) {
                        // K-major, 128-byte swizzle: slab ks / 4, 32 bytes per 16-column step inside it
                        const uint32_t ko = (ks / 4) * (QR * 128) + (ks % 4) * 32;
                        const uint64_t dC = make_desc(cA + ko, 16, 1024, kSwizzle128B);
                        mma_ss(tmem + cS, dC, make_desc(bA + ko, 16, 1024, kSwizzle128B), idS, ks > 0);
                        // state operand: MN-major (p), K = n rows in 8-row groups of 1024 bytes
                        mma_ss(tmem + cYi, dC, make_desc(hA + ks * 2048, 0, 1024, kSwizzle128B), idYi, ks > 0);
                    }
                }
#pragma unroll
                for (int ks = 0; ks < QR / 16; ++ks) {
                    // B~ read as the MN-major A operand (M = n in 64-wide slabs, K = rows j)
                    mma_ss(tmem + cSn, make_desc(bA + ks * 2048, QR * 128, 1024, kSwizzle128B),
                           make_desc(xh + ks * 2048, 0, 1024, kSwizzle128B), idSn, ks > 0);
                }
                mma_commit(bars + kMma1 + p);
                mma_commit(bars + kRawEmpty + p);   // MMA 2 reads only TMEM and x'
                if (OUT) {
                    wait(kPReady + p, ph, true);
                    fence_after();
                    const uint32_t xb = smem_u32(sm + S::oXp + p * Cf::XT);
#pragma unroll
                    for (int ks = 0; ks < QR / 16; ++ks)
                        mma_ts(tmem + cYa, tmem + cP + ks * 8, make_desc(xb + ks * 2048, 0, 1024, kSwizzle128B),
                               idYa, ks > 0);
                    mma_commit(bars + kMma2 + p);
                }
            }
            if (*abort_flag && nchunks > 0) {
                // let the last MMAs finish before TMEM is released
                const int it = nchunks - 1;
                mbar_wait(bars + (OUT ? kMma2 : kMma1) + (it & 1), (it >> 1) & 1, kWaitNs);
            }
        }
        __syncwarp();
    } else if (warp < kEpiW0) {
        // ================================================================ prologue
        const int ptid = tid - kProW0 * 32, pw = warp - kProW0;
        const int slab = pw % NSLAB, seg = pw / NSLAB, k = 32 * slab + lane;
        // Without BC normalisation each lane turns two adjacent pairs (kp = 32 slab + 2 kc and kp + 1) of
        // half of its warp's tokens (half hh), so that its shared-memory words are 8 bytes; with it, one
        // pair k per lane (the two-pair form measured slower there, its gains and biases held or reloaded)
        constexpr bool kPair2 = !BCN;
        // Rows past the sequence end come in as zeros (the input maps end there) and rotate to zeros, so
        // the two-pair rotation needs no selects for them; the SISO N = 64 build keeps them (without, the
        // compiler's schedule spills at the register cap and runs 5 % slower)
        constexpr bool kSelects = R == 1 && N == 64;
        constexpr int TH = TPS / 2;   // tokens per lane with two pairs
        static_assert(!kPair2 || TPS % 2 == 0, "two halves of whole tokens");
        const int kc = lane & 15, hh = lane >> 4, kp = 32 * slab + 2 * kc;
        // per-token scalars of the next chunk, loaded one chunk ahead into registers
        // (raw values: nothing waits on these loads until the chunk is processed)
        __nv_bfloat16 r_dt, r_A, r_l, r_ln, r_dtn;
        auto fetch = [&](int it, const Pos &u) {
            const __nv_bfloat16 z = __float2bfloat16_rn(0.f);
            r_dt = r_A = r_l = r_ln = r_dtn = z;
            const int t = u.c * Q + ptid;
            if (ptid < Q && it < nchunks && t < t_stop) {
                const size_t ti = tokq(u, t);
                r_dt = dtp[ti];
                r_A = Ap[ti];
                r_l = lp[ti];
                if (t + 1 < L) {
                    const size_t tn = ti + H;   // the next token of the sequence
                    r_ln = lp[tn];
                    r_dtn = dtp[tn];
                } else {
                    r_ln = __float2bfloat16_rn(1.f);   // (1 - lambda) dt = 0 past the sequence end
                }
            }
        };
        Pos pu = piece_at(0);   // this chunk
        fetch(0, pu);
        float acc_cA = 0.f;   // pass 1: total log2-decay of the segment (prologue thread 0)
        float *bss = reinterpret_cast<float *>(sm + S::oSS);    // [B, C][QR] inverse RMS of the rows
        const float *bw = reinterpret_cast<const float *>(sm + S::oBW);   // [B, C][N]
        const float *bb = reinterpret_cast<const float *>(sm + S::oBB);   // [B, C][R][N]
        const float *bnd = reinterpret_cast<const float *>(sm + S::oBnd); // [B, C]
        if constexpr (BCN) {
            // this head's gains and biases into shared memory, and the bounds |v'| <= sqrt(N) max|w| +
            // max|bias| (|v| / rms(v) <= sqrt(N)) that replace the tile maxima of B and C
            float *w = reinterpret_cast<float *>(sm + S::oBW), *bi = reinterpret_cast<float *>(sm + S::oBB);
#pragma unroll
            for (int tsr = 0; tsr < 2; ++tsr) {
                const float *ws = tsr ? a.bc.wC : a.bc.wB, *bs = tsr ? a.bc.bC : a.bc.bB;
                float mw = 0.f, mb = 0.f;
                for (int n = ptid; n < N; n += kProThreads) {
                    const float v = ws ? ws[(size_t)h * N + n] : 1.f;
                    w[tsr * N + n] = v;
                    mw = fmaxf(mw, fabsf(v));
                }
                for (int rn = ptid; rn < R * N; rn += kProThreads) {
                    const float v = bs ? bs[(size_t)h * R * N + rn] : 0.f;
                    bi[tsr * R * N + rn] = v;
                    mb = fmaxf(mb, fabsf(v));
                }
                mw = warp_max(mw);
                mb = warp_max(mb);
                if (lane == 0) mx[pw * 4 + tsr] = sqrtf((float)N) * mw + mb;
            }
            named_sync(kBarPro, kProThreads);
            if (ptid < 2) {
                float m = 0.f;
                for (int q = 0; q < kProWarps; ++q) m = fmaxf(m, mx[q * 4 + ptid]);
                reinterpret_cast<float *>(sm + S::oBnd)[ptid] = m;
            }
            named_sync(kBarPro, kProThreads);
        }
        for (int it = 0; it < nchunks; ++it, pu = pos_next(pu)) {
            const int p = it & 1;
            const int s0 = pu.c * Q, Qc = min(Q, t_stop - s0), e = Qc - 1;
            unsigned char *slot = sm + p * S::SLOT;
            float *cA2 = v_cA(p), *gv = v_g(p), *wv = v_w(p), *vj = v_vj(p), *dts = v_dt(p);
            if (it >= 2) wait(kEpiDone + p, ((it - 2) >> 1) & 1);
            // ---- P1: token scalars
            const float c_dt = to_f(r_dt), c_a = c_dt * to_f(r_A) * kLog2e, c_g = to_f(r_l) * c_dt;
            const float c_w = c_g + (1.f - to_f(r_ln)) * to_f(r_dtn);
            // inclusive scan of dt A within each warp of tokens (shuffles); the warp totals
            // are added after the barrier
            float c_scan = c_a;
            if (pw * 32 < Q) {
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float t = __shfl_up_sync(0xffffffffu, c_scan, o);
                    if (lane >= o) c_scan += t;
                }
                if (lane == 31) wtot[pw] = c_scan;
            }
            if (ptid < Q) {
                dts[ptid] = c_dt;
                gv[ptid] = c_g;
                wv[ptid] = c_w;
            }
            fetch(it + 1, pos_next(pu));
            // one thread waits for the chunk's TMA; the named barrier (which costs the
            // other warps no issue slots) releases the rest
            if (ptid == 0) wait(kRawFull + p, (it >> 1) & 1);
            named_sync(kBarPro, kProThreads);
            // ---- P2: chunk-local cumsum of dt A, angle partial sums, bounds of |B|, |C|, |x|, w
            if (ptid < Q) {
                float off = 0.f;
#pragma unroll
                for (int q = 0; q < (Q + 31) / 32 - 1; ++q) off += (q < pw) ? wtot[q] : 0.f;
                cA2[ptid] = c_scan + off;
            }
            const __nv_bfloat16 *rawT = reinterpret_cast<const __nv_bfloat16 *>(slot + S::sT);
            float mW = ptid < Qc ? fabsf(c_w) : 0.f;
            // this thread's tokens: dt (0 past the sequence end) and its pair's angle rate
            float dd[TPS], th[TPS];
            float dd2[TH];
            float2 th2[TH], lo2 = f2(0.f);   // two pairs: rates; the first half's partial sums (hh = 1)
            if constexpr (kPair2) {
#pragma unroll
                for (int i = 0; i < TH; ++i) {
                    const int t = seg * TPS + hh * TH + i;
                    dd2[i] = dts[t];
                    const uint32_t w = *reinterpret_cast<const uint32_t *>(rawT + t * K + kp);
                    th2[i] = f2u(w << 16, w & 0xFFFF0000u);
                }
                float2 ps = f2(0.f);
#pragma unroll
                for (int i = 0; i < TH; ++i) ps = __ffma2_rn(f2(dd2[i]), th2[i], ps);
                const float2 other = make_float2(__shfl_xor_sync(0xffffffffu, ps.x, 16),
                                                 __shfl_xor_sync(0xffffffffu, ps.y, 16));
                if (hh == 0) {
                    part[seg * K + kp] = ps.x + other.x;
                    part[seg * K + kp + 1] = ps.y + other.y;
                } else {
                    lo2 = other;
                }
            } else {
#pragma unroll
                for (int i = 0; i < TPS; ++i) {
                    const int t = seg * TPS + i;
                    dd[i] = dts[t];
                    th[i] = __bfloat162float(rawT[t * K + k]);
                }
                float ps = 0.f;
#pragma unroll
                for (int i = 0; i < TPS; ++i) ps = fmaf(dd[i], th[i], ps);
                part[seg * K + k] = ps;
            }
            // bounds of |B|, |C|, |x| over the raw tiles: packed maxima of the bf16 magnitudes
            // (their bit patterns order like the values)
            auto tile_max = [&](const unsigned char *base, auto bytes_c) {
                constexpr uint32_t bytes = decltype(bytes_c)::value;
                static_assert(bytes % (16u * kProThreads) == 0, "whole 16-byte words per thread");
                uint32_t m2 = 0;
#pragma unroll
                for (uint32_t o = 0; o < bytes; o += 16u * kProThreads) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(base + o + 16u * ptid);
                    m2 = __vmaxu2(m2, v.x & 0x7FFF7FFFu);
                    m2 = __vmaxu2(m2, v.y & 0x7FFF7FFFu);
                    m2 = __vmaxu2(m2, v.z & 0x7FFF7FFFu);
                    m2 = __vmaxu2(m2, v.w & 0x7FFF7FFFu);
                }
                return fmaxf(bf16_lo_f(m2), bf16_hi_f(m2));
            };
            using BTc = std::integral_constant<uint32_t, Cf::BT>;
            using XTc = std::integral_constant<uint32_t, Cf::XT>;
            float mB, mC;
            if constexpr (BCN) {
                // inverse RMS of the raw B (and C) rows: the 8 consecutive threads reading one 128-byte
                // row of the first slab (64 entries) also read the same row of the other slab, add
                // their squares with three shuffles, and one of them writes rsqrt(mean + eps)
                auto row_ss = [&](const unsigned char *base, float *dst) {
                    static_assert((QR * 128) % (16 * kProThreads) == 0, "whole rows per pass");
#pragma unroll
                    for (uint32_t o = 16u * ptid; o < QR * 128u; o += 16u * kProThreads) {
                        float2 acc = f2(0.f);
#pragma unroll
                        for (int sl = 0; sl < NSLAB; ++sl) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(base + sl * (QR * 128) + o);
                            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                            for (int z = 0; z < 4; ++z) {
                                const float2 e2 = f2u(wv[z] << 16, wv[z] & 0xFFFF0000u);
                                acc = __ffma2_rn(e2, e2, acc);
                            }
                        }
                        float ssq = acc.x + acc.y;
                        ssq += __shfl_xor_sync(0xffffffffu, ssq, 1);
                        ssq += __shfl_xor_sync(0xffffffffu, ssq, 2);
                        ssq += __shfl_xor_sync(0xffffffffu, ssq, 4);
                        if ((ptid & 7) == 0) dst[o / 128u] = rsqrtf(fmaf(ssq, 1.f / N, a.bc.eps));
                    }
                };
                row_ss(slot + S::sB, bss);
                if (OUT) row_ss(slot + S::sC, bss + QR);
                mB = bnd[0];
                mC = OUT ? bnd[1] : 0.f;
            } else {
                mB = tile_max(slot + S::sB, BTc{});
                mC = OUT ? tile_max(slot + S::sC, BTc{}) : 0.f;
            }
            float mX = tile_max(slot + S::sX, XTc{});
            mB = warp_max(mB);
            mC = warp_max(mC);
            mX = warp_max(mX);
            mW = warp_max(mW);
            if (lane == 0) {
                mx[pw * 4 + 0] = mB;
                mx[pw * 4 + 1] = mC;
                mx[pw * 4 + 2] = mX;
                mx[pw * 4 + 3] = mW;
            }
            named_sync(kBarPro, kProThreads);
            // ---- P3: scales, rotation of B and C in place (fp16), X^, mask column factors
            float MB, MC, MX, MW;
            {
                const bool rd = lane < kProWarps;
                MB = warp_max(rd ? mx[lane * 4 + 0] : 0.f);
                MC = warp_max(rd ? mx[lane * 4 + 1] : 0.f);
                MX = warp_max(rd ? mx[lane * 4 + 2] : 0.f);
                MW = warp_max(rd ? mx[lane * 4 + 3] : 0.f);
            }
            // |B~| <= sqrt 2 max|B| (rotation of a pair);  |X^| <= max w max|x|;
            // |P| <= N max|B~| max|C~| max(w, lambda dt)
            // one scale for B~ and C~ (their rotations then share the scaled cos / sin)
            const float sgB = pow2_scale(1.5f * fmaxf(MB, MC)), sgC = sgB, sgX = pow2_scale(MX * MW);
            const float sgXp = pow2_scale(MX), tauP = pow2_scale((float)N * 2.25f * MB * MC * MW);
            if (ptid == 0) {
                float *sg = v_sig(p);
                sg[0] = sgB;
                sg[1] = sgC;
                sg[2] = sgX;
                sg[3] = tauP * pow2_inv(sgB) * pow2_inv(sgC);
                sg[4] = pow2_inv(sgB) * pow2_inv(sgX);
                sg[5] = pow2_inv(sgC);
                sg[6] = pow2_inv(tauP) * pow2_inv(sgXp);
                if (!OUT) acc_cA += cA2[e];
            }
            if constexpr (kPair2) {
                // two pairs a lane: both pairs' angles as one packed pair, 8-byte words of B and C
                float2 phi2 = lo2;
#pragma unroll
                for (int sg = 0; sg < Cf::NSEG - 1; ++sg)
                    if (sg < seg) phi2 = __fadd2_rn(phi2, make_float2(part[sg * K + kp], part[sg * K + kp + 1]));
                float2 ph2[TH];
#pragma unroll
                for (int i = 0; i < TH; ++i) {
                    phi2 = __ffma2_rn(f2(dd2[i]), th2[i], phi2);
                    ph2[i] = phi2;
                }
                const int t0 = seg * TPS + hh * TH;
                const int ie = e - t0;   // the chunk's last token, if it is this lane's
                unsigned char *bs = slot + S::sB + slab * (QR * 128), *cs = slot + S::sC + slab * (QR * 128);
                uint2 rb2[TH * R], rc2[TH * R];
                constexpr int kLA = TH < 4 ? TH : 4;
                auto load_tok = [&](int i) {
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const uint32_t off = sw128((t0 + i) * R + r, 4 * kc);
                        rb2[i * R + r] = *reinterpret_cast<const uint2 *>(bs + off);
                        if (OUT) rc2[i * R + r] = *reinterpret_cast<const uint2 *>(cs + off);
                    }
                };
#pragma unroll
                for (int i = 0; i < kLA; ++i) load_tok(i);
                // sin / cos as in the one-pair layout below (Cody-Waite by 2 pi, then the hardware
                // approximations), the two lanes of each packed pair now the lane's two pairs
#pragma unroll
                for (int i = 0; i < TH; ++i) {
                    if (i + kLA < TH) load_tok(i + kLA);
                    const float2 x2 = ph2[i];
                    const float2 n2 = __fadd2_rn(__ffma2_rn(x2, f2(0.15915494309189535f), f2(12582912.f)),
                                                 f2(-12582912.f));
                    float2 r2 = __ffma2_rn(n2, f2(-6.28318548202514648f), x2);
                    r2 = __ffma2_rn(n2, f2(1.7484555314695172e-7f), r2);
                    float c0, s0, c1, s1;
                    __sincosf(r2.x, &s0, &c0);
                    __sincosf(r2.y, &s1, &c1);
                    if (i == ie) {   // the chunk's last token: rotation of the state at the chunk end
                        v_cos(p)[kp] = c0;
                        v_cos(p)[kp + 1] = c1;
                        v_sin(p)[kp] = s0;
                        v_sin(p)[kp + 1] = s1;
                        if (!OUT) {
                            tot[1 + kp] += x2.x;
                            tot[1 + kp + 1] += x2.y;
                        }
                    }
                    const float2 cb = __fmul2_rn(make_float2(c0, c1), f2(sgB));
                    const float2 sb = __fmul2_rn(make_float2(s0, s1), f2(sgB));
                    const float2 nsb = __fmul2_rn(make_float2(s0, s1), f2(-sgB));
                    const bool valid = kSelects ? t0 + i < Qc : true;
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const uint32_t off = sw128((t0 + i) * R + r, 4 * kc);
                        // entries 2k (even) and 2k + 1 (odd) of the two pairs
                        const uint2 vb = rb2[i * R + r];
                        const float2 be = f2u(vb.x << 16, vb.y << 16), bo = f2u(vb.x & 0xFFFF0000u, vb.y & 0xFFFF0000u);
                        const float2 oe = __ffma2_rn(cb, be, __fmul2_rn(sb, bo));
                        const float2 oo = __ffma2_rn(cb, bo, __fmul2_rn(nsb, be));
                        *reinterpret_cast<uint2 *>(bs + off) =
                            valid ? make_uint2(pack_f16x2(oe.x, oo.x), pack_f16x2(oe.y, oo.y)) : make_uint2(0u, 0u);
                        if (OUT) {
                            const uint2 vc = rc2[i * R + r];
                            const float2 ge = f2u(vc.x << 16, vc.y << 16), go = f2u(vc.x & 0xFFFF0000u, vc.y & 0xFFFF0000u);
                            const float2 qe = __ffma2_rn(cb, ge, __fmul2_rn(sb, go));
                            const float2 qo = __ffma2_rn(cb, go, __fmul2_rn(nsb, ge));
                            *reinterpret_cast<uint2 *>(cs + off) =
                                valid ? make_uint2(pack_f16x2(qe.x, qo.x), pack_f16x2(qe.y, qo.y)) : make_uint2(0u, 0u);
                        }
                    }
                }
            } else {
                float phi = 0.f;
#pragma unroll
                for (int sg = 0; sg < Cf::NSEG - 1; ++sg) phi += (sg < seg) ? part[sg * K + k] : 0.f;
                unsigned char *bs = slot + S::sB + slab * (QR * 128);
                unsigned char *cs = slot + S::sC + slab * (QR * 128);
                if constexpr (R == 1 || N != 64) {
                    // (BC normalisation) SISO and N = 128: fully unrolled, the raw words loaded a few tokens ahead
                    // angles of all the thread's tokens first (a short FMA chain), then
                    // independent rotations the scheduler can overlap
                    float ph[TPS];
#pragma unroll
                    for (int i = 0; i < TPS; ++i) {
                        phi = fmaf(dd[i], th[i], phi);
                        ph[i] = phi;
                    }
                    const int ie = e - seg * TPS;   // the chunk's last token, if it is this thread's
                    // this thread's BC gains (entries 2k, 2k + 1 of B and of C)
                    float2 wkB = f2(1.f), wkC = f2(1.f);
                    if constexpr (BCN) {
                        wkB = *reinterpret_cast<const float2 *>(bw + 2 * k);
                        wkC = *reinterpret_cast<const float2 *>(bw + N + 2 * k);
                    }
                    // raw words are loaded kLA tokens ahead of their use (each load precedes, in
                    // program order, the in-place stores it could alias, so none waits on a store)
                    uint32_t rb[TPS * R], rc[TPS * R];
                    constexpr int kLA = TPS < 4 ? TPS : 4;
                    auto load_tok = [&](int i) {
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const uint32_t off = sw128((seg * TPS + i) * R + r, 2 * lane);
                            rb[i * R + r] = *reinterpret_cast<const uint32_t *>(bs + off);
                            if (OUT) rc[i * R + r] = *reinterpret_cast<const uint32_t *>(cs + off);
                        }
                    };
#pragma unroll
                    for (int i = 0; i < kLA; ++i) load_tok(i);
                    // two tokens at a time on packed fp32.  sin / cos: Cody-Waite reduction by 2 pi
                    // (two-constant split) to [-pi, pi], n = round(x / 2 pi) by the 1.5 * 2^23
                    // addition (exact for |x / 2 pi| < 2^22, and on the FMA pipe rather than the
                    // conversion unit), then the hardware approximations there
                    static_assert(TPS % 2 == 0, "token pairs");
#pragma unroll
                    for (int i = 0; i < TPS; i += 2) {
                        if (i + kLA < TPS) load_tok(i + kLA);
                        if (i + kLA + 1 < TPS) load_tok(i + kLA + 1);
                        const float2 x2 = make_float2(ph[i], ph[i + 1]);
                        const float2 n2 = __fadd2_rn(__ffma2_rn(x2, f2(0.15915494309189535f), f2(12582912.f)),
                                                     f2(-12582912.f));
                        float2 r2 = __ffma2_rn(n2, f2(-6.28318548202514648f), x2);
                        r2 = __ffma2_rn(n2, f2(1.7484555314695172e-7f), r2);
                        float c0, s0, c1, s1;
                        __sincosf(r2.x, &s0, &c0);
                        __sincosf(r2.y, &s1, &c1);
                        if (i == ie || i + 1 == ie) {   // the chunk's last token: rotation of the state at the chunk end
                            const bool first = i == ie;
                            v_cos(p)[k] = first ? c0 : c1;
                            v_sin(p)[k] = first ? s0 : s1;
                            if (!OUT) tot[1 + k] += first ? ph[i] : ph[i + 1];
                        }
                        const float2 cb = __fmul2_rn(make_float2(c0, c1), f2(sgB));
                        const float2 sb = __fmul2_rn(make_float2(s0, s1), f2(sgB));
                        const float2 nsb = __fmul2_rn(make_float2(s0, s1), f2(-sgB));
                        const int t = seg * TPS + i;
                        const bool valid0 = t < Qc, valid1 = t + 1 < Qc;
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const uint32_t off0 = sw128(t * R + r, 2 * lane), off1 = sw128((t + 1) * R + r, 2 * lane);
                            const uint32_t vb0 = rb[i * R + r], vb1 = rb[(i + 1) * R + r];
                            float2 b0 = f2u(vb0 << 16, vb1 << 16), b1 = f2u(vb0 & 0xFFFF0000u, vb1 & 0xFFFF0000u);
                            // BC normalisation of the two tokens' rows: v * (w / rms) + bias, entries 2k, 2k + 1
                            auto bc_norm = [&](int tsr, float2 &e0, float2 &e1) {
                                const float *iv = bss + tsr * QR + t * R + r;
                                const float2 inv = make_float2(iv[0], iv[R]);
                                const float2 wk = tsr ? wkC : wkB;
                                const float2 bk = *reinterpret_cast<const float2 *>(bb + (tsr * R + r) * N + 2 * k);
                                e0 = __ffma2_rn(e0, __fmul2_rn(inv, f2(wk.x)), f2(bk.x));
                                e1 = __ffma2_rn(e1, __fmul2_rn(inv, f2(wk.y)), f2(bk.y));
                            };
                            if constexpr (BCN) bc_norm(0, b0, b1);
                            const float2 o0 = __ffma2_rn(cb, b0, __fmul2_rn(sb, b1));
                            const float2 o1 = __ffma2_rn(cb, b1, __fmul2_rn(nsb, b0));
                            *reinterpret_cast<uint32_t *>(bs + off0) = valid0 ? pack_f16x2(o0.x, o1.x) : 0u;
                            *reinterpret_cast<uint32_t *>(bs + off1) = valid1 ? pack_f16x2(o0.y, o1.y) : 0u;
                            if (OUT) {
                                const uint32_t vc0 = rc[i * R + r], vc1 = rc[(i + 1) * R + r];
                                float2 e0 = f2u(vc0 << 16, vc1 << 16), e1 = f2u(vc0 & 0xFFFF0000u, vc1 & 0xFFFF0000u);
                                if constexpr (BCN) bc_norm(1, e0, e1);
                                const float2 q0 = __ffma2_rn(cb, e0, __fmul2_rn(sb, e1));
                                const float2 q1 = __ffma2_rn(cb, e1, __fmul2_rn(nsb, e0));
                                *reinterpret_cast<uint32_t *>(cs + off0) = valid0 ? pack_f16x2(q0.x, q1.x) : 0u;
                                *reinterpret_cast<uint32_t *>(cs + off1) = valid1 ? pack_f16x2(q0.y, q1.y) : 0u;
                            }
                        }
                    }
                } else {
                    // (BC normalisation) MIMO with N = 64: a few tokens per thread; one token pair per
                    // iteration of a rolled loop keeps the code (and the instruction-cache footprint) small
                    const int ie = e - seg * TPS;   // the chunk's last token, if it is this thread's
                    // this thread's BC gains (entries 2k, 2k + 1 of B and of C)
                    float2 wkB = f2(1.f), wkC = f2(1.f);
                    if constexpr (BCN) {
                        wkB = *reinterpret_cast<const float2 *>(bw + 2 * k);
                        wkC = *reinterpret_cast<const float2 *>(bw + N + 2 * k);
                    }
                    // two tokens at a time on packed fp32, each pair's angles and raw words loaded in its
                    // own iteration (the loop stays rolled: the kernel's code must fit the instruction
                    // cache).  sin / cos: Cody-Waite reduction by 2 pi (two-constant split) to [-pi, pi],
                    // n = round(x / 2 pi) by the 1.5 * 2^23 addition (exact for |x / 2 pi| < 2^22, and on
                    // the FMA pipe rather than the conversion unit), then the hardware approximations there
                    static_assert(TPS % 2 == 0, "token pairs");
#pragma unroll 2
                    for (int i = 0; i < TPS; i += 2) {
                        const int t = seg * TPS + i;
                        const float ph0 = fmaf(dts[t], __bfloat162float(rawT[t * K + k]), phi);
                        phi = fmaf(dts[t + 1], __bfloat162float(rawT[(t + 1) * K + k]), ph0);
                        uint32_t rb[2 * R], rc[2 * R];
#pragma unroll
                        for (int z = 0; z < 2; ++z)
#pragma unroll
                            for (int r = 0; r < R; ++r) {
                                const uint32_t off = sw128((t + z) * R + r, 2 * lane);
                                rb[z * R + r] = *reinterpret_cast<const uint32_t *>(bs + off);
                                if (OUT) rc[z * R + r] = *reinterpret_cast<const uint32_t *>(cs + off);
                            }
                        const float2 x2 = make_float2(ph0, phi);
                        const float2 n2 = __fadd2_rn(__ffma2_rn(x2, f2(0.15915494309189535f), f2(12582912.f)),
                                                     f2(-12582912.f));
                        float2 r2 = __ffma2_rn(n2, f2(-6.28318548202514648f), x2);
                        r2 = __ffma2_rn(n2, f2(1.7484555314695172e-7f), r2);
                        float c0, s0, c1, s1;
                        __sincosf(r2.x, &s0, &c0);
                        __sincosf(r2.y, &s1, &c1);
                        if (i == ie || i + 1 == ie) {   // the chunk's last token: rotation of the state at the chunk end
                            const bool first = i == ie;
                            v_cos(p)[k] = first ? c0 : c1;
                            v_sin(p)[k] = first ? s0 : s1;
                            if (!OUT) tot[1 + k] += first ? ph0 : phi;
                        }
                        const float2 cb = __fmul2_rn(make_float2(c0, c1), f2(sgB));
                        const float2 sb = __fmul2_rn(make_float2(s0, s1), f2(sgB));
                        const float2 nsb = __fmul2_rn(make_float2(s0, s1), f2(-sgB));
                        const bool valid0 = t < Qc, valid1 = t + 1 < Qc;
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const uint32_t off0 = sw128(t * R + r, 2 * lane), off1 = sw128((t + 1) * R + r, 2 * lane);
                            const uint32_t vb0 = rb[r], vb1 = rb[R + r];
                            float2 b0 = f2u(vb0 << 16, vb1 << 16), b1 = f2u(vb0 & 0xFFFF0000u, vb1 & 0xFFFF0000u);
                            // BC normalisation of the two tokens' rows: v * (w / rms) + bias, entries 2k, 2k + 1
                            auto bc_norm = [&](int tsr, float2 &e0, float2 &e1) {
                                const float *iv = bss + tsr * QR + t * R + r;
                                const float2 inv = make_float2(iv[0], iv[R]);
                                const float2 wk = tsr ? wkC : wkB;
                                const float2 bk = *reinterpret_cast<const float2 *>(bb + (tsr * R + r) * N + 2 * k);
                                e0 = __ffma2_rn(e0, __fmul2_rn(inv, f2(wk.x)), f2(bk.x));
                                e1 = __ffma2_rn(e1, __fmul2_rn(inv, f2(wk.y)), f2(bk.y));
                            };
                            if constexpr (BCN) bc_norm(0, b0, b1);
                            const float2 o0 = __ffma2_rn(cb, b0, __fmul2_rn(sb, b1));
                            const float2 o1 = __ffma2_rn(cb, b1, __fmul2_rn(nsb, b0));
                            *reinterpret_cast<uint32_t *>(bs + off0) = valid0 ? pack_f16x2(o0.x, o1.x) : 0u;
                            *reinterpret_cast<uint32_t *>(bs + off1) = valid1 ? pack_f16x2(o0.y, o1.y) : 0u;
                            if (OUT) {
                                const uint32_t vc0 = rc[r], vc1 = rc[R + r];
                                float2 e0 = f2u(vc0 << 16, vc1 << 16), e1 = f2u(vc0 & 0xFFFF0000u, vc1 & 0xFFFF0000u);
                                if constexpr (BCN) bc_norm(1, e0, e1);
                                const float2 q0 = __ffma2_rn(cb, e0, __fmul2_rn(sb, e1));
                                const float2 q1 = __ffma2_rn(cb, e1, __fmul2_rn(nsb, e0));
                                *reinterpret_cast<uint32_t *>(cs + off0) = valid0 ? pack_f16x2(q0.x, q1.x) : 0u;
                                *reinterpret_cast<uint32_t *>(cs + off1) = valid1 ? pack_f16x2(q0.y, q1.y) : 0u;
                            }
                        }
                    }
                }
            }
            {
                unsigned char *xh = sm + S::oXh + p * Cf::XT;
                unsigned char *xp = sm + S::oXp + p * Cf::XT;
                const float ce = cA2[e];
                static_assert((QR * 8) % kProThreads == 0, "whole items per thread");
                constexpr int kItems = QR * 8 / kProThreads;
                uint4 xv[kItems];
#pragma unroll
                for (int i = 0; i < kItems; ++i) {
                    const int item = ptid + i * kProThreads;
                    xv[i] = *reinterpret_cast<const uint4 *>(slot + S::sX + sw128(item >> 3, 8 * (item & 7)));
                }
#pragma unroll
                for (int i = 0; i < kItems; ++i) {
                    const int item = ptid + i * kProThreads;
                    const int row = item >> 3, c8 = item & 7, t = row / R;
                    const uint32_t off = sw128(row, 8 * c8);
                    uint4 o = make_uint4(0, 0, 0, 0), q = o;
                    // rows past the sequence end: x came in as zeros and w is 0 there, so both tiles get zeros
                    // without a test (kept in the 16-bit-y SISO N = 64 build, whose schedule is 3 % faster with it)
                    constexpr bool kXGuard = YB == 2 && N == 64 && R == 1;
                    if (!kXGuard || t < Qc) {
                        const float sj = fast_exp2(ce - cA2[t]) * wv[t] * sgX;
                        const uint4 v = xv[i];
                        const float f[8] = {bf16_lo_f(v.x), bf16_hi_f(v.x), bf16_lo_f(v.y), bf16_hi_f(v.y),
                                            bf16_lo_f(v.z), bf16_hi_f(v.z), bf16_lo_f(v.w), bf16_hi_f(v.w)};
                        uint32_t ow[4], qw[4];
#pragma unroll
                        for (int z = 0; z < 4; ++z) {
                            const float2 fz = make_float2(f[2 * z], f[2 * z + 1]);
                            const float2 a = __fmul2_rn(f2(sj), fz);
                            ow[z] = pack_f16x2(a.x, a.y);
                            if (OUT) {   // x' = sX' x, exact in fp16
                                const float2 b2 = __fmul2_rn(f2(sgXp), fz);
                                qw[z] = pack_f16x2(b2.x, b2.y);
                            }
                        }
                        o = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                        if (OUT) q = make_uint4(qw[0], qw[1], qw[2], qw[3]);
                    }
                    *reinterpret_cast<uint4 *>(xh + off) = o;
                    if (OUT) *reinterpret_cast<uint4 *>(xp + off) = q;
                }
                if (ptid < Q) {
                    const int bt = (ptid / TB) * TB;
                    vj[ptid] = ptid < Qc ? fast_exp2(cA2[bt] - cA2[ptid]) * wv[ptid] : 0.f;
                }
            }
            fence_proxy_async();
            mbar_arrive(bars + kTilesFull + p);
        }
        if (!OUT) {
            named_sync(kBarPro, kProThreads);
            if (!*abort_flag) {
                float *dst = a.ws_tot + ((size_t)bh * (ws_stride - 1) + g) * (1 + K);
                if (ptid == 0) dst[0] = acc_cA / kLog2e;
                for (int i = ptid; i < K; i += kProThreads) dst[1 + i] = tot[1 + i];
            }
        }
    } else {
        // ================================================================ epilogue
        const int ew = warp - kEpiW0, eq = warp & 3, eh = ew >> 2;   // lane quadrant, column half
        const uint32_t lane_base = static_cast<uint32_t>(eq * 32) << 16;
        // state rows loaded at the start: row n of the N x P state, columns [32 eh, 32 eh + 32)
        const bool st_owner = kStateM64 ? (lane < 16) : true;
        const int st_row = kStateM64 ? eq * 16 + lane : eq * 32 + lane;
        // state rows updated per chunk: N = 64 (the M = 64 layout: 16 lanes per quadrant) uses the 16-lane
        // TMEM shape, so that every thread holds 16 columns of a row: threads 16-31 take the same rows as
        // 0-15, 16 columns further; N = 128 keeps one row per thread, 32 columns.  The BC-normalised MIMO
        // builds keep half the lanes idle instead (at their register cap the 16-lane form was slower)
        constexpr bool kState16 = kStateM64 && !(BCN && R > 1);
        const bool up_own = (kStateM64 && !kState16) ? lane < 16 : true;
        const int up_row = kState16 ? eq * 16 + (lane & 15) : st_row;
        const int up_col = kState16 ? 32 * eh + 16 * (lane >> 4) : 32 * eh;
        // score / output rows owned: with QR = 64 (the M = 64 layout) the 16-lane TMEM shape, threads
        // 16-31 taking the rows of threads 0-15 sixteen columns further (hf = 1)
        const int row = kRowsM64 ? eq * 16 + (lane & 15) : eq * 32 + lane;
        const int hf = kRowsM64 ? lane >> 4 : 0;
        const int ti = row / R;
        // The fp32 state lives in TMEM columns [cH, cH + 64): row n in the lane of the Sn
        // accumulator's row n, column p; this thread holds columns [32 eh, 32 eh + 32).
        const uint32_t hcol = tmem + lane_base + cH + 32 * eh;
        // bounded wait for the hand-off flag of the CTA before (balanced plan)
        auto wait_flag = [&](const unsigned long long *f) {
            const uint64_t t0 = global_ns();
            for (uint32_t n = 0;; ++n) {
                if (flag_acquire(f) == epoch) return;
                __nanosleep(128);
                if ((n & 15u) == 15u) {
                    if (*abort_flag) return;
                    if (global_ns() - t0 > kWaitNs) break;
                }
            }
            *abort_flag = 1;
            atomicOr(status, kStatusTimeout);
        };
        // The state entering piece u into TMEM (this thread's rows, columns [32 eh, 32 eh + 32)); returns
        // the thread's max |h|.  A sequence's first chunk: h0 plus the carry's left-endpoint term; a later
        // segment's: its workspace state; a balanced tail's: the state the CTA before handed over.
        auto load_start = [&](const Pos &u) -> float {
            const int sq = p_seq(u), n = st_row;
            const float *src = nullptr;
            bool from_h0;
            if constexpr (BAL) {
                from_h0 = u.c == 0;
                if (!from_h0) {
                    if (ew == 0 && lane == 0) wait_flag(hflags + blockIdx.x - 1);
                    named_sync(kBarEpi, kEpiThreads);
                    src = a.ws_state + (size_t)(blockIdx.x - 1) * N * kP;
                }
            } else {
                from_h0 = nseg == 1;
                if (!from_h0) src = a.ws_state + ((size_t)bh * ws_stride + (size_t)g * ws_step) * N * kP;
            }
            float hm = 0.f;
            const float left0 = (OUT && from_h0) ? (1.f - to_f(lp[tokq(u, 0)])) * to_f(dtp[tokq(u, 0)]) : 0.f;
            const __nv_bfloat16 *bq = static_cast<const __nv_bfloat16 *>(a.Bprev);
            const __nv_bfloat16 *xq = static_cast<const __nv_bfloat16 *>(a.xprev);
            // the carried B row entries n of every rank, BC-normalised when BCN
            float bqn[R];
#pragma unroll
            for (int r = 0; r < R; ++r) bqn[r] = 0.f;
            if (OUT && st_owner && from_h0 && bq && xq) {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const __nv_bfloat16 *row = bq + ((size_t)sq * R + r) * N;
                    bqn[r] = to_f(row[n]);
                    if constexpr (BCN) {
                        float ssq = 0.f;
                        for (int m = 0; m < N; ++m) ssq = fmaf(to_f(row[m]), to_f(row[m]), ssq);
                        bqn[r] = bc_apply(bqn[r], 1.f / sqrtf(ssq / (float)N + a.bc.eps), a.bc.wB, a.bc.bB,
                                          p_qh(u), r, R, N, n);
                    }
                }
            }
#pragma unroll
            for (int h16 = 0; h16 < 32; h16 += 16) {
                uint32_t w[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int pp = 32 * eh + h16 + j;
                    float v = 0.f;
                    if (OUT && st_owner) {
                        if (from_h0) {
                            v = a.h0 ? a.h0[((size_t)sq * N + n) * kP + pp] : 0.f;
                            if (bq && xq) {
                                float uu = 0.f;
#pragma unroll
                                for (int r = 0; r < R; ++r) uu += bqn[r] * to_f(xq[((size_t)sq * R + r) * kP + pp]);
                                v += left0 * uu;
                            }
                        } else {
                            v = __ldcg(src + (size_t)n * kP + pp);
                        }
                    }
                    hm = fmaxf(hm, fabsf(v));
                    w[j] = __float_as_uint(v);
                }
                tmem_st16(hcol + h16, w);
            }
            return hm;
        };
        // the carry out of sequence sq (its last token's B and x), at the sequence's end
        auto carry_out = [&](const Pos &u) {
            if (!(OUT && a.Bprev_out && a.xprev_out && L > 0 && !*abort_flag)) return;
            const int et = tid - kEpiW0 * 32, sq = p_seq(u);
            const size_t tl = tokq(u, L - 1);
            const size_t tlg = ((size_t)p_qb(u) * L + L - 1) * a.G + p_qh(u) / (H / a.G);   // its B / C group row
            const __nv_bfloat16 *Bm = static_cast<const __nv_bfloat16 *>(a.B);
            const __nv_bfloat16 *xm = static_cast<const __nv_bfloat16 *>(a.x);
            __nv_bfloat16 *bo = static_cast<__nv_bfloat16 *>(a.Bprev_out);
            __nv_bfloat16 *xo = static_cast<__nv_bfloat16 *>(a.xprev_out);
            for (int i = et; i < R * N; i += kEpiThreads) bo[(size_t)sq * R * N + i] = Bm[tlg * R * N + i];
            for (int i = et; i < R * kP; i += kEpiThreads) xo[(size_t)sq * R * kP + i] = xm[tl * R * kP + i];
        };
        // fp16 copy of the state (scaled) for the C~ H MMA (MN-major, 128-byte swizzle, rows n)
        auto publish_state = [&](int slot_parity, float m) {
            if (!OUT) return;
            m = warp_max(m);
            if (lane == 0) mxH[slot_parity * kEpiWarps + ew] = m;
            named_sync(kBarEpi, kEpiThreads);
            float M = 0.f;
#pragma unroll
            for (int q = 0; q < kEpiWarps; ++q) M = fmaxf(M, mxH[slot_parity * kEpiWarps + q]);
            const float sg = pow2_scale(M);
            if (ew == 0 && lane == 0) {
                sigH[slot_parity] = sg;
                sigH[2 + slot_parity] = pow2_inv(sg);
            }
            constexpr int kCols = kState16 ? 16 : 32;   // columns per thread
            uint32_t hv[32];
            if constexpr (kState16) {
                tmem_ld16x2_nw(hcol, hv);
                tmem_wait_ld16(hv);
            } else {
                tmem_ld16_nw(hcol, hv);
                tmem_ld16_nw(hcol + 16, hv + 16);
                tmem_wait_ld(hv);
            }
#pragma unroll
            for (int q4 = 0; q4 < kCols / 8; ++q4) {
                if (!up_own) break;
                uint32_t w4[4];
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    const float2 v2 = __fmul2_rn(f2u(hv[8 * q4 + 2 * e2], hv[8 * q4 + 2 * e2 + 1]), f2(sg));
                    w4[e2] = pack_f16x2(v2.x, v2.y);
                }
                *reinterpret_cast<uint4 *>(sm + S::oH + sw128(up_row, up_col + 8 * q4)) =
                    make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
        };

        // the first piece's start state; a later piece's is loaded where the piece before ends (below), so
        // that the loop holds one copy of the load and of the fp16 publication (instruction cache)
        publish_state(0, load_start(piece_at(0)));
        fence_proxy_async();
        fence_before();
        mbar_arrive(bars + kStateReady + 0);
        Pos eu = piece_at(0);
        int it = 0;
        // pieces (one without the balanced plan), then their chunks: a later piece's start state is loaded
        // and published here, outside the chunk loop, whose code then holds none of it (instruction cache)
        for (int pi = 0; pi < (BAL ? npc : 1); ++pi) {
        if constexpr (BAL) {
            if (pi > 0) {
                eu = piece_at(pi);
                const float hm = load_start(eu);
                publish_state(it & 1, hm);
                fence_proxy_async();
                fence_before();
                mbar_arrive(bars + kStateReady + (it & 1));
            }
        }
        for (; it < nchunks && (!BAL || eu.c < p_ce(eu)); ++it, ++eu.c) {
            const int p = it & 1;
            const uint32_t ph = (it >> 1) & 1;
            const int s0 = eu.c * Q, Qc = min(Q, t_stop - s0), e = Qc - 1;
            const float *cA2 = v_cA(p), *gv = v_g(p), *vj = v_vj(p), *sg = v_sig(p);
            const bool last_chunk = it == nchunks - 1;
            const bool piece_end = BAL && eu.c == p_ce(eu) - 1;   // (balanced plan) the last chunk of a piece
            // one thread waits for the chunk's vectors and first MMAs; the named barrier
            // releases the other epilogue warps without them polling
            if (ew == 0 && lane == 0) {
                wait(kTilesFull + p, ph);
                wait(kMma1 + p, ph);
            }
            named_sync(kBarEpi, kEpiThreads);
            fence_after();
            // ---- masked score -> TMEM (fp16, scaled by tauP)
            if (OUT) {
                constexpr int COLS = QR / 2;    // score columns per thread
                const int t = min(ti, Q - 1);
                const float ca = cA2[t], invBC = sg[3];   // tauP / (sB sC)
                const float gd = gv[t] * invBC;
                // token range of this warp's rows (warp-uniform): blocks past tmax are zero,
                // blocks ending before tmin need no causal test
                const int tmax = (kRowsM64 ? eq * 16 + 15 : eq * 32 + 31) / R;
                const int tmin = (kRowsM64 ? eq * 16 : eq * 32) / R;
                if constexpr (kRowsM64) {
                    // one 32-column block per warp half (COLS = 32); this thread: 16 of its columns
                    static_assert(COLS == 32, "QR = 64");
                    constexpr int TH = TB / 2;            // tokens of 16 columns
                    const int cb = eh * COLS, btok = eh * TB, tq0 = hf * TH;
                    uint32_t p8[8];
                    if (btok > tmax) {
#pragma unroll
                        for (int q = 0; q < 8; ++q) p8[q] = 0u;
                    } else {
                        uint32_t sv[16];
                        tmem_ld16x2_nw(tmem + lane_base + cS + cb, sv);
                        const float u = (btok < ti) ? fast_exp2(ca - cA2[btok]) * invBC : 0.f;
                        float um[TH];
#pragma unroll
                        for (int q = 0; q < TH; ++q) um[q] = u * vj[btok + tq0 + q];
                        tmem_wait_ld16(sv);
                        if (btok + TB <= tmin) {
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const float2 v2 = __fmul2_rn(f2u(sv[2 * q], sv[2 * q + 1]),
                                                             make_float2(um[(2 * q) / R], um[(2 * q + 1) / R]));
                                p8[q] = pack_f16x2(v2.x, v2.y);
                            }
                        } else {
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                float mz[2];
#pragma unroll
                                for (int z = 0; z < 2; ++z) {
                                    const int jq = (2 * q + z) / R;
                                    const int tj = btok + tq0 + jq;
                                    mz[z] = (tj < ti) ? um[jq] : ((tj == ti) ? gd : 0.f);
                                }
                                const float2 v2 = __fmul2_rn(f2u(sv[2 * q], sv[2 * q + 1]), make_float2(mz[0], mz[1]));
                                p8[q] = pack_f16x2(v2.x, v2.y);
                            }
                        }
                    }
                    tmem_st8x2(tmem + lane_base + cP + cb / 2, p8);
                } else {
#pragma unroll 1
                for (int cc = 0; cc < COLS; cc += 32) {
                    const int cb = eh * COLS + cc;   // first score column of this 32-column block
                    const int btok = (cb / 32) * TB; // first token of the block
                    uint32_t p16[16];
                    if (btok > tmax) {
#pragma unroll
                        for (int q = 0; q < 16; ++q) p16[q] = 0u;
                    } else {
                        uint32_t sv[32];
                        tmem_ld16_nw(tmem + lane_base + cS + cb, sv);
                        tmem_ld16_nw(tmem + lane_base + cS + cb + 16, sv + 16);
                        // exp2(cA_t - cA_btok) <= 1 wherever it is used (btok <= tj < t)
                        const float u = (btok < ti) ? fast_exp2(ca - cA2[btok]) * invBC : 0.f;
                        if (R == 1 && YB == 4 && btok + TB <= tmin) {
                            // SISO block wholly before the row's token: (S o vj) u on packed pairs, no
                            // per-column factors (fp32 y only: the 16-bit-y builds schedule it 6 % slower)
                            float4 v4[TB / 4];
#pragma unroll
                            for (int q = 0; q < TB / 4; ++q) v4[q] = *reinterpret_cast<const float4 *>(vj + btok + 4 * q);
                            tmem_wait_ld(sv);
#pragma unroll
                            for (int q = 0; q < 16; ++q) {
                                const float4 w4 = v4[q / 2];
                                const float2 w2 = (q & 1) ? make_float2(w4.z, w4.w) : make_float2(w4.x, w4.y);
                                const float2 v2 = __fmul2_rn(__fmul2_rn(f2u(sv[2 * q], sv[2 * q + 1]), w2), f2(u));
                                p16[q] = pack_f16x2(v2.x, v2.y);
                            }
                            tmem_st16(tmem + lane_base + cP + cb / 2, p16);
                            continue;
                        }
                        float um[TB];
#pragma unroll
                        for (int q = 0; q < TB; q += 4) {
                            const float4 v4 = *reinterpret_cast<const float4 *>(vj + btok + q);
                            um[q] = u * v4.x;
                            if (q + 1 < TB) um[q + 1] = u * v4.y;
                            if (q + 2 < TB) um[q + 2] = u * v4.z;
                            if (q + 3 < TB) um[q + 3] = u * v4.w;
                        }
                        tmem_wait_ld(sv);
                        if (btok + TB <= tmin) {
#pragma unroll
                            for (int q = 0; q < 16; ++q) {
                                const float2 v2 = __fmul2_rn(f2u(sv[2 * q], sv[2 * q + 1]),
                                                             make_float2(um[(2 * q) / R], um[(2 * q + 1) / R]));
                                p16[q] = pack_f16x2(v2.x, v2.y);
                            }
                        } else {
#pragma unroll
                            for (int q = 0; q < 16; ++q) {
                                float mz[2];
#pragma unroll
                                for (int z = 0; z < 2; ++z) {
                                    const int jq = (2 * q + z) / R;   // token offset in the block
                                    const int tj = btok + jq;
                                    mz[z] = (tj < ti) ? um[jq] : ((tj == ti) ? gd : 0.f);
                                }
                                const float2 v2 = __fmul2_rn(f2u(sv[2 * q], sv[2 * q + 1]), make_float2(mz[0], mz[1]));
                                p16[q] = pack_f16x2(v2.x, v2.y);
                            }
                        }
                    }
                    tmem_st16(tmem + lane_base + cP + cb / 2, p16);
                }
                }
                fence_before();
                mbar_arrive(bars + kPReady + p);
            }
            // ---- state update: H <- R(phi_e) [exp(cA_e) H + Sn]
            {
                const float rho = fast_exp2(cA2[e]), invBX = sg[4];
                const int n = up_row, kk = n >> 1;
                const float c = up_own ? v_cos(p)[kk] : 1.f, s = up_own ? v_sin(p)[kk] : 0.f;
                const bool odd = n & 1;
                float *dst = nullptr;
                if constexpr (BAL) {
                    if (piece_end && up_own && !*abort_flag) {
                        if (p_ce(eu) < ncs) dst = a.ws_state + ((size_t)blockIdx.x * N + n) * kP + up_col;   // hand-off
                        else if (a.h_out) dst = a.h_out + ((size_t)p_seq(eu) * N + n) * kP + up_col;
                    }
                } else if (last_chunk && up_own && !*abort_flag) {
                    if (!OUT) dst = a.ws_state + (((size_t)bh * ws_stride + g + 1) * N + n) * kP + up_col;
                    else if (g == nseg - 1 && a.h_out) dst = a.h_out + ((size_t)bh * N + n) * kP + up_col;
                }
                float m = 0.f;
                // 16 columns: sh [0, 16) Sn, [16, 32) H -> hv; the pair partner (row n ^ 1) is lane ^ 1
                auto update16 = [&](const uint32_t *sh, uint32_t *hv, float *d) {
                    const float sgn_s = odd ? s : -s;
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        const float2 v = __ffma2_rn(f2(rho), f2u(sh[16 + j], sh[16 + j + 1]),
                                                    __fmul2_rn(f2u(sh[j], sh[j + 1]), f2(invBX)));
                        const float2 pv = make_float2(__shfl_xor_sync(0xffffffffu, v.x, 1),
                                                      __shfl_xor_sync(0xffffffffu, v.y, 1));
                        const float2 nv = __ffma2_rn(f2(sgn_s), pv, __fmul2_rn(f2(c), v));
                        m = fmaxf(m, up_own ? fmaxf(fabsf(nv.x), fabsf(nv.y)) : 0.f);
                        hv[j] = __float_as_uint(nv.x);
                        hv[j + 1] = __float_as_uint(nv.y);
                    }
                    if (d) {
#pragma unroll
                        for (int j = 0; j < 16; j += 4)
                            *reinterpret_cast<float4 *>(d + j) =
                                make_float4(__uint_as_float(hv[j]), __uint_as_float(hv[j + 1]),
                                            __uint_as_float(hv[j + 2]), __uint_as_float(hv[j + 3]));
                    }
                };
                if constexpr (kState16) {
                    uint32_t sh[32];
                    tmem_ld16x2_nw(tmem + lane_base + cSn + 32 * eh, sh);
                    tmem_ld16x2_nw(hcol, sh + 16);
                    tmem_wait_ld(sh);
                    uint32_t hv[16];
                    update16(sh, hv, dst);
                    tmem_st16x2(hcol, hv);
                } else {
#pragma unroll
                    for (int h16 = 0; h16 < 32; h16 += 16) {
                        uint32_t sh[32];
                        tmem_ld16_nw(tmem + lane_base + cSn + 32 * eh + h16, sh);
                        tmem_ld16_nw(hcol + h16, sh + 16);
                        tmem_wait_ld(sh);
                        uint32_t hv[16];
                        update16(sh, hv, dst ? dst + h16 : nullptr);
                        tmem_st16(hcol + h16, *reinterpret_cast<const uint32_t(*)[16]>(hv));
                    }
                }
                if constexpr (BAL) {
                    if (piece_end) {
                        if (p_ce(eu) < ncs) {
                            // this CTA's head state is in its slot: release it to the CTA after
                            __threadfence();
                            named_sync(kBarEpi, kEpiThreads);
                            if (ew == 0 && lane == 0) flag_release(hflags + blockIdx.x, epoch);
                        } else {
                            carry_out(eu);
                        }
                    }
                }
                if (!(piece_end && it + 1 < nchunks)) {   // (a next piece publishes its own start state)
                    publish_state((it + 1) & 1, m);
                    fence_proxy_async();
                    fence_before();
                    mbar_arrive(bars + kStateReady + ((it + 1) & 1));
                }
            }
            // ---- y = Ya + exp(cA_t) Yi
            if (OUT) {
                if (ew == 0 && lane == 0) {
                    wait(kMma2 + p, ph);
                    bulk_wait_read<0>();   // the previous chunk's y stores have left the staging tile
                }
                named_sync(kBarEpi, kEpiThreads);
                fence_after();
                const float sc = fast_exp2(cA2[min(ti, Q - 1)]) * sg[5] * sigH[2 + p], sa = sg[6];
                // the last read of this chunk's vectors (and MMA 2, the last reader of its x' tile, is
                // done): the prologue may refill them while y is formed
                mbar_arrive(bars + kEpiDone + p);
                // y rows go through a shared-memory tile (this thread: row `row`, columns
                // [32 eh, 32 eh + 32), or with QR = 64 the 16 of them at 16 hf) and leave by TMA: rows past
                // the sequence end are clipped by the map, and the global writes are whole lines
#pragma unroll 1
                for (int half16 = 16 * hf; half16 < 32; half16 += (kRowsM64 ? 32 : 16)) {
                    uint32_t yy[32];   // [0, 16): Ya, [16, 32): Yi
                    if constexpr (kRowsM64) {
                        tmem_ld16x2_nw(tmem + lane_base + cYa + 32 * eh, yy);
                        tmem_ld16x2_nw(tmem + lane_base + cYi0 + 64 * p + 32 * eh, yy + 16);
                    } else {
                        tmem_ld16_nw(tmem + lane_base + cYa + 32 * eh + half16, yy);
                        tmem_ld16_nw(tmem + lane_base + cYi0 + 64 * p + 32 * eh + half16, yy + 16);
                    }
                    tmem_wait_ld(yy);
                    const uint32_t *ya = yy, *yi = yy + 16;
                    {
                        if constexpr (YB == 4) {
                            // fp32: two halves [QR][32] of 128-byte rows
                            unsigned char *ys = sm + S::oYs + eh * (QR * 128);
#pragma unroll
                            for (int j = 0; j < 16; j += 4) {
                                const float2 u0 = __ffma2_rn(f2(sc), f2u(yi[j], yi[j + 1]),
                                                             __fmul2_rn(f2(sa), f2u(ya[j], ya[j + 1])));
                                const float2 u1 = __ffma2_rn(f2(sc), f2u(yi[j + 2], yi[j + 3]),
                                                             __fmul2_rn(f2(sa), f2u(ya[j + 2], ya[j + 3])));
                                *reinterpret_cast<float4 *>(ys + sw128f(row, half16 + j)) =
                                    make_float4(u0.x, u0.y, u1.x, u1.y);
                            }
                        } else {
                            // 16-bit: one [QR][64] tile of 128-byte rows, rounded once from fp32
                            uint32_t w[8];
#pragma unroll
                            for (int j = 0; j < 16; j += 2) {
                                const float2 u = __ffma2_rn(f2(sc), f2u(yi[j], yi[j + 1]),
                                                            __fmul2_rn(f2(sa), f2u(ya[j], ya[j + 1])));
                                w[j / 2] = YT == M3_F16 ? pack_f16x2(u.x, u.y) : pack_bf16x2(u.x, u.y);
                            }
                            const int c0 = 32 * eh + half16;
                            *reinterpret_cast<uint4 *>(sm + S::oYs + sw128(row, c0)) = make_uint4(w[0], w[1], w[2], w[3]);
                            *reinterpret_cast<uint4 *>(sm + S::oYs + sw128(row, c0 + 8)) =
                                make_uint4(w[4], w[5], w[6], w[7]);
                        }
                    }
                }
                fence_proxy_async();
                named_sync(kBarEpi, kEpiThreads);
                if (ew == 0 && lane == 0) {
                    if (!*abort_flag) {
                        tma_store_5d(&maps.Y, sm + S::oYs, 0, 0, p_qh(eu), s0, p_qb(eu));
                        if (YB == 4) tma_store_5d(&maps.Y, sm + S::oYs + QR * 128, 32, 0, p_qh(eu), s0, p_qb(eu));
                    }
                    bulk_commit();
                }
            }
            if (!OUT) mbar_arrive(bars + kEpiDone + p);
        }
        }
        if (OUT && ew == 0 && lane == 0) bulk_wait<0>();
        // ---- carry out (last segment; the balanced plan wrote it at each sequence's end)
        if (!BAL && g == nseg - 1) carry_out(piece_at(0));
    }
    fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- host side
// L2 promotion of the loads through a map: how far past the requested bytes a fetch into L2 extends.
// 256 bytes suits launches whose CTAs read neighbouring heads' rows of a token at the same time; a
// launch whose CTAs do not (the balanced pass) promotes no further than one head's contiguous row.
CUtensorMapL2promotion promo_for(int row_bytes) {
    return row_bytes <= 64 ? CU_TENSOR_MAP_L2_PROMOTION_L2_64B
                           : (row_bytes <= 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

// 5-d map over a [batch][L][H][R][inner] bf16 tensor, box = {64, R, 1, Q, 1}, 128-byte swizzle.  Token
// rows past a sequence's end are outside the map and arrive as zeros.
bool map5(CUtensorMap *m, const void *base, int inner, int R, int H, int L, int batch, int Q,
          CUtensorMapL2promotion prom = CU_TENSOR_MAP_L2_PROMOTION_L2_256B) {
    EncodeFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[5] = {(cuuint64_t)inner, (cuuint64_t)R, (cuuint64_t)H, (cuuint64_t)L, (cuuint64_t)batch};
    const cuuint64_t row = (cuuint64_t)inner * 2 * R * H;   // bytes per token
    const cuuint64_t strides[4] = {(cuuint64_t)inner * 2, (cuuint64_t)inner * 2 * R, row, row * (cuuint64_t)L};
    const cuuint32_t box[5] = {64, (cuuint32_t)R, 1, (cuuint32_t)Q, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, prom,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// 4-d map over a [batch][L][H][inner] bf16 tensor, box = {inner, 1, Q, 1} (rows past the end arrive as zeros)
bool map4t(CUtensorMap *m, const void *base, int inner, int H, int L, int batch, int Q,
           CUtensorMapL2promotion prom = CU_TENSOR_MAP_L2_PROMOTION_L2_256B) {
    EncodeFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)H, (cuuint64_t)L, (cuuint64_t)batch};
    const cuuint64_t row = (cuuint64_t)inner * 2 * H;
    const cuuint64_t strides[3] = {(cuuint64_t)inner * 2, row, row * (cuuint64_t)L};
    const cuuint32_t box[4] = {(cuuint32_t)inner, 1, (cuuint32_t)Q, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, prom,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 5-d map over y [batch][L][H][R][64] of type yd: box = {32, R, 1, Q, 1} for fp32, {64, R, 1, Q, 1}
// for 16-bit y (128-byte lines either way), 128-byte swizzle
bool map_y(CUtensorMap *m, void *base, int yd, int R, int H, int L, int batch, int Q) {
    EncodeFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t eb = yd == M3_F32 ? 4 : 2;
    const cuuint64_t dims[5] = {64, (cuuint64_t)R, (cuuint64_t)H, (cuuint64_t)L, (cuuint64_t)batch};
    const cuuint64_t strides[4] = {64 * eb, (cuuint64_t)R * 64 * eb, (cuuint64_t)H * R * 64 * eb,
                                   (cuuint64_t)L * H * R * 64 * eb};
    const cuuint32_t box[5] = {(cuuint32_t)(128 / eb), (cuuint32_t)R, 1, (cuuint32_t)Q, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    const CUtensorMapDataType ty = yd == M3_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : yd == M3_F16  ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    return enc(m, ty, 5, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int N, int R, bool OUT, int YT = M3_F32, bool BCN = false, int QRT = (N == 64 ? 128 : 64)>
// ws_stride: workspace state slots per sequence; ws_step: slots per segment of this pass
cudaError_t launch_pass(const TcMaps &maps, const ScanArgs &a, const ScanPlan &pl, int nlaunch, int ws_stride,
                        int ws_step, cudaStream_t s) {
    using Sm = Smem<N, R, OUT, YT == M3_F32 ? 4 : 2, BCN, QRT>;
    static_assert(Sm::kAlloc <= 227 * 1024, "shared memory over the per-CTA limit");
    auto kern = tc_segment_kernel<N, R, OUT, YT, BCN, QRT>;
    cudaError_t e = allow_dynamic_smem<tc_segment_kernel<N, R, OUT, YT, BCN, QRT>>(Sm::kAlloc);
    if (e != cudaSuccess) return e;
    unsigned *status = device_status_word();
    if (!status) return cudaErrorUnknown;
    const long long grid = (long long)a.batch * a.H * nlaunch;
    const int kid = OUT ? M3_KERNEL_PREFILL_OUTPUT : M3_KERNEL_PREFILL_STATE;
    // a programmatic dependent of the kernel before it in the stream (see the kernel's set-up)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Sm::kAlloc;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    trace_mark(kid, s, 0);
    e = cudaLaunchKernelEx(&cfg, kern, maps, a, pl.seglen, pl.nseg, nlaunch, ws_stride, ws_step, status, 0ull, 0);
    trace_mark(kid, s, 1);
    if (e != cudaSuccess) return e;
    count_launch();
    return cudaGetLastError();
}

// A fresh value of the hand-off flags per balanced launch (so that flags left in a reused workspace never
// match); the start is taken from the clock so that another process's leftovers do not either.
unsigned long long next_epoch() {
    static std::atomic<unsigned long long> e{0};
    unsigned long long v = e.fetch_add(1) + 1;
    static const unsigned long long base =
        (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count() * 0x9E3779B97F4A7C15ull;
    return (base + v) | 1ull;   // never 0
}

// The balanced output pass (one segment): pl.bal CTAs, all resident at once (a cooperative launch, which
// fails rather than runs them in turns); returns cudaErrorCooperativeLaunchTooLarge when they cannot be.
template <int N, int R, int YT, int QRT>
cudaError_t launch_bal(const TcMaps &maps, const ScanArgs &a, const ScanPlan &pl, cudaStream_t s) {
    using Sm = Smem<N, R, true, YT == M3_F32 ? 4 : 2, false, QRT>;
    auto kern = tc_segment_kernel<N, R, true, YT, false, QRT, true>;
    cudaError_t e = allow_dynamic_smem<tc_segment_kernel<N, R, true, YT, false, QRT, true>>(Sm::kAlloc);
    if (e != cudaSuccess) return e;
    int dev = 0, per_sm = 0, coop = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    if (!coop || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, Sm::kAlloc) != cudaSuccess ||
        per_sm * sm_count() < pl.bal)
        return cudaErrorCooperativeLaunchTooLarge;
    unsigned *status = device_status_word();
    if (!status) return cudaErrorUnknown;
    int seglen = pl.seglen, nseg = 1, nlaunch = 1, ws_stride = 1, ws_step = 1, nbal = pl.bal;
    unsigned long long epoch = next_epoch();
    void *args[] = {(void *)&maps, (void *)&a, &seglen, &nseg, &nlaunch, &ws_stride, &ws_step, &status, &epoch, &nbal};
    trace_mark(M3_KERNEL_PREFILL_OUTPUT, s, 0);
    e = cudaLaunchCooperativeKernel((const void *)kern, dim3(pl.bal), dim3(kThreads), args, Sm::kAlloc, s);
    trace_mark(M3_KERNEL_PREFILL_OUTPUT, s, 1);
    if (e == cudaSuccess) count_launch();
    return e;
}

template <int N, int R, bool BCN, int QRT = (N == 64 ? 128 : 64)>
cudaError_t run_tc(const ScanArgs &a, const ScanPlan &pl, cudaStream_t s) {
    using Cf = Cfg<N, R, QRT>;
    const int L = a.L, nb = a.batch;
    TcMaps maps;
    if (!map5(&maps.B, a.B, N, R, a.G, L, nb, Cf::Q) || !map5(&maps.C, a.C, N, R, a.G, L, nb, Cf::Q) ||
        !map5(&maps.X, a.x, kP, R, a.H, L, nb, Cf::Q) || !map4t(&maps.T, a.theta, N / 2, a.H, L, nb, Cf::Q) ||
        !map_y(&maps.Y, a.y, a.ydtype, R, a.H, a.L, a.batch, Cf::Q))
        return cudaErrorInvalidValue;
    cudaError_t e;
    // The state pass works on pieces of seglen / nsub tokens (one CTA each) covering segments
    // 0 .. nseg - 2; the segment pass chains the pieces' end states; the output pass starts
    // segment g from the state at piece g * nsub.
    const int npieces = pl.nseg > 1 ? (pl.nseg - 1) * pl.nsub + 1 : 1;
    if (pl.nseg > 1) {
        ScanPlan pp = pl;
        pp.nseg = npieces;
        pp.seglen = pl.seglen / pl.nsub;
        // The state pass holds no score, output or state-copy tiles, so with N = 128 its chunk takes twice
        // the rows of the output pass's (the per-chunk state update then serves twice the tokens).  A CTA
        // starts at a whole chunk (its first is t_begin / Q), so the pieces must be whole chunks of it; the
        // planner cuts them so, and a plan that is not gets the output pass's chunk here.
        constexpr int QRS = (N == 128 && QRT == 64) ? 128 : QRT;
        using Cs = Cfg<N, R, QRS>;
        if (QRS != QRT && pp.seglen % Cs::Q == 0) {
            TcMaps smaps = maps;
            if (!map5(&smaps.B, a.B, N, R, a.G, L, nb, Cs::Q) || !map5(&smaps.X, a.x, kP, R, a.H, L, nb, Cs::Q) ||
                !map4t(&smaps.T, a.theta, N / 2, a.H, L, nb, Cs::Q))
                return cudaErrorInvalidValue;
            e = launch_pass<N, R, false, M3_F32, BCN, QRS>(smaps, a, pp, npieces - 1, npieces, 1, s);
        } else {
            e = launch_pass<N, R, false, M3_F32, BCN, QRT>(maps, a, pp, npieces - 1, npieces, 1, s);
        }
        if (e != cudaSuccess) return e;
        if ((e = segment_pass(a, pp, s)) != cudaSuccess) return e;
    }
    if constexpr (!BCN) {
        if (pl.bal > 0 && pl.nseg == 1) {
            // rows of one (token, head): B and C R N, x R P, theta N / 2 elements (a 64-wide slab of each
            // B and C row for N = 128, the neighbouring slab loaded next)
            TcMaps bm = maps;
            if (!map5(&bm.B, a.B, N, R, a.G, L, nb, Cf::Q, promo_for(R * 64 * 2)) ||
                !map5(&bm.C, a.C, N, R, a.G, L, nb, Cf::Q, promo_for(R * 64 * 2)) ||
                !map5(&bm.X, a.x, kP, R, a.H, L, nb, Cf::Q, promo_for(R * kP * 2)) ||
                !map4t(&bm.T, a.theta, N / 2, a.H, L, nb, Cf::Q, promo_for(N)))
                return cudaErrorInvalidValue;
            cudaError_t eb = a.ydtype == M3_F16    ? launch_bal<N, R, M3_F16, QRT>(bm, a, pl, s)
                             : a.ydtype == M3_BF16 ? launch_bal<N, R, M3_BF16, QRT>(bm, a, pl, s)
                                                   : launch_bal<N, R, M3_F32, QRT>(bm, a, pl, s);
            if (eb != cudaErrorCooperativeLaunchTooLarge) return eb;
            cudaGetLastError();   // not resident at once here: the plain plan below
        }
    }
    if (a.ydtype == M3_F16)
        return launch_pass<N, R, true, M3_F16, BCN, QRT>(maps, a, pl, pl.nseg, npieces, pl.nsub, s);
    if (a.ydtype == M3_BF16)
        return launch_pass<N, R, true, M3_BF16, BCN, QRT>(maps, a, pl, pl.nseg, npieces, pl.nsub, s);
    return launch_pass<N, R, true, M3_F32, BCN, QRT>(maps, a, pl, pl.nseg, npieces, pl.nsub, s);
}

}  // namespace
}  // namespace m3
