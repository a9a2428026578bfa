// Chunked prefill on the tensor cores: planning and dispatch.  The kernel itself is in
// m3_scan_tc.cuh (a warp-specialised tcgen05 / TMA pipeline; see there), instantiated by
// m3_scan_tc_n64.cu, m3_scan_tc_n64_bc.cu, m3_scan_tc_n128.cu and m3_scan_tc_n128_bc.cu.
#include "m3_internal.cuh"

namespace m3 {

// the per-(N, BC variant) instantiations
cudaError_t tc_scan_n64(const ScanArgs &a, const ScanPlan &pl, cudaStream_t s);
cudaError_t tc_scan_n64_bc(const ScanArgs &a, const ScanPlan &pl, cudaStream_t s);
cudaError_t tc_scan_n128(const ScanArgs &a, const ScanPlan &pl, cudaStream_t s);
cudaError_t tc_scan_n128_bc(const ScanArgs &a, const ScanPlan &pl, cudaStream_t s);
cudaError_t tc_scan_n64_q64(const ScanArgs &a, const ScanPlan &pl, cudaStream_t s);
cudaError_t tc_scan_n64_q64_bc(const ScanArgs &a, const ScanPlan &pl, cudaStream_t s);

namespace {

// tokens per chunk of the default tile (128 rows (t, r) for N = 64, 64 for N = 128)
int tc_chunk(int N, int R) { return (N == 64 ? 128 : 64) / R; }

// tokens per chunk of the state pass: 128 rows for both N (it has room for them with N = 128)
int tc_state_chunk(int N, int R, int Q) { return N == 128 ? 128 / R : Q; }

// The chunk rule of the pages, Q = N / R tokens (N rows per chunk): a tile of its own for N = 64,
// R <= 4 (N = 128 would need 128-row tiles of B, C and theta that do not fit shared memory).
bool tc_rule_chunk(int N, int R, int chunk) { return N == 64 && R <= 4 && chunk == N / R; }

}  // namespace

bool tc_supported(const m3_dims &d) {
    if (d.dtype != M3_BF16 || d.headdim != 64) return false;
    if (d.dstate != 64 && d.dstate != 128) return false;
    if (d.rank != 1 && d.rank != 2 && d.rank != 4 && d.rank != 8) return false;
    if (d.chunk != 0 && d.chunk != tc_chunk(d.dstate, d.rank) && !tc_rule_chunk(d.dstate, d.rank, d.chunk))
        return false;
    if ((long long)d.batch * d.seqlen >= (1LL << 31)) return false;   // TMA row coordinates are int32
    return true;
}

bool tc_plan(const m3_dims &d, int sms, ScanPlan *pl) {
    if (!tc_supported(d)) return false;
    const int Q = tc_rule_chunk(d.dstate, d.rank, d.chunk) ? d.chunk : tc_chunk(d.dstate, d.rank);
    const long long seqs = (long long)d.batch * d.nheads;
    const int L = d.seqlen;
    int nseg = 1;
    if (seqs > 0 && L > 0 && seqs < (long long)(0.8 * sms)) {
        // fill the SMs with one wave of CTAs (one per SM; a second, partial wave would
        // double the time of the output pass); segments of at least 8 chunks
        const int max_seg = (L + 8 * Q - 1) / (8 * Q);
        long long want = sms / seqs;
        nseg = (int)(want < max_seg ? want : max_seg);
        if (nseg < 1) nseg = 1;
    }
    // segments and the state pass's pieces are whole chunks of the pass that walks them: a segment
    // of the output pass's chunks, a piece of the state pass's
    const int Qs = nseg > 1 ? tc_state_chunk(d.dstate, d.rank, Q) : Q;
    int seglen = L > 0 ? (L + nseg - 1) / nseg : Q;
    seglen = ((seglen + Qs - 1) / Qs) * Qs;
    nseg = L > 0 ? (L + seglen - 1) / seglen : 1;
    // the state pass covers segments 0 .. nseg - 2, cut into nsub whole pieces (of at least 8 output-pass
    // chunks) each: one CTA a piece, in as many waves as it takes.  Its time goes as waves / nsub (a
    // wave lasts one piece), so nsub is the smallest count that minimises that: more, shorter pieces
    // let the last wave fill the SMs (64 sequences: 16 pieces, 7 waves, 0.4375 of a segment a CTA
    // slot against 0.5 for one wave of 2 pieces)
    int nsub = 1;
    if (nseg > 1) {
        const long long units = seqs * (nseg - 1);
        const int chunks = seglen / Q, schunks = seglen / Qs;
        double best = (double)((units + sms - 1) / sms);
        for (int c = 2; c <= 64 && chunks / c >= 8; ++c) {
            if (schunks % c) continue;
            const double t = (double)((units * c + sms - 1) / sms) / c;
            if (t < best - 1e-9) {
                best = t;
                nsub = c;
            }
        }
    }
    pl->Q = Q;
    pl->nseg = nseg;
    pl->seglen = seglen;
    pl->nsub = nsub;
    pl->path = kPathTc;
    pl->ws_bytes = scan_workspace_bytes(d.batch, d.nheads, d.dstate, d.headdim,
                                        nseg > 1 ? (nseg - 1) * nsub + 1 : 1);
    // More sequences than SMs in a last wave that would leave a tenth of the machine idle: the balanced
    // output pass (one CTA per SM, equal shares of all sequences' chunks, a state slot and a flag per
    // CTA).  Not with the chunk-rule tile (its own instantiation) or BC normalisation (falls back).
    pl->bal = 0;
    if (nseg == 1 && seqs > sms && Q * d.rank == (d.dstate == 64 ? 128 : 64)) {
        const long long waves = (seqs + sms - 1) / sms;
        if ((double)seqs / (double)(waves * sms) < 0.9) {
            pl->bal = sms;
            const size_t need = (size_t)sms * d.dstate * d.headdim * sizeof(float) + (size_t)sms * 8;
            if (need > pl->ws_bytes) pl->ws_bytes = need;
        }
    }
    return true;
}

cudaError_t tc_scan(const ScanArgs &a, const ScanPlan &pl, cudaStream_t s) {
    // the chunk rule Q = N / R has a tile of its own (the plan's segments are whole chunks of it)
    if (a.N == 64 && pl.Q * a.R == 64) return a.bc.on ? tc_scan_n64_q64_bc(a, pl, s) : tc_scan_n64_q64(a, pl, s);
    if (a.N == 64) return a.bc.on ? tc_scan_n64_bc(a, pl, s) : tc_scan_n64(a, pl, s);
    if (a.N == 128) return a.bc.on ? tc_scan_n128_bc(a, pl, s) : tc_scan_n128(a, pl, s);
    return cudaErrorInvalidValue;
}

}  // namespace m3
