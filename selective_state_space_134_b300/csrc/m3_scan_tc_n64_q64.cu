// Instantiation of the tensor-core prefill for N = 64 with 64 rows (t, r) per chunk, i.e. the chunk
// rule Q = N / R tokens (linkstar.cloud/article/869, section "训练怎么办": the chunk length N / R keeps
// the chunked algorithm's cost at R times, not R^2 times, that of SISO); ranks 1, 2 and 4.
#include "m3_scan_tc.cuh"

namespace m3 {

cudaError_t tc_scan_n64_q64(const ScanArgs &a, const ScanPlan &pl, cudaStream_t s) {
    switch (a.R) {
        case 1: return run_tc<64, 1, false, 64>(a, pl, s);
        case 2: return run_tc<64, 2, false, 64>(a, pl, s);
        case 4: return run_tc<64, 4, false, 64>(a, pl, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace m3
