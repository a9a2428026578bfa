// Instantiation of the tensor-core prefill for N = 64.
#include "m3_scan_tc.cuh"

namespace m3 {

cudaError_t tc_scan_n64(const ScanArgs &a, const ScanPlan &pl, cudaStream_t s) {
    switch (a.R) {
        case 1: return run_tc<64, 1, false>(a, pl, s);
        case 2: return run_tc<64, 2, false>(a, pl, s);
        case 4: return run_tc<64, 4, false>(a, pl, s);
        case 8: return run_tc<64, 8, false>(a, pl, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace m3
