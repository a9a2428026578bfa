// Instantiation of the tensor-core prefill for N = 128, with BC normalisation and bias.
#include "m3_scan_tc.cuh"

namespace m3 {

cudaError_t tc_scan_n128_bc(const ScanArgs &a, const ScanPlan &pl, cudaStream_t s) {
    switch (a.R) {
        case 1: return run_tc<128, 1, true>(a, pl, s);
        case 2: return run_tc<128, 2, true>(a, pl, s);
        case 4: return run_tc<128, 4, true>(a, pl, s);
        case 8: return run_tc<128, 8, true>(a, pl, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace m3
