// Self-test of the bounded device-side waits: a kernel waits on an mbarrier that nothing arrives at,
// with the same bounded wait the pipelines use, gives up after the limit and reports the timeout in
// the device status word; the context stays usable.
#include "m3_internal.cuh"
#include "m3_tc.cuh"

namespace m3 {
namespace {

__global__ void wait_timeout_kernel(uint64_t limit_ns, unsigned *status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        tc::mbar_init_fence();
    }
    __syncthreads();
    // no thread arrives on `bar` and no copy completes on it: phase 0 never completes
    const bool ok = tc::mbar_wait(&bar, 0, limit_ns);
    if (__syncthreads_or(!ok) && threadIdx.x == 0) atomicOr(status, kStatusTimeout);
}

}  // namespace
}  // namespace m3

extern "C" m3_status mamba3_selftest_wait_timeout(uint64_t limit_ns, void *stream) {
    if (limit_ns == 0 || limit_ns > 100000000ull) return M3_ERR_INVALID_ARG;   // (0, 100 ms]
    unsigned *status = m3::device_status_word();
    if (!status) return M3_ERR_CUDA;
    m3::wait_timeout_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, status);
    m3::count_launch();
    return cudaGetLastError() == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}
