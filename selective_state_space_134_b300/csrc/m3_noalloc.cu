// mamba3_scan_fwd_noalloc: the prefill for callers that cannot allocate device
// memory.  Its scratch (the per-segment states that the prefill passes hand to
// one another) lives in a static device array defined in this file instead of
// a caller-provided workspace.
#include <mutex>

#include "m3_internal.cuh"

// One copy per device that loads this library, held until the process exits.
static __device__ __align__(256) unsigned char m3_noalloc_scratch[M3_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices];   // device address of m3_noalloc_scratch, per device

// In host code `m3_noalloc_scratch` only names the symbol; its device address
// comes from cudaGetSymbolAddress, looked up once per device with that device
// current (the first call on each device does this).
m3_status scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return M3_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, m3_noalloc_scratch) != cudaSuccess || p == nullptr) return M3_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return M3_OK;
}

}  // namespace

extern "C" m3_status mamba3_scan_fwd_noalloc(const m3_dims *dims, const void *x, const void *B, const void *C,
                                             const void *dt, const void *A, const void *lambda,
                                             const void *theta, const m3_state *state_in, void *y,
                                             const m3_state *state_out, void *stream) {
    size_t need = 0;
    m3_status st = mamba3_scan_fwd_workspace(dims, &need);
    if (st != M3_OK) return st;
    if (need > (size_t)M3_NOALLOC_SCRATCH_BYTES) return M3_ERR_WORKSPACE;   // before any launch
    void *scratch = nullptr;
    if (need > 0 && dims->batch > 0 && dims->seqlen > 0) {
        if ((st = scratch_address(&scratch)) != M3_OK) return st;
    }
    // The prefill writes every scratch byte it reads before reading it, so the
    // previous call's leftovers need no clearing.
    return mamba3_scan_fwd(dims, x, B, C, dt, A, lambda, theta, state_in, y, state_out, scratch,
                           scratch ? (size_t)M3_NOALLOC_SCRATCH_BYTES : 0, stream);
}
