// Internal declarations of the Mamba-3 recurrence library (not part of the C ABI).
#pragma once

#include <atomic>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mamba3.h"

namespace m3 {

// ---------------------------------------------------------------- element types
__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// One element of y, rounded once (to nearest even) from fp32 to the output type `yd` (m3_dtype).
__device__ __forceinline__ void store_y(void *y, size_t i, float v, int yd) {
    if (yd == M3_F32) static_cast<float *>(y)[i] = v;
    else if (yd == M3_BF16) static_cast<__nv_bfloat16 *>(y)[i] = __float2bfloat16_rn(v);
    else static_cast<__half *>(y)[i] = __float2half_rn(v);
}

// Device status word bits (read and cleared by mamba3_device_status).
enum : unsigned { kStatusTimeout = 1u, kStatusBadIndex = 2u };

// ---------------------------------------------------------------- launch plumbing
void count_launch();                 // +1 to the library's launch counter
// Tracing marks around a launch of `kernel` (m3_kernel) on stream s:
// phase 0 just before the launch, phase 1 just after it.
void trace_mark(int kernel, cudaStream_t s, int phase);
unsigned *device_status_word();      // address of this device's status word (nullptr on error)
int sm_count();                      // SMs of the current device (cached)

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the current device.  The
// driver call (microseconds of host time) is made only when the limit has to grow.
constexpr int kSmemLimitDevices = 64;
template <auto Kern>
cudaError_t allow_dynamic_smem(size_t bytes) {
    static std::atomic<int> limit[kSmemLimitDevices];
    int dev = -1;
    cudaGetDevice(&dev);
    const bool cached = dev >= 0 && dev < kSmemLimitDevices;
    if (cached && limit[dev].load(std::memory_order_acquire) >= (int)bytes) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess && cached) {
        int cur = limit[dev].load(std::memory_order_relaxed);
        while (cur < (int)bytes && !limit[dev].compare_exchange_weak(cur, (int)bytes)) {
        }
    }
    return e;
}
void *tensor_map_encoder();          // the driver's cuTensorMapEncodeTiled (nullptr if unavailable)
cudaStream_t input_stream();         // the staged prefill's stream for copies in (this device; nullptr on error)

// ---------------------------------------------------------------- prefill plan
// Prefill runs over segments of `seglen` tokens (a multiple of the chunk Q).
// Segment g of every (b, h) sequence starts from state H'_g:
//   - pass 1 (segment_state, g < nseg-1): state at the segment end from a zero
//     start, plus the segment's total log-decay and angles;
//   - pass 2 (segment_pass): H'_0 = h0 + carry term, H'_{g+1} = T_g H'_g + S_g;
//   - pass 3 (segment_output): y for every token of the segment and, for the
//     last segment, the final state and carry.
// With nseg == 1 only pass 3 runs and it reads h0 and the carry itself.
struct ScanPlan {
    int Q;        // tokens per chunk
    int nseg;     // segments per sequence
    int seglen;   // tokens per segment (multiple of Q), last one may be shorter
    int nsub;     // state-pass pieces per segment (the pass that feeds the segment starts)
    int path;     // kPathSimt or kPathTc
    int bal;      // > 0: the balanced output pass on this many CTAs (tensor-core path, one segment)
    size_t ws_bytes;
};
enum { kPathSimt = 0, kPathTc = 1 };

// BC normalisation and bias (m3_bc_norm); on = 0: B and C enter the recurrence as given.
struct BcNorm {
    const float *wB, *bB, *wC, *bC;   // [H][N] gains (null = 1), [H][R][N] biases (null = 0)
    float eps;
    int on;
};

// The normalised value of entry n of a row whose inverse RMS is `inv` (head h, rank r).
__device__ __forceinline__ float bc_apply(float v, float inv, const float *w, const float *bias, int h, int r,
                                          int R, int N, int n) {
    const float g = w ? __ldg(w + (size_t)h * N + n) : 1.f;
    const float c = bias ? __ldg(bias + ((size_t)h * R + r) * N + n) : 0.f;
    return fmaf(v * inv, g, c);
}

struct ScanArgs {
    int dtype, ydtype, batch, L, H, P, N, R;
    BcNorm bc;
    int G;                      // B / C groups (G = H: one per head)
    const void *x, *B, *C, *dt, *A, *lam, *theta;
    const float *h0;            // may be null (zero state)
    const void *Bprev, *xprev;  // may be null (no carry)
    void *y;
    float *h_out;               // may be null
    void *Bprev_out, *xprev_out;  // may be null
    float *ws_state;            // [b*H][nseg][N][P]  (nseg > 1)
    float *ws_tot;              // [b*H][nseg-1][1 + N/2]
};

// Backward pass (mamba3_scan_bwd): forward inputs, incoming and outgoing gradients (fp32).
struct BwdArgs {
    int dtype, batch, L, H, P, N, R;
    const void *x, *B, *C, *dt, *A, *lam, *theta;
    const float *h0;
    const void *Bprev, *xprev;
    const float *dy, *dh_out, *dBprev_out, *dxprev_out;
    float *dx, *dB, *dC, *ddt, *dA, *dlam, *dtheta, *dh0, *dBprev, *dxprev;
    float *ws;                  // [b*H][L/Q + 1][N][P] state checkpoints
};
// esz: bytes per element of the token inputs
int bwd_chunk(int N, int P, int R, int esz);                           // tokens per chunk
size_t bwd_smem_bytes(int N, int P, int R, int esz);
size_t bwd_workspace_bytes(int batch, int H, int L, int N, int P, int R, int esz);
cudaError_t scan_bwd(const BwdArgs &a, cudaStream_t s);

// Workspace layout sizes (bytes) for a plan.
size_t scan_workspace_bytes(int batch, int H, int N, int P, int nseg);

// SIMT path (any supported shape and dtype).
bool simt_plan(const m3_dims &d, int sms, ScanPlan *plan);   // false = unsupported
cudaError_t simt_scan(const ScanArgs &a, const ScanPlan &plan, cudaStream_t s);

// Tensor-core path (bf16, P = 64, N in {64, 128}, R in {1, 2, 4, 8}).
bool tc_supported(const m3_dims &d);
bool tc_plan(const m3_dims &d, int sms, ScanPlan *plan);      // false = unsupported
cudaError_t tc_scan(const ScanArgs &a, const ScanPlan &plan, cudaStream_t s);

// Segment state passing (shared by both paths).
cudaError_t segment_pass(const ScanArgs &a, const ScanPlan &plan, cudaStream_t s);

// Decode step.
// bc: BC normalisation (null or bc->on == 0: none; then the tensor-core kernel may serve the call)
cudaError_t decode_step(int dtype, int ydtype, int batch, int H, int G, int P, int N, int R, const void *x,
                        const void *B, const void *C, const void *dt, const void *A,
                        const void *lam, const void *theta, float *h, void *Bprev, void *xprev,
                        void *y, cudaStream_t s, const BcNorm *bc = nullptr);
// The tensor-core decode's shapes (pooled and grouped decode run only there), and the pooled launch.
bool decode_tc_ok(int dtype, int P, int N, int R, long long heads, const void *const *ptrs, int nptr);
cudaError_t decode_step_pooled(int ydtype, int batch, int H, int G, int P, int N, int R, const int *slot, int pool,
                               const void *x, const void *B, const void *C, const void *dt, const void *A,
                               const void *lam, const void *theta, float *h, void *Bprev, void *xprev, void *y,
                               cudaStream_t s);

}  // namespace m3
