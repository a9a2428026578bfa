// Host side of the C ABI declared in include/mamba3.h: argument validation,
// planning of the prefill segments, kernel dispatch, status reporting.
#include <atomic>
#include <mutex>
#include <vector>

#include "m3_internal.cuh"

namespace m3 {

static std::atomic<uint64_t> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// ---- tracing: event pairs around the launches of one kernel
static std::mutex g_trace_mu;
static int g_trace_kernel = -1;
static int g_trace_max = 0;
static std::vector<cudaEvent_t> g_trace_ev;   // [2 * max]: start, stop
static int g_trace_n = 0;

void trace_mark(int kernel, cudaStream_t s, int phase) {
    std::lock_guard<std::mutex> lock(g_trace_mu);
    if (kernel != g_trace_kernel || g_trace_n >= g_trace_max) return;
    cudaEventRecord(g_trace_ev[2 * g_trace_n + phase], s);
    if (phase == 1) ++g_trace_n;
}

static void trace_release_locked() {
    for (cudaEvent_t e : g_trace_ev) cudaEventDestroy(e);
    g_trace_ev.clear();
    g_trace_kernel = -1;
    g_trace_max = 0;
    g_trace_n = 0;
}

// One status word per device (a module-scope __device__ variable exists once
// per device context); kernels set bits, mamba3_device_status reads + clears.
__device__ unsigned g_status_word;

static constexpr int kMaxDevices = 64;
static std::mutex g_mu;
static unsigned *g_status_ptr[kMaxDevices];
static int g_sms[kMaxDevices];

unsigned *device_status_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<unsigned *>(p);
    }
    return g_status_ptr[dev];
}

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_sms[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return 148;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

// The library's stream for the staged prefill's copies in, one per device (created on first use, kept for the
// life of the process); nullptr on error.
static cudaStream_t g_in_stream[kMaxDevices];
cudaStream_t input_stream() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_in_stream[dev] && cudaStreamCreateWithFlags(&g_in_stream[dev], cudaStreamNonBlocking) != cudaSuccess)
        g_in_stream[dev] = nullptr;
    return g_in_stream[dev];
}

void *tensor_map_encoder() {
    static std::once_flag once;
    static void *fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = p;
    });
    return fn;
}

}  // namespace m3

using namespace m3;

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape / dtype check shared by both entry points.
m3_status check_dims(const m3_dims *d, bool prefill) {
    if (!d) return M3_ERR_INVALID_ARG;
    if (d->batch < 0 || d->nheads < 1 || (prefill && d->seqlen < 0) || d->chunk < 0)
        return M3_ERR_INVALID_ARG;
    if (d->dtype != M3_F32 && d->dtype != M3_BF16) return M3_ERR_UNSUPPORTED;
    if (d->headdim < 1 || d->headdim > 128 || (d->headdim % 4) != 0) return M3_ERR_UNSUPPORTED;
    if (d->dstate < 2 || d->dstate > 256 || (d->dstate % 2) != 0) return M3_ERR_UNSUPPORTED;
    if (d->rank < 1 || d->rank > 8) return M3_ERR_UNSUPPORTED;
    if (d->ngroups < 0 || (d->ngroups > 0 && d->nheads % d->ngroups != 0)) return M3_ERR_INVALID_ARG;
    if (d->ydtype != M3_F32 && d->ydtype != M3_BF16 && d->ydtype != M3_F16) return M3_ERR_UNSUPPORTED;
    return M3_OK;
}

// B / C groups of a problem (ngroups = 0 means one per head)
int groups_of(const m3_dims &d) { return d.ngroups > 0 ? d.ngroups : d.nheads; }

// Per-token inputs, y and the carry need only element alignment; the fp32
// state and the workspace are read as float4 and need 16 bytes.
bool ptr_ok(const void *p, size_t align) { return p && (reinterpret_cast<uintptr_t>(p) % align) == 0; }

// The workspace covers both plans, so a call may take either path: the
// tensor-core one when the shape is supported and the pointers are 16-byte
// aligned (TMA), the SIMT one otherwise.
m3_status plan_scan(const m3_dims &d, ScanPlan *simt, ScanPlan *tc, bool *has_tc, size_t *ws) {
    const int sms = sm_count();
    const bool ok_simt = simt_plan(d, sms, simt);
    *has_tc = tc_plan(d, sms, tc);
    if (!ok_simt && !*has_tc) return M3_ERR_UNSUPPORTED;
    size_t w = 0;
    if (ok_simt) w = simt->ws_bytes;
    else simt->path = -1;
    if (*has_tc && tc->ws_bytes > w) w = tc->ws_bytes;
    *ws = w;
    return M3_OK;
}

size_t elem_size(int dtype) { return dtype == M3_F32 ? 4 : 2; }

}  // namespace

extern "C" {

m3_status mamba3_scan_fwd_workspace(const m3_dims *dims, size_t *bytes) {
    if (!bytes) return M3_ERR_INVALID_ARG;
    m3_status st = check_dims(dims, true);
    if (st != M3_OK) return st;
    ScanPlan simt, tc;
    bool has_tc = false;
    if ((st = plan_scan(*dims, &simt, &tc, &has_tc, bytes)) != M3_OK) return st;
    return M3_OK;
}

}  // extern "C"

namespace {

// Validates an m3_bc_norm (null = none) into `out`.
m3_status bc_args(const m3_bc_norm *bc, BcNorm *out) {
    *out = BcNorm{};
    if (!bc) return M3_OK;
    for (const float *p : {bc->B_weight, bc->B_bias, bc->C_weight, bc->C_bias})
        if (p && (reinterpret_cast<uintptr_t>(p) & 3u)) return M3_ERR_INVALID_ARG;
    if (!(bc->eps >= 0.f)) return M3_ERR_INVALID_ARG;   // also NaN
    *out = BcNorm{bc->B_weight, bc->B_bias, bc->C_weight, bc->C_bias, bc->eps, 1};
    return M3_OK;
}

m3_status scan_impl(const m3_dims *dims, const void *x, const void *B, const void *C, const void *dt, const void *A,
                    const void *lambda, const void *theta, const m3_bc_norm *bcn, const m3_state *state_in, void *y,
                    const m3_state *state_out, void *workspace, size_t workspace_bytes, void *stream) {
    m3_status st = check_dims(dims, true);
    if (st != M3_OK) return st;
    const m3_dims &d = *dims;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    BcNorm bc;
    if ((st = bc_args(bcn, &bc)) != M3_OK) return st;
    if (d.batch == 0) return M3_OK;   // nothing to read or write; pointers are not inspected
    const bool work = d.seqlen > 0;
    const size_t es = elem_size(d.dtype);
    if (work) {
        for (const void *p : {x, B, C, dt, A, lambda, theta})
            if (!ptr_ok(p, es)) return M3_ERR_INVALID_ARG;
        if (!ptr_ok(y, elem_size(d.ydtype))) return M3_ERR_INVALID_ARG;
    }
    for (const m3_state *st : {state_in, state_out}) {
        if (!st) continue;
        if (!ptr_ok(st->h, 16)) return M3_ERR_INVALID_ARG;
        if ((st->B_prev == nullptr) != (st->x_prev == nullptr)) return M3_ERR_INVALID_ARG;
        if (st->B_prev && (!ptr_ok(st->B_prev, es) || !ptr_ok(st->x_prev, es))) return M3_ERR_INVALID_ARG;
    }
    ScanPlan simt, tc;
    bool has_tc = false;
    size_t ws_need = 0;
    if ((st = plan_scan(d, &simt, &tc, &has_tc, &ws_need)) != M3_OK) return st;
    bool use_tc = has_tc;
    for (const void *p : {x, B, C, theta, (const void *)y})
        if (!aligned16(p)) use_tc = false;
    if (!use_tc && groups_of(d) != d.nheads) return M3_ERR_UNSUPPORTED;   // grouped B / C: tensor cores only
    if (!use_tc && simt.path < 0) return M3_ERR_UNSUPPORTED;
    const ScanPlan &pl = use_tc ? tc : simt;

    const size_t bh = (size_t)d.batch * d.nheads;
    const size_t hbytes = bh * d.dstate * d.headdim * sizeof(float);
    const size_t bbytes = bh * d.rank * d.dstate * es, xbytes = bh * d.rank * d.headdim * es;
    if (!work) {
        // L = 0: the state and carry pass through unchanged (zeros without state_in)
        if (!state_out) return M3_OK;
        cudaError_t e = cudaSuccess;
        if (state_in && state_in->h != state_out->h)
            e = cudaMemcpyAsync(state_out->h, state_in->h, hbytes, cudaMemcpyDeviceToDevice, s);
        else if (!state_in)
            e = cudaMemsetAsync(state_out->h, 0, hbytes, s);
        if (e == cudaSuccess && state_out->B_prev) {
            if (state_in && state_in->B_prev) {
                if (state_in->B_prev != state_out->B_prev)
                    e = cudaMemcpyAsync(state_out->B_prev, state_in->B_prev, bbytes, cudaMemcpyDeviceToDevice, s);
                if (e == cudaSuccess && state_in->x_prev != state_out->x_prev)
                    e = cudaMemcpyAsync(state_out->x_prev, state_in->x_prev, xbytes, cudaMemcpyDeviceToDevice, s);
            } else {
                e = cudaMemsetAsync(state_out->B_prev, 0, bbytes, s);
                if (e == cudaSuccess) e = cudaMemsetAsync(state_out->x_prev, 0, xbytes, s);
            }
        }
        return e == cudaSuccess ? M3_OK : M3_ERR_CUDA;
    }
    if (ws_need > 0 && (!workspace || workspace_bytes < ws_need || !aligned16(workspace)))
        return M3_ERR_WORKSPACE;

    ScanArgs a{};
    a.dtype = d.dtype; a.ydtype = d.ydtype; a.batch = d.batch; a.L = d.seqlen; a.H = d.nheads; a.G = groups_of(d);
    a.bc = bc;
    a.P = d.headdim; a.N = d.dstate; a.R = d.rank;
    a.x = x; a.B = B; a.C = C; a.dt = dt; a.A = A; a.lam = lambda; a.theta = theta;
    a.h0 = state_in ? state_in->h : nullptr;
    a.Bprev = state_in ? state_in->B_prev : nullptr;
    a.xprev = state_in ? state_in->x_prev : nullptr;
    a.y = y;
    a.h_out = state_out ? state_out->h : nullptr;
    a.Bprev_out = state_out ? state_out->B_prev : nullptr;
    a.xprev_out = state_out ? state_out->x_prev : nullptr;
    if (pl.ws_bytes > 0) {
        // state slots per sequence: one per state-pass piece boundary (see scan_workspace_bytes)
        const size_t slots = pl.nseg > 1 ? (size_t)(pl.nseg - 1) * pl.nsub + 1 : 1;
        const size_t state_b = bh * slots * d.dstate * d.headdim * sizeof(float);
        a.ws_state = static_cast<float *>(workspace);
        a.ws_tot = reinterpret_cast<float *>(static_cast<char *>(workspace) + ((state_b + 255) / 256) * 256);
    }
    cudaError_t e = use_tc ? tc_scan(a, pl, s) : simt_scan(a, pl, s);
    return e == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}

m3_status decode_impl(const m3_dims *dims, const void *x, const void *B, const void *C, const void *dt, const void *A,
                      const void *lambda, const void *theta, const m3_bc_norm *bcn, const m3_state *state, void *y,
                      void *stream) {
    m3_status st = check_dims(dims, false);
    if (st != M3_OK) return st;
    const m3_dims &d = *dims;
    BcNorm bc;
    if ((st = bc_args(bcn, &bc)) != M3_OK) return st;
    if (d.batch == 0) return M3_OK;   // nothing to read or write; pointers are not inspected
    if (!state) return M3_ERR_INVALID_ARG;
    const size_t es = elem_size(d.dtype);
    for (const void *p : {x, B, C, dt, A, lambda, theta, (const void *)state->B_prev,
                          (const void *)state->x_prev})
        if (!ptr_ok(p, es)) return M3_ERR_INVALID_ARG;
    if (!ptr_ok(y, elem_size(d.ydtype))) return M3_ERR_INVALID_ARG;
    if (!ptr_ok(state->h, 16)) return M3_ERR_INVALID_ARG;
    const int G = groups_of(d);
    if (G != d.nheads) {
        if (bc.on) return M3_ERR_UNSUPPORTED;   // grouped B / C: tensor-core kernel only, which has no BC step
        const void *ptrs[] = {x, B, C, theta, state->h, state->B_prev, state->x_prev};
        if (!decode_tc_ok(d.dtype, d.headdim, d.dstate, d.rank, (long long)d.batch * d.nheads, ptrs, 7))
            return M3_ERR_UNSUPPORTED;
    }
    cudaError_t e = decode_step(d.dtype, d.ydtype, d.batch, d.nheads, G, d.headdim, d.dstate, d.rank, x, B, C, dt,
                                A, lambda, theta, state->h, state->B_prev, state->x_prev, y,
                                static_cast<cudaStream_t>(stream), &bc);
    return e == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}

}  // namespace

extern "C" {

m3_status mamba3_scan_fwd(const m3_dims *dims, const void *x, const void *B, const void *C,
                          const void *dt, const void *A, const void *lambda, const void *theta,
                          const m3_state *state_in, void *y, const m3_state *state_out,
                          void *workspace, size_t workspace_bytes, void *stream) {
    return scan_impl(dims, x, B, C, dt, A, lambda, theta, nullptr, state_in, y, state_out, workspace,
                     workspace_bytes, stream);
}

m3_status mamba3_scan_fwd_bc(const m3_dims *dims, const void *x, const void *B, const void *C,
                             const void *dt, const void *A, const void *lambda, const void *theta,
                             const m3_bc_norm *bc, const m3_state *state_in, void *y,
                             const m3_state *state_out, void *workspace, size_t workspace_bytes,
                             void *stream) {
    return scan_impl(dims, x, B, C, dt, A, lambda, theta, bc, state_in, y, state_out, workspace,
                     workspace_bytes, stream);
}

// Token range [l0, l1) of slice i when L tokens are cut into ns slices.
static void slice_range(int L, int ns, int i, int *l0, int *l1) {
    const int base = L / ns, extra = L % ns;
    *l0 = i * base + (i < extra ? i : extra);
    *l1 = *l0 + base + (i < extra ? 1 : 0);
}

m3_status mamba3_scan_fwd_staged_workspace(const m3_dims *dims, int slices, size_t *bytes) {
    if (!bytes || !dims || slices < 1) return M3_ERR_INVALID_ARG;
    m3_status st = check_dims(dims, true);
    if (st != M3_OK) return st;
    const int L = dims->seqlen;
    const int ns = slices < L ? slices : (L > 0 ? L : 1);
    size_t need = 0;
    for (int ls : {(L + ns - 1) / ns, L / ns}) {   // slices hold ceil(L / ns) or floor(L / ns) tokens
        if (ls < 1) continue;
        m3_dims sd = *dims;
        sd.seqlen = ls;
        size_t w = 0;
        if ((st = mamba3_scan_fwd_workspace(&sd, &w)) != M3_OK) return st;
        if (w > need) need = w;
    }
    *bytes = need;
    return M3_OK;
}

m3_status mamba3_scan_fwd_staged(const m3_dims *dims, const m3_token_inputs *host_in, const m3_token_inputs *dev_in,
                                 void *host_y, void *dev_y, const m3_state *dev_state_in,
                                 const m3_state *dev_state_out, float *host_h_out, void *workspace,
                                 size_t workspace_bytes, int slices, void *stream, void *copy_stream) {
    m3_status st = check_dims(dims, true);
    if (st != M3_OK) return st;
    if (!host_in || !dev_in || slices < 1) return M3_ERR_INVALID_ARG;
    const m3_dims &d = *dims;
    if (d.batch == 0) return M3_OK;
    if (host_h_out && !dev_state_out) return M3_ERR_INVALID_ARG;
    const int L = d.seqlen, ns = slices < L ? slices : (L > 0 ? L : 1);
    if (ns > 1 && !(dev_state_out && dev_state_out->B_prev)) return M3_ERR_INVALID_ARG;   // carries the slices
    for (const void *p : {host_in->x, host_in->B, host_in->C, host_in->dt, host_in->A, host_in->lambda,
                          host_in->theta, dev_in->x, dev_in->B, dev_in->C, dev_in->dt, dev_in->A, dev_in->lambda,
                          dev_in->theta})
        if (!p) return M3_ERR_INVALID_ARG;
    if (L > 0 && (!dev_y || !host_y)) return M3_ERR_INVALID_ARG;
    size_t need = 0;
    if ((st = mamba3_scan_fwd_staged_workspace(dims, slices, &need)) != M3_OK) return st;
    if (need > 0 && (!workspace || workspace_bytes < need)) return M3_ERR_WORKSPACE;
    const size_t es = elem_size(d.dtype);
    const size_t H = (size_t)d.nheads, P = (size_t)d.headdim, N = (size_t)d.dstate, R = (size_t)d.rank;
    const size_t nb = (size_t)d.batch;
    // bytes per token (all heads) of every tensor
    const size_t G = (size_t)groups_of(d);
    const size_t tx = H * R * P * es, tB = G * R * N * es, ts = H * es, tth = H * (N / 2) * es, ty = H * R * P * elem_size(d.ydtype);
    const cudaStream_t s = static_cast<cudaStream_t>(stream), cs = static_cast<cudaStream_t>(copy_stream);
    // `to` waits for the work queued on `from` so far
    auto follow = [](cudaStream_t to, cudaStream_t from) {
        cudaEvent_t ev;
        if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) return false;
        cudaError_t e = cudaEventRecord(ev, from);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(to, ev, 0);
        cudaEventDestroy(ev);   // released once the wait has been satisfied
        return e == cudaSuccess;
    };
    // the previous call's copies out read buffers this call rewrites: start after them
    if (!follow(s, cs)) return M3_ERR_CUDA;
    if (L == 0) {
        st = mamba3_scan_fwd(dims, dev_in->x, dev_in->B, dev_in->C, dev_in->dt, dev_in->A, dev_in->lambda,
                             dev_in->theta, dev_state_in, dev_y, dev_state_out, workspace, workspace_bytes, stream);
        if (st == M3_OK && host_h_out &&
            cudaMemcpyAsync(host_h_out, dev_state_out->h, nb * H * N * P * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
            st = M3_ERR_CUDA;
        return st;
    }
    // The copies in run on the library's input stream, ahead of the kernels: range i + 1 comes in while
    // range i is scanned and range i - 1 goes out, so both directions of the link stay busy.  They start
    // after everything queued on `stream` so far (the previous call's kernels read the staging buffers).
    const cudaStream_t is = input_stream();
    if (!is || !follow(is, s)) return M3_ERR_CUDA;
    // Slice i holds tokens [l0, l1) of every sequence; its device copy is the contiguous
    // [batch][l1 - l0][...] block at offset batch * l0 * (bytes per token) of each device buffer.
    for (int i = 0; i < ns; ++i) {
        int l0, l1;
        slice_range(L, ns, i, &l0, &l1);
        const size_t ls = (size_t)(l1 - l0);
        const struct { const void *h; const void *dv; size_t tb; } in[7] = {
            {host_in->x, dev_in->x, tx}, {host_in->B, dev_in->B, tB}, {host_in->C, dev_in->C, tB},
            {host_in->dt, dev_in->dt, ts}, {host_in->A, dev_in->A, ts}, {host_in->lambda, dev_in->lambda, ts},
            {host_in->theta, dev_in->theta, tth}};
        const void *dp[7];
        for (int k = 0; k < 7; ++k) {
            char *dst = static_cast<char *>(const_cast<void *>(in[k].dv)) + nb * (size_t)l0 * in[k].tb;
            const char *src = static_cast<const char *>(in[k].h) + (size_t)l0 * in[k].tb;
            dp[k] = dst;
            if (cudaMemcpy2DAsync(dst, ls * in[k].tb, src, (size_t)L * in[k].tb, ls * in[k].tb, nb,
                                  cudaMemcpyHostToDevice, is) != cudaSuccess)
                return M3_ERR_CUDA;
        }
        if (!follow(s, is)) return M3_ERR_CUDA;
        m3_dims sd = d;
        sd.seqlen = (int)ls;
        char *ydev = static_cast<char *>(dev_y) + nb * (size_t)l0 * ty;
        st = mamba3_scan_fwd(&sd, dp[0], dp[1], dp[2], dp[3], dp[4], dp[5], dp[6],
                             i == 0 ? dev_state_in : dev_state_out, ydev, dev_state_out, workspace, workspace_bytes,
                             stream);
        if (st != M3_OK) return st;
        if (!follow(cs, s)) return M3_ERR_CUDA;
        if (cudaMemcpy2DAsync(static_cast<char *>(host_y) + (size_t)l0 * ty, (size_t)L * ty, ydev, ls * ty, ls * ty, nb,
                              cudaMemcpyDeviceToHost, cs) != cudaSuccess)
            return M3_ERR_CUDA;
    }
    if (host_h_out &&
        cudaMemcpyAsync(host_h_out, dev_state_out->h, nb * H * N * P * 4, cudaMemcpyDeviceToHost, cs) != cudaSuccess)
        return M3_ERR_CUDA;
    return M3_OK;
}

m3_status mamba3_decode_step(const m3_dims *dims, const void *x, const void *B, const void *C,
                             const void *dt, const void *A, const void *lambda, const void *theta,
                             const m3_state *state, void *y, void *stream) {
    return decode_impl(dims, x, B, C, dt, A, lambda, theta, nullptr, state, y, stream);
}

m3_status mamba3_decode_step_bc(const m3_dims *dims, const void *x, const void *B, const void *C,
                                const void *dt, const void *A, const void *lambda, const void *theta,
                                const m3_bc_norm *bc, const m3_state *state, void *y, void *stream) {
    return decode_impl(dims, x, B, C, dt, A, lambda, theta, bc, state, y, stream);
}

m3_status mamba3_decode_step_pooled(const m3_dims *dims, const int *slot, const void *x, const void *B,
                                    const void *C, const void *dt, const void *A, const void *lambda,
                                    const void *theta, const m3_state *pool, int pool_size, void *y,
                                    void *stream) {
    m3_status st = check_dims(dims, false);
    if (st != M3_OK) return st;
    const m3_dims &d = *dims;
    if (d.batch == 0) return M3_OK;   // nothing to read or write; pointers are not inspected
    if (!pool || pool_size < 1 || !ptr_ok(slot, 4)) return M3_ERR_INVALID_ARG;
    const size_t es = elem_size(d.dtype);
    for (const void *p : {x, B, C, dt, A, lambda, theta, (const void *)pool->B_prev, (const void *)pool->x_prev})
        if (!ptr_ok(p, es)) return M3_ERR_INVALID_ARG;
    if (!ptr_ok(y, elem_size(d.ydtype))) return M3_ERR_INVALID_ARG;
    if (!ptr_ok(pool->h, 16)) return M3_ERR_INVALID_ARG;
    const void *ptrs[] = {x, B, C, theta, pool->h, pool->B_prev, pool->x_prev};
    const long long heads = (long long)(d.batch > pool_size ? d.batch : pool_size) * d.nheads;
    if (!decode_tc_ok(d.dtype, d.headdim, d.dstate, d.rank, heads, ptrs, 7)) return M3_ERR_UNSUPPORTED;
    cudaError_t e = decode_step_pooled(d.ydtype, d.batch, d.nheads, groups_of(d), d.headdim, d.dstate, d.rank, slot,
                                       pool_size, x, B, C, dt, A, lambda, theta, pool->h, pool->B_prev,
                                       pool->x_prev, y, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}

m3_status mamba3_scan_bwd_workspace(const m3_dims *dims, size_t *bytes) {
    if (!bytes) return M3_ERR_INVALID_ARG;
    m3_status st = check_dims(dims, true);
    if (st != M3_OK) return st;
    const m3_dims &d = *dims;
    const int esz = (int)elem_size(d.dtype);
    if (groups_of(d) != d.nheads || (size_t)d.dstate * d.headdim > 8192 ||
        bwd_smem_bytes(d.dstate, d.headdim, d.rank, esz) > 227u * 1024u)
        return M3_ERR_UNSUPPORTED;
    *bytes = bwd_workspace_bytes(d.batch, d.nheads, d.seqlen, d.dstate, d.headdim, d.rank, esz);
    return M3_OK;
}

m3_status mamba3_scan_bwd(const m3_dims *dims, const m3_token_inputs *in, const m3_state *state_in,
                          const m3_grads_in *gin, const m3_grads_out *gout, void *workspace, size_t workspace_bytes,
                          void *stream) {
    size_t need = 0;
    m3_status st = mamba3_scan_bwd_workspace(dims, &need);
    if (st != M3_OK) return st;
    const m3_dims &d = *dims;
    if (!in || !gin || !gout) return M3_ERR_INVALID_ARG;
    if (d.batch == 0) return M3_OK;
    const size_t es = elem_size(d.dtype);
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (state_in) {
        if (state_in->h && !ptr_ok(state_in->h, 4)) return M3_ERR_INVALID_ARG;
        if ((state_in->B_prev == nullptr) != (state_in->x_prev == nullptr)) return M3_ERR_INVALID_ARG;
        if (state_in->B_prev && (!ptr_ok(state_in->B_prev, es) || !ptr_ok(state_in->x_prev, es)))
            return M3_ERR_INVALID_ARG;
    }
    for (const float *p : {gin->dh_out, gin->dB_prev_out, gin->dx_prev_out})
        if (p && !ptr_ok(p, 4)) return M3_ERR_INVALID_ARG;
    for (float *p : {gout->dh0, gout->dB_prev, gout->dx_prev})
        if (p && !ptr_ok(p, 4)) return M3_ERR_INVALID_ARG;
    const size_t bh = (size_t)d.batch * d.nheads;
    if (d.seqlen == 0) {
        // nothing scanned: the state's and carry's gradients pass through
        const struct { float *dst; const float *src; size_t n; } pass[3] = {
            {gout->dh0, gin->dh_out, bh * d.dstate * d.headdim},
            {gout->dB_prev, gin->dB_prev_out, bh * d.rank * d.dstate},
            {gout->dx_prev, gin->dx_prev_out, bh * d.rank * d.headdim}};
        for (const auto &q : pass) {
            if (!q.dst) continue;
            const cudaError_t e = q.src ? cudaMemcpyAsync(q.dst, q.src, q.n * 4, cudaMemcpyDeviceToDevice, s)
                                        : cudaMemsetAsync(q.dst, 0, q.n * 4, s);
            if (e != cudaSuccess) return M3_ERR_CUDA;
        }
        return M3_OK;
    }
    for (const void *p : {in->x, in->B, in->C, in->dt, in->A, in->lambda, in->theta})
        if (!ptr_ok(p, es)) return M3_ERR_INVALID_ARG;
    if (!ptr_ok(gin->dy, 4)) return M3_ERR_INVALID_ARG;
    for (float *p : {gout->dx, gout->dB, gout->dC, gout->ddt, gout->dA, gout->dlambda, gout->dtheta})
        if (!ptr_ok(p, 4)) return M3_ERR_INVALID_ARG;
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace))) return M3_ERR_WORKSPACE;
    BwdArgs a{};
    a.dtype = d.dtype; a.batch = d.batch; a.L = d.seqlen; a.H = d.nheads; a.P = d.headdim; a.N = d.dstate;
    a.R = d.rank;
    a.x = in->x; a.B = in->B; a.C = in->C; a.dt = in->dt; a.A = in->A; a.lam = in->lambda; a.theta = in->theta;
    a.h0 = state_in ? state_in->h : nullptr;
    a.Bprev = state_in ? state_in->B_prev : nullptr;
    a.xprev = state_in ? state_in->x_prev : nullptr;
    a.dy = gin->dy; a.dh_out = gin->dh_out; a.dBprev_out = gin->dB_prev_out; a.dxprev_out = gin->dx_prev_out;
    a.dx = gout->dx; a.dB = gout->dB; a.dC = gout->dC; a.ddt = gout->ddt; a.dA = gout->dA; a.dlam = gout->dlambda;
    a.dtheta = gout->dtheta; a.dh0 = gout->dh0; a.dBprev = gout->dB_prev; a.dxprev = gout->dx_prev;
    a.ws = static_cast<float *>(workspace);
    return scan_bwd(a, s) == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}

m3_status mamba3_device_status(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return M3_ERR_CUDA;
    unsigned *w = device_status_word();
    if (!w) return M3_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return M3_ERR_CUDA;
    if (v != 0) {
        const unsigned zero = 0;
        if (cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return M3_ERR_CUDA;
    }
    if (v & kStatusTimeout) return M3_ERR_TIMEOUT;
    return (v & kStatusBadIndex) ? M3_ERR_INDEX : M3_OK;
}

const char *mamba3_status_string(int status) {
    switch (status) {
        case M3_OK: return "ok";
        case M3_ERR_INVALID_ARG: return "invalid argument";
        case M3_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case M3_ERR_WORKSPACE: return "workspace missing or too small";
        case M3_ERR_CUDA: return "CUDA error";
        case M3_ERR_TIMEOUT: return "device-side wait timed out";
        case M3_ERR_INDEX: return "pooled decode slot index outside the pool";
        default: return "unknown status";
    }
}

m3_status mamba3_trace_begin(int kernel, int max_launches) {
    if (kernel < 0 || kernel >= M3_KERNEL_COUNT || max_launches < 1) return M3_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_trace_mu);
    trace_release_locked();
    g_trace_ev.resize(2 * (size_t)max_launches, nullptr);
    for (auto &e : g_trace_ev) {
        if (cudaEventCreate(&e) != cudaSuccess) {
            e = nullptr;
            for (auto &f : g_trace_ev)
                if (f) cudaEventDestroy(f);
            g_trace_ev.clear();
            return M3_ERR_CUDA;
        }
    }
    g_trace_kernel = kernel;
    g_trace_max = max_launches;
    g_trace_n = 0;
    return M3_OK;
}

m3_status mamba3_trace_end(int *launches, double *total_ms) {
    std::lock_guard<std::mutex> lock(g_trace_mu);
    if (g_trace_kernel < 0) return M3_ERR_INVALID_ARG;
    double total = 0.0;
    m3_status st = M3_OK;
    for (int i = 0; i < g_trace_n; ++i) {
        float ms = 0.f;
        if (cudaEventSynchronize(g_trace_ev[2 * i + 1]) != cudaSuccess ||
            cudaEventElapsedTime(&ms, g_trace_ev[2 * i], g_trace_ev[2 * i + 1]) != cudaSuccess) {
            st = M3_ERR_CUDA;
            break;
        }
        total += ms;
    }
    if (launches) *launches = g_trace_n;
    if (total_ms) *total_ms = total;
    trace_release_locked();
    return st;
}

uint64_t mamba3_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int mamba3_version(void) { return 100; }

}  // extern "C"
