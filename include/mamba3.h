/*
 * mamba3.h -- C ABI of the B300 (sm_103a) Mamba-3 layer-recurrence library.
 *
 * The library computes the Mamba-3 selective state-space recurrence for every
 * (batch, head) sequence:
 *
 *   h_t = alpha_t h_{t-1} + beta_t B_{t-1} x_{t-1}^T + gamma_t B_t x_t^T,
 *   alpha_t = exp(dt_t (A_t + i theta_t)),  beta_t = (1 - lambda_t) dt_t alpha_t,
 *   gamma_t = lambda_t dt_t,                y_t = C_t^T h_t,
 *
 * with a complex state realised as a real one whose (2k, 2k+1) entries are
 * rotated by the data-dependent angle dt_t theta_{t,k}, and MIMO rank R
 * (B_t is N x R, x_t is P x R).  Sources (Mamba-3 pages):
 *   - exponential-trapezoidal update: linkstar.cloud/article/869, section
 *     "第一刀：指数梯形离散化 / Mamba-3的升级";
 *   - complex state as 2x2 block rotations and its RoPE form: same page,
 *     sections "第二刀：复值状态空间" and "RoPE技巧";
 *   - MIMO: same page, section "第三刀：多输入多输出";
 *   - chunked prefill, recurrent decode: same page, sections "第一刀"
 *     (parallel form) and "训练怎么办" (chunked algorithm).
 *
 * Conventions shared by every call
 *   - All tensor pointers are caller-owned DEVICE memory on the current CUDA
 *     device, row-major and contiguous.  The fp32 state h and the workspace
 *     must be 16-byte aligned; every other pointer must be aligned to its
 *     element size (a misaligned or NULL pointer is M3_ERR_INVALID_ARG).  No
 *     call allocates device memory at run time; the prefill workspace is
 *     supplied by the caller after a size query.  The one static reservation
 *     is the M3_NOALLOC_SCRATCH_BYTES scratch array behind
 *     mamba3_scan_fwd_noalloc, which the module holds on every device it is
 *     loaded on.
 *   - Element type of the per-token inputs is dims->dtype (fp32 or bf16);
 *     the output y has dims->ydtype (fp32 unless chosen otherwise: rounding y
 *     to bf16 would by itself cost up to half a bf16 ulp of the largest |y|,
 *     about 1-2 % of rms(y), which is the whole error budget of a bf16-input
 *     run; fp16 costs an eighth of that).  The state h is always fp32.  The
 *     carry (B_prev, x_prev) has the input dtype.
 *   - dt, A, lambda are already activated (dt >= 0, A <= 0, 0 <= lambda <= 1
 *     for a stable recurrence; other values are computed as given); theta is
 *     in radians.
 *   - Calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *     default stream).  The return value reports argument validation and
 *     launch status; on an argument error nothing is launched or written.
 *     Device-side wait limits report through mamba3_device_status().
 *     The tensor-core prefill (one-wave plans) and decode kernels are
 *     launched as programmatic dependents of the kernel before them in the
 *     stream: they may be scheduled while it finishes, and touch no global
 *     memory until it has completed (ordering on the stream is unchanged).
 *   - batch = 0 is a successful call that touches nothing (pointers are not
 *     inspected).
 *   - Inputs must not overlap outputs, except that a state may be updated in
 *     place where a call says so.
 *   - Supported shapes: N even with 2 <= N <= 256, 1 <= P <= 128, P a
 *     multiple of 4, 1 <= R <= 8, nheads >= 1, batch >= 0, seqlen >= 0.
 *     Anything else returns M3_ERR_UNSUPPORTED.
 */
#ifndef MAMBA3_H
#define MAMBA3_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    M3_OK = 0,
    M3_ERR_INVALID_ARG = 1,   /* NULL / misaligned pointer, negative size, NULL dims */
    M3_ERR_UNSUPPORTED = 2,   /* shape or dtype outside the supported set */
    M3_ERR_WORKSPACE = 3,     /* workspace missing or smaller than the queried size */
    M3_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
    M3_ERR_TIMEOUT = 5,       /* a device-side wait gave up (see mamba3_device_status) */
    M3_ERR_INDEX = 6          /* a pooled decode read a slot index outside [0, pool_size) */
} m3_status;

typedef enum { M3_F32 = 0, M3_BF16 = 1, M3_F16 = 2 } m3_dtype;

/* Problem sizes.  P = head dim, N = real state size (N/2 complex pairs),
 * R = MIMO rank.  chunk = tokens per chunk of the prefill kernels, 0 = the
 * library's choice; the result does not depend on it beyond rounding.
 * ngroups = G: B and C are shared by groups of H / G consecutive heads
 * (head h reads group h / (H / G)), so their per-token blocks are [G][R][N]
 * instead of [H][R][N]; 0 (or H) = one B and C per head.  G must divide H
 * (else M3_ERR_INVALID_ARG).  Grouped B and C are a layout of the inputs, not
 * a change of the recurrence, and are not from the Mamba-3 pages.  They are
 * supported on the tensor-core paths only (bf16 inputs, P = 64, N in
 * {64, 128}, 16-byte-aligned pointers); elsewhere M3_ERR_UNSUPPORTED.  The
 * state's carry stays per head.
 * ydtype: element type of the output y (an m3_dtype; 0 = M3_F32).  The
 * arithmetic is the same for all three; y is rounded once (to nearest even)
 * from fp32.  M3_F16 keeps y at the input element size with an 11-bit
 * significand (rounding costs at most 2^-11 |y|); its range ends at 65504,
 * beyond which a value becomes infinite.  M3_BF16 has the input's format;
 * its 8-bit significand alone can cost up to 2^-9 |y|.  Inputs must be
 * M3_F32 or M3_BF16. */
typedef struct {
    int batch;
    int seqlen;      /* L; ignored by mamba3_decode_step */
    int nheads;      /* H */
    int headdim;     /* P */
    int dstate;      /* N */
    int rank;        /* R */
    int chunk;
    int dtype;       /* m3_dtype */
    int ngroups;     /* G, 0 = H */
    int ydtype;      /* m3_dtype of y, 0 = fp32 */
} m3_dims;

/* Recurrent state of every (batch, head): the checkpoint between calls.
 *   h      [batch][H][N][P] fp32, the true (unrotated) state after the last token;
 *   B_prev [batch][H][R][N] dtype, that token's B (unrotated);
 *   x_prev [batch][H][R][P] dtype, that token's x.
 * (B_prev, x_prev) feed the next call's beta (left-endpoint) term. */
typedef struct {
    float *h;
    void *B_prev;
    void *x_prev;
} m3_state;

/*
 * Workspace bytes mamba3_scan_fwd needs for `dims` on the current device
 * (0 is a valid answer).  Returns M3_ERR_INVALID_ARG for NULL arguments and
 * M3_ERR_UNSUPPORTED for unsupported shapes.
 */
m3_status mamba3_scan_fwd_workspace(const m3_dims *dims, size_t *bytes);

/*
 * Chunked prefill over L = dims->seqlen tokens of every (b, h) sequence.
 *
 * Inputs (dtype unless stated):
 *   x      [batch][L][H][R][P]      B, C [batch][L][H][R][N]
 *   dt, A, lambda [batch][L][H]     theta [batch][L][H][N/2]
 *   state_in: initial state and carry, or NULL for h0 = 0 and no carry.
 * Outputs:
 *   y      [batch][L][H][R][P] of dims->ydtype, y_t = C_t^T h_t;
 *   state_out: final state h_L (fp32) and carry (B_{L-1}, x_{L-1}); NULL = not
 *     written.  state_out may equal state_in (in-place update); otherwise the
 *     two must not overlap.
 *   workspace: device buffer of at least the queried size (may be NULL when the
 *     query returned 0).  It holds per-segment fp32 states between kernels.
 * L = 0 copies state_in (or zeros) to state_out.
 */
m3_status mamba3_scan_fwd(const m3_dims *dims, const void *x, const void *B, const void *C,
                          const void *dt, const void *A, const void *lambda, const void *theta,
                          const m3_state *state_in, void *y, const m3_state *state_out,
                          void *workspace, size_t workspace_bytes, void *stream);

/*
 * BC normalisation and bias (linkstar.cloud/article/869, section
 * "架构上的其他改动": BC归一化 -- B and C are RMS-normalised like a QK-norm --
 * and BC偏置 -- a learnable, data-independent bias is added to B and C).  The
 * page gives no formula; the reading taken: every row of B (and of C) -- the N
 * entries of one (token, head, rank) -- becomes
 *     v'[n] = v[n] / sqrt(mean_m v[m]^2 + eps) * weight[h][n] + bias[h][r][n]
 * before the recurrence (and before the rotation of its RoPE form).  The carry
 * keeps the raw B of the last token; the call that consumes it normalises it.
 *   B_weight, C_weight [H][N] fp32 device arrays, or NULL for a gain of 1;
 *   B_bias, C_bias  [H][R][N] fp32 device arrays, or NULL for no bias;
 *   eps >= 0 (a row of zeros with eps = 0 gives a non-finite result).
 * Pointers must be 4-byte aligned.  With grouped B / C the gain and bias are
 * still per head (the heads of a group share the raw B, not the normalised one).
 */
typedef struct {
    const float *B_weight;
    const float *B_bias;
    const float *C_weight;
    const float *C_bias;
    float eps;
} m3_bc_norm;

/* The seven per-token input tensors of a prefill (layouts as in mamba3_scan_fwd). */
typedef struct {
    const void *x, *B, *C, *dt, *A, *lambda, *theta;
} m3_token_inputs;

/*
 * Workspace bytes mamba3_scan_fwd_staged needs for `dims` cut into `slices`
 * token slices (0 is a valid answer).  Errors as mamba3_scan_fwd_workspace;
 * slices < 1 is M3_ERR_INVALID_ARG.
 */
m3_status mamba3_scan_fwd_staged_workspace(const m3_dims *dims, int slices, size_t *bytes);

/*
 * The prefill from and to host memory, with the host <-> device copies
 * overlapped: the sequences are cut into `slices` consecutive token ranges
 * (at most L); range i of every sequence is copied in, then scanned on `stream`
 * (starting from range i-1's final state and carry), and its y is copied out
 * on `copy_stream` while range i+1 is copied in.  The copies in run on a
 * stream the library keeps for them (one per device, created on first use),
 * queued ahead of the scans so that both directions of the host link stay
 * busy.  The host buffers should be pinned (page-locked) for the copies to be
 * asynchronous.
 *   host_in, host_y:   the inputs and y in host memory, full layouts;
 *   dev_in, dev_y:     device buffers of the same sizes (caller-owned staging;
 *                      range i occupies the block of batch * L_i tokens that
 *                      follows the earlier ranges' blocks);
 *   dev_state_in:      initial state and carry on the device, or NULL (zero);
 *   dev_state_out:     final state and carry on the device; required (with its
 *                      carry) when slices > 1, as it carries the state between
 *                      the ranges; may equal dev_state_in;
 *   host_h_out:        if non-NULL (needs dev_state_out), the final state h is
 *                      also copied to this host buffer [batch][H][N][P] fp32;
 *   workspace:         at least mamba3_scan_fwd_staged_workspace(dims, slices).
 * Work on `stream` first waits for the copies already queued on `copy_stream`
 * (a previous call's outputs), and the copies in wait for the work already
 * queued on `stream`, so consecutive calls may share the buffers.
 * Returns when everything is enqueued; `copy_stream` holds the last copies
 * (synchronise it before reading the host outputs).  Argument errors are
 * reported before anything is enqueued; a failing range reports M3_ERR_CUDA.
 * Not from the Mamba-3 pages: a host-side convenience around mamba3_scan_fwd.
 */
m3_status mamba3_scan_fwd_staged(const m3_dims *dims, const m3_token_inputs *host_in, const m3_token_inputs *dev_in,
                                 void *host_y, void *dev_y, const m3_state *dev_state_in,
                                 const m3_state *dev_state_out, float *host_h_out, void *workspace,
                                 size_t workspace_bytes, int slices, void *stream, void *copy_stream);

/* Gradients flowing into the backward pass: fp32 device arrays of the forward outputs' layouts. */
typedef struct {
    const float *dy;            /* [batch][L][H][R][P], required */
    const float *dh_out;        /* [batch][H][N][P], or NULL (zero) */
    const float *dB_prev_out;   /* [batch][H][R][N], or NULL: gradient of the carry returned */
    const float *dx_prev_out;   /* [batch][H][R][P], or NULL */
} m3_grads_in;

/* Gradients out: fp32 device arrays of the forward inputs' layouts (overwritten). */
typedef struct {
    float *dx, *dB, *dC;        /* [batch][L][H][R][P], [..][N], [..][N]; required */
    float *ddt, *dA, *dlambda;  /* [batch][L][H]; required */
    float *dtheta;              /* [batch][L][H][N/2]; required */
    float *dh0;                 /* [batch][H][N][P], or NULL (not written) */
    float *dB_prev, *dx_prev;   /* [batch][H][R][N], [batch][H][R][P], or NULL */
} m3_grads_out;

/*
 * Workspace bytes mamba3_scan_bwd needs (the forward states at every chunk boundary:
 * batch x H x (L / Q + 1) x N x P floats).  Errors as mamba3_scan_fwd_workspace.
 */
m3_status mamba3_scan_bwd_workspace(const m3_dims *dims, size_t *bytes);

/*
 * Backward pass of mamba3_scan_fwd (reverse mode, for training through the chunked
 * form; linkstar.cloud/article/869, section "训练怎么办"): the gradient of
 *   Loss = sum(dy * y) + sum(dh_out * h_out) + sum(dB_prev_out * B_prev_out)
 *          + sum(dx_prev_out * x_prev_out)
 * with respect to x, B, C, dt, A, lambda, theta and the initial state and carry,
 * for the forward call with the same dims, inputs and state_in (NULL = zero state
 * and no carry; the carry's gradients are then zero).  The forward states are
 * recomputed here (chunk checkpoints in the workspace), so the forward outputs
 * are not needed.  Arithmetic is fp32 on CUDA cores.
 * Supported: every forward shape with N * P <= 8192 and one B and C per head
 * (ngroups 0 or H); otherwise M3_ERR_UNSUPPORTED.  dims->ydtype is ignored.
 * Errors as mamba3_scan_fwd (M3_ERR_INVALID_ARG for a missing required pointer).
 */
m3_status mamba3_scan_bwd(const m3_dims *dims, const m3_token_inputs *inputs, const m3_state *state_in,
                          const m3_grads_in *grads_in, const m3_grads_out *grads_out, void *workspace,
                          size_t workspace_bytes, void *stream);

/* Size of the static scratch array behind mamba3_scan_fwd_noalloc (16 MiB). */
#define M3_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * mamba3_scan_fwd without a caller-provided workspace, for callers that cannot
 * allocate device memory: a runtime or engine that owns and pre-plans every
 * device allocation and forbids extra ones, a latency-critical path that
 * cannot afford cudaMalloc's implicit synchronisation, or a plain C caller
 * with no allocator at hand.  (The Mamba-3 pages have no counterpart; this is
 * an interface convenience, not part of the method.)
 *
 * Same arguments, results and errors as mamba3_scan_fwd minus the workspace.
 * The scratch is a static device array of M3_NOALLOC_SCRATCH_BYTES inside the
 * library; every GPU that loads the library holds it until the process exits.
 * A problem whose workspace query exceeds that size returns M3_ERR_WORKSPACE
 * before anything is launched.  The call allocates nothing (no cudaMalloc,
 * cudaFree or allocating library routine).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents
 *     (nothing in it needs to start at zero).  Calls that overlap on the GPU
 *     (concurrent streams, other host threads) race on it: serialise them.
 */
m3_status mamba3_scan_fwd_noalloc(const m3_dims *dims, const void *x, const void *B, const void *C,
                                  const void *dt, const void *A, const void *lambda, const void *theta,
                                  const m3_state *state_in, void *y, const m3_state *state_out,
                                  void *stream);

/*
 * mamba3_scan_fwd with BC normalisation and bias (see m3_bc_norm) applied to
 * B and C in front of the recurrence, fused into the prefill kernels.  bc =
 * NULL is mamba3_scan_fwd.  The workspace query is mamba3_scan_fwd_workspace.
 * Errors as mamba3_scan_fwd, plus M3_ERR_INVALID_ARG for a misaligned bc
 * pointer or eps < 0 (or NaN).
 */
m3_status mamba3_scan_fwd_bc(const m3_dims *dims, const void *x, const void *B, const void *C,
                             const void *dt, const void *A, const void *lambda, const void *theta,
                             const m3_bc_norm *bc, const m3_state *state_in, void *y,
                             const m3_state *state_out, void *workspace, size_t workspace_bytes,
                             void *stream);

/*
 * One-token recurrent step for every (b, h), updating `state` in place
 * (linkstar.cloud article, section "第一刀": the recursion used at inference).
 *
 * Inputs (dtype): x [batch][H][R][P]; B, C [batch][H][R][N];
 *   dt, A, lambda [batch][H]; theta [batch][H][N/2].
 * state: h (fp32) and carry; on return h is the state after this token and
 *   the carry is (B, x) of this token.  All three pointers are required.
 * Output: y [batch][H][R][P] of dims->ydtype.
 * dims->seqlen and dims->chunk are ignored.
 */
m3_status mamba3_decode_step(const m3_dims *dims, const void *x, const void *B, const void *C,
                             const void *dt, const void *A, const void *lambda, const void *theta,
                             const m3_state *state, void *y, void *stream);

/*
 * mamba3_decode_step with BC normalisation and bias (see m3_bc_norm) applied to
 * this token's B and C and to the carried B_prev; the carry written back is
 * this token's raw B.  bc = NULL is mamba3_decode_step.  Runs on the decode
 * kernels with per-thread FMA arithmetic (M3_DECODE_STREAM or
 * M3_DECODE_GENERIC).  Grouped B / C is not supported here
 * (M3_ERR_UNSUPPORTED).  Errors otherwise as mamba3_decode_step and
 * mamba3_scan_fwd_bc.
 */
m3_status mamba3_decode_step_bc(const m3_dims *dims, const void *x, const void *B, const void *C,
                                const void *dt, const void *A, const void *lambda, const void *theta,
                                const m3_bc_norm *bc, const m3_state *state, void *y, void *stream);

/*
 * One decode step for a batch whose states live in a caller-owned state pool
 * (serving: sequences join and leave, each keeps its slot).  Not from the
 * Mamba-3 pages: the step is exactly mamba3_decode_step, with the state of
 * batch row b read from and written back to pool slot slot[b].
 *
 * slot:  device int32 [batch].  slot[b] in [0, pool_size) selects the pool
 *   state of row b; slot[b] < 0 marks an inactive row: nothing of it is read
 *   from the pool or written (its y row is left as it was).  Active rows must
 *   name distinct slots (two rows on one slot race).  A slot >= pool_size is
 *   skipped like an inactive row and sets M3_ERR_INDEX in the device status
 *   word (see mamba3_device_status).
 * pool:  h [pool_size][H][N][P] fp32, B_prev [pool_size][H][R][N], x_prev
 *   [pool_size][H][R][P] (input dtype), updated in place for the active rows.
 * x, B, C, dt, A, lambda, theta, y: as mamba3_decode_step, indexed by batch
 *   row.
 * Supported shapes: those of the tensor-core decode kernel (bf16 inputs,
 * P = 64, N in {64, 128}, R in {1, 2, 4, 8}, 16-byte-aligned pointers); others
 * return M3_ERR_UNSUPPORTED.  pool_size < 1 or a NULL pointer is
 * M3_ERR_INVALID_ARG; nothing is launched on an argument error.
 */
m3_status mamba3_decode_step_pooled(const m3_dims *dims, const int *slot, const void *x, const void *B,
                                    const void *C, const void *dt, const void *A, const void *lambda,
                                    const void *theta, const m3_state *pool, int pool_size, void *y,
                                    void *stream);

/* The decode kernels (one per class of shapes; the results agree within
 * rounding).  Not from the Mamba-3 pages: an implementation detail exposed so
 * that a caller or a test can see which kernel served a call. */
typedef enum {
    M3_DECODE_GENERIC = 0,   /* any supported shape: one CTA per head, global loads */
    M3_DECODE_STREAM = 1,    /* P in {32, 64, 128}, 16-byte aligned blocks: staged FMA pipeline */
    M3_DECODE_TENSOR = 2     /* bf16, P = 64, N in {64, 128}: warp-level MMA pipeline */
} m3_decode_variant;

/* The m3_decode_variant that served the most recent decode call (plain or
 * pooled) in this process, on any thread or device; -1 before the first. */
int mamba3_decode_last_variant(void);

/*
 * Synchronises `stream`, then reads and clears the library's device status
 * word on the current device.  Returns M3_OK, or M3_ERR_TIMEOUT when a kernel
 * gave up a bounded wait since the last call (its outputs are then invalid),
 * M3_ERR_INDEX when a pooled decode met a slot index outside the pool (that
 * row was skipped), or M3_ERR_CUDA when the synchronisation itself failed.
 */
m3_status mamba3_device_status(void *stream);

/*
 * Self-test of the device-side wait limit (failure detection without a fault):
 * launches one kernel that waits, with the library's bounded mbarrier wait, on a
 * barrier that nothing ever completes; after `limit_ns` nanoseconds (0 <
 * limit_ns <= 1e8, else M3_ERR_INVALID_ARG) it gives up and sets the timeout bit
 * of the device status word, so that the next mamba3_device_status() returns
 * M3_ERR_TIMEOUT.  The context stays usable.  Not from the Mamba-3 pages.
 */
m3_status mamba3_selftest_wait_timeout(uint64_t limit_ns, void *stream);

/* Human-readable name of a status code (static string). */
const char *mamba3_status_string(int status);

/* Number of kernels this library has launched since it was loaded (all
 * devices, all streams); lets a caller count launches in a timed region. */
uint64_t mamba3_launch_count(void);

/* Kernels of the library, for tracing. */
typedef enum {
    M3_KERNEL_PREFILL_STATE = 0,    /* prefill pass 1: per-segment end states */
    M3_KERNEL_SEGMENT_PASS = 1,     /* prefill pass 2: state passing across segments */
    M3_KERNEL_PREFILL_OUTPUT = 2,   /* prefill pass 3: outputs, final state, carry */
    M3_KERNEL_DECODE = 3,           /* decode step */
    M3_KERNEL_BACKWARD = 4,         /* backward pass of the prefill */
    M3_KERNEL_COUNT = 5
} m3_kernel;

/*
 * Starts tracing: each of the next `max_launches` launches of `kernel` (an
 * m3_kernel) is bracketed by two CUDA events recorded on the stream it is
 * launched on.  Events are created here on the current device (no device
 * memory is allocated).  A trace already running is discarded.  Returns
 * M3_ERR_INVALID_ARG for a bad kernel id or max_launches < 1.  The events
 * sit between launches on the stream, so a traced launch does not overlap
 * the kernel before it (see programmatic dependents above): time rates with
 * events around a whole untraced run, and trace for one kernel's share.
 */
m3_status mamba3_trace_begin(int kernel, int max_launches);

/*
 * Ends tracing: waits for the traced launches, returns how many there were
 * and their summed device time in milliseconds, and releases the events.
 * Returns M3_ERR_INVALID_ARG when no trace is running.
 */
m3_status mamba3_trace_end(int *launches, double *total_ms);

/* Library version, major * 10000 + minor * 100 + patch. */
int mamba3_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MAMBA3_H */
