/*
 * ssd.h — C ABI of the GB300 (sm_103a) Mamba-2 SSD core: forward and analytic
 * backward of the selective state-space scan.
 *
 * What is computed (burn_dragon_kernel 0.5.0, src/sequence/mamba2/backward.rs,
 * `ssd_forward_state_history_reference` for the recurrence and the `y_grouped`
 * expression of `tensorized_mamba2_backward_impl` for the output): for every
 * batch row b and head h, with g the group of h,
 *
 *     h_t = exp(dt_t * A_h) * h_{t-1} + dt_t * x_t B_t^T        ([P x N] state)
 *     y_t = h_t C_t + D_h * x_t
 *
 * starting from h_{-1} = h0 (or zeros).  The backward returns the gradients
 * of L = sum(dy * y) w.r.t. x, dt, A, B, C, D and h0, the quantities of
 * `ssd_backward_reference` on the same page (that page returns the gradient
 * w.r.t. a_log = log(-A); here dA is returned, and d a_log = dA * A).
 *
 * Heads map to groups as h = g * (H / G) + j (the page reshapes nheads into
 * [ngroups, heads_per_group]); the heads of one group share B and C.
 *
 * Layouts: every tensor is dense row-major, in device memory, 16-byte aligned.
 *   x, y, dy, dx      [B][T][H][P]          `dtype`
 *   B, C, dB, dC      [B][T][G][N]          `dtype`
 *   dt, ddt           [B][T][H]             fp32
 *   A, D, dA, dD      [H]                   fp32
 *   h0, final, dh0    [B][H][P][N]          fp32
 *   chunk_states      [B][nc][H][P][N]      fp32, nc = T / chunk; entry c is
 *                                           the state *before* step c*chunk
 *                                           (entry 0 is h0 or zeros)
 * The caller owns all memory, including the workspace.  Nothing is allocated
 * by the library on the device or the host.
 *
 * Calls are asynchronous on `cuda_stream` (a cudaStream_t; NULL = legacy
 * default stream).  They return after launching; launch errors are returned,
 * device-side faults surface at the caller's next synchronisation.  Outputs
 * are overwritten, never accumulated.  Results are deterministic: no floating
 * point atomics; every reduction runs in a fixed order.
 */
#ifndef SSD_GB300_H
#define SSD_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SSD_API __attribute__((visibility("default")))
#else
#define SSD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Storage type of x, B, C, dy, y, dx, dB, dC.  Every other tensor is fp32 and
 * every accumulation runs in fp32. */
typedef enum { SSD_F32 = 0, SSD_BF16 = 1 } ssd_dtype;

/* Return codes. */
enum {
  SSD_OK = 0,
  SSD_ERR_INVALID_ARG = 1,    /* null required pointer, bad size, small workspace */
  SSD_ERR_UNSUPPORTED = 2,    /* valid but unsupported shape (see ssd_forward) */
  SSD_ERR_ALIGNMENT = 3,      /* a pointer is not 16-byte aligned */
  SSD_ERR_CUDA = 4,           /* a CUDA runtime call failed (message has it) */
  SSD_ERR_DEVICE_TIMEOUT = 5  /* a bounded device-side wait gave up */
};

typedef struct {
  int64_t batch;    /* B  >= 1 */
  int64_t seqlen;   /* T  >= 1, multiple of chunk */
  int64_t nheads;   /* H  >= 1, multiple of ngroups */
  int64_t headdim;  /* P  in [16, 128], multiple of 16 */
  int64_t dstate;   /* N  in [16, 256], multiple of 16; P * N <= 16384 */
  int64_t ngroups;  /* G  >= 1 */
  int64_t chunk;    /* Q  one of 16, 32, 64, 128, 256 */
  int32_t dtype;    /* ssd_dtype */
  int32_t reserved; /* must be 0 */
} ssd_dims;

/* Bytes of device workspace needed for these dims.  which = 0: ssd_forward;
 * 1: ssd_backward given the chunk history; 2: ssd_backward with
 * chunk_states = NULL (history recomputed inside the call); 3, 4, 5: the same
 * three for ssd_forward_raw / ssd_backward_raw.  Returns 0 for dims the
 * library rejects (ssd_last_error then says why). */
SSD_API size_t ssd_workspace_bytes(const ssd_dims* dims, int which);

/*
 * Forward.  Inputs x, dt, A, B, C, D (required) and h0 (NULL = zeros).
 * Outputs: y (required); final_state (NULL = not written); chunk_states
 * (NULL = not written; pass it to ssd_backward to skip the recompute).
 * workspace: device memory of at least ssd_workspace_bytes(dims, 0) bytes,
 * 256-byte aligned, contents ignored and clobbered.
 * Errors: SSD_ERR_INVALID_ARG, SSD_ERR_UNSUPPORTED (T % chunk != 0, chunk not
 * in {16..256}, P or N out of range), SSD_ERR_ALIGNMENT, SSD_ERR_CUDA.  On an
 * error nothing is launched.
 */
SSD_API int ssd_forward(const ssd_dims* dims,
                        const void* x, const float* dt, const float* A,
                        const void* B, const void* C, const float* D,
                        const float* h0,
                        void* y, float* final_state, float* chunk_states,
                        void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * Backward of L = sum(dy * y).  Same inputs as ssd_forward plus dy.
 * chunk_states: the history ssd_forward wrote for the same inputs, or NULL to
 * recompute it inside this call (needs ssd_workspace_bytes(dims, 2)).  At
 * chunk 256 the tensor-core block family (headdim 64 with d_state 64;
 * headdim 128) works on 128-step sub-chunks and recomputes their start
 * states in either case (the same kernels as ssd_forward, so the results do
 * not depend on the argument).
 * Outputs (all required except dh0): dx, ddt, dA, dB, dC, dD; dh0 (NULL = not
 * written; when h0 is NULL it is the gradient w.r.t. the zero initial state).
 * The gradient w.r.t. the final state is taken as zero.
 */
SSD_API int ssd_backward(const ssd_dims* dims,
                         const void* x, const float* dt, const float* A,
                         const void* B, const void* C, const float* D,
                         const float* h0, const void* dy, const float* chunk_states,
                         void* dx, float* ddt, float* dA, void* dB, void* dC, float* dD,
                         float* dh0,
                         void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * The core with the dt and A preprocessing in front of it
 * (burn_dragon_kernel 0.5.0, src/sequence/mamba2/backward.rs,
 * `tensorized_mamba2_backward_impl`, where dt = softplus(dt_raw + dt_bias)
 * per head and A = -exp(a_log); its backward multiplies the gradient w.r.t.
 * dt by sigmoid(dt_raw + dt_bias) and sums it over batch and time for
 * dt_bias; `ssd_backward_reference` gives the gradient w.r.t. a_log as the
 * summed gradient w.r.t. A times -exp(a_log)).
 *   dt_raw, d_dt_raw   [B][T][H] fp32
 *   dt_bias, a_log, d_dt_bias, d_a_log   [H] fp32
 * Every other argument, layout, error and rule is that of ssd_forward /
 * ssd_backward; the workspace is ssd_workspace_bytes(dims, 3) (forward), 4
 * (backward given the history) or 5 (backward recomputing it).  The history
 * written by ssd_forward_raw is the core's history for dt and A.  Where the
 * fused tensor-core path applies, the transforms run inside the core's
 * kernels; elsewhere a preprocessing kernel writes dt and A into the
 * workspace and a gradient pass follows the core.
 */
SSD_API int ssd_forward_raw(const ssd_dims* dims,
                            const void* x, const float* dt_raw, const float* dt_bias,
                            const float* a_log, const void* B, const void* C, const float* D,
                            const float* h0,
                            void* y, float* final_state, float* chunk_states,
                            void* workspace, size_t workspace_bytes, void* cuda_stream);
SSD_API int ssd_backward_raw(const ssd_dims* dims,
                             const void* x, const float* dt_raw, const float* dt_bias,
                             const float* a_log, const void* B, const void* C, const float* D,
                             const float* h0, const void* dy, const float* chunk_states,
                             void* dx, float* d_dt_raw, float* d_dt_bias, float* d_a_log,
                             void* dB, void* dC, float* dD, float* dh0,
                             void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * Gated RMSNorm, the step after the core (burn_dragon_kernel 0.5.0,
 * src/sequence/mamba2/backward.rs, `rmsnorm_gated_forward_from_inv_rms` and
 * `rmsnorm_gated_backward_from_inv_rms`; inv_rms as
 * `tensorized_mamba2_backward_impl` forms it), on `rows` rows of `width`
 * (for the SSD output: rows = B*T, width = H*P):
 *   inv_rms[r] = 1 / sqrt(mean_w y[r][w]^2 + eps)
 *   out[r][w]  = y[r][w] * inv_rms[r] * weight[w] * silu(z[r][w])
 * The backward returns dy, dz and dweight (summed over the rows) for the
 * gradient dout of out; inv_rms may be the forward's (NULL = recomputed).
 *   y, z, out, dout, dy, dz   [rows][width]   `dtype` (ssd_dtype)
 *   weight, dweight           [width]         fp32
 *   inv_rms                   [rows]          fp32
 * width: a multiple of 256 (bf16) or 128 (fp32), at most 4096.  Pointers
 * 16-byte aligned; the backward's workspace is
 * ssd_rmsnorm_gated_workspace_bytes(rows, width) bytes (0 = rejected).
 * Errors as for ssd_forward; results are deterministic (fixed-order sums).
 */
SSD_API size_t ssd_rmsnorm_gated_workspace_bytes(int64_t rows, int64_t width);
SSD_API int ssd_rmsnorm_gated_forward(int64_t rows, int64_t width, int32_t dtype,
                                      const void* y, const void* z, const float* weight,
                                      float eps, void* out, float* inv_rms, void* cuda_stream);
SSD_API int ssd_rmsnorm_gated_backward(int64_t rows, int64_t width, int32_t dtype,
                                       const void* y, const void* z, const float* weight,
                                       float eps, const float* inv_rms, const void* dout,
                                       void* dy, void* dz, float* dweight,
                                       void* workspace, size_t workspace_bytes,
                                       void* cuda_stream);

/*
 * Causal depthwise conv1d + SiLU on xBC, the step before the core
 * (burn_dragon_kernel 0.5.0, src/sequence/mamba2/backward.rs,
 * `depthwise_conv_preact_with_history` and the fallback conv backward of
 * `tensorized_mamba2_backward_impl`).  Per batch row and channel c, with the
 * history h = [init_state (d_conv entries) | x (seqlen entries)]:
 *   out[t] = silu(bias[c] + sum_{k < d_conv} weight[c][k] * h[t + k + 1])
 * (h[t + d_conv] = x[t]; init_state NULL = zeros, bias NULL = 0).  The
 * backward returns dx, dweight and dbias (dbias may be NULL); the gradient
 * w.r.t. the initial state is not formed, as on the page.
 *   x, out, dout, dx      [batch][seqlen][channels]   `dtype` (ssd_dtype)
 *   weight, dweight       [channels][d_conv]          fp32
 *   bias, dbias           [channels]                  fp32
 *   init_state            [batch][channels][d_conv]   fp32
 * channels: a multiple of 8 (bf16) or 4 (fp32); d_conv in [1, 4]; batch <=
 * 65535 and batch * seqlen below 2^31 - 1024 (x and dout are read as
 * [batch*seqlen][channels] TMA tensors with 32-bit row coordinates).
 * Pointers 16-byte aligned; the backward's workspace is
 * ssd_conv1d_silu_workspace_bytes(batch, seqlen, channels, d_conv) bytes.
 * Errors as for ssd_forward (SSD_ERR_CUDA also when the driver cannot encode
 * the tensor maps); results are deterministic.  The kernels' waits on their
 * copies are bounded and report through ssd_device_status.
 */
SSD_API size_t ssd_conv1d_silu_workspace_bytes(int64_t batch, int64_t seqlen, int64_t channels,
                                               int32_t d_conv);
SSD_API int ssd_conv1d_silu_forward(int64_t batch, int64_t seqlen, int64_t channels,
                                    int32_t d_conv, int32_t dtype, const void* x,
                                    const float* weight, const float* bias,
                                    const float* init_state, void* out, void* cuda_stream);
SSD_API int ssd_conv1d_silu_backward(int64_t batch, int64_t seqlen, int64_t channels,
                                     int32_t d_conv, int32_t dtype, const void* x,
                                     const float* weight, const float* bias,
                                     const float* init_state, const void* dout, void* dx,
                                     float* dweight, float* dbias,
                                     void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * Forward pass that allocates nothing (no counterpart on the pages: an
 * addition of this library for callers that cannot allocate).
 * Same inputs, outputs, layouts, errors and launch sequence as ssd_forward
 * (its outputs are bit-for-bit those of ssd_forward for the same dims), but
 * no workspace argument: it works in a fixed device array of
 * SSD_NOALLOC_SCRATCH_BYTES that is part of the library image, for callers
 * that own all device memory through their own pool, run where an
 * allocation may synchronise the device or fail, or have no allocator at
 * hand.  It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - The array lives on every GPU that loads the library until the process
 *     exits.  The first call on a device looks up its address on that device
 *     (cudaGetSymbolAddress); make that first call before any stream
 *     capture.  Only a successful lookup is kept; after a failure
 *     (SSD_ERR_CUDA) the next call looks again.
 *   - All calls on a device share the array and it keeps the last call's
 *     contents: calls whose kernels may overlap on the GPU (several streams
 *     or host threads) race; order them.  What must start at zero is
 *     cleared by each call on its own stream.
 *   - Scratch used: B*H*nc floats and B*nc*H + 1 words, plus B*nc*H*P*N
 *     floats when chunk_states is NULL (each rounded up to 256 bytes); the
 *     tensor-core block family at chunk 256 counts nc as T / 128 and always
 *     keeps its chunk states in the scratch.
 *     Larger problems are rejected with SSD_ERR_UNSUPPORTED and a message;
 *     nothing is launched.
 */
#define SSD_NOALLOC_SCRATCH_BYTES (8u << 20)
SSD_API int ssd_forward_noalloc(const ssd_dims* dims,
                                const void* x, const float* dt, const float* A,
                                const void* B, const void* C, const float* D,
                                const float* h0,
                                void* y, float* final_state, float* chunk_states,
                                void* cuda_stream);

/* Message for the last non-zero return on this thread ("" if none). */
SSD_API const char* ssd_last_error(void);

/* Number of kernels this process has launched through the library so far
 * (all threads).  Diagnostic counter for benchmarks. */
SSD_API uint64_t ssd_kernel_launch_count(void);

/* Per-kernel timing trace (diagnostics).  While a trace is open, every kernel
 * the library launches is bracketed by a pair of CUDA events recorded on the
 * launch stream.  ssd_trace_begin(capacity) opens a trace for up to
 * `capacity` launches (creates 2*capacity events; needs a current device);
 * ssd_trace_end() stops recording; ssd_trace_read(i, ...) synchronises on the
 * recorded events and returns, for the i-th distinct kernel name in first
 * launch order, its name, the summed event time in milliseconds and its
 * launch count (returns SSD_ERR_INVALID_ARG past the last name);
 * ssd_trace_reset() destroys the events.  Launches beyond `capacity` are
 * counted but not timed (ssd_trace_read reports them in `untimed`).  Not
 * thread-safe against concurrent library calls on other threads. */
SSD_API int ssd_trace_begin(int capacity);
SSD_API int ssd_trace_end(void);
SSD_API int ssd_trace_read(int index, char* name, int name_len, double* total_ms,
                           int* launches, int* untimed);
SSD_API int ssd_trace_reset(void);

/* Which kernel family ssd_forward/ssd_backward select for these dims:
 * 0 = SIMT fp32 kernels, 1 = tcgen05 tensor-core kernels.  -1 if rejected. */
SSD_API int ssd_kernel_path(const ssd_dims* dims);

/* Restrict kernel selection: path = 0 uses the SIMT kernels for every shape,
 * path = -1 restores automatic selection.  Process-wide; for tests. */
SSD_API int ssd_force_kernel_path(int path);

/* Reads and clears the device-side error words that bounded waits inside the
 * tensor-core kernels and the conv1d kernels set when they give up
 * (synchronous: it copies from the device).  Returns SSD_OK,
 * SSD_ERR_DEVICE_TIMEOUT or SSD_ERR_CUDA. */
SSD_API int ssd_device_status(void);

/* Failure-path self test: launches one CTA whose bounded wait on an mbarrier
 * that nothing completes gives up after about one second and sets the
 * device error word; the kernel then returns normally.  After the caller
 * synchronises, ssd_device_status() reports SSD_ERR_DEVICE_TIMEOUT (once).
 * Returns SSD_OK or SSD_ERR_CUDA (launch failure). */
SSD_API int ssd_selftest_wait_timeout(void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* SSD_GB300_H */
