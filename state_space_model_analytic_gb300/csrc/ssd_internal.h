// Host-side problem description shared by the C-ABI layer and the kernel
// launchers.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/ssd.h"

namespace ssd {

struct Problem {
  int B, T, H, P, N, G, Q, nc, hpg;
  int bf16;  // storage type of x, B, C, dy, y, dx, dB, dC: 0 fp32, 1 bf16

  // inputs
  const void* x;
  const float* dt;
  const float* A;
  const void* Bm;
  const void* Cm;
  const float* D;
  const float* h0;  // nullable
  const void* dy;   // backward only
  // raw-dt mode of the fused tensor-core path (both set, else nullptr): dt
  // holds dt_raw, dt = softplus(dt_raw + dt_bias), A = -exp(a_log); the
  // backward writes the gradients w.r.t. dt_raw, a_log (into ddt, dA) and
  // dt_bias
  const float* dt_bias;
  const float* a_log;
  float* d_dt_bias;

  // forward outputs
  void* y;
  float* final_state;  // nullable
  float* hist;         // [B][nc][H][P][N]: chunk-start states (user buffer or workspace)
  // the block family with chunks longer than its 128-step blocks runs on
  // 128-step sub-chunks: their start states [B][T/128][H][P][N] (workspace)
  float* hist_sub;

  // backward outputs
  void* dx;
  float* ddt;
  float* dA;
  void* dB;
  void* dC;
  float* dD;
  float* dh0;  // nullable

  // workspace carve-up
  float* cs_last;  // [B][H][nc]   total log-decay of each chunk
  float* dstate;   // [B][nc][H][P][N]  R_c, then the state gradient at chunk end
  float* rowsum;   // [B][T][H]
  float* colsum;   // [B][T][H]
  float* statein;  // [B][T][H]
  float* eout;     // [B][T][H]
  float* drive;    // [B][T][H]
  float* dA_part;  // [B][nc][Q/16][H]  (the used prefix depends on the kernel family)
  float* dD_part;  // [B][nc][Q/16][H]  (tile-count upper bound)
  float* dtb_part; // raw-dt mode: per-(b, chunk, block) sums of the dt_raw gradient, same layout
  unsigned int* tickets;  // [1 + 2 units] completion counters of the tensor-core backward
  int ntickets;
  float* bwd_part;        // tensor-core backward: fp32 dC, dB partials, 2 slots per CTA
  unsigned int* fwd_flags;  // [B*nc*H + 1]: single-pass forward slot flags, then its tile counter
  void* hT;        // [B][nc][H][N][P] bf16: chunk-start states, rows n (tensor-core backward)
  void* gT;        // [B][nc][H][N][P] bf16: chunk-end state gradients, rows n
  void* gmT;       // chunks of 256: [B][nc][H][N][P] bf16 state gradients at step 127, rows n

  cudaStream_t stream;
};

// Argument checks and problem set-up shared by the entry points
// (ssd_api.cu): each check returns SSD_OK or an SSD_ERR_* code and sets the
// thread's last-error message.
int validate_dims(const ssd_dims* d);
Problem problem_of(const ssd_dims* d);  // call after validate_dims succeeded
int check_shared_memory(const Problem& p);

// The kernels of one forward call for a carved problem (ssd_api.cu); *where
// names the kernel whose launch failed.
cudaError_t forward_launches(Problem& p, const char** where);

// Gated RMSNorm after the core (ssd_norm.cu).  The backward keeps per-CTA
// column sums of the weight gradient in part[grid][width], grid <=
// kNormMaxCtas.
constexpr int kNormMaxCtas = 512;
cudaError_t norm_forward(long long rows, int width, bool bf16, const void* y, const void* z,
                         const float* w, float eps, void* out, float* inv_rms, cudaStream_t s);
cudaError_t norm_backward(long long rows, int width, bool bf16, const void* y, const void* z,
                          const float* w, float eps, const float* inv_rms, const void* g, void* dy,
                          void* dz, float* dw, float* part, cudaStream_t s);

// Causal depthwise conv1d + SiLU before the core (ssd_conv.cu): a warp owns
// kConvCols channels of one batch row over a run of steps; the backward's
// CTAs are kConvBwdWarps such runs and keep per-CTA partials of dw, dbias in
// [B * ctas_per_column][C][K + 1], ctas_per_column <=
// conv_max_ctas_per_column(T) (runs of kConvMinRun steps or more).
constexpr int kConvCols = 128;
constexpr int kConvBwdWarps = 8;
constexpr int kConvMinRun = 16;
inline long long conv_max_ctas_per_column(long long T) {
  const long long c =
      (T + (long long)kConvBwdWarps * kConvMinRun - 1) / ((long long)kConvBwdWarps * kConvMinRun);
  return c < 1 ? 1 : c;
}
// reads and clears the conv kernels' device error word (a TMA wait gave up)
cudaError_t conv_read_and_clear_error(unsigned int* out);
cudaError_t conv_forward(long long B, int T_, int C, int K, bool bf16, const void* x,
                         const float* w, const float* bias, const float* init, void* out,
                         cudaStream_t s);
cudaError_t conv_backward(long long B, int T_, int C, int K, bool bf16, const void* x,
                          const float* w, const float* bias, const float* init, const void* dout,
                          void* dx, float* dw, float* dbias, float* part, cudaStream_t s);

// Upper bound on the CTAs of the tensor-core backward (one per SM).
constexpr size_t kBwdMaxCtas = 160;

// Kernel launchers (SIMT family).  Each returns the CUDA launch status and
// bumps the launch counter.
cudaError_t simt_forward_states(const Problem& p, float* hist, float* cs_last);
cudaError_t simt_state_pass_fwd(const Problem& p, float* hist, const float* cs_last);
// the block family with chunks longer than its 128-step blocks (ssd_tc64.cu)
bool tc64_subchunks(const Problem& p);
Problem tc64_sub_problem(const Problem& p);
cudaError_t simt_forward_scan(const Problem& p);
cudaError_t simt_backward(const Problem& p);
cudaError_t simt_state_pass_bwd(const Problem& p);
cudaError_t simt_reduce_heads(const Problem& p, int n_a, int n_d);

void count_launch(int n = 1);

// dt = softplus(dt_raw + dt_bias), A = -exp(a_log) for the core kernels, and
// the chain rule back to dt_raw, dt_bias and a_log (ssd_dtprep.cu).
cudaError_t dt_prep(const Problem& p, const float* dt_raw, const float* dt_bias,
                    const float* a_log, float* dt, float* A);
// slices of the (b, t) rows in the dt gradient pass; part holds
// kDtPostSlices * H floats of per-slice sums
constexpr int kDtPostSlices = 32;
cudaError_t dt_post(const Problem& p, const float* dt_raw, const float* dt_bias,
                    const float* a_log, float* d_dt_raw, float* d_dt_bias, float* d_a_log,
                    float* part);

// 2D row-major [rows][cols] tensor map (bf16 or fp32) with an unswizzled
// {box_cols, box_rows} box, through the driver entry point (ssd_tc.cu);
// false if the driver does not provide the encoder or rejects the map.
bool encode_rows_2d(CUtensorMap* m, const void* base, bool bf16, uint64_t rows, uint64_t cols,
                    uint32_t box_cols, uint32_t box_rows);

// Per-kernel event trace (see ssd_trace_begin in include/ssd.h).  A
// LaunchScope brackets exactly one kernel launch: it records the start event
// (when a trace is open), and on destruction the end event plus the launch
// count.
int trace_open_slot(const char* name, cudaStream_t s);
void trace_close_slot(int slot, cudaStream_t s);

struct LaunchScope {
  int slot;
  cudaStream_t stream;
  LaunchScope(const char* name, cudaStream_t s) : slot(trace_open_slot(name, s)), stream(s) {}
  ~LaunchScope() {
    trace_close_slot(slot, stream);
    count_launch();
  }
};

}  // namespace ssd
