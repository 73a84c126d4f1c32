// The dt and A preprocessing in front of the SSD core and its backward
// (burn_dragon_kernel 0.5.0, src/sequence/mamba2/backward.rs,
// `tensorized_mamba2_backward_impl`: dt = softplus(dt_raw + dt_bias[h]);
// the gradient w.r.t. dt is multiplied by sigmoid(dt_raw + dt_bias) and
// summed over batch and time for dt_bias; `ssd_backward_reference`: the
// gradient w.r.t. a_log is the summed gradient w.r.t. A times -exp(a_log)).
//
// Both passes touch B*T*H + H floats: a prep kernel writes dt and A for the
// core kernels, a post kernel turns the core's ddt and dA into the gradients
// w.r.t. dt_raw, dt_bias and a_log.  These kernels never let the next kernel
// start early (no griddepcontrol.launch_dependents): the core kernels that
// read dt and A before their griddepcontrol.wait start only once the prep
// kernel has completed.
#include "ssd_common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

// softplus(z) = log(1 + e^z), evaluated as max(z, 0) + log1p(e^{-|z|}) (no overflow)
__device__ __forceinline__ float softplus_f(float z) { return fmaxf(z, 0.f) + log1pf(expf(-fabsf(z))); }

__global__ void k_dt_prep(long long n, int H, const float* __restrict__ dt_raw,
                          const float* __restrict__ dt_bias, const float* __restrict__ a_log,
                          float* __restrict__ dt, float* __restrict__ A) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    dt[i] = softplus_f(dt_raw[i] + dt_bias[i % H]);
  if (blockIdx.x == 0)
    for (int h = threadIdx.x; h < H; h += blockDim.x) A[h] = -expf(a_log[h]);
}

// CTA (h, s): d_dt_raw (holding ddt on entry) *= sigmoid(dt_raw + bias) on
// the (b, t) rows of slice s (rows j with (j / 256) % S == s), and the slice's
// sum of the result, in a fixed order, into part[s][h].
__global__ void k_dt_post(long long bt, int H, const float* __restrict__ dt_raw,
                          const float* __restrict__ dt_bias, float* __restrict__ d_dt_raw,
                          float* __restrict__ part) {
  __shared__ float scratch[32];
  const int h = blockIdx.x, s = blockIdx.y, S = gridDim.y;
  const float bias = dt_bias[h];
  float acc = 0.f;
  for (long long j0 = (long long)s * 256; j0 < bt; j0 += (long long)S * 256) {
    const long long j = j0 + threadIdx.x;
    if (j < bt) {
      const long long i = j * H + h;
      const float z = dt_raw[i] + bias;
      const float v = d_dt_raw[i] / (1.f + expf(-z));
      d_dt_raw[i] = v;
      acc += v;
    }
  }
  const float total = block_sum(acc, scratch);
  if (threadIdx.x == 0) part[(size_t)s * H + h] = total;
}

// d_dt_bias[h] = sum of the slice sums in slice order; d_a_log[h] (holding dA
// on entry) *= -exp(a_log[h]).
__global__ void k_dt_finish(int H, int S, const float* __restrict__ part,
                            const float* __restrict__ a_log, float* __restrict__ d_dt_bias,
                            float* __restrict__ d_a_log) {
  for (int h = blockIdx.x * blockDim.x + threadIdx.x; h < H; h += gridDim.x * blockDim.x) {
    float t = 0.f;
    for (int s = 0; s < S; ++s) t += part[(size_t)s * H + h];
    d_dt_bias[h] = t;
    d_a_log[h] = d_a_log[h] * -expf(a_log[h]);
  }
}

}  // namespace

cudaError_t dt_prep(const Problem& p, const float* dt_raw, const float* dt_bias,
                    const float* a_log, float* dt, float* A) {
  const long long n = (long long)p.B * p.T * p.H;
  int blocks = (int)((n + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  {
    LaunchScope ls("dt_prep", p.stream);
    k_dt_prep<<<blocks, 256, 0, p.stream>>>(n, p.H, dt_raw, dt_bias, a_log, dt, A);
  }
  return cudaGetLastError();
}

int dt_post_slices(const Problem& p) {
  const long long bt = (long long)p.B * p.T;
  const long long tiles = (bt + 255) / 256;
  return (int)(tiles < kDtPostSlices ? tiles : kDtPostSlices);
}

cudaError_t dt_post(const Problem& p, const float* dt_raw, const float* dt_bias,
                    const float* a_log, float* d_dt_raw, float* d_dt_bias, float* d_a_log,
                    float* part) {
  const int S = dt_post_slices(p);
  {
    LaunchScope ls("dt_post", p.stream);
    k_dt_post<<<dim3(p.H, S), 256, 0, p.stream>>>((long long)p.B * p.T, p.H, dt_raw, dt_bias,
                                                 d_dt_raw, part);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    LaunchScope ls("dt_finish", p.stream);
    k_dt_finish<<<(p.H + 127) / 128, 128, 0, p.stream>>>(p.H, S, part, a_log, d_dt_bias, d_a_log);
  }
  return cudaGetLastError();
}

}  // namespace ssd
