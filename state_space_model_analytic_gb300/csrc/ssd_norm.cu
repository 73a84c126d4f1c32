// Gated RMSNorm, the step after the SSD core (burn_dragon_kernel 0.5.0,
// src/sequence/mamba2/backward.rs, `rmsnorm_gated_forward_from_inv_rms` and
// `rmsnorm_gated_backward_from_inv_rms`, with inv_rms = 1 / sqrt(mean(y^2) +
// eps) over the row as `tensorized_mamba2_backward_impl` forms it):
//   out = (y * inv_rms) * w * silu(z)
// backward, with g = d out, gate = silu(z), n = y * inv_rms:
//   dw    = sum over rows of g * gate * n
//   gn    = g * gate * w;  dot = sum_w gn * y
//   dy    = gn * inv_rms - y * dot * inv_rms^3 / width
//   dz    = g * n * w * silu'(z),  silu'(z) = s (1 + z (1 - s)), s = sigmoid(z)
//
// One warp per row, 16-byte vector accesses (the rows are HBM-streamed; the
// second pass over y re-reads it from L1).  dw: each warp sums its rows'
// products for the columns its lanes own into a per-warp shared-memory row,
// the CTA sums its warps in order, and a final kernel sums the CTAs in order
// (deterministic).
#include <cuda_bf16.h>

#include "ssd_common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kNormWarps = 8;  // warps (rows in flight) per CTA

template <typename T>
struct Vec;  // 16 bytes of T
template <>
struct Vec<float> {
  static constexpr int n = 4;
  __device__ static void load(const void* p, float* v) {
    const float4 q = *(const float4*)p;
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  }
  __device__ static void store(void* p, const float* v) { *(float4*)p = make_float4(v[0], v[1], v[2], v[3]); }
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int n = 8;
  __device__ static void load(const void* p, float* v) {
    const uint4 q = *(const uint4*)p;
    const __nv_bfloat162* h = (const __nv_bfloat162*)&q;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
  __device__ static void store(void* p, const float* v) {
    uint4 q;
    __nv_bfloat162* h = (__nv_bfloat162*)&q;
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    *(uint4*)p = q;
  }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float sigmoidf_(float z) { return 1.f / (1.f + expf(-z)); }

template <typename T>
__global__ void __launch_bounds__(32 * kNormWarps)
k_norm_fwd(long long rows, int width, float eps, const T* __restrict__ y, const T* __restrict__ z,
           const float* __restrict__ w, T* __restrict__ out, float* __restrict__ inv_rms) {
  constexpr int E = Vec<T>::n;
  const int lane = threadIdx.x & 31;
  const long long r = (long long)blockIdx.x * kNormWarps + (threadIdx.x >> 5);
  if (r >= rows) return;
  const T* yr = y + r * width;
  float ss = 0.f;
#pragma unroll 4
  for (int c = lane * E; c < width; c += 32 * E) {
    float v[E];
    Vec<T>::load(yr + c, v);
#pragma unroll
    for (int i = 0; i < E; ++i) ss = fmaf(v[i], v[i], ss);
  }
  const float inv = 1.f / sqrtf(warp_sum(ss) / (float)width + eps);
  const T* zr = z + r * width;
  T* orow = out + r * width;
#pragma unroll 4
  for (int c = lane * E; c < width; c += 32 * E) {
    float v[E], zz[E], wv[E], o[E];
    Vec<T>::load(yr + c, v);
    Vec<T>::load(zr + c, zz);
    Vec<float>::load(w + c, wv);
    if constexpr (E == 8) Vec<float>::load(w + c + 4, wv + 4);
#pragma unroll
    for (int i = 0; i < E; ++i) o[i] = (v[i] * inv) * wv[i] * (zz[i] * sigmoidf_(zz[i]));
    Vec<T>::store(orow + c, o);
  }
  if (inv_rms && lane == 0) inv_rms[r] = inv;
}

// Persistent: warp j of CTA b takes rows (b * kNormWarps + j) + k * (grid * kNormWarps).
// part: [grid][width] per-CTA column sums of g * gate * n.
template <typename T>
__global__ void __launch_bounds__(32 * kNormWarps)
k_norm_bwd(long long rows, int width, float eps, const T* __restrict__ y, const T* __restrict__ z,
           const float* __restrict__ w, const float* __restrict__ inv_in, const T* __restrict__ g,
           T* __restrict__ dy, T* __restrict__ dz, float* __restrict__ part) {
  constexpr int E = Vec<T>::n;
  extern __shared__ float s_dw[];  // [kNormWarps][width]
  const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
  float* my = s_dw + (size_t)wp * width;
  for (int c = lane; c < width; c += 32) my[c] = 0.f;
  __syncwarp();
  const long long stride = (long long)gridDim.x * kNormWarps;
  for (long long r = (long long)blockIdx.x * kNormWarps + wp; r < rows; r += stride) {
    const T* yr = y + r * width;
    const T* zr = z + r * width;
    const T* gr = g + r * width;
    float inv;
    if (inv_in) {
      inv = inv_in[r];
    } else {
      float ss = 0.f;
    #pragma unroll 4
  for (int c = lane * E; c < width; c += 32 * E) {
        float v[E];
        Vec<T>::load(yr + c, v);
#pragma unroll
        for (int i = 0; i < E; ++i) ss = fmaf(v[i], v[i], ss);
      }
      inv = 1.f / sqrtf(warp_sum(ss) / (float)width + eps);
    }
    // dot = sum_w (g * gate * w) * y
    float dot = 0.f;
  #pragma unroll 4
  for (int c = lane * E; c < width; c += 32 * E) {
      float v[E], zz[E], gg[E], wv[E];
      Vec<T>::load(yr + c, v);
      Vec<T>::load(zr + c, zz);
      Vec<T>::load(gr + c, gg);
      Vec<float>::load(w + c, wv);
      if constexpr (E == 8) Vec<float>::load(w + c + 4, wv + 4);
#pragma unroll
      for (int i = 0; i < E; ++i) dot = fmaf(gg[i] * (zz[i] * sigmoidf_(zz[i])) * wv[i], v[i], dot);
    }
    dot = warp_sum(dot);
    const float k3 = dot * inv * inv * inv / (float)width;
  #pragma unroll 4
  for (int c = lane * E; c < width; c += 32 * E) {
      float v[E], zz[E], gg[E], wv[E], oy[E], oz[E], dwv[E];
      Vec<T>::load(yr + c, v);
      Vec<T>::load(zr + c, zz);
      Vec<T>::load(gr + c, gg);
      Vec<float>::load(w + c, wv);
      if constexpr (E == 8) Vec<float>::load(w + c + 4, wv + 4);
#pragma unroll
      for (int i = 0; i < E; ++i) {
        const float s = sigmoidf_(zz[i]);
        const float gate = zz[i] * s;
        const float nrm = v[i] * inv;
        oy[i] = gg[i] * gate * wv[i] * inv - v[i] * k3;
        oz[i] = gg[i] * nrm * wv[i] * (s * (1.f + zz[i] * (1.f - s)));
        dwv[i] = gg[i] * gate * nrm;
      }
#pragma unroll
      for (int i = 0; i < E; i += 4) {
        float4 a = *(float4*)(my + c + i);
        a.x += dwv[i]; a.y += dwv[i + 1]; a.z += dwv[i + 2]; a.w += dwv[i + 3];
        *(float4*)(my + c + i) = a;
      }
      Vec<T>::store(dy + r * width + c, oy);
      Vec<T>::store(dz + r * width + c, oz);
    }
  }
  __syncthreads();
  // this CTA's column sums, warps in order
  for (int c = threadIdx.x; c < width; c += blockDim.x) {
    float t = 0.f;
    for (int j = 0; j < kNormWarps; ++j) t += s_dw[(size_t)j * width + c];
    part[(size_t)blockIdx.x * width + c] = t;
  }
}


__global__ void k_norm_dw(int ncta, int width, const float* __restrict__ part, float* __restrict__ dw) {
  for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < width; c += gridDim.x * blockDim.x) {
    float t = 0.f;
    for (int b = 0; b < ncta; ++b) t += part[(size_t)b * width + c];
    dw[c] = t;
  }
}

}  // namespace

int norm_bwd_ctas(long long rows) {
  int nsm = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  long long want = (rows + kNormWarps - 1) / kNormWarps;
  long long cap = 3LL * (nsm > 0 ? nsm : 1);  // three 64 KB CTAs per SM at width 2048
  if (cap > kNormMaxCtas) cap = kNormMaxCtas;
  return (int)(want < cap ? want : cap);
}

cudaError_t norm_forward(long long rows, int width, bool bf16, const void* y, const void* z,
                         const float* w, float eps, void* out, float* inv_rms, cudaStream_t s) {
  const unsigned grid = (unsigned)((rows + kNormWarps - 1) / kNormWarps);
  LaunchScope ls("rmsnorm_gated_fwd", s);
  if (bf16)
    k_norm_fwd<__nv_bfloat16><<<grid, 32 * kNormWarps, 0, s>>>(
        rows, width, eps, (const __nv_bfloat16*)y, (const __nv_bfloat16*)z, w,
        (__nv_bfloat16*)out, inv_rms);
  else
    k_norm_fwd<float><<<grid, 32 * kNormWarps, 0, s>>>(rows, width, eps, (const float*)y,
                                                      (const float*)z, w, (float*)out, inv_rms);
  return cudaGetLastError();
}

cudaError_t norm_backward(long long rows, int width, bool bf16, const void* y, const void* z,
                          const float* w, float eps, const float* inv_rms, const void* g, void* dy,
                          void* dz, float* dw, float* part, cudaStream_t s) {
  const int ncta = norm_bwd_ctas(rows);
  const size_t smem = (size_t)kNormWarps * width * sizeof(float);
  cudaError_t e;
  if (bf16)
    e = cudaFuncSetAttribute(k_norm_bwd<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  else
    e = cudaFuncSetAttribute(k_norm_bwd<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  {
    LaunchScope ls("rmsnorm_gated_bwd", s);
    if (bf16)
      k_norm_bwd<__nv_bfloat16><<<ncta, 32 * kNormWarps, smem, s>>>(
          rows, width, eps, (const __nv_bfloat16*)y, (const __nv_bfloat16*)z, w, inv_rms,
          (const __nv_bfloat16*)g, (__nv_bfloat16*)dy, (__nv_bfloat16*)dz, part);
    else
      k_norm_bwd<float><<<ncta, 32 * kNormWarps, smem, s>>>(
          rows, width, eps, (const float*)y, (const float*)z, w, inv_rms, (const float*)g,
          (float*)dy, (float*)dz, part);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  {
    LaunchScope ls("rmsnorm_gated_dw", s);
    k_norm_dw<<<(width + 255) / 256, 256, 0, s>>>(ncta, width, part, dw);
  }
  return cudaGetLastError();
}

}  // namespace ssd
