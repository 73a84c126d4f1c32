// Device helpers shared by the SSD kernels: storage-type conversion and
// block-wide scans/reductions with a fixed evaluation order.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssd {

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// Inclusive prefix sum over the block (blockDim.x a multiple of 32, <= 1024).
// `scratch` holds at least blockDim.x / 32 floats.  All threads must call.
// The result is a pure function of the inputs (fixed order of additions).
__device__ __forceinline__ float block_inclusive_scan(float v, float* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  __syncthreads();
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  float base = 0.f;
  for (int w = 0; w < warp; ++w) base += scratch[w];
  return v + base;
}

// Sum over the block in a fixed order (warp butterfly, then warps in order).
// Every thread receives the total.  `scratch` holds blockDim.x / 32 floats.
__device__ __forceinline__ float block_sum(float v, float* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  float s = 0.f;
  const int nw = blockDim.x >> 5;
  for (int w = 0; w < nw; ++w) s += scratch[w];
  return s;
}

// Inclusive prefix sums of two values at once (same fixed order as above).
// `scratch` holds at least blockDim.x / 32 float2.
__device__ __forceinline__ float2 block_inclusive_scan2(float2 v, float2* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float tx = __shfl_up_sync(0xffffffffu, v.x, o);
    const float ty = __shfl_up_sync(0xffffffffu, v.y, o);
    if (lane >= o) {
      v.x += tx;
      v.y += ty;
    }
  }
  __syncthreads();
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  float2 base = make_float2(0.f, 0.f);
  for (int w = 0; w < warp; ++w) {
    base.x += scratch[w].x;
    base.y += scratch[w].y;
  }
  return make_float2(v.x + base.x, v.y + base.y);
}

// Sum of two values over the block in a fixed order; every thread gets both.
__device__ __forceinline__ float2 block_sum2(float2 v, float2* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
    v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
  }
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  float2 t = make_float2(0.f, 0.f);
  const int nw = blockDim.x >> 5;
  for (int w = 0; w < nw; ++w) {
    t.x += scratch[w].x;
    t.y += scratch[w].y;
  }
  return t;
}

}  // namespace ssd
