// Causal depthwise conv1d + SiLU on xBC, the step before the SSD core
// (burn_dragon_kernel 0.5.0, src/sequence/mamba2/backward.rs,
// `depthwise_conv_preact_with_history` and the fallback backward of
// `tensorized_mamba2_backward_impl`).  Per batch row and channel c, with
// the history h = [init (K entries) | x (T entries)]:
//   pre[t] = bias[c] + sum_{k<K} w[c][k] h[t + k + 1]      (h[t + K] = x[t])
//   out[t] = silu(pre[t])
// backward, with gp[t] = dout[t] silu'(pre[t]):
//   dx[t]   = sum_{k<K, t + K - 1 - k < T} gp[t + K - 1 - k] w[c][k]
//   dw[c][k] = sum_{b,t} gp[t] h[t + k + 1],  dbias[c] = sum_{b,t} gp[t]
// (the gradient w.r.t. the initial state is not formed, as on the page).
//
// Layouts: x, out, dout, dx [B][T][C] (`dtype`); w [C][K], bias [C], init
// [B][C][K], dw [C][K], dbias [C] fp32.  A thread owns 4 channels (one 8-byte
// bf16 or 16-byte fp32 vector; a warp-row of kConvChunks threads is one
// coalesced run) and one tile of steps; a CTA stacks consecutive tiles.
// The tile's loads are unconditional (indices clamped into the sequence,
// the extra values unused), so the walk, unrolled by 4, can issue them
// ahead.  The backward walks forward in time over the tile
// plus K - 1 steps past it, keeping the last K inputs and the K - 1 dx
// values still open; it stores dx of a step once the gradient of the step
// K - 1 later is in.  dw and dbias: the CTA sums its tiles in shared memory
// in order, a last kernel sums the CTAs along time in order.
#include <cuda_bf16.h>

#include "ssd_common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kE = 4;  // channels per thread

template <typename T>
struct CVec;
template <>
struct CVec<float> {
  __device__ static void load(const void* p, float* v) {
    const float4 q = *(const float4*)p;
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  }
  __device__ static void store(void* p, const float* v) { *(float4*)p = make_float4(v[0], v[1], v[2], v[3]); }
};
template <>
struct CVec<__nv_bfloat16> {
  __device__ static void load(const void* p, float* v) {
    const uint2 q = *(const uint2*)p;
    const float2 a = __bfloat1622float2(*(const __nv_bfloat162*)&q.x);
    const float2 b = __bfloat1622float2(*(const __nv_bfloat162*)&q.y);
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
  }
  __device__ static void store(void* p, const float* v) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
    const __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
    *(uint2*)p = make_uint2(*(const unsigned*)&a, *(const unsigned*)&b);
  }
};

// logistic sigmoid with the fast exponential and divide; the exponent is
// capped at 80 so that the divisor stays below 2^126, where the fast divide
// is accurate (for z < -80 the result, below 2e-35, is immaterial to silu)
__device__ __forceinline__ float sig(float z) {
  return __fdividef(1.f, 1.f + __expf(fminf(-z, 80.f)));
}

// history value of step s (s >= -K, s < T) for the channels at c0
template <typename T, int K>
__device__ __forceinline__ void hist_load(const T* x, const float* init, int b, int s, int C, int c0,
                                          long long T_, float* v) {
  if (s >= 0) {
    CVec<T>::load(x + ((long long)b * T_ + s) * C + c0, v);
  } else {
#pragma unroll
    for (int e = 0; e < kE; ++e) v[e] = init ? init[((long long)b * C + c0 + e) * K + K + s] : 0.f;
  }
}

template <int K>
__device__ __forceinline__ void load_params(const float* w, const float* bias, int c0,
                                            float (&wv)[K][kE], float (&bv)[kE]) {
#pragma unroll
  for (int e = 0; e < kE; ++e) {
    bv[e] = bias ? bias[c0 + e] : 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) wv[k][e] = w[(c0 + e) * K + k];
  }
}

template <typename T, int K>
__global__ void __launch_bounds__(kConvChunks * kConvFwdSlots)
k_conv_fwd(int T_, int C, const T* __restrict__ x, const float* __restrict__ w,
           const float* __restrict__ bias, const float* __restrict__ init, T* __restrict__ out) {
  const int c0 = (blockIdx.x * kConvChunks + threadIdx.x) * kE, b = blockIdx.z;
  if (c0 >= C) return;
  const int t0 = (blockIdx.y * kConvFwdSlots + threadIdx.y) * kConvFwdTile;
  if (t0 >= T_) return;
  const int t1 = min(T_, t0 + kConvFwdTile);
  float wv[K][kE], bv[kE], win[K][kE];  // win[k] = h of step t - K + 1 + k
  load_params<K>(w, bias, c0, wv, bv);
#pragma unroll
  for (int k = 0; k < K - 1; ++k) hist_load<T, K>(x, init, b, t0 - K + 1 + k, C, c0, T_, win[k]);
  const T* xr = x + (long long)b * T_ * C + c0;
  T* orow = out + (long long)b * T_ * C + c0;
#pragma unroll 4
  for (int i = 0; i < kConvFwdTile; ++i) {
    const int t = t0 + i;
    CVec<T>::load(xr + (long long)min(t, t1 - 1) * C, win[K - 1]);
    float o[kE];
#pragma unroll
    for (int e = 0; e < kE; ++e) {
      float p = bv[e];
#pragma unroll
      for (int k = 0; k < K; ++k) p = fmaf(wv[k][e], win[k][e], p);
      o[e] = p * sig(p);
    }
    if (t < t1) CVec<T>::store(orow + (long long)t * C, o);
#pragma unroll
    for (int k = 0; k < K - 1; ++k)
#pragma unroll
      for (int e = 0; e < kE; ++e) win[k][e] = win[k + 1][e];
  }
}

// part: [B * gridDim.y][C][K + 1] (dw taps, then dbias) per (b, CTA row along time)
template <typename T, int K>
__global__ void __launch_bounds__(kConvChunks * kConvBwdSlots, kConvBwdMinCtas)
k_conv_bwd(int T_, int C, const T* __restrict__ x, const float* __restrict__ w,
           const float* __restrict__ bias, const float* __restrict__ init, const T* __restrict__ dout,
           T* __restrict__ dx, float* __restrict__ part) {
  __shared__ float s_red[kConvBwdSlots][kConvChunks * kE * (K + 1)];
  const int c0 = (blockIdx.x * kConvChunks + threadIdx.x) * kE, b = blockIdx.z;
  const int t0 = (blockIdx.y * kConvBwdSlots + threadIdx.y) * kConvBwdTile;
  const int t1 = min(T_, t0 + kConvBwdTile);
  float dw[K][kE], db[kE];
#pragma unroll
  for (int e = 0; e < kE; ++e) {
    db[e] = 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) dw[k][e] = 0.f;
  }
  if (c0 < C && t0 < T_) {
    float wv[K][kE], bv[kE];
    load_params<K>(w, bias, c0, wv, bv);
    float xw[K][kE];  // xw[k] = h of step t - K + 1 + k
#pragma unroll
    for (int k = 0; k < K - 1; ++k) hist_load<T, K>(x, init, b, t0 - K + 1 + k, C, c0, T_, xw[k]);
    // open[j]: dx of step t - K + 1 + j summed over the gradients of steps < t
    float open[K > 1 ? K - 1 : 1][kE];
#pragma unroll
    for (int j = 0; j < K - 1; ++j)
#pragma unroll
      for (int e = 0; e < kE; ++e) open[j][e] = 0.f;
    const long long row = (long long)b * T_ * C + c0;
#pragma unroll 4
    for (int i = 0; i < kConvBwdTile + K - 1; ++i) {
      const int t = t0 + i;
      const long long tc = (long long)min(t, T_ - 1) * C;
      float d[kE], g[kE], o[kE];
      CVec<T>::load(x + row + tc, xw[K - 1]);
      CVec<T>::load(dout + row + tc, d);
      const bool in_seq = t < T_, owned = t < t1;
#pragma unroll
      for (int e = 0; e < kE; ++e) {
        float p = bv[e];
#pragma unroll
        for (int k = 0; k < K; ++k) p = fmaf(wv[k][e], xw[k][e], p);
        const float sg = sig(p);
        g[e] = in_seq ? d[e] * sg * (1.f + p * (1.f - sg)) : 0.f;
        if (owned) {
          db[e] += g[e];
#pragma unroll
          for (int k = 0; k < K; ++k) dw[k][e] = fmaf(g[e], xw[k][e], dw[k][e]);
        }
        // this step's gradient reaches dx of steps t - K + 1 .. t through taps 0 .. K - 1
        if (K > 1) {
          o[e] = fmaf(g[e], wv[0][e], open[0][e]);
#pragma unroll
          for (int j = 0; j + 1 < K - 1; ++j) open[j][e] = fmaf(g[e], wv[j + 1][e], open[j + 1][e]);
          open[K > 1 ? K - 2 : 0][e] = g[e] * wv[K - 1][e];
        } else {
          o[e] = g[e] * wv[0][e];
        }
      }
      const int s = t - K + 1;  // dx of step s is complete
      if (s >= t0 && s < t1) CVec<T>::store(dx + row + (long long)s * C, o);
#pragma unroll
      for (int k = 0; k < K - 1; ++k)
#pragma unroll
        for (int e = 0; e < kE; ++e) xw[k][e] = xw[k + 1][e];
    }
  }
  // this CTA's tiles summed in order (slot 0 first), per channel and tap
  float* mine = &s_red[threadIdx.y][threadIdx.x * kE * (K + 1)];
#pragma unroll
  for (int e = 0; e < kE; ++e) {
#pragma unroll
    for (int k = 0; k < K; ++k) mine[e * (K + 1) + k] = dw[k][e];
    mine[e * (K + 1) + K] = db[e];
  }
  __syncthreads();
  const int n = kConvChunks * kE * (K + 1);
  const int cbase = blockIdx.x * kConvChunks * kE;
  float* pr = part + ((size_t)(b * gridDim.y + blockIdx.y) * C + cbase) * (K + 1);
  for (int i = threadIdx.y * kConvChunks + threadIdx.x; i < n; i += kConvChunks * kConvBwdSlots) {
    if (cbase + i / (K + 1) >= C) continue;
    float t = 0.f;
    for (int sl = 0; sl < kConvBwdSlots; ++sl) t += s_red[sl][i];
    pr[i] = t;
  }
}

// dw, dbias: the (b, tile) partials summed in order
__global__ void k_conv_dw(int nparts, int C, int K, const float* __restrict__ part,
                          float* __restrict__ dw, float* __restrict__ dbias) {
  const int n = C * (K + 1);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    float t = 0.f;
    for (int p = 0; p < nparts; ++p) t += part[(size_t)p * n + i];
    const int c = i / (K + 1), k = i % (K + 1);
    if (k < K) dw[c * K + k] = t;
    else if (dbias) dbias[c] = t;
  }
}

template <typename T, int K>
cudaError_t conv_fwd_t(long long B, int T_, int C, const void* x, const float* w,
                       const float* bias, const float* init, void* out, cudaStream_t s) {
  const dim3 grid((C / kE + kConvChunks - 1) / kConvChunks, (T_ + kConvFwdRows - 1) / kConvFwdRows,
                  (unsigned)B);
  k_conv_fwd<T, K><<<grid, dim3(kConvChunks, kConvFwdSlots), 0, s>>>(T_, C, (const T*)x, w, bias,
                                                                  init, (T*)out);
  return cudaGetLastError();
}

template <typename T, int K>
cudaError_t conv_bwd_t(long long B, int T_, int C, const void* x, const float* w,
                       const float* bias, const float* init, const void* dout, void* dx,
                       float* part, cudaStream_t s) {
  const dim3 grid((C / kE + kConvChunks - 1) / kConvChunks, (T_ + kConvBwdRows - 1) / kConvBwdRows,
                  (unsigned)B);
  k_conv_bwd<T, K><<<grid, dim3(kConvChunks, kConvBwdSlots), 0, s>>>(T_, C, (const T*)x, w, bias,
                                                                  init, (const T*)dout, (T*)dx, part);
  return cudaGetLastError();
}

}  // namespace

cudaError_t conv_forward(long long B, int T_, int C, int K, bool bf16, const void* x,
                         const float* w, const float* bias, const float* init, void* out,
                         cudaStream_t s) {
  LaunchScope ls("conv1d_silu_fwd", s);
#define SSD_CONV_F(TT, KK) return conv_fwd_t<TT, KK>(B, T_, C, x, w, bias, init, out, s)
  if (bf16) {
    switch (K) {
      case 1: SSD_CONV_F(__nv_bfloat16, 1);
      case 2: SSD_CONV_F(__nv_bfloat16, 2);
      case 3: SSD_CONV_F(__nv_bfloat16, 3);
      default: SSD_CONV_F(__nv_bfloat16, 4);
    }
  }
  switch (K) {
    case 1: SSD_CONV_F(float, 1);
    case 2: SSD_CONV_F(float, 2);
    case 3: SSD_CONV_F(float, 3);
    default: SSD_CONV_F(float, 4);
  }
#undef SSD_CONV_F
}

cudaError_t conv_backward(long long B, int T_, int C, int K, bool bf16, const void* x,
                          const float* w, const float* bias, const float* init, const void* dout,
                          void* dx, float* dw, float* dbias, float* part, cudaStream_t s) {
  cudaError_t e;
  {
    LaunchScope ls("conv1d_silu_bwd", s);
#define SSD_CONV_B(TT, KK) e = conv_bwd_t<TT, KK>(B, T_, C, x, w, bias, init, dout, dx, part, s)
    if (bf16) {
      switch (K) {
        case 1: SSD_CONV_B(__nv_bfloat16, 1); break;
        case 2: SSD_CONV_B(__nv_bfloat16, 2); break;
        case 3: SSD_CONV_B(__nv_bfloat16, 3); break;
        default: SSD_CONV_B(__nv_bfloat16, 4); break;
      }
    } else {
      switch (K) {
        case 1: SSD_CONV_B(float, 1); break;
        case 2: SSD_CONV_B(float, 2); break;
        case 3: SSD_CONV_B(float, 3); break;
        default: SSD_CONV_B(float, 4); break;
      }
    }
#undef SSD_CONV_B
  }
  if (e != cudaSuccess) return e;
  const int nparts = (int)(B * ((T_ + kConvBwdRows - 1) / kConvBwdRows));
  {
    LaunchScope ls("conv1d_silu_dw", s);
    k_conv_dw<<<(C * (K + 1) + 255) / 256, 256, 0, s>>>(nparts, C, K, part, dw, dbias);
  }
  return cudaGetLastError();
}

}  // namespace ssd
