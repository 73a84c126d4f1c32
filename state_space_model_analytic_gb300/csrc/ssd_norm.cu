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
// Work split: a CTA of up to 256 threads spans the row (thread t owns the
// 16-byte column vectors t, t + blockDim, ...: V of them, V in {1, 2, 4}) and
// walks groups of R rows (forward 4 / V, backward 2 / V or 1), persistently
// over the rows (CTA j takes groups j, j + grid, ...).  A thread copies its
// vectors of the next group into shared memory (cp.async, double-buffered)
// while it computes the current one, so two groups of 16-byte loads per
// operand are in flight per thread at no register cost; the row sums (sum
// y^2, and the backward's dot) go through one block reduction per group
// (warp shuffles, then the warps' partials in order from shared memory).  The backward keeps its columns' dw
// in registers over all its rows, writes them as the CTA's partial row, and a
// final kernel sums the CTAs in a fixed order (deterministic for a given grid,
// which follows the GPU's SM count).
#include <cuda_bf16.h>

#include "f32x2.cuh"
#include "ssd_common.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kNormThreads = 256;
constexpr int kNormWarpsMax = kNormThreads / 32;

template <typename T>
struct Vec;  // 16 bytes of T
template <>
struct Vec<float> {
  static constexpr int n = 4;
  using raw = float4;
  __device__ static void cvt(const raw& q, float* v) {
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  }
  __device__ static void store(void* p, const float* v) { *(float4*)p = make_float4(v[0], v[1], v[2], v[3]); }
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int n = 8;
  using raw = uint4;
  __device__ static void cvt(const raw& q, float* v) {
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

// 16-byte asynchronous copy global -> shared (each thread later reads back
// only what it copied itself, so waiting for its own groups suffices)
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((unsigned)__cvta_generic_to_shared(smem)),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// logistic sigmoid 1 / (1 + 2^(-z log2 e)) of a pair of values from the
// hardware base-2 exponential and reciprocal approximations (about 1e-6
// relative, exact limits at both ends), the multiply and the add packed
// (f32x2)
__device__ __forceinline__ float2 sigmoid2(float2 z) {
  const float2 u = mul2(z, make_float2(-1.4426950408889634f, -1.4426950408889634f));
  float2 e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.x) : "f"(u.x));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.y) : "f"(u.y));
  const float2 den = add2(make_float2(1.f, 1.f), e);
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.x) : "f"(den.x));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.y) : "f"(den.y));
  return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}


// Block sums of NV values per thread (row partials): every thread gets the
// totals, the warps' partials added in warp order.  red: [2][NV][warps]
// shared floats, alternated between calls (buf) so that one barrier per call
// suffices.
template <int NV>
__device__ __forceinline__ void block_sums(float (&v)[NV], float* red, int buf) {
  const int nw = blockDim.x >> 5, wp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* r = red + buf * NV * kNormWarpsMax;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const float s = warp_sum(v[i]);
    if (lane == 0) r[i * kNormWarpsMax + wp] = s;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    float t = 0.f;
    for (int j = 0; j < nw; ++j) t += r[i * kNormWarpsMax + j];
    v[i] = t;
  }
}

template <typename T, int V>
__global__ void __launch_bounds__(kNormThreads)
k_norm_fwd(long long rows, int width, float eps, const T* __restrict__ y, const T* __restrict__ z,
           const float* __restrict__ w, T* __restrict__ out, float* __restrict__ inv_rms) {
  constexpr int E = Vec<T>::n, R = 4 / V;
  using raw = typename Vec<T>::raw;
  __shared__ float red[2 * R * kNormWarpsMax];
  // [stage][r][operand y, z][v][thread] 16-byte slots (a warp's slots are contiguous)
  extern __shared__ uint4 stage[];
  const int nt = blockDim.x, t = threadIdx.x;
  auto slot = [&](int st, int r, int op, int v) -> uint4* {
    return stage + ((((size_t)st * R + r) * 2 + op) * V + v) * nt + t;
  };
  float wv[V][E];
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int c = (v * nt + t) * E;
#pragma unroll
    for (int i = 0; i < E; ++i) wv[v][i] = w[c + i];
  }
  const long long ngroups = (rows + R - 1) / R;
  auto fetch = [&](long long gi, int st) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const long long row = min(gi * R + r, rows - 1);  // past the end: a valid row, unused
        const long long off = row * width + (long long)(v * nt + t) * E;
        cp_async16(slot(st, r, 0, v), y + off);
        cp_async16(slot(st, r, 1, v), z + off);
      }
  };
  if ((long long)blockIdx.x < ngroups) fetch(blockIdx.x, 0);
  cp_async_commit();
  int buf = 0, st = 0;
  for (long long gi = blockIdx.x; gi < ngroups; gi += gridDim.x, buf ^= 1, st ^= 1) {
    const long long r0 = gi * R;
    if (gi + gridDim.x < ngroups) fetch(gi + gridDim.x, st ^ 1);
    cp_async_commit();
    cp_async_wait<1>();  // this group's copies (the thread's own) are in
    raw qy[R][V], qz[R][V];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int v = 0; v < V; ++v) {
        qy[r][v] = *(const raw*)slot(st, r, 0, v);
        qz[r][v] = *(const raw*)slot(st, r, 1, v);
      }
    float ss[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      ss[r] = 0.f;
#pragma unroll
      for (int v = 0; v < V; ++v) {
        float a[E];
        Vec<T>::cvt(qy[r][v], a);
        float2 s2 = make_float2(0.f, 0.f);  // even and odd columns (f32x2)
#pragma unroll
        for (int i = 0; i < E; i += 2) {
          const float2 a2 = make_float2(a[i], a[i + 1]);
          s2 = fma2(a2, a2, s2);
        }
        ss[r] += s2.x + s2.y;
      }
    }
    block_sums<R>(ss, red, buf);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (r0 + r >= rows) break;
      const float inv = 1.f / sqrtf(ss[r] / (float)width + eps);
#pragma unroll
      for (int v = 0; v < V; ++v) {
        float a[E], zz[E], o[E];
        Vec<T>::cvt(qy[r][v], a);
        Vec<T>::cvt(qz[r][v], zz);
        const float2 inv2 = make_float2(inv, inv);
#pragma unroll
        for (int i = 0; i < E; i += 2) {  // (a * inv) * w * (z * sigmoid(z)), pairs in f32x2
          const float2 z2 = make_float2(zz[i], zz[i + 1]);
          const float2 o2 = mul2(mul2(mul2(make_float2(a[i], a[i + 1]), inv2),
                                      make_float2(wv[v][i], wv[v][i + 1])),
                                 mul2(z2, sigmoid2(z2)));
          o[i] = o2.x;
          o[i + 1] = o2.y;
        }
        Vec<T>::store(out + (r0 + r) * width + (long long)(v * nt + t) * E, o);
      }
      if (inv_rms && t == 0) inv_rms[r0 + r] = inv;
    }
  }
  cp_async_wait<0>();
}

// part: [grid][width] per-CTA column sums of g * gate * n.
template <typename T, int V>
__global__ void __launch_bounds__(kNormThreads, 2)
k_norm_bwd(long long rows, int width, float eps, const T* __restrict__ y, const T* __restrict__ z,
           const float* __restrict__ w, const float* __restrict__ inv_in, const T* __restrict__ g,
           T* __restrict__ dy, T* __restrict__ dz, float* __restrict__ part) {
  constexpr int E = Vec<T>::n, R = V < 2 ? 2 : 1;
  using raw = typename Vec<T>::raw;
  __shared__ float red[2 * 2 * R * kNormWarpsMax];
  // [stage][r][operand y, z, g][v][thread] 16-byte slots
  extern __shared__ uint4 stage[];
  const int nt = blockDim.x, t = threadIdx.x;
  auto slot = [&](int st, int r, int op, int v) -> uint4* {
    return stage + ((((size_t)st * R + r) * 3 + op) * V + v) * nt + t;
  };
  float wv[V][E], dw[V][E];
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int c = (v * nt + t) * E;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      wv[v][i] = w[c + i];
      dw[v][i] = 0.f;
    }
  }
  const long long ngroups = (rows + R - 1) / R;
  auto fetch = [&](long long gi, int st) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const long long row = min(gi * R + r, rows - 1);  // past the end: a valid row, unused
        const long long off = row * width + (long long)(v * nt + t) * E;
        cp_async16(slot(st, r, 0, v), y + off);
        cp_async16(slot(st, r, 1, v), z + off);
        cp_async16(slot(st, r, 2, v), g + off);
      }
  };
  if ((long long)blockIdx.x < ngroups) fetch(blockIdx.x, 0);
  cp_async_commit();
  int buf = 0, st = 0;
  for (long long gi = blockIdx.x; gi < ngroups; gi += gridDim.x, buf ^= 1, st ^= 1) {
    const long long r0 = gi * R;
    float inv[R];
#pragma unroll
    for (int r = 0; r < R; ++r) inv[r] = inv_in ? inv_in[min(r0 + r, rows - 1)] : 0.f;
    if (gi + gridDim.x < ngroups) fetch(gi + gridDim.x, st ^ 1);
    cp_async_commit();
    cp_async_wait<1>();  // this group's copies (the thread's own) are in
    raw qy[R][V], qz[R][V], qg[R][V];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int v = 0; v < V; ++v) {
        qy[r][v] = *(const raw*)slot(st, r, 0, v);
        qz[r][v] = *(const raw*)slot(st, r, 1, v);
        qg[r][v] = *(const raw*)slot(st, r, 2, v);
      }
    // per row: dot = sum_w (g * gate * w) * y, and sum y^2 when inv_rms is not given
    float sums[2 * R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float dot = 0.f, ss = 0.f;
#pragma unroll
      for (int v = 0; v < V; ++v) {
        float a[E], zz[E], gg[E];
        Vec<T>::cvt(qy[r][v], a);
        Vec<T>::cvt(qz[r][v], zz);
        Vec<T>::cvt(qg[r][v], gg);
        float2 dot2 = make_float2(0.f, 0.f), ss2 = make_float2(0.f, 0.f);  // f32x2 pairs
#pragma unroll
        for (int i = 0; i < E; i += 2) {
          const float2 z2 = make_float2(zz[i], zz[i + 1]), a2 = make_float2(a[i], a[i + 1]);
          const float2 gw = mul2(mul2(make_float2(gg[i], gg[i + 1]), mul2(z2, sigmoid2(z2))),
                                 make_float2(wv[v][i], wv[v][i + 1]));
          dot2 = fma2(gw, a2, dot2);
          ss2 = fma2(a2, a2, ss2);
        }
        dot += dot2.x + dot2.y;
        ss += ss2.x + ss2.y;
      }
      sums[2 * r] = dot;
      sums[2 * r + 1] = ss;
    }
    block_sums<2 * R>(sums, red, buf);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (r0 + r >= rows) break;
      const float iv = inv_in ? inv[r] : 1.f / sqrtf(sums[2 * r + 1] / (float)width + eps);
      const float k3 = sums[2 * r] * iv * iv * iv / (float)width;
#pragma unroll
      for (int v = 0; v < V; ++v) {
        float a[E], zz[E], gg[E], oy[E], oz[E];
        Vec<T>::cvt(qy[r][v], a);
        Vec<T>::cvt(qz[r][v], zz);
        Vec<T>::cvt(qg[r][v], gg);
        const float2 iv2 = make_float2(iv, iv), nk3 = make_float2(-k3, -k3);
        const float2 one2 = make_float2(1.f, 1.f);
#pragma unroll
        for (int i = 0; i < E; i += 2) {  // pairs of columns in f32x2
          const float2 z2 = make_float2(zz[i], zz[i + 1]), a2 = make_float2(a[i], a[i + 1]);
          const float2 g2 = make_float2(gg[i], gg[i + 1]), w2 = make_float2(wv[v][i], wv[v][i + 1]);
          const float2 s2 = sigmoid2(z2);
          const float2 gate = mul2(z2, s2);
          const float2 nrm = mul2(a2, iv2);
          const float2 y2 = fma2(a2, nk3, mul2(mul2(mul2(g2, gate), w2), iv2));
          // silu'(z) = s (1 + z (1 - s))
          const float2 ds = mul2(s2, fma2(z2, fma2(s2, make_float2(-1.f, -1.f), one2), one2));
          const float2 z2o = mul2(mul2(mul2(g2, nrm), w2), ds);
          const float2 dw2 = fma2(mul2(g2, gate), nrm, make_float2(dw[v][i], dw[v][i + 1]));
          oy[i] = y2.x;
          oy[i + 1] = y2.y;
          oz[i] = z2o.x;
          oz[i + 1] = z2o.y;
          dw[v][i] = dw2.x;
          dw[v][i + 1] = dw2.y;
        }
        const long long off = (r0 + r) * width + (long long)(v * nt + t) * E;
        Vec<T>::store(dy + off, oy);
        Vec<T>::store(dz + off, oz);
      }
    }
  }
  cp_async_wait<0>();
  // this CTA's column sums
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int c = (v * nt + t) * E;
#pragma unroll
    for (int i = 0; i < E; ++i) part[(size_t)blockIdx.x * width + c + i] = dw[v][i];
  }
}

// dw[c] = sum over the CTAs' partial rows, in a fixed order: a CTA takes 32
// columns; thread (slice sl, column j) sums the partials sl, sl + 32, ... in
// order (a warp reads 32 consecutive floats of one partial row), then the 32
// slice sums of each column are added in slice order.
constexpr int kNormDwSlices = 32;
__global__ void __launch_bounds__(32 * kNormDwSlices)
k_norm_dw(int ncta, int width, const float* __restrict__ part, float* __restrict__ dw) {
  __shared__ float sl_sum[kNormDwSlices][33];
  const int j = threadIdx.x & 31, sl = threadIdx.x >> 5;
  const int c = blockIdx.x * 32 + j;
  float t = 0.f;
  if (c < width)
    for (int b = sl; b < ncta; b += kNormDwSlices) t += part[(size_t)b * width + c];
  sl_sum[sl][j] = t;
  __syncthreads();
  if (sl == 0 && c < width) {
    float u = 0.f;
    for (int i = 0; i < kNormDwSlices; ++i) u += sl_sum[i][j];
    dw[c] = u;
  }
}

// threads per CTA and vectors per thread for a row of `width` elements of
// `esz` bytes (16-byte vectors; width / (16 / esz) is a multiple of 32)
void norm_shape(int width, int esz, int* threads, int* V) {
  const int nvec = width / (16 / esz);
  *threads = nvec < kNormThreads ? nvec : kNormThreads;
  *V = nvec / *threads;
}

template <typename KernelT>
int norm_grid(KernelT kernel, int threads, size_t smem, long long ngroups, int cap) {
  int dev = 0, nsm = 0, occ = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, smem);
  long long g = (long long)(nsm > 0 ? nsm : 1) * (occ > 0 ? occ : 1);
  if (g > cap) g = cap;
  if (g > ngroups) g = ngroups;
  return (int)(g < 1 ? 1 : g);
}

template <typename T, int V>
cudaError_t norm_fwd_t(long long rows, int width, int threads, const void* y, const void* z,
                       const float* w, float eps, void* out, float* inv_rms, cudaStream_t s) {
  const long long ngroups = (rows + 4 / V - 1) / (4 / V);
  const size_t smem = (size_t)2 * 4 * 2 * threads * 16;  // 2 stages x (R x V = 4) x (y, z)
  const int grid = norm_grid(k_norm_fwd<T, V>, threads, smem, ngroups, 1 << 20);
  k_norm_fwd<T, V><<<grid, threads, smem, s>>>(rows, width, eps, (const T*)y, (const T*)z, w,
                                               (T*)out, inv_rms);
  return cudaGetLastError();
}

template <typename T, int V>
cudaError_t norm_bwd_t(long long rows, int width, int threads, const void* y, const void* z,
                       const float* w, float eps, const float* inv_rms, const void* g, void* dy,
                       void* dz, float* part, int* ncta, cudaStream_t s) {
  constexpr int R = V < 2 ? 2 : 1;
  const long long ngroups = (rows + R - 1) / R;
  const size_t smem = (size_t)2 * R * V * 3 * threads * 16;  // 2 stages x R x V x (y, z, g)
  const int grid = norm_grid(k_norm_bwd<T, V>, threads, smem, ngroups, kNormMaxCtas);
  *ncta = grid;
  k_norm_bwd<T, V><<<grid, threads, smem, s>>>(rows, width, eps, (const T*)y, (const T*)z, w,
                                               inv_rms, (const T*)g, (T*)dy, (T*)dz, part);
  return cudaGetLastError();
}

}  // namespace

cudaError_t norm_forward(long long rows, int width, bool bf16, const void* y, const void* z,
                         const float* w, float eps, void* out, float* inv_rms, cudaStream_t s) {
  int threads = 0, V = 0;
  norm_shape(width, bf16 ? 2 : 4, &threads, &V);
  LaunchScope ls("rmsnorm_gated_fwd", s);
#define SSD_NORM_F(TT, VV) return norm_fwd_t<TT, VV>(rows, width, threads, y, z, w, eps, out, inv_rms, s)
  if (bf16) {  // width <= 4096: at most 2 vectors a thread
    if (V == 1) SSD_NORM_F(__nv_bfloat16, 1);
    SSD_NORM_F(__nv_bfloat16, 2);
  }
  if (V == 1) SSD_NORM_F(float, 1);
  if (V == 2) SSD_NORM_F(float, 2);
  SSD_NORM_F(float, 4);
#undef SSD_NORM_F
}

cudaError_t norm_backward(long long rows, int width, bool bf16, const void* y, const void* z,
                          const float* w, float eps, const float* inv_rms, const void* g, void* dy,
                          void* dz, float* dw, float* part, cudaStream_t s) {
  int threads = 0, V = 0, ncta = 1;
  norm_shape(width, bf16 ? 2 : 4, &threads, &V);
  cudaError_t e;
  {
    LaunchScope ls("rmsnorm_gated_bwd", s);
#define SSD_NORM_B(TT, VV) \
  e = norm_bwd_t<TT, VV>(rows, width, threads, y, z, w, eps, inv_rms, g, dy, dz, part, &ncta, s)
    if (bf16) {  // width <= 4096: at most 2 vectors a thread
      if (V == 1) SSD_NORM_B(__nv_bfloat16, 1);
      else SSD_NORM_B(__nv_bfloat16, 2);
    } else {
      if (V == 1) SSD_NORM_B(float, 1);
      else if (V == 2) SSD_NORM_B(float, 2);
      else SSD_NORM_B(float, 4);
    }
#undef SSD_NORM_B
  }
  if (e != cudaSuccess) return e;
  {
    LaunchScope ls("rmsnorm_gated_dw", s);
    k_norm_dw<<<(width + 31) / 32, 32 * kNormDwSlices, 0, s>>>(ncta, width, part, dw);
  }
  return cudaGetLastError();
}

}  // namespace ssd
