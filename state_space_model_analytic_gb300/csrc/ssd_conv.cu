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
// [B][C][K], dw [C][K], dbias [C] fp32.
//
// Work split.  A warp owns kConvCols = 128 channels (lane l: channels
// 4l..4l+3, one 8-byte bf16 / 16-byte fp32 shared-memory read per step, a
// warp reads one contiguous row) of one batch row over a run of consecutive
// steps; a CTA is a few warps (4 forward, kConvBwdWarps backward) with
// consecutive runs of the same channels and batch row.  The host splits each
// (channel block, batch row) column into gridDim.y * (warps per CTA)
// balanced runs, as many as the GPU holds at once (one wave), so every warp
// walks one run.
//
// Data movement.  Each warp has its own ring of stages in shared memory and
// its own mbarriers: lane 0 keeps the next stages in flight with 2D TMA
// boxes of 16 (forward) or 8 (backward) steps x 128 channels (x, and dout
// for the backward, viewed as [B*T][C]); no barrier spans warps.  The K - 1
// inputs before a run come from plain loads (or the initial state before
// step 0).
//
// Compute.  A thread keeps the last K inputs in registers and walks its run
// step by step, its 4 channels as two pairs in packed f32x2 arithmetic.  The
// backward walks on K - 1 steps past its run, keeping the K - 1 dx values
// still open and storing each once the gradient of the step K - 1 later is
// in (steps past T carry no gradient); dw and dbias stay in registers over
// the run, are summed over the CTA's warps in shared memory in order and
// over the CTAs along time in order by a last kernel.
//
// Waits on the TMA barriers are bounded: a wait that gives up sets a device
// error word; the warp then waits (bounded) for the copies it still has in
// flight and stops walking.
#include <cuda.h>
#include <cuda_bf16.h>

#include "f32x2.cuh"
#include "ssd_common.cuh"
#include "ssd_internal.h"
#include "tc_util.cuh"

namespace ssd {
namespace {

using namespace tc;

// forward: 4 warps a CTA, stages of 16 steps, 3 stages a warp; backward:
// kConvBwdWarps warps a CTA, stages of 8 steps, 2 stages a warp (measured
// best among 2-4 stages, 8-16 steps and 4-8 warps on the xBC workload)
constexpr int kConvFwdWarps = 4;
constexpr int kConvFwdStep = 16;
constexpr int kConvFwdStages = 3;
constexpr int kConvBwdStep = 8;
constexpr int kConvBwdStages = 2;
constexpr uint64_t kConvWaitNs = 1000000000ull;

__device__ unsigned int g_conv_error;

template <typename T>
struct ConvT;
template <>
struct ConvT<float> {
  // 4 channels from a shared-memory row at lane's offset
  __device__ static void lds(const uint8_t* row, int lane, float* v) {
    const float4 q = *(const float4*)(row + 16 * lane);
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  }
  __device__ static void ldg(const float* p, float* v) {
    const float4 q = *(const float4*)p;
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  }
  __device__ static void stg(float* p, const float* v) { *(float4*)p = make_float4(v[0], v[1], v[2], v[3]); }
};
template <>
struct ConvT<__nv_bfloat16> {
  __device__ static void cvt(uint2 q, float* v) {
    const float2 a = __bfloat1622float2(*(const __nv_bfloat162*)&q.x);
    const float2 b = __bfloat1622float2(*(const __nv_bfloat162*)&q.y);
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
  }
  __device__ static void lds(const uint8_t* row, int lane, float* v) {
    cvt(*(const uint2*)(row + 8 * lane), v);
  }
  __device__ static void ldg(const __nv_bfloat16* p, float* v) { cvt(*(const uint2*)p, v); }
  __device__ static void stg(__nv_bfloat16* p, const float* v) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
    const __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
    *(uint2*)p = make_uint2(*(const unsigned*)&a, *(const unsigned*)&b);
  }
};

// Shared-memory geometry: a stage of one tensor is (step) rows of 128
// elements; a warp's ring is S stages (of x, or of x and dout).
template <typename T, int K>
struct ConvGeom {
  static constexpr int ROWB = kConvCols * (int)sizeof(T);
  static constexpr int FTILE = kConvFwdStep * ROWB;
  static constexpr int BTILE = kConvBwdStep * ROWB;
  static constexpr int FWD_WARP = kConvFwdStages * FTILE;
  static constexpr int BWD_WARP = kConvBwdStages * 2 * BTILE;
  static constexpr size_t fwd_smem() { return (size_t)kConvFwdWarps * FWD_WARP + 1024; }
  static constexpr size_t bwd_smem() {
    const size_t ring = (size_t)kConvBwdWarps * BWD_WARP;
    const size_t red = (size_t)kConvBwdWarps * 32 * 4 * (K + 1) * sizeof(float);
    return (ring > red ? ring : red) + 1024;
  }
};

// logistic sigmoid 1 / (1 + 2^(-z log2 e)) from the hardware base-2
// exponential and reciprocal approximations (about 1e-6 relative for
// |z| < 80, and exact limits: 2^(+large) = inf gives 0, 2^(-large) = 0
// gives 1)
__device__ __forceinline__ float sig(float z) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(z * -1.4426950408889634f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + e));
  return r;
}

// input of step s for the thread's channels: x for s >= 0, else the initial
// state (zeros without one); zeros for channels past C
template <typename T, int K>
__device__ __forceinline__ void hist_load(const T* x, const float* init, long long rowb, int b, int C,
                                          int c0, bool valid, int s, float* v) {
  if (valid && s >= 0) {
    ConvT<T>::ldg(x + (rowb + s) * C + c0, v);
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      v[e] = (valid && init) ? init[((long long)b * C + c0 + e) * K + K + s] : 0.f;
  }
}

// per channel pair e: channels c0 + 2e, c0 + 2e + 1
template <int K>
__device__ __forceinline__ void load_params(const float* w, const float* bias, int c0, bool valid,
                                            float2 (&wv)[K][2], float2 (&bv)[2]) {
  auto at = [&](int c, int k) { return valid ? w[c * K + k] : 0.f; };
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int c = c0 + 2 * e;
    bv[e] = (valid && bias) ? make_float2(bias[c], bias[c + 1]) : make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < K; ++k) wv[k][e] = make_float2(at(c, k), at(c + 1, k));
  }
}

// The warp's balanced run of the column: [ws, we)
struct Run {
  int ws, we;
};
template <int WARPS>
__device__ __forceinline__ Run warp_run(int T_) {
  const int nr = gridDim.y * WARPS, r = blockIdx.y * WARPS + (threadIdx.x >> 5);
  return Run{(int)((long long)r * T_ / nr), (int)((long long)(r + 1) * T_ / nr)};
}

// After the wait for stage j gave up (uniform over the warp): flag it, and
// let lane 0 wait (bounded) for the copies it still has in flight: stages
// j .. min(ntiles, j + S) - 1 (stage j' + S is issued after stage j' is
// walked).
__device__ __forceinline__ void conv_abort(uint64_t* full, int stages, int j, int ntiles) {
  if ((threadIdx.x & 31) != 0) return;
  atomicOr(&g_conv_error, 1u);
  const int last = min(ntiles, j + stages) - 1;
  for (int i = j; i <= last; ++i) (void)mbar_wait(&full[i % stages], (i / stages) & 1, kConvWaitNs);
}

template <typename T, int K>
__global__ void __launch_bounds__(kConvFwdWarps * 32)
k_conv_fwd(const __grid_constant__ CUtensorMap xmap, int T_, int C, const T* __restrict__ x,
           const float* __restrict__ w, const float* __restrict__ bias,
           const float* __restrict__ init, T* __restrict__ out) {
  using G = ConvGeom<T, K>;
  constexpr int S = kConvFwdStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_all[kConvFwdWarps][S];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = align1024(smem_raw) + warp * G::FWD_WARP;
  uint64_t* full = full_all[warp];
  const int cs = blockIdx.x * kConvCols, c0 = cs + 4 * lane, b = blockIdx.z;
  const Run run = warp_run<kConvFwdWarps>(T_);
  const int ntiles = (run.we - run.ws + kConvFwdStep - 1) / kConvFwdStep;
  const long long rowb = (long long)b * T_;
  auto issue = [&](int j) {
    mbar_expect_tx(&full[j % S], G::FTILE);
    tma_load_2d(ring + (j % S) * G::FTILE, &xmap, cs, (int)(rowb + run.ws + j * kConvFwdStep),
                &full[j % S]);
  };
  if (lane == 0) {
    prefetch_tmap(&xmap);
    for (int i = 0; i < S; ++i) mbar_init(&full[i], 1);
    fence_mbar_init();
    for (int j = 0; j < min(S, ntiles); ++j) issue(j);
  }
  __syncwarp();
  const bool cvalid = c0 < C;
  float2 wv[K][2], bv[2], win[K][2];  // win[k] = input of step t - K + 1 + k (channel pairs)
  load_params<K>(w, bias, c0, cvalid, wv, bv);
#pragma unroll
  for (int k = 0; k < K - 1; ++k)
    hist_load<T, K>(x, init, rowb, b, C, c0, cvalid && ntiles > 0, run.ws - (K - 1) + k,
                    (float*)win[k]);
  T* op = out + (rowb + run.ws) * C + c0;
  for (int j = 0; j < ntiles; ++j) {
    const bool ok = mbar_wait(&full[j % S], (j / S) & 1, kConvWaitNs);
    if (!__all_sync(0xffffffffu, ok)) {
      conv_abort(full, S, j, ntiles);
      return;
    }
    const uint8_t* st = ring + (j % S) * G::FTILE;
    const int n = min(kConvFwdStep, run.we - run.ws - j * kConvFwdStep);
#pragma unroll
    for (int i = 0; i < kConvFwdStep; ++i) {
      ConvT<T>::lds(st + i * G::ROWB, lane, (float*)win[K - 1]);
      float2 o[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float2 p = bv[e];
#pragma unroll
        for (int k = 0; k < K; ++k) p = fma2(wv[k][e], win[k][e], p);
        o[e] = mul2(p, make_float2(sig(p.x), sig(p.y)));
      }
      if (cvalid && i < n) ConvT<T>::stg(op, (const float*)o);
      op += C;
#pragma unroll
      for (int k = 0; k < K - 1; ++k)
#pragma unroll
        for (int e = 0; e < 2; ++e) win[k][e] = win[k + 1][e];
    }
    __syncwarp();
    if (lane == 0 && j + S < ntiles) issue(j + S);
  }
}

// part: [B * gridDim.y][C][K + 1] (dw taps, then dbias) per CTA
template <typename T, int K>
__global__ void __launch_bounds__(kConvBwdWarps * 32)
k_conv_bwd(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap gmap,
           int T_, int C, const T* __restrict__ x, const float* __restrict__ w,
           const float* __restrict__ bias, const float* __restrict__ init, T* __restrict__ dx,
           float* __restrict__ part) {
  using G = ConvGeom<T, K>;
  constexpr int S = kConvBwdStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_all[kConvBwdWarps][S];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* base = align1024(smem_raw);
  uint8_t* ring = base + warp * G::BWD_WARP;
  uint64_t* full = full_all[warp];
  const int cs = blockIdx.x * kConvCols, c0 = cs + 4 * lane, b = blockIdx.z;
  const Run run = warp_run<kConvBwdWarps>(T_);
  // steps walked: the run and the K - 1 after it
  const int nwalk = run.we > run.ws ? run.we - run.ws + K - 1 : 0;
  const int ntiles = (nwalk + kConvBwdStep - 1) / kConvBwdStep;
  const long long rowb = (long long)b * T_;
  auto issue = [&](int j) {
    uint8_t* st = ring + (j % S) * 2 * G::BTILE;
    const int r = (int)(rowb + run.ws + j * kConvBwdStep);
    mbar_expect_tx(&full[j % S], 2 * G::BTILE);
    tma_load_2d(st, &xmap, cs, r, &full[j % S]);
    tma_load_2d(st + G::BTILE, &gmap, cs, r, &full[j % S]);
  };
  if (lane == 0) {
    prefetch_tmap(&xmap);
    prefetch_tmap(&gmap);
    for (int i = 0; i < S; ++i) mbar_init(&full[i], 1);
    fence_mbar_init();
    for (int j = 0; j < min(S, ntiles); ++j) issue(j);
  }
  __syncwarp();
  const bool cvalid = c0 < C;
  const float2 zero2 = make_float2(0.f, 0.f), one2 = make_float2(1.f, 1.f);
  float2 wv[K][2], bv[2];  // channel pairs
  load_params<K>(w, bias, c0, cvalid, wv, bv);
  float2 dw[K][2], db[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    db[e] = zero2;
#pragma unroll
    for (int k = 0; k < K; ++k) dw[k][e] = zero2;
  }
  float2 xw[K][2];  // xw[k] = input of step s - K + 1 + k
#pragma unroll
  for (int k = 0; k < K - 1; ++k)
    hist_load<T, K>(x, init, rowb, b, C, c0, cvalid && ntiles > 0, run.ws - (K - 1) + k,
                    (float*)xw[k]);
  // open[k]: dx of step s - K + 1 + k summed over the gradients of steps < s
  float2 open[K > 1 ? K - 1 : 1][2];
#pragma unroll
  for (int k = 0; k < K - 1; ++k)
#pragma unroll
    for (int e = 0; e < 2; ++e) open[k][e] = zero2;
  T* dp = dx + (rowb + run.ws) * C + c0;  // dx of the next step to complete
  for (int j = 0; j < ntiles; ++j) {
    const bool ok = mbar_wait(&full[j % S], (j / S) & 1, kConvWaitNs);
    if (!__all_sync(0xffffffffu, ok)) {
      conv_abort(full, S, j, ntiles);
      break;
    }
    const uint8_t* xs = ring + (j % S) * 2 * G::BTILE;
    const uint8_t* gs = xs + G::BTILE;
#pragma unroll
    for (int i = 0; i < kConvBwdStep; ++i) {
      const int s = run.ws + j * kConvBwdStep + i;
      float2 d[2], o[2];
      ConvT<T>::lds(xs + i * G::ROWB, lane, (float*)xw[K - 1]);
      ConvT<T>::lds(gs + i * G::ROWB, lane, (float*)d);
      const bool in_seq = s < T_, owned = s < run.we;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float2 p = bv[e];
#pragma unroll
        for (int k = 0; k < K; ++k) p = fma2(wv[k][e], xw[k][e], p);
        const float2 sg = make_float2(sig(p.x), sig(p.y));
        // g = d sg (1 + p (1 - sg))
        const float2 oms = fma2(sg, make_float2(-1.f, -1.f), one2);
        const float2 g = in_seq ? mul2(mul2(d[e], sg), fma2(p, oms, one2)) : zero2;
        if (owned) {
          db[e] = add2(db[e], g);
#pragma unroll
          for (int k = 0; k < K; ++k) dw[k][e] = fma2(g, xw[k][e], dw[k][e]);
        }
        // this step's gradient reaches dx of steps s - K + 1 .. s through taps 0 .. K - 1
        if (K > 1) {
          o[e] = fma2(g, wv[0][e], open[0][e]);
#pragma unroll
          for (int k = 0; k + 1 < K - 1; ++k) open[k][e] = fma2(g, wv[k + 1][e], open[k + 1][e]);
          open[K > 1 ? K - 2 : 0][e] = mul2(g, wv[K - 1][e]);
        } else {
          o[e] = mul2(g, wv[0][e]);
        }
      }
      const int sd = s - (K - 1);  // dx of step sd is complete
      if (sd >= run.ws && sd < run.we) {
        if (cvalid) ConvT<T>::stg(dp, (const float*)o);
        dp += C;
      }
#pragma unroll
      for (int k = 0; k < K - 1; ++k)
#pragma unroll
        for (int e = 0; e < 2; ++e) xw[k][e] = xw[k + 1][e];
    }
    __syncwarp();
    if (lane == 0 && j + S < ntiles) issue(j + S);
  }
  // the CTA's warps summed in order (warp 0 first), per channel and tap; every
  // warp is past its ring (all copies waited for, or given up on and flagged)
  __syncthreads();
  float* red = (float*)base;
  float* mine = red + (size_t)threadIdx.x * 4 * (K + 1);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int pe = e >> 1;
#pragma unroll
    for (int k = 0; k < K; ++k) mine[e * (K + 1) + k] = (e & 1) ? dw[k][pe].y : dw[k][pe].x;
    mine[e * (K + 1) + K] = (e & 1) ? db[pe].y : db[pe].x;
  }
  __syncthreads();
  constexpr int n = 32 * 4 * (K + 1);  // one warp's channels x (taps + bias)
  float* pr = part + ((size_t)(b * gridDim.y + blockIdx.y) * C + cs) * (K + 1);
  for (int i = threadIdx.x; i < n; i += kConvBwdWarps * 32) {
    if (cs + i / (K + 1) >= C) continue;
    float t = 0.f;
    for (int wi = 0; wi < kConvBwdWarps; ++wi) t += red[wi * n + i];
    pr[i] = t;
  }
}

// dw, dbias: the per-CTA partials summed along time in order
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

template <typename T>
bool conv_map(CUtensorMap* m, const void* base, long long rows, int C, int box_rows) {
  return encode_rows_2d(m, base, sizeof(T) == 2, (uint64_t)rows, (uint64_t)C, kConvCols,
                        (uint32_t)box_rows);
}

// CTAs per (channel block, batch row) column: as many as fill the GPU once
// (from the kernel's occupancy), at most conv_max_ctas_per_column(T) (runs
// of about kConvMinRun steps or more with kConvBwdWarps warps a CTA) and at
// least 1.
template <typename KernelT>
cudaError_t conv_ctas_per_column(KernelT kernel, int threads, size_t smem, long long cols, int T_,
                                 int* out) {
  int dev = 0, nsm = 0, occ = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, smem);
  if (e != cudaSuccess) return e;
  long long cpc = (long long)nsm * occ / cols;
  const long long cap = conv_max_ctas_per_column(T_);
  if (cpc > cap) cpc = cap;
  *out = cpc < 1 ? 1 : (int)cpc;
  return cudaSuccess;
}

template <typename T, int K>
cudaError_t conv_fwd_t(long long B, int T_, int C, const void* x, const float* w,
                       const float* bias, const float* init, void* out, cudaStream_t s) {
  using G = ConvGeom<T, K>;
  CUtensorMap xm;
  if (!conv_map<T>(&xm, x, B * T_, C, kConvFwdStep)) return cudaErrorInvalidValue;
  const size_t smem = G::fwd_smem();
  const long long stripes = (C + kConvCols - 1) / kConvCols;
  int cpc = 1;
  cudaError_t e = conv_ctas_per_column(k_conv_fwd<T, K>, kConvFwdWarps * 32, smem, stripes * B, T_,
                                       &cpc);
  if (e != cudaSuccess) return e;
  k_conv_fwd<T, K><<<dim3((unsigned)stripes, (unsigned)cpc, (unsigned)B), kConvFwdWarps * 32, smem,
                     s>>>(
      xm, T_, C, (const T*)x, w, bias, init, (T*)out);
  return cudaGetLastError();
}

template <typename T, int K>
cudaError_t conv_bwd_t(long long B, int T_, int C, const void* x, const float* w,
                       const float* bias, const float* init, const void* dout, void* dx,
                       float* part, int* nparts, cudaStream_t s) {
  using G = ConvGeom<T, K>;
  CUtensorMap xm, gm;
  if (!conv_map<T>(&xm, x, B * T_, C, kConvBwdStep) ||
      !conv_map<T>(&gm, dout, B * T_, C, kConvBwdStep))
    return cudaErrorInvalidValue;
  const size_t smem = G::bwd_smem();
  const long long stripes = (C + kConvCols - 1) / kConvCols;
  int cpc = 1;
  cudaError_t e = conv_ctas_per_column(k_conv_bwd<T, K>, kConvBwdWarps * 32, smem, stripes * B, T_,
                                       &cpc);
  if (e != cudaSuccess) return e;
  *nparts = (int)(B * cpc);
  k_conv_bwd<T, K><<<dim3((unsigned)stripes, (unsigned)cpc, (unsigned)B), kConvBwdWarps * 32, smem,
                     s>>>(
      xm, gm, T_, C, (const T*)x, w, bias, init, (T*)dx, part);
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
  int nparts = 1;
  {
    LaunchScope ls("conv1d_silu_bwd", s);
#define SSD_CONV_B(TT, KK) e = conv_bwd_t<TT, KK>(B, T_, C, x, w, bias, init, dout, dx, part, &nparts, s)
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
  {
    LaunchScope ls("conv1d_silu_dw", s);
    k_conv_dw<<<(C * (K + 1) + 255) / 256, 256, 0, s>>>(nparts, C, K, part, dw, dbias);
  }
  return cudaGetLastError();
}

cudaError_t conv_read_and_clear_error(unsigned int* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_conv_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_conv_error, &zero, sizeof(unsigned int));
}

}  // namespace ssd
