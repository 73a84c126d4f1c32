// Tensor-core (tcgen05 / TMEM / TMA) kernels of the chunked SSD core.
//
// Scope: bf16 storage, headdim P = 64, d_state N = 128, chunk Q in {128, 256}.
// A chunk is processed as Q/128 blocks of 128 rows (the MMA M size).  Inside a
// chunk the second block reaches the first through the mid-chunk state
//     H_mid = exp(cs_127) H_{c-1} + S_0,
//     S_0   = sum_{j<128} exp(cs_127 - cs_j) dt_j x_j B_j^T,
// which is exact in real arithmetic (it is the recurrence of
// `ssd_forward_state_history_reference`, burn_dragon_kernel 0.5.0,
// src/sequence/mamba2/backward.rs, unrolled over 128 steps) and replaces the
// off-diagonal 128 x 128 block of the quadratic form by two rank-N products.
//
// Decay masks.  For a 128-row block, warp w owns rows r..r+31, r = 32 w.  For
// a column j < r (a 32-column chunk left of the warp's diagonal chunk)
//     exp(cs_i - cs_j) = exp(cs_i - cs_r) * exp(cs_r - cs_j),
// both factors <= 1 because cs is non-increasing (dt >= 0, A <= 0), so no
// factor overflows and an underflowed factor means the product underflows.
// The column factors are a per-warp table in shared memory; only the 32 x 32
// diagonal chunk evaluates one exp per element, with the exponent set to
// -inf above the diagonal before exp.
#include <cuda.h>
#include <cuda_bf16.h>

#include <climits>
#include <cstdlib>
#include <mutex>

#include "ssd_common.cuh"
#include "ssd_internal.h"
#include "tc_util.cuh"

namespace ssd {

using namespace tc;

namespace {

constexpr int kTcThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;
// Wall time (ns) an mbarrier wait may take before the kernel gives up and
// records a timeout.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// ---------------------------------------------------------------------------
// Device error word: a bounded wait that gives up sets it; the host reads it
// only through the test hooks.  Kernels finish (no trap) after a timeout.
__device__ unsigned int g_tc_error;

// Every thread of the CTA waits; the outcome is made uniform across the CTA
// (so a timeout never splits the threads at a later barrier).
__device__ __forceinline__ bool wait_or_flag(uint64_t* bar, uint32_t parity) {
  const bool mine = mbar_wait(bar, parity, kWaitLimitNs);
  const bool all = __syncthreads_and(mine) != 0;
  if (!all && threadIdx.x == 0) atomicOr(&g_tc_error, 1u);
  return all;
}

struct TcDims {
  int B, T, H, P, N, G, Q, nc, hpg;
  // raw-dt mode (both set): the dt argument holds dt_raw and the kernels use
  // dt = softplus(dt_raw + dt_bias[h]) and A = -exp(a_log[h]); else nullptr
  const float* dt_bias;
  const float* a_log;
};

// softplus(z) = log(1 + e^z), evaluated as max(z, 0) + log1p(e^{-|z|}) (no overflow)
__device__ __forceinline__ float softplus_tc(float z) {
  return fmaxf(z, 0.f) + log1pf(expf(-fabsf(z)));
}
// dt of one element from the value stored in the dt argument (kRaw: the
// kernel instantiation of the raw-dt mode, so the plain kernels carry none of
// its code)
template <bool kRaw>
__device__ __forceinline__ float dt_of(const TcDims& d, float stored, int h) {
  if (!kRaw) return stored;
  return softplus_tc(stored + d.dt_bias[h]);
}
// A of head h
template <bool kRaw>
__device__ __forceinline__ float a_of(const TcDims& d, const float* __restrict__ A, int h) {
  if (!kRaw) return A[h];
  return -expf(d.a_log[h]);
}

// Column sums over the 32 lanes of a warp, for 16 columns: lane l returns the
// sum over all lanes of v[l % 16].
__device__ __forceinline__ float warp_column_sum16(float (&v)[16]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int s = 8; s >= 1; s >>= 1) {
    const bool upper = (lane & s) != 0;
#pragma unroll
    for (int k = 0; k < s; ++k) {
      const float send = upper ? v[k] : v[k + s];
      const float keep = upper ? v[k + s] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, s);
    }
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 16);
}

__device__ __forceinline__ void store_row_bf16(uint8_t* tile, int row, int chunk0,
                                               const float* v8) {
  uint4 o;
  o.x = pack_bf16(v8[0], v8[1]);
  o.y = pack_bf16(v8[2], v8[3]);
  o.z = pack_bf16(v8[4], v8[5]);
  o.w = pack_bf16(v8[6], v8[7]);
  *(uint4*)(tile + sw128(row, chunk0)) = o;
}

__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
  const __nv_bfloat162* p = (const __nv_bfloat162*)&v;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float2 x = __bfloat1622float2(p[t]);
    f[2 * t] = x.x;
    f[2 * t + 1] = x.y;
  }
}

// Scale the 16-byte chunks e = first, first + step, ... of a SW128 bf16 tile
// (rows of 8 chunks) by a per-row factor.
template <typename F>
__device__ __forceinline__ void scale_tile_rows(uint8_t* tile, int nchunks, F&& factor) {
  for (int e = threadIdx.x; e < nchunks; e += blockDim.x) {
    const float s = factor(e >> 3);
    float f[8];
    unpack8(*(const uint4*)(tile + e * 16), f);
#pragma unroll
    for (int t = 0; t < 8; ++t) f[t] *= s;
    uint4 o;
    o.x = pack_bf16(f[0], f[1]);
    o.y = pack_bf16(f[2], f[3]);
    o.z = pack_bf16(f[4], f[5]);
    o.w = pack_bf16(f[6], f[7]);
    *(uint4*)(tile + e * 16) = o;
  }
}

// dt of step `tid` of chunk c, head h (0 past the chunk), for 256 threads.
template <bool kRaw = false>
__device__ __forceinline__ float load_dt_256(const TcDims& d, const float* __restrict__ dt, int b,
                                             int c, int h) {
  const int tid = threadIdx.x;
  return tid < d.Q ? dt_of<kRaw>(d, dt[((size_t)b * d.T + (size_t)c * d.Q + tid) * d.H + h], h)
                    : 0.f;
}

// Chunk-local inclusive cumsum (log2 units) with 256 threads, one value each.
template <bool kRaw = false>
__device__ __forceinline__ void chunk_cumsum_256(const TcDims& d, const float* __restrict__ dt,
                                                 const float* __restrict__ A, int b, int c, int h,
                                                 float* s_cs2, float* s_dt, float* scratch) {
  const int tid = threadIdx.x;
  const float dv = load_dt_256<kRaw>(d, dt, b, c, h);
  const float cs = block_inclusive_scan(dv * (a_of<kRaw>(d, A, h) * kLog2e), scratch);
  if (tid < d.Q) {
    s_cs2[tid] = cs;
    s_dt[tid] = dv;
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Chunk outer product on tensor cores: out[b][c][h] (P x N, fp32) =
//   MODE 0: sum_j exp(cs_last - cs_j) dt_j x_j B_j^T   (chunk state S_c)
//   MODE 1: sum_j exp(cs_j) dy_j C_j^T                 (chunk dstate R_c)
// computed transposed, D[n][p] = V^T (w o U), M = N = 128 rows (n), N = P = 64.
struct OuterMaps {
  CUtensorMap u;  // x or dy: [B*T][H*P] bf16, box {64, Q}
  CUtensorMap v;  // B or C:  [B*T][G*N] bf16, box {64, Q}
  CUtensorMap o;  // output [B*nc*H*P][N] fp32, box {32, 64} (store)
};

template <int MODE>
__global__ void __launch_bounds__(256)
k_chunk_outer_tc(const __grid_constant__ OuterMaps maps, TcDims d, const float* __restrict__ dt,
                 const float* __restrict__ A, float* __restrict__ out,
                 float* __restrict__ cs_last) {
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  const int Q = d.Q;
  uint8_t* sV = sm;                      // 2 MN blocks of [Q rows][128 B]
  uint8_t* sU = sm + 2 * Q * 128;        // [Q rows][128 B]
  __shared__ float s_cs2[256], s_dt[256], s_w[256], scratch[8];
  __shared__ uint64_t bar_load, bar_mma;
  __shared__ uint32_t tmem_base;
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = h / d.hpg, tid = threadIdx.x, wg = tid >> 7, q = (tid >> 5) & 3;
  const int row0 = b * d.T + c * Q;

  if (tid == 0) {
    prefetch_tmap(&maps.u);
    prefetch_tmap(&maps.v);
    mbar_init(&bar_load, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
  }
  if (tid < 32) {
    tmem_alloc(&tmem_base, 64);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tm = tmem_base;
  if (tid == 0) {
    mbar_expect_tx(&bar_load, (uint32_t)(3 * Q * 128));
    tma_load_2d(sV, &maps.v, g * d.N, row0, &bar_load);
    tma_load_2d(sV + Q * 128, &maps.v, g * d.N + 64, row0, &bar_load);
    tma_load_2d(sU, &maps.u, h * d.P, row0, &bar_load);
  }
  chunk_cumsum_256(d, dt, A, b, c, h, s_cs2, s_dt, scratch);
  const float last2 = s_cs2[Q - 1];
  if (tid < Q) s_w[tid] = (MODE == 0) ? exp2f(last2 - s_cs2[tid]) * s_dt[tid] : exp2f(s_cs2[tid]);
  if (tid == 0) cs_last[((size_t)b * d.H + h) * d.nc + c] = last2 * (1.0f / kLog2e);
  const bool loaded = wait_or_flag(&bar_load, 0);  // also publishes s_w
  if (loaded) scale_tile_rows(sU, Q * 8, [&](int r) { return s_w[r]; });
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (tid == 0 && loaded) {
    const uint32_t idesc = idesc_bf16(128, 64, true, true);
    for (int ks = 0; ks < Q / 16; ++ks) {
      const uint64_t ad = desc_sw128(smem_u32(sV) + ks * 2048, Q * 128, 1024);
      const uint64_t bd = desc_sw128(smem_u32(sU) + ks * 2048, Q * 128, 1024);
      mma_bf16(tm, ad, bd, idesc, ks > 0);
    }
    mma_commit(&bar_mma);
  }
  const bool done = loaded && wait_or_flag(&bar_mma, 0);
  fence_after_sync();
  if (done) {
    // thread (wg, n): columns p in [32 wg, 32 wg + 32) of row n of D = out^T,
    // written as out[p][n] into four SW128 fp32 staging boxes [64 p][32 n]
    // (the dead operand tiles), then stored by TMA
    const int n = tid & 127, box = n >> 5, cc = (n & 31) >> 2, w4 = n & 3;
    float v[32];
    tmem_ld32(tm + ((uint32_t)(q * 32) << 16) + wg * 32, v);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int pp = wg * 32 + i;
      *(float*)(sV + box * 8192 + pp * 128 + ((cc ^ (pp & 7)) << 4) + w4 * 4) = v[i];
    }
    fence_async_smem();
  }
  __syncthreads();
  if (tid == 0 && done) {
    const int srow = ((b * d.nc + c) * d.H + h) * d.P;
    for (int k = 0; k < 4; ++k) tma_store_2d(&maps.o, sV + k * 8192, 32 * k, srow);
    bulk_commit();
    bulk_wait0();
  }
  fence_before_sync();
  __syncthreads();
  if (tid < 32) tmem_dealloc(tm, 64);
}

// ---------------------------------------------------------------------------
// Fused chunk-state + state pass, one CTA per (b, h), warp-specialised.
// Warp 8 (issuer) streams the chunks' tiles in by TMA (two stages) and issues
// the product D[n][p] = V^T (w o U) of each chunk on tcgen05 into one of
// kScanBufs TMEM buffers of 64 columns.  Warps 4-7 (scalers) build each
// chunk's decay tables and scale the rows of U by w in shared memory (MODE 1:
// they also convert the fp32 history into bf16 rows).  Warps 0-3 (consumer)
// hold the running state, thread n owning row n (64 p values): per chunk they wait for
// the product, read it out of TMEM, free the buffer and advance the
// recurrence, so the products of later chunks overlap the recurrence and the
// state writes of earlier ones.  The bf16 rows go out through a 128-byte
// swizzled shared-memory tile and a TMA store (one coalesced 16 KB block per
// (b, chunk, h)).
// MODE 0 (forward, chunks in order):
//   S_c^T = B_c^T (w o X_c), w_j = exp(cs_last - cs_j) dt_j;
//   hist[c] = H_{c-1} (fp32) and its bf16 copy as rows n (hT);
//   H_c = exp(cs_last) H_{c-1} + S_c;  final = H_{nc-1}.
// MODE 1 (backward, chunks in reverse):
//   R_c^T = C_c^T (e o dY_c), e_i = exp(cs_i);
//   gT[c] = g_c and hT[c] = H_{c-1} from hist, both bf16 rows n;
//   g_{c-1} = exp(cs_last) g_c + R_c;  dh0 = g_{-1}.
//   With gmid, chunks of 256 steps go through their middle: the product is
//   taken in two halves, R_1^T over rows i >= 128 with e_i = exp(cs_i -
//   cs_127) and R_0^T over rows i < 128 with e_i = exp(cs_i), and
//   g_mid = exp(cs_255 - cs_127) g_c + R_1 (bf16 rows n, rows3 map),
//   g_{c-1} = exp(cs_127) g_mid + R_0.
struct ScanStateMaps {
  CUtensorMap u;     // x or dy: [B*T][H*P] bf16, box {64, Q}
  CUtensorMap v;     // B or C:  [B*T][G*N] bf16, box {64, Q}
  CUtensorMap rows;  // hT (MODE 0) or gT (MODE 1): [B*nc*H*N][P] bf16, box {64, 128} (store)
  CUtensorMap rows2; // hT (MODE 1), same layout (store)
  CUtensorMap rows3; // g_mid rows (MODE 1, chunks of 256), same layout (store)
};

constexpr int kScanBufs = 4;  // TMEM product buffers (64 columns each; 128 when split in halves)

__device__ __forceinline__ void named_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Barrier over `nthreads` threads that also returns the OR of `pred` over them.
__device__ __forceinline__ bool named_sync_or(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// Bounded wait that also gives up as soon as another warp of the CTA has
// recorded a timeout in *abort (then the caller stops touching guarded data).
__device__ __forceinline__ bool wait_ws(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      atomicOr(&g_tc_error, 1u);
      return false;
    }
  }
}

constexpr int kScanThreads = 288;  // consumer warps 0-3, scaler warps 4-7, issuer warp 8

template <int MODE, bool kRaw>
__global__ void __launch_bounds__(kScanThreads, 1)
k_state_scan_tc(const __grid_constant__ ScanStateMaps maps, TcDims d, const float* __restrict__ dt,
                const float* __restrict__ A, const float* __restrict__ h0,
                float* __restrict__ hist, float* __restrict__ final_or_dh0,
                unsigned int* __restrict__ tickets, int ntickets, int gmid) {
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  const int Q = d.Q;
  const uint32_t stage_bytes = 3u * Q * 128;  // V: 2 MN blocks of [Q][128 B]; U: [Q][128 B]
  __shared__ float s_wsum[2][4], s_lastq[4], s_last[kScanBufs], s_midq[4], s_mid[kScanBufs];
  __shared__ uint64_t bar_load[2], bar_sfree[2], bar_scaled[2], bar_full[kScanBufs],
      bar_free[kScanBufs];
  __shared__ uint32_t tmem_base;
  __shared__ volatile int s_abort;
  const int h = blockIdx.x, b = blockIdx.y;
  const int g = h / d.hpg, tid = threadIdx.x;
  const int nc = d.nc;
  const size_t PN = (size_t)d.P * d.N;
  auto chunk_of = [&](int it) { return MODE == 0 ? it : nc - 1 - it; };
  // MODE 1 at 256 steps: the product in two halves (columns [0, 64): rows
  // 128-255, [64, 128): rows 0-127 of the chunk) and g_mid on the way
  const bool split = MODE == 1 && Q == 256 && gmid;
  const uint32_t buf_cols = split ? 128 : 64;

  if (tid == 0) {
    prefetch_tmap(&maps.u);
    prefetch_tmap(&maps.v);
    for (int k = 0; k < 2; ++k) {
      mbar_init(&bar_load[k], 1);
      mbar_init(&bar_sfree[k], 1);
      mbar_init(&bar_scaled[k], 4);  // one arrive per scaler warp
    }
    for (int k = 0; k < kScanBufs; ++k) {
      mbar_init(&bar_full[k], 2);   // the product's commit + the issuer's table arrive
      mbar_init(&bar_free[k], 4);   // one arrive per consumer warp
    }
    s_abort = 0;
    fence_mbar_init();
  }
  if (tid < 32) {
    tmem_alloc(&tmem_base, buf_cols * kScanBufs);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tm = tmem_base;

  if (tid >= 256) {
    // ===================== issuer (warp 8) =====================
    if (tid == 256) {
      auto issue = [&](int it) {
        const int c = chunk_of(it), k = it & 1;
        uint8_t* st = sm + k * stage_bytes;
        const int row0 = b * d.T + c * Q;
        mbar_expect_tx(&bar_load[k], stage_bytes);
        tma_load_2d(st, &maps.v, g * d.N, row0, &bar_load[k]);
        tma_load_2d(st + Q * 128, &maps.v, g * d.N + 64, row0, &bar_load[k]);
        tma_load_2d(st + 2 * Q * 128, &maps.u, h * d.P, row0, &bar_load[k]);
      };
      // the first tiles are inputs that no kernel of this library writes: they
      // are fetched before waiting for the kernel launched ahead of this one
      issue(0);
      if (nc > 1) issue(1);
      grid_dep_wait();
      int loads_issued = nc > 1 ? 2 : 1, mma_issued = 0;
      const uint32_t idesc = idesc_bf16(128, 64, true, true);
      for (int it = 0; it < nc; ++it) {
        const int k = it & 1, buf = it % kScanBufs;
        // chunk it scaled; its decay total; the buffer's previous product read out
        if (!wait_ws(&bar_scaled[k], (it >> 1) & 1, &s_abort)) break;
        const float last2 = s_lastq[it & 3], mid2 = s_midq[it & 3];
        if (it >= kScanBufs && !wait_ws(&bar_free[buf], ((it / kScanBufs) - 1) & 1, &s_abort)) break;
        s_last[buf] = last2;
        s_mid[buf] = mid2;
        mbar_arrive(&bar_full[buf]);
        fence_after_sync();
        uint8_t* sV = sm + k * stage_bytes;
        uint8_t* sU = sV + 2 * Q * 128;
        const uint32_t tb = tm + buf_cols * buf;
        for (int ks = 0; ks < Q / 16; ++ks) {
          // split: K-steps 8-15 (rows 128-255) into columns [0, 64), 0-7 into [64, 128)
          const bool hi = ks >= 8;
          mma_bf16(split && !hi ? tb + 64 : tb, desc_sw128(smem_u32(sV) + ks * 2048, Q * 128, 1024),
                   desc_sw128(smem_u32(sU) + ks * 2048, Q * 128, 1024), idesc,
                   split ? (ks & 7) > 0 : ks > 0);
        }
        mma_commit(&bar_full[buf]);
        mma_commit(&bar_sfree[k]);
        ++mma_issued;
        // stage k takes chunk it + 2 once this product has read it
        if (it + 2 < nc) {
          if (!wait_ws(&bar_sfree[k], (it >> 1) & 1, &s_abort)) break;
          issue(it + 2);
          ++loads_issued;
        }
      }
      // drain: no TMA write or product may still be in flight when the CTA ends
      // (bounded waits; in the normal case all have completed already)
      for (int i = mma_issued; i < loads_issued; ++i)
        (void)mbar_wait(&bar_load[i & 1], (i >> 1) & 1, kWaitLimitNs);
      if (mma_issued > 0)
        (void)mbar_wait(&bar_sfree[(mma_issued - 1) & 1], ((mma_issued - 1) >> 1) & 1, kWaitLimitNs);
    }
    if (tid != 256) grid_dep_wait();
    __syncwarp();
  } else if (tid >= 128) {
    // ===================== scalers (warps 4-7) =====================
    grid_dep_wait();
    // MODE 1: the backward kernel that follows counts its finished CTAs and
    // unit segments here
    if (tickets)
      for (int i = (b * (int)gridDim.x + h) * 128 + (tid - 128); i < ntickets;
           i += (int)(gridDim.x * gridDim.y) * 128)
        tickets[i] = 0u;
    const int pt = tid - 128, lane = tid & 31, pw = pt >> 5;
    const float a2 = a_of<kRaw>(d, A, h) * kLog2e;
    const int per = Q / 128;  // dt values per thread: 1 or 2, consecutive
    auto load_dt = [&](int it, float (&v)[2]) {
      const size_t t0 = (size_t)b * d.T + (size_t)chunk_of(it) * Q + (size_t)pt * per;
      v[0] = dt[t0 * d.H + h];
      v[1] = per == 2 ? dt[(t0 + 1) * d.H + h] : 0.f;
    };
    float dv[2], dv_next[2] = {0.f, 0.f};
    load_dt(0, dv);
    if (nc > 1) load_dt(1, dv_next);
    for (int it = 0; it < nc; ++it) {
      const int k = it & 1;
      // the stored values were fetched ahead; raw-dt mode: dt = softplus(...)
      if (kRaw) {
        dv[0] = dt_of<kRaw>(d, dv[0], h);
        dv[1] = per == 2 ? dt_of<kRaw>(d, dv[1], h) : 0.f;
      }
      // ---- decay tables: chunk-local inclusive cumsum of dt * A (log2 units)
      const float x0 = dv[0] * a2, x1 = dv[1] * a2;
      float run = x0 + x1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, run, o);
        if (lane >= o) run += t;
      }
      if (lane == 31) s_wsum[k][pw] = run;
      named_sync(1, 128);
      float base = 0.f, last2 = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float ws = s_wsum[k][w];
        if (w < pw) base += ws;
        last2 += ws;
      }
      const float cs0 = base + run - x1;  // cs of this thread's first value
      const float cs1 = base + run;       // and of its second
      // weights of this thread's rows pt * per + {0, 1}; split: rows from 128
      // on (threads 64-127) relative to cs_127, the end of warps 0-1's rows
      const float mid2 = split ? s_wsum[k][0] + s_wsum[k][1] : 0.f;
      const float ref = split && pt >= 64 ? mid2 : 0.f;
      const float w0 = MODE == 0 ? exp2f(last2 - cs0) * dv[0] : exp2f(cs0 - ref);
      const float w1 = MODE == 0 ? exp2f(last2 - cs1) * dv[1] : exp2f(cs1 - ref);
      if (pt == 0) {
        s_lastq[it & 3] = last2;
        s_midq[it & 3] = mid2;
      }
      dv[0] = dv_next[0];
      dv[1] = dv_next[1];
      if (it + 2 < nc) load_dt(it + 2, dv_next);
      // ---- this chunk's tiles; U rows times w (bf16 pairs).  The barrier
      // makes the decision to stop uniform over the scalers.
      const bool got = wait_ws(&bar_load[k], (it >> 1) & 1, &s_abort);
      if (named_sync_or(1, 128, !got || s_abort)) break;
      uint8_t* sU = sm + k * stage_bytes + 2 * Q * 128;
      for (int rr = 0; rr < per; ++rr) {
        // a whole 128-byte row has one factor, so the swizzle does not matter;
        // the lane-rotated chunk order keeps the accesses bank-conflict free
        uint8_t* row = sU + (pt * per + rr) * 128;
        const __nv_bfloat162 w2 = __float2bfloat162_rn(rr ? w1 : w0);
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = *(const uint4*)(row + 16 * ((j + lane) & 7));
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          __nv_bfloat162* hv2 = (__nv_bfloat162*)&v[j];
#pragma unroll
          for (int t = 0; t < 4; ++t) hv2[t] = __hmul2(hv2[t], w2);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) *(uint4*)(row + 16 * ((j + lane) & 7)) = v[j];
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_scaled[k]);  // s_lastq too (release)
      if (MODE == 1) {
        // hT[c] = H_{c-1} as bf16 rows n, off the consumers' path: this
        // thread's share of the fp32 history (p in [16 pw, 16 pw + 16) of
        // rows n = 4 lane .. 4 lane + 3, 16-byte loads coalesced over the
        // lanes), loaded only now: the proxy fence before the arrive above
        // would otherwise wait for these loads
        const int c = chunk_of(it);
        float4 hv[16];
        {
          const float* hsrc = hist + (((size_t)b * nc + c) * d.H + h) * PN +
                              (size_t)(16 * pw) * d.N + 4 * lane;
#pragma unroll
          for (int pp = 0; pp < 16; ++pp) hv[pp] = *(const float4*)(hsrc + (size_t)pp * d.N);
        }
        uint8_t* sRows2 = sm + 2 * stage_bytes + 16384;  // [128 rows n][64 p] bf16, SW128
        if (pt == 0) bulk_wait_read0();  // the previous store of sRows2 has read it
        named_sync(1, 128);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float v8[8];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const float4 f = hv[8 * half + t];
              v8[t] = i == 0 ? f.x : i == 1 ? f.y : i == 2 ? f.z : f.w;
            }
            store_row_bf16(sRows2, 4 * lane + i, 2 * pw + half, v8);
          }
        }
        fence_async_smem();
        named_sync(1, 128);
        if (pt == 0) {
          tma_store_2d(&maps.rows2, sRows2, 0, ((b * nc + c) * d.H + h) * d.N);
          bulk_commit();
        }
      }
    }
    if (pt == 0) bulk_wait0();
  } else {
    // ===================== consumer (warps 0-3) =====================
    grid_dep_wait();
    const int n = tid, q = tid >> 5;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    uint8_t* sRows = sm + 2 * stage_bytes;  // [128 rows n][64 p] bf16, SW128
    if (tid == 0) prefetch_tmap(&maps.rows);
    // 64 values of row n as bf16 into the staging tile, then one TMA store of
    // the tile to rows [srow, srow + 128) (the tile is free again once the
    // previous store has read it)
    auto put_rows = [&](const float (&v)[64], const CUtensorMap* map, int srow) {
      if (tid == 0) bulk_wait_read0();
      named_sync(2, 128);
#pragma unroll
      for (int j = 0; j < 8; ++j) store_row_bf16(sRows, n, j, &v[8 * j]);
      fence_async_smem();
      named_sync(2, 128);
      if (tid == 0) {
        tma_store_2d(map, sRows, 0, srow);
        bulk_commit();
      }
    };
    float st[64];
    if (MODE == 0 && h0) {
      const float* src = h0 + ((size_t)b * d.H + h) * PN + n;
#pragma unroll
      for (int p = 0; p < 64; ++p) st[p] = src[(size_t)p * d.N];
    } else {
#pragma unroll
      for (int p = 0; p < 64; ++p) st[p] = 0.f;
    }
    bool ok = true;
    for (int it = 0; it < nc; ++it) {
      const int c = chunk_of(it), buf = it % kScanBufs;
      const int srow = ((b * nc + c) * d.H + h) * d.N;
      if (MODE == 0) {  // hist[c] = H_{c-1}: fp32 [P][N] (coalesced over n) and bf16 rows n
        float* hblk = hist + (((size_t)b * nc + c) * d.H + h) * PN + n;
#pragma unroll
        for (int p = 0; p < 64; ++p) hblk[(size_t)p * d.N] = st[p];
      }
      put_rows(st, &maps.rows, srow);  // MODE 0: hT[c] = H_{c-1}; MODE 1: gT[c] = g_c
      ok = __all_sync(0xffffffffu, wait_ws(&bar_full[buf], (it / kScanBufs) & 1, &s_abort));
      // warp-uniform; the other consumer warps still reach the named barriers
      // st = e st + (the 64 columns at col of the buffer)
      auto advance = [&](float e, uint32_t col) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float v[32];
          tmem_ld32(tm + buf_cols * buf + col + 32 * half + lane_base, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) st[32 * half + i] = fmaf(e, st[32 * half + i], v[i]);
        }
      };
      if (split) {
        // g_mid = exp(cs_255 - cs_127) g_c + R_1 out as bf16 rows through the
        // staging tile (every consumer warp reaches its barriers), then R_0
        if (ok) {
          fence_after_sync();
          advance(exp2f(s_last[buf] - s_mid[buf]), 0);
        }
        if (named_sync_or(2, 128, !ok)) {
          ok = false;
          break;
        }
        put_rows(st, &maps.rows3, srow);
        advance(exp2f(s_mid[buf]), 64);
        fence_before_sync();
        __syncwarp();
        if ((tid & 31) == 0) mbar_arrive(&bar_free[buf]);
      } else if (ok) {
        fence_after_sync();
        advance(exp2f(s_last[buf]), 0);
        fence_before_sync();
        __syncwarp();
        if ((tid & 31) == 0) mbar_arrive(&bar_free[buf]);
      }
      if (named_sync_or(2, 128, !ok)) {
        ok = false;
        break;
      }
    }
    if (ok && final_or_dh0) {
      float* dst = final_or_dh0 + ((size_t)b * d.H + h) * PN + n;
#pragma unroll
      for (int p = 0; p < 64; ++p) dst[(size_t)p * d.N] = st[p];
    }
    if (tid == 0) bulk_wait0();
  }
  grid_dep_launch();
  fence_before_sync();
  __syncthreads();
  if (tid < 32) tmem_dealloc(tm, buf_cols * kScanBufs);
}

// ---------------------------------------------------------------------------
// Forward chunk scan: y for one (b, chunk, head) per CTA, block by block.
struct ScanMaps {
  CUtensorMap x;   // [B*T][H*P] bf16, box {64, 128}
  CUtensorMap B;   // [B*T][G*N] bf16, box {64, 128}
  CUtensorMap C;   // [B*T][G*N] bf16, box {64, 128}
  CUtensorMap y;   // [B*T][H*P] bf16, box {64, 128} (store)
};

// shared-memory layout of k_fwd_scan_tc (offsets from the 1024-aligned base);
// 96 KB so that two CTAs fit on one SM
constexpr uint32_t kScanR1 = 0;       // C tile (32K) + B tile (32K); M and y staging reuse the C part
constexpr uint32_t kScanX = 65536;    // X block [128 rows][64 p]
constexpr uint32_t kScanH = 81920;    // state as bf16 B operand, row n, 64 p (MN-major)
constexpr uint32_t kScanBytes = 98304;

// The chunk-start state comes as fp32 [P][N] from the history, converted to
// bf16 rows by the threads.
__global__ void __launch_bounds__(256, 2)
k_fwd_scan_tc(const __grid_constant__ ScanMaps maps, TcDims d, const float* __restrict__ dt,
              const float* __restrict__ A, const float* __restrict__ D,
              const float* __restrict__ hist) {
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  uint8_t* sC = sm + kScanR1;
  uint8_t* sB = sm + kScanR1 + 32768;
  uint8_t* sM = sm + kScanR1;   // after the CB / Ys products are done
  uint8_t* sY = sm + kScanR1;   // after the Y product is done
  uint8_t* sX = sm + kScanX;
  uint8_t* sH = sm + kScanH;
  __shared__ float s_cs2[256], s_dt[256], scratch[8];
  __shared__ __align__(16) float s_E[4][128];  // per-warp column factors exp(cs_r - cs_j) dt_j
  __shared__ uint64_t bar_load, bar_mma;
  __shared__ uint32_t tmem_base;
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = h / d.hpg, tid = threadIdx.x, wg = tid >> 7, q = (tid >> 5) & 3;
  const int row = tid & 127;  // TMEM lane / tile row, shared by the two warpgroups
  const int Q = d.Q, nblk = Q / 128;
  const float Dh = D[h];
  const uint32_t lane_base = (uint32_t)(q * 32) << 16;

  if (tid == 0) {
    prefetch_tmap(&maps.x);
    prefetch_tmap(&maps.B);
    prefetch_tmap(&maps.C);
    prefetch_tmap(&maps.y);
    mbar_init(&bar_load, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
  }
  if (tid < 32) {
    tmem_alloc(&tmem_base, 256);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tm = tmem_base;
  const uint32_t tCB = tm, tY = tm, tYs = tm + 128, tS0 = tm + 192;
  uint32_t load_phase = 0, mma_phase = 0;
  bool ok = true;

  auto issue_loads = [&](int row0) {
    mbar_expect_tx(&bar_load, 80 * 1024);
    tma_load_2d(sC, &maps.C, g * d.N, row0, &bar_load);
    tma_load_2d(sC + 16384, &maps.C, g * d.N + 64, row0, &bar_load);
    tma_load_2d(sB, &maps.B, g * d.N, row0, &bar_load);
    tma_load_2d(sB + 16384, &maps.B, g * d.N + 64, row0, &bar_load);
    tma_load_2d(sX, &maps.x, h * d.P, row0, &bar_load);
  };
  const int crow = b * d.T + c * Q;
  // C, B, x are inputs that no kernel of this library writes: fetched before
  // waiting for the kernel launched ahead of this one; the states after
  if (tid == 0) issue_loads(crow);
  grid_dep_wait();

  // H_{c-1} as bf16 rows n (64 p each): the MN-major B operand of C H^T.
  const float* Hg = hist + (((size_t)b * d.nc + c) * d.H + h) * (size_t)(64 * 128);
  chunk_cumsum_256(d, dt, A, b, c, h, s_cs2, s_dt, scratch);
  {  // thread (wg, n) converts p in [32 wg, 32 wg + 32) from fp32 [P][N]
    const int n = row;
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
      float v8[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) v8[t] = Hg[(size_t)(wg * 32 + ch * 8 + t) * 128 + n];
      store_row_bf16(sH, n, wg * 4 + ch, v8);
    }
  }

  for (int blk = 0; blk < nblk && ok; ++blk) {
    const int row0 = crow + blk * 128;
    // per-warp column factors of this block: E[w][jj] = exp(cs_r - cs_J) dt_J, J < r
    const int base = blk * 128;
    for (int e = tid; e < 4 * 128; e += 256) {
      const int w = e >> 7, jj = e & 127;
      const int r = base + 32 * w, J = base + jj;
      s_E[w][jj] = (J < r) ? exp2f(s_cs2[r] - s_cs2[J]) * s_dt[J] : 0.f;
    }
    // reference log-decay of the block's state term: cs before row `base`
    const float ref2 = blk == 0 ? 0.f : s_cs2[base - 1];
    fence_async_smem();
    ok = wait_or_flag(&bar_load, load_phase);
    load_phase ^= 1;
    if (!ok) break;
    fence_after_sync();
    if (tid == 0) {
      // CB = C_blk B_blk^T  (128 x 128, K = N)
      const uint32_t id_cb = idesc_bf16(128, 128, false, false);
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
        mma_bf16(tCB, desc_sw128(smem_u32(sC) + off, 16, 1024),
                 desc_sw128(smem_u32(sB) + off, 16, 1024), id_cb, kk > 0);
      }
      // Ys = C_blk Hin^T  (128 x 64, K = N); Hin rows n, MN-major
      const uint32_t id_ys = idesc_bf16(128, 64, false, true);
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t aoff = (kk >> 2) * 16384 + (kk & 3) * 32;
        mma_bf16(tYs, desc_sw128(smem_u32(sC) + aoff, 16, 1024),
                 desc_sw128(smem_u32(sH) + kk * 2048, 16384, 1024), id_ys, kk > 0);
      }
      mma_commit(&bar_mma);
    }
    ok = wait_or_flag(&bar_mma, mma_phase);
    mma_phase ^= 1;
    fence_after_sync();
    if (!ok) break;

    const int I = base + row;  // row inside the chunk
    // M = CB o L o dt (masked), bf16 K-major A operand: row, K = j (two 64-wide tiles).
    // Warpgroup wg writes columns [64 wg, 64 wg + 64).
    {
      const float fi = exp2f(s_cs2[I] - s_cs2[base + 32 * q]);
      const float csI = s_cs2[I];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int jc = 2 * wg + u;
        float v[32];
        if (jc <= q) {  // warp-uniform
          tmem_ld32(tCB + lane_base + jc * 32, v);
          tmem_wait_ld();
          if (jc < q) {
#pragma unroll
            for (int t4 = 0; t4 < 8; ++t4) {
              const float4 e4 = *(const float4*)&s_E[q][jc * 32 + t4 * 4];
              v[t4 * 4 + 0] *= fi * e4.x;
              v[t4 * 4 + 1] *= fi * e4.y;
              v[t4 * 4 + 2] *= fi * e4.z;
              v[t4 * 4 + 3] *= fi * e4.w;
            }
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const int J = base + jc * 32 + k;
              const float ex = (J <= I) ? exp2f(csI - s_cs2[J]) : 0.f;
              v[k] *= ex * s_dt[J];
            }
          }
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = 0.f;
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int j = jc * 32 + q4 * 8;
          store_row_bf16(sM + (j >> 6) * 16384, row, (j & 63) >> 3, &v[q4 * 8]);
        }
      }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (tid == 0) {
      // Y = M X_blk (128 x 64, K = j); X is MN-major (row j, 64 p)
      const uint32_t id_y = idesc_bf16(128, 64, false, true);
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t aoff = (kk >> 2) * 16384 + (kk & 3) * 32;
        mma_bf16(tY, desc_sw128(smem_u32(sM) + aoff, 16, 1024),
                 desc_sw128(smem_u32(sX) + kk * 2048, 16384, 1024), id_y, kk > 0);
      }
      mma_commit(&bar_mma);
    }
    ok = wait_or_flag(&bar_mma, mma_phase);
    mma_phase ^= 1;
    fence_after_sync();
    if (!ok) break;
    // epilogue: y = Y + exp(cs_I - ref) Ys + D x  -> bf16 staging -> TMA store;
    // warpgroup wg handles p in [32 wg, 32 wg + 32)
    {
      const float sc = exp2f(s_cs2[I] - ref2);
      float yv[32], ys[32];
      tmem_ld32(tY + lane_base + wg * 32, yv);
      tmem_ld32(tYs + lane_base + wg * 32, ys);
      tmem_wait_ld();
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int ch = wg * 4 + k;
        float xf[8], o8[8];
        unpack8(*(const uint4*)(sX + sw128(row, ch)), xf);
#pragma unroll
        for (int t = 0; t < 8; ++t) o8[t] = fmaf(sc, ys[k * 8 + t], yv[k * 8 + t]) + Dh * xf[t];
        store_row_bf16(sY, row, ch, o8);
      }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (tid == 0) {
      tma_store_2d(&maps.y, sY, h * d.P, row0);
      bulk_commit();
    }
    if (blk + 1 < nblk) {
      // mid-chunk state: X_0 rows j scaled in place by exp(cs_127 - cs_j) dt_j,
      // S_0^T = B_0^T (w o X_0) (M = n, N = p, K = j), H_mid = exp(cs_127) H + S_0
      scale_tile_rows(sX, 128 * 8, [&](int r) { return exp2f(s_cs2[127] - s_cs2[r]) * s_dt[r]; });
      fence_async_smem();
      fence_before_sync();
      __syncthreads();
      fence_after_sync();
      if (tid == 0) {
        const uint32_t id_s0 = idesc_bf16(128, 64, true, true);
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16(tS0, desc_sw128(smem_u32(sB) + kk * 2048, 16384, 1024),
                   desc_sw128(smem_u32(sX) + kk * 2048, 16384, 1024), id_s0, kk > 0);
        mma_commit(&bar_mma);
      }
      ok = wait_or_flag(&bar_mma, mma_phase);
      mma_phase ^= 1;
      fence_after_sync();
      if (!ok) break;
      const float e127 = exp2f(s_cs2[127]);
      const int n = row;
      float v[32];
      tmem_ld32(tS0 + lane_base + wg * 32, v);
      tmem_wait_ld();
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float v8[8];
#pragma unroll
        for (int t = 0; t < 8; ++t)
          v8[t] = fmaf(e127, Hg[(size_t)(wg * 32 + k * 8 + t) * 128 + n], v[k * 8 + t]);
        store_row_bf16(sH, n, wg * 4 + k, v8);
      }
      if (tid == 0) {
        bulk_wait_read0();  // y staging (region R1) is reloaded next
        issue_loads(row0 + 128);
      }
      // sH written by every thread: visible to the next block's MMA
      fence_async_smem();
      fence_before_sync();
      __syncthreads();
      fence_after_sync();
    }
  }
  grid_dep_launch();
  if (tid == 0) bulk_wait0();
  fence_before_sync();
  __syncthreads();
  if (tid < 32) tmem_dealloc(tm, 256);
}

// ---------------------------------------------------------------------------
// Single-pass forward: the chunk-state pass folded into the chunk scan with a
// bounded look-back, for the shapes whose per-(b, h) state scan fills the GPU.
// Tiles are (b, chunk, head), taken from a counter chunk-major by resident
// CTAs (two per SM, each looping over tiles): the tile of chunk c - 1 of the
// same (b, h) was taken earlier by a CTA that processes its tiles in the
// order it took them, and every wait is on an earlier tile, so no wait can
// be on a tile nobody is processing.  A CTA takes its next tile at the start
// of its current tile's last y block and fetches that tile's dt meanwhile.
// Per tile:
//   A. before any wait, the chunk's state contributions block by block, the
//      last block first: S_k^T = B_k^T (w o X_k), w_j = exp(cs_end(k) - cs_j)
//      dt_j, end(k) the block's last row, with w o X_k written into the C
//      tile (idle until C) so that block 0's B and X stay as loaded for C;
//   B. the look-back: wait (bounded) for the flag of the history slot c,
//      which chunk c - 1 fills with H_{c-1} (slot 0 = h0 or zeros, written
//      here); H_mid = exp(cs_127) H_{c-1} + S_0 and
//      H_c = exp(cs_{Q-1} - cs_127) H_mid + S_1 (one block: H_c =
//      exp(cs_127) H_{c-1} + S_0); publish H_c into slot c + 1 and release
//      its flag, or write the final state;
//   C. y block by block as in k_fwd_scan_tc, with H_{c-1} and then H_mid as
//      the state term.
// flags: [B][nc][H] slot-ready words, then the tile counter; all zero at
// launch.  A wait that gives up sets the device error word and goes on with
// the slot as it is, and every CTA releases its successor's flag, so that a
// failure does not make every later chunk wait out its limit too (the outputs
// are then wrong; nothing hangs).
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned int* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(unsigned int* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Bounded wait (about kWaitLimitNs) until the counter *f reaches `target`;
// false if it gave up.  Not inlined: it runs once per split unit, and kept
// apart it leaves the register allocation of its callers' loops alone.
__device__ __noinline__ bool wait_count_at_least(const unsigned int* f, unsigned int target) {
  bool got = ld_acquire_gpu(f) >= target;
  if (!got) {
    const uint64_t t0 = globaltimer_ns();
    while (!got) {
#pragma unroll 1
      for (int i = 0; i < 32 && !got; ++i) got = ld_acquire_gpu(f) >= target;
      if (!got && globaltimer_ns() - t0 > kWaitLimitNs) break;
    }
  }
  return got;
}

template <bool kRaw>
__global__ void __launch_bounds__(256, 2)
k_fwd_single_tc(const __grid_constant__ ScanMaps maps, TcDims d, const float* __restrict__ dt,
                const float* __restrict__ A, const float* __restrict__ D,
                const float* __restrict__ h0, float* hist, float* __restrict__ final_state,
                unsigned int* flags) {
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  uint8_t* sB = sm + kScanR1 + 32768;  // the state phase's B_1 (B_0 of one block)
  uint8_t* sX = sm + kScanX;
  uint8_t* sH = sm + kScanH;
  __shared__ float s_cs2[256], s_dt[256], scratch[8];
  __shared__ __align__(16) float s_E[4][128];  // per-warp column factors exp(cs_r - cs_j) dt_j
  __shared__ uint64_t bar_load, bar_mma, bar_c0;
  __shared__ uint32_t tmem_base;
  __shared__ int s_tile;
  const int tid = threadIdx.x, wg = tid >> 7, q = (tid >> 5) & 3;
  const int row = tid & 127;  // TMEM lane / tile row, shared by the two warpgroups
  const int Q = d.Q, nblk = Q / 128;
  const uint32_t lane_base = (uint32_t)(q * 32) << 16;
  const size_t PN = 64 * 128;
  const int ntiles = d.B * d.nc * d.H;
  unsigned int* counter = flags + (size_t)ntiles;

  if (tid == 0) {
    s_tile = (int)atomicAdd(counter, 1u);
    prefetch_tmap(&maps.x);
    prefetch_tmap(&maps.B);
    prefetch_tmap(&maps.C);
    prefetch_tmap(&maps.y);
    mbar_init(&bar_load, 1);
    mbar_init(&bar_mma, 1);
    mbar_init(&bar_c0, 1);
    fence_mbar_init();
  }
  if (tid < 32) {
    tmem_alloc(&tmem_base, 256);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const int bh = d.B * d.H;
  const uint32_t tm = tmem_base;
  const uint32_t tCB = tm, tY = tm, tYs = tm + 128, tS0 = tm + 192;
  const uint32_t tS1 = tm + 128;  // block 1's state contribution, read out before Ys reuses it
  uint32_t load_phase = 0, mma_phase = 0, c0_phase = 0;
  bool ok = true;
  int tile = s_tile;
  // a tile's stored dt of row tid of its chunk and its head's A (raw-dt mode:
  // dt_raw, a_log and dt_bias), fetched a tile ahead and used at its start
  float dv, av, bv;
  auto fetch = [&](int t) {
    const int hh = t % d.H;
    dv = t < ntiles && tid < Q
             ? dt[((size_t)((t % bh) / d.H) * d.T + (size_t)(t / bh) * Q + tid) * d.H + hh]
             : 0.f;
    av = t < ntiles ? (kRaw ? d.a_log[hh] : A[hh]) : 0.f;
    bv = kRaw && t < ntiles ? d.dt_bias[hh] : 0.f;
  };
  fetch(tile);

  while (tile < ntiles && ok) {
  const int c = tile / bh, b = (tile % bh) / d.H, h = tile % d.H;
  const int g = h / d.hpg;
  const float Dh = D[h];
  const int crow = b * d.T + c * Q;

  auto issue_state_loads = [&](int row0) {  // B and X of one block
    mbar_expect_tx(&bar_load, 48 * 1024);
    tma_load_2d(sB, &maps.B, g * d.N, row0, &bar_load);
    tma_load_2d(sB + 16384, &maps.B, g * d.N + 64, row0, &bar_load);
    tma_load_2d(sX, &maps.x, h * d.P, row0, &bar_load);
  };
  if (tid == 0) {
    bulk_wait_read0();  // the previous tile's last y store has read its staging
    issue_state_loads(crow + (nblk - 1) * 128);
  }
  {
    // the chunk-local inclusive cumsum of dt * A (log2 units)
    const float dtv = kRaw && tid < Q ? softplus_tc(dv + bv) : dv;
    const float a2 = (kRaw ? -expf(av) : av) * kLog2e;
    const float cs = block_inclusive_scan(dtv * a2, scratch);
    if (tid < Q) {
      s_cs2[tid] = cs;
      s_dt[tid] = dtv;
    }
    __syncthreads();
  }

  // ---- tile places, in 16 KB tiles R0-R5 of the 96 KB:
  //   one block (Q = 128): C R0-R1 (later M, then the y staging), B R2-R3,
  //   X R4, the state term R5;
  //   two blocks: the state phase takes B_1 R2-R3, X_1 R4 and w o X R0, then
  //   X_0 R4 and B_0 R1 + R5 (fetched under block 1's state product); C_0
  //   lands in R2-R3 once block 1's product is done, the state term (bf16
  //   rows) goes to R0, and block 1's B and C follow into R1 + R5 and R2-R3
  //   as block 0's products release them.  B is K-major with its K-half
  //   n 64-127 at kB1 from n 0-63.
  const bool two = nblk == 2;
  uint8_t* const tC = two ? sm + 32768 : sm;
  uint8_t* const tB = two ? sm + 16384 : sm + 32768;
  const uint32_t kB1 = two ? 65536u : 16384u;
  uint8_t* const tH = two ? sm : sH;

  // ---- A: the chunk's state contributions, the last block first
  uint8_t* sWX = sm;  // w o X_k (R0)
  for (int blk = nblk - 1; blk >= 0 && ok; --blk) {
    const int base = blk * 128, end = base + 127;
    // block 0's B is in its y-phase place (R2-R3 for one block, R1 + R5 for two)
    uint8_t* const sBk = blk == 0 ? tB : sB;
    const uint32_t lbo = blk == 0 ? kB1 : 16384u;
    ok = wait_or_flag(&bar_load, load_phase);
    load_phase ^= 1;
    if (!ok) break;
    fence_after_sync();
    for (int e = tid; e < 128 * 8; e += 256) {
      const int r = e >> 3;
      const float w = exp2f(s_cs2[end] - s_cs2[base + r]) * s_dt[base + r];
      float f[8];
      unpack8(*(const uint4*)(sX + e * 16), f);
      *(uint4*)(sWX + e * 16) = make_uint4(pack_bf16(f[0] * w, f[1] * w), pack_bf16(f[2] * w, f[3] * w),
                                           pack_bf16(f[4] * w, f[5] * w), pack_bf16(f[6] * w, f[7] * w));
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (tid == 0) {
      // S_k^T = B_k^T (w o X_k)  (M = n, N = p, K = j; both operands MN-major)
      const uint32_t id_s = idesc_bf16(128, 64, true, true);
      const uint32_t tS = blk == 0 ? tS0 : tS1;
      for (int kk = 0; kk < 8; ++kk)
        mma_bf16(tS, desc_sw128(smem_u32(sBk) + kk * 2048, lbo, 1024),
                 desc_sw128(smem_u32(sWX) + kk * 2048, 16384, 1024), id_s, kk > 0);
      mma_commit(&bar_mma);
      if (blk == 1) {  // block 0's state tiles, under this product
        mbar_expect_tx(&bar_load, 48 * 1024);
        tma_load_2d(tB, &maps.B, g * d.N, crow, &bar_load);
        tma_load_2d(tB + kB1, &maps.B, g * d.N + 64, crow, &bar_load);
        tma_load_2d(sX, &maps.x, h * d.P, crow, &bar_load);
      }
    }
    ok = wait_or_flag(&bar_mma, mma_phase);
    mma_phase ^= 1;
    fence_after_sync();
    if (!ok) break;
    // C_0 into the tiles this product has released: R2-R3 after block 1's
    // product (two blocks), R0-R1 after block 0's (one block)
    if (tid == 0 && (blk == 1 || !two)) {
      uint64_t* bar = two ? &bar_c0 : &bar_load;
      mbar_expect_tx(bar, 32 * 1024);
      tma_load_2d(tC, &maps.C, g * d.N, crow, bar);
      tma_load_2d(tC + 16384, &maps.C, g * d.N + 64, crow, bar);
    }
  }

  // ---- B: the look-back and the chunk-end state
  float hv[32];  // H_{c-1}[p][n] for p = 32 wg + k, n = row
  float* slot_in = hist + (((size_t)b * d.nc + c) * d.H + h) * PN;
  if (c == 0) {
    const float* h0p = h0 ? h0 + ((size_t)b * d.H + h) * PN : nullptr;
#pragma unroll
    for (int k = 0; k < 32; ++k) hv[k] = h0p ? h0p[(size_t)(wg * 32 + k) * 128 + row] : 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k) slot_in[(size_t)(wg * 32 + k) * 128 + row] = hv[k];
  } else {
    if (tid == 0) {
      const unsigned int* f = flags + ((size_t)b * d.nc + c) * d.H + h;
      bool got = ld_acquire_gpu(f) != 0u;
      if (!got) {
        const uint64_t t0 = globaltimer_ns();
        while (!got) {
#pragma unroll 1
          for (int i = 0; i < 32 && !got; ++i) got = ld_acquire_gpu(f) != 0u;
          if (!got && globaltimer_ns() - t0 > kWaitLimitNs) break;
        }
      }
      if (!got) atomicOr(&g_tc_error, 1u);
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 32; ++k) hv[k] = __ldcg(slot_in + (size_t)(wg * 32 + k) * 128 + row);
  }
  uint32_t hmid[16];  // H_mid as bf16 pairs (two-block chunks), the state term of block 1
  if (ok) {
    float hn[32];
    {
      float s0[32];
      tmem_ld32(tS0 + lane_base + wg * 32, s0);
      tmem_wait_ld();
      const float e0 = exp2f(s_cs2[127]);
#pragma unroll
      for (int k = 0; k < 32; ++k) hn[k] = fmaf(e0, hv[k], s0[k]);
    }
    if (nblk == 2) {
#pragma unroll
      for (int k = 0; k < 16; ++k) hmid[k] = pack_bf16(hn[2 * k], hn[2 * k + 1]);
      float s1[32];
      tmem_ld32(tS1 + lane_base + wg * 32, s1);
      tmem_wait_ld();
      const float e1 = exp2f(s_cs2[Q - 1] - s_cs2[127]);
#pragma unroll
      for (int k = 0; k < 32; ++k) hn[k] = fmaf(e1, hn[k], s1[k]);
    }
    if (c + 1 < d.nc) {
      // made visible to chunk c + 1 by the barrier below and one thread's release
      float* slot_out = hist + (((size_t)b * d.nc + c + 1) * d.H + h) * PN;
#pragma unroll
      for (int k = 0; k < 32; ++k) slot_out[(size_t)(wg * 32 + k) * 128 + row] = hn[k];
    } else if (final_state) {
      float* fo = final_state + ((size_t)b * d.H + h) * PN;
#pragma unroll
      for (int k = 0; k < 32; ++k) fo[(size_t)(wg * 32 + k) * 128 + row] = hn[k];
    }
    // H_{c-1} as bf16 rows n (64 p each): the MN-major B operand of C H^T
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) store_row_bf16(tH, row, wg * 4 + ch, &hv[ch * 8]);
  }
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  // released even after a wait that gave up (the error word is set then), so
  // that the next chunk does not wait out its own limit as well.  The
  // barrier above orders every thread's history writes before this release
  // (cumulative at gpu scope); a thread other than the MMA issuer does it.
  if (c + 1 < d.nc && tid == 32) {
    __threadfence();
    st_release_gpu(flags + ((size_t)b * d.nc + c + 1) * d.H + h, 1u);
  }

  // ---- C: y block by block
  for (int blk = 0; blk < nblk && ok; ++blk) {
    const int row0 = crow + blk * 128;
    const int base = blk * 128;
    if (blk == nblk - 1 && tid == 0) s_tile = (int)atomicAdd(counter, 1u);  // the next tile
    for (int e = tid; e < 4 * 128; e += 256) {
      const int w = e >> 7, jj = e & 127;
      const int r = base + 32 * w, J = base + jj;
      s_E[w][jj] = (J < r) ? exp2f(s_cs2[r] - s_cs2[J]) * s_dt[J] : 0.f;
    }
    // reference log-decay of the block's state term: cs before row `base`
    const float ref2 = blk == 0 ? 0.f : s_cs2[base - 1];
    fence_async_smem();
    if (two && blk == 0) {
      ok = wait_or_flag(&bar_c0, c0_phase);
      c0_phase ^= 1;
    } else {
      ok = wait_or_flag(&bar_load, load_phase);
      load_phase ^= 1;
    }
    if (!ok) break;
    fence_after_sync();
    if (tid == 0) {
      const uint32_t id_cb = idesc_bf16(128, 128, false, false);
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
        const uint32_t boff = (kk >> 2) * kB1 + (kk & 3) * 32;
        mma_bf16(tCB, desc_sw128(smem_u32(tC) + off, 16, 1024),
                 desc_sw128(smem_u32(tB) + boff, 16, 1024), id_cb, kk > 0);
      }
      const uint32_t id_ys = idesc_bf16(128, 64, false, true);
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t aoff = (kk >> 2) * 16384 + (kk & 3) * 32;
        mma_bf16(tYs, desc_sw128(smem_u32(tC) + aoff, 16, 1024),
                 desc_sw128(smem_u32(tH) + kk * 2048, 16384, 1024), id_ys, kk > 0);
      }
      mma_commit(&bar_mma);
    }
    ok = wait_or_flag(&bar_mma, mma_phase);
    mma_phase ^= 1;
    fence_after_sync();
    if (!ok) break;
    if (tid == 0 && two && blk == 0) {
      // block 1's B into the B tiles (B_0 has been read); its C and X follow
      // once block 0's y is out
      mbar_expect_tx_only(&bar_load, 32 * 1024);
      tma_load_2d(tB, &maps.B, g * d.N, row0 + 128, &bar_load);
      tma_load_2d(tB + kB1, &maps.B, g * d.N + 64, row0 + 128, &bar_load);
    }

    const int I = base + row;
    {
      const float fi = exp2f(s_cs2[I] - s_cs2[base + 32 * q]);
      const float csI = s_cs2[I];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int jc = 2 * wg + u;
        float v[32];
        if (jc <= q) {  // warp-uniform
          tmem_ld32(tCB + lane_base + jc * 32, v);
          tmem_wait_ld();
          if (jc < q) {
#pragma unroll
            for (int t4 = 0; t4 < 8; ++t4) {
              const float4 e4 = *(const float4*)&s_E[q][jc * 32 + t4 * 4];
              v[t4 * 4 + 0] *= fi * e4.x;
              v[t4 * 4 + 1] *= fi * e4.y;
              v[t4 * 4 + 2] *= fi * e4.z;
              v[t4 * 4 + 3] *= fi * e4.w;
            }
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const int J = base + jc * 32 + k;
              const float ex = (J <= I) ? exp2f(csI - s_cs2[J]) : 0.f;
              v[k] *= ex * s_dt[J];
            }
          }
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = 0.f;
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int j = jc * 32 + q4 * 8;
          store_row_bf16(tC + (j >> 6) * 16384, row, (j & 63) >> 3, &v[q4 * 8]);
        }
      }
    }
    // block 0 of two: the state term of block 1 (H_mid) replaces H_{c-1}, which
    // the Ys product above has read
    if (blk == 0 && nblk == 2) {
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
        *(uint4*)(tH + sw128(row, wg * 4 + ch)) =
            make_uint4(hmid[4 * ch], hmid[4 * ch + 1], hmid[4 * ch + 2], hmid[4 * ch + 3]);
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (blk == nblk - 1) fetch(s_tile);  // the next tile (published by the barrier), under this block
    if (tid == 0) {
      const uint32_t id_y = idesc_bf16(128, 64, false, true);
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t aoff = (kk >> 2) * 16384 + (kk & 3) * 32;
        mma_bf16(tY, desc_sw128(smem_u32(tC) + aoff, 16, 1024),
                 desc_sw128(smem_u32(sX) + kk * 2048, 16384, 1024), id_y, kk > 0);
      }
      mma_commit(&bar_mma);
    }
    ok = wait_or_flag(&bar_mma, mma_phase);
    mma_phase ^= 1;
    fence_after_sync();
    if (!ok) break;
    {
      const float sc = exp2f(s_cs2[I] - ref2);
      float yv[32], ys[32];
      tmem_ld32(tY + lane_base + wg * 32, yv);
      tmem_ld32(tYs + lane_base + wg * 32, ys);
      tmem_wait_ld();
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int ch = wg * 4 + k;
        float xf[8], o8[8];
        unpack8(*(const uint4*)(sX + sw128(row, ch)), xf);
#pragma unroll
        for (int t = 0; t < 8; ++t) o8[t] = fmaf(sc, ys[k * 8 + t], yv[k * 8 + t]) + Dh * xf[t];
        store_row_bf16(tC, row, ch, o8);  // y staging in the M tile
      }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (tid == 0) {
      tma_store_2d(&maps.y, tC, h * d.P, row0);
      bulk_commit();
      if (blk + 1 < nblk) {
        // block 1's C into the y staging's tiles once the store has read
        // them, and its X (block 0's has been read); its B is on its way
        bulk_wait_read0();
        mbar_expect_tx(&bar_load, 48 * 1024);
        tma_load_2d(tC, &maps.C, g * d.N, row0 + 128, &bar_load);
        tma_load_2d(tC + 16384, &maps.C, g * d.N + 64, row0 + 128, &bar_load);
        tma_load_2d(sX, &maps.x, h * d.P, row0 + 128, &bar_load);
      }
    }
  }
  // the tile's TMEM reads and shared-memory use are done; its successor
  // (taken above, or past the last tile: the loop ends)
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  tile = s_tile;
  }
  grid_dep_launch();
  if (tid == 0) bulk_wait0();
  fence_before_sync();
  __syncthreads();
  if (tid < 32) tmem_dealloc(tm, 256);
}

// ---------------------------------------------------------------------------
// Backward on tensor cores.  The work items are (unit, head) pairs, a unit
// being one (128-row block k, chunk c, group g, batch b); one CTA per SM takes
// an equal contiguous range of items, i.e. one or more segments of
// consecutive heads of a unit.  Per segment the CTA loops over its heads and
// accumulates dC and dB of the block over them in TMEM (fixed head order).  A
// unit covered by one segment writes dC, dB directly; of a unit split over
// several CTAs, the last segment to finish (a per-unit ticket) keeps its sums
// in TMEM, and the others write fp32 partials and count them in a per-unit
// counter that it waits for; it sums all in segment order (deterministic).
// Each block is treated as a chunk of 128 steps with
//   state in  Hin  = H_{c-1} (k = 0) or H_mid  (k = 1),
//   grad out  gout = g_c     (last block) or g_mid = exp(cs_255 - cs_127) g_c + R_1 (k = 0 of 2),
//   R_1 = sum_{i >= 128} exp(cs_i - cs_127) dy_i C_i^T,
// and the per-block formulas of the chunked backward (see ssd_simt.cu).  The
// strict row and column sums of M_ij = W_ij (C_i.B_j) come from the rows the
// threads hold (row sums) and a warp-transposed reduction (column sums).
// 4-byte asynchronous global -> shared copy, and the wait for this thread's copies
__device__ __forceinline__ void cp_async4(float* smem, const float* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(smem)), "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Work split of the backward.  Items are (unit, head) pairs, item = unit *
// hpg + head in group, unit = ((b * G + g) * nc + c) * nblk + k.  A head of
// the second block of a 256-step chunk forms the mid-chunk state from the
// first block's tiles, so it weighs more; the CTAs take contiguous item
// ranges of equal weight: item i goes to CTA floor(W(i) ncta / W(nitems)),
// W(i) being the weight of the items before it.  The host computes the first
// item of every CTA.  The weights are measured: 1.10 against 1.0, 1.18 and
// 1.26 for the second block gave the shortest backward on the B4 T2048 H32
// bf16 workload.
constexpr long long kBwW0 = 100, kBwW1 = 110;
inline long long bw_weight_before(long long i, int hpg, int nblk) {
  if (nblk == 1) return i * kBwW0;
  const long long u = i / hpg, r = i % hpg;
  const long long w = (u >> 1) * hpg * (kBwW0 + kBwW1);
  return (u & 1) ? w + hpg * kBwW0 + r * kBwW1 : w + r * kBwW0;
}
struct BwdSplit {
  int first[kBwdMaxCtas + 1];  // first item of each CTA, then the item count
};

struct BwdMaps {
  CUtensorMap x;   // [B*T][H*P] bf16, box {64, 128}
  CUtensorMap dy;  // [B*T][H*P] bf16, box {64, 128}
  CUtensorMap B;   // [B*T][G*N] bf16, box {64, 128}
  CUtensorMap C;   // [B*T][G*N] bf16, box {64, 128}
  CUtensorMap dx;  // [B*T][H*P] bf16, box {64, 128} (store)
  CUtensorMap dB;  // [B*T][G*N] bf16, box {64, 128} (store)
  CUtensorMap dC;  // [B*T][G*N] bf16, box {64, 128} (store)
  CUtensorMap ht;  // chunk-start states, bf16 rows n: [B*nc*H*N][P], box {64, 128}
  CUtensorMap gt;  // chunk-end state gradients, same layout
  CUtensorMap gmt; // mid-chunk state gradients (chunks of two blocks), same layout
};

constexpr int kBwThreads = 512;       // four warpgroups share each TMEM lane quarter
constexpr uint32_t kBwC = 0;          // C_k: 2 K-major tiles [128][128 B]
constexpr uint32_t kBwB = 32768;      // B_k
constexpr uint32_t kBwO = 65536;      // L o CB (2 tiles, same layout as W), then dx staging
constexpr uint32_t kBwX = 98304;      // X_k  [128 rows][64 p]
constexpr uint32_t kBwDY = 114688;    // dY_k
constexpr uint32_t kBwXO = 131072;    // X_0 (k = 1) or dY_1 (k = 0), row-scaled; then e o dY_k
constexpr uint32_t kBwH = 147456;     // Hin  bf16, row n, 64 p
constexpr uint32_t kBwG = 163840;     // gout bf16, row n, 64 p
constexpr uint32_t kBwW = 180224;     // B_0 (k = 1) / C_1 (k = 0) per head, then W
constexpr uint32_t kBwBytes = 212992;

template <bool kRaw>
__global__ void __launch_bounds__(kBwThreads, 1)
k_bwd_tc(const __grid_constant__ BwdMaps maps, const __grid_constant__ BwdSplit split, TcDims d,
         long long nitems,
         const float* __restrict__ dt, const float* __restrict__ A, const float* __restrict__ D,
         float* __restrict__ ddt, float* __restrict__ dA_part, float* __restrict__ dD_part,
         float* __restrict__ dtb_part, float* __restrict__ d_dt_bias,
         void* __restrict__ dB_out, void* __restrict__ dC_out, float* __restrict__ dA,
         float* __restrict__ dD, unsigned int* __restrict__ tickets,
         unsigned int* __restrict__ written, float* __restrict__ part, int gmid) {
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  uint8_t* sC = sm + kBwC;
  uint8_t* sB = sm + kBwB;
  uint8_t* sO = sm + kBwO;
  uint8_t* sX = sm + kBwX;
  uint8_t* sDY = sm + kBwDY;
  uint8_t* sXO = sm + kBwXO;
  uint8_t* sH = sm + kBwH;
  uint8_t* sG = sm + kBwG;
  uint8_t* sW = sm + kBwW;
  // decay tables of the current head, and the next head's (s_cs2n, s_dtn),
  // built by warpgroups 1-3 while warpgroup 0 finishes the current head; at
  // the next head's start they are copied into place and give s_E, s_Edt
  __shared__ float s_cs2[256], s_dt[256], s_cs2n[256], s_dtn[256];
  __shared__ __align__(16) float s_E[4][128];    // exp(cs_r - cs_J), J < r = base + 32 q
  __shared__ __align__(16) float s_Edt[4][128];  // the same times dt_J
  __shared__ float s_col[4][128];                // per-warp strict column sums of M
  __shared__ float s_rs[3][128];                 // row-sum partials of warpgroups 1-3
  __shared__ float s_hg[4][128];                 // <gout, Hin> partials per warpgroup and row
  __shared__ float4 s_wtot[4];                   // warpgroup 0: per-warp totals (d(cs), e, <g, H>)
  __shared__ float2 s_wad[4];                    // warpgroup 0: per-warp dA, dD partials
  __shared__ float s_gsum[4];  // raw-dt mode: per-warp sums of the dt_raw gradient
  __shared__ uint64_t bar_shared, bar_head, bar_mma;
  __shared__ uint32_t tmem_base;
  __shared__ int s_flag;

  const int nblk = d.Q / 128;
  const int tid = threadIdx.x, wg = tid >> 7, q = (tid >> 5) & 3, lane = tid & 31;
  const int row = tid & 127;  // TMEM lane / tile row owned (with the other warpgroups)
  const uint32_t lane_base = (uint32_t)(q * 32) << 16;
  // items [it_begin, it_end) of this CTA (ranges of equal weight)
  const int ncta = (int)gridDim.x;
  const long long it_begin = split.first[blockIdx.x], it_end = split.first[blockIdx.x + 1];
  auto cta_of = [&](long long item) {  // the CTA whose range holds `item`
    int lo = 0, hi = ncta - 1;
    while (lo < hi) {
      const int m = (lo + hi + 1) >> 1;
      if (split.first[m] <= item)
        lo = m;
      else
        hi = m - 1;
    }
    return lo;
  };
  // the current segment's unit
  int k = 0, c = 0, g = 0, b = 0, base = 0, crow = 0, row0 = 0;
  const bool two = nblk == 2;
  // a block whose head forms the mid-chunk state (k = 1) or state gradient
  // (k = 0, unless the state pass has written it: gmid) from the other
  // block's tiles
  auto mid_of = [&](int kk) { return two && (kk == 1 || !gmid); };

  if (tid == 0) {
    prefetch_tmap(&maps.x);
    prefetch_tmap(&maps.dy);
    prefetch_tmap(&maps.B);
    prefetch_tmap(&maps.C);
    prefetch_tmap(&maps.ht);
    prefetch_tmap(&maps.gt);
    prefetch_tmap(&maps.gmt);
    mbar_init(&bar_shared, 1);
    mbar_init(&bar_head, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
  }
  if (tid < 32) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tm = tmem_base;
  const uint32_t T0 = tm, T1 = tm + 128, TdC = tm + 256, TdB = tm + 384;

  // the state-gradient rows a head of block kk reads: g_c, or g_mid for the
  // first block of two when the state pass has written it
  auto gout_map = [&](int kk) { return two && kk == 0 && gmid ? &maps.gmt : &maps.gt; };
  // with_state: also the head's state and state-gradient rows (outputs of the
  // state pass); the first head fetches them after waiting for that kernel
  // tiles of head h of unit uu (the head's own and, where it forms the
  // mid-chunk state or state gradient, the other block's tiles for it)
  auto issue_head_loads = [&](int uu, int h, bool with_state) {
    const int kk = uu % nblk, cc = (uu / nblk) % d.nc, gg = (uu / (nblk * d.nc)) % d.G;
    const int bb = uu / (nblk * d.nc * d.G);
    const int crow_u = bb * d.T + cc * d.Q, row0_u = crow_u + 128 * kk;
    mbar_expect_tx(&bar_head, (mid_of(kk) ? 80 : 32) * 1024 + 32 * 1024);
    tma_load_2d(sX, &maps.x, h * d.P, row0_u, &bar_head);
    tma_load_2d(sDY, &maps.dy, h * d.P, row0_u, &bar_head);
    if (mid_of(kk)) {
      if (kk == 1) {
        tma_load_2d(sXO, &maps.x, h * d.P, crow_u, &bar_head);
        tma_load_2d(sW, &maps.B, gg * d.N, crow_u, &bar_head);
        tma_load_2d(sW + 16384, &maps.B, gg * d.N + 64, crow_u, &bar_head);
      } else {
        tma_load_2d(sXO, &maps.dy, h * d.P, crow_u + 128, &bar_head);
        tma_load_2d(sW, &maps.C, gg * d.N, crow_u + 128, &bar_head);
        tma_load_2d(sW + 16384, &maps.C, gg * d.N + 64, crow_u + 128, &bar_head);
      }
    }
    if (with_state) {
      const int srow = ((bb * d.nc + cc) * d.H + h) * d.N;
      tma_load_2d(sH, &maps.ht, 0, srow, &bar_head);
      tma_load_2d(sG, gout_map(kk), 0, srow, &bar_head);
    }
  };
  // C_k and B_k of unit uu
  auto issue_unit_loads = [&](int uu) {
    const int kk = uu % nblk, cc = (uu / nblk) % d.nc, gg = (uu / (nblk * d.nc)) % d.G;
    const int bb = uu / (nblk * d.nc * d.G);
    const int row0_u = bb * d.T + cc * d.Q + 128 * kk;
    mbar_expect_tx(&bar_shared, 64 * 1024);
    tma_load_2d(sC, &maps.C, gg * d.N, row0_u, &bar_shared);
    tma_load_2d(sC + 16384, &maps.C, gg * d.N + 64, row0_u, &bar_shared);
    tma_load_2d(sB, &maps.B, gg * d.N, row0_u, &bar_shared);
    tma_load_2d(sB + 16384, &maps.B, gg * d.N + 64, row0_u, &bar_shared);
  };
  // dt of step tid - 256 of chunk cc, head hh, in the threads of warpgroups
  // 2 and 3 (0 past the chunk and in the other threads)
  auto load_dt_hi = [&](int bb, int cc, int hh) -> float {
    const int r = tid - 256;
    return r >= 0 && r < d.Q ? dt[((size_t)bb * d.T + (size_t)cc * d.Q + r) * d.H + hh] : 0.f;
  };
  // The next head's cumsum into s_cs2n (threads of warpgroups 1-3 only,
  // `sync` a barrier over them, after warpgroups 2-3 have staged dt in
  // s_dtn): warp 4 scans dt * A (log2 units, a2) over the 256 steps (eight
  // steps per lane in order, then the lanes).
  auto build_tables = [&](float a2, auto&& sync) {
    float* ncs = s_cs2n;
    const float* ndt = s_dtn;
    sync();
    if (wg == 1 && q == 0) {
      // the lane's eight partial sums are formed twice (the same order both
      // times), so that few registers are live here
      float run = 0.f;
#pragma unroll
      for (int t = 0; t < 8; ++t) run += ndt[lane * 8 + t] * a2;
      float inc = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
      }
      float off = __shfl_up_sync(0xffffffffu, inc, 1);
      if (lane == 0) off = 0.f;
      run = 0.f;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        run += ndt[lane * 8 + t] * a2;
        ncs[lane * 8 + t] = off + run;
      }
    }
  };
  const auto sync_wg123 = [] { named_sync(2, kBwThreads - 128); };
  uint32_t mma_phase = 0, head_phase = 0, shared_phase = 0;
  bool ok = true;
  for (long long x = it_begin; x < it_end && ok;) {
  // ---- segment: heads [j0, j0 + kh) of unit u
  const int u = (int)(x / d.hpg), j0 = (int)(x % d.hpg);
  const int kh = (int)((long long)(d.hpg - j0) < it_end - x ? (long long)(d.hpg - j0) : it_end - x);
  k = u % nblk;
  c = (u / nblk) % d.nc;
  g = (u / (nblk * d.nc)) % d.G;
  b = u / (nblk * d.nc * d.G);
  base = 128 * k;
  crow = b * d.T + c * d.Q;  // first row of the chunk
  row0 = crow + base;
  const int h_first = g * d.hpg + j0;
  const bool first_seg = x == it_begin;
  const bool mid = mid_of(k);
  if (tid == 0) {
    issue_unit_loads(u);
    issue_head_loads(u, h_first, !first_seg);
  }
  if (first_seg) {
    grid_dep_wait();
    if (tid == 0) {
      const int srow = ((b * d.nc + c) * d.H + h_first) * d.N;
      tma_load_2d(sH, &maps.ht, 0, srow, &bar_head);
      tma_load_2d(sG, gout_map(k), 0, srow, &bar_head);
    }
  }
  // A and D of the next head are loaded one head ahead and its dt goes
  // straight into s_dtn (raw-dt mode: dt_raw and a_log, transformed where
  // they are used), so the loads stay hidden; the first head's tables are
  // built here, the others' at the end of the head before them
  float A_next = kRaw ? d.a_log[h_first] : A[h_first], D_next = D[h_first];
  {
    const float dt0 = load_dt_hi(b, c, h_first);
    if (wg >= 2)
      s_dtn[tid - 256] = (kRaw && tid - 256 < d.Q) ? dt_of<kRaw>(d, dt0, h_first) : dt0;
    if (wg > 0) build_tables((kRaw ? -expf(A_next) : A_next) * kLog2e, sync_wg123);
    __syncthreads();
  }
  ok = wait_or_flag(&bar_shared, shared_phase);
  shared_phase ^= 1;

  for (int hh = 0; hh < kh && ok; ++hh) {
    const int h = h_first + hh;
    const float Ah = kRaw ? -expf(A_next) : A_next, Dh = D_next;
    if (hh + 1 < kh) {
      A_next = kRaw ? d.a_log[h + 1] : A[h + 1];
      D_next = D[h + 1];
    }
    // this head's tables into place, and s_E, s_Edt from them (published by
    // the barrier of the wait below)
    if (tid < 256)
      s_cs2[tid] = s_cs2n[tid];
    else
      s_dt[tid - 256] = s_dtn[tid - 256];
    {
      const int w = tid >> 7, jj = tid & 127;
      const int r = base + 32 * w, J = base + jj;
      const float ev = (J < r) ? exp2f(s_cs2n[r] - s_cs2n[J]) : 0.f;
      s_E[w][jj] = ev;
      s_Edt[w][jj] = ev * s_dtn[J];
    }
    const float ref2 = k == 0 ? 0.f : s_cs2n[base - 1];
    const float end2 = s_cs2n[base + 127];
    ok = wait_or_flag(&bar_head, head_phase);  // also publishes the tables
    head_phase ^= 1;
    if (!ok) break;

    // ---- mid-chunk state or state gradient (chunks of two blocks)
    if (mid) {
      if (k == 1)  // X_0 rows j by exp(cs_127 - cs_j) dt_j
        scale_tile_rows(sXO, 128 * 8, [&](int r) { return exp2f(s_cs2[127] - s_cs2[r]) * s_dt[r]; });
      else  // dY_1 rows i by exp(cs_i - cs_127)
        scale_tile_rows(sXO, 128 * 8, [&](int r) { return exp2f(s_cs2[128 + r] - s_cs2[127]); });
      fence_async_smem();
      fence_before_sync();
      __syncthreads();
      fence_after_sync();
      if (tid == 0) {
        // S_0^T = B_0^T (w o X_0)  or  R_1^T = C_1^T (e o dY_1):  M = n, N = p, K = rows
        const uint32_t id = idesc_bf16(128, 64, true, true);
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16(T1, desc_sw128(smem_u32(sW) + kk * 2048, 16384, 1024),
                   desc_sw128(smem_u32(sXO) + kk * 2048, 16384, 1024), id, kk > 0);
        mma_commit(&bar_mma);
      }
      ok = wait_or_flag(&bar_mma, mma_phase);
      mma_phase ^= 1;
      fence_after_sync();
      if (!ok) break;
      // row n, p in [16 wg, 16 wg + 16): H_mid = e^{cs_127} H + S_0 or g_mid = e^{..} g + R_1
      float v[16];
      tmem_ld16(T1 + lane_base + wg * 16, v);
      tmem_wait_ld();
      uint8_t* tile = (k == 1) ? sH : sG;
      const float sc = (k == 1) ? exp2f(s_cs2[127]) : exp2f(s_cs2[d.Q - 1] - s_cs2[127]);
#pragma unroll
      for (int q4 = 0; q4 < 2; ++q4) {
        float f[8];
        unpack8(*(const uint4*)(tile + sw128(row, wg * 2 + q4)), f);
#pragma unroll
        for (int t = 0; t < 8; ++t) f[t] = fmaf(sc, f[t], v[q4 * 8 + t]);
        store_row_bf16(tile, row, wg * 2 + q4, f);
      }
    }
    // <gout, Hin> over this thread's quarter row (bf16 operands, fp32 sum);
    // summed over the block with the d(cs) suffix sums at the end of the head
    {
      float hg = 0.f;
#pragma unroll
      for (int q4 = 0; q4 < 2; ++q4) {
        float fh[8], fg[8];
        unpack8(*(const uint4*)(sH + sw128(row, wg * 2 + q4)), fh);
        unpack8(*(const uint4*)(sG + sw128(row, wg * 2 + q4)), fg);
#pragma unroll
        for (int t = 0; t < 8; ++t) hg = fmaf(fh[t], fg[t], hg);
      }
      s_hg[wg][row] = hg;
    }
    if (mid) {  // every thread's T1 reads before the next products reuse T1
      fence_async_smem();
      fence_before_sync();
      __syncthreads();
      fence_after_sync();
    }

    // ---- phase A: CB = C_k B_k^T -> T0 ; dYX = dY_k X_k^T -> T1
    if (tid == 0) {
      const uint32_t id = idesc_bf16(128, 128, false, false);
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
        mma_bf16(T0, desc_sw128(smem_u32(sC) + off, 16, 1024),
                 desc_sw128(smem_u32(sB) + off, 16, 1024), id, kk > 0);
      }
      for (int kk = 0; kk < 4; ++kk)
        mma_bf16(T1, desc_sw128(smem_u32(sDY) + kk * 32, 16, 1024),
                 desc_sw128(smem_u32(sX) + kk * 32, 16, 1024), id, kk > 0);
      mma_commit(&bar_mma);
    }
    ok = wait_or_flag(&bar_mma, mma_phase);
    mma_phase ^= 1;
    fence_after_sync();
    if (!ok) break;

    // the next head's dt into s_dtn (read at this head's start), by
    // asynchronous copies that warpgroups 2-3 wait for where they use them;
    // issued here, about 2 us before the next proxy fence (which would
    // otherwise wait for them)
    if (wg >= 2 && hh + 1 < kh) {
      const int r = tid - 256;
      if (r < d.Q)
        cp_async4(&s_dtn[r], dt + ((size_t)b * d.T + (size_t)c * d.Q + r) * d.H + h + 1);
      else
        s_dtn[r] = 0.f;
    }

    // ---- W = L o dt_j o dYX -> sW, L o CB -> sO, row / column sums of M.
    // Warpgroup wg covers the 32 columns [32 wg, 32 wg + 32) of row `row`, in
    // two halves of 16.
    const int I = base + row;
    const float fi = exp2f(s_cs2[I] - s_cs2[base + 32 * q]);
    const float csI = s_cs2[I];
    float rowsum = 0.f;
    {
      const int jc = wg;
      if (jc <= q) {  // warp-uniform
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int col0 = jc * 32 + hf * 16;
          float cb[16], xy[16], wv[16];
          tmem_ld16(T0 + lane_base + col0, cb);
          tmem_ld16(T1 + lane_base + col0, xy);
          tmem_wait_ld();
          if (jc < q) {
#pragma unroll
            for (int t4 = 0; t4 < 4; ++t4) {
              const float4 e4 = *(const float4*)&s_E[q][col0 + t4 * 4];
              const float4 d4 = *(const float4*)&s_Edt[q][col0 + t4 * 4];
              const float ee[4] = {e4.x, e4.y, e4.z, e4.w};
              const float dd4[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const int m = t4 * 4 + t;
                wv[m] = fi * dd4[t] * xy[m];
                const float mm = wv[m] * cb[m];
                rowsum += mm;
                xy[m] = mm;
                cb[m] *= fi * ee[t];
              }
            }
          } else {
#pragma unroll
            for (int m = 0; m < 16; ++m) {
              const int J = base + col0 + m;
              const float L = (J <= I) ? exp2f(csI - s_cs2[J]) : 0.f;
              wv[m] = L * s_dt[J] * xy[m];
              const float mm = (J < I) ? wv[m] * cb[m] : 0.f;
              rowsum += mm;
              xy[m] = mm;
              cb[m] *= L;
            }
          }
          const float cs = warp_column_sum16(xy);
          if (lane < 16) s_col[q][col0 + lane] = cs;
#pragma unroll
          for (int q4 = 0; q4 < 2; ++q4) {
            const int j = col0 + q4 * 8;
            store_row_bf16(sW + (j >> 6) * 16384, row, (j & 63) >> 3, &wv[q4 * 8]);
            store_row_bf16(sO + (j >> 6) * 16384, row, (j & 63) >> 3, &cb[q4 * 8]);
          }
        }
      } else {  // above the diagonal: zeros
        const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int j = jc * 32 + q4 * 8;
          store_row_bf16(sW + (j >> 6) * 16384, row, (j & 63) >> 3, z);
          store_row_bf16(sO + (j >> 6) * 16384, row, (j & 63) >> 3, z);
        }
      }
    }
    if (wg > 0) s_rs[wg - 1][row] = rowsum;
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    // ---- phases B and C together: dC += W B_k ; dB += W^T C_k ;
    //      Gx = (L o CB)^T dY_k -> T0[0,64) ; Gs = B_k gout^T -> T0[64,128) ;
    //      CH = C_k Hin^T -> T1[0,64)
    if (tid == 0) {
      const uint32_t id_dc = idesc_bf16(128, 128, false, true);
      const uint32_t id_db = idesc_bf16(128, 128, true, true);
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t aoff = (kk >> 2) * 16384 + (kk & 3) * 32;
        mma_bf16(TdC, desc_sw128(smem_u32(sW) + aoff, 16, 1024),
                 desc_sw128(smem_u32(sB) + kk * 2048, 16384, 1024), id_dc, (hh > 0) || (kk > 0));
      }
      for (int kk = 0; kk < 8; ++kk)
        mma_bf16(TdB, desc_sw128(smem_u32(sW) + kk * 2048, 16384, 1024),
                 desc_sw128(smem_u32(sC) + kk * 2048, 16384, 1024), id_db, (hh > 0) || (kk > 0));
      const uint32_t id_mm = idesc_bf16(128, 64, true, true);
      const uint32_t id_km = idesc_bf16(128, 64, false, true);
      for (int kk = 0; kk < 8; ++kk)
        mma_bf16(T0, desc_sw128(smem_u32(sO) + kk * 2048, 16384, 1024),
                 desc_sw128(smem_u32(sDY) + kk * 2048, 16384, 1024), id_mm, kk > 0);
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t aoff = (kk >> 2) * 16384 + (kk & 3) * 32;
        mma_bf16(T0 + 64, desc_sw128(smem_u32(sB) + aoff, 16, 1024),
                 desc_sw128(smem_u32(sG) + kk * 2048, 16384, 1024), id_km, kk > 0);
        mma_bf16(T1, desc_sw128(smem_u32(sC) + aoff, 16, 1024),
                 desc_sw128(smem_u32(sH) + kk * 2048, 16384, 1024), id_km, kk > 0);
      }
      mma_commit(&bar_mma);
    }
    // under the B and C products: this thread's quarter rows of x_j and dy_i
    // (unscaled) into registers, X scaled in place (not an operand of those
    // products) by exp(cs_end - cs_j) dt_j, and dY scaled by exp(cs_i - ref)
    // into the XO tile (free since the mid-chunk product), for phase D (every
    // 16-byte chunk belongs to exactly one thread: row `row`, chunks 2wg, 2wg+1)
    uint4 xr[2], dyr[2];
    {
      const float sx = exp2f(end2 - s_cs2[base + row]) * s_dt[base + row];
      const float sy = exp2f(s_cs2[base + row] - ref2);
#pragma unroll
      for (int q4 = 0; q4 < 2; ++q4) {
        uint8_t* px = sX + sw128(row, wg * 2 + q4);
        xr[q4] = *(const uint4*)px;
        dyr[q4] = *(const uint4*)(sDY + sw128(row, wg * 2 + q4));
        float f[8];
        unpack8(xr[q4], f);
#pragma unroll
        for (int t = 0; t < 8; ++t) f[t] *= sx;
        store_row_bf16(sX, row, wg * 2 + q4, f);
        unpack8(dyr[q4], f);
#pragma unroll
        for (int t = 0; t < 8; ++t) f[t] *= sy;
        store_row_bf16(sXO, row, wg * 2 + q4, f);
      }
    }
    fence_async_smem();
    ok = wait_or_flag(&bar_mma, mma_phase);  // also publishes the scaled tiles
    mma_phase ^= 1;
    fence_after_sync();
    if (!ok) break;

    // ---- phase D: dC += (e o dY_k) Hin ; dB += (f o X_k) gout   (K = p)
    if (tid == 0) {
      const uint32_t id = idesc_bf16(128, 128, false, false);
      for (int kk = 0; kk < 4; ++kk) {
        mma_bf16(TdC, desc_sw128(smem_u32(sXO) + kk * 32, 16, 1024),
                 desc_sw128(smem_u32(sH) + kk * 32, 16, 1024), id, 1);
        mma_bf16(TdB, desc_sw128(smem_u32(sX) + kk * 32, 16, 1024),
                 desc_sw128(smem_u32(sG) + kk * 32, 16, 1024), id, 1);
      }
      mma_commit(&bar_mma);
    }

    // ---- epilogue of the head (overlaps phase D): dx, drive, e, statein, dD
    const float sgs = exp2f(end2 - s_cs2[I]);
    const float dtI = s_dt[I];
    float drive = 0.f, ej = 0.f, stin = 0.f, dd = 0.f;
    {
      float gx[16], gs[16], ch[16];
      tmem_ld16(T0 + lane_base + wg * 16, gx);
      tmem_ld16(T0 + lane_base + 64 + wg * 16, gs);
      tmem_ld16(T1 + lane_base + wg * 16, ch);
      tmem_wait_ld();
#pragma unroll
      for (int q4 = 0; q4 < 2; ++q4) {
        float xf[8], yf[8], o8[8];
        unpack8(xr[q4], xf);
        unpack8(dyr[q4], yf);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int m = q4 * 8 + t;
          const float gg = fmaf(sgs, gs[m], gx[m]);
          o8[t] = fmaf(dtI, gg, Dh * yf[t]);
          drive = fmaf(xf[t], gg, drive);
          ej = fmaf(xf[t], gs[m], ej);
          stin = fmaf(yf[t], ch[m], stin);
          dd = fmaf(yf[t], xf[t], dd);
        }
        store_row_bf16(sO, row, wg * 2 + q4, o8);  // dx staging: tile [128 rows][64 p]
      }
    }
    // dx is staged in sO (L o CB was last read by the Gx product), the
    // partials of warpgroups 1-3 16 KB further on
    float* ered = (float*)(sO + 16384);
    if (wg > 0) {
      ered[((wg - 1) * 4 + 0) * 128 + row] = drive;
      ered[((wg - 1) * 4 + 1) * 128 + row] = ej;
      ered[((wg - 1) * 4 + 2) * 128 + row] = stin;
      ered[((wg - 1) * 4 + 3) * 128 + row] = dd;
    }
    fence_async_smem();
    // phase D done (the barrier also publishes the dx staging and the
    // partials): dx goes out, X, dY, Hin, gout are free and the next head's
    // tiles go out now, under this head's dcs work (issued from warpgroup 3,
    // which has slack here, so that warpgroup 0's chain starts at once)
    ok = wait_or_flag(&bar_mma, mma_phase);
    mma_phase ^= 1;
    fence_after_sync();
    if (tid == 0) {
      tma_store_2d(&maps.dx, sO, h * d.P, row0);
      bulk_commit();
    }
    if (tid == kBwThreads - 128 && ok && hh + 1 < kh) issue_head_loads(u, h + 1, true);
    if (wg == 0) {
      // ---- dcs, its suffix sums (da), ddt, dA and dD partials: warpgroup 0,
      // one row per thread.  The end-of-block term (sum_j e_j + exp(cs_end -
      // ref) <gout, Hin>) sits at the last row, so it adds to every da_j: the
      // suffix sums run over dcs without it, with the totals of e and <g, H>
      // alongside.
      float hg = s_hg[0][row];
#pragma unroll
      for (int w = 0; w < 3; ++w) {
        rowsum += s_rs[w][row];
        drive += ered[(w * 4 + 0) * 128 + row];
        ej += ered[(w * 4 + 1) * 128 + row];
        stin += ered[(w * 4 + 2) * 128 + row];
        dd += ered[(w * 4 + 3) * 128 + row];
        hg += s_hg[w + 1][row];
      }
      ej *= sgs * dtI;
      stin *= exp2f(s_cs2[I] - ref2);
      float colsum = 0.f;
      for (int w = row >> 5; w < 4; ++w) colsum += s_col[w][row];
      // suffix sums within the warp (rows row .. 32 q + 31), then the later warps' totals
      float vd = rowsum - colsum + stin - ej, ve = ej, vh = hg;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float td = __shfl_down_sync(0xffffffffu, vd, o);
        const float te = __shfl_down_sync(0xffffffffu, ve, o);
        const float th = __shfl_down_sync(0xffffffffu, vh, o);
        if (lane + o < 32) {
          vd += td;
          ve += te;
          vh += th;
        }
      }
      if (lane == 0) s_wtot[q] = make_float4(vd, ve, vh, 0.f);
      named_sync(1, 128);
      float later = 0.f, esum = 0.f, hgsum = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float4 t = s_wtot[w];
        if (w > q) later += t.x;
        esum += t.y;
        hgsum += t.z;
      }
      const float da = (vd + later) + esum + exp2f(end2 - ref2) * hgsum;
      // ddt; raw-dt mode: the gradient w.r.t. dt_raw, ddt times sigmoid(dt_raw
      // + dt_bias) = 1 - exp(-dt) (dt being its softplus), with per-warp sums
      float gdt = drive + Ah * da;
      if (kRaw) {
        gdt *= -expm1f(-s_dt[I]);
        float gw = gdt;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) gw += __shfl_xor_sync(0xffffffffu, gw, o);
        if (lane == 0) s_gsum[q] = gw;
      }
      ddt[((size_t)crow + I) * d.H + h] = gdt;
      float pa = s_dt[I] * da, pd = dd;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        pa += __shfl_xor_sync(0xffffffffu, pa, o);
        pd += __shfl_xor_sync(0xffffffffu, pd, o);
      }
      if (lane == 0) s_wad[q] = make_float2(pa, pd);
      named_sync(1, 128);
      if (tid == 0) {
        const size_t slot = (((size_t)b * d.nc + c) * nblk + k) * d.H + h;
        dA_part[slot] = ((s_wad[0].x + s_wad[1].x) + s_wad[2].x) + s_wad[3].x;
        dD_part[slot] = ((s_wad[0].y + s_wad[1].y) + s_wad[2].y) + s_wad[3].y;
        if (kRaw) dtb_part[slot] = ((s_gsum[0] + s_gsum[1]) + s_gsum[2]) + s_gsum[3];
      }
    } else if (hh + 1 < kh) {
      // ---- meanwhile warpgroups 1-3 build the next head's tables
      if (wg >= 2) {
        cp_async_wait_all();
        const int r = tid - 256;
        if (kRaw && r < d.Q) s_dtn[r] = dt_of<kRaw>(d, s_dtn[r], h + 1);
      }
      build_tables((kRaw ? -expf(A_next) : A_next) * kLog2e, sync_wg123);
    }
    // ---- end of head: the next head's tables are published, and the dx
    // staging (sO) is free for the next head's L o CB or the final dC, dB sums
    if (tid == 0) bulk_wait_read0();
    __syncthreads();
  }

  // ---- dC and dB of the segment, summed over its heads in TMEM.
  // Warpgroup wg handles columns [32 wg, 32 wg + 32); dC first, then dB.
  // A split unit: each segment takes the unit's arrival ticket as it ends;
  // the last to arrive keeps its sums in TMEM and waits (bounded) for the
  // others' fp32 partials, which they write and then count in the unit's
  // written counter (`written`, after the arrival tickets).
  {
    const long long u0 = (long long)u * d.hpg;
    const int cta0 = cta_of(u0), nseg = cta_of(u0 + d.hpg - 1) - cta0 + 1;
    const int jc = wg;
    bool reducer = false;
    if (nseg > 1) {
      if (tid == 0) s_flag = atomicAdd(&tickets[1 + u], 1u) == (unsigned int)(nseg - 1);
      __syncthreads();
      reducer = s_flag != 0;
      if (!reducer) {
        // fp32 partial in this CTA's slot (0 for its first segment, 1 for its
        // last), float4 i4 of every thread contiguous: [which][i4][thread]
        float4* pslot = (float4*)(part + ((size_t)blockIdx.x * 2 + (first_seg ? 0 : 1)) * 32768);
        if (ok) {
#pragma unroll 1
          for (int which = 0; which < 2; ++which) {
            float v[32];
            tmem_ld32((which ? TdB : TdC) + lane_base + jc * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4)
              pslot[(which * 8 + i4) * kBwThreads + tid] =
                  make_float4(v[4 * i4], v[4 * i4 + 1], v[4 * i4 + 2], v[4 * i4 + 3]);
          }
        }
        __syncthreads();
        if (tid == 0) {
          __threadfence();
          atomicAdd(written + u, 1u);
        }
      } else if (tid == 0) {
        // (a wait that gives up sets the error word; the sums are then wrong)
        if (!wait_count_at_least(written + u, (unsigned int)(nseg - 1))) atomicOr(&g_tc_error, 1u);
        __threadfence();
      }
      if (reducer) __syncthreads();
    }
    // the unit's output: a single segment from TMEM, else by its last segment
    // as the sum over the segments in order (its own from TMEM, the others'
    // partials); bf16 -> staging in sO (dead since the last head's Gx
    // product) -> TMA store, dC then dB
    const bool write_out = ok && (nseg == 1 || reducer);
    if (write_out) {
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        float v[32];
        if (nseg == 1) {
          tmem_ld32((which ? TdB : TdC) + lane_base + jc * 32, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
#pragma unroll 1
          for (int j = 0; j < nseg; ++j) {
            const int cj = cta0 + j;
            if (cj == (int)blockIdx.x) {
              float t[32];
              tmem_ld32((which ? TdB : TdC) + lane_base + jc * 32, t);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] += t[i];
            } else {
              // slot 0 unless the unit starts inside that CTA's range
              const int side = (j == 0 && split.first[cj] < u0) ? 1 : 0;
              const float4* q = (const float4*)(part + ((size_t)cj * 2 + side) * 32768);
#pragma unroll
              for (int i4 = 0; i4 < 8; ++i4) {
                const float4 f = __ldcg(q + (which * 8 + i4) * kBwThreads + tid);
                v[4 * i4] += f.x;
                v[4 * i4 + 1] += f.y;
                v[4 * i4 + 2] += f.z;
                v[4 * i4 + 3] += f.w;
              }
            }
          }
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int nn = jc * 32 + q4 * 8;
          store_row_bf16(sO + (nn >> 6) * 16384, row, (nn & 63) >> 3, &v[q4 * 8]);
        }
        fence_async_smem();
        __syncthreads();
        if (tid == 0) {
          const CUtensorMap* m = which ? &maps.dB : &maps.dC;
          tma_store_2d(m, sO, g * d.N, row0);
          tma_store_2d(m, sO + 16384, g * d.N + 64, row0);
          bulk_commit();
          bulk_wait_read0();  // sO is rewritten by dB, then by the next W build
        }
        __syncthreads();
      }
    }
    // TMEM accumulators and the ticket flag are reused by the next segment
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
  }
  x += kh;
  }
  grid_dep_launch();
  grid_dep_wait();  // (a CTA without items has not waited yet; the tickets are zeroed before)
  if (tid == 0) bulk_wait0();
  fence_before_sync();
  __syncthreads();
  if (tid < 32) tmem_dealloc(tm, 512);

  // ---- the last CTA to finish sums the dA, dD partials of every (b, chunk,
  // block) per head, in a fixed order (lane-strided sums, then a butterfly)
  if (tid == 0) {
    __threadfence();  // this CTA's partials before its ticket
    s_flag = atomicAdd(&tickets[0], 1u) == gridDim.x - 1u;
  }
  __syncthreads();
  if (s_flag) {
    __threadfence();
    const int nparts = d.B * d.nc * nblk;
    // raw-dt mode: dA goes out as the gradient w.r.t. a_log (dA times A), and
    // the dt_raw gradient sums as the gradient w.r.t. dt_bias
    for (int hr = tid >> 5; hr < d.H; hr += kBwThreads / 32) {
      float sa = 0.f, sd = 0.f, sb = 0.f;
      for (int kk = lane; kk < nparts; kk += 32) {
        sa += __ldcg(dA_part + (size_t)kk * d.H + hr);
        sd += __ldcg(dD_part + (size_t)kk * d.H + hr);
        if (kRaw) sb += __ldcg(dtb_part + (size_t)kk * d.H + hr);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        sa += __shfl_xor_sync(0xffffffffu, sa, o);
        sd += __shfl_xor_sync(0xffffffffu, sd, o);
        if (kRaw) sb += __shfl_xor_sync(0xffffffffu, sb, o);
      }
      if (lane == 0) {
        dA[hr] = kRaw ? sa * a_of<kRaw>(d, A, hr) : sa;
        dD[hr] = sd;
        if (kRaw) d_dt_bias[hr] = sb;
      }
    }
  }
}

// Reverse state pass of the tensor-core backward.  Per (b, h) and a tile of
// 16 columns n, walks the chunks from last to first: g_c (gradient of the
// state at the end of chunk c) = exp(cs_last[c+1]) g_{c+1} + R_{c+1}, g_{nc-1}
// = 0, dh0 = exp(cs_last[0]) g_0 + R_0.  Writes g_c and the chunk-start state
// H_{c-1} (read from the history) as bf16 rows n x 64 p ([b][c][h][n][p]),
// the operand layout of k_bwd_tc, through a shared-memory transpose.
__global__ void __launch_bounds__(256)
k_state_pass_bwd_t(TcDims d, unsigned int* __restrict__ tickets, int ntickets,
                   const float* __restrict__ R,
                   const float* __restrict__ hist,
                   const float* __restrict__ cs_last, __nv_bfloat16* __restrict__ gT,
                   __nv_bfloat16* __restrict__ hT, float* __restrict__ dh0) {
  __shared__ __align__(16) __nv_bfloat16 s_g[16][72];  // [n][p], padded rows
  __shared__ __align__(16) __nv_bfloat16 s_h[16][72];
  const int nt = blockIdx.x, h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
  const int p = tid >> 2, n4 = (tid & 3) * 4;  // this thread: row p, columns n0 + n4 .. + 3
  const int n0 = nt * 16;
  const int PN = d.P * d.N;
  const size_t bh = (size_t)b * d.H + h;
  const float* cl = cs_last + bh * d.nc;
  auto at = [&](int c) { return (((size_t)b * d.nc + c) * d.H + h) * (size_t)PN + (size_t)p * d.N + n0 + n4; };
  float4 gc = make_float4(0.f, 0.f, 0.f, 0.f);
  const int last = d.nc - 1;
  // the next kDepth chunks' R_c, H_{c-1} and decay totals in flight in a
  // register ring while one chunk is updated
  constexpr int kDepth = 4;
  float4 r_ring[kDepth], h_ring[kDepth];
  float l_ring[kDepth];
#pragma unroll
  for (int k = 0; k < kDepth; ++k)
    if (last - k >= 0) {
      r_ring[k] = *(const float4*)(R + at(last - k));
      h_ring[k] = *(const float4*)(hist + at(last - k));
      l_ring[k] = cl[last - k];
    }
  for (int i0 = 0; i0 <= last; i0 += kDepth) {
#pragma unroll
  for (int k = 0; k < kDepth; ++k) {
    const int c = last - (i0 + k);
    if (c < 0) break;  // uniform over the CTA
    const float4 r = r_ring[k], hv = h_ring[k];
    const float lc = l_ring[k];
    if (c - kDepth >= 0) {  // refill the slot with chunk c - depth
      r_ring[k] = *(const float4*)(R + at(c - kDepth));
      h_ring[k] = *(const float4*)(hist + at(c - kDepth));
      l_ring[k] = cl[c - kDepth];
    }
    __syncthreads();  // previous chunk's rows are written out
    s_g[n4 + 0][p] = __float2bfloat16_rn(gc.x);
    s_g[n4 + 1][p] = __float2bfloat16_rn(gc.y);
    s_g[n4 + 2][p] = __float2bfloat16_rn(gc.z);
    s_g[n4 + 3][p] = __float2bfloat16_rn(gc.w);
    s_h[n4 + 0][p] = __float2bfloat16_rn(hv.x);
    s_h[n4 + 1][p] = __float2bfloat16_rn(hv.y);
    s_h[n4 + 2][p] = __float2bfloat16_rn(hv.z);
    s_h[n4 + 3][p] = __float2bfloat16_rn(hv.w);
    __syncthreads();
    {
      // 16 rows x 64 p bf16 = 16 x 8 chunks of 16 bytes per tile
      const int t = tid & 127, rr = t >> 3, ch = t & 7;
      const size_t orow = ((((size_t)b * d.nc + c) * d.H + h) * d.N + n0 + rr) * d.P + ch * 8;
      if (tid < 128) *(uint4*)(gT + orow) = *(const uint4*)&s_g[rr][ch * 8];
      else *(uint4*)(hT + orow) = *(const uint4*)&s_h[rr][ch * 8];
    }
    const float e = expf(lc);
    gc.x = fmaf(e, gc.x, r.x);
    gc.y = fmaf(e, gc.y, r.y);
    gc.z = fmaf(e, gc.z, r.z);
    gc.w = fmaf(e, gc.w, r.w);
  }
  }
  if (dh0) *(float4*)(dh0 + bh * PN + (size_t)p * d.N + n0 + n4) = gc;
  // completion counters of the backward kernel that follows
  for (int i = ((b * (int)gridDim.y + h) * (int)gridDim.x + nt) * 256 + tid; i < ntickets;
       i += (int)(gridDim.x * gridDim.y * gridDim.z) * 256)
    tickets[i] = 0u;
}

// ---------------------------------------------------------------------------
// Host side: tensor maps through the driver entry point (no libcuda link).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  });
  return fn;
}

// 2D bf16 row-major [rows][cols] map with a {64, box_rows} SW128 box.
bool map_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D fp32 row-major [rows][cols] map with a {box_cols, box_rows} SW128 box
// (box_cols * 4 = 128 bytes).
bool map_f32(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
             uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 4};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

TcDims tc_dims(const Problem& p) {
  return TcDims{p.B, p.T, p.H, p.P, p.N, p.G, p.Q, p.nc, p.hpg, p.dt_bias, p.a_log};
}

template <typename K>
cudaError_t set_smem_tc(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// Launch with programmatic stream serialization: the kernel may start while
// the kernel ahead of it on the stream finishes; it waits for that kernel
// (griddepcontrol.wait) before touching anything the earlier kernels write.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace

bool encode_rows_2d(CUtensorMap* m, const void* base, bool bf16, uint64_t rows, uint64_t cols,
                    uint32_t box_cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const uint64_t esz = bf16 ? 2 : 4;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * esz};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
            const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int g_force_path = -1;  // -1 automatic, 0 SIMT only

bool tc_supported(const Problem& p) {
  if (g_force_path == 0) return false;
  return p.bf16 && p.P == 64 && p.N == 128 && (p.Q == 128 || p.Q == 256) && encode_fn() != nullptr;
}

void tc_force_path(int path) { g_force_path = path; }

bool tc_forced_simt() { return g_force_path == 0; }

bool tc_backward_supported(const Problem& p) { return tc_supported(p); }

// S_c (mode 0, from x and B) or R_c (mode 1, from dy and C) into `out`; cs_last.
cudaError_t tc_chunk_outer(const Problem& p, int mode, float* out) {
  OuterMaps maps;
  const void* u = mode == 0 ? p.x : p.dy;
  const void* v = mode == 0 ? p.Bm : p.Cm;
  if (!map_bf16(&maps.u, u, (uint64_t)p.B * p.T, (uint64_t)p.H * p.P, p.Q) ||
      !map_bf16(&maps.v, v, (uint64_t)p.B * p.T, (uint64_t)p.G * p.N, p.Q) ||
      !map_f32(&maps.o, out, (uint64_t)p.B * p.nc * p.H * p.P, (uint64_t)p.N, 32, 64))
    return cudaErrorInvalidValue;
  const size_t smem = 3 * (size_t)p.Q * 128 + 1024;
  const TcDims d = tc_dims(p);
  cudaError_t e;
  if (mode == 0) {
    if ((e = set_smem_tc(k_chunk_outer_tc<0>, smem)) != cudaSuccess) return e;
    LaunchScope ls("chunk_state_tc", p.stream);
    k_chunk_outer_tc<0><<<dim3(p.nc, p.H, p.B), 256, smem, p.stream>>>(maps, d, p.dt, p.A,
                                                                              out, p.cs_last);
  } else {
    if ((e = set_smem_tc(k_chunk_outer_tc<1>, smem)) != cudaSuccess) return e;
    LaunchScope ls("chunk_dstate_tc", p.stream);
    k_chunk_outer_tc<1><<<dim3(p.nc, p.H, p.B), 256, smem, p.stream>>>(maps, d, p.dt, p.A,
                                                                              out, p.cs_last);
  }
  return cudaGetLastError();
}

// Whether the fused per-(b, h) state scans have enough CTAs to fill the GPU.
bool tc_fused_states(const Problem& p) {
  int nsm = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  return (long)p.B * p.H * 4 >= 3L * nsm;
}

template <int MODE>
cudaError_t tc_state_scan(const Problem& p, const char* name, float* final_or_dh0) {
  ScanStateMaps maps;
  const void* u = MODE == 0 ? p.x : p.dy;
  const void* v = MODE == 0 ? p.Bm : p.Cm;
  const uint64_t srows = (uint64_t)p.B * p.nc * p.H * p.N;
  if (!map_bf16(&maps.u, u, (uint64_t)p.B * p.T, (uint64_t)p.H * p.P, p.Q) ||
      !map_bf16(&maps.v, v, (uint64_t)p.B * p.T, (uint64_t)p.G * p.N, p.Q) ||
      !map_bf16(&maps.rows, MODE == 0 ? p.hT : p.gT, srows, (uint64_t)p.P, 128) ||
      !map_bf16(&maps.rows2, p.hT, srows, (uint64_t)p.P, 128) ||
      !map_bf16(&maps.rows3, MODE == 1 && p.gmT ? p.gmT : p.hT, srows, (uint64_t)p.P, 128))
    return cudaErrorInvalidValue;
  // two pipeline stages of tiles + the bf16 row staging tile(s)
  const size_t smem = 2 * 3 * (size_t)p.Q * 128 + (MODE == 1 ? 2 : 1) * 16384 + 1024;
  auto kern = p.dt_bias ? k_state_scan_tc<MODE, true> : k_state_scan_tc<MODE, false>;
  cudaError_t e = set_smem_tc(kern, smem);
  if (e != cudaSuccess) return e;
  {
    LaunchScope ls(name, p.stream);
    e = launch_pdl(kern, dim3(p.H, p.B), dim3(kScanThreads), smem, p.stream, maps,
                   tc_dims(p), p.dt, p.A, p.h0, p.hist, final_or_dh0,
                   MODE == 1 ? p.tickets : (unsigned int*)nullptr, p.ntickets,
                   (int)(MODE == 1 && p.Q == 256 && p.gmT != nullptr));
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t tc_forward_states(const Problem& p) {
  return tc_state_scan<0>(p, "state_scan_fwd_tc", p.final_state);
}

cudaError_t tc_forward_scan(const Problem& p) {
  ScanMaps maps;
  const uint64_t rows = (uint64_t)p.B * p.T;
  if (!map_bf16(&maps.x, p.x, rows, (uint64_t)p.H * p.P, 128) ||
      !map_bf16(&maps.B, p.Bm, rows, (uint64_t)p.G * p.N, 128) ||
      !map_bf16(&maps.C, p.Cm, rows, (uint64_t)p.G * p.N, 128) ||
      !map_bf16(&maps.y, p.y, rows, (uint64_t)p.H * p.P, 128))
    return cudaErrorInvalidValue;
  const size_t smem = kScanBytes + 1024;
  cudaError_t e = set_smem_tc(k_fwd_scan_tc, smem);
  if (e != cudaSuccess) return e;
  {
    LaunchScope ls("chunk_scan_tc", p.stream);
    e = launch_pdl(k_fwd_scan_tc, dim3(p.nc, p.H, p.B), dim3(256), smem, p.stream, maps,
                   tc_dims(p), p.dt, p.A, p.D, p.hist);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t tc_forward_single(const Problem& p) {
  ScanMaps maps;
  const uint64_t rows = (uint64_t)p.B * p.T;
  if (!map_bf16(&maps.x, p.x, rows, (uint64_t)p.H * p.P, 128) ||
      !map_bf16(&maps.B, p.Bm, rows, (uint64_t)p.G * p.N, 128) ||
      !map_bf16(&maps.C, p.Cm, rows, (uint64_t)p.G * p.N, 128) ||
      !map_bf16(&maps.y, p.y, rows, (uint64_t)p.H * p.P, 128))
    return cudaErrorInvalidValue;
  const size_t nflags = (size_t)p.B * p.nc * p.H + 1;
  cudaError_t e = cudaMemsetAsync(p.fwd_flags, 0, nflags * sizeof(unsigned int), p.stream);
  if (e != cudaSuccess) return e;
  const size_t smem = kScanBytes + 1024;
  auto kern = p.dt_bias ? k_fwd_single_tc<true> : k_fwd_single_tc<false>;
  if ((e = set_smem_tc(kern, smem)) != cudaSuccess) return e;
  // resident CTAs, two per SM, each looping over tiles from the counter
  int nsm = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  const long long ntiles = (long long)(nflags - 1);
  const unsigned grid = (unsigned)(ntiles < 2LL * nsm ? ntiles : 2LL * nsm);
  {
    LaunchScope ls("fwd_single_tc", p.stream);
    kern<<<grid, 256, smem, p.stream>>>(maps, tc_dims(p), p.dt, p.A, p.D, p.h0, p.hist,
                                        p.final_state, p.fwd_flags);
  }
  return cudaGetLastError();
}

cudaError_t tc_backward(const Problem& p) {
  cudaError_t e;
  // the fused state scan also writes the mid-chunk state gradients of
  // 256-step chunks, which the backward then reads instead of forming them
  const bool fused = tc_fused_states(p), gmid = fused && p.Q == 256 && p.gmT != nullptr;
  if (fused) {
    if ((e = tc_state_scan<1>(p, "state_scan_bwd_tc", p.dh0)) != cudaSuccess) return e;
  } else {
    if ((e = tc_chunk_outer(p, 1, p.dstate)) != cudaSuccess) return e;
    {
      LaunchScope ls("state_pass_bwd_tc", p.stream);
      k_state_pass_bwd_t<<<dim3(p.N / 16, p.H, p.B), 256, 0, p.stream>>>(
          tc_dims(p), p.tickets, p.ntickets, p.dstate, p.hist, p.cs_last, (__nv_bfloat16*)p.gT, (__nv_bfloat16*)p.hT,
          p.dh0);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  BwdMaps maps;
  const uint64_t rows = (uint64_t)p.B * p.T;
  const uint64_t srows = (uint64_t)p.B * p.nc * p.H * p.N;
  if (!map_bf16(&maps.x, p.x, rows, (uint64_t)p.H * p.P, 128) ||
      !map_bf16(&maps.dy, p.dy, rows, (uint64_t)p.H * p.P, 128) ||
      !map_bf16(&maps.B, p.Bm, rows, (uint64_t)p.G * p.N, 128) ||
      !map_bf16(&maps.C, p.Cm, rows, (uint64_t)p.G * p.N, 128) ||
      !map_bf16(&maps.dx, p.dx, rows, (uint64_t)p.H * p.P, 128) ||
      !map_bf16(&maps.dB, p.dB, rows, (uint64_t)p.G * p.N, 128) ||
      !map_bf16(&maps.dC, p.dC, rows, (uint64_t)p.G * p.N, 128) ||
      !map_bf16(&maps.ht, p.hT, srows, (uint64_t)p.P, 128) ||
      !map_bf16(&maps.gt, p.gT, srows, (uint64_t)p.P, 128) ||
      !map_bf16(&maps.gmt, gmid ? p.gmT : p.gT, srows, (uint64_t)p.P, 128))
    return cudaErrorInvalidValue;
  const size_t smem = kBwBytes + 1024;
  auto kern = p.dt_bias ? k_bwd_tc<true> : k_bwd_tc<false>;
  if ((e = set_smem_tc(kern, smem)) != cudaSuccess) return e;
  const int nblk = p.Q / 128;
  // one CTA per SM (at most kBwdMaxCtas, at most one per item), each taking an
  // equal contiguous range of the (unit, head) items
  int nsm = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  const long long nitems = (long long)p.B * p.G * p.nc * nblk * p.hpg;
  long long ncta = nsm < (int)kBwdMaxCtas ? nsm : (long long)kBwdMaxCtas;
  // every range at least as heavy as the heaviest item, so that no CTA is
  // left without items (a unit's segments are then its CTAs cta_of(first) ..
  // cta_of(last))
  const long long wmax = nblk == 2 ? kBwW1 : kBwW0;
  const long long wtot = bw_weight_before(nitems, p.hpg, nblk);
  if (ncta > wtot / wmax) ncta = wtot / wmax;
  if (nitems > INT_MAX) return cudaErrorInvalidValue;
  BwdSplit split;
  for (long long c = 0; c <= ncta; ++c) {  // the least item whose CTA is c or later
    long long lo = 0, hi = nitems;
    while (lo < hi) {
      const long long m = (lo + hi) >> 1;
      if (bw_weight_before(m, p.hpg, nblk) * ncta / wtot >= c)
        hi = m;
      else
        lo = m + 1;
    }
    split.first[c] = (int)lo;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ncta, 1, 1);
  cfg.blockDim = dim3(kBwThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = p.stream;
  cudaLaunchAttribute attr[1];
  // may start while the state pass ahead of it finishes (see launch_pdl)
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  {
    LaunchScope ls("bwd_tc", p.stream);
    e = cudaLaunchKernelEx(&cfg, kern, maps, split, tc_dims(p), nitems, p.dt, p.A, p.D, p.ddt,
                           p.dA_part, p.dD_part, p.dtb_part, p.d_dt_bias, p.dB, p.dC, p.dA, p.dD,
                           p.tickets, p.tickets + 1 + nitems / p.hpg, p.bwd_part, (int)gmid);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// One CTA waits on an mbarrier that nothing arrives on; the bounded wait gives
// up after kWaitLimitNs and sets the device error word.  Exercises the
// timeout path without faulting or hanging the GPU.
__global__ void k_selftest_wait() {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  (void)wait_or_flag(&bar, 0);
}

cudaError_t tc_selftest_timeout(cudaStream_t s) {
  {
    LaunchScope ls("selftest_wait", s);
    k_selftest_wait<<<1, kTcThreads, 0, s>>>();
  }
  return cudaGetLastError();
}

cudaError_t tc_read_and_clear_error(unsigned int* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_tc_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(unsigned int));
}

}  // namespace ssd
