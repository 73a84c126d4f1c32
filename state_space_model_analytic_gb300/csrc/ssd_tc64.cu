// Tensor-core (tcgen05 / TMEM) kernels of the chunked SSD core on 128-step
// blocks: headdim P = 64 with d_state N = 64 (fp32 or bf16 storage) or
// N = 128 (bf16), and P = 128 with N = 64 or 128 (bf16); any chunk Q in {16, 32,
// 64, 128} (seqlen a multiple of 128), and Q = 256 run by the host as
// 128-step sub-chunks (tc64_sub_problem).  A bf16 row of 128 values occupies
// the bytes of an fp32 row of 64 carried as two bf16 tiles, so the 128-wide
// operands of the bf16 shapes take the lo tiles' places of the fp32 layout.
//
// Blocks.  The chunk scan and the backward work on blocks of 128 steps (the
// MMA M size).  A block holds 128 / Q whole chunks; inside it the decays are
// block-local cumulative sums, which is exact (chunking is a regrouping of
// the recurrence), and the block's start state is the history entry of its
// first chunk.  The chunk-state kernel and the state passes work per chunk,
// as the history is defined per chunk.
//
// Split products (fp32 storage).  Every fp32 operand a is carried as two
// bf16 tiles,
//     hi = bf16(a),  lo = bf16(a - hi),
// so a = hi + lo + r with |r| <= 2^-18 |a|, and every product as three bf16
// MMAs accumulated in fp32 TMEM:
//     A B ~ Ah Bh + Ah Bl + Al Bh,
// dropping Al Bl and the remainders (each at most about 2^-18 |A||B| per
// term).  bf16 storage uses the hi tiles alone and one MMA per product, like
// the bf16 kernels of ssd_tc.cu.  The layouts are those kernels' (128-byte
// swizzled rows of 64 bf16).  Inputs come from global memory by coalesced
// 16-byte loads and are converted by the threads; elementwise math (decays,
// masks, epilogues) runs in fp32; the epilogues read x and dy back from the
// tiles (hi + lo: within 2^-18 of the stored fp32 value; exact for bf16).
//
// The chunked algebra is that of the SIMT kernels (ssd_simt.cu), derived from
// the recurrence of `ssd_forward_state_history_reference` and the reverse-time
// adjoint of `ssd_backward_reference` (burn_dragon_kernel 0.5.0,
// src/sequence/mamba2/backward.rs).  Kernels:
//   k_outer64<0>  S_c = sum_j exp(cs_last - cs_j) dt_j x_j B_j^T       (b, c, h)
//   k_outer64<1>  R_c = sum_i exp(cs_i) dy_i C_i^T                      (b, c, h)
//   k_scan64      y_i = sum_{j<=i} exp(cs_i-cs_j) dt_j (C_i.B_j) x_j
//                       + exp(cs_i) H_in C_i + D x_i                    (b, block, h)
//   k_bwd64_x     dx, d(dt), and the per-(b, block) partials of dA, dD  (b, block, h)
//   k_bwd64_bc    dC, dB of a (b, block, g) unit over a segment of its heads:
//                 W = sum_h exp(cs_i-cs_j) dt_j (dy_i.x_j) (summed over the
//                 segment's heads in registers), then W B, W^T C, plus the
//                 state terms sum_h (e o dY) H and sum_h (f o X) g
//   k_sum64_bc    the segments' dC, dB partials summed in segment order
// The state passes between them are the SIMT ones (fp32, sequential over
// chunks).  Every wait is bounded; a wait that gives up sets a device error
// word and the kernel finishes without touching the guarded data.
#include <cuda.h>
#include <cuda_bf16.h>

#include <type_traits>

#include "ssd_common.cuh"
#include "ssd_internal.h"
#include "tc_util.cuh"

namespace ssd {

using namespace tc;

bool tc_forced_simt();

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr int kQ = 128;  // rows of a block (the MMA M size)

__device__ unsigned int g_tc64_error;

__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity) {
  const bool mine = mbar_wait(bar, parity, kWaitLimitNs);
  const bool all = __syncthreads_and(mine) != 0;
  if (!all && threadIdx.x == 0) atomicOr(&g_tc64_error, 1u);
  return all;
}

struct D64 {
  int B, T, H, G, nc, hpg;
  int Q, nb, cpb;  // chunk size, 128-row blocks, chunks per block
};

// storage element type
template <bool kBf>
using Elem = typename std::conditional<kBf, __nv_bfloat16, float>::type;

// ---- split tiles ----------------------------------------------------------
// 8 consecutive values of one tile row as (hi, lo) bf16 chunks at byte offset
// `off` of the hi and lo tiles (kBf: the hi chunk only).
template <bool kBf = false>
__device__ __forceinline__ void store_split8(uint8_t* hi, uint8_t* lo, uint32_t off,
                                             const float* v) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const __nv_bfloat16 a = __float2bfloat16_rn(v[2 * t]);
    const __nv_bfloat16 b = __float2bfloat16_rn(v[2 * t + 1]);
    h[t] = pack_bf16(__bfloat162float(a), __bfloat162float(b));
    if (!kBf)
      l[t] = pack_bf16(v[2 * t] - __bfloat162float(a), v[2 * t + 1] - __bfloat162float(b));
  }
  *(uint4*)(hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
  if (!kBf) *(uint4*)(lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
}

// 8 consecutive fp32 values
struct Raw8 {
  float4 a, b;
};
__device__ __forceinline__ Raw8 ld8(const float* p) {
  return Raw8{__ldg((const float4*)p), __ldg((const float4*)p + 1)};
}
__device__ __forceinline__ void unpack8_bf16(const uint4& u, float* f) {
  const __nv_bfloat162* q = (const __nv_bfloat162*)&u;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float2 x = __bfloat1622float2(q[t]);
    f[2 * t] = x.x;
    f[2 * t + 1] = x.y;
  }
}
__device__ __forceinline__ void unpack_raw(const Raw8& r, float* f) {
  f[0] = r.a.x; f[1] = r.a.y; f[2] = r.a.z; f[3] = r.a.w;
  f[4] = r.b.x; f[5] = r.b.y; f[6] = r.b.z; f[7] = r.b.w;
}
// 8 values to storage at p (16 or 32 bytes)
__device__ __forceinline__ void st8(float* p, const float* f) {
  ((float4*)p)[0] = make_float4(f[0], f[1], f[2], f[3]);
  ((float4*)p)[1] = make_float4(f[4], f[5], f[6], f[7]);
}
__device__ __forceinline__ void st8(__nv_bfloat16* p, const float* f) {
  *(uint4*)p = make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]),
                          pack_bf16(f[6], f[7]));
}

// One thread's share of rows [0, nrows) (nrows <= ROWS) of a 64-wide slab
// (row r at src + r * stride elements), fetched into registers by fetch()
// and written into split tiles (rows of 64 bf16, SW128) by put(), each value
// times scale(r).  Separate phases let a kernel keep the next tile's loads
// in flight while it converts the current one.
// W = 128 (bf16 storage only): the row's second 64 values go to a second
// tile at the lo tile's place (a bf16 row of 128 takes the bytes of an fp32
// row of 64 split in two).
template <int NT, int ROWS, typename E, int W = 64>
struct RowTile {
  static constexpr bool kBf = std::is_same<E, __nv_bfloat16>::value;
  static_assert(W == 64 || (W == 128 && kBf), "128-wide rows are bf16 only");
  static constexpr int kCh = W / 8;  // 16-byte chunks of bf16 per row
  static constexpr int kPer = ROWS * kCh / NT;
  // bf16 values stay packed (4 registers per 8 values) until put()
  typename std::conditional<kBf, uint4, Raw8>::type v[kPer];
  __device__ __forceinline__ void fetch(const E* __restrict__ src, size_t stride,
                                        int nrows = ROWS) {
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int e = threadIdx.x + NT * k, r = e / kCh, ch = e % kCh;
      if (r < nrows) {
        if constexpr (kBf)
          v[k] = __ldg((const uint4*)(src + (size_t)r * stride + ch * 8));
        else
          v[k] = ld8(src + (size_t)r * stride + ch * 8);
      }
    }
  }
  template <typename F>
  __device__ __forceinline__ void put(uint8_t* hi, uint8_t* lo, F&& scale, int nrows = ROWS) {
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int e = threadIdx.x + NT * k, r = e / kCh, ch = e % kCh;
      if (r >= nrows) continue;
      const float sc = scale(r);
      float f[8];
      if constexpr (kBf)
        unpack8_bf16(v[k], f);
      else
        unpack_raw(v[k], f);
#pragma unroll
      for (int t = 0; t < 8; ++t) f[t] *= sc;
      if (W == 64)
        store_split8<kBf>(hi, lo, sw128(r, ch), f);
      else
        store_split8<true>((ch >> 3) ? lo : hi, nullptr, sw128(r, ch & 7), f);
    }
  }
};

// 8 values of a split tile row as fp32: hi + lo (hi alone for bf16 storage,
// where it holds the stored value exactly; for fp32 the sum is within 2^-18
// of it)
template <bool kBf>
__device__ __forceinline__ void read_split8(const uint8_t* hi, const uint8_t* lo, uint32_t off,
                                            float* f) {
  unpack8_bf16(*(const uint4*)(hi + off), f);
  if (!kBf) {
    float g[8];
    unpack8_bf16(*(const uint4*)(lo + off), g);
#pragma unroll
    for (int t = 0; t < 8; ++t) f[t] += g[t];
  }
}

// A [64 p][NS n] fp32 state block as rows p into tiles: split for fp32
// storage (NS = 64), bf16 for bf16 storage (NS = 128: n 64-127 in a second
// tile at the lo tile's place).
template <int NT, int NS, bool kBf, int PR = 64>
struct StateRowTile {
  static_assert(NS == 64 || (NS == 128 && kBf), "d_state 128 is bf16 only");
  static_assert(PR == 64 || (PR == 128 && kBf), "headdim 128 is bf16");
  static constexpr int kCh = NS / 8;
  // PR = 128: rows 64-127 follow rows 0-63; with NS = 128 the n 64-127 block
  // (PR rows) is at the lo pointer
  static constexpr int kPer = PR * kCh / NT;
  Raw8 v[kPer];
  __device__ __forceinline__ void fetch(const float* __restrict__ src) {
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int e = threadIdx.x + NT * k, r = e / kCh, ch = e % kCh;
      v[k] = ld8(src + (size_t)r * NS + ch * 8);
    }
  }
  __device__ __forceinline__ void put(uint8_t* hi, uint8_t* lo) {
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int e = threadIdx.x + NT * k, r = e / kCh, ch = e % kCh;
      float f[8];
      unpack_raw(v[k], f);
      if (NS == 64)
        store_split8<kBf>(hi, lo, sw128(r, ch), f);
      else
        store_split8<true>((ch >> 3) ? lo : hi, nullptr, sw128(r, ch & 7), f);
    }
  }
};

// fetch, then put (no overlap)
template <int NT, int ROWS, typename E, typename F>
__device__ __forceinline__ void load_split(uint8_t* hi, uint8_t* lo, const E* __restrict__ src,
                                           size_t stride, F&& scale, int nrows = ROWS) {
  RowTile<NT, ROWS, E, 64> t;
  t.fetch(src, stride, nrows);
  t.put(hi, lo, scale, nrows);
}

// Rows [0, ROWS) of split tiles rescaled in place: each row r times scale(r),
// from the value the tiles hold (hi + lo, or hi alone for bf16 storage).
template <int NT, int ROWS, bool kBf, int W = 64, typename F>
__device__ __forceinline__ void rescale_split(uint8_t* hi, uint8_t* lo, F&& scale) {
  static_assert(W == 64 || (W == 128 && kBf), "128-wide rows are bf16 only");
  constexpr int kCh = W / 8;
  constexpr int kPer = ROWS * kCh / NT;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int e = threadIdx.x + NT * k, r = e / kCh, cw = e % kCh, ch = cw & 7;
    // the row's second 64 values (W = 128, bf16 only) are in the lo tile's place
    uint8_t* th = W == 128 && (cw >> 3) ? lo : hi;
    const uint32_t off = sw128(r, ch);
    float f[8], g[8];
    unpack8_bf16(*(const uint4*)(th + off), f);
    if (!kBf) {
      unpack8_bf16(*(const uint4*)(lo + off), g);
#pragma unroll
      for (int t = 0; t < 8; ++t) f[t] += g[t];
    }
    const float sc = scale(r);
#pragma unroll
    for (int t = 0; t < 8; ++t) f[t] *= sc;
    store_split8<kBf>(th, lo, off, f);
  }
}

// A [PS p][NS n] fp32 state block (p-major) transposed into split tiles of
// rows n with 64 p each; NS = 128 (bf16 only): rows 64-127 follow rows 0-63;
// PS = 128 (bf16 only): p 64-127 go to a second tile of NS rows at the lo
// pointer.  Returns this thread's share of sum(src * other) when `other`
// is given (the same elements of a second block, for <g, H>).
template <int NT, bool kBf, int NS = 64, int PS = 64>
__device__ __forceinline__ float load_split_transposed(uint8_t* hi, uint8_t* lo,
                                                       const float* __restrict__ src,
                                                       const float* __restrict__ other) {
  static_assert(NS == 64 || (NS == 128 && kBf), "d_state 128 is bf16 only");
  static_assert(PS == 64 || (PS == 128 && kBf), "headdim 128 is bf16");
  constexpr int kPer = NS * (PS / 8) / NT;
  float dot = 0.f;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int e = threadIdx.x + NT * k, n = e % NS, pc = e / NS;
    float f[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) f[t] = __ldg(src + (size_t)(pc * 8 + t) * NS + n);
    if (other) {
#pragma unroll
      for (int t = 0; t < 8; ++t) dot = fmaf(f[t], __ldg(other + (size_t)(pc * 8 + t) * NS + n), dot);
    }
    if (PS == 64)
      store_split8<kBf>(hi, lo, sw128(n, pc), f);
    else
      store_split8<true>((pc >> 3) ? lo : hi, nullptr, sw128(n, pc & 7), f);
  }
  return dot;
}

// D (+)= A B over the split tiles (lo tiles at the given byte distance from
// the hi tiles): three bf16 MMAs, or one (kBf: the hi tiles hold the
// operands exactly).
template <bool kBf>
__device__ __forceinline__ void mma3(uint32_t d, uint32_t a_hi, uint32_t a_lo_off, uint32_t a_lbo,
                                     bool a_mn, uint32_t b_hi, uint32_t b_lo_off, uint32_t b_lbo,
                                     uint32_t idesc, uint32_t acc) {
  (void)a_mn;
  const uint64_t ah = desc_sw128(a_hi, a_lbo, 1024), bh = desc_sw128(b_hi, b_lbo, 1024);
  mma_bf16(d, ah, bh, idesc, acc);
  if (!kBf) {
    const uint64_t al = desc_sw128(a_hi + a_lo_off, a_lbo, 1024);
    const uint64_t bl = desc_sw128(b_hi + b_lo_off, b_lbo, 1024);
    mma_bf16(d, ah, bl, idesc, 1u);
    mma_bf16(d, al, bh, idesc, 1u);
  }
}

// Inclusive cumsum of dt * A (log2 units) over `len` steps starting at step
// t0 of batch row b, for the block's first `len` threads; s_cs2, s_dt
// filled, ends synced.
__device__ __forceinline__ void step_tables(const D64& d, const float* __restrict__ dt, float a2,
                                            int b, size_t t0, int len, int h, float* s_cs2,
                                            float* s_dt, float* scratch) {
  const int tid = threadIdx.x;
  const float dv = tid < len ? dt[((size_t)b * d.T + t0 + tid) * d.H + h] : 0.f;
  const float cs = block_inclusive_scan(dv * a2, scratch);
  if (tid < len) {
    s_cs2[tid] = cs;
    s_dt[tid] = dv;
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Chunk outer products, one CTA per (b, c, h) for chunks of Q <= 128 steps,
// 256 threads.
//   MODE 0: out = S_c  from u = x,  v = B, w_j = exp(cs_last - cs_j) dt_j
//   MODE 1: out = R_c  from u = dy, v = C, w_i = exp(cs_i)
// as D[n][p] = V^T (w o U) (M = n padded to 128: the second half of the A
// operand reads the U tiles and its rows are never read back), then written
// out[b][c][h][p][n]; also cs_last[b][h][c] (natural-log units).  PS: headdim.
template <int MODE, bool kBf, int NS, int PS>
__global__ void __launch_bounds__(256) k_outer64(D64 d, const Elem<kBf>* __restrict__ U,
                                                 const Elem<kBf>* __restrict__ V,
                                                 const float* __restrict__ dt,
                                                 const float* __restrict__ A,
                                                 float* __restrict__ out,
                                                 float* __restrict__ cs_last) {
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  uint8_t* sVh = sm;           // [128 rows j][64 n] (NS = 128: n 64-127 in the lo tile's place)
  uint8_t* sVl = sm + 16384;
  uint8_t* sUh = sm + 32768;   // [128 rows j][64 p], rows scaled by w (PS = 128: p 64-127 at the lo tile)
  uint8_t* sUl = sm + 49152;
  __shared__ float s_cs2[kQ], s_dt[kQ], s_w[kQ], scratch[8];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
  const int g = h / d.hpg, Q = d.Q;
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  if (tid < 32) {
    tmem_alloc(&tmem_base, PS);
    tmem_relinquish();
  }
  // the tiles' loads are in flight while the decay tables are built
  const size_t row0 = (size_t)b * d.T + (size_t)c * Q;
  RowTile<256, kQ, Elem<kBf>, NS> tv;
  RowTile<256, kQ, Elem<kBf>, PS> tu;
  tv.fetch(V + (row0 * d.G + g) * NS, (size_t)d.G * NS, Q);
  tu.fetch(U + (row0 * d.H + h) * PS, (size_t)d.H * PS, Q);
  step_tables(d, dt, A[h] * kLog2e, b, (size_t)c * Q, Q, h, s_cs2, s_dt, scratch);
  const float last2 = s_cs2[Q - 1];
  if (tid < Q) s_w[tid] = MODE == 0 ? exp2f(last2 - s_cs2[tid]) * s_dt[tid] : exp2f(s_cs2[tid]);
  if (tid == 0) cs_last[((size_t)b * d.H + h) * d.nc + c] = last2 * (1.0f / kLog2e);
  __syncthreads();
  tv.put(sVh, sVl, [](int) { return 1.f; }, Q);
  tu.put(sUh, sUl, [&](int r) { return s_w[r]; }, Q);
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tm = tmem_base;
  if (tid == 0) {
    const uint32_t id = idesc_bf16(128, PS, true, true);
    // A = V^T, M = n: NS = 64 pads M to 128 with a second block read from
    // the U tiles (rows never read back); NS = 128 has its second block of n
    // in the lo tile's place.  N = p: PS = 128 has its second block of p in
    // the U lo tile's place (16 KB on).
    for (int ks = 0; ks < Q / 16; ++ks)
      mma3<kBf>(tm, smem_u32(sVh) + ks * 2048, 16384, NS == 128 ? 16384 : 32768, true,
                smem_u32(sUh) + ks * 2048, 16384, 16384, id, ks > 0);
    mma_commit(&bar);
  }
  const bool ok = wait_all(&bar, 0);
  fence_after_sync();
  const int wg = tid >> 7, r = tid & 127;
  if (ok && r < NS) {  // lanes (rows n) below NS; warpgroup wg takes p in [PS/2 wg, +PS/2)
    float* dst = out + (((size_t)b * d.nc + c) * d.H + h) * (PS * NS) + r;
#pragma unroll
    for (int p32 = 0; p32 < PS / 64; ++p32) {
      const int pc = wg * (PS / 2) + p32 * 32;
      float v[32];
      tmem_ld32(tm + ((uint32_t)((r >> 5) * 32) << 16) + pc, v);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) dst[(size_t)(pc + i) * NS] = v[i];
    }
  }
  fence_before_sync();
  __syncthreads();
  if (tid < 32) tmem_dealloc(tm, PS);
}

// ---------------------------------------------------------------------------
// Chunk scan: y of one (b, 128-step block, h) per CTA, 256 threads, two
// CTAs per SM (80 KB of shared memory, 256 TMEM columns each).
//   CB = C B^T, Ys = C H^T (H = the state before the block: the history entry
//   of its first chunk, as rows n),
//   M = CB o L o dt (masked, split), Y = M X,
//   y = Y + exp(cs_i) Ys + D x.
// fp32 storage forms M (split) in two 64-column halves in the C tile's
// place, each followed by its half of Y = M X (K = the half's 64 rows of X).
// bf16 storage forms M whole in the C tile's 32 KB (CB and Ys have read C)
// and Y = M X is one batch with K = 128; Y then takes CB's TMEM columns (CB
// has been read), which leaves room for a 128-wide Y and Ys (headdim 128).
// X is fetched into registers at the start and written into the B tile's
// place once CB is formed (PS = 128: X's second 64 columns at the lo place).
// Decay masks as in the bf16 kernels: for warp q's rows and a 32-column chunk
// left of its diagonal chunk, exp(cs_i - cs_j) = exp(cs_i - cs_r) exp(cs_r -
// cs_j) with r = 32 q (both factors <= 1); the diagonal chunk evaluates the
// exponent only where j <= i.
// The tiles of the transposed state (H^T, g^T), the stride between their
// 64-p blocks (bf16) or their hi and lo tiles (fp32), and the shared memory
// of the kernels that hold them.
template <bool kBf, int NS, int PS>
constexpr uint32_t state_tile_bytes() { return (uint32_t)NS * PS * 2 * (kBf ? 1 : 2); }
template <bool kBf, int NS>
constexpr uint32_t state_block_stride() { return kBf ? NS * 128u : 8192u; }
template <bool kBf, int NS, int PS>
constexpr uint32_t scan64_bytes() {  // C (later M) 32K | B (later X) 32K | H^T
  return 65536u + state_tile_bytes<kBf, NS, PS>();
}

template <bool kBf, int NS, int PS>
__global__ void __launch_bounds__(256, 2) k_scan64(D64 d, const Elem<kBf>* __restrict__ x,
                                                   const float* __restrict__ dt,
                                                   const float* __restrict__ A,
                                                   const Elem<kBf>* __restrict__ Bm,
                                                   const Elem<kBf>* __restrict__ Cm,
                                                   const float* __restrict__ D,
                                                   const float* __restrict__ hist,
                                                   Elem<kBf>* __restrict__ y) {
  constexpr bool kWholeM = kBf;
  static_assert(PS == 64 || kBf, "headdim 128 is bf16");
  constexpr uint32_t kHpb = state_block_stride<kBf, NS>();
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  uint8_t* sCh = sm;            // [128 rows i][64 n] K-major (NS = 128: n 64-127 at the lo tile)
  uint8_t* sCl = sm + 16384;
  uint8_t* sMh = sm;            // M [128 rows i][64 j] K-major (after CB, Ys); kWholeM: j 64-127
  uint8_t* sMl = sm + 16384;    // at the lo tile
  uint8_t* sBh = sm + 32768;    // [128 rows j][64 n] K-major
  uint8_t* sBl = sm + 49152;
  uint8_t* sXh = sm + 32768;    // [128 rows j][64 p] MN-major B operand (after CB)
  uint8_t* sXl = sm + 49152;
  uint8_t* sHh = sm + 65536;    // [NS rows n][64 p] MN-major B operand (fp32: its lo tile;
  uint8_t* sHl = sHh + kHpb;    // PS = 128: p 64-127 there)
  __shared__ float s_cs2[kQ], s_dt[kQ], scratch[8];
  __shared__ __align__(16) float s_E[4][kQ];  // exp(cs_r - cs_j) dt_j, j < r = 32 w
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
  const int g = h / d.hpg, wg = tid >> 7, q = (tid >> 5) & 3, row = tid & 127;
  const uint32_t lane_base = (uint32_t)(q * 32) << 16;
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  if (tid < 32) {
    tmem_alloc(&tmem_base, 256);
    tmem_relinquish();
  }
  const size_t row0 = (size_t)b * d.T + (size_t)blk * kQ;
  const size_t c0 = (size_t)blk * d.cpb;  // the block's first chunk
  const auto one = [](int) { return 1.f; };
  // C, B and X loads in flight under the tables; X stays in registers until
  // the B tile is free (with a 128-wide tile, X is fetched under the products)
  constexpr bool kEarlyX = NS == 64 && PS == 64;
  RowTile<256, kQ, Elem<kBf>, NS> ta, tb;
  RowTile<256, kQ, Elem<kBf>, PS> tx;
  ta.fetch(Cm + (row0 * d.G + g) * NS, (size_t)d.G * NS);
  if (NS == 64) tb.fetch(Bm + (row0 * d.G + g) * NS, (size_t)d.G * NS);
  if (kEarlyX) tx.fetch(x + (row0 * d.H + h) * PS, (size_t)d.H * PS);
  step_tables(d, dt, A[h] * kLog2e, b, (size_t)blk * kQ, kQ, h, s_cs2, s_dt, scratch);
  for (int e = tid; e < 4 * kQ; e += 256) {
    const int w = e >> 7, j = e & 127, r = 32 * w;
    s_E[w][j] = j < r ? exp2f(s_cs2[r] - s_cs2[j]) * s_dt[j] : 0.f;
  }
  ta.put(sCh, sCl, one);
  if (NS == 128) ta.fetch(Bm + (row0 * d.G + g) * NS, (size_t)d.G * NS);
  if (NS == 64) tb.put(sBh, sBl, one);
  else ta.put(sBh, sBl, one);
  (void)load_split_transposed<256, kBf, NS, PS>(
      sHh, sHl, hist + (((size_t)b * d.nc + c0) * d.H + h) * (PS * NS), nullptr);
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tm = tmem_base, tCB = tm, tYs = tm + 128, tY = kWholeM ? tm : tm + 192;
  if (tid == 0) {
    // K = n: NS / 16 steps, the second 64 of n (NS = 128) at the lo tiles
    const uint32_t id_cb = idesc_bf16(128, 128, false, false);
    const uint32_t id_ys = idesc_bf16(128, PS, false, true);
    for (int kk = 0; kk < NS / 16; ++kk) {
      const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
      mma3<kBf>(tCB, smem_u32(sCh) + ko, 16384, 16, false, smem_u32(sBh) + ko, 16384, 16, id_cb,
                kk > 0);
      mma3<kBf>(tYs, smem_u32(sCh) + ko, 16384, 16, false, smem_u32(sHh) + kk * 2048, kHpb, kHpb,
                id_ys, kk > 0);
    }
    mma_commit(&bar);
  }
  if (!kEarlyX) tx.fetch(x + (row0 * d.H + h) * PS, (size_t)d.H * PS);  // under the products
  bool ok = wait_all(&bar, 0);
  uint32_t phase = 1;
  fence_after_sync();
  // the C and B tiles are free: X into the B tile's place
  tx.put(sXh, sXl, one);
  const int I = row;
  const float fi = exp2f(s_cs2[I] - s_cs2[32 * q]), csI = s_cs2[I];
  const uint32_t id_y = idesc_bf16(128, PS, false, true);
#pragma unroll 1
  for (int half = 0; half < 2 && ok; ++half) {
    // M columns [64 half, 64 half + 64): warpgroup wg writes its 32-column chunk jc
    const int jc = 2 * half + wg;
    uint8_t* mt = kWholeM && half ? sMl : sMh;
    {
      float v[32];
      if (jc <= q) {  // warp-uniform
        tmem_ld32(tCB + lane_base + jc * 32, v);
        tmem_wait_ld();
        if (jc < q) {
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] *= fi * s_E[q][jc * 32 + k];
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const int J = jc * 32 + k;
            v[k] *= J <= I ? exp2f(csI - s_cs2[J]) * s_dt[J] : 0.f;
          }
        }
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] = 0.f;
      }
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        store_split8<kBf>(mt, sMl, sw128(row, wg * 4 + q4), &v[q4 * 8]);
    }
    if (kWholeM && half == 0) continue;  // the whole M first
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (tid == 0) {
      if (kWholeM) {
        // Y = M X: K = all 128 rows j (the j 64-127 half of M at the lo tile)
        for (int kk = 0; kk < 8; ++kk)
          mma3<kBf>(tY, smem_u32(sMh) + (kk >> 2) * 16384 + (kk & 3) * 32, 16384, 16, false,
                    smem_u32(sXh) + kk * 2048, 16384, 16384, id_y, kk > 0);
      } else {
        // Y += M[:, half] X[half rows, :]: K = the half's 64 rows j
        for (int kk = 0; kk < 4; ++kk)
          mma3<kBf>(tY, smem_u32(sMh) + kk * 32, 16384, 16, false,
                    smem_u32(sXh) + (4 * half + kk) * 2048, 16384, 16384, id_y,
                    half > 0 || kk > 0);
      }
      mma_commit(&bar);
    }
    ok = wait_all(&bar, phase);  // the M half is rewritten next
    phase ^= 1;
    fence_after_sync();
  }
  if (ok) {
    // y = Y + exp(cs_i) Ys + D x; warpgroup wg takes p in [PS/2 wg, PS/2 (wg + 1))
    const float sc = exp2f(s_cs2[row]), Dh = D[h];
    const size_t off = ((row0 + row) * d.H + h) * PS + wg * (PS / 2);
#pragma unroll
    for (int hp = 0; hp < PS / 32; ++hp) {
      float yv[16], yst[16];
      tmem_ld16(tY + lane_base + wg * (PS / 2) + hp * 16, yv);
      tmem_ld16(tYs + lane_base + wg * (PS / 2) + hp * 16, yst);
      tmem_wait_ld();
#pragma unroll
      for (int k8 = 0; k8 < 2; ++k8) {
        const int cw = (wg * (PS / 2) + hp * 16) / 8 + k8;  // 8-column chunk of the row
        float xf[8], o[8];
        read_split8<kBf>(sXh + (cw >> 3) * 16384, sXl, sw128(row, cw & 7), xf);
#pragma unroll
        for (int t = 0; t < 8; ++t) o[t] = fmaf(sc, yst[k8 * 8 + t], yv[k8 * 8 + t]) + Dh * xf[t];
        st8(y + off + hp * 16 + k8 * 8, o);
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  if (tid < 32) tmem_dealloc(tm, 256);
}

// ---------------------------------------------------------------------------
// Column sums over the 32 lanes of a warp, for 16 columns: lane l returns the
// sum over all lanes of v[l % 16].
__device__ __forceinline__ float col_sum16(float (&v)[16]) {
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

// Backward, gradient w.r.t. x and dt: one (b, 128-step block, h) per CTA,
// 256 threads; cs, L are block-local.
//   batch A: CB = C B^T, dYX = dY X^T, Gs = B g^T, CH = C H^T
//            (g, the state gradient at the block end: the reverse pass's
//            value for its last chunk; H, the state before the block)
//   build:   W = L o dt o dYX and M = W o CB (row sums and strict column
//            sums of M, for d(cs)); O = L o CB (split) into the C/B tiles
//   batch B: Gx = O^T dY
//   epilogue: dx_j = D dy_j + dt_j (Gx_j + f_j Gs_j), f_j = exp(cs_last - cs_j);
//            drive_j = x_j.(Gx_j + f_j Gs_j), e_j = f_j dt_j x_j.Gs_j,
//            statein_i = exp(cs_i) dy_i.CH_i, and dy.x for dD
//   dcs_i = rowsum_i - colsum_i + statein_i - e_i (+ sum_j e_j +
//            exp(cs_last) <g, H> at i = Q - 1); da_j = sum_{i >= j} dcs_i;
//            ddt_j = drive_j + A da_j; partials sum_j dt_j da_j and sum dy.x.
// Headdim PS = 128 (bf16): X, dY, H^T and g^T keep p 64-127 in their lo
// places; Gx then takes CB's TMEM columns (CB has been read).
template <bool kBf, int NS, int PS>
constexpr uint32_t bwdx64_bytes() {  // C, B (later O) 64K | X 32K | dY 32K | H^T | g^T
  return 131072u + 2 * state_tile_bytes<kBf, NS, PS>();
}

template <bool kBf, int NS, int PS>
__global__ void __launch_bounds__(512, 1) k_bwd64_x(D64 d, const Elem<kBf>* __restrict__ x,
                                                    const float* __restrict__ dt,
                                                    const float* __restrict__ A,
                                                    const Elem<kBf>* __restrict__ Bm,
                                                    const Elem<kBf>* __restrict__ Cm,
                                                    const float* __restrict__ D,
                                                    const Elem<kBf>* __restrict__ dy,
                                                    const float* __restrict__ hist,
                                                    const float* __restrict__ gstate,
                                                    Elem<kBf>* __restrict__ dx,
                                                    float* __restrict__ ddt,
                                                    float* __restrict__ dA_part,
                                                    float* __restrict__ dD_part) {
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  uint8_t* sCh = sm;            // [128 rows i][64 n] K-major
  uint8_t* sCl = sm + 16384;
  uint8_t* sBh = sm + 32768;    // [128 rows j][64 n] K-major
  uint8_t* sBl = sm + 49152;
  uint8_t* sOh = sm;            // O [128 rows i][128 j] (two 64-column tiles), after batch A
  uint8_t* sOl = sm + 32768;
  uint8_t* sXh = sm + 65536;    // [128 rows j][64 p]
  uint8_t* sXl = sm + 81920;
  uint8_t* sYh = sm + 98304;    // dY [128 rows i][64 p]
  uint8_t* sYl = sm + 114688;
  static_assert(PS == 64 || (PS == 128 && kBf), "headdim 128 is bf16");
  constexpr uint32_t kHpb = state_block_stride<kBf, NS>();
  uint8_t* sHh = sm + 131072;   // H^T [NS rows n][64 p] (fp32: its lo tile; PS = 128: p
  uint8_t* sHl = sHh + kHpb;    // 64-127 there)
  uint8_t* sGh = sHh + state_tile_bytes<kBf, NS, PS>();  // g^T, the same
  uint8_t* sGl = sGh + kHpb;
  __shared__ float s_cs2[kQ], s_dt[kQ], scratch[16];
  __shared__ __align__(16) float s_E[4][kQ];    // exp(cs_r - cs_j), j < r = 32 w
  __shared__ __align__(16) float s_Edt[4][kQ];  // the same times dt_j
  __shared__ float s_col[4][kQ];                // per-warp strict column sums of M
  __shared__ float s_red[3][5][kQ];             // warpgroups 1-3: row partials
  __shared__ float s_v[kQ];
  __shared__ float2 s_v2[kQ], scratch2[16];
  __shared__ float s_esum;
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
  const int g = h / d.hpg, wg = tid >> 7, q = (tid >> 5) & 3, row = tid & 127, lane = tid & 31;
  const uint32_t lane_base = (uint32_t)(q * 32) << 16;
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  if (tid < 32) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  const float Ah = A[h], Dh = D[h];
  const size_t row0 = (size_t)b * d.T + (size_t)blk * kQ;
  const size_t c0 = (size_t)blk * d.cpb, c1 = c0 + d.cpb - 1;  // first, last chunk
  const size_t st_in = (((size_t)b * d.nc + c0) * d.H + h) * (PS * NS);
  const size_t st_out = (((size_t)b * d.nc + c1) * d.H + h) * (PS * NS);
  const auto one = [](int) { return 1.f; };
  // two tiles' loads in flight at a time, the first two under the tables
  RowTile<512, kQ, Elem<kBf>, NS> ta, tb;
  RowTile<512, kQ, Elem<kBf>, PS> tc, td;
  ta.fetch(Cm + (row0 * d.G + g) * NS, (size_t)d.G * NS);
  tb.fetch(Bm + (row0 * d.G + g) * NS, (size_t)d.G * NS);
  step_tables(d, dt, Ah * kLog2e, b, (size_t)blk * kQ, kQ, h, s_cs2, s_dt, scratch);
  for (int e = tid; e < 4 * kQ; e += 512) {
    const int w = e >> 7, j = e & 127, r = 32 * w;
    const float ev = j < r ? exp2f(s_cs2[r] - s_cs2[j]) : 0.f;
    s_E[w][j] = ev;
    s_Edt[w][j] = ev * s_dt[j];
  }
  ta.put(sCh, sCl, one);
  tc.fetch(x + (row0 * d.H + h) * PS, (size_t)d.H * PS);
  tb.put(sBh, sBl, one);
  td.fetch(dy + (row0 * d.H + h) * PS, (size_t)d.H * PS);
  (void)load_split_transposed<512, kBf, NS, PS>(sHh, sHl, hist + st_in, nullptr);
  tc.put(sXh, sXl, one);
  float hg = load_split_transposed<512, kBf, NS, PS>(sGh, sGl, gstate + st_out, hist + st_in);
  td.put(sYh, sYl, one);
  hg = block_sum(hg, scratch);  // <g_c, H_{c-1}> (syncs)
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tm = tmem_base;
  const uint32_t T0 = tm, T1 = tm + 128, TGs = tm + 256, TCH = tm + 256 + PS;
  const uint32_t TGx = PS == 64 ? tm + 384 : T0;
  if (tid == 0) {
    const uint32_t id_sq = idesc_bf16(128, 128, false, false);
    const uint32_t id_km = idesc_bf16(128, PS, false, true);
    // K = p (dY X^T): PS / 16 steps; K = n (CB, Gs, CH): NS / 16 steps; the
    // second 64 of p or n at the lo tiles
    for (int kk = 0; kk < PS / 16; ++kk) {
      const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
      mma3<kBf>(T1, smem_u32(sYh) + ko, 16384, 16, false, smem_u32(sXh) + ko, 16384, 16, id_sq,
                kk > 0);
    }
    for (int kk = 0; kk < NS / 16; ++kk) {
      const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
      mma3<kBf>(T0, smem_u32(sCh) + ko, 16384, 16, false, smem_u32(sBh) + ko, 16384, 16, id_sq,
                kk > 0);
      mma3<kBf>(TGs, smem_u32(sBh) + ko, 16384, 16, false, smem_u32(sGh) + kk * 2048, kHpb, kHpb,
                id_km, kk > 0);
      mma3<kBf>(TCH, smem_u32(sCh) + ko, 16384, 16, false, smem_u32(sHh) + kk * 2048, kHpb, kHpb,
                id_km, kk > 0);
    }
    mma_commit(&bar);
  }
  bool ok = wait_all(&bar, 0);
  fence_after_sync();

  // ---- build: W, M sums and O = L o CB; warpgroup wg covers the 32
  // columns [32 wg, 32 wg + 32)
  const int I = row;
  const float fi = exp2f(s_cs2[I] - s_cs2[32 * q]), csI = s_cs2[I];
  float rowsum = 0.f;
  if (ok) {
    {
      const int jc = wg;
      if (jc <= q) {  // warp-uniform
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          const int col0 = jc * 32 + hf * 16;
          float cb[16], xy[16];
          tmem_ld16(T0 + lane_base + col0, cb);
          tmem_ld16(T1 + lane_base + col0, xy);
          tmem_wait_ld();
          if (jc < q) {
#pragma unroll
            for (int m = 0; m < 16; ++m) {
              const float wv = fi * s_Edt[q][col0 + m] * xy[m];
              const float mm = wv * cb[m];
              rowsum += mm;
              xy[m] = mm;
              cb[m] *= fi * s_E[q][col0 + m];
            }
          } else {
#pragma unroll
            for (int m = 0; m < 16; ++m) {
              const int J = col0 + m;
              const float L = J <= I ? exp2f(csI - s_cs2[J]) : 0.f;
              const float wv = L * s_dt[J] * xy[m];
              const float mm = J < I ? wv * cb[m] : 0.f;
              rowsum += mm;
              xy[m] = mm;
              cb[m] *= L;
            }
          }
          const float cs = col_sum16(xy);
          if (lane < 16) s_col[q][col0 + lane] = cs;
#pragma unroll
          for (int q4 = 0; q4 < 2; ++q4) {
            const int j = col0 + q4 * 8;
            store_split8<kBf>(sOh + (j >> 6) * 16384, sOl + (j >> 6) * 16384,
                              sw128(row, (j & 63) >> 3), &cb[q4 * 8]);
          }
        }
      } else {
        const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int j = jc * 32 + q4 * 8;
          store_split8<kBf>(sOh + (j >> 6) * 16384, sOl + (j >> 6) * 16384,
                            sw128(row, (j & 63) >> 3), z);
        }
      }
    }
  }
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (tid == 0 && ok) {
    // Gx = O^T dY: M = j (O as MN-major, two 64-column blocks), K = i, N = p
    const uint32_t id = idesc_bf16(128, PS, true, true);
    for (int kk = 0; kk < 8; ++kk)
      mma3<kBf>(TGx, smem_u32(sOh) + kk * 2048, 32768, 16384, true, smem_u32(sYh) + kk * 2048,
                16384, 16384, id, kk > 0);
    mma_commit(&bar);
  }
  ok = ok && wait_all(&bar, 1);
  fence_after_sync();

  // ---- epilogue: this thread's row (j for dx, drive, e; i for statein), p in
  // [PS/4 wg, PS/4 (wg + 1))
  const float last2 = s_cs2[kQ - 1];
  const float fj = exp2f(last2 - s_cs2[row]), dtj = s_dt[row];
  float drive = 0.f, ej = 0.f, stin = 0.f, dd = 0.f;
  if (ok) {
    const size_t off = ((row0 + row) * d.H + h) * PS + wg * (PS / 4);
#pragma unroll
    for (int hp = 0; hp < PS / 64; ++hp) {
      const int pc = wg * (PS / 4) + hp * 16;  // the 16 columns of this pass
      float gx[16], gs[16], ch[16];
      tmem_ld16(TGx + lane_base + pc, gx);
      tmem_ld16(TGs + lane_base + pc, gs);
      tmem_ld16(TCH + lane_base + pc, ch);
      tmem_wait_ld();
#pragma unroll
      for (int k8 = 0; k8 < 2; ++k8) {
        const int cw = pc / 8 + k8;  // 8-column chunk of the row
        float xa[8], ya[8], o[8];
        read_split8<kBf>(sXh + (cw >> 3) * 16384, sXl, sw128(row, cw & 7), xa);
        read_split8<kBf>(sYh + (cw >> 3) * 16384, sYl, sw128(row, cw & 7), ya);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int m = 8 * k8 + t;
          const float gg = fmaf(fj, gs[m], gx[m]);
          o[t] = fmaf(dtj, gg, Dh * ya[t]);
          drive = fmaf(xa[t], gg, drive);
          ej = fmaf(xa[t], gs[m], ej);
          stin = fmaf(ya[t], ch[m], stin);
          dd = fmaf(ya[t], xa[t], dd);
        }
        st8(dx + off + hp * 16 + k8 * 8, o);
      }
    }
  }
  if (wg > 0) {
    s_red[wg - 1][0][row] = rowsum;
    s_red[wg - 1][1][row] = drive;
    s_red[wg - 1][2][row] = ej;
    s_red[wg - 1][3][row] = stin;
    s_red[wg - 1][4][row] = dd;
  }
  __syncthreads();
  if (wg == 0) {
#pragma unroll
    for (int w = 0; w < 3; ++w) {  // warpgroups in order
      rowsum += s_red[w][0][row];
      drive += s_red[w][1][row];
      ej += s_red[w][2][row];
      stin += s_red[w][3][row];
      dd += s_red[w][4][row];
    }
    ej *= fj * dtj;
    stin *= exp2f(s_cs2[row]);
    float colsum = 0.f;
    for (int w = row >> 5; w < 4; ++w) colsum += s_col[w][row];
    s_v2[row] = make_float2(rowsum - colsum + stin - ej, ej);
  } else {
    dd = 0.f;
  }
  __syncthreads();
  // da_j = sum_{i >= j} dcs_i: an inclusive scan over the reversed rows
  const float2 rv = wg == 0 ? s_v2[kQ - 1 - row] : make_float2(0.f, 0.f);
  const float2 sc2 = block_inclusive_scan2(rv, scratch2);
  const int Jr = kQ - 1 - row;
  if (wg == 0) s_v[row] = drive;
  if (tid == kQ - 1) s_esum = sc2.y;
  __syncthreads();
  const float da = sc2.x + s_esum + exp2f(last2) * hg;
  if (wg == 0 && ok) ddt[(row0 + Jr) * d.H + h] = s_v[Jr] + Ah * da;
  const float2 ad = block_sum2(make_float2(wg == 0 ? s_dt[Jr] * da : 0.f, dd), scratch2);
  if (tid == 0 && ok) {
    const size_t slot = ((size_t)b * d.nb + blk) * d.H + h;
    dA_part[slot] = ad.x;
    dD_part[slot] = ad.y;
  }
  fence_before_sync();
  __syncthreads();
  if (tid < 32) tmem_dealloc(tm, 512);
}

// ---------------------------------------------------------------------------
// Backward, gradients w.r.t. B and C: one (b, 128-step block, g) unit and a
// segment of its heads per CTA, 512 threads.  Per head: dYX = dY X^T (TMEM), W = L o dt o dYX
// summed over the segment's heads in registers (thread (wg, row) holds
// columns [32 wg, 32 wg + 32) of its row); then X and dY are reloaded scaled
// (f_j = exp(cs_last - cs_j) dt_j, e_i = exp(cs_i)) for
//   dC += (e o dY) H,  dB += (f o X) g      (TMEM accumulators over heads).
// After the segment: W into split tiles, dC += W B, dB += W^T C, and the fp32
// sums of the segment written as partials [unit][segment][dC|dB][128][64].
// Headdim PS = 128 (bf16): X, dY keep p 64-127 in their lo places and H, g
// their rows p 64-127 (d_state 128: their n 64-127 blocks at the lo
// pointers, PS rows on).
template <bool kBf, int NS, int PS>
constexpr uint32_t bwdbc64_bytes() {  // B 32K | C 32K | X 32K | dY 32K | H | g
  return 131072u + 2 * state_tile_bytes<kBf, NS, PS>();
}

template <bool kBf, int NS, int PS>
__global__ void __launch_bounds__(512, 1) k_bwd64_bc(D64 d, int seg_heads,
                                                     const Elem<kBf>* __restrict__ x,
                                                     const float* __restrict__ dt,
                                                     const float* __restrict__ A,
                                                     const Elem<kBf>* __restrict__ Bm,
                                                     const Elem<kBf>* __restrict__ Cm,
                                                     const Elem<kBf>* __restrict__ dy,
                                                     const float* __restrict__ hist,
                                                     const float* __restrict__ gstate,
                                                     float* __restrict__ part) {
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t* sm = align1024(smraw);
  uint8_t* sBh = sm;            // [128 rows j][64 n] MN-major B operand
  uint8_t* sBl = sm + 16384;
  uint8_t* sCh = sm + 32768;    // [128 rows i][64 n]
  uint8_t* sCl = sm + 49152;
  uint8_t* sXh = sm + 65536;    // [128 rows j][64 p]
  uint8_t* sXl = sm + 81920;
  uint8_t* sYh = sm + 98304;    // dY [128 rows i][64 p]
  uint8_t* sYl = sm + 114688;
  uint8_t* sWh = sm + 65536;    // W [128 rows i][128 j] after the last head (X, dY region)
  uint8_t* sWl = sm + 98304;
  constexpr uint32_t kSpb = state_block_stride<kBf, PS>();  // n-block stride: PS rows p
  uint8_t* sHh = sm + 131072;   // H [PS rows p][64 n] MN-major B operand (fp32: its lo tile;
  uint8_t* sHl = sHh + kSpb;    // NS = 128: n 64-127 there)
  uint8_t* sGh = sHh + state_tile_bytes<kBf, NS, PS>();  // g, the same
  uint8_t* sGl = sGh + kSpb;
  __shared__ float s_cs2[kQ], s_dt[kQ], scratch[16];
  __shared__ __align__(16) float s_E[4][kQ];  // exp(cs_r - cs_j) dt_j, j < r = 32 w
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  const int seg = blockIdx.x, blk = blockIdx.y, bg = blockIdx.z;
  const int b = bg / d.G, g = bg % d.G;
  const int tid = threadIdx.x, wg = tid >> 7, q = (tid >> 5) & 3, row = tid & 127;
  const uint32_t lane_base = (uint32_t)(q * 32) << 16;
  const int h0 = g * d.hpg + seg * seg_heads;
  const int nh = min(seg_heads, d.hpg - seg * seg_heads);
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  constexpr uint32_t kCols = NS == 128 ? 512 : 256;  // dY X^T 128 + dC, dB NS each
  if (tid < 32) {
    tmem_alloc(&tmem_base, kCols);
    tmem_relinquish();
  }
  const size_t row0 = (size_t)b * d.T + (size_t)blk * kQ;
  const size_t c0 = (size_t)blk * d.cpb, c1 = c0 + d.cpb - 1;  // first, last chunk
  const auto one = [](int) { return 1.f; };
  {
    RowTile<512, kQ, Elem<kBf>, NS> tb;
    tb.fetch(Bm + (row0 * d.G + g) * NS, (size_t)d.G * NS);
    tb.put(sBh, sBl, one);
    tb.fetch(Cm + (row0 * d.G + g) * NS, (size_t)d.G * NS);
    tb.put(sCh, sCl, one);
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tm = tmem_base, T1 = tm, TdC = tm + 128, TdB = tm + 128 + NS;
  uint32_t phase = 0;
  bool ok = true;
  float wsum[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) wsum[k] = 0.f;
  const int I = row, jc = wg;  // this thread's row and 32-column chunk of W
  // a head's tiles are fetched into registers while the previous head's
  // state-term products run (the first head's before the loop)
  RowTile<512, kQ, Elem<kBf>, PS> tx, ty;
  StateRowTile<512, NS, kBf, PS> th, tg;  // the states as rows p of NS values
  // (NS = 128 or PS = 128: the state tiles are fetched at the head's start
  // instead, to stay within the registers; with both at 128, one after the
  // other through th)
  constexpr bool kEarlyStates = NS == 64 && PS == 64;
  constexpr bool kOneState = NS == 128 && PS == 128;
  auto st_in_of = [&](int h) { return (((size_t)b * d.nc + c0) * d.H + h) * (PS * NS); };
  auto st_out_of = [&](int h) { return (((size_t)b * d.nc + c1) * d.H + h) * (PS * NS); };
  auto fetch_states = [&](int h) {
    th.fetch(hist + st_in_of(h));
    tg.fetch(gstate + st_out_of(h));
  };
  auto fetch_head = [&](int h) {
    tx.fetch(x + (row0 * d.H + h) * PS, (size_t)d.H * PS);
    ty.fetch(dy + (row0 * d.H + h) * PS, (size_t)d.H * PS);
    if (kEarlyStates) fetch_states(h);
  };
  if (nh > 0) fetch_head(h0);
  for (int hh = 0; hh < nh && ok; ++hh) {
    const int h = h0 + hh;
    if (!kEarlyStates && !kOneState) fetch_states(h);
    if (kOneState) th.fetch(hist + st_in_of(h));
    step_tables(d, dt, A[h] * kLog2e, b, (size_t)blk * kQ, kQ, h, s_cs2, s_dt, scratch);
    for (int e = tid; e < 4 * kQ; e += 512) {
      const int w = e >> 7, j = e & 127, r = 32 * w;
      s_E[w][j] = j < r ? exp2f(s_cs2[r] - s_cs2[j]) * s_dt[j] : 0.f;
    }
    tx.put(sXh, sXl, one);
    ty.put(sYh, sYl, one);
    th.put(sHh, sHl);
    if (kOneState) {
      th.fetch(gstate + st_out_of(h));
      th.put(sGh, sGl);
    } else {
      tg.put(sGh, sGl);
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (tid == 0) {
      // K = p: PS / 16 steps, p 64-127 (PS = 128) at the lo tiles
      const uint32_t id = idesc_bf16(128, 128, false, false);
      for (int kk = 0; kk < PS / 16; ++kk) {
        const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
        mma3<kBf>(T1, smem_u32(sYh) + ko, 16384, 16, false, smem_u32(sXh) + ko, 16384, 16, id,
                  kk > 0);
      }
      mma_commit(&bar);
    }
    ok = wait_all(&bar, phase);
    phase ^= 1;
    fence_after_sync();
    if (!ok) break;
    // W += L o dt o dYX over this thread's 32 columns
    if (jc <= q) {  // warp-uniform
      const float fi = exp2f(s_cs2[I] - s_cs2[32 * q]), csI = s_cs2[I];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int col0 = jc * 32 + hf * 16;
        float xy[16];
        tmem_ld16(T1 + lane_base + col0, xy);
        tmem_wait_ld();
        if (jc < q) {
#pragma unroll
          for (int m = 0; m < 16; ++m) wsum[hf * 16 + m] = fmaf(fi * s_E[q][col0 + m], xy[m], wsum[hf * 16 + m]);
        } else {
#pragma unroll
          for (int m = 0; m < 16; ++m) {
            const int J = col0 + m;
            const float L = J <= I ? exp2f(csI - s_cs2[J]) * s_dt[J] : 0.f;
            wsum[hf * 16 + m] = fmaf(L, xy[m], wsum[hf * 16 + m]);
          }
        }
      }
    }
    // X, dY rescaled in place (the dYX product has read them): X rows j by
    // exp(cs_last - cs_j) dt_j, dY rows i by exp(cs_i)
    const float last2 = s_cs2[kQ - 1];
    rescale_split<512, kQ, kBf, PS>(sXh, sXl,
                                    [&](int r) { return exp2f(last2 - s_cs2[r]) * s_dt[r]; });
    rescale_split<512, kQ, kBf, PS>(sYh, sYl, [&](int r) { return exp2f(s_cs2[r]); });
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (tid == 0) {
      // N = n: NS (the second 64 of n at the lo tiles, 8 KB on); K = p:
      // PS / 16 steps (p 64-127 of X, dY at their lo tiles; rows p of H, g
      // continue there)
      const uint32_t id = idesc_bf16(128, NS, false, true);
      for (int kk = 0; kk < PS / 16; ++kk) {
        const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
        mma3<kBf>(TdC, smem_u32(sYh) + ko, 16384, 16, false, smem_u32(sHh) + kk * 2048, kSpb,
                  kSpb, id, hh > 0 || kk > 0);
        mma3<kBf>(TdB, smem_u32(sXh) + ko, 16384, 16, false, smem_u32(sGh) + kk * 2048, kSpb,
                  kSpb, id, hh > 0 || kk > 0);
      }
      mma_commit(&bar);
    }
    if (hh + 1 < nh) fetch_head(h + 1);
    ok = wait_all(&bar, phase);  // the tiles are rewritten by the next head
    phase ^= 1;
    fence_after_sync();
  }
  // W of the segment into split tiles (X, dY region), then dC += W B, dB += W^T C
  if (ok) {
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const int j = jc * 32 + q4 * 8;
      store_split8<kBf>(sWh + (j >> 6) * 16384, sWl + (j >> 6) * 16384,
                        sw128(row, (j & 63) >> 3), &wsum[q4 * 8]);
    }
  }
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (tid == 0 && ok) {
    const uint32_t id_dc = idesc_bf16(128, NS, false, true);
    const uint32_t id_db = idesc_bf16(128, NS, true, true);
    for (int kk = 0; kk < 8; ++kk) {
      // dC: A = W (K-major, K = j), B = B (MN-major rows j, N = n)
      mma3<kBf>(TdC, smem_u32(sWh) + (kk >> 2) * 16384 + (kk & 3) * 32, 32768, 16, false,
           smem_u32(sBh) + kk * 2048, 16384, 16384, id_dc, 1);
      // dB: A = W^T (MN-major rows i = K, M = j), B = C (MN-major rows i, N = n)
      mma3<kBf>(TdB, smem_u32(sWh) + kk * 2048, 32768, 16384, true, smem_u32(sCh) + kk * 2048, 16384,
           16384, id_db, 1);
    }
    mma_commit(&bar);
  }
  ok = ok && wait_all(&bar, phase);
  fence_after_sync();
  if (ok) {
    // warpgroup wg writes columns [NS/4 wg, NS/4 (wg + 1)) of row `row` of dC and dB
    constexpr int kC = NS / 4;
    const size_t unit = ((size_t)b * d.nb + blk) * d.G + g;
    float* pbase = part + (unit * gridDim.x + seg) * (2 * kQ * NS);
#pragma unroll
    for (int which = 0; which < 2; ++which) {
#pragma unroll
      for (int c16 = 0; c16 < kC / 16; ++c16) {
        float v[16];
        tmem_ld16((which ? TdB : TdC) + lane_base + wg * kC + c16 * 16, v);
        tmem_wait_ld();
        float4* dst = (float4*)(pbase + which * (kQ * NS) + (size_t)row * NS + wg * kC + c16 * 16);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
          dst[k4] = make_float4(v[4 * k4], v[4 * k4 + 1], v[4 * k4 + 2], v[4 * k4 + 3]);
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  if (tid < 32) tmem_dealloc(tm, kCols);
}

// dC, dB of every unit: the segments' partials summed in segment order.
__device__ __forceinline__ void st4(float* p, float4 v) { *(float4*)p = v; }
__device__ __forceinline__ void st4(__nv_bfloat16* p, float4 v) {
  *(uint2*)p = make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
}

template <bool kBf, int NS>
__global__ void __launch_bounds__(256) k_sum64_bc(D64 d, int nseg, const float* __restrict__ part,
                                                  Elem<kBf>* __restrict__ dB,
                                                  Elem<kBf>* __restrict__ dC) {
  const size_t unit = blockIdx.x;  // ((b * nb + block) * G + g)
  const int g = (int)(unit % d.G), blk = (int)((unit / d.G) % d.nb);
  const int b = (int)(unit / ((size_t)d.G * d.nb));
  const float* base = part + unit * nseg * (2 * kQ * NS);
  for (int e = threadIdx.x; e < 2 * kQ * NS / 4; e += blockDim.x) {
    const int which = e / (kQ * NS / 4), r = (e % (kQ * NS / 4)) / (NS / 4), n4 = e % (NS / 4);
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < nseg; ++k) {
      const float4 v = ((const float4*)(base + (size_t)k * (2 * kQ * NS) + which * (kQ * NS) +
                                        (size_t)r * NS))[n4];
      s.x += v.x;
      s.y += v.y;
      s.z += v.z;
      s.w += v.w;
    }
    Elem<kBf>* out = which ? dB : dC;
    st4(out + (((size_t)b * d.T + (size_t)blk * kQ + r) * d.G + g) * NS + 4 * n4, s);
  }
}

D64 d64_of(const Problem& p) {
  return D64{p.B, p.T, p.H, p.G, p.nc, p.hpg, p.Q, p.T / kQ, kQ / p.Q};
}

template <typename K>
cudaError_t set_smem64(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <bool kBf, int NS, int PS>
cudaError_t chunk_outer_t(const Problem& p, int mode, float* out) {
  using E = Elem<kBf>;
  const size_t smem = 65536 + 1024;
  cudaError_t e;
  if (mode == 0) {
    if ((e = set_smem64(k_outer64<0, kBf, NS, PS>, smem)) != cudaSuccess) return e;
    LaunchScope ls("chunk_state_tc64", p.stream);
    k_outer64<0, kBf, NS, PS><<<dim3(p.nc, p.H, p.B), 256, smem, p.stream>>>(
        d64_of(p), (const E*)p.x, (const E*)p.Bm, p.dt, p.A, out, p.cs_last);
  } else {
    if ((e = set_smem64(k_outer64<1, kBf, NS, PS>, smem)) != cudaSuccess) return e;
    LaunchScope ls("chunk_dstate_tc64", p.stream);
    k_outer64<1, kBf, NS, PS><<<dim3(p.nc, p.H, p.B), 256, smem, p.stream>>>(
        d64_of(p), (const E*)p.dy, (const E*)p.Cm, p.dt, p.A, out, p.cs_last);
  }
  return cudaGetLastError();
}

template <bool kBf, int NS, int PS>
cudaError_t forward_scan_t(const Problem& p) {
  using E = Elem<kBf>;
  const size_t smem = scan64_bytes<kBf, NS, PS>() + 1024;
  cudaError_t e = set_smem64(k_scan64<kBf, NS, PS>, smem);
  if (e != cudaSuccess) return e;
  {
    LaunchScope ls("chunk_scan_tc64", p.stream);
    k_scan64<kBf, NS, PS><<<dim3(p.T / kQ, p.H, p.B), 256, smem, p.stream>>>(
        d64_of(p), (const E*)p.x, p.dt, p.A, (const E*)p.Bm, (const E*)p.Cm, p.D, p.hist,
        (E*)p.y);
  }
  return cudaGetLastError();
}

}  // namespace

// seqlen a multiple of 128, and
//   headdim 64, d_state 64 (fp32 or bf16), chunk 16-256;
//   headdim 64, d_state 128 (bf16, chunks 16-64: the bf16 kernels of
//     ssd_tc.cu take chunks 128 and 256);
//   headdim 128, d_state 64 or 128 (bf16), chunk 16-256.
// Chunks of 256 run as 128-step sub-chunks (tc64_subchunks).
bool tc64_supported(const Problem& p) {
  if (tc_forced_simt()) return false;
  if (p.T % kQ != 0) return false;
  if (p.Q != 16 && p.Q != 32 && p.Q != 64 && p.Q != 128 && p.Q != 256) return false;
  if (p.P == 64) return p.N == 64 || (p.N == 128 && p.bf16 && p.Q < 128);
  return p.P == 128 && (p.N == 64 || p.N == 128) && p.bf16;
}

// Chunks longer than a block: the kernels run on the problem regrouped into
// 128-step chunks (exact: chunking regroups the recurrence), whose start
// states include those of the caller's chunks (every Q/128-th).
bool tc64_subchunks(const Problem& p) { return tc64_supported(p) && p.Q > kQ; }

Problem tc64_sub_problem(const Problem& p) {
  Problem s = p;
  s.Q = kQ;
  s.nc = p.T / kQ;
  s.hist = p.hist_sub;
  return s;
}

// Heads per segment of the dB, dC kernel (one CTA per SM): the number of
// segments per unit that minimises waves x (heads per segment + a CTA's own
// work, about two heads': the B, C tiles, the W products and the partials'
// write) over kBcSlots CTA slots (the SMs of a GB300), the fewest segments
// among equals.  The split sets the order of the dB, dC sums,
// so it depends on this constant and not on the device: results and
// workspace sizes are the same on every GPU.
constexpr long long kBcSlots = 152;

int tc64_seg_heads(const Problem& p) {
  const long long units = (long long)p.B * (p.T / kQ) * p.G;
  long long best_seg = 1, best_cost = -1;
  for (long long nseg = 1; nseg <= p.hpg; ++nseg) {
    const long long heads = (p.hpg + nseg - 1) / nseg;
    if ((p.hpg + heads - 1) / heads != nseg) continue;  // same split as a smaller count
    const long long cost = ((units * nseg + kBcSlots - 1) / kBcSlots) * (heads + 2);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_seg = nseg;
    }
  }
  return (int)((p.hpg + best_seg - 1) / best_seg);
}

size_t tc64_bc_part_floats(const Problem& p) {
  const int sh = tc64_seg_heads(p);
  const long long nseg = (p.hpg + sh - 1) / sh;
  return (size_t)p.B * (p.T / kQ) * p.G * nseg * 2 * kQ * p.N;
}

cudaError_t tc64_chunk_outer(const Problem& p, int mode, float* out) {
  if (!p.bf16) return chunk_outer_t<false, 64, 64>(p, mode, out);
  if (p.P == 128)
    return p.N == 128 ? chunk_outer_t<true, 128, 128>(p, mode, out)
                      : chunk_outer_t<true, 64, 128>(p, mode, out);
  return p.N == 128 ? chunk_outer_t<true, 128, 64>(p, mode, out)
                    : chunk_outer_t<true, 64, 64>(p, mode, out);
}

cudaError_t tc64_forward_scan(const Problem& p) {
  if (!p.bf16) return forward_scan_t<false, 64, 64>(p);
  if (p.P == 128)
    return p.N == 128 ? forward_scan_t<true, 128, 128>(p) : forward_scan_t<true, 64, 128>(p);
  return p.N == 128 ? forward_scan_t<true, 128, 64>(p) : forward_scan_t<true, 64, 64>(p);
}

namespace {
template <bool kBf, int NS, int PS>
cudaError_t backward_t(const Problem& p) {
  using E = Elem<kBf>;
  cudaError_t e;
  if ((e = chunk_outer_t<kBf, NS, PS>(p, 1, p.dstate)) != cudaSuccess) return e;
  if ((e = simt_state_pass_bwd(p)) != cudaSuccess) return e;
  const D64 d = d64_of(p);
  const int nb = p.T / kQ;
  {
    const size_t smem = bwdx64_bytes<kBf, NS, PS>() + 1024;
    if ((e = set_smem64(k_bwd64_x<kBf, NS, PS>, smem)) != cudaSuccess) return e;
    LaunchScope ls("bwd_x_tc64", p.stream);
    k_bwd64_x<kBf, NS, PS><<<dim3(nb, p.H, p.B), 512, smem, p.stream>>>(
        d, (const E*)p.x, p.dt, p.A, (const E*)p.Bm, (const E*)p.Cm, p.D, (const E*)p.dy,
        p.hist, p.dstate, (E*)p.dx, p.ddt, p.dA_part, p.dD_part);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int sh = tc64_seg_heads(p);
  const int nseg = (p.hpg + sh - 1) / sh;
  {
    const size_t smem = bwdbc64_bytes<kBf, NS, PS>() + 1024;
    if ((e = set_smem64(k_bwd64_bc<kBf, NS, PS>, smem)) != cudaSuccess) return e;
    LaunchScope ls("bwd_bc_tc64", p.stream);
    k_bwd64_bc<kBf, NS, PS><<<dim3(nseg, nb, p.B * p.G), 512, smem, p.stream>>>(
        d, sh, (const E*)p.x, p.dt, p.A, (const E*)p.Bm, (const E*)p.Cm, (const E*)p.dy,
        p.hist, p.dstate, p.bwd_part);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  {
    LaunchScope ls("sum_bc_tc64", p.stream);
    k_sum64_bc<kBf, NS><<<(unsigned)((size_t)p.B * nb * p.G), 256, 0, p.stream>>>(
        d, nseg, p.bwd_part, (E*)p.dB, (E*)p.dC);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return simt_reduce_heads(p, p.B * nb, p.B * nb);
}
}  // namespace

// R_c, the reverse state pass (g_c in place, dh0), the dx / d(dt) kernel, the
// dB / dC kernel and its segment sums, and the dA, dD reduction.
cudaError_t tc64_backward(const Problem& p) {
  if (!p.bf16) return backward_t<false, 64, 64>(p);
  if (p.P == 128)
    return p.N == 128 ? backward_t<true, 128, 128>(p) : backward_t<true, 64, 128>(p);
  return p.N == 128 ? backward_t<true, 128, 64>(p) : backward_t<true, 64, 64>(p);
}

cudaError_t tc64_read_and_clear_error(unsigned int* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_tc64_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_tc64_error, &zero, sizeof(unsigned int));
}

}  // namespace ssd
