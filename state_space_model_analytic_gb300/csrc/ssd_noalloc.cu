// ssd_forward_noalloc: the forward pass for callers that must not allocate
// device memory.
//
// ssd_forward needs a caller-provided workspace.  Some callers cannot
// provide one on demand: a host framework that owns every byte of device
// memory through its own pool and forbids other allocations, code on a
// latency-critical path where a cudaMalloc may synchronise the device or
// fail with out-of-memory at the worst moment, or an embedding that simply
// has no allocator at hand.  This entry point takes the same inputs and
// outputs as ssd_forward and uses, instead of a workspace, a fixed scratch
// array that is part of the library image: it calls no cudaMalloc, cudaFree
// or any allocating routine.
//
// The scratch is a file-scope device array of SSD_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads the library keeps it until the process exits.  Its
// device address is looked up once per device (cudaGetSymbolAddress, with
// that device current) by the first call on that device; that first call
// should therefore come before any stream capture.  All calls on a device
// share the one array and it keeps whatever the last call left in it, so
// calls whose kernels may overlap on the GPU (different streams, or
// different host threads) race on it; callers must order them.  Nothing in
// it needs to start at zero: the forward fully writes every scratch value
// (per-chunk decay totals and, without a caller history buffer, the chunk
// states) before reading it.
#include <cstring>
#include <mutex>

#include "../../include/ssd.h"
#include "ssd_internal.h"

namespace ssd {

bool tc_supported(const Problem& p);
cudaError_t tc_chunk_outer(const Problem& p, int mode, float* out);
cudaError_t tc_forward_scan(const Problem& p);
size_t simt_smem_need(const Problem& p);
void set_last_error(const char* msg);

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SSD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

struct DeviceScratch {
  std::once_flag once;
  void* ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
DeviceScratch g_scratch[kMaxDevices];

// Device address of the scratch array on the current device (looked up once).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  DeviceScratch& s = g_scratch[dev];
  std::call_once(s.once, [&s] {
    void* p = nullptr;
    s.err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    s.ptr = (s.err == cudaSuccess) ? p : nullptr;
  });
  *out = s.ptr;
  return s.err;
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

int reject(int code, const char* msg) {
  set_last_error(msg);
  return code;
}

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" int ssd_forward_noalloc(const ssd_dims* dims, const void* x, const float* dt,
                                   const float* A, const void* B, const void* C, const float* D,
                                   const float* h0, void* y, float* final_state,
                                   float* chunk_states, void* cuda_stream) {
  set_last_error("");
  // validation and shape limits of ssd_forward (0 = rejected, message already set)
  if (ssd_workspace_bytes(dims, 0) == 0) return SSD_ERR_UNSUPPORTED;
  if (!x || !dt || !A || !B || !C || !D || !y)
    return reject(SSD_ERR_INVALID_ARG, "ssd_forward_noalloc: a required pointer is NULL");
  const void* ptrs[] = {x, dt, A, B, C, D, h0, y, final_state, chunk_states};
  for (const void* q : ptrs)
    if (q && ((uintptr_t)q & 15u))
      return reject(SSD_ERR_ALIGNMENT, "ssd_forward_noalloc: a pointer is not 16-byte aligned");

  Problem p;
  memset(&p, 0, sizeof p);
  p.B = (int)dims->batch;
  p.T = (int)dims->seqlen;
  p.H = (int)dims->nheads;
  p.P = (int)dims->headdim;
  p.N = (int)dims->dstate;
  p.G = (int)dims->ngroups;
  p.Q = (int)dims->chunk;
  p.nc = p.T / p.Q;
  p.hpg = p.H / p.G;
  p.bf16 = dims->dtype == SSD_BF16;
  if (simt_smem_need(p) > 227 * 1024)
    return reject(SSD_ERR_UNSUPPORTED, "ssd_forward_noalloc: shape needs too much shared memory");

  // scratch: per-chunk decay totals, plus the chunk states when the caller
  // passes no history buffer
  const size_t cl_bytes = align256((size_t)p.B * p.H * p.nc * sizeof(float));
  const size_t st_bytes = chunk_states ? 0 : align256((size_t)p.B * p.nc * p.H * p.P * p.N * sizeof(float));
  if (cl_bytes + st_bytes > (size_t)SSD_NOALLOC_SCRATCH_BYTES)
    return reject(SSD_ERR_UNSUPPORTED,
                  chunk_states
                      ? "ssd_forward_noalloc: problem needs more scratch than the built-in array "
                        "holds; use ssd_forward with a workspace"
                      : "ssd_forward_noalloc: without a chunk_states buffer the chunk states do "
                        "not fit in the built-in scratch; pass chunk_states or use ssd_forward");
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess || !scratch)
    return reject(SSD_ERR_CUDA, "ssd_forward_noalloc: cudaGetSymbolAddress of the scratch failed");

  p.x = x; p.dt = dt; p.A = A; p.Bm = B; p.Cm = C; p.D = D; p.h0 = h0;
  p.y = y; p.final_state = final_state;
  p.cs_last = (float*)scratch;
  p.hist = chunk_states ? chunk_states : (float*)((char*)scratch + cl_bytes);
  p.stream = (cudaStream_t)cuda_stream;

  const bool tc = tc_supported(p);
  e = tc ? tc_chunk_outer(p, 0, p.hist) : simt_forward_states(p, p.hist, p.cs_last);
  if (e == cudaSuccess) e = simt_state_pass_fwd(p, p.hist, p.cs_last);
  if (e == cudaSuccess) e = tc ? tc_forward_scan(p) : simt_forward_scan(p);
  if (e != cudaSuccess) return reject(SSD_ERR_CUDA, cudaGetErrorString(e));
  return SSD_OK;
}
