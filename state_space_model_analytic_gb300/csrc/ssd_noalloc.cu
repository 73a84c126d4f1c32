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
// device address is looked up per device (cudaGetSymbolAddress, with that
// device current) by the first call on that device that succeeds in the
// lookup; that first call should therefore come before any stream capture.
// A failed lookup is not remembered: the next call tries again.  All calls
// on a device share the one array and it keeps whatever the last call left
// in it, so calls whose kernels may overlap on the GPU (different streams,
// or different host threads) race on it; callers must order them.  The
// launch sequence is ssd_forward's for the same dims, so the outputs are
// bit-for-bit those of ssd_forward.  What must start at zero is cleared by
// the call itself on its stream (the single-pass forward's flags); every
// other scratch value is written before it is read.
#include <cstring>
#include <mutex>

#include "../../include/ssd.h"
#include "ssd_internal.h"

namespace ssd {

void set_last_error(const char* msg);

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SSD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  Only a
// successful lookup is cached; a failure is returned and retried next call.
cudaError_t scratch_address(void** out) {
  *out = nullptr;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
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
  int rc = validate_dims(dims);  // the codes and messages of ssd_forward
  if (rc != SSD_OK) return rc;
  if (!x || !dt || !A || !B || !C || !D || !y)
    return reject(SSD_ERR_INVALID_ARG, "ssd_forward_noalloc: a required pointer is NULL");
  const void* ptrs[] = {x, dt, A, B, C, D, h0, y, final_state, chunk_states};
  for (const void* q : ptrs)
    if (q && ((uintptr_t)q & 15u))
      return reject(SSD_ERR_ALIGNMENT, "ssd_forward_noalloc: a pointer is not 16-byte aligned");
  Problem p = problem_of(dims);
  if ((rc = check_shared_memory(p)) != SSD_OK) return rc;

  // scratch: per-chunk decay totals, the single-pass forward's flags (one per
  // history slot and its tile counter), and the chunk states when the caller
  // passes no history buffer; the block family on 128-step sub-chunks keeps
  // its decay totals and chunk states per sub-chunk, always in the scratch
  const bool sub = tc64_subchunks(p);
  const size_t ncw = sub ? (size_t)p.T / 128 : (size_t)p.nc;
  const size_t cl_bytes = align256((size_t)p.B * p.H * ncw * sizeof(float));
  const size_t fl_bytes = align256(((size_t)p.B * p.nc * p.H + 1) * sizeof(unsigned int));
  const size_t st_bytes = chunk_states && !sub
                              ? 0
                              : align256((size_t)p.B * ncw * p.H * p.P * p.N * sizeof(float));
  if (cl_bytes + fl_bytes + st_bytes > (size_t)SSD_NOALLOC_SCRATCH_BYTES)
    return reject(SSD_ERR_UNSUPPORTED,
                  chunk_states
                      ? "ssd_forward_noalloc: problem needs more scratch than the built-in array "
                        "holds; use ssd_forward with a workspace"
                      : "ssd_forward_noalloc: without a chunk_states buffer the chunk states do "
                        "not fit in the built-in scratch; pass chunk_states or use ssd_forward");
  // an error left by an earlier asynchronous launch is not this call's: clear
  // it so that the lookup below reports only its own outcome
  (void)cudaGetLastError();
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess || !scratch)
    return reject(SSD_ERR_CUDA, "ssd_forward_noalloc: cudaGetSymbolAddress of the scratch failed");

  p.x = x; p.dt = dt; p.A = A; p.Bm = B; p.Cm = C; p.D = D; p.h0 = h0;
  p.y = y; p.final_state = final_state;
  char* s = (char*)scratch;
  p.cs_last = (float*)s;
  p.fwd_flags = (unsigned int*)(s + cl_bytes);
  float* st = (float*)(s + cl_bytes + fl_bytes);
  if (sub) {
    p.hist_sub = st;
    p.hist = chunk_states;
  } else {
    p.hist = chunk_states ? chunk_states : st;
  }
  p.stream = (cudaStream_t)cuda_stream;

  // the launch sequence of ssd_forward for these dims
  const char* where = "";
  e = forward_launches(p, &where);
  if (e != cudaSuccess) return reject(SSD_ERR_CUDA, cudaGetErrorString(e));
  return SSD_OK;
}
