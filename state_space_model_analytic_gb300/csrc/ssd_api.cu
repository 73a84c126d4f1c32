// C ABI of the SSD core: argument validation, workspace carve-up and the
// launch sequence of each call.  Declarations and contracts: include/ssd.h.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/ssd.h"
#include "ssd_internal.h"

namespace ssd {

static std::atomic<uint64_t> g_launches{0};
void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

namespace {
struct TraceEvent {
  int name_id;
  cudaEvent_t start, stop;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
std::vector<TraceEvent> g_trace_slots;  // created by ssd_trace_begin
size_t g_trace_used = 0;
std::vector<std::string> g_trace_names;
std::vector<int> g_trace_untimed;

int trace_name_id(const char* name) {
  for (size_t i = 0; i < g_trace_names.size(); ++i)
    if (g_trace_names[i] == name) return (int)i;
  g_trace_names.emplace_back(name);
  g_trace_untimed.push_back(0);
  return (int)g_trace_names.size() - 1;
}
}  // namespace

int trace_open_slot(const char* name, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (!g_trace_on) return -1;
  const int id = trace_name_id(name);
  if (g_trace_used >= g_trace_slots.size()) {
    g_trace_untimed[id] += 1;
    return -1;
  }
  TraceEvent& ev = g_trace_slots[g_trace_used];
  ev.name_id = id;
  if (cudaEventRecord(ev.start, s) != cudaSuccess) return -1;
  return (int)g_trace_used++;
}

void trace_close_slot(int slot, cudaStream_t s) {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  cudaEventRecord(g_trace_slots[slot].stop, s);
}

size_t simt_smem_need(const Problem& p);
int simt_row_tile(const Problem& p);
bool tc_supported(const Problem& p);
bool tc_backward_supported(const Problem& p);
void tc_force_path(int path);
cudaError_t tc_chunk_outer(const Problem& p, int mode, float* out);
cudaError_t tc_forward_scan(const Problem& p);
cudaError_t tc_forward_single(const Problem& p);
bool tc_fused_states(const Problem& p);
cudaError_t tc_forward_states(const Problem& p);
cudaError_t tc_backward(const Problem& p);
cudaError_t tc_read_and_clear_error(unsigned int* out);
cudaError_t tc_selftest_timeout(cudaStream_t s);
bool tc64_supported(const Problem& p);
size_t tc64_bc_part_floats(const Problem& p);
cudaError_t tc64_chunk_outer(const Problem& p, int mode, float* out);
cudaError_t tc64_forward_scan(const Problem& p);
cudaError_t tc64_backward(const Problem& p);
cudaError_t tc64_read_and_clear_error(unsigned int* out);

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(SSD_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr size_t kAlign = 256;
size_t up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int validate(const ssd_dims* d) {
  if (!d) return fail(SSD_ERR_INVALID_ARG, "dims is NULL");
  if (d->batch < 1 || d->seqlen < 1 || d->nheads < 1 || d->headdim < 1 || d->dstate < 1 ||
      d->ngroups < 1 || d->chunk < 1)
    return fail(SSD_ERR_INVALID_ARG, "every dimension must be >= 1");
  if (d->reserved != 0) return fail(SSD_ERR_INVALID_ARG, "dims.reserved must be 0");
  if (d->dtype != SSD_F32 && d->dtype != SSD_BF16)
    return fail(SSD_ERR_INVALID_ARG, "dtype %d is not SSD_F32 or SSD_BF16", (int)d->dtype);
  if (d->nheads % d->ngroups)
    return fail(SSD_ERR_INVALID_ARG, "nheads %lld is not a multiple of ngroups %lld",
                (long long)d->nheads, (long long)d->ngroups);
  const int64_t q = d->chunk;
  if (q != 16 && q != 32 && q != 64 && q != 128 && q != 256)
    return fail(SSD_ERR_UNSUPPORTED, "chunk %lld not in {16,32,64,128,256}", (long long)q);
  if (d->seqlen % q)
    return fail(SSD_ERR_UNSUPPORTED, "seqlen %lld is not a multiple of chunk %lld",
                (long long)d->seqlen, (long long)q);
  if (d->headdim % 16 || d->headdim > 128)
    return fail(SSD_ERR_UNSUPPORTED, "headdim %lld must be a multiple of 16 in [16,128]",
                (long long)d->headdim);
  if (d->dstate % 16 || d->dstate > 256)
    return fail(SSD_ERR_UNSUPPORTED, "dstate %lld must be a multiple of 16 in [16,256]",
                (long long)d->dstate);
  if (d->headdim * d->dstate > 16384)
    return fail(SSD_ERR_UNSUPPORTED, "headdim * dstate must be <= 16384");
  // every flat index must fit comfortably in 63 bits and grid limits
  if (d->batch > 65535 / 2 || d->nheads > 65535)
    return fail(SSD_ERR_UNSUPPORTED, "batch or nheads too large for the launch grid");
  const double elems = (double)d->batch * (double)d->seqlen * (double)d->nheads * (double)d->headdim;
  if (elems > 4.0e12) return fail(SSD_ERR_UNSUPPORTED, "problem too large");
  return SSD_OK;
}

Problem base_problem(const ssd_dims* d) {
  Problem p;
  memset(&p, 0, sizeof p);
  p.B = (int)d->batch;
  p.T = (int)d->seqlen;
  p.H = (int)d->nheads;
  p.P = (int)d->headdim;
  p.N = (int)d->dstate;
  p.G = (int)d->ngroups;
  p.Q = (int)d->chunk;
  p.nc = p.T / p.Q;
  p.hpg = p.H / p.G;
  p.bf16 = d->dtype == SSD_BF16;
  return p;
}

// Workspace layout.  which: 0 forward, 1 backward with history, 2 backward
// recomputing the history.  Carves into `p` when base != nullptr.
size_t carve(Problem* p, char* base, int which) {
  const size_t B = p->B, T = p->T, H = p->H, P = p->P, N = p->N, nc = p->nc, Q = p->Q;
  // the block family on 128-step sub-chunks keeps its per-chunk buffers (the
  // decay totals, the state gradients and its own chunk-start states) at
  // sub-chunk granularity
  const bool sub = tc64_subchunks(*p);
  const size_t ncw = sub ? T / 128 : nc;
  const size_t states = B * ncw * H * P * N * sizeof(float);
  const size_t tokh = B * T * H * sizeof(float);
  size_t off = 0;
  auto take = [&](size_t bytes) -> char* {
    char* r = base ? base + off : nullptr;
    off += up(bytes);
    return r;
  };
  p->cs_last = (float*)take(B * H * ncw * sizeof(float));
  if (sub) {
    p->hist_sub = (float*)take(states);
    if (which == 0) return off;
  }
  if (which == 0) {
    float* h = (float*)take(states);
    if (!p->hist) p->hist = h;
    // single-pass tensor-core forward: one ready flag per history slot, then
    // its tile counter
    p->fwd_flags = (unsigned int*)take((B * nc * H + 1) * sizeof(unsigned int));
    return off;
  }
  p->dstate = (float*)take(states);
  p->rowsum = (float*)take(tokh);
  p->colsum = (float*)take(tokh);
  p->statein = (float*)take(tokh);
  p->eout = (float*)take(tokh);
  p->drive = (float*)take(tokh);
  p->dA_part = (float*)take(B * nc * (Q / 16) * H * sizeof(float));  // per (chunk, tile or block)
  p->dD_part = (float*)take(B * nc * (Q / 16) * H * sizeof(float));
  p->dtb_part = (float*)take(B * nc * (Q / 16) * H * sizeof(float));
  // tensor-core backward: one counter for all CTAs, then per (b, g, chunk,
  // 128-row block) unit an arrival ticket and a written-partials counter; fp32
  // partials of dC, dB (2 x 128 x 128 floats) in two slots per CTA, at most
  // kBwdMaxCtas CTAs and one per (unit, head) item
  const size_t units = B * (size_t)p->G * nc * ((Q + 127) / 128);
  const size_t items = units * (size_t)p->hpg;
  p->ntickets = (int)(1 + 2 * units);
  p->tickets = (unsigned int*)take((1 + 2 * units) * sizeof(unsigned int));
  // (the d_state-64 tensor-core backward keeps its per-segment dC, dB partials there)
  size_t part_floats = (items < kBwdMaxCtas ? items : kBwdMaxCtas) * 2 * 32768;
  if (tc64_supported(*p) && tc64_bc_part_floats(*p) > part_floats)
    part_floats = tc64_bc_part_floats(*p);
  p->bwd_part = (float*)take(part_floats * sizeof(float));
  if (sub) return off;  // (its backward recomputes hist_sub itself)
  p->hT = take(states / 2);  // bf16 copies for the tensor-core backward
  p->gT = take(states / 2);
  if (Q == 256) p->gmT = take(states / 2);
  if (which == 2) p->hist = (float*)take(states);
  return off;
}

// Workspace in front of the core's for ssd_forward_raw / ssd_backward_raw:
// dt [B][T][H] fp32, then A [H] fp32, then the per-slice dt_bias sums
// [kDtPostSlices][H] fp32 of the backward.
size_t raw_extra_bytes(const Problem& p) {
  return up((size_t)p.B * p.T * p.H * sizeof(float)) + up((size_t)p.H * sizeof(float)) +
         up((size_t)kDtPostSlices * p.H * sizeof(float));
}

int check_smem(const Problem& p) {
  if (simt_smem_need(p) > 227 * 1024)
    return fail(SSD_ERR_UNSUPPORTED, "shape needs %zu bytes of shared memory per block",
                simt_smem_need(p));
  return SSD_OK;
}

}  // namespace

void set_last_error(const char* msg) { g_err = msg; }

// The kernels of one forward call for the carved problem `p` (shared with
// ssd_forward_noalloc, so both run the same sequence); *where names the
// kernel whose launch failed.
cudaError_t forward_launches(Problem& p, const char** where) {
  const bool tc = tc_supported(p);
  cudaError_t e;
  if (tc && tc_fused_states(p)) {
    // one kernel: chunk states, the state pass (look-back) and y
    *where = "single-pass forward kernel";
    return tc_forward_single(p);
  }
  if (tc64_supported(p)) {  // the block family (fp32 through split bf16 products)
    const bool sub = tc64_subchunks(p);
    Problem s = sub ? tc64_sub_problem(p) : p;
    *where = "forward chunk-state kernel";
    if ((e = tc64_chunk_outer(s, 0, s.hist)) != cudaSuccess) return e;
    *where = "forward state-pass kernel";
    if ((e = simt_state_pass_fwd(s, s.hist, s.cs_last)) != cudaSuccess) return e;
    *where = "forward chunk-scan kernel";
    if ((e = tc64_forward_scan(s)) != cudaSuccess) return e;
    if (sub && p.hist) {
      // the caller's chunk-start states: every (Q / 128)-th sub-chunk's
      *where = "forward history copy";
      const size_t blk = (size_t)p.H * p.P * p.N * sizeof(float);
      return cudaMemcpy2DAsync(p.hist, blk, s.hist, blk * (p.Q / 128), blk, (size_t)p.B * p.nc,
                               cudaMemcpyDeviceToDevice, p.stream);
    }
    return cudaSuccess;
  }
  p.hT = nullptr;  // the scan converts the fp32 history itself
  *where = "forward chunk-state kernel";
  e = tc ? tc_chunk_outer(p, 0, p.hist) : simt_forward_states(p, p.hist, p.cs_last);
  if (e != cudaSuccess) return e;
  *where = "forward state-pass kernel";
  if ((e = simt_state_pass_fwd(p, p.hist, p.cs_last)) != cudaSuccess) return e;
  *where = "forward chunk-scan kernel";
  return tc ? tc_forward_scan(p) : simt_forward_scan(p);
}


// The checks and problem set-up of ssd_forward, for the other entry points.
int validate_dims(const ssd_dims* d) { return validate(d); }
Problem problem_of(const ssd_dims* d) { return base_problem(d); }
int check_shared_memory(const Problem& p) { return check_smem(p); }

}  // namespace ssd

using namespace ssd;

extern "C" {

const char* ssd_last_error(void) { return g_err.c_str(); }

int ssd_trace_reset(void) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  for (auto& e : g_trace_slots) {
    cudaEventDestroy(e.start);
    cudaEventDestroy(e.stop);
  }
  g_trace_slots.clear();
  g_trace_used = 0;
  g_trace_names.clear();
  g_trace_untimed.clear();
  g_trace_on = false;
  return SSD_OK;
}

int ssd_trace_begin(int capacity) {
  g_err.clear();
  if (capacity < 1 || capacity > (1 << 20))
    return fail(SSD_ERR_INVALID_ARG, "trace capacity %d out of range", capacity);
  ssd_trace_reset();
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_slots.reserve((size_t)capacity);
  for (int i = 0; i < capacity; ++i) {
    TraceEvent e{0, nullptr, nullptr};
    cudaError_t r = cudaEventCreate(&e.start);
    if (r == cudaSuccess) r = cudaEventCreate(&e.stop);
    if (r != cudaSuccess) return cuda_fail(r, "ssd_trace_begin: cudaEventCreate");
    g_trace_slots.push_back(e);
  }
  g_trace_on = true;
  return SSD_OK;
}

int ssd_trace_end(void) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_on = false;
  return SSD_OK;
}

int ssd_trace_read(int index, char* name, int name_len, double* total_ms, int* launches,
                   int* untimed) {
  g_err.clear();
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (index < 0 || index >= (int)g_trace_names.size())
    return fail(SSD_ERR_INVALID_ARG, "trace index %d out of range", index);
  double ms = 0.0;
  int n = 0;
  for (size_t i = 0; i < g_trace_used; ++i) {
    const TraceEvent& e = g_trace_slots[i];
    if (e.name_id != index) continue;
    cudaError_t r = cudaEventSynchronize(e.stop);
    float t = 0.f;
    if (r == cudaSuccess) r = cudaEventElapsedTime(&t, e.start, e.stop);
    if (r != cudaSuccess) return cuda_fail(r, "ssd_trace_read");
    ms += t;
    ++n;
  }
  if (name && name_len > 0) snprintf(name, (size_t)name_len, "%s", g_trace_names[index].c_str());
  if (total_ms) *total_ms = ms;
  if (launches) *launches = n;
  if (untimed) *untimed = g_trace_untimed[index];
  return SSD_OK;
}

uint64_t ssd_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

size_t ssd_workspace_bytes(const ssd_dims* dims, int which) {
  if (validate(dims) != SSD_OK || which < 0 || which > 5) return 0;
  Problem p = base_problem(dims);
  // 3..5: the raw-dt entry points, dt and A in front of the core's workspace
  return (which >= 3 ? raw_extra_bytes(p) : 0) + carve(&p, nullptr, which % 3);
}

int ssd_force_kernel_path(int path) {
  if (path != -1 && path != 0) return fail(SSD_ERR_INVALID_ARG, "path must be -1 or 0");
  tc_force_path(path);
  return SSD_OK;
}

int ssd_device_status(void) {
  g_err.clear();
  unsigned int flag = 0, conv_flag = 0, tc64_flag = 0;
  cudaError_t e = tc_read_and_clear_error(&flag);
  if (e == cudaSuccess) e = conv_read_and_clear_error(&conv_flag);
  if (e == cudaSuccess) e = tc64_read_and_clear_error(&tc64_flag);
  if (e != cudaSuccess) return cuda_fail(e, "ssd_device_status");
  flag |= conv_flag << 8;
  flag |= tc64_flag << 16;
  if (flag) return fail(SSD_ERR_DEVICE_TIMEOUT, "a device-side wait gave up (flag 0x%x)", flag);
  return SSD_OK;
}

int ssd_selftest_wait_timeout(void* cuda_stream) {
  g_err.clear();
  cudaError_t e = tc_selftest_timeout((cudaStream_t)cuda_stream);
  if (e != cudaSuccess) return cuda_fail(e, "ssd_selftest_wait_timeout");
  return SSD_OK;
}

int ssd_kernel_path(const ssd_dims* dims) {
  if (validate(dims) != SSD_OK) return -1;
  Problem p = base_problem(dims);
  return (tc_supported(p) || tc64_supported(p)) ? 1 : 0;
}

// The raw-dt mode of the fused tensor-core path (ssd_forward_raw /
// ssd_backward_raw): dt holds dt_raw; the kernels apply softplus(dt_raw +
// dt_bias) and A = -exp(a_log) where they read dt and A, and the backward
// returns the gradients w.r.t. dt_raw (in ddt), a_log (in dA) and dt_bias.
struct RawDt {
  const float* dt_bias;
  const float* a_log;
  float* d_dt_bias;
};

namespace {
int forward_impl(const ssd_dims* dims, const void* x, const float* dt, const float* A,
                const void* B, const void* C, const float* D, const float* h0, void* y,
                float* final_state, float* chunk_states, void* workspace, size_t workspace_bytes,
                void* cuda_stream, const RawDt* raw) {
  g_err.clear();
  int rc = validate(dims);
  if (rc) return rc;
  if (!x || !dt || !A || !B || !C || !D || !y || !workspace)
    return fail(SSD_ERR_INVALID_ARG, "ssd_forward: a required pointer is NULL");
  const void* ptrs[] = {x, dt, A, B, C, D, h0, y, final_state, chunk_states};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return fail(SSD_ERR_ALIGNMENT, "ssd_forward: pointer %p is not 16-byte aligned", q);
  if (((uintptr_t)workspace & 255u) != 0)
    return fail(SSD_ERR_ALIGNMENT, "ssd_forward: workspace must be 256-byte aligned");
  Problem p = base_problem(dims);
  if ((rc = check_smem(p))) return rc;
  p.x = x; p.dt = dt; p.A = A; p.Bm = B; p.Cm = C; p.D = D; p.h0 = h0;
  p.y = y; p.final_state = final_state; p.hist = chunk_states;
  if (raw) {
    p.dt_bias = raw->dt_bias;
    p.a_log = raw->a_log;
  }
  const size_t need = carve(&p, nullptr, 0);
  if (workspace_bytes < need)
    return fail(SSD_ERR_INVALID_ARG, "ssd_forward: workspace %zu bytes < %zu needed",
                workspace_bytes, need);
  p.hist = chunk_states;
  carve(&p, (char*)workspace, 0);
  p.stream = (cudaStream_t)cuda_stream;

  if (raw && !(tc_supported(p) && tc_fused_states(p)))
    return fail(SSD_ERR_UNSUPPORTED, "ssd_forward: raw-dt mode needs the fused tensor-core path");
  const char* where = "";
  const cudaError_t e = forward_launches(p, &where);
  if (e != cudaSuccess) return cuda_fail(e, where);
  return SSD_OK;
}
}  // namespace

int ssd_forward(const ssd_dims* dims, const void* x, const float* dt, const float* A,
                const void* B, const void* C, const float* D, const float* h0, void* y,
                float* final_state, float* chunk_states, void* workspace, size_t workspace_bytes,
                void* cuda_stream) {
  return forward_impl(dims, x, dt, A, B, C, D, h0, y, final_state, chunk_states, workspace,
                      workspace_bytes, cuda_stream, nullptr);
}

namespace {
int backward_impl(const ssd_dims* dims, const void* x, const float* dt, const float* A,
                 const void* B, const void* C, const float* D, const float* h0, const void* dy,
                 const float* chunk_states, void* dx, float* ddt, float* dA, void* dB, void* dC,
                 float* dD, float* dh0, void* workspace, size_t workspace_bytes,
                 void* cuda_stream, const RawDt* raw) {
  g_err.clear();
  int rc = validate(dims);
  if (rc) return rc;
  if (!x || !dt || !A || !B || !C || !D || !dy || !dx || !ddt || !dA || !dB || !dC || !dD ||
      !workspace)
    return fail(SSD_ERR_INVALID_ARG, "ssd_backward: a required pointer is NULL");
  const void* ptrs[] = {x, dt, A, B, C, D, h0, dy, chunk_states, dx, ddt, dA, dB, dC, dD, dh0};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return fail(SSD_ERR_ALIGNMENT, "ssd_backward: pointer %p is not 16-byte aligned", q);
  if (((uintptr_t)workspace & 255u) != 0)
    return fail(SSD_ERR_ALIGNMENT, "ssd_backward: workspace must be 256-byte aligned");
  Problem p = base_problem(dims);
  if ((rc = check_smem(p))) return rc;
  const int which = chunk_states ? 1 : 2;
  const size_t need = carve(&p, nullptr, which);
  if (workspace_bytes < need)
    return fail(SSD_ERR_INVALID_ARG, "ssd_backward: workspace %zu bytes < %zu needed%s",
                workspace_bytes, need, chunk_states ? "" : " (recomputing chunk states)");
  p.x = x; p.dt = dt; p.A = A; p.Bm = B; p.Cm = C; p.D = D; p.h0 = h0; p.dy = dy;
  p.dx = dx; p.ddt = ddt; p.dA = dA; p.dB = dB; p.dC = dC; p.dD = dD; p.dh0 = dh0;
  if (raw) {
    p.dt_bias = raw->dt_bias;
    p.a_log = raw->a_log;
    p.d_dt_bias = raw->d_dt_bias;
    if (!(tc_supported(p) && tc_fused_states(p)))
      return fail(SSD_ERR_UNSUPPORTED, "ssd_backward: raw-dt mode needs the fused tensor-core path");
  }
  p.hist = nullptr;
  carve(&p, (char*)workspace, which);
  if (chunk_states) p.hist = const_cast<float*>(chunk_states);
  p.stream = (cudaStream_t)cuda_stream;

  cudaError_t e;
  if (tc64_subchunks(p)) {
    // the block family on 128-step sub-chunks: their start states are not in
    // the caller's chunk-level history, so they are recomputed (the same
    // kernels as the forward: the caller's history holds the same values)
    Problem s = tc64_sub_problem(p);
    s.final_state = nullptr;
    e = tc64_chunk_outer(s, 0, s.hist);
    if (e == cudaSuccess) e = simt_state_pass_fwd(s, s.hist, s.cs_last);
    if (e != cudaSuccess) return cuda_fail(e, "backward sub-chunk state kernels");
    e = tc64_backward(s);
    if (e != cudaSuccess) return cuda_fail(e, "backward kernels");
    return SSD_OK;
  }
  if (!chunk_states) {
    // recompute the chunk-start states into the workspace (final state not needed)
    Problem f = p;
    f.final_state = nullptr;
    if (tc_supported(f) && tc_fused_states(f)) {
      e = tc_forward_states(f);
      if (e != cudaSuccess) return cuda_fail(e, "backward recompute state-scan kernel");
    } else {
      e = tc_supported(f)     ? tc_chunk_outer(f, 0, f.hist)
          : tc64_supported(f) ? tc64_chunk_outer(f, 0, f.hist)
                              : simt_forward_states(f, f.hist, f.cs_last);
      if (e != cudaSuccess) return cuda_fail(e, "backward recompute chunk-state kernel");
      e = simt_state_pass_fwd(f, f.hist, f.cs_last);
      if (e != cudaSuccess) return cuda_fail(e, "backward recompute state-pass kernel");
    }
  }
  e = tc_backward_supported(p) ? tc_backward(p)
      : tc64_supported(p)       ? tc64_backward(p)
                                : simt_backward(p);
  if (e != cudaSuccess) return cuda_fail(e, "backward kernels");
  return SSD_OK;
}
}  // namespace

int ssd_backward(const ssd_dims* dims, const void* x, const float* dt, const float* A,
                 const void* B, const void* C, const float* D, const float* h0, const void* dy,
                 const float* chunk_states, void* dx, float* ddt, float* dA, void* dB, void* dC,
                 float* dD, float* dh0, void* workspace, size_t workspace_bytes,
                 void* cuda_stream) {
  return backward_impl(dims, x, dt, A, B, C, D, h0, dy, chunk_states, dx, ddt, dA, dB, dC, dD,
                       dh0, workspace, workspace_bytes, cuda_stream, nullptr);
}

// ---- dt and A preprocessing in front of the core (ssd_dtprep.cu) ----------

int ssd_forward_raw(const ssd_dims* dims, const void* x, const float* dt_raw, const float* dt_bias,
                    const float* a_log, const void* B, const void* C, const float* D,
                    const float* h0, void* y, float* final_state, float* chunk_states,
                    void* workspace, size_t workspace_bytes, void* cuda_stream) {
  g_err.clear();
  int rc = validate(dims);
  if (rc) return rc;
  if (!x || !dt_raw || !dt_bias || !a_log || !B || !C || !D || !y || !workspace)
    return fail(SSD_ERR_INVALID_ARG, "ssd_forward_raw: a required pointer is NULL");
  const void* ptrs[] = {x, dt_raw, dt_bias, a_log, B, C, D, h0, y, final_state, chunk_states};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return fail(SSD_ERR_ALIGNMENT, "ssd_forward_raw: pointer %p is not 16-byte aligned", q);
  if (((uintptr_t)workspace & 255u) != 0)
    return fail(SSD_ERR_ALIGNMENT, "ssd_forward_raw: workspace must be 256-byte aligned");
  Problem p = base_problem(dims);
  if ((rc = check_smem(p))) return rc;
  const size_t need = ssd_workspace_bytes(dims, 3), extra = raw_extra_bytes(p);
  if (workspace_bytes < need)
    return fail(SSD_ERR_INVALID_ARG, "ssd_forward_raw: workspace %zu bytes < %zu needed",
                workspace_bytes, need);
  // the fused tensor-core path applies softplus and -exp where it reads dt and A
  if (tc_supported(p) && tc_fused_states(p)) {
    const RawDt raw{dt_bias, a_log, nullptr};
    return forward_impl(dims, x, dt_raw, a_log, B, C, D, h0, y, final_state, chunk_states,
                        (char*)workspace + extra, workspace_bytes - extra, cuda_stream, &raw);
  }
  float* dt = (float*)workspace;
  float* A = (float*)((char*)workspace + up((size_t)p.B * p.T * p.H * sizeof(float)));
  p.stream = (cudaStream_t)cuda_stream;
  cudaError_t e = dt_prep(p, dt_raw, dt_bias, a_log, dt, A);
  if (e != cudaSuccess) return cuda_fail(e, "dt preprocessing kernel");
  return ssd_forward(dims, x, dt, A, B, C, D, h0, y, final_state, chunk_states,
                     (char*)workspace + extra, workspace_bytes - extra, cuda_stream);
}

int ssd_backward_raw(const ssd_dims* dims, const void* x, const float* dt_raw,
                     const float* dt_bias, const float* a_log, const void* B, const void* C,
                     const float* D, const float* h0, const void* dy, const float* chunk_states,
                     void* dx, float* d_dt_raw, float* d_dt_bias, float* d_a_log, void* dB,
                     void* dC, float* dD, float* dh0, void* workspace, size_t workspace_bytes,
                     void* cuda_stream) {
  g_err.clear();
  int rc = validate(dims);
  if (rc) return rc;
  if (!x || !dt_raw || !dt_bias || !a_log || !B || !C || !D || !dy || !dx || !d_dt_raw ||
      !d_dt_bias || !d_a_log || !dB || !dC || !dD || !workspace)
    return fail(SSD_ERR_INVALID_ARG, "ssd_backward_raw: a required pointer is NULL");
  const void* ptrs[] = {x, dt_raw, dt_bias, a_log, B, C, D, h0, dy, chunk_states, dx,
                        d_dt_raw, d_dt_bias, d_a_log, dB, dC, dD, dh0};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return fail(SSD_ERR_ALIGNMENT, "ssd_backward_raw: pointer %p is not 16-byte aligned", q);
  if (((uintptr_t)workspace & 255u) != 0)
    return fail(SSD_ERR_ALIGNMENT, "ssd_backward_raw: workspace must be 256-byte aligned");
  Problem p = base_problem(dims);
  if ((rc = check_smem(p))) return rc;
  const size_t need = ssd_workspace_bytes(dims, chunk_states ? 4 : 5), extra = raw_extra_bytes(p);
  if (workspace_bytes < need)
    return fail(SSD_ERR_INVALID_ARG, "ssd_backward_raw: workspace %zu bytes < %zu needed%s",
                workspace_bytes, need, chunk_states ? "" : " (recomputing chunk states)");
  // the fused tensor-core path: softplus and -exp where dt and A are read, the
  // gradients w.r.t. dt_raw, dt_bias and a_log formed where ddt and dA are
  if (tc_supported(p) && tc_fused_states(p)) {
    const RawDt raw{dt_bias, a_log, d_dt_bias};
    return backward_impl(dims, x, dt_raw, a_log, B, C, D, h0, dy, chunk_states, dx, d_dt_raw,
                         d_a_log, dB, dC, dD, dh0, (char*)workspace + extra,
                         workspace_bytes - extra, cuda_stream, &raw);
  }
  float* dt = (float*)workspace;
  float* A = (float*)((char*)workspace + up((size_t)p.B * p.T * p.H * sizeof(float)));
  p.stream = (cudaStream_t)cuda_stream;
  cudaError_t e = dt_prep(p, dt_raw, dt_bias, a_log, dt, A);
  if (e != cudaSuccess) return cuda_fail(e, "dt preprocessing kernel");
  // the core writes ddt into d_dt_raw and dA into d_a_log; the post kernel
  // turns them into the gradients w.r.t. dt_raw, dt_bias and a_log in place
  rc = ssd_backward(dims, x, dt, A, B, C, D, h0, dy, chunk_states, dx, d_dt_raw, d_a_log, dB, dC,
                    dD, dh0, (char*)workspace + extra, workspace_bytes - extra, cuda_stream);
  if (rc) return rc;
  float* part = (float*)((char*)A + up((size_t)p.H * sizeof(float)));
  e = dt_post(p, dt_raw, dt_bias, a_log, d_dt_raw, d_dt_bias, d_a_log, part);
  if (e != cudaSuccess) return cuda_fail(e, "dt gradient kernel");
  return SSD_OK;
}

// ---- gated RMSNorm after the core (ssd_norm.cu) ---------------------------

namespace {
int norm_check(const char* who, long long rows, long long width, int dtype, float eps) {
  if (rows < 1) return fail(SSD_ERR_INVALID_ARG, "%s: rows must be >= 1", who);
  if (dtype != SSD_F32 && dtype != SSD_BF16) return fail(SSD_ERR_INVALID_ARG, "%s: bad dtype", who);
  const long long unit = dtype == SSD_BF16 ? 256 : 128;  // 32 lanes x 16 bytes
  if (width < unit || width > 4096 || width % unit != 0)
    return fail(SSD_ERR_UNSUPPORTED, "%s: width %lld must be a multiple of %lld in [%lld, 4096]",
                who, width, unit, unit);
  if (!(eps >= 0.f)) return fail(SSD_ERR_INVALID_ARG, "%s: eps must be >= 0", who);
  return SSD_OK;
}
}  // namespace

size_t ssd_rmsnorm_gated_workspace_bytes(int64_t rows, int64_t width) {
  if (rows < 1 || width < 1 || width > 4096) return 0;
  return up((size_t)kNormMaxCtas * width * sizeof(float));
}

int ssd_rmsnorm_gated_forward(int64_t rows, int64_t width, int32_t dtype, const void* y,
                              const void* z, const float* weight, float eps, void* out,
                              float* inv_rms, void* cuda_stream) {
  g_err.clear();
  int rc = norm_check("ssd_rmsnorm_gated_forward", rows, width, dtype, eps);
  if (rc) return rc;
  if (!y || !z || !weight || !out)
    return fail(SSD_ERR_INVALID_ARG, "ssd_rmsnorm_gated_forward: a required pointer is NULL");
  const void* ptrs[] = {y, z, weight, out, inv_rms};
  for (const void* q : ptrs)
    if (q && !aligned16(q))
      return fail(SSD_ERR_ALIGNMENT, "ssd_rmsnorm_gated_forward: pointer %p is not 16-byte aligned", q);
  cudaError_t e = norm_forward(rows, (int)width, dtype == SSD_BF16, y, z, weight, eps, out, inv_rms,
                               (cudaStream_t)cuda_stream);
  if (e != cudaSuccess) return cuda_fail(e, "gated RMSNorm forward kernel");
  return SSD_OK;
}

int ssd_rmsnorm_gated_backward(int64_t rows, int64_t width, int32_t dtype, const void* y,
                               const void* z, const float* weight, float eps,
                               const float* inv_rms, const void* dout, void* dy, void* dz,
                               float* dweight, void* workspace, size_t workspace_bytes,
                               void* cuda_stream) {
  g_err.clear();
  int rc = norm_check("ssd_rmsnorm_gated_backward", rows, width, dtype, eps);
  if (rc) return rc;
  if (!y || !z || !weight || !dout || !dy || !dz || !dweight || !workspace)
    return fail(SSD_ERR_INVALID_ARG, "ssd_rmsnorm_gated_backward: a required pointer is NULL");
  const void* ptrs[] = {y, z, weight, inv_rms, dout, dy, dz, dweight, workspace};
  for (const void* q : ptrs)
    if (q && !aligned16(q))
      return fail(SSD_ERR_ALIGNMENT, "ssd_rmsnorm_gated_backward: pointer %p is not 16-byte aligned", q);
  const size_t need = ssd_rmsnorm_gated_workspace_bytes(rows, width);
  if (workspace_bytes < need)
    return fail(SSD_ERR_INVALID_ARG, "ssd_rmsnorm_gated_backward: workspace %zu bytes < %zu needed",
                workspace_bytes, need);
  cudaError_t e = norm_backward(rows, (int)width, dtype == SSD_BF16, y, z, weight, eps, inv_rms,
                                dout, dy, dz, dweight, (float*)workspace, (cudaStream_t)cuda_stream);
  if (e != cudaSuccess) return cuda_fail(e, "gated RMSNorm backward kernels");
  return SSD_OK;
}

// ---- causal depthwise conv1d + SiLU before the core (ssd_conv.cu) --------

namespace {
int conv_check(const char* who, long long B, long long T, long long C, int K, int dtype) {
  if (B < 1 || B > 65535 || T < 1 || B * T > (1ll << 31) - 1024)
    return fail(SSD_ERR_INVALID_ARG, "%s: batch must be in [1, 65535], seqlen >= 1 and batch * "
                "seqlen below 2^31 - 1024", who);
  if (dtype != SSD_F32 && dtype != SSD_BF16) return fail(SSD_ERR_INVALID_ARG, "%s: bad dtype", who);
  const long long e = dtype == SSD_BF16 ? 8 : 4;  // channels per 16-byte chunk
  if (C < e || C % e != 0)
    return fail(SSD_ERR_UNSUPPORTED, "%s: channels must be a positive multiple of %lld", who, e);
  if (K < 1 || K > 4) return fail(SSD_ERR_UNSUPPORTED, "%s: d_conv must be in [1, 4]", who);
  return SSD_OK;
}
}  // namespace

size_t ssd_conv1d_silu_workspace_bytes(int64_t batch, int64_t seqlen, int64_t channels,
                                       int32_t d_conv) {
  if (batch < 1 || seqlen < 1 || channels < 1 || d_conv < 1 || d_conv > 4) return 0;
  const size_t tiles = (size_t)conv_max_ctas_per_column(seqlen);
  return up((size_t)batch * tiles * channels * (d_conv + 1) * sizeof(float));
}

int ssd_conv1d_silu_forward(int64_t batch, int64_t seqlen, int64_t channels, int32_t d_conv,
                            int32_t dtype, const void* x, const float* weight, const float* bias,
                            const float* init_state, void* out, void* cuda_stream) {
  g_err.clear();
  int rc = conv_check("ssd_conv1d_silu_forward", batch, seqlen, channels, d_conv, dtype);
  if (rc) return rc;
  if (!x || !weight || !out)
    return fail(SSD_ERR_INVALID_ARG, "ssd_conv1d_silu_forward: a required pointer is NULL");
  const void* ptrs[] = {x, weight, bias, init_state, out};
  for (const void* q : ptrs)
    if (q && !aligned16(q))
      return fail(SSD_ERR_ALIGNMENT, "ssd_conv1d_silu_forward: pointer %p is not 16-byte aligned", q);
  cudaError_t e = conv_forward(batch, (int)seqlen, (int)channels, d_conv, dtype == SSD_BF16, x,
                               weight, bias, init_state, out, (cudaStream_t)cuda_stream);
  if (e != cudaSuccess) return cuda_fail(e, "conv1d forward kernel");
  return SSD_OK;
}

int ssd_conv1d_silu_backward(int64_t batch, int64_t seqlen, int64_t channels, int32_t d_conv,
                             int32_t dtype, const void* x, const float* weight, const float* bias,
                             const float* init_state, const void* dout, void* dx, float* dweight,
                             float* dbias, void* workspace, size_t workspace_bytes,
                             void* cuda_stream) {
  g_err.clear();
  int rc = conv_check("ssd_conv1d_silu_backward", batch, seqlen, channels, d_conv, dtype);
  if (rc) return rc;
  if (!x || !weight || !dout || !dx || !dweight || !workspace)
    return fail(SSD_ERR_INVALID_ARG, "ssd_conv1d_silu_backward: a required pointer is NULL");
  const void* ptrs[] = {x, weight, bias, init_state, dout, dx, dweight, dbias, workspace};
  for (const void* q : ptrs)
    if (q && !aligned16(q))
      return fail(SSD_ERR_ALIGNMENT, "ssd_conv1d_silu_backward: pointer %p is not 16-byte aligned", q);
  const size_t need = ssd_conv1d_silu_workspace_bytes(batch, seqlen, channels, d_conv);
  if (workspace_bytes < need)
    return fail(SSD_ERR_INVALID_ARG, "ssd_conv1d_silu_backward: workspace %zu bytes < %zu needed",
                workspace_bytes, need);
  cudaError_t e = conv_backward(batch, (int)seqlen, (int)channels, d_conv, dtype == SSD_BF16, x,
                                weight, bias, init_state, dout, dx, dweight, dbias,
                                (float*)workspace, (cudaStream_t)cuda_stream);
  if (e != cudaSuccess) return cuda_fail(e, "conv1d backward kernels");
  return SSD_OK;
}

}  // extern "C"
