// Host runtime of libafd: the C ABI of include/afd.h, the context's arenas,
// the exchange state machine and the kernel launches.
//
// The call order, ownership and stream rules are those of the afdEP-comm
// "API contract" page (Roles and tensors; Graphs, streams and lifetime),
// restated for one GPU: sources and workers are index arguments on one
// context, and the exchange's kernels are ordered by the caller's stream(s).
// No call allocates device memory after afd_create and none synchronizes
// unless read_host_counts asks for it, so a complete exchange can be captured
// in a CUDA graph.

#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <new>

#include "afd.h"
#include "afd_internal.cuh"

using afd::CombineParams;
using afd::DispatchParams;
using afd::SourceDesc;

namespace {

enum Phase { kIdle = 0, kStaging = 1, kDispatched = 2, kReplied = 3 };

int64_t align_up64(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

}  // namespace

struct afd_ctx {
  afd_config cfg;
  int device;
  int sm_count;
  int sm_cap;
  int layout_max_ctas;  // largest layout cluster this device runs
  int wait_polls;       // polls of a bulk row load before the scatter gives up
  int Ef;
  int row_bytes;
  int nscale;
  int64_t R_arena;

  // device arenas (owned)
  uint8_t* rows;
  float* row_scales;
  float* row_w;
  int32_t* row_src;
  int32_t* starts;
  int32_t* ends;
  int32_t* hcounts;
  int2* routes;
  int32_t* route_tmp;
  unsigned long long* err;
  uint16_t* inbox;
  // pinned host
  int32_t* host_counts;
  unsigned long long* host_err;

  cudaEvent_t order_ev;
  cudaStream_t last_stream;
  bool last_captured;
  bool has_last;

  // current exchange
  uint64_t gen;
  int phase;
  int bucket;
  int rhc;
  bool cached;          // this exchange reuses the last layout
  // the last call of this exchange launched a combine on combine_stream (the
  // next combine on that stream may start without the dependency wait)
  bool combine_last;
  cudaStream_t combine_stream;
  bool combine_captured;
  // the last layout that a dispatch computed (what a cached dispatch reuses)
  bool layout_valid;
  int layout_bucket;
  int32_t layout_T[afd::kMaxSources];
  int staged_n;
  int replied_n;
  int collected_n;
  SourceDesc src[afd::kMaxSources];
  bool staged[afd::kMaxSources];
  bool collected[afd::kMaxSources];
  bool received[afd::kMaxWorkers];
  bool replied[afd::kMaxWorkers];
  int64_t recv_rows[afd::kMaxWorkers];
  const uint16_t* reply[afd::kMaxWorkers];

  char detail[256];
};

namespace {

afd_status fail(afd_ctx* c, afd_status st, const char* fmt, ...) {
  if (c) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(c->detail, sizeof c->detail, fmt, ap);
    va_end(ap);
  }
  return st;
}

afd_status cuda_fail(afd_ctx* c, cudaError_t e, const char* what) {
  return fail(c, AFD_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Makes the context's device current for the duration of a call.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

bool is_capturing(cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &st) != cudaSuccess) return false;
  return st != cudaStreamCaptureStatusNone;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The address the kernels use for a caller buffer: device memory of the
// context's device, managed memory, or page-locked host memory (reached over
// the host link through its mapped device address). Pageable host memory is
// refused: a kernel cannot dereference it.
afd_status resolve_ptr(afd_ctx* c, const void* p, const char* what, const void** out,
                       bool* on_device = nullptr) {
  DeviceGuard guard(c->device);  // a mapped host address is the current device's
  if (on_device) *on_device = false;
  cudaPointerAttributes a;
  memset(&a, 0, sizeof a);
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(c, AFD_ERR_ARG, "%s: not a pointer CUDA knows", what);
  }
  switch (a.type) {
    case cudaMemoryTypeDevice:
      if (a.device != c->device)
        return fail(c, AFD_ERR_ARG, "%s is on device %d, the context on device %d", what, a.device, c->device);
      *out = p;
      if (on_device) *on_device = true;
      return AFD_OK;
    case cudaMemoryTypeManaged:
      *out = p;
      return AFD_OK;
    case cudaMemoryTypeHost:
      if (!a.devicePointer) return fail(c, AFD_ERR_ARG, "%s: pinned host memory not mapped for the device", what);
      *out = a.devicePointer;
      return AFD_OK;
    default:
      return fail(c, AFD_ERR_ARG, "%s is pageable host memory: pin it or copy it to the device", what);
  }
}

template <typename T>
afd_status resolve(afd_ctx* c, T* p, const char* what, T** out) {
  const void* r = nullptr;
  afd_status st = resolve_ptr(c, p, what, &r);
  *out = static_cast<T*>(const_cast<void*>(r));
  return st;
}

// Orders `s` after the context's previous call when the stream changes. A
// wait never crosses a capture boundary (CUDA forbids a captured stream to
// depend on work recorded outside its capture, and the reverse is
// meaningless): across that boundary the caller orders the work, as when it
// synchronizes before capturing a graph.
afd_status order_stream(afd_ctx* c, cudaStream_t s) {
  if (c->has_last && s != c->last_stream && is_capturing(s) == c->last_captured) {
    cudaError_t e = cudaStreamWaitEvent(s, c->order_ev, 0);
    if (e != cudaSuccess) return cuda_fail(c, e, "cudaStreamWaitEvent");
  }
  return AFD_OK;
}

// Every call records the mark, even one that enqueued nothing: the mark also
// covers the caller's own work before the call on that stream (the expert
// before worker_reply, the producer of x before source_dispatch), which a
// later call on another stream must wait for.
afd_status mark_stream(afd_ctx* c, cudaStream_t s) {
  cudaError_t e = cudaEventRecord(c->order_ev, s);
  if (e != cudaSuccess) return cuda_fail(c, e, "cudaEventRecord");
  c->last_stream = s;
  c->last_captured = is_capturing(s);
  c->has_last = true;
  return AFD_OK;
}

int64_t recv_rows_for(const afd_ctx* c, int64_t bucket) {
  const afd_config& g = c->cfg;
  const int64_t per_token = g.top_k < c->Ef ? g.top_k : c->Ef;
  return align_up64((int64_t)g.num_sources * bucket * per_token +
                        (int64_t)c->Ef * (g.expert_alignment - 1),
                    g.expert_alignment);
}

void reset_exchange(afd_ctx* c) {
  c->phase = kIdle;
  c->cached = false;
  c->combine_last = false;
  c->combine_stream = nullptr;
  c->combine_captured = false;
  c->staged_n = c->replied_n = c->collected_n = 0;
  c->bucket = -1;
  c->rhc = -1;
  for (int i = 0; i < afd::kMaxSources; ++i) c->staged[i] = c->collected[i] = false;
  for (int i = 0; i < afd::kMaxWorkers; ++i) {
    c->received[i] = c->replied[i] = false;
    c->recv_rows[i] = -1;
    c->reply[i] = nullptr;
  }
}

void free_all(afd_ctx* c) {
  cudaFree(c->rows);
  cudaFree(c->row_scales);
  cudaFree(c->row_w);
  cudaFree(c->row_src);
  cudaFree(c->starts);
  cudaFree(c->ends);
  cudaFree(c->hcounts);
  cudaFree(c->routes);
  cudaFree(c->route_tmp);
  cudaFree(c->err);
  cudaFree(c->inbox);
  cudaFreeHost(c->host_counts);
  cudaFreeHost(c->host_err);
  if (c->order_ev) cudaEventDestroy(c->order_ev);
}

template <typename T>
bool dev_alloc(T** p, size_t count) {
  if (count == 0) count = 1;
  return cudaMalloc(reinterpret_cast<void**>(p), count * sizeof(T)) == cudaSuccess;
}

afd_status check_config(const afd_config* g, afd_ctx* c) {
  if (g->num_sources < 1 || g->num_sources > afd::kMaxSources)
    return fail(c, AFD_ERR_UNSUPPORTED, "num_sources must be in [1, %d]", afd::kMaxSources);
  if (g->num_workers < 1 || g->num_workers > afd::kMaxWorkers)
    return fail(c, AFD_ERR_UNSUPPORTED, "num_workers must be in [1, %d]", afd::kMaxWorkers);
  if (g->num_experts < 1 || g->num_experts > afd::kMaxExperts)
    return fail(c, AFD_ERR_UNSUPPORTED, "num_experts must be in [1, %d]", afd::kMaxExperts);
  if (g->num_experts % g->num_workers != 0)
    return fail(c, AFD_ERR_ARG, "num_experts must divide evenly over the workers");
  if (g->top_k < 1 || g->top_k > afd::kMaxTopK || g->top_k > g->num_experts)
    return fail(c, AFD_ERR_ARG, "top_k must be in [1, min(32, num_experts)]");
  if (g->hidden < 256 || g->hidden % 256 != 0)
    return fail(c, AFD_ERR_ARG, "hidden must be a positive multiple of 256");
  if (g->capacity < 1) return fail(c, AFD_ERR_ARG, "capacity must be >= 1");
  if (g->expert_alignment < 1) return fail(c, AFD_ERR_ARG, "expert_alignment must be >= 1");
  if (g->dtype != AFD_BF16 && g->dtype != AFD_FP8_E4M3)
    return fail(c, AFD_ERR_ARG, "dtype must be AFD_BF16 or AFD_FP8_E4M3");
  if (g->num_sms < 0) return fail(c, AFD_ERR_ARG, "num_sms must be >= 0");
  if (g->combine_mode < AFD_COMBINE_FUSED || g->combine_mode > AFD_COMBINE_TWO_STAGE_FP8)
    return fail(c, AFD_ERR_ARG, "unknown combine_mode");
  if (g->combine_mode != AFD_COMBINE_FUSED && g->top_k > 8)
    return fail(c, AFD_ERR_UNSUPPORTED, "the two-stage combine modes need top_k <= 8");
  return AFD_OK;
}

// Builds the exchange's launch parameters from the staged sources and
// launches its dispatch: the layout and scatter, or (cached) only the copy of
// the rows along the last layout.
afd_status launch_exchange_dispatch(afd_ctx* c, cudaStream_t stream, bool cached) {
  const afd_config& g = c->cfg;
  DispatchParams p;
  memset(&p, 0, sizeof p);
  int tok = 0;
  p.x_device = 1;
  for (int s = 0; s < g.num_sources; ++s) {
    p.src[s] = c->src[s];
    p.src[s].tok_off = tok;
    c->src[s].tok_off = tok;
    tok += c->src[s].T;
    if (c->src[s].T > 0 && !c->src[s].x_device) p.x_device = 0;
  }
  p.A = g.num_sources;
  p.F = g.num_workers;
  p.E = g.num_experts;
  p.Ef = c->Ef;
  p.K = g.top_k;
  p.alpha = g.expert_alignment;
  p.bucket = c->bucket;
  p.row_bytes = c->row_bytes;
  p.nscale = c->nscale;
  p.total_tokens = tok;
  p.R_arena = c->R_arena;
  p.wait_polls = c->wait_polls;
  p.route_tmp = c->route_tmp;
  p.layout_ctas = afd::layout_ctas_for(tok, c->sm_cap, c->layout_max_ctas);
  p.err = c->err;
  p.starts = c->starts;
  p.ends = c->ends;
  p.hcounts = c->hcounts;
  p.routes = c->routes;
  p.row_src = c->row_src;
  p.row_w = c->row_w;
  p.rows = c->rows;
  p.row_scales = c->row_scales;
  cudaError_t e = cached ? afd::launch_cached_scatter(p, c->sm_cap, stream)
                         : afd::launch_dispatch(p, c->sm_cap, stream);
  if (e != cudaSuccess) return cuda_fail(c, e, "dispatch launch");
  if (!cached) {
    c->layout_valid = true;
    c->layout_bucket = c->bucket;
    for (int s = 0; s < g.num_sources; ++s) c->layout_T[s] = c->src[s].T;
  }
  c->phase = kDispatched;
  return AFD_OK;
}

}  // namespace

extern "C" {

const char* afd_status_string(afd_status s) {
  switch (s) {
    case AFD_OK: return "ok";
    case AFD_ERR_ARG: return "invalid argument";
    case AFD_ERR_STATE: return "call out of exchange order";
    case AFD_ERR_BUCKET: return "bucket or read_host_counts mismatch";
    case AFD_ERR_RECEIPT: return "receipt or receive shape mismatch";
    case AFD_ERR_ROUTE_RANGE: return "top-k ID outside [-1, num_experts)";
    case AFD_ERR_ROUTE_DUP: return "repeated top-k ID within a token";
    case AFD_ERR_CUDA: return "CUDA runtime error";
    case AFD_ERR_OOM: return "allocation failed";
    case AFD_ERR_CAPTURING: return "host synchronization requested during stream capture";
    case AFD_ERR_UNSUPPORTED: return "configuration not supported by this build";
    case AFD_ERR_TIMEOUT: return "a bounded device-side wait gave up";
  }
  return "unknown status";
}

int32_t afd_version(void) { return (0 << 16) | 1; }

const char* afd_error_detail(const afd_ctx* c) { return c ? c->detail : "no context"; }

int64_t afd_arena_rows(const afd_ctx* c) { return c ? c->R_arena : -1; }

int64_t afd_recv_rows_for_bucket(const afd_ctx* c, int32_t bucket) {
  if (!c || bucket < 0 || bucket > c->cfg.capacity) return -1;
  return recv_rows_for(c, bucket);
}

afd_status afd_create(const afd_config* config, int32_t device, afd_ctx** out) {
  if (!config || !out) return AFD_ERR_ARG;
  *out = nullptr;
  afd_ctx* c = new (std::nothrow) afd_ctx;
  if (!c) return AFD_ERR_OOM;
  memset(c, 0, sizeof *c);
  c->detail[0] = 0;
  afd_status st = check_config(config, c);
  if (st != AFD_OK) {
    // the caller gets no context, so the message goes to stderr
    fprintf(stderr, "afd_create: %s\n", c->detail);
    delete c;
    return st;
  }
  c->cfg = *config;
  c->device = device;

  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
    delete c;
    return AFD_ERR_CUDA;
  }
  DeviceGuard guard(device);
  if (!guard.ok) {
    delete c;
    return AFD_ERR_CUDA;
  }
  cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, device);
  c->sm_cap = config->num_sms > 0 && config->num_sms < c->sm_count ? config->num_sms : c->sm_count;

  const afd_config& g = c->cfg;
  c->Ef = g.num_experts / g.num_workers;
  c->row_bytes = g.dtype == AFD_FP8_E4M3 ? g.hidden : 2 * g.hidden;
  c->nscale = g.dtype == AFD_FP8_E4M3 ? g.hidden / 128 : 0;
  c->R_arena = recv_rows_for(c, g.capacity);
  if (c->R_arena >= (int64_t)1 << afd::kWorkerShift) {
    fprintf(stderr, "afd_create: a worker arena of %lld rows exceeds 2^24\n",
            (long long)c->R_arena);
    delete c;
    return AFD_ERR_UNSUPPORTED;
  }

  const int64_t F = g.num_workers, A = g.num_sources, E = g.num_experts, K = g.top_k;
  bool ok = dev_alloc(&c->rows, (size_t)(F * c->R_arena * c->row_bytes)) &&
            dev_alloc(&c->row_w, (size_t)(F * c->R_arena)) &&
            dev_alloc(&c->row_src, (size_t)(F * c->R_arena)) &&
            dev_alloc(&c->starts, (size_t)E) && dev_alloc(&c->ends, (size_t)E) &&
            dev_alloc(&c->hcounts, (size_t)E) &&
            dev_alloc(&c->routes, (size_t)(A * g.capacity * K)) &&
            dev_alloc(&c->route_tmp, (size_t)(A * g.capacity * K)) &&
            dev_alloc(&c->err, 1);
  if (ok && c->nscale) ok = dev_alloc(&c->row_scales, (size_t)(F * c->R_arena * c->nscale));
  if (ok && F == 1) ok = dev_alloc(&c->inbox, (size_t)(A * g.capacity * g.hidden));
  if (ok) ok = cudaMallocHost(reinterpret_cast<void**>(&c->host_counts), E * sizeof(int32_t)) == cudaSuccess;
  if (ok) ok = cudaMallocHost(reinterpret_cast<void**>(&c->host_err), sizeof(unsigned long long)) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    free_all(c);
    delete c;
    return AFD_ERR_OOM;
  }
  cudaError_t e = cudaEventCreateWithFlags(&c->order_ev, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaMemset(c->err, 0xff, sizeof(unsigned long long));
  if (e == cudaSuccess) e = cudaMemset(c->row_src, 0xff, (size_t)(F * c->R_arena) * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemset(c->row_w, 0, (size_t)(F * c->R_arena) * sizeof(float));
  if (e == cudaSuccess) e = afd::configure_dispatch_kernels(&c->layout_max_ctas);
  if (e == cudaSuccess) e = afd::configure_combine_kernels();
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    fprintf(stderr, "afd_create: %s\n", cudaGetErrorString(e));
    free_all(c);
    delete c;
    return AFD_ERR_CUDA;
  }
  c->gen = 1;
  c->wait_polls = afd::kDefaultWaitPolls;
  reset_exchange(c);
  *out = c;
  return AFD_OK;
}

afd_status afd_destroy(afd_ctx* c) {
  if (!c) return AFD_OK;
  DeviceGuard guard(c->device);
  cudaError_t e = cudaDeviceSynchronize();
  free_all(c);
  delete c;
  return e == cudaSuccess ? AFD_OK : AFD_ERR_CUDA;
}

afd_status afd_reset_exchange(afd_ctx* c) {
  if (!c) return AFD_ERR_ARG;
  reset_exchange(c);
  c->gen += 1;
  return AFD_OK;
}

afd_status afd_source_dispatch(afd_ctx* c, int32_t source, const void* x, const int64_t* ids,
                               const float* weights, const float* x_scale,
                               int64_t scale_stride_t, int64_t scale_stride_b,
                               int32_t num_tokens, int32_t bucket, int32_t read_host_counts,
                               afd_stream stream_) {
  if (!c) return AFD_ERR_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const afd_config& g = c->cfg;
  if (source < 0 || source >= g.num_sources) return fail(c, AFD_ERR_ARG, "source %d out of range", source);
  if (c->phase != kIdle && c->phase != kStaging)
    return fail(c, AFD_ERR_STATE, "the previous exchange is not collected yet");
  if (c->staged[source]) return fail(c, AFD_ERR_STATE, "source %d already dispatched", source);
  if (c->phase == kStaging && c->cached)
    return fail(c, AFD_ERR_STATE, "this exchange reuses the last routing (cached dispatch)");
  if (read_host_counts != 0 && read_host_counts != 1)
    return fail(c, AFD_ERR_ARG, "read_host_counts must be 0 or 1");
  if (bucket < 0 || bucket > g.capacity)
    return fail(c, AFD_ERR_BUCKET, "bucket %d outside [0, capacity %d]", bucket, g.capacity);
  if (num_tokens < 0 || num_tokens > bucket)
    return fail(c, AFD_ERR_BUCKET, "num_tokens %d outside [0, bucket %d]", num_tokens, bucket);
  if (c->phase == kStaging && (bucket != c->bucket || read_host_counts != c->rhc))
    return fail(c, AFD_ERR_BUCKET, "every role of one exchange passes the same bucket and read_host_counts");
  const void* dx = nullptr;
  const int64_t* dids = nullptr;
  const float* dw = nullptr;
  const float* dsc = nullptr;
  bool x_dev = true;
  if (num_tokens > 0) {
    if (!x || !ids || !weights) return fail(c, AFD_ERR_ARG, "x, ids and weights are required");
    if (g.dtype == AFD_FP8_E4M3 && !x_scale) return fail(c, AFD_ERR_ARG, "FP8 dispatch needs x_scale");
    if (g.dtype == AFD_FP8_E4M3 && (scale_stride_t < 0 || scale_stride_b < 0))
      return fail(c, AFD_ERR_ARG, "scale strides must be non-negative");
    afd_status r = resolve_ptr(c, x, "x", &dx, &x_dev);
    if (r == AFD_OK) r = resolve(c, ids, "ids", &dids);
    if (r == AFD_OK) r = resolve(c, weights, "weights", &dw);
    if (r == AFD_OK && g.dtype == AFD_FP8_E4M3) r = resolve(c, x_scale, "x_scale", &dsc);
    if (r != AFD_OK) return r;
    if (!aligned16(dx)) return fail(c, AFD_ERR_ARG, "x must be 16-byte aligned");
  }
  if (read_host_counts && is_capturing(stream))
    return fail(c, AFD_ERR_CAPTURING, "read_host_counts=1 cannot be captured");
  DeviceGuard guard(c->device);
  if (!guard.ok) return fail(c, AFD_ERR_CUDA, "cannot select device %d", c->device);

  afd_status st = order_stream(c, stream);
  if (st != AFD_OK) return st;

  SourceDesc& d = c->src[source];
  d.x = static_cast<const uint8_t*>(dx);
  d.x_device = x_dev ? 1 : 0;
  d.ids = dids;
  d.w = dw;
  d.scale = dsc;
  d.sst = scale_stride_t;
  d.ssb = scale_stride_b;
  d.T = num_tokens;
  c->staged[source] = true;
  c->staged_n += 1;
  c->phase = kStaging;
  c->bucket = bucket;
  c->rhc = read_host_counts;

  if (c->staged_n == g.num_sources) {
    st = launch_exchange_dispatch(c, stream, false);
    if (st != AFD_OK) return st;
  }
  return mark_stream(c, stream);
}

afd_status afd_source_dispatch_cached(afd_ctx* c, int32_t source, const void* x, const float* weights,
                                      const float* x_scale, int64_t scale_stride_t,
                                      int64_t scale_stride_b, int32_t num_tokens, int32_t bucket,
                                      int32_t read_host_counts, afd_stream stream_) {
  if (!c) return AFD_ERR_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const afd_config& g = c->cfg;
  if (source < 0 || source >= g.num_sources) return fail(c, AFD_ERR_ARG, "source %d out of range", source);
  if (c->phase != kIdle && c->phase != kStaging)
    return fail(c, AFD_ERR_STATE, "the previous exchange is not collected yet");
  if (c->staged[source]) return fail(c, AFD_ERR_STATE, "source %d already dispatched", source);
  if (c->phase == kStaging && !c->cached)
    return fail(c, AFD_ERR_STATE, "this exchange computes a new layout (afd_source_dispatch)");
  if (!c->layout_valid) return fail(c, AFD_ERR_STATE, "no earlier layout to reuse");
  if (bucket != c->layout_bucket || num_tokens != c->layout_T[source])
    return fail(c, AFD_ERR_STATE, "cached dispatch needs the last layout's num_tokens and bucket");
  if (read_host_counts != 0 && read_host_counts != 1)
    return fail(c, AFD_ERR_ARG, "read_host_counts must be 0 or 1");
  if (c->phase == kStaging && read_host_counts != c->rhc)
    return fail(c, AFD_ERR_BUCKET, "every role of one exchange passes the same read_host_counts");
  const void* dx = nullptr;
  const float* dw = nullptr;
  const float* dsc = nullptr;
  bool x_dev = true;
  if (num_tokens > 0) {
    if (!x) return fail(c, AFD_ERR_ARG, "x is required");
    if (g.dtype == AFD_FP8_E4M3 && !x_scale) return fail(c, AFD_ERR_ARG, "FP8 dispatch needs x_scale");
    if (g.dtype == AFD_FP8_E4M3 && (scale_stride_t < 0 || scale_stride_b < 0))
      return fail(c, AFD_ERR_ARG, "scale strides must be non-negative");
    afd_status r = resolve_ptr(c, x, "x", &dx, &x_dev);
    if (r == AFD_OK && weights) r = resolve(c, weights, "weights", &dw);
    if (r == AFD_OK && g.dtype == AFD_FP8_E4M3) r = resolve(c, x_scale, "x_scale", &dsc);
    if (r != AFD_OK) return r;
    if (!aligned16(dx)) return fail(c, AFD_ERR_ARG, "x must be 16-byte aligned");
  }
  if (read_host_counts && is_capturing(stream))
    return fail(c, AFD_ERR_CAPTURING, "read_host_counts=1 cannot be captured");
  DeviceGuard guard(c->device);
  if (!guard.ok) return fail(c, AFD_ERR_CUDA, "cannot select device %d", c->device);
  afd_status st = order_stream(c, stream);
  if (st != AFD_OK) return st;

  SourceDesc& d = c->src[source];
  d.x = static_cast<const uint8_t*>(dx);
  d.x_device = x_dev ? 1 : 0;
  d.ids = nullptr;
  d.w = dw;
  d.scale = dsc;
  d.sst = scale_stride_t;
  d.ssb = scale_stride_b;
  d.T = num_tokens;
  c->staged[source] = true;
  c->staged_n += 1;
  c->phase = kStaging;
  c->cached = true;
  c->bucket = bucket;
  c->rhc = read_host_counts;
  if (c->staged_n == g.num_sources) {
    st = launch_exchange_dispatch(c, stream, true);
    if (st != AFD_OK) return st;
  }
  return mark_stream(c, stream);
}

afd_status afd_worker_receive(afd_ctx* c, int32_t worker, int32_t bucket, int32_t read_host_counts,
                              afd_stream stream_, afd_recv* out) {
  if (!c || !out) return AFD_ERR_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const afd_config& g = c->cfg;
  if (worker < 0 || worker >= g.num_workers) return fail(c, AFD_ERR_ARG, "worker %d out of range", worker);
  if (c->phase != kDispatched) return fail(c, AFD_ERR_STATE, "no dispatched exchange to receive");
  if (c->received[worker]) return fail(c, AFD_ERR_STATE, "worker %d already received", worker);
  if (bucket != c->bucket || read_host_counts != c->rhc)
    return fail(c, AFD_ERR_BUCKET, "every role of one exchange passes the same bucket and read_host_counts");
  if (read_host_counts && is_capturing(stream))
    return fail(c, AFD_ERR_CAPTURING, "read_host_counts=1 cannot be captured");
  DeviceGuard guard(c->device);
  if (!guard.ok) return fail(c, AFD_ERR_CUDA, "cannot select device %d", c->device);
  afd_status st = order_stream(c, stream);
  if (st != AFD_OK) return st;

  const int64_t off = (int64_t)worker * c->R_arena;
  memset(out, 0, sizeof *out);
  out->rows = c->rows + off * c->row_bytes;
  out->row_scales = c->nscale ? c->row_scales + off * c->nscale : nullptr;
  out->weights = c->row_w + off;
  out->row_src = c->row_src + off;
  out->ends = c->ends + (int64_t)worker * c->Ef;
  out->receipt = (c->gen << 8) | (uint64_t)worker;
  afd_status result = AFD_OK;
  if (read_host_counts) {
    cudaError_t e = cudaMemcpyAsync(c->host_counts + (int64_t)worker * c->Ef,
                                    c->hcounts + (int64_t)worker * c->Ef, c->Ef * sizeof(int32_t),
                                    cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(c->host_err, c->err, sizeof(unsigned long long), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "host counts");
    int64_t n = 0;
    for (int l = 0; l < c->Ef; ++l) n += c->host_counts[(int64_t)worker * c->Ef + l];
    out->num_rows = n;
    out->host_counts = c->host_counts + (int64_t)worker * c->Ef;
    const unsigned long long key = *c->host_err;
    if (key != afd::kNoError) {
      const int code = (int)(key & 0xff);
      result = fail(c, (afd_status)code, "invalid route at source %d token %d k %d",
                    (int)(key >> 56), (int)((key >> 16) & 0xffffffffull), (int)((key >> 8) & 0xff));
    }
  } else {
    out->num_rows = recv_rows_for(c, c->bucket);
  }
  c->received[worker] = true;
  c->recv_rows[worker] = out->num_rows;
  st = mark_stream(c, stream);
  return result != AFD_OK ? result : st;
}

afd_status afd_worker_reply(afd_ctx* c, int32_t worker, const void* rows, int64_t num_rows,
                            uint64_t receipt, afd_stream stream_) {
  if (!c) return AFD_ERR_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const afd_config& g = c->cfg;
  if (worker < 0 || worker >= g.num_workers) return fail(c, AFD_ERR_ARG, "worker %d out of range", worker);
  if (c->phase != kDispatched) return fail(c, AFD_ERR_STATE, "no exchange awaiting replies");
  if (!c->received[worker]) return fail(c, AFD_ERR_STATE, "worker %d replies before receiving", worker);
  if (c->replied[worker]) return fail(c, AFD_ERR_STATE, "worker %d already replied", worker);
  if (receipt != ((c->gen << 8) | (uint64_t)worker))
    return fail(c, AFD_ERR_RECEIPT, "receipt does not match worker %d's receive", worker);
  if (num_rows != c->recv_rows[worker])
    return fail(c, AFD_ERR_RECEIPT, "reply has %lld rows, the receive had %lld", (long long)num_rows,
                (long long)c->recv_rows[worker]);
  if (num_rows > 0 && !rows) return fail(c, AFD_ERR_ARG, "reply rows are required");
  if (rows) {
    afd_status r = resolve_ptr(c, rows, "reply rows", &rows);
    if (r != AFD_OK) return r;
    if (!aligned16(rows)) return fail(c, AFD_ERR_ARG, "reply rows must be 16-byte aligned");
  }
  DeviceGuard guard(c->device);
  if (!guard.ok) return fail(c, AFD_ERR_CUDA, "cannot select device %d", c->device);
  afd_status st = order_stream(c, stream);
  if (st != AFD_OK) return st;

  c->reply[worker] = static_cast<const uint16_t*>(rows);
  c->replied[worker] = true;
  c->replied_n += 1;
  if (c->replied_n == g.num_workers) c->phase = kReplied;
  return mark_stream(c, stream);
}

afd_status afd_source_collect(afd_ctx* c, int32_t source, void* out, int32_t view,
                              afd_stream stream_, afd_view* view_out) {
  if (!c) return AFD_ERR_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const afd_config& g = c->cfg;
  if (source < 0 || source >= g.num_sources) return fail(c, AFD_ERR_ARG, "source %d out of range", source);
  if (c->phase != kReplied) return fail(c, AFD_ERR_STATE, "replies are not complete");
  if (c->collected[source]) return fail(c, AFD_ERR_STATE, "source %d already collected", source);
  if (view && !view_out) return fail(c, AFD_ERR_ARG, "view = 1 needs view_out");
  const int T = c->src[source].T;
  const bool as_view = view && g.num_workers == 1;
  void* user_out = out;
  if (!as_view && T > 0) {
    if (!out) return fail(c, AFD_ERR_ARG, "out is required");
    afd_status r = resolve(c, out, "out", &out);
    if (r != AFD_OK) return r;
    if (!aligned16(out)) return fail(c, AFD_ERR_ARG, "out must be 16-byte aligned");
  }
  DeviceGuard guard(c->device);
  if (!guard.ok) return fail(c, AFD_ERR_CUDA, "cannot select device %d", c->device);
  afd_status st = order_stream(c, stream);
  if (st != AFD_OK) return st;

  uint16_t* inbox = c->inbox ? c->inbox + (int64_t)source * g.capacity * g.hidden : nullptr;
  if (T > 0) {
    CombineParams p;
    memset(&p, 0, sizeof p);
    // Started at once when the previous call was a collect of this exchange
    // that launched a combine on the same stream (and capture state): the
    // stream then holds nothing between the two combines but host-side marks.
    p.early = AFD_COMBINE_EARLY && c->combine_last && c->combine_stream == stream &&
              c->combine_captured == is_capturing(stream);
    p.share = g.num_sources;  // each source collects on its own
    p.routes[0] = c->routes + (int64_t)c->src[source].tok_off * g.top_k;
    p.out[0] = as_view ? inbox : static_cast<uint16_t*>(out);
    p.out_stride[0] = g.hidden;
    p.tok_off[0] = 0;
    for (int f = 0; f < g.num_workers; ++f) p.reply[f] = c->reply[f];
    p.mode = g.combine_mode;
    p.A = 1;
    p.K = g.top_k;
    p.H = g.hidden;
    p.total_tokens = T;
    cudaError_t e = afd::launch_combine(p, c->sm_cap, stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "combine launch");
  }
  c->combine_last = T > 0;
  c->combine_stream = stream;
  c->combine_captured = is_capturing(stream);
  if (view_out) {
    view_out->data = as_view ? static_cast<const void*>(inbox) : static_cast<const void*>(user_out);
    view_out->row_stride = g.hidden;
    view_out->num_tokens = T;
    view_out->is_view = as_view ? 1 : 0;
  }
  c->collected[source] = true;
  c->collected_n += 1;
  if (c->collected_n == g.num_sources) {
    reset_exchange(c);
    c->gen += 1;
  }
  return mark_stream(c, stream);
}

afd_status afd_source_collect_all(afd_ctx* c, void* const* outs, int32_t view, afd_stream stream_,
                                  afd_view* views) {
  if (!c) return AFD_ERR_ARG;
  const afd_config& g = c->cfg;
  if (c->phase != kReplied) return fail(c, AFD_ERR_STATE, "replies are not complete");
  if (c->collected_n != 0) return fail(c, AFD_ERR_STATE, "some sources are already collected");
  const bool as_view = view && g.num_workers == 1;
  if (!outs && !as_view) return fail(c, AFD_ERR_ARG, "outs is required");
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  void* dout[afd::kMaxSources] = {};
  for (int s = 0; s < g.num_sources; ++s) {
    if (c->src[s].T == 0) continue;
    if (as_view) {
      dout[s] = c->inbox + (int64_t)s * g.capacity * g.hidden;
      continue;
    }
    if (!outs[s]) return fail(c, AFD_ERR_ARG, "outs[%d] is required", s);
    afd_status r = resolve(c, outs[s], "outs[s]", &dout[s]);
    if (r != AFD_OK) return r;
    if (!aligned16(dout[s])) return fail(c, AFD_ERR_ARG, "outs[%d] must be 16-byte aligned", s);
  }
  DeviceGuard guard(c->device);
  if (!guard.ok) return fail(c, AFD_ERR_CUDA, "cannot select device %d", c->device);
  afd_status st = order_stream(c, stream);
  if (st != AFD_OK) return st;
  CombineParams p;
  memset(&p, 0, sizeof p);
  int tok = 0;
  for (int s = 0; s < g.num_sources; ++s) {
    p.routes[s] = c->routes + (int64_t)c->src[s].tok_off * g.top_k;
    p.out[s] = static_cast<uint16_t*>(dout[s]);
    p.out_stride[s] = g.hidden;
    p.tok_off[s] = tok;
    tok += c->src[s].T;
  }
  for (int f = 0; f < g.num_workers; ++f) p.reply[f] = c->reply[f];
  p.mode = g.combine_mode;
  p.A = g.num_sources;
  p.K = g.top_k;
  p.H = g.hidden;
  p.total_tokens = tok;
  cudaError_t e = afd::launch_combine(p, c->sm_cap, stream);
  if (e != cudaSuccess) return cuda_fail(c, e, "combine launch");
  for (int s = 0; s < g.num_sources; ++s) {
    if (views) {
      views[s].data = as_view ? static_cast<const void*>(dout[s]) : static_cast<const void*>(outs[s]);
      views[s].row_stride = g.hidden;
      views[s].num_tokens = c->src[s].T;
      views[s].is_view = as_view ? 1 : 0;
    }
  }
  reset_exchange(c);
  c->gen += 1;
  return mark_stream(c, stream);
}

afd_status afd_get_error(afd_ctx* c, int32_t* code, int32_t* source, int32_t* token, int32_t* k) {
  if (!c) return AFD_ERR_ARG;
  if (c->has_last && is_capturing(c->last_stream))
    return fail(c, AFD_ERR_CAPTURING, "afd_get_error synchronizes; not allowed during capture");
  DeviceGuard guard(c->device);
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(c->host_err, c->err, sizeof(unsigned long long), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(c, e, "reading the route error");
  const unsigned long long key = *c->host_err;
  const bool none = key == afd::kNoError;
  if (code) *code = none ? AFD_OK : (int32_t)(key & 0xff);
  if (source) *source = none ? -1 : (int32_t)(key >> 56);
  if (token) *token = none ? -1 : (int32_t)((key >> 16) & 0xffffffffull);
  if (k) *k = none ? -1 : (int32_t)((key >> 8) & 0xff);
  return AFD_OK;
}

afd_status afd_set_wait_limit(afd_ctx* c, int32_t polls) {
  if (!c) return AFD_ERR_ARG;
  if (polls < 0) return fail(c, AFD_ERR_ARG, "polls must be >= 0");
  c->wait_polls = polls;
  return AFD_OK;
}

afd_status afd_l2_flush(void* scratch, int64_t bytes, afd_stream stream_) {
  if (!scratch || bytes <= 0 || bytes % 32 != 0 || reinterpret_cast<uintptr_t>(scratch) % 16 != 0)
    return AFD_ERR_ARG;
  cudaError_t e = afd::launch_l2_flush(static_cast<uint4*>(scratch), bytes / 32,
                                       reinterpret_cast<cudaStream_t>(stream_));
  return e == cudaSuccess ? AFD_OK : AFD_ERR_CUDA;
}

afd_status afd_phase_stamps(afd_ctx* c, uint64_t* host, int64_t count, int32_t clear) {
#if AFD_PHASE_TIMERS
  if (!c || !host) return AFD_ERR_ARG;
  const int64_t half = 2ll * afd::kStampBlocks * afd::kStampPoints;
  if (count < 2 * half) return fail(c, AFD_ERR_ARG, "count must be at least %lld", (long long)(2 * half));
  DeviceGuard guard(c->device);
  if (!guard.ok) return fail(c, AFD_ERR_CUDA, "cannot select device %d", c->device);
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = afd::read_dispatch_stamps(reinterpret_cast<unsigned long long*>(host), clear != 0);
  if (e == cudaSuccess) e = afd::read_combine_stamps(reinterpret_cast<unsigned long long*>(host + half), clear != 0);
  if (e == cudaSuccess && clear) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(c, e, "reading the phase stamps");
  return AFD_OK;
#else
  (void)c;
  (void)host;
  (void)count;
  (void)clear;
  return AFD_ERR_UNSUPPORTED;
#endif
}

afd_status afd_clear_error(afd_ctx* c, afd_stream stream_) {
  if (!c) return AFD_ERR_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  DeviceGuard guard(c->device);
  afd_status st = order_stream(c, stream);
  if (st != AFD_OK) return st;
  cudaError_t e = cudaMemsetAsync(c->err, 0xff, sizeof(unsigned long long), stream);
  if (e != cudaSuccess) return cuda_fail(c, e, "clearing the route error");
  c->combine_last = false;  // the next combine waits for the work before it
  return mark_stream(c, stream);
}

}  // extern "C"
