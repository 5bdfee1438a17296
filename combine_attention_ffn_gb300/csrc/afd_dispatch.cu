// Dispatch kernels: route layout (validate, histogram, aligned scan, ranks)
// and the scatter of source rows into expert-major worker arenas.
//
// What they compute follows the afdEP-comm "API contract" (Roles and tensors:
// ID rules, worker-owned expert blocks, the ends[] prefix sums with
// expert_alignment padding, aligned host counts) and "DeepEP V2 ElasticBuffer
// first principles" section 3 (count routes per expert, give every route a
// slot, copy each token's row to every selected expert; section 7: FP8 rows
// travel with their scales). Unlike the atomic slot counters described there,
// slots here come from a stable counting sort, so rows inside an expert
// follow (source, token) order and every run gives the same layout.
//
// Counting: tokens are taken in chunks of 256, one token per thread. For
// each warp and expert a shared-memory lane mask records which of the warp's
// 32 tokens route to that expert; a route's rank inside the chunk is the
// count of earlier warps' tokens plus the popcount of the earlier lanes of
// its own mask. A repeated ID shows up as a mask bit that is already set.
//
// Two paths:
//  * small exchanges (at most kSmallRoutes routes): one kernel. Every block
//    counts all routes itself (they are few and sit in L2), scans in shared
//    memory, then copies its share of the rows. No block waits for another.
//  * large exchanges: layout_kernel (one block per chunk of 256 tokens; the
//    last block to finish, found with a completion counter, scans the chunk
//    counts; nobody waits) then scatter_kernel (a warp per token), launched
//    as a programmatic dependent: its blocks start early and load their first
//    source rows while the layout is still running.

#include <cuda_runtime.h>
#include <stdint.h>

#include "afd_device.cuh"
#include "afd_internal.cuh"

namespace afd {
namespace {

__device__ __forceinline__ int source_of_chunk(const DispatchParams& p, int g) {
  int s = 0;
  while (s + 1 < p.A && g >= p.src[s + 1].chunk_off) ++s;
  return s;
}

__device__ __forceinline__ int source_of_token(const DispatchParams& p, int gt) {
  int s = 0;
  while (s + 1 < p.A && gt >= p.src[s + 1].tok_off) ++s;
  return s;
}

// Validates the K IDs of token (s, t) held by this thread and marks the valid
// ones in its warp's lane masks (wmask = this warp's [E] masks). Returns the
// set of valid routes (bit k). IDs are read as int64 so that a value outside
// int32 is out of range, not truncated. Errors go to `err` when it is given.
__device__ __forceinline__ uint32_t mark_token(const int64_t* ids, int K, int E, uint32_t* wmask,
                                               int lane, int s, int t, unsigned long long* err) {
  uint32_t valid = 0u;
  for (int k0 = 0; k0 < K; k0 += 8) {
    int64_t v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = (k0 + j < K) ? ids[k0 + j] : -1;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int k = k0 + j;
      const int64_t id = v[j];
      if (k >= K || id == -1) continue;
      if (id < -1 || id >= E) {
        if (err) atomicMin(err, route_error_key(s, t, k, kErrRange));
        continue;
      }
      const uint32_t old = atomicOr(wmask + (int)id, 1u << lane);
      if (old & (1u << lane)) {  // this token already routed to this expert
        if (err) atomicMin(err, route_error_key(s, t, k, kErrDup));
        continue;
      }
      valid |= 1u << k;
    }
  }
  return valid;
}

// Per worker: start = exclusive scan of align_up(count, alpha) over its local
// experts, ends = start + count ("API contract": expert e occupies
// [align_up(ends[e-1], alpha), ends[e]) with ends[-1] = 0). One warp per
// worker. Writes sh_start; with `out`, also the global starts/ends/counts.
__device__ __forceinline__ void worker_scan(const DispatchParams& p, const int32_t* sh_total,
                                            int32_t* sh_start, bool out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  for (int f = warp; f < p.F; f += nwarps) {
    int carry = 0;
    for (int l0 = 0; l0 < p.Ef; l0 += 32) {
      const int l = l0 + lane;
      const int e = f * p.Ef + l;
      const int cnt = l < p.Ef ? sh_total[e] : 0;
      const int al = align_up_dev(cnt, p.alpha);
      const int incl = warp_inclusive_scan(al);
      if (l < p.Ef) {
        const int start = carry + incl - al;
        sh_start[e] = start;
        if (out) {
          p.starts[e] = start;
          p.ends[e] = start + cnt;
          p.hcounts[e] = al;
        }
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
}

// Padding rows between ends[e] and the next aligned start hold no route:
// row_src -1, weight +0. One warp per expert, lanes over its padding rows.
__device__ __forceinline__ void fill_padding(const DispatchParams& p, const int32_t* ends_of) {
  if (p.alpha <= 1) return;
  const int lane = threadIdx.x & 31;
  const int gwarp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  for (int e = gwarp; e < p.E; e += nwarps) {
    const int end = ends_of[e];
    const int lim = align_up_dev(end, p.alpha);
    const int64_t base = (int64_t)(e / p.Ef) * p.R_arena;
    for (int row = end + lane; row < lim; row += 32) {
      p.row_src[base + row] = -1;
      p.row_w[base + row] = 0.0f;
    }
  }
}

// A warp copies token (s, t)'s row to each of its routes. `code` is this
// lane's route (lane < K): (worker << 24) | row, or -1. The row is moved in
// pieces of 32 x kScatterVecs 16-byte vectors; `pre` holds the first piece
// when the caller loaded it early (have_pre).
constexpr int kScatterVecs = 8;  // 16-byte vectors per lane in flight

__device__ __forceinline__ void load_piece(uint4 (&buf)[kScatterVecs], const uint4* xrow, int v0,
                                           int nvec) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < kScatterVecs; ++j) {
    const int v = v0 + j * 32 + lane;
    if (v < nvec) buf[j] = ld_once(xrow + v);
  }
}

template <bool kPre>
__device__ __forceinline__ void copy_token(const DispatchParams& p, const SourceDesc& src, int t,
                                           int code, const uint4 (&pre)[kScatterVecs]) {
  const int lane = threadIdx.x & 31;
  const int K = p.K;
  const int nvec = p.row_bytes >> 4;
  const uint4* xrow = reinterpret_cast<const uint4*>(src.x + (int64_t)t * p.row_bytes);
  for (int v0 = 0; v0 < nvec; v0 += 32 * kScatterVecs) {
    uint4 buf[kScatterVecs];
    if (kPre && v0 == 0) {
#pragma unroll
      for (int j = 0; j < kScatterVecs; ++j) buf[j] = pre[j];
    } else {
      load_piece(buf, xrow, v0, nvec);
    }
    for (int k = 0; k < K; ++k) {
      const int c = __shfl_sync(0xffffffffu, code, k);
      if (c < 0) continue;
      uint4* dst = reinterpret_cast<uint4*>(
          p.rows + ((int64_t)(c >> kWorkerShift) * p.R_arena + (c & kRowMask)) * p.row_bytes);
#pragma unroll
      for (int j = 0; j < kScatterVecs; ++j) {
        const int v = v0 + j * 32 + lane;
        if (v < nvec) dst[v] = buf[j];
      }
    }
  }
  // FP8: the row's block scales follow it (read through the caller's strides).
  for (int b0 = 0; b0 < p.nscale; b0 += 32) {
    const int b = b0 + lane;
    float sc = 0.0f;
    if (b < p.nscale) sc = src.scale[(int64_t)t * src.sst + (int64_t)b * src.ssb];
    for (int k = 0; k < K; ++k) {
      const int c = __shfl_sync(0xffffffffu, code, k);
      if (c < 0 || b >= p.nscale) continue;
      p.row_scales[((int64_t)(c >> kWorkerShift) * p.R_arena + (c & kRowMask)) * p.nscale + b] = sc;
    }
  }
}

// Writes route (s, t, lane)'s receipt entries for a final row and returns its
// route code. Called by lanes < K.
__device__ __forceinline__ int write_route(const DispatchParams& p, int s, int t, int gt, int e,
                                           int row, float w) {
  const int f = e / p.Ef;
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)f * p.R_arena + row;
  p.row_src[r] = (s * p.bucket + t) * p.K + lane;
  p.row_w[r] = w;
  const int code = (f << kWorkerShift) | row;
  p.routes[(int64_t)gt * p.K + lane] = make_int2(code, __float_as_int(w));
  return code;
}

// One token of the scatter: finish each route's row from the layout (the
// chunk's first row of the expert plus the route's rank inside the chunk),
// write the receipt, copy the row. kPre: the row's first piece and the
// weights were loaded early into pre / pre_w.
template <bool kPre, typename RowOf>
__device__ __forceinline__ void scatter_token(const DispatchParams& p, int gt, RowOf row_of,
                                              float pre_w, const uint4 (&pre)[kScatterVecs]) {
  const int lane = threadIdx.x & 31;
  const int K = p.K;
  const int s = source_of_token(p, gt);
  const SourceDesc& src = p.src[s];
  const int t = gt - src.tok_off;
  int code = -1;
  if (lane < K) {
    int e = -1, row = 0;
    if (row_of(gt, s, t, e, row)) {
      const float w = kPre ? pre_w : src.w[(int64_t)t * K + lane];
      code = write_route(p, s, t, gt, e, row, w);
    } else {
      p.routes[(int64_t)gt * K + lane] = make_int2(-1, 0);
    }
  }
  copy_token<kPre>(p, src, t, code, pre);
}

// Loads warp `gwarp`'s first token's first row piece and weights.
__device__ __forceinline__ bool preload_first(const DispatchParams& p, int gwarp,
                                              uint4 (&pre)[kScatterVecs], float& pre_w) {
  if (gwarp >= p.total_tokens) return false;
  const int lane = threadIdx.x & 31;
  const int s0 = source_of_token(p, gwarp);
  const int t0 = gwarp - p.src[s0].tok_off;
  load_piece(pre, reinterpret_cast<const uint4*>(p.src[s0].x + (int64_t)t0 * p.row_bytes), 0,
             p.row_bytes >> 4);
  if (lane < p.K) pre_w = p.src[s0].w[(int64_t)t0 * p.K + lane];
  return true;
}

// ---------------------------------------------------------------- large path

// Sums the chunk counts per expert, scans per worker, and writes each chunk's
// first row per expert. Runs in the last block of the layout launch; the
// chunk loop of each expert is split into slices so that loads overlap.
__device__ void layout_finish(const DispatchParams& p, int32_t* sm) {
  const int E = p.E, G = p.total_chunks, nthr = blockDim.x;
  const int P = E <= nthr ? nthr / E : 1;  // slices per expert
  int32_t* part = sm;                      // [P][E]
  int32_t* sh_total = part + P * E;        // [E]
  int32_t* sh_start = sh_total + E;        // [E]
  const int32_t* cc = p.chunk_counts;

  for (int idx = threadIdx.x; idx < P * E; idx += nthr) {
    const int e = idx % E, sl = idx / E;
    const int g0 = (int)((int64_t)G * sl / P), g1 = (int)((int64_t)G * (sl + 1) / P);
    int sum = 0, g = g0;
    for (; g + 8 <= g1; g += 8) {
      int v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = __ldcg(cc + (int64_t)(g + j) * E + e);
#pragma unroll
      for (int j = 0; j < 8; ++j) sum += v[j];
    }
    for (; g < g1; ++g) sum += __ldcg(cc + (int64_t)g * E + e);
    part[sl * E + e] = sum;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += nthr) {
    int run = 0;
    for (int sl = 0; sl < P; ++sl) {
      const int v = part[sl * E + e];
      part[sl * E + e] = run;
      run += v;
    }
    sh_total[e] = run;
  }
  __syncthreads();
  worker_scan(p, sh_total, sh_start, true);
  __syncthreads();
  for (int idx = threadIdx.x; idx < P * E; idx += nthr) {
    const int e = idx % E, sl = idx / E;
    const int g0 = (int)((int64_t)G * sl / P), g1 = (int)((int64_t)G * (sl + 1) / P);
    int run = sh_start[e] + part[sl * E + e], g = g0;
    for (; g + 8 <= g1; g += 8) {
      int v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = __ldcg(cc + (int64_t)(g + j) * E + e);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        p.chunk_start[(int64_t)(g + j) * E + e] = run;
        run += v[j];
      }
    }
    for (; g < g1; ++g) {
      const int c = __ldcg(cc + (int64_t)g * E + e);
      p.chunk_start[(int64_t)g * E + e] = run;
      run += c;
    }
  }
}

__global__ void __launch_bounds__(kChunk) layout_kernel(const __grid_constant__ DispatchParams p) {
  extern __shared__ __align__(16) uint32_t smem[];
  uint32_t* mask = smem;                                                   // [8][E]
  uint16_t* wbase = reinterpret_cast<uint16_t*>(smem + kChunkWarps * p.E);  // [8][E]
  __shared__ int is_last;
  pdl_launch_dependents();

  const int E = p.E, K = p.K;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = blockIdx.x;

  if (g < p.total_chunks) {
    const int s = source_of_chunk(p, g);
    const SourceDesc& src = p.src[s];
    const int t = (g - src.chunk_off) * kChunk + threadIdx.x;
    const bool live = t < src.T;

    for (int i = threadIdx.x; i < kChunkWarps * E; i += blockDim.x) mask[i] = 0u;
    __syncthreads();
    const int64_t* ids = src.ids + (int64_t)t * K;
    const uint32_t valid = live ? mark_token(ids, K, E, mask + warp * E, lane, s, t, p.err) : 0u;
    __syncthreads();

    // Warp offsets inside the chunk and the chunk's count per expert.
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int run = 0;
#pragma unroll
      for (int w = 0; w < kChunkWarps; ++w) {
        wbase[w * E + e] = (uint16_t)run;
        run += __popc(mask[w * E + e]);
      }
      p.chunk_counts[(int64_t)g * E + e] = run;
    }
    __syncthreads();

    if (live) {
      int32_t* rt = p.route_tmp + (int64_t)(src.tok_off + t) * K;
      const uint32_t lanes_before = (1u << lane) - 1u;
      for (int k = 0; k < K; ++k) {
        int code = -1;
        if ((valid >> k) & 1u) {
          const int e = (int)ids[k];
          const int rank = wbase[warp * E + e] + __popc(mask[warp * E + e] & lanes_before);
          code = (e << kRankBits) | rank;
        }
        rt[k] = code;
      }
    }
  }

  // The last block to arrive finishes the layout; nobody waits.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = (atomicAdd(p.done, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  layout_finish(p, reinterpret_cast<int32_t*>(smem));
  if (threadIdx.x == 0) *p.done = 0u;
}

__global__ void __launch_bounds__(AFD_SCATTER_BLOCK) scatter_kernel(const __grid_constant__ DispatchParams p) {
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int gwarp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const int K = p.K, E = p.E;

  // The source rows and weights are inputs, not layout outputs: start loading
  // this warp's first token while the layout kernel is still running.
  uint4 pre[kScatterVecs];
  float pre_w = 0.0f;
  const bool have_pre = preload_first(p, gwarp, pre, pre_w);
  pdl_wait();  // the layout kernel's outputs
  const int32_t* chunk_start = p.chunk_start;

  auto row_of = [&](int gt, int s, int t, int& e, int& row) -> bool {
    const int rt = p.route_tmp[(int64_t)gt * K + lane];
    if (rt < 0) return false;
    e = rt >> kRankBits;
    const int g = p.src[s].chunk_off + t / kChunk;
    row = chunk_start[g * E + e] + (rt & ((1 << kRankBits) - 1));
    return true;
  };
  int gt = gwarp;
  if (have_pre) {
    scatter_token<true>(p, gt, row_of, pre_w, pre);
    gt += nwarps;
  }
  for (; gt < p.total_tokens; gt += nwarps) scatter_token<false>(p, gt, row_of, 0.0f, pre);
  fill_padding(p, p.ends);
}

// ---------------------------------------------------------------- small path

__global__ void __launch_bounds__(256) dispatch_small_kernel(const __grid_constant__ DispatchParams p) {
  extern __shared__ __align__(16) uint32_t smem[];
  const int E = p.E, K = p.K, N = p.total_tokens;
  const int G = (N + kChunk - 1) / kChunk;
  uint32_t* mask = smem;                                   // [8][E]
  uint32_t* rinfo = mask + kChunkWarps * E;                // [N*K]: (e << 8 | rank) or ~0
  int32_t* sh_start = reinterpret_cast<int32_t*>(rinfo + N * K);  // [E]
  int32_t* sh_total = sh_start + E;                        // [E]
  uint16_t* wbase = reinterpret_cast<uint16_t*>(sh_total + E);    // [8][E]
  uint16_t* ccnt = wbase + kChunkWarps * E;                // [G][E]

  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long* err = blockIdx.x == 0 ? p.err : nullptr;
  const int gwarp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;

  // Load this warp's first row and weights now, so that their latency
  // overlaps the counting below.
  uint4 pre[kScatterVecs];
  float pre_w = 0.0f;
  const bool have_pre = preload_first(p, gwarp, pre, pre_w);

  // Pass 1 (every block, all routes): ranks inside each chunk, chunk counts.
  for (int c = 0; c < G; ++c) {
    for (int i = threadIdx.x; i < kChunkWarps * E; i += blockDim.x) mask[i] = 0u;
    __syncthreads();
    const int gt = c * kChunk + threadIdx.x;
    const bool live = gt < N;
    int s = 0, t = 0;
    const int64_t* ids = nullptr;
    uint32_t valid = 0u;
    if (live) {
      s = source_of_token(p, gt);
      t = gt - p.src[s].tok_off;
      ids = p.src[s].ids + (int64_t)t * K;
      valid = mark_token(ids, K, E, mask + warp * E, lane, s, t, err);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int run = 0;
#pragma unroll
      for (int w = 0; w < kChunkWarps; ++w) {
        wbase[w * E + e] = (uint16_t)run;
        run += __popc(mask[w * E + e]);
      }
      ccnt[c * E + e] = (uint16_t)run;
    }
    __syncthreads();
    if (live) {
      const uint32_t lanes_before = (1u << lane) - 1u;
      for (int k = 0; k < K; ++k) {
        uint32_t info = ~0u;
        if ((valid >> k) & 1u) {
          const int e = (int)ids[k];
          info = ((uint32_t)e << kRankBits) |
                 (uint32_t)(wbase[warp * E + e] + __popc(mask[warp * E + e] & lanes_before));
        }
        rinfo[gt * K + k] = info;
      }
    }
    __syncthreads();
  }

  // Scan: chunk prefixes per expert (in place), totals, aligned starts.
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int c = 0; c < G; ++c) {
      const int v = ccnt[c * E + e];
      ccnt[c * E + e] = (uint16_t)run;
      run += v;
    }
    sh_total[e] = run;
  }
  __syncthreads();
  worker_scan(p, sh_total, sh_start, blockIdx.x == 0);
  __syncthreads();

  // Pass 2: this block's share of the tokens.
  auto row_of = [&](int gt, int, int, int& e, int& row) -> bool {
    const uint32_t info = rinfo[gt * K + lane];
    if (info == ~0u) return false;
    e = (int)(info >> kRankBits);
    row = sh_start[e] + ccnt[(gt / kChunk) * E + e] + (int)(info & ((1u << kRankBits) - 1));
    return true;
  };
  int gt = gwarp;
  if (have_pre) {
    scatter_token<true>(p, gt, row_of, pre_w, pre);
    gt += nwarps;
  }
  for (; gt < N; gt += nwarps) scatter_token<false>(p, gt, row_of, 0.0f, pre);

  // Padding rows, from this block's own copy of the layout.
  for (int e = threadIdx.x; e < E; e += blockDim.x) sh_total[e] += sh_start[e];  // ends
  __syncthreads();
  fill_padding(p, sh_total);
}

// ---------------------------------------------------------------- cached path

// Dispatch with the previous exchange's routing: the receipt already holds
// every route's row, so a warp per token only copies the row (and, when new
// weights are given, refreshes the weights in both receipts).
__global__ void __launch_bounds__(AFD_SCATTER_BLOCK) cached_scatter_kernel(const __grid_constant__ DispatchParams p) {
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int gwarp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const int K = p.K;
  uint4 none[kScatterVecs];
  for (int gt = gwarp; gt < p.total_tokens; gt += nwarps) {
    const int s = source_of_token(p, gt);
    const SourceDesc& src = p.src[s];
    const int t = gt - src.tok_off;
    int code = -1;
    if (lane < K) {
      int2* r = p.routes + (int64_t)gt * K + lane;
      code = r->x;
      if (src.w != nullptr && code >= 0) {
        const float w = src.w[(int64_t)t * K + lane];
        r->y = __float_as_int(w);
        p.row_w[(int64_t)(code >> kWorkerShift) * p.R_arena + (code & kRowMask)] = w;
      }
    }
    copy_token<false>(p, src, t, code, none);
  }
}

// ---------------------------------------------------------------- tiny path

// At most 32 tokens in the whole exchange: one-warp blocks. Every block
// counts all the routes itself with one lane mask per expert (lane = token),
// so ranks are popcounts of earlier lanes and no block-wide barrier is
// needed; block b < N then scatters token b, and all blocks share the padding
// rows.
__global__ void __launch_bounds__(32) dispatch_tiny_kernel(const __grid_constant__ DispatchParams p) {
  extern __shared__ __align__(16) uint32_t tsm[];
  const int E = p.E, K = p.K, N = p.total_tokens;
  uint32_t* mask = tsm;                                     // [E]
  int32_t* sh_start = reinterpret_cast<int32_t*>(mask + E);  // [E]
  int32_t* sh_end = sh_start + E;                           // [E]
  pdl_launch_dependents();
  const int lane = threadIdx.x;

  uint4 pre[kScatterVecs];
  float pre_w = 0.0f;
  const bool has_token = preload_first(p, blockIdx.x, pre, pre_w);  // token blockIdx.x, if any

  for (int e = lane; e < E; e += 32) mask[e] = 0u;
  __syncwarp();
  uint32_t valid = 0u;
  if (lane < N) {
    const int s = source_of_token(p, lane);
    const int t = lane - p.src[s].tok_off;
    valid = mark_token(p.src[s].ids + (int64_t)t * K, K, E, mask, lane, s, t,
                       blockIdx.x == 0 ? p.err : nullptr);
  }
  __syncwarp();
  // aligned scan per worker, one warp
  for (int f = 0; f < p.F; ++f) {
    int carry = 0;
    for (int l0 = 0; l0 < p.Ef; l0 += 32) {
      const int l = l0 + lane;
      const int e = f * p.Ef + l;
      const int cnt = l < p.Ef ? __popc(mask[e]) : 0;
      const int al = align_up_dev(cnt, p.alpha);
      const int incl = warp_inclusive_scan(al);
      if (l < p.Ef) {
        const int start = carry + incl - al;
        sh_start[e] = start;
        sh_end[e] = start + cnt;
        if (blockIdx.x == 0) {
          p.starts[e] = start;
          p.ends[e] = start + cnt;
          p.hcounts[e] = al;
        }
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncwarp();

  auto row_of = [&](int gt, int s, int t, int& e, int& row) -> bool {
    if (!((__shfl_sync(0xffffffffu, valid, gt) >> lane) & 1u)) return false;
    e = (int)p.src[s].ids[(int64_t)t * K + lane];
    row = sh_start[e] + __popc(mask[e] & ((1u << gt) - 1u));
    return true;
  };
  // the route rows of one token; all 32 lanes take part (the valid mask is
  // gathered with a shuffle), lanes >= K only copy
  const int gt = blockIdx.x;
  if (has_token) {
    const int s = source_of_token(p, gt);
    const SourceDesc& src = p.src[s];
    const int t = gt - src.tok_off;
    int e = -1, row = 0;
    const bool ok = row_of(gt, s, t, e, row);
    int code = -1;
    if (lane < K) {
      if (ok) {
        code = write_route(p, s, t, gt, e, row, pre_w);
      } else {
        p.routes[(int64_t)gt * K + lane] = make_int2(-1, 0);
      }
    }
    copy_token<true>(p, src, t, code, pre);
  }
  // padding rows, spread over the blocks
  if (p.alpha > 1) {
    for (int e = blockIdx.x; e < E; e += gridDim.x) {
      const int end = sh_end[e];
      const int lim = align_up_dev(end, p.alpha);
      const int64_t base = (int64_t)(e / p.Ef) * p.R_arena;
      for (int row = end + lane; row < lim; row += 32) {
        p.row_src[base + row] = -1;
        p.row_w[base + row] = 0.0f;
      }
    }
  }
}

size_t layout_smem(int E) {
  const size_t count = (size_t)kChunkWarps * E * (sizeof(uint32_t) + sizeof(uint16_t));
  const size_t finish = (size_t)(kChunk + 2 * E) * sizeof(int32_t);
  return count > finish ? count : finish;
}

size_t small_smem(int E, int N, int K) {
  const int G = (N + kChunk - 1) / kChunk;
  return (size_t)kChunkWarps * E * 4 + (size_t)N * K * 4 + (size_t)2 * E * 4 +
         (size_t)kChunkWarps * E * 2 + (size_t)G * E * 2;
}

template <typename Kernel>
cudaError_t launch(Kernel kernel, int grid, int block, size_t smem, cudaStream_t stream, bool pdl,
                   const DispatchParams& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace

bool dispatch_is_small(const DispatchParams& p) {
  return (int64_t)p.total_tokens * p.K <= kSmallRoutes &&
         small_smem(p.E, p.total_tokens, p.K) <= (size_t)kSmallSmemMax;
}

cudaError_t configure_dispatch_kernels() {
  cudaError_t e = cudaFuncSetAttribute(layout_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)layout_smem(kMaxExperts));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(dispatch_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmallSmemMax);
  return e;
}

// Launches the exchange's dispatch. The first kernel waits for all earlier
// work on the stream (a normal launch), so it never overlaps the previous
// exchange's combine, which still reads the arenas it overwrites.
cudaError_t launch_dispatch(const DispatchParams& p, int sm_cap, cudaStream_t stream) {
  const int block = 256;
  if (p.total_tokens >= 1 && p.total_tokens <= 32 && AFD_TINY_DISPATCH) {
    // one block per token, and at least 16 blocks to share the padding rows
    const int grid = p.total_tokens > 16 ? p.total_tokens : 16;
    return launch(dispatch_tiny_kernel, grid, 32, (size_t)3 * p.E * sizeof(int32_t), stream, false, p);
  }
  if (dispatch_is_small(p)) {
    int grid = (p.total_tokens + 7) / 8;
    if (grid > sm_cap) grid = sm_cap;
    if (grid < 1) grid = 1;
    return launch(dispatch_small_kernel, grid, block, small_smem(p.E, p.total_tokens, p.K), stream,
                  false, p);
  }
  const int lgrid = p.total_chunks > 0 ? p.total_chunks : 1;
  cudaError_t e = launch(layout_kernel, lgrid, kChunk, layout_smem(p.E), stream, false, p);
  if (e != cudaSuccess) return e;
  // small blocks, a warp per token, so that blocks spread evenly over the SMs
  constexpr int kWarps = AFD_SCATTER_BLOCK / 32;
  int grid = (p.total_tokens + kWarps - 1) / kWarps;
  if (grid > sm_cap * (2048 / AFD_SCATTER_BLOCK)) grid = sm_cap * (2048 / AFD_SCATTER_BLOCK);
  if (grid < 1) grid = 1;
  return launch(scatter_kernel, grid, AFD_SCATTER_BLOCK, 0, stream, true, p);
}

}  // namespace afd

namespace afd {

// Launched normally (not as a programmatic dependent): it rewrites the rows
// that the previous exchange's combine reads.
cudaError_t launch_cached_scatter(const DispatchParams& p, int sm_cap, cudaStream_t stream) {
  constexpr int kWarps = AFD_SCATTER_BLOCK / 32;
  int grid = (p.total_tokens + kWarps - 1) / kWarps;
  if (grid > sm_cap * (2048 / AFD_SCATTER_BLOCK)) grid = sm_cap * (2048 / AFD_SCATTER_BLOCK);
  if (grid < 1) grid = 1;
  return launch(cached_scatter_kernel, grid, AFD_SCATTER_BLOCK, 0, stream, false, p);
}

}  // namespace afd
