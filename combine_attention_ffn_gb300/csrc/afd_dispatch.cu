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
// Three paths:
//  * at most 32 tokens: dispatch_tiny_kernel, one-warp blocks, one per
//    (token, route); a lane per token counts with one mask word per expert.
//  * at most kSmallRoutes routes: dispatch_small_kernel, one kernel, a warp
//    per (token, route). Every block counts all routes itself (they are few
//    and sit in L2) and scans in shared memory; no block waits for another.
//  * larger exchanges: cluster_layout_kernel (one thread-block cluster; the
//    CTAs share their counts through distributed shared memory and write
//    every route's final code) then scatter_kernel (a warp per token, which
//    reads its row once and writes it to each route), launched as a
//    programmatic dependent: its blocks start early and load their first
//    source rows while the layout is still running.

#include <cuda_runtime.h>
#include <stdint.h>

#include "afd_device.cuh"
#include "afd_internal.cuh"

namespace afd {

#if AFD_PHASE_TIMERS
// [kind 0: first dispatch kernel, kind 1: scatter][block][point]
__device__ unsigned long long g_dispatch_stamps[2][kStampBlocks][kStampPoints];

cudaError_t read_dispatch_stamps(unsigned long long* host, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(host, g_dispatch_stamps, sizeof(g_dispatch_stamps));
  if (e == cudaSuccess && clear) {
    void* d = nullptr;
    e = cudaGetSymbolAddress(&d, g_dispatch_stamps);
    if (e == cudaSuccess) e = cudaMemset(d, 0, sizeof(g_dispatch_stamps));
  }
  return e;
}
#endif

namespace {

__device__ __forceinline__ int source_of_token(const DispatchParams& p, int gt) {
  int s = 0;
  while (s + 1 < p.A && gt >= p.src[s + 1].tok_off) ++s;
  return s;
}

// The order the scatter kernels take tokens in: the i-th is a token of the
// last source first, then of the one before it, ..., tokens in order inside
// each source. Sources are usually collected in order, each collect reading
// its source's rows soon after the scatter wrote them, so the rows the first
// collect reads are written last and are the likeliest to be in L2 still
// (2A2F H2048 T=2048 round trip 50.0 -> 48.0 us, H4096 100.2 -> 96.3 us, skew
// 3A:1F 73.7 -> 69.6 us; one source: unchanged).
__device__ __forceinline__ int scatter_token_of(const DispatchParams& p, int i) {
  int s = p.A - 1;
  while (s > 0 && i >= p.src[s].T) {
    i -= p.src[s].T;
    --s;
  }
  return p.src[s].tok_off + i;
}

// Validates the K IDs of token (s, t) held by this thread and marks the valid
// ones in its warp's lane masks (wmask = this warp's [E] masks). Returns the
// set of valid routes (bit k). IDs are read as int64 so that a value outside
// int32 is out of range, not truncated. Errors go to `err` when it is given.
// The experts of routes 0..7 stay in e8 (registers), so that the caller can
// rank them without reading the IDs again (meaningful for valid routes only).
__device__ __forceinline__ uint32_t mark_token(const int64_t* ids, int K, int E, uint32_t* wmask,
                                               int lane, int s, int t, unsigned long long* err,
                                               int (&e8)[8]) {
  uint32_t valid = 0u;
  for (int k0 = 0; k0 < K; k0 += 8) {
    int64_t v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = (k0 + j < K) ? ids[k0 + j] : -1;
    if (k0 == 0) {
#pragma unroll
      for (int j = 0; j < 8; ++j) e8[j] = (int)v[j];
    }
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

// Writes route (s, t, lane)'s receipt entries for its final code
// ((worker << 24) | row). Called by lanes < K.
__device__ __forceinline__ void write_route(const DispatchParams& p, int s, int t, int gt, int code, float w) {
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)(code >> kWorkerShift) * p.R_arena + (code & kRowMask);
  p.row_src[r] = (s * p.bucket + t) * p.K + lane;
  p.row_w[r] = w;
  p.routes[(int64_t)gt * p.K + lane] = make_int2(code, __float_as_int(w));
}

// One token of the scatter: lane k < K holds route k's final code from the
// layout ((worker << 24) | row, or -1). Writes the receipt and copies the
// row. kPre: the row's first piece and the weights were loaded early into
// pre / pre_w.
template <bool kPre>
__device__ __forceinline__ void scatter_token(const DispatchParams& p, int gt, int code, float pre_w,
                                              const uint4 (&pre)[kScatterVecs]) {
  const int lane = threadIdx.x & 31;
  const int K = p.K;
  const int s = source_of_token(p, gt);
  const SourceDesc& src = p.src[s];
  const int t = gt - src.tok_off;
  if (lane < K) {
    if (code >= 0)
      write_route(p, s, t, gt, code, kPre ? pre_w : src.w[(int64_t)t * K + lane]);
    else
      p.routes[(int64_t)gt * K + lane] = make_int2(-1, 0);
  }
  copy_token<kPre>(p, src, t, lane < K ? code : -1, pre);
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

// The layout is one thread-block cluster of n CTAs (n <= 16). CTA r counts
// the tokens [r * tpc, (r + 1) * tpc) of the flattened (source, token) order
// (tpc = ceil(N / n)) in slices of 256, keeping a running count per expert in
// its shared memory, and gives each valid route its rank among the CTA's
// routes to the same expert (kept in shared memory). After a cluster barrier
// every CTA reads all n count vectors through distributed shared memory, so
// each one computes the totals, the aligned per-worker scan and the first
// row of its own run of each expert (start[e] plus the counts of CTAs
// r' < r) without a global-memory round trip, and writes its routes' final
// codes: (worker << 24) | (that first row + rank). The scatter kernel,
// spread over every SM, writes the receipts from them. Because the CTAs hold
// consecutive token ranges and ranks follow token order inside a CTA, rows
// inside an expert follow (source, token) order.
constexpr int kLocalRankBits = 21;  // local code = (expert << 21) | rank in the CTA
constexpr int kLayoutCodesMax = 8192;  // local codes a CTA keeps in shared memory (32 KB)

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Reads the int32 at the same shared-memory offset as `local` in CTA `rank`
// of this cluster. Only called between cluster barriers, when the value no
// longer changes, so the loads may be reordered and overlapped freely.
__device__ __forceinline__ int32_t ld_cluster(const int32_t* local, uint32_t rank) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
  uint32_t ra;
  int32_t v;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm("ld.shared::cluster.b32 %0, [%1];" : "=r"(v) : "r"(ra));
  return v;
}

__device__ __forceinline__ int layout_tpc(const DispatchParams& p) {
  return (p.total_tokens + p.layout_ctas - 1) / p.layout_ctas;
}

__global__ void __launch_bounds__(kChunk, 1) cluster_layout_kernel(const __grid_constant__ DispatchParams p) {
  AFD_STAMP_REGS;
  AFD_STAMP_REG(0);
  extern __shared__ __align__(16) uint32_t smem[];
  const int E = p.E, K = p.K, N = p.total_tokens;
  uint32_t* mask = smem;                                        // [8][E]
  int32_t* wbase = reinterpret_cast<int32_t*>(mask + kChunkWarps * E);  // [8][E]
  int32_t* cnt = wbase + kChunkWarps * E;                       // [E] this CTA's counts
  int32_t* total = cnt + E;                                     // [E]
  int32_t* start = total + E;                                   // [E]
  int32_t* before = start + E;                                  // [E] counts of earlier CTAs
  int32_t* codes_sm = before + E;                               // [tpc * K] when they fit
  // The first kernel of an exchange is a programmatic dependent of whatever
  // ran before it on the stream: it waits for that work (which may produce
  // the IDs, weights and rows, or still read the arenas) before touching
  // memory, and only then lets the scatter launch.
  pdl_wait();
  AFD_STAMP_REG(1);
  pdl_launch_dependents();

  const int n = gridDim.x;
  const uint32_t r = cluster_rank();
  const int tpc = layout_tpc(p);
  const int lo = min(N, (int)r * tpc), hi = min(N, lo + tpc);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t lanes_before = (1u << lane) - 1u;
  // each route's (expert, rank in this CTA) until the scan gives its row: in
  // shared memory when they fit, else in the route-code scratch itself
  int32_t* codes = (int64_t)tpc * K <= kLayoutCodesMax ? codes_sm : p.route_tmp + (int64_t)lo * K;

  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  for (int c0 = lo; c0 < hi; c0 += kChunk) {
    const int gt = c0 + threadIdx.x;
    const bool live = gt < hi;
    int s = 0, t = 0;
    if (live) {
      s = source_of_token(p, gt);
      t = gt - p.src[s].tok_off;
      // start the IDs' first read while the masks are cleared
      asm volatile("prefetch.global.L1 [%0];" ::"l"(p.src[s].ids + (int64_t)t * K));
    }
    for (int i = threadIdx.x; i < kChunkWarps * E; i += blockDim.x) mask[i] = 0u;
    __syncthreads();
    const int64_t* ids = p.src[s].ids + (int64_t)t * K;
    int e8[8];
    const uint32_t valid = live ? mark_token(ids, K, E, mask + warp * E, lane, s, t, p.err, e8) : 0u;
    __syncthreads();
    if (c0 == lo) AFD_STAMP_REG(2);  // the first slice's IDs read and marked
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int run = cnt[e];
#pragma unroll
      for (int w = 0; w < kChunkWarps; ++w) {
        wbase[w * E + e] = run;
        run += __popc(mask[w * E + e]);
      }
      cnt[e] = run;
    }
    __syncthreads();
    if (live) {
      int32_t* mine = codes + (int64_t)(gt - lo) * K;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (k >= K) continue;
        int code = -1;
        if ((valid >> k) & 1u) {
          const int e = e8[k];
          code = (e << kLocalRankBits) | (wbase[warp * E + e] + __popc(mask[warp * E + e] & lanes_before));
        }
        mine[k] = code;
      }
      for (int k = 8; k < K; ++k) {
        int code = -1;
        if ((valid >> k) & 1u) {
          const int e = (int)ids[k];
          code = (e << kLocalRankBits) | (wbase[warp * E + e] + __popc(mask[warp * E + e] & lanes_before));
        }
        mine[k] = code;
      }
    }
    __syncthreads();  // the masks are cleared for the next slice
  }

  AFD_STAMP_REG(3);
  // Every CTA's counts are final: read them all through the cluster.
  cluster_arrive();
  cluster_wait();
  AFD_STAMP_REG(4);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int v[kLayoutMaxCtas];
#pragma unroll
    for (int q = 0; q < kLayoutMaxCtas; ++q) v[q] = q < n ? ld_cluster(cnt + e, (uint32_t)q) : 0;
    int b = 0, all = 0;
#pragma unroll
    for (int q = 0; q < kLayoutMaxCtas; ++q) {
      b += q < (int)r ? v[q] : 0;
      all += v[q];
    }
    before[e] = b;
    total[e] = all;
  }
  AFD_STAMP_REG(5);
  // no CTA may leave (and free its shared memory) while others still read it
  cluster_arrive();
  __syncthreads();
  worker_scan(p, total, start, r == 0);
  __syncthreads();
  AFD_STAMP_REG(6);
  // this CTA's first code per expert: (worker << 24) | its first row
  for (int e = threadIdx.x; e < E; e += blockDim.x) start[e] = ((e / p.Ef) << kWorkerShift) + start[e] + before[e];
  __syncthreads();
  // every route's final code: (worker << 24) | row, or -1
  for (int i = threadIdx.x; i < (hi - lo) * K; i += blockDim.x) {
    const int c = codes[i];
    p.route_tmp[(int64_t)lo * K + i] =
        c < 0 ? -1 : start[c >> kLocalRankBits] + (c & ((1 << kLocalRankBits) - 1));
  }
  AFD_STAMP_REG(7);
  cluster_wait();
  AFD_STAMP_REGS_STORE(g_dispatch_stamps, 0);
}

__global__ void __launch_bounds__(AFD_SCATTER_BLOCK) scatter_kernel(const __grid_constant__ DispatchParams p) {
  AFD_STAMP(g_dispatch_stamps, 1, 0);
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int gwarp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const int K = p.K;

  // The source rows and weights are inputs, not layout outputs: start loading
  // this warp's first token while the layout kernel is still running.
  uint4 pre[kScatterVecs];
  float pre_w = 0.0f;
  const bool have_pre =
      preload_first(p, gwarp < p.total_tokens ? scatter_token_of(p, gwarp) : gwarp, pre, pre_w);
  pdl_wait();  // the layout kernel's outputs
  AFD_STAMP(g_dispatch_stamps, 1, 1);

  auto code_of = [&](int gt) { return lane < K ? __ldcg(p.route_tmp + (int64_t)gt * K + lane) : -1; };
  int i = gwarp;
  if (have_pre) {
    const int gt = scatter_token_of(p, i);
    scatter_token<true>(p, gt, code_of(gt), pre_w, pre);
    i += nwarps;
  }
  for (; i < p.total_tokens; i += nwarps) {
    const int gt = scatter_token_of(p, i);
    scatter_token<false>(p, gt, code_of(gt), 0.0f, pre);
  }
  fill_padding(p, p.ends);
  AFD_STAMP(g_dispatch_stamps, 1, 5);
}

// ---- bulk-copy scatter (rows of at most kBulkRowMax bytes in device memory)

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// One bulk copy of `bytes` from global memory into shared memory, completing
// on the barrier (which expects that many bytes).
__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src, uint32_t bytes, uint64_t* mbar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(mbar)), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst_smem)),
               "l"(src), "r"(bytes), "r"(smem_addr(mbar))
               : "memory");
}

// One poll of the barrier's phase `parity` (the thread may be suspended for a
// while inside it); true once that phase has completed.
__device__ __forceinline__ bool phase_done(uint64_t* mbar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(done)
      : "r"(smem_addr(mbar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the barrier's phase `parity`, at most `polls` polls. Every lane
// polls, and the warp leaves the loop together: once all lanes have seen the
// phase complete (true), or when the limit is reached (false). A completed
// phase stays visible until the next arrival, which only lane 0 makes after
// this wait, so the lanes cannot disagree for long.
__device__ __forceinline__ bool wait_phase_warp(uint64_t* mbar, uint32_t parity, int polls) {
  for (int i = 0; i < polls; ++i)
    if (__all_sync(0xffffffffu, phase_done(mbar, parity))) return true;
  return false;
}

// The wait for a load still in flight after a wait gave up: bounded by time
// (kDrainNs of the global timer), so that it ends however long each poll
// suspends the thread. The warp decides together, as above.
constexpr unsigned long long kDrainNs = 2000000000ull;  // 2 s
__device__ __forceinline__ bool drain_phase_warp(uint64_t* mbar, uint32_t parity) {
  const unsigned long long t0 = global_timer_ns();
  for (;;) {
    if (__all_sync(0xffffffffu, phase_done(mbar, parity))) return true;
    const unsigned long long dt = global_timer_ns() - t0;  // lane 0's clock decides for the warp
    if (__shfl_sync(0xffffffffu, dt, 0) > kDrainNs) return false;
  }
}

// One bulk copy of `bytes` from shared memory to global memory, with an L2
// evict-last policy: the rows are read again soon, by the combine (with the
// identity expert) or by the expert, and kept dirty in L2 they are not
// written back while the combine streams its replies (round trips at T=2048
// after an L2 flush that evicts such lines too: FP8 2A2F 51.4 -> 49.7 us,
// skew 3A:1F 69.6 -> 68.1, H4096 95.6 -> 94.2; 2A2F H2048 48.1 -> 48.6,
// within the run-to-run spread, and 49.1 -> 47.2 back to back).
__device__ __forceinline__ void bulk_store(void* dst, const void* src_smem, uint32_t bytes) {
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dst),
               "r"(smem_addr(src_smem)), "r"(bytes), "l"(pol)
               : "memory");
}

// The scatter with bulk (TMA) copies: a warp per token; lane 0 brings the
// row into the warp's shared-memory buffer with one bulk copy, and lane k < K
// writes it to route k's row with one bulk copy, while the lanes write the
// receipts (and FP8 scales) with ordinary stores. The buffer is reused for
// the warp's next token once every lane's copies have read it.
// kCached: the copy along the last exchange's receipts (cached dispatch):
// the route codes come from the receipt, and new weights, when given,
// replace the old ones in both receipts.
template <bool kCached>
__global__ void __launch_bounds__(64) scatter_bulk_kernel(const __grid_constant__ DispatchParams p) {
  if (!kCached) AFD_STAMP(g_dispatch_stamps, 1, 0);
  extern __shared__ __align__(128) uint8_t bsm[];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(bsm) + wib;       // one barrier per warp
  uint8_t* buf = bsm + 128 + (size_t)wib * p.row_bytes;          // one row per warp
  const int gwarp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const int K = p.K;
  const uint32_t rb = (uint32_t)p.row_bytes;
  if (lane == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(mbar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  if (kCached) {  // the first kernel of the exchange (see cluster_layout_kernel)
    pdl_wait();
    pdl_launch_dependents();
  } else {
    pdl_launch_dependents();
  }
  // the source rows (and FP8 scales) are inputs, not layout outputs: load
  // the first token's while the layout is still running
  float sc_first = 0.0f;
  if (gwarp < p.total_tokens) {
    const int g0 = scatter_token_of(p, gwarp);
    const int s0 = source_of_token(p, g0);
    const int t0 = g0 - p.src[s0].tok_off;
    if (lane == 0) bulk_load(buf, p.src[s0].x + (int64_t)t0 * rb, rb, mbar);
    if (lane < p.nscale) sc_first = p.src[s0].scale[(int64_t)t0 * p.src[s0].sst + (int64_t)lane * p.src[s0].ssb];
  }
  if (!kCached) pdl_wait();  // the layout kernel's route codes
  if (!kCached) AFD_STAMP(g_dispatch_stamps, 1, 1);

  uint32_t parity = 0;
  // false once a wait of this warp gave up: the warp then writes only the
  // receipts of its remaining tokens (valid codes, so that the combine never
  // reads outside the arenas) and moves no more rows
  bool copying = true;
  for (int gi = gwarp; gi < p.total_tokens; gi += nwarps) {
    const int gt = scatter_token_of(p, gi);
    const bool first = gi == gwarp;
    const int s = source_of_token(p, gt);
    const SourceDesc& src = p.src[s];
    const int t = gt - src.tok_off;
    if (copying && !first && lane == 0) bulk_load(buf, src.x + (int64_t)t * rb, rb, mbar);
    int code = -1;
    if (kCached) {
      if (lane < K) {
        int2* r = p.routes + (int64_t)gt * K + lane;
        code = r->x;
        if (src.w != nullptr && code >= 0) {
          const float w = src.w[(int64_t)t * K + lane];
          r->y = __float_as_int(w);
          p.row_w[(int64_t)(code >> kWorkerShift) * p.R_arena + (code & kRowMask)] = w;
        }
      }
    } else {
      code = lane < K ? __ldcg(p.route_tmp + (int64_t)gt * K + lane) : -1;
      if (lane < K) {
        if (code >= 0)
          write_route(p, s, t, gt, code, src.w[(int64_t)t * K + lane]);
        else
          p.routes[(int64_t)gt * K + lane] = make_int2(-1, 0);
      }
    }
    if (copying) {
      if (!wait_phase_warp(mbar, parity, p.wait_polls)) {
        // the row's load did not complete in time: report it, and wait
        // (bounded by time) for the load still in flight before the buffer
        // is abandoned
        if (lane == 0) atomicMin(p.err, route_error_key(s, t, 0, kErrTimeout));
        drain_phase_warp(mbar, parity);
        copying = false;
      } else {
        if (!kCached && first) AFD_STAMP(g_dispatch_stamps, 1, 2);  // first row in shared memory
        parity ^= 1u;
        if (code >= 0)
          bulk_store(p.rows + ((int64_t)(code >> kWorkerShift) * p.R_arena + (code & kRowMask)) * rb, buf, rb);
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      }
    }
    // FP8: the row's block scales follow it, written while its bulk stores run
    for (int b0 = 0; b0 < p.nscale; b0 += 32) {
      const int b = b0 + lane;
      float sc = 0.0f;
      if (b < p.nscale)
        sc = (first && b0 == 0) ? sc_first : src.scale[(int64_t)t * src.sst + (int64_t)b * src.ssb];
      for (int k = 0; k < K; ++k) {
        const int c = __shfl_sync(0xffffffffu, code, k);
        if (c >= 0 && b < p.nscale)
          p.row_scales[((int64_t)(c >> kWorkerShift) * p.R_arena + (c & kRowMask)) * p.nscale + b] = sc;
      }
    }
    if (copying) {
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");  // this lane's copies have read buf
      __syncwarp();
    }
  }
  if (!kCached) AFD_STAMP(g_dispatch_stamps, 1, 3);
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");  // this lane's copies are complete
  if (!kCached) AFD_STAMP(g_dispatch_stamps, 1, 4);
  if (!kCached) fill_padding(p, p.ends);
  if (!kCached) AFD_STAMP(g_dispatch_stamps, 1, 5);
}

// Copies token (s, t)'s row to one route's row (code = (worker << 24) | row,
// or -1 for none). kPre: `pre` holds the row's first piece.
template <bool kPre>
__device__ __forceinline__ void copy_route(const DispatchParams& p, const SourceDesc& src, int t, int code,
                                           const uint4 (&pre)[kScatterVecs]) {
  if (code < 0) return;
  const int lane = threadIdx.x & 31;
  const int nvec = p.row_bytes >> 4;
  const uint4* xrow = reinterpret_cast<const uint4*>(src.x + (int64_t)t * p.row_bytes);
  const int64_t r = (int64_t)(code >> kWorkerShift) * p.R_arena + (code & kRowMask);
  uint4* dst = reinterpret_cast<uint4*>(p.rows + r * p.row_bytes);
  for (int v0 = 0; v0 < nvec; v0 += 32 * kScatterVecs) {
    uint4 buf[kScatterVecs];
    if (kPre && v0 == 0) {
#pragma unroll
      for (int j = 0; j < kScatterVecs; ++j) buf[j] = pre[j];
    } else {
      load_piece(buf, xrow, v0, nvec);
    }
#pragma unroll
    for (int j = 0; j < kScatterVecs; ++j) {
      const int v = v0 + j * 32 + lane;
      if (v < nvec) dst[v] = buf[j];
    }
  }
  for (int b = lane; b < p.nscale; b += 32)
    p.row_scales[r * p.nscale + b] = src.scale[(int64_t)t * src.sst + (int64_t)b * src.ssb];
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

  AFD_STAMP(g_dispatch_stamps, 0, 0);
  pdl_wait();  // the work before the exchange (see cluster_layout_kernel)
  AFD_STAMP(g_dispatch_stamps, 0, 1);
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long* err = blockIdx.x == 0 ? p.err : nullptr;
  const int gwarp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;

  // Load this warp's first two (token, route) pairs' rows and weights now,
  // so that their latency overlaps the counting below (a launch has at most
  // two pairs per warp up to kSmallRoutes routes on a full device).
  uint4 pre[kScatterVecs], pre2[kScatterVecs];
  float pre_w = 0.0f, pre2_w = 0.0f;
  if (gwarp < N * K) {
    const int gt = gwarp / K, s = source_of_token(p, gt), t = gt - p.src[s].tok_off;
    load_piece(pre, reinterpret_cast<const uint4*>(p.src[s].x + (int64_t)t * p.row_bytes), 0, p.row_bytes >> 4);
    if (lane == 0) pre_w = p.src[s].w[(int64_t)t * K + (gwarp - gt * K)];
  }
  if (gwarp + nwarps < N * K) {
    const int pr = gwarp + nwarps;
    const int gt = pr / K, s = source_of_token(p, gt), t = gt - p.src[s].tok_off;
    load_piece(pre2, reinterpret_cast<const uint4*>(p.src[s].x + (int64_t)t * p.row_bytes), 0, p.row_bytes >> 4);
    if (lane == 0) pre2_w = p.src[s].w[(int64_t)t * K + (pr - gt * K)];
  }

  // Pass 1 (every block, all routes): ranks inside each chunk, chunk counts.
  for (int c = 0; c < G; ++c) {
    for (int i = threadIdx.x; i < kChunkWarps * E; i += blockDim.x) mask[i] = 0u;
    __syncthreads();
    const int gt = c * kChunk + threadIdx.x;
    const bool live = gt < N;
    int s = 0, t = 0;
    const int64_t* ids = nullptr;
    uint32_t valid = 0u;
    int e8[8];
    if (live) {
      s = source_of_token(p, gt);
      t = gt - p.src[s].tok_off;
      ids = p.src[s].ids + (int64_t)t * K;
      valid = mark_token(ids, K, E, mask + warp * E, lane, s, t, err, e8);
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
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (k >= K) continue;
        uint32_t info = ~0u;
        if ((valid >> k) & 1u) {
          const int e = e8[k];
          info = ((uint32_t)e << kRankBits) |
                 (uint32_t)(wbase[warp * E + e] + __popc(mask[warp * E + e] & lanes_before));
        }
        rinfo[gt * K + k] = info;
      }
      for (int k = 8; k < K; ++k) {
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

  // Pass 2: a warp per (token, route) pair: the route's receipt and its row.
  for (int pr = gwarp; pr < N * K; pr += nwarps) {
    const int gt = pr / K, kk = pr - gt * K;
    const int s = source_of_token(p, gt);
    const SourceDesc& src = p.src[s];
    const int t = gt - src.tok_off;
    int code = -1;
    if (lane == 0) {
      const uint32_t info = rinfo[gt * K + kk];
      const float w = pr == gwarp ? pre_w : pr == gwarp + nwarps ? pre2_w : src.w[(int64_t)t * K + kk];
      if (info != ~0u) {
        const int e = (int)(info >> kRankBits);
        const int row = sh_start[e] + ccnt[(gt / kChunk) * E + e] + (int)(info & ((1u << kRankBits) - 1));
        const int f = e / p.Ef;
        const int64_t r = (int64_t)f * p.R_arena + row;
        p.row_src[r] = (s * p.bucket + t) * K + kk;
        p.row_w[r] = w;
        code = (f << kWorkerShift) | row;
        p.routes[(int64_t)gt * K + kk] = make_int2(code, __float_as_int(w));
      } else {
        p.routes[(int64_t)gt * K + kk] = make_int2(-1, 0);
      }
    }
    code = __shfl_sync(0xffffffffu, code, 0);
    if (pr == gwarp)
      copy_route<true>(p, src, t, code, pre);
    else if (pr == gwarp + nwarps)
      copy_route<true>(p, src, t, code, pre2);
    else
      copy_route<false>(p, src, t, code, pre);
  }

  // Padding rows, from this block's own copy of the layout.
  for (int e = threadIdx.x; e < E; e += blockDim.x) sh_total[e] += sh_start[e];  // ends
  __syncthreads();
  fill_padding(p, sh_total);
  AFD_STAMP(g_dispatch_stamps, 0, 7);
}

// ---------------------------------------------------------------- cached path

// Dispatch with the previous exchange's routing: the receipt already holds
// every route's row, so a warp per token only copies the row (and, when new
// weights are given, refreshes the weights in both receipts).
__global__ void __launch_bounds__(AFD_SCATTER_BLOCK) cached_scatter_kernel(const __grid_constant__ DispatchParams p) {
  pdl_wait();  // the work before the exchange (see cluster_layout_kernel)
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int gwarp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const int K = p.K;
  uint4 none[kScatterVecs];
  for (int gi = gwarp; gi < p.total_tokens; gi += nwarps) {
    const int gt = scatter_token_of(p, gi);
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

// One warp scans all E experts in one pass: lane i owns the experts
// [i * epl, (i + 1) * epl), epl = ceil(E / 32); the first expert of every
// worker starts a new segment of the (segmented) scan of aligned counts.
// count_of(e) gives expert e's count. Writes sh_start / sh_end, and with
// `out` the context's starts, ends and aligned counts.
template <typename CountOf>
__device__ __forceinline__ void warp_worker_scan(const DispatchParams& p, CountOf count_of,
                                                 int32_t* sh_start, int32_t* sh_end, bool out) {
  const int lane = threadIdx.x & 31;
  const int E = p.E, Ef = p.Ef;
  const int epl = (E + 31) >> 5;
  const int e0 = lane * epl, e1 = min(E, e0 + epl);
  // the sum of aligned counts since the last worker start in this lane's range
  int v = 0, f = 0;
  for (int e = e0, l = e0 % Ef; e < e1; ++e, l = (l + 1 == Ef ? 0 : l + 1)) {
    if (l == 0) {
      v = 0;
      f = 1;
    }
    v += align_up_dev(count_of(e), p.alpha);
  }
  // inclusive segmented scan over the lanes: (v, f) after (v', f') is
  // (f ? v : v' + v, f | f')
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int vu = __shfl_up_sync(0xffffffffu, v, d);
    const int fu = __shfl_up_sync(0xffffffffu, f, d);
    if (lane >= d) {
      if (!f) v += vu;
      f |= fu;
    }
  }
  int run = __shfl_up_sync(0xffffffffu, v, 1);  // running sum at the end of the previous lane
  if (lane == 0) run = 0;
  for (int e = e0, l = e0 % Ef; e < e1; ++e, l = (l + 1 == Ef ? 0 : l + 1)) {
    if (l == 0) run = 0;
    const int cnt = count_of(e);
    const int al = align_up_dev(cnt, p.alpha);
    sh_start[e] = run;
    sh_end[e] = run + cnt;
    if (out) {
      p.starts[e] = run;
      p.ends[e] = run + cnt;
      p.hcounts[e] = al;
    }
    run += al;
  }
}

// At most 32 tokens in the whole exchange: one-warp blocks, one per (token,
// route) pair (and at least one per expert up to 128; they share the padding
// rows). Every block
// counts all the routes itself with one lane mask per expert (lane = token),
// so ranks are popcounts of earlier lanes and no block waits for another;
// block b then writes the receipt of route b % K of token b / K and copies
// the token's row there.
__global__ void __launch_bounds__(32) dispatch_tiny_kernel(const __grid_constant__ DispatchParams p) {
  extern __shared__ __align__(16) uint32_t tsm[];
  const int E = p.E, K = p.K, N = p.total_tokens;
  uint32_t* mask = tsm;                                     // [E]
  int32_t* sh_start = reinterpret_cast<int32_t*>(mask + E);  // [E]
  int32_t* sh_end = sh_start + E;                           // [E]
  AFD_STAMP(g_dispatch_stamps, 0, 0);
  pdl_wait();  // the work before the exchange (see cluster_layout_kernel)
  AFD_STAMP(g_dispatch_stamps, 0, 1);
  pdl_launch_dependents();
  const int lane = threadIdx.x;

  // this block's route: token gt, route kk; its row, weight and ID load now
  const bool has_pair = (int)blockIdx.x < N * K;
  const int gt = has_pair ? (int)blockIdx.x / K : 0;
  const int kk = (int)blockIdx.x - gt * K;
  const int s = source_of_token(p, gt);
  const SourceDesc& src = p.src[s];
  const int t = gt - src.tok_off;
  uint4 pre[kScatterVecs];
  float w = 0.0f;
  int64_t id = -1;
  if (has_pair) {
    load_piece(pre, reinterpret_cast<const uint4*>(src.x + (int64_t)t * p.row_bytes), 0, p.row_bytes >> 4);
    if (lane == 0) {
      w = src.w[(int64_t)t * K + kk];
      id = src.ids[(int64_t)t * K + kk];
    }
  }

  for (int e = lane; e < E; e += 32) mask[e] = 0u;
  __syncwarp();
  uint32_t valid = 0u;
  if (lane < N) {
    const int ls = source_of_token(p, lane);
    const int lt = lane - p.src[ls].tok_off;
    int e8[8];
    valid = mark_token(p.src[ls].ids + (int64_t)lt * K, K, E, mask, lane, ls, lt,
                       blockIdx.x == 0 ? p.err : nullptr, e8);
  }
  __syncwarp();
  warp_worker_scan(p, [&](int e) { return __popc(mask[e]); }, sh_start, sh_end, blockIdx.x == 0);
  __syncwarp();

  if (has_pair) {
    const bool ok = (__shfl_sync(0xffffffffu, valid, gt) >> kk) & 1u;
    int code = -1;
    if (lane == 0) {
      if (ok) {
        const int e = (int)id;
        const int row = sh_start[e] + __popc(mask[e] & ((1u << gt) - 1u));
        const int f = e / p.Ef;
        const int64_t r = (int64_t)f * p.R_arena + row;
        p.row_src[r] = (s * p.bucket + t) * K + kk;
        p.row_w[r] = w;
        code = (f << kWorkerShift) | row;
        p.routes[(int64_t)gt * K + kk] = make_int2(code, __float_as_int(w));
      } else {
        p.routes[(int64_t)gt * K + kk] = make_int2(-1, 0);
      }
    }
    copy_route<true>(p, src, t, __shfl_sync(0xffffffffu, code, 0), pre);
  }
  // padding rows, spread over the blocks: block b takes the experts
  // b, b + gridDim.x, ...; its lanes look at 32 of them at once, then the
  // warp writes the padding rows of each one that has some
  if (p.alpha > 1) {
    for (int i0 = 0; (int)blockIdx.x + i0 * (int)gridDim.x < E; i0 += 32) {
      const int e = (int)blockIdx.x + (i0 + lane) * (int)gridDim.x;
      int end = 0, lim = 0;
      if (e < E) {
        end = sh_end[e];
        lim = align_up_dev(end, p.alpha);
      }
      uint32_t todo = __ballot_sync(0xffffffffu, lim > end);
      while (todo) {
        const int src = __ffs(todo) - 1;
        todo &= todo - 1u;
        const int pe = __shfl_sync(0xffffffffu, end, src), pl = __shfl_sync(0xffffffffu, lim, src);
        const int ee = (int)blockIdx.x + (i0 + src) * (int)gridDim.x;
        const int64_t base = (int64_t)(ee / p.Ef) * p.R_arena;
        for (int row = pe + lane; row < pl; row += 32) {
          p.row_src[base + row] = -1;
          p.row_w[base + row] = 0.0f;
        }
      }
    }
  }
  AFD_STAMP(g_dispatch_stamps, 0, 7);
}

size_t layout_smem(int E) { return (size_t)kChunkWarps * E * 8 + (size_t)4 * E * 4 + (size_t)kLayoutCodesMax * 4; }


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

int layout_ctas_for(int total_tokens, int sm_cap, int max_ctas) {
  int n = (total_tokens + kChunk - 1) / kChunk;
  if (n > max_ctas) n = max_ctas;
  if (n > sm_cap) n = sm_cap;
  return n < 1 ? 1 : n;
}

bool dispatch_is_small(const DispatchParams& p) {
  return (int64_t)p.total_tokens * p.K <= kSmallRoutes &&
         small_smem(p.E, p.total_tokens, p.K) <= (size_t)kSmallSmemMax;
}

// Sets the kernels' shared-memory and cluster attributes on the current
// device and returns in *max_ctas the largest layout cluster it can run.
cudaError_t configure_dispatch_kernels(int* max_ctas) {
  cudaError_t e = cudaFuncSetAttribute(cluster_layout_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)layout_smem(kMaxExperts));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(cluster_layout_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(dispatch_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmallSmemMax);
  for (const void* k : {(const void*)cluster_layout_kernel, (const void*)scatter_kernel,
                        (const void*)scatter_bulk_kernel<false>, (const void*)scatter_bulk_kernel<true>,
                        (const void*)dispatch_small_kernel, (const void*)dispatch_tiny_kernel,
                        (const void*)cached_scatter_kernel})
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, kSharedCarveout);
  if (e != cudaSuccess) return e;
  // the largest cluster that fits with the largest shared-memory request
  for (int n = kLayoutMaxCtas; n >= 1; n /= 2) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n);
    cfg.blockDim = dim3(kChunk);
    cfg.dynamicSmemBytes = layout_smem(kMaxExperts);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = n;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, cluster_layout_kernel, &cfg) != cudaSuccess) {
      cudaGetLastError();  // this size is not available: try a smaller one
      continue;
    }
    if (clusters >= 1) {
      *max_ctas = n;
      return cudaSuccess;
    }
  }
  return cudaErrorInvalidConfiguration;
}

// Launches the exchange's dispatch. Every kernel is a programmatic dependent
// of the one before it. The first one waits (griddepcontrol.wait) for all
// earlier work on the stream before it reads or writes anything, so it never
// overlaps the producer of its inputs or the previous exchange's combine,
// which still reads the arenas; it lets its own dependents launch only after
// that wait.
cudaError_t launch_dispatch(const DispatchParams& p, int sm_cap, cudaStream_t stream) {
  const int block = 256;
  if (p.total_tokens >= 1 && p.total_tokens <= 32 && AFD_TINY_DISPATCH) {
    // one block per (token, route), and at least one per expert (up to 128)
    // so that each block has the padding rows of one expert at most: with 16
    // blocks for 128 experts the round trip at one token per source took 2 us
    // longer
    const int pairs = p.total_tokens * p.K;
    const int min_blocks = p.E < AFD_TINY_MIN_BLOCKS ? p.E : AFD_TINY_MIN_BLOCKS;
    const int grid = pairs > min_blocks ? pairs : min_blocks;
    return launch(dispatch_tiny_kernel, grid, 32, (size_t)3 * p.E * sizeof(int32_t), stream, true, p);
  }
  if (dispatch_is_small(p)) {
    int grid = (p.total_tokens * p.K + 7) / 8;  // a warp per (token, route)
    if (grid > sm_cap) grid = sm_cap;
    if (grid < 1) grid = 1;
    return launch(dispatch_small_kernel, grid, block, small_smem(p.E, p.total_tokens, p.K), stream,
                  true, p);
  }
  // the layout cluster (its size was chosen with the launch parameters)
  const int n = p.layout_ctas;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n);
  cfg.blockDim = dim3(kChunk);
  cfg.dynamicSmemBytes = layout_smem(p.E);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = n;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, cluster_layout_kernel, p);
  if (e != cudaSuccess) return e;
  // small blocks, a warp per token, so that blocks spread evenly over the SMs
  constexpr int kWarps = AFD_SCATTER_BLOCK / 32;
  int grid = (p.total_tokens + kWarps - 1) / kWarps;
  if (grid > sm_cap * (2048 / AFD_SCATTER_BLOCK)) grid = sm_cap * (2048 / AFD_SCATTER_BLOCK);
  if (grid < 1) grid = 1;
  if (p.x_device && p.row_bytes <= kBulkRowMax) {
    // small blocks with a row buffer per warp, so that they spread evenly over
    // the SMs: two warps, or one for rows of at most 2 KB (FP8 at H=2048),
    // whose blocks all fit the shared memory at once (FP8 2A2F T=2048 round
    // trip 49.6 -> 48.5 us, 49.1 -> 47.6 back to back; FP8 2A1F and T=1024
    // unchanged; one-warp blocks for 4 KB rows: 48.0 -> 49.7 us)
    const int kBulkWarps = p.row_bytes <= 2048 ? 1 : 2;
    int bgrid = (p.total_tokens + kBulkWarps - 1) / kBulkWarps;
    if (bgrid > sm_cap * 32) bgrid = sm_cap * 32;
    return launch(scatter_bulk_kernel<false>, bgrid, 32 * kBulkWarps, 128 + (size_t)kBulkWarps * p.row_bytes,
                  stream, true, p);
  }
  return launch(scatter_kernel, grid, AFD_SCATTER_BLOCK, 0, stream, true, p);
}

}  // namespace afd

namespace afd {

// A programmatic dependent of the work before it, which it waits for before
// it rewrites the rows that the previous exchange's combine reads.
cudaError_t launch_cached_scatter(const DispatchParams& p, int sm_cap, cudaStream_t stream) {
  if (p.x_device && p.row_bytes <= kBulkRowMax) {
    constexpr int kBulkWarps = 2;
    int bgrid = (p.total_tokens + kBulkWarps - 1) / kBulkWarps;
    if (bgrid > sm_cap * 32) bgrid = sm_cap * 32;
    if (bgrid < 1) bgrid = 1;
    return launch(scatter_bulk_kernel<true>, bgrid, 32 * kBulkWarps, 128 + (size_t)kBulkWarps * p.row_bytes,
                  stream, true, p);
  }
  constexpr int kWarps = AFD_SCATTER_BLOCK / 32;
  int grid = (p.total_tokens + kWarps - 1) / kWarps;
  if (grid > sm_cap * (2048 / AFD_SCATTER_BLOCK)) grid = sm_cap * (2048 / AFD_SCATTER_BLOCK);
  if (grid < 1) grid = 1;
  return launch(cached_scatter_kernel, grid, AFD_SCATTER_BLOCK, 0, stream, true, p);
}

}  // namespace afd
