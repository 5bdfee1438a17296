// Dispatch kernels: route layout (validate, histogram, aligned scan, ranks)
// and the scatter of source rows into expert-major worker arenas.
//
// What they compute follows the afdEP-comm "API contract" (Roles and tensors:
// ID rules, worker-owned expert blocks, the ends[] prefix sums with
// expert_alignment padding, aligned host counts) and "DeepEP V2 ElasticBuffer
// first principles" section 3 (count routes per expert, give every route a
// slot, copy each token's row to every selected expert; section 7: FP8 rows
// travel with their scales). Unlike the atomic slot counters described there,
// slots here are assigned by a stable counting sort, so rows inside an expert
// follow (source, token) order and every run gives the same layout.
//
// Layout (one launch): each 256-thread block owns a chunk of 256 tokens of
// one source, one token per thread. Per warp and expert a shared-memory lane
// mask collects which of the warp's 32 tokens route to the expert; a route's
// rank inside the chunk is the count of earlier warps' tokens plus the popcount
// of earlier lanes in its own mask. A repeated ID shows up as a bit that is
// already set. The last block to finish (a completion counter, no waiting)
// sums the chunk counts per expert, runs the aligned exclusive scan per
// worker, and turns chunk counts into per-chunk starting rows.
//
// Scatter (one launch): a warp per token reads its route codes, finishes
// each route's row (chunk start + rank), writes the receipt entries, then
// reads the source row once with 16-byte loads and stores it to each of the K
// destination rows.

#include <cuda_runtime.h>
#include <stdint.h>

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

__device__ __forceinline__ int align_up(int v, int a) { return (v + a - 1) / a * a; }

__device__ __forceinline__ int warp_inclusive_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    int u = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += u;
  }
  return v;
}

// Sums the chunk counts, runs the aligned scan per worker and writes the
// per-chunk starting rows. Runs in the last block of the layout launch.
__device__ void layout_finish(const DispatchParams& p, int32_t* sh_total, int32_t* sh_start) {
  const int E = p.E, G = p.total_chunks;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;

  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int g = 0; g < G; ++g) run += __ldcg(p.chunk_counts + (int64_t)g * E + e);
    sh_total[e] = run;
  }
  __syncthreads();

  // Per worker: start = exclusive scan of align_up(count, alpha) over its
  // local experts; ends = start + count ("API contract": expert e occupies
  // [align_up(ends[e-1], alpha), ends[e]) with ends[-1] = 0).
  for (int f = warp; f < p.F; f += nwarps) {
    int carry = 0;
    for (int l0 = 0; l0 < p.Ef; l0 += 32) {
      const int l = l0 + lane;
      const int e = f * p.Ef + l;
      const int cnt = l < p.Ef ? sh_total[e] : 0;
      const int al = align_up(cnt, p.alpha);
      const int incl = warp_inclusive_scan(al);
      if (l < p.Ef) {
        const int start = carry + incl - al;
        sh_start[e] = start;
        p.starts[e] = start;
        p.ends[e] = start + cnt;
        p.hcounts[e] = al;
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();

  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = sh_start[e];
    for (int g = 0; g < G; ++g) {
      const int c = __ldcg(p.chunk_counts + (int64_t)g * E + e);
      p.chunk_start[(int64_t)g * E + e] = run;
      run += c;
    }
  }
}

__global__ void __launch_bounds__(kChunk) layout_kernel(const __grid_constant__ DispatchParams p) {
  extern __shared__ uint32_t smem[];
  uint32_t* mask = smem;                                   // [kChunkWarps][E]
  uint16_t* wbase = reinterpret_cast<uint16_t*>(smem + kChunkWarps * p.E);  // [kChunkWarps][E]
  __shared__ int is_last;

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

    // Validate and mark. IDs are read as int64 so that a value outside int32
    // is caught as out of range rather than truncated.
    uint32_t valid = 0u;
    const int64_t* ids = src.ids + (int64_t)t * K;
    if (live) {
      for (int k = 0; k < K; ++k) {
        const int64_t id = ids[k];
        if (id == -1) continue;
        if (id < -1 || id >= E) {
          atomicMin(p.err, route_error_key(s, t, k, kErrRange));
          continue;
        }
        const uint32_t old = atomicOr(mask + warp * E + (int)id, 1u << lane);
        if (old & (1u << lane)) {  // this token already routed to this expert
          atomicMin(p.err, route_error_key(s, t, k, kErrDup));
          continue;
        }
        valid |= 1u << k;
      }
    }
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
  int32_t* sh_total = reinterpret_cast<int32_t*>(smem);
  int32_t* sh_start = sh_total + E;
  layout_finish(p, sh_total, sh_start);
  if (threadIdx.x == 0) *p.done = 0u;
}

constexpr int kScatterVecs = 8;  // 16-byte vectors per lane in flight

__global__ void __launch_bounds__(256) scatter_kernel(const __grid_constant__ DispatchParams p) {
  const int lane = threadIdx.x & 31;
  const int gwarp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const int K = p.K;
  const int nvec = p.row_bytes >> 4;

  for (int gt = gwarp; gt < p.total_tokens; gt += nwarps) {
    const int s = source_of_token(p, gt);
    const SourceDesc& src = p.src[s];
    const int t = gt - src.tok_off;

    int code = -1;
    if (lane < K) {
      const int rt = p.route_tmp[(int64_t)gt * K + lane];
      const float w = src.w[(int64_t)t * K + lane];
      float wr = 0.0f;
      if (rt >= 0) {
        const int e = rt >> kRankBits;
        const int rank = rt & ((1 << kRankBits) - 1);
        const int g = src.chunk_off + t / kChunk;
        const int row = p.chunk_start[(int64_t)g * p.E + e] + rank;
        const int f = e / p.Ef;
        code = (f << kWorkerShift) | row;
        const int64_t r = (int64_t)f * p.R_arena + row;
        p.row_src[r] = (s * p.bucket + t) * K + lane;
        p.row_w[r] = w;
        wr = w;
      }
      p.routes[(int64_t)gt * K + lane] = make_int2(code, __float_as_int(wr));
    }

    // Read the row once, write it to every selected expert row.
    const uint4* xrow = reinterpret_cast<const uint4*>(src.x + (int64_t)t * p.row_bytes);
    for (int v0 = 0; v0 < nvec; v0 += 32 * kScatterVecs) {
      uint4 buf[kScatterVecs];
#pragma unroll
      for (int j = 0; j < kScatterVecs; ++j) {
        const int v = v0 + j * 32 + lane;
        if (v < nvec) buf[j] = __ldg(xrow + v);
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

  // Padding rows between ends[e] and the next aligned start: no route, so
  // row_src -1 and weight +0.
  if (p.alpha > 1) {
    const int64_t per = p.alpha - 1;
    const int64_t items = (int64_t)p.E * per;
    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < items; i += nthreads) {
      const int e = (int)(i / per);
      const int j = (int)(i % per);
      const int end = p.ends[e];
      const int row = end + j;
      if (row < align_up(end, p.alpha)) {
        const int64_t r = (int64_t)(e / p.Ef) * p.R_arena + row;
        p.row_src[r] = -1;
        p.row_w[r] = 0.0f;
      }
    }
  }
}

}  // namespace

static size_t layout_smem(int E) {
  return (size_t)kChunkWarps * E * sizeof(uint32_t) + (size_t)kChunkWarps * E * sizeof(uint16_t);
}

cudaError_t configure_kernels(int max_experts) {
  return cudaFuncSetAttribute(layout_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)layout_smem(max_experts));
}

cudaError_t launch_layout(const DispatchParams& p, int /*sm_cap*/, cudaStream_t stream) {
  const int grid = p.total_chunks > 0 ? p.total_chunks : 1;
  layout_kernel<<<grid, kChunk, layout_smem(p.E), stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_scatter(const DispatchParams& p, int sm_cap, cudaStream_t stream) {
  const int block = 256;
  const int warps_needed = p.total_tokens;
  int grid = (warps_needed + 7) / 8;
  const int pad_items = p.alpha > 1 ? p.E * (p.alpha - 1) : 0;
  if (grid < (pad_items + block - 1) / block) grid = (pad_items + block - 1) / block;
  const int cap = sm_cap * 8;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  scatter_kernel<<<grid, block, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace afd
