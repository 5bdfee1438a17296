// afd_route_layout_noalloc: the routing layout (route checks, per-expert
// counts, ends[] with expert_alignment padding, one row per valid route) for
// callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at all: code that runs inside another
// framework's memory pool, an allocator hook, or a process whose device
// memory is fully reserved up front. This entry point needs no allocation
// from them or from the library: its scratch (per-chunk counts, route ranks
// and the error key) lives in a fixed file-scope device array. The caller
// passes only its inputs and outputs.
//
// The scratch array is a device symbol. Host code may not hand the symbol
// itself to a kernel (on the host it is only a stand-in, not a device
// address); the device address comes from cudaGetSymbolAddress, looked up
// once per device, with that device current, on the first call made there.

#include <cuda_runtime.h>
#include <stdint.h>

#include <climits>
#include <mutex>

#include "afd.h"
#include "afd_device.cuh"

namespace {

constexpr int kNaMaxTokens = 8192;
constexpr int kNaMaxRoutes = 65536;       // tokens x top_k
constexpr int kNaMaxExperts = 1024;
constexpr int kNaMaxTopK = 32;
constexpr int kNaChunk = 256;             // tokens per counting block
constexpr int kNaWarps = kNaChunk / 32;
constexpr int kNaMaxChunks = kNaMaxTokens / kNaChunk;
constexpr int kNaMaxDevices = 64;

// Scratch layout (int32 words): [0, 2) the error key (uint64), padding to
// word 64, then per-chunk counts [chunks][E], then route ranks [T*K].
constexpr int kNaCountsOff = 64;
constexpr int kNaRanksOff = kNaCountsOff + kNaMaxChunks * kNaMaxExperts;
constexpr int kNaScratchWords = kNaRanksOff + kNaMaxRoutes;  // 98,368 words = 384 KiB

static __device__ __align__(256) int32_t g_layout_scratch[kNaScratchWords];

constexpr unsigned long long kNaNoError = ~0ull;
constexpr int kNaErrRange = AFD_ERR_ROUTE_RANGE;
constexpr int kNaErrDup = AFD_ERR_ROUTE_DUP;

__device__ __forceinline__ unsigned long long na_error_key(int t, int k, int code) {
  return ((unsigned long long)(uint32_t)t << 16) | ((unsigned long long)k << 8) |
         (unsigned long long)code;
}

// One block per chunk of 256 tokens, one token per thread: check the IDs,
// mark them in per-warp lane masks, write the chunk's count per expert and
// each route's rank inside the chunk ((expert << 8) | rank, or -1).
__global__ void __launch_bounds__(kNaChunk) na_count_kernel(const int64_t* ids, int T, int K, int E,
                                                            int32_t* scratch) {
  extern __shared__ __align__(16) uint32_t smem[];
  uint32_t* mask = smem;                                             // [8][E]
  uint16_t* wbase = reinterpret_cast<uint16_t*>(smem + kNaWarps * E);  // [8][E]
  unsigned long long* err = reinterpret_cast<unsigned long long*>(scratch);
  int32_t* counts = scratch + kNaCountsOff;
  int32_t* ranks = scratch + kNaRanksOff;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = blockIdx.x;
  const int t = g * kNaChunk + threadIdx.x;
  const bool live = t < T;

  for (int i = threadIdx.x; i < kNaWarps * E; i += blockDim.x) mask[i] = 0u;
  __syncthreads();
  uint32_t valid = 0u;
  const int64_t* tid = ids + (int64_t)t * K;
  if (live) {
    for (int k = 0; k < K; ++k) {
      const int64_t id = tid[k];
      if (id == -1) continue;
      if (id < -1 || id >= E) {
        atomicMin(err, na_error_key(t, k, kNaErrRange));
        continue;
      }
      const uint32_t old = atomicOr(mask + warp * E + (int)id, 1u << lane);
      if (old & (1u << lane)) {
        atomicMin(err, na_error_key(t, k, kNaErrDup));
        continue;
      }
      valid |= 1u << k;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < kNaWarps; ++w) {
      wbase[w * E + e] = (uint16_t)run;
      run += __popc(mask[w * E + e]);
    }
    counts[g * E + e] = run;
  }
  __syncthreads();
  if (live) {
    const uint32_t before = (1u << lane) - 1u;
    for (int k = 0; k < K; ++k) {
      int code = -1;
      if ((valid >> k) & 1u) {
        const int e = (int)tid[k];
        code = (e << 8) | (wbase[warp * E + e] + __popc(mask[warp * E + e] & before));
      }
      ranks[t * K + k] = code;
    }
  }
}

// One block: chunk prefixes per expert, the aligned scan per worker (ends),
// every route's row, and the error report.
__global__ void __launch_bounds__(1024) na_finish_kernel(int T, int K, int E, int F, int alpha,
                                                         int32_t* scratch, int32_t* ends,
                                                         int32_t* slots, int32_t* error) {
  __shared__ int32_t sh_total[kNaMaxExperts];
  __shared__ int32_t sh_start[kNaMaxExperts];
  int32_t* counts = scratch + kNaCountsOff;
  const int32_t* ranks = scratch + kNaRanksOff;
  const int G = (T + kNaChunk - 1) / kNaChunk;
  const int Ef = E / F;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;

  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int g = 0; g < G; ++g) {
      const int c = counts[g * E + e];
      counts[g * E + e] = run;
      run += c;
    }
    sh_total[e] = run;
  }
  __syncthreads();
  for (int f = warp; f < F; f += nwarps) {
    int carry = 0;
    for (int l0 = 0; l0 < Ef; l0 += 32) {
      const int l = l0 + lane;
      const int e = f * Ef + l;
      const int cnt = l < Ef ? sh_total[e] : 0;
      const int al = afd::align_up_dev(cnt, alpha);
      const int incl = afd::warp_inclusive_scan(al);
      if (l < Ef) {
        sh_start[e] = carry + incl - al;
        ends[e] = carry + incl - al + cnt;
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < T * K; i += blockDim.x) {
    const int code = ranks[i];
    if (code < 0) {
      slots[i] = -1;
    } else {
      const int e = code >> 8;
      const int g = (i / K) / kNaChunk;
      slots[i] = sh_start[e] + counts[g * E + e] + (code & 0xff);
    }
  }
  if (threadIdx.x == 0) {
    const unsigned long long key = *reinterpret_cast<unsigned long long*>(scratch);
    const bool none = key == kNaNoError;
    error[0] = none ? AFD_OK : (int32_t)(key & 0xff);
    error[1] = none ? -1 : (int32_t)(key >> 16);
    error[2] = none ? -1 : (int32_t)((key >> 8) & 0xff);
  }
}

std::mutex g_setup_mu;
int32_t* g_scratch_ptr[kNaMaxDevices];

// Device address of the scratch array on the current device (looked up once
// per device).
afd_status scratch_for_current_device(int32_t** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNaMaxDevices) return AFD_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_layout_scratch) != cudaSuccess || !p) return AFD_ERR_CUDA;
    if (cudaFuncSetAttribute(na_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kNaWarps * kNaMaxExperts * 6) != cudaSuccess)
      return AFD_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  return AFD_OK;
}

// The address a kernel on the current device uses for a caller buffer: the
// buffer itself in that device's memory or in managed memory, the mapped
// device address of page-locked host memory. Pageable host memory, and
// memory of another device, are refused before anything is enqueued.
template <typename T>
bool device_view(T* p, T** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  cudaPointerAttributes a = {};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if ((a.type == cudaMemoryTypeDevice && a.device == dev) || a.type == cudaMemoryTypeManaged) {
    *out = p;
    return true;
  }
  if (a.type == cudaMemoryTypeHost && a.devicePointer) {
    *out = static_cast<T*>(a.devicePointer);
    return true;
  }
  return false;
}

}  // namespace

extern "C" AFD_API afd_status afd_route_layout_noalloc(const int64_t* ids, int32_t num_tokens,
                                                       int32_t top_k, int32_t num_experts,
                                                       int32_t num_workers, int32_t expert_alignment,
                                                       int32_t* ends, int32_t* slots, int32_t* error,
                                                       afd_stream stream_) {
  const int T = num_tokens, K = top_k, E = num_experts, F = num_workers;
  if (!ends || !error || (T > 0 && (!ids || !slots))) return AFD_ERR_ARG;
  if (T < 0 || K < 1 || E < 1 || F < 1 || expert_alignment < 1 || K > E || E % F != 0)
    return AFD_ERR_ARG;
  if (T > kNaMaxTokens || K > kNaMaxTopK || E > kNaMaxExperts || (int64_t)T * K > kNaMaxRoutes)
    return AFD_ERR_UNSUPPORTED;
  // Every row index inside a worker, and every intermediate sum of the
  // aligned scan, is at most align_up(T*K + (E/F)*(alpha-1), alpha); it must
  // fit the int32 arithmetic of the kernels.
  {
    const int64_t a = expert_alignment;
    const int64_t bound = ((int64_t)T * K + (int64_t)(E / F) * (a - 1) + a - 1) / a * a;
    if (bound > INT32_MAX) return AFD_ERR_UNSUPPORTED;
  }
  if ((T > 0 && (!device_view(ids, &ids) || !device_view(slots, &slots))) || !device_view(ends, &ends) ||
      !device_view(error, &error))
    return AFD_ERR_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int32_t* scratch = nullptr;
  afd_status st = scratch_for_current_device(&scratch);
  if (st != AFD_OK) return st;

  // The error key must start at "none" on every call; counts and ranks are
  // overwritten in full. Each step's own return code decides the status, so
  // an error left pending by unrelated earlier work is neither reported here
  // nor taken from its owner.
  if (cudaMemsetAsync(scratch, 0xff, sizeof(unsigned long long), stream) != cudaSuccess)
    return AFD_ERR_CUDA;
  const int G = (T + kNaChunk - 1) / kNaChunk;
  if (G > 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(kNaChunk);
    cfg.dynamicSmemBytes = (size_t)kNaWarps * E * 6;
    cfg.stream = stream;
    if (cudaLaunchKernelEx(&cfg, na_count_kernel, ids, T, K, E, scratch) != cudaSuccess) return AFD_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(1024);
  cfg.stream = stream;
  if (cudaLaunchKernelEx(&cfg, na_finish_kernel, T, K, E, F, (int)expert_alignment, scratch, ends, slots,
                         error) != cudaSuccess)
    return AFD_ERR_CUDA;
  return AFD_OK;
}
