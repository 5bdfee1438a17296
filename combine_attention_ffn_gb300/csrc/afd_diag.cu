// Diagnostics for benchmarks: an L2 flush that also evicts the lines the
// scatter writes with an evict-last policy (afd_l2_flush in afd.h). Not on
// the exchange's path.

#include <cuda_runtime.h>
#include <stdint.h>

#include "afd_internal.cuh"

namespace {

__device__ __forceinline__ uint64_t evict_last_policy() {
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__global__ void l2_flush_write_kernel(uint4* dst, int64_t n) {
  const uint64_t pol = evict_last_policy();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %1, %1, %1}, %2;" ::"l"(dst + i), "r"(0u), "l"(pol)
                 : "memory");
}

__global__ void l2_flush_read_kernel(const uint4* src, int64_t n, uint4* sink) {
  const uint64_t pol = evict_last_policy();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  uint32_t acc = 0;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    uint4 v;
    asm volatile("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(src + i), "l"(pol));
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  if (acc == 0xdeadbeefu) sink[0] = make_uint4(acc, acc, acc, acc);  // keeps the loads
}

// Drops the (clean) lines of the read pass from L2 without writing them back,
// so that the step after the flush finds no line at all of the flush there.
__global__ void l2_flush_discard_kernel(char* base, int64_t lines) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < lines; i += stride)
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(base + i * 128) : "memory");
}

}  // namespace

namespace afd {

cudaError_t launch_l2_flush(uint4* scratch, int64_t vecs, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int grid = sms * 4;
  l2_flush_write_kernel<<<grid, 256, 0, stream>>>(scratch, vecs);
  e = cudaPeekAtLastError();
  if (e != cudaSuccess) return e;
  l2_flush_read_kernel<<<grid, 256, 0, stream>>>(scratch + vecs, vecs, scratch);
  e = cudaPeekAtLastError();
  if (e != cudaSuccess) return e;
  // whole 128-byte lines of the read half (its start is 16-byte aligned)
  char* lo = reinterpret_cast<char*>(scratch + vecs);
  char* first = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(lo) + 127) & ~uintptr_t(127));
  const int64_t lines = ((lo + vecs * 16) - first) / 128;
  if (lines > 0) l2_flush_discard_kernel<<<grid, 256, 0, stream>>>(first, lines);
  return cudaPeekAtLastError();
}

}  // namespace afd
