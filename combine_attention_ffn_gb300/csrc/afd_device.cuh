// Device helpers shared by the library's kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace afd {

// Programmatic dependent launch (sm_90+). A kernel launched with programmatic
// stream serialization may start while the previous kernel in the stream is
// still running; it must call pdl_wait() before touching anything that
// kernel writes. pdl_launch_dependents() lets the next kernel's blocks be
// scheduled early. Both are no-ops for a kernel launched normally.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 16-byte load of data read exactly once: skip L1.
__device__ __forceinline__ uint4 ld_once(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Rounds v up to a multiple of a (a >= 1); a power of two (the usual
// expert_alignment) takes a mask instead of a division.
__device__ __forceinline__ int align_up_dev(int v, int a) {
  return (a & (a - 1)) == 0 ? (v + a - 1) & -a : (v + a - 1) / a * a;
}

__device__ __forceinline__ int warp_inclusive_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += u;
  }
  return v;
}

}  // namespace afd
