// Device helpers shared by the library's kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "afd_internal.cuh"

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

// Phase timers (diagnostic builds only: -DAFD_PHASE_TIMERS=1). Thread 0 of
// each block records %globaltimer (ns) at numbered points of its kernel; the
// translation unit holding the kernel keeps the stamps in a device array
// [kind][block][point] that afd_phase_stamps copies out. Kinds: 0 the first
// dispatch kernel (layout, one-kernel or one-warp dispatch), 1 the scatter,
// 2 a combine that waits first, 3 an early-started combine (later launches of
// a kind overwrite earlier ones). Blocks past kStampBlocks are not recorded.
// In the default build every macro is empty and no array exists.
__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

#if AFD_PHASE_TIMERS
// A stamp stored at once (kernels whose later fences do not wait on it).
#define AFD_STAMP(arr, kind, point)                                                  \
  do {                                                                               \
    if (threadIdx.x == 0 && blockIdx.x < ::afd::kStampBlocks)                        \
      arr[kind][blockIdx.x][point] = ::afd::global_timer_ns();                       \
  } while (0)
// Stamps kept in registers and stored at the kernel's end (the layout, whose
// cluster barriers release every earlier store of the thread).
#define AFD_STAMP_REGS unsigned long long afd_ts_[::afd::kStampPoints] = {}
#define AFD_STAMP_REG(point)                                        \
  do {                                                              \
    if (threadIdx.x == 0) afd_ts_[point] = ::afd::global_timer_ns(); \
  } while (0)
#define AFD_STAMP_REGS_STORE(arr, kind)                                              \
  do {                                                                               \
    if (threadIdx.x == 0 && blockIdx.x < ::afd::kStampBlocks)                        \
      for (int i_ = 0; i_ < ::afd::kStampPoints; ++i_) arr[kind][blockIdx.x][i_] = afd_ts_[i_]; \
  } while (0)
#else
#define AFD_STAMP(arr, kind, point) \
  do {                              \
  } while (0)
#define AFD_STAMP_REGS \
  do {                 \
  } while (0)
#define AFD_STAMP_REG(point) \
  do {                       \
  } while (0)
#define AFD_STAMP_REGS_STORE(arr, kind) \
  do {                                  \
  } while (0)
#endif

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
