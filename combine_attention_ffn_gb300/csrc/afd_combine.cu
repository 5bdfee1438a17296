// Combine kernel: gathers each token's reply rows and sums them with the
// routing weights, and the collect copy kernel.
//
// What it computes follows the afdEP-comm "API contract" (source_collect:
// BF16 [T,H] summed over the selected experts in original token order, the
// routing weight applied exactly once) and the design page's "19. FP8 combine
// replies" (FP32 sum in slot order, one rounding to BF16). Every element is
//   acc = +0.0f;  for k = 0..K-1 with a valid route: acc = fma(w_k, reply_k, acc)
//   out = bf16_round_nearest_even(acc)
// so the result does not depend on the launch shape.
//
// Shape: a warp per token. Each lane owns 16-byte slices (8 BF16) of the
// hidden row; for a group of up to 8 routes it issues all the slice loads
// first and then the FMAs in ascending k, so up to 8 x kCombineVecs loads per
// lane are in flight ("10. Single-FFN reduction" of the design page: the
// reduction over the top-k rows is branch-free across the slices of a row).

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "afd_internal.cuh"

namespace afd {
namespace {

constexpr int kCombineVecs = 2;   // 16-byte slices per lane per step
constexpr int kGroup = 8;         // routes whose loads are issued together

__device__ __forceinline__ int source_of(const CombineParams& p, int gt) {
  int s = 0;
  while (s + 1 < p.A && gt >= p.tok_off[s + 1]) ++s;
  return s;
}

__device__ __forceinline__ void fma8(float (&acc)[8], float w, const uint4& v) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] = __fmaf_rn(w, __uint_as_float(u[i] << 16), acc[2 * i]);
    acc[2 * i + 1] = __fmaf_rn(w, __uint_as_float(u[i] & 0xffff0000u), acc[2 * i + 1]);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}

__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ CombineParams p) {
  const int lane = threadIdx.x & 31;
  const int gwarp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const int K = p.K;
  const int nvec = p.H >> 3;  // 8 BF16 per 16-byte slice

  for (int gt = gwarp; gt < p.total_tokens; gt += nwarps) {
    const int s = source_of(p, gt);
    const int t = gt - p.tok_off[s];
    int2 r = make_int2(-1, 0);
    if (lane < K) r = p.routes[s][(int64_t)t * K + lane];
    uint4* out_row = reinterpret_cast<uint4*>(p.out[s] + (int64_t)t * p.out_stride[s]);

    for (int v0 = 0; v0 < nvec; v0 += 32 * kCombineVecs) {
      float acc[kCombineVecs][8];
#pragma unroll
      for (int u = 0; u < kCombineVecs; ++u)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[u][i] = 0.0f;

      for (int k0 = 0; k0 < K; k0 += kGroup) {
        uint4 buf[kGroup][kCombineVecs];
        float wk[kGroup];
        bool ok[kGroup];
#pragma unroll
        for (int j = 0; j < kGroup; ++j) {
          const int k = k0 + j;
          const int c = __shfl_sync(0xffffffffu, r.x, k & 31);
          const float w = __int_as_float(__shfl_sync(0xffffffffu, r.y, k & 31));
          ok[j] = (k < K) && (c >= 0);
          wk[j] = w;
          if (ok[j]) {
            const uint4* row = reinterpret_cast<const uint4*>(
                p.reply[c >> kWorkerShift] + (int64_t)(c & kRowMask) * p.H);
#pragma unroll
            for (int u = 0; u < kCombineVecs; ++u) {
              const int v = v0 + u * 32 + lane;
              if (v < nvec) buf[j][u] = __ldg(row + v);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < kGroup; ++j) {
          if (!ok[j]) continue;
#pragma unroll
          for (int u = 0; u < kCombineVecs; ++u)
            if (v0 + u * 32 + lane < nvec) fma8(acc[u], wk[j], buf[j][u]);
        }
      }

#pragma unroll
      for (int u = 0; u < kCombineVecs; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < nvec) {
          uint4 o;
          o.x = pack_bf16x2(acc[u][0], acc[u][1]);
          o.y = pack_bf16x2(acc[u][2], acc[u][3]);
          o.z = pack_bf16x2(acc[u][4], acc[u][5]);
          o.w = pack_bf16x2(acc[u][6], acc[u][7]);
          out_row[v] = o;
        }
      }
    }
  }
}

__global__ void __launch_bounds__(256) copy_kernel(const __grid_constant__ CopyParams p) {
  const int nvec = p.H >> 3;
  const int64_t total = (int64_t)p.rows * nvec;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int64_t row = i / nvec;
    const int v = (int)(i % nvec);
    const uint4* src = reinterpret_cast<const uint4*>(p.src + row * p.src_stride);
    uint4* dst = reinterpret_cast<uint4*>(p.dst + row * p.dst_stride);
    dst[v] = __ldg(src + v);
  }
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, int sm_cap, cudaStream_t stream) {
  if (p.total_tokens <= 0) return cudaSuccess;
  int grid = (p.total_tokens + 7) / 8;
  const int cap = sm_cap * 8;
  if (grid > cap) grid = cap;
  combine_kernel<<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_copy(const CopyParams& p, int sm_cap, cudaStream_t stream) {
  const int64_t total = (int64_t)p.rows * (p.H >> 3);
  if (total <= 0) return cudaSuccess;
  int64_t grid = (total + 255) / 256;
  const int64_t cap = (int64_t)sm_cap * 8;
  if (grid > cap) grid = cap;
  copy_kernel<<<(int)grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace afd
