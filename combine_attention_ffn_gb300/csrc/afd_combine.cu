// Combine kernels: gather each token's reply rows and sum them with the
// routing weights.
//
// What it computes follows the afdEP-comm "API contract" (source_collect:
// BF16 [T,H] summed over the selected experts in the source's token order,
// each routing weight applied once) and the design page's "19. FP8 combine
// replies" (FP32 sum in slot order, one rounding to BF16). Every element is
//   acc = +0.0f;  for k = 0..K-1 with a valid route: acc = fma(w_k, reply_k, acc)
//   out = bf16_round_nearest_even(acc)
// so the result does not depend on the launch shape.
//
// Two kernels compute it:
//  * combine_token_kernel (K <= 8, at least 4 tokens per SM): a warp per
//    token walks the row in 512-byte segments with a two-stage register
//    pipeline (the next segment's loads, one per route, are in flight while
//    the current one is summed and stored).
//  * combine_kernel<U> (fewer tokens, or K > 8): work items are (token,
//    segment), a segment being U x 32 consecutive 16-byte slices of the row;
//    a warp issues the loads of up to 8 routes at once, then their FMAs in
//    ascending k. Splitting a token's row into segments spreads a few tokens
//    over many warps ("R2" of the afdEP-comm design page spreads few-token
//    combines the same way).
// The two-stage modes (design page section 19) use the same two kernels
// with per-worker partials (combine_two_stage_kernel is the segmented one).

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "afd.h"
#include "afd_device.cuh"
#include "afd_internal.cuh"

namespace afd {

#if AFD_PHASE_TIMERS
// [0: a combine that waits first, 1: an early-started combine][block][point]
__device__ unsigned long long g_combine_stamps[2][kStampBlocks][kStampPoints];

cudaError_t read_combine_stamps(unsigned long long* host, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(host, g_combine_stamps, sizeof(g_combine_stamps));
  if (e == cudaSuccess && clear) {
    void* d = nullptr;
    e = cudaGetSymbolAddress(&d, g_combine_stamps);
    if (e == cudaSuccess) e = cudaMemset(d, 0, sizeof(g_combine_stamps));
  }
  return e;
}
#endif

namespace {

constexpr int kGroup = 8;  // routes whose loads are issued together

// Resident blocks per SM of combine_kernel<1> and <2> (set by configure_combine_kernels).
int g_seg1_blocks_per_sm = 0;
int g_seg2_blocks_per_sm = 0;

// Reply rows: 16-byte non-coherent loads that skip L1 allocation (the
// texture path streams this gather much faster than L2-only loads). Route
// receipts: L2-only loads.
//
// A combine launched right after the previous combine of the same exchange
// on the same stream (p.early != 0) needs no dependency wait to start: its
// launch implies that every block of that combine has passed its own wait
// (it lets dependents launch only after it), so the scatter, the expert and
// everything before them have completed, and the replies stay unchanged for
// this kernel's whole lifetime, which is what non-coherent loads require. It
// waits at its end instead, so that it completes only after its predecessor
// (what comes after it in the stream may rely on the whole exchange being
// done). Any other combine waits first and then lets dependents launch.
// An early start takes one of two forms (kEarlyFence, kEarlyL2):
//  * kEarlyFence: a device-scope acquire fence first, so that no line an
//    earlier kernel left in this SM's L1 is used, then the streaming loads;
//  * kEarlyL2 (launches of fewer tokens than the per-token kernel takes):
//    every reply and receipt load reads L2 only, which holds the completed
//    writes, so no fence is needed; at these sizes L2-only loads cost no
//    more than the streaming ones.
constexpr int kEarlyFence = 1, kEarlyL2 = 2;

__device__ __forceinline__ uint4 ld_l2(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}


// combine_kernel's reply loads: the same streaming loads with an L2
// evict-first policy (replies are read once). Measured with few tokens per
// launch: 2A2F round trip back to back T=1 10.3 -> 8.4 us, T=32 12.3 -> 10.9,
// T=512 22.6 -> 20.5 (evict_normal or evict_last policies measure the same;
// the per-token kernel, which streams far more bytes, and the segmented
// two-stage kernel are slower with them). kL2: L2-only loads with the same
// policy (the instantiation launched for an early start of kind kEarlyL2).
template <bool kL2>
__device__ __forceinline__ uint4 ld_reply_seg(const uint4* p) {
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  uint4 v;
  if (kL2)
    asm volatile("ld.global.cg.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
  else
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
  return v;
}

__device__ __forceinline__ void combine_begin(const CombineParams& p) {
  AFD_STAMP(g_combine_stamps, p.early ? 1 : 0, 0);
  if (!p.early) {
    pdl_wait();
  } else if (p.early == kEarlyFence) {
#if AFD_EARLY_FENCE
    // a device-scope acquire before the first load: no line an earlier
    // kernel left in this SM's L1 is used
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
#endif
  }
  pdl_launch_dependents();
  AFD_STAMP(g_combine_stamps, p.early ? 1 : 0, 1);
}
__device__ __forceinline__ void combine_end(const CombineParams& p) {
  AFD_STAMP(g_combine_stamps, p.early ? 1 : 0, 2);  // this block's sums are stored
  if (p.early) pdl_wait();
  AFD_STAMP(g_combine_stamps, p.early ? 1 : 0, 3);
}

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

template <int U, bool kL2>
__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ CombineParams p) {
  combine_begin(p);  // receipts and replies come from earlier kernels
  const int lane = threadIdx.x & 31;
  const int64_t gwarp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int K = p.K;
  const int nseg = (p.H >> 8) / U;  // 32 lanes x 8 BF16 = 256 elements per slice step
  const int64_t items = (int64_t)p.total_tokens * nseg;

  for (int64_t it = gwarp; it < items; it += nwarps) {
    const int gt = (int)(it / nseg);
    const int seg = (int)(it - (int64_t)gt * nseg);
    const int s = source_of(p, gt);
    const int t = gt - p.tok_off[s];
    int2 r = make_int2(-1, 0);
    if (lane < K) r = __ldcg(p.routes[s] + (int64_t)t * K + lane);
    const int v0 = seg * 32 * U + lane;

    float acc[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[u][i] = 0.0f;

    for (int k0 = 0; k0 < K; k0 += kGroup) {
      uint4 buf[kGroup][U];
      float wk[kGroup];
      bool ok[kGroup];
#pragma unroll
      for (int j = 0; j < kGroup; ++j) {
        const int k = k0 + j;
        const int c = __shfl_sync(0xffffffffu, r.x, k & 31);
        wk[j] = __int_as_float(__shfl_sync(0xffffffffu, r.y, k & 31));
        ok[j] = (k < K) && (c >= 0);
        if (ok[j]) {
          const uint4* row = reinterpret_cast<const uint4*>(
              p.reply[c >> kWorkerShift] + (int64_t)(c & kRowMask) * p.H);
#pragma unroll
          for (int u = 0; u < U; ++u) buf[j][u] = ld_reply_seg<kL2>(row + v0 + u * 32);
        }
      }
#pragma unroll
      for (int j = 0; j < kGroup; ++j) {
        if (!ok[j]) continue;
#pragma unroll
        for (int u = 0; u < U; ++u) fma8(acc[u], wk[j], buf[j][u]);
      }
    }

    uint4* out_row = reinterpret_cast<uint4*>(p.out[s] + (int64_t)t * p.out_stride[s]);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      uint4 o;
      o.x = pack_bf16x2(acc[u][0], acc[u][1]);
      o.y = pack_bf16x2(acc[u][2], acc[u][3]);
      o.z = pack_bf16x2(acc[u][4], acc[u][5]);
      o.w = pack_bf16x2(acc[u][6], acc[u][7]);
      out_row[v0 + u * 32] = o;
    }
  }
  combine_end(p);
}

// ---- two-stage combine (optionally with E4M3 partials) ----

// Rounds a and b to BF16 (nearest even) with one paired conversion.
__device__ __forceinline__ void bf16_round2(float& a, float& b) {
  const uint32_t u = pack_bf16x2(a, b);
  a = __uint_as_float(u << 16);
  b = __uint_as_float(u & 0xffff0000u);
}

// 2^e as an FP32 value (e in [-126, 127]).
__device__ __forceinline__ float exp2_int(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

// The smallest integer e >= -117 with amax <= 448 * 2^e, from amax's FP32
// bits: amax = (1 + m) * 2^E fits under 1.75 * 2^(E) exactly when m <= 0.75.
// An infinite amax gives 120; zero or subnormal amax gives -117.
__device__ __forceinline__ int group_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int E = (int)((b >> 23) & 0xffu);
  if (E == 0) return -117;
  int e = (E - 127) - 8 + ((b & 0x7fffffu) > 0x600000u ? 1 : 0);
  return e < -117 ? -117 : e;
}

// Rounds v to E4M3 (nearest even, saturating) and back, exactly as the
// conversion instructions do.
__device__ __forceinline__ void e4m3_round_trip2(float& a, float& b) {
  uint16_t q;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(q) : "f"(a), "f"(b));
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(q));
  const __half2 hv = *reinterpret_cast<const __half2*>(&h2);
  a = __high2float(hv);
  b = __low2float(hv);
}

// ---- per-token combine ----

// Large batches, K <= 8: a warp per token. The token's route codes are read
// once; the hidden row is then walked in 512-byte segments (one 16-byte
// slice per lane) with a two-stage register pipeline: the loads of segment
// i+1 (one per route) are in flight while segment i is summed and stored.
//
// The token's routes from its receipt entries (lane j < K holds route j):
// row pointers, weights and workers (-1 for a skipped route). Returns the
// valid routes as bits.
__device__ __forceinline__ uint32_t token_routes(const CombineParams& p, int2 r, const uint16_t* (&rowp)[kGroup],
                                                 float (&wk)[kGroup]) {
  uint32_t okmask = 0u;
#pragma unroll
  for (int j = 0; j < kGroup; ++j) {
    const int c = __shfl_sync(0xffffffffu, r.x, j);
    wk[j] = __int_as_float(__shfl_sync(0xffffffffu, r.y, j));
    const bool ok = (j < p.K) && (c >= 0);
    okmask |= (ok ? 1u : 0u) << j;
    rowp[j] = ok ? p.reply[c >> kWorkerShift] + (int64_t)(c & kRowMask) * p.H : p.reply[0];
  }
  return okmask;
}

// The two-stage modes take a token's routes in summation order instead:
// grouped by worker, the groups in the order of each worker's last route,
// ascending k inside a group (the order of the design page's section 19).
// Slot j gets route perm[j]; bit j of *bnd marks the last slot of a group.
// Lane k < K ranks its own route by key (last route of its worker) * 8 + k
// (skipped routes after all others), and a ballot per slot finds the lane
// that holds it.
__device__ __forceinline__ uint32_t token_routes_grouped(const CombineParams& p, int2 r,
                                                         const uint16_t* (&rowp)[kGroup], float (&wk)[kGroup],
                                                         uint32_t& bnd) {
  const int lane = threadIdx.x & 31;
  const int wf_me = (lane < p.K && r.x >= 0) ? (r.x >> kWorkerShift) : -1;
  int wf[kGroup];
#pragma unroll
  for (int j = 0; j < kGroup; ++j) wf[j] = __shfl_sync(0xffffffffu, wf_me, j);
  int last = lane;
#pragma unroll
  for (int j = 1; j < kGroup; ++j) last = (j > lane && wf[j] == wf_me) ? j : last;
  const int key_me = wf_me >= 0 ? last * kGroup + lane : kGroup * kGroup + lane;
  int rank = 0;
#pragma unroll
  for (int j = 0; j < kGroup; ++j) rank += __shfl_sync(0xffffffffu, key_me, j) < key_me ? 1 : 0;
  uint32_t okmask = 0u;
  int prev_wf = -1;
  bnd = 0u;
#pragma unroll
  for (int j = 0; j < kGroup; ++j) {
    const int src = __ffs(__ballot_sync(0xffffffffu, lane < kGroup && rank == j)) - 1;
    const int c = __shfl_sync(0xffffffffu, r.x, src);
    wk[j] = __int_as_float(__shfl_sync(0xffffffffu, r.y, src));
    const bool ok = (src < p.K) && (c >= 0);
    const int w = ok ? (c >> kWorkerShift) : -1;
    okmask |= (ok ? 1u : 0u) << j;
    rowp[j] = ok ? p.reply[w] + (int64_t)(c & kRowMask) * p.H : p.reply[0];
    // the slot before ends its group when this one belongs to another worker
    if (j > 0 && prev_wf >= 0 && w != prev_wf) bnd |= 1u << (j - 1);
    prev_wf = w;
  }
  if (prev_wf >= 0) bnd |= 1u << (kGroup - 1);
  return okmask;
}

// kL2: L2-only loads (an early start of kind kEarlyL2; segmented launches
// only), else the streaming loads.
template <bool kL2>
__device__ __forceinline__ void load_seg(uint4 (&buf)[kGroup], const uint16_t* const (&rowp)[kGroup],
                                         uint32_t okmask, int v) {
#pragma unroll
  for (int j = 0; j < kGroup; ++j)
    if ((okmask >> j) & 1u) {
      const uint4* a = reinterpret_cast<const uint4*>(rowp[j]) + v;
      buf[j] = kL2 ? ld_l2(a) : ld_once(a);
    }
}

// Sums one segment (this lane's 8 elements of every route) and stores it.
// AFD_COMBINE_FUSED: one FP32 chain over the routes in ascending k, one BF16
// rounding. Two-stage modes (design page, section 19): each worker's routes
// form a partial (FP32 chain in ascending k, rounded to BF16; in the FP8
// mode also scaled by its group's power of two, rounded to E4M3 and back);
// the partials are added in FP32 in the order of each worker's last route,
// then rounded to BF16 once.
template <int kMode>
__device__ __forceinline__ void sum_seg(uint4* out_row, const uint4 (&buf)[kGroup], const float (&wk)[kGroup],
                                        uint32_t bnd, uint32_t okmask, int v) {
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  if (kMode == AFD_COMBINE_FUSED) {
#pragma unroll
    for (int j = 0; j < kGroup; ++j)
      if ((okmask >> j) & 1u) fma8(acc, wk[j], buf[j]);
  } else {
    // slots in summation order (token_routes_grouped): one worker's partial
    // is an FP32 chain over its run of slots, finished at the run's end
    float part[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) part[e] = 0.0f;
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      if ((okmask >> j) & 1u) fma8(part, wk[j], buf[j]);
      if (!((bnd >> j) & 1u)) continue;  // the same for the whole warp
#pragma unroll
      for (int e = 0; e < 8; e += 2) bf16_round2(part[e], part[e + 1]);
      if (kMode == AFD_COMBINE_TWO_STAGE_FP8) {
        // one power-of-two scale per 128 elements: 16 lanes x 8 elements
        float amax = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(part[e]));
#pragma unroll
        for (int d = 1; d < 16; d <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
        const int ge = group_exponent(amax);
        const float down = exp2_int(-ge), up = exp2_int(ge);
        // the decoded partial is an FP32 value of its own before the sum
        // (a group amax of 248 * 2^120 or more decodes to infinity), so the
        // product and the sum are rounded separately, never fused
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          float a = part[e] * down, b = part[e + 1] * down;
          e4m3_round_trip2(a, b);
          acc[e] = __fadd_rn(acc[e], __fmul_rn(a, up));
          acc[e + 1] = __fadd_rn(acc[e + 1], __fmul_rn(b, up));
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = acc[e] + part[e];
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) part[e] = 0.0f;
    }
  }
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  out_row[v] = o;
}

template <int kMode>
__global__ void __launch_bounds__(64, kMode == AFD_COMBINE_FUSED               ? 0
                                     : kMode == AFD_COMBINE_TWO_STAGE_FP8 ? AFD_TWO_STAGE_FP8_BLOCKS
                                                                          : AFD_TWO_STAGE_BLOCKS)
    combine_token_kernel(const __grid_constant__ CombineParams p) {
  combine_begin(p);
  const int lane = threadIdx.x & 31;
  const int gwarp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const int K = p.K;
  // a warp takes 1/split of a token's segments (split divides the count)
  const int nseg_all = p.H >> 8;
  const int split = nseg_all % AFD_COMBINE_SPLIT == 0 ? AFD_COMBINE_SPLIT : 1;
  const int nseg = nseg_all / split;
  const int items = p.total_tokens * split;

  for (int item = gwarp; item < items; item += nwarps) {
    const int gt = item / split;
    const int seg0 = (item - gt * split) * nseg;
    const int s = source_of(p, gt);
    const int t = gt - p.tok_off[s];
    int2 r = make_int2(-1, 0);
    if (lane < K) r = __ldcg(p.routes[s] + (int64_t)t * K + lane);
    const uint16_t* rowp[kGroup];
    float wk[kGroup];
    uint32_t bnd = 0u;
    const uint32_t okmask = kMode == AFD_COMBINE_FUSED ? token_routes(p, r, rowp, wk)
                                                       : token_routes_grouped(p, r, rowp, wk, bnd);
    uint4* out_row = reinterpret_cast<uint4*>(p.out[s] + (int64_t)t * p.out_stride[s]) + seg0 * 32;
#pragma unroll
    for (int j = 0; j < kGroup; ++j) rowp[j] += seg0 * 256;
    uint4 a[kGroup], b[kGroup];
    load_seg<false>(a, rowp, okmask, lane);
    int seg = 0;
    for (; seg + 2 <= nseg; seg += 2) {
      load_seg<false>(b, rowp, okmask, (seg + 1) * 32 + lane);
      sum_seg<kMode>(out_row, a, wk, bnd, okmask, seg * 32 + lane);
      if (seg + 2 < nseg) load_seg<false>(a, rowp, okmask, (seg + 2) * 32 + lane);
      sum_seg<kMode>(out_row, b, wk, bnd, okmask, (seg + 1) * 32 + lane);
    }
    if (seg < nseg) sum_seg<kMode>(out_row, a, wk, bnd, okmask, seg * 32 + lane);
  }
  combine_end(p);
}

// Few tokens: a warp per (token, 512-byte segment), as combine_kernel<1>,
// with the two-stage rule.
template <int kMode, bool kL2>
__global__ void __launch_bounds__(256) combine_two_stage_kernel(const __grid_constant__ CombineParams p) {
  combine_begin(p);
  const int lane = threadIdx.x & 31;
  const int64_t gwarp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int K = p.K;  // <= kGroup
  const int nseg = p.H >> 8;
  const int64_t items = (int64_t)p.total_tokens * nseg;

  for (int64_t it = gwarp; it < items; it += nwarps) {
    const int gt = (int)(it / nseg);
    const int seg = (int)(it - (int64_t)gt * nseg);
    const int s = source_of(p, gt);
    const int t = gt - p.tok_off[s];
    int2 r = make_int2(-1, 0);
    if (lane < K) r = __ldcg(p.routes[s] + (int64_t)t * K + lane);
    const uint16_t* rowp[kGroup];
    float wk[kGroup];
    uint32_t bnd = 0u;
    const uint32_t okmask = kMode == AFD_COMBINE_FUSED ? token_routes(p, r, rowp, wk)
                                                       : token_routes_grouped(p, r, rowp, wk, bnd);
    uint4 buf[kGroup];
    load_seg<kL2>(buf, rowp, okmask, seg * 32 + lane);
    sum_seg<kMode>(reinterpret_cast<uint4*>(p.out[s] + (int64_t)t * p.out_stride[s]), buf, wk, bnd,
                   okmask, seg * 32 + lane);
  }
  combine_end(p);
}

template <typename Kernel, typename Params>
cudaError_t launch_pdl(Kernel kernel, int64_t grid, int block, cudaStream_t stream, const Params& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(block);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace

// Both kernels start as programmatic dependents of the previous kernel on the
// stream and wait for it before reading anything.
cudaError_t launch_combine(const CombineParams& p_in, int sm_cap, cudaStream_t stream) {
  if (p_in.total_tokens <= 0) return cudaSuccess;
  CombineParams p = p_in;
  const bool small = p.total_tokens < sm_cap * AFD_TOKEN_COMBINE_MIN;
  if (p.early) p.early = small ? kEarlyL2 : kEarlyFence;
  if (p.K <= kGroup && !small) {
    // enough tokens for a warp each on every SM: the pipelined per-token
    // kernel, in two-warp blocks so that tokens spread evenly over the SMs
    int64_t grid = ((int64_t)p.total_tokens * AFD_COMBINE_SPLIT + 1) / 2;
    if (grid > (int64_t)sm_cap * 8) grid = (int64_t)sm_cap * 8;
    switch (p.mode) {
      case AFD_COMBINE_TWO_STAGE: return launch_pdl(combine_token_kernel<AFD_COMBINE_TWO_STAGE>, grid, 64, stream, p);
      case AFD_COMBINE_TWO_STAGE_FP8:
        return launch_pdl(combine_token_kernel<AFD_COMBINE_TWO_STAGE_FP8>, grid, 64, stream, p);
      default: return launch_pdl(combine_token_kernel<AFD_COMBINE_FUSED>, grid, 64, stream, p);
    }
  }
  const bool l2 = p.early == kEarlyL2;
  if (p.mode != AFD_COMBINE_FUSED) {
    const int64_t items = (int64_t)p.total_tokens * (p.H >> 8);
    int64_t grid = (items + 7) / 8;
    if (grid > (int64_t)sm_cap * 8) grid = (int64_t)sm_cap * 8;
    if (p.mode == AFD_COMBINE_TWO_STAGE_FP8)
      return l2 ? launch_pdl(combine_two_stage_kernel<AFD_COMBINE_TWO_STAGE_FP8, true>, grid, 256, stream, p)
                : launch_pdl(combine_two_stage_kernel<AFD_COMBINE_TWO_STAGE_FP8, false>, grid, 256, stream, p);
    return l2 ? launch_pdl(combine_two_stage_kernel<AFD_COMBINE_TWO_STAGE, true>, grid, 256, stream, p)
              : launch_pdl(combine_two_stage_kernel<AFD_COMBINE_TWO_STAGE, false>, grid, 256, stream, p);
  }
  const int64_t slices = (int64_t)p.total_tokens * (p.H >> 8);
  // Two slices per item when one slice per warp would need more warps than
  // the SMs hold at once: every warp then still has exactly one item, in a
  // single wave, instead of a second wave paying the whole latency again.
  const int64_t resident1 = (int64_t)sm_cap * (g_seg1_blocks_per_sm > 0 ? g_seg1_blocks_per_sm : 1) * 8;
  const bool wide = (p.H % 512 == 0) && slices > resident1;
  if (AFD_COMBINE_SHARE && p.share > 1 && p.H % 512 == 0) {
    // One combine per source, each started while the one before it runs
    // (early start). When their blocks could not all be resident at once,
    // every launch gets an equal share of the SMs instead (two slices per
    // item, a few items per warp), so that they run side by side rather than
    // each waiting for the previous one's blocks to leave.
    const int64_t need = ((wide ? slices / 2 : slices) + 7) / 8;
    const int bps0 = wide ? g_seg2_blocks_per_sm : g_seg1_blocks_per_sm;
    if (need * p.share > (int64_t)sm_cap * (bps0 > 0 ? bps0 : 1)) {
      int64_t grid = (int64_t)sm_cap * (g_seg2_blocks_per_sm > 0 ? g_seg2_blocks_per_sm : 1) / p.share;
      const int64_t need2 = (slices / 2 + 7) / 8;
      if (grid > need2) grid = need2;
      if (grid < 1) grid = 1;
      return l2 ? launch_pdl(combine_kernel<2, true>, grid, 256, stream, p)
                : launch_pdl(combine_kernel<2, false>, grid, 256, stream, p);
    }
  }
  const int64_t cap = (int64_t)sm_cap * 8;  // blocks of 8 warps
  const int64_t items = wide ? slices / 2 : slices;
  int64_t grid = (items + 7) / 8;
  if (grid > cap) grid = cap;
  if (wide)
    return l2 ? launch_pdl(combine_kernel<2, true>, grid, 256, stream, p)
              : launch_pdl(combine_kernel<2, false>, grid, 256, stream, p);
  return l2 ? launch_pdl(combine_kernel<1, true>, grid, 256, stream, p)
            : launch_pdl(combine_kernel<1, false>, grid, 256, stream, p);
}

cudaError_t configure_combine_kernels() {
  cudaError_t e = cudaSuccess;
  for (const void* k : {(const void*)combine_token_kernel<AFD_COMBINE_FUSED>,
                        (const void*)combine_token_kernel<AFD_COMBINE_TWO_STAGE>,
                        (const void*)combine_token_kernel<AFD_COMBINE_TWO_STAGE_FP8>,
                        (const void*)combine_kernel<1, false>, (const void*)combine_kernel<2, false>,
                        (const void*)combine_kernel<1, true>, (const void*)combine_kernel<2, true>,
                        (const void*)combine_two_stage_kernel<AFD_COMBINE_TWO_STAGE, false>,
                        (const void*)combine_two_stage_kernel<AFD_COMBINE_TWO_STAGE_FP8, false>,
                        (const void*)combine_two_stage_kernel<AFD_COMBINE_TWO_STAGE, true>,
                        (const void*)combine_two_stage_kernel<AFD_COMBINE_TWO_STAGE_FP8, true>})
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, kSharedCarveout);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g_seg1_blocks_per_sm, combine_kernel<1, false>, 256, 0);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g_seg2_blocks_per_sm, combine_kernel<2, false>, 256, 0);
  return e;
}

}  // namespace afd
