// Internal declarations shared by the libafd translation units: launch
// parameter blocks and the kernel launchers. Not part of the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace afd {

constexpr int kMaxSources = 64;
constexpr int kMaxWorkers = 64;
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kChunk = 256;          // tokens counted per pass = threads per layout block
constexpr int kChunkWarps = kChunk / 32;
constexpr int kWorkerShift = 24;     // receipt route code = (worker << 24) | row
constexpr int32_t kRowMask = (1 << kWorkerShift) - 1;
constexpr int kLayoutMaxCtas = 16;   // largest layout cluster
constexpr int kRankBits = 8;         // one-kernel dispatch code = (expert << 8) | rank in chunk
#ifndef AFD_SMALL_ROUTES
#define AFD_SMALL_ROUTES 2048         // exchanges up to this many routes take the one-kernel dispatch
#endif
constexpr int kSmallRoutes = AFD_SMALL_ROUTES;
constexpr int kSmallSmemMax = 110 * 1024;
// Launch-shape constants. They only change speed, never results; a build may
// override them (-D...) to compare shapes.
#ifndef AFD_SCATTER_BLOCK
#define AFD_SCATTER_BLOCK 128    // threads per scatter block (a warp per token)
#endif
#ifndef AFD_TINY_MIN_BLOCKS
#define AFD_TINY_MIN_BLOCKS 128   // the one-warp dispatch runs min(E, this) blocks at least (they share the padding rows)
#endif
#ifndef AFD_TINY_DISPATCH
#define AFD_TINY_DISPATCH 1       // exchanges of at most 32 tokens take the one-warp dispatch
#endif
#ifndef AFD_COMBINE_SPLIT
#define AFD_COMBINE_SPLIT 1       // warps per token in the per-token combine
#endif
#ifndef AFD_TWO_STAGE_BLOCKS
#define AFD_TWO_STAGE_BLOCKS 7    // resident two-warp blocks per SM asked of the two-stage per-token combine
#endif
#ifndef AFD_TWO_STAGE_FP8_BLOCKS
#define AFD_TWO_STAGE_FP8_BLOCKS 8  // the same, with E4M3 partials
#endif
#ifndef AFD_EARLY_FENCE
#define AFD_EARLY_FENCE 1         // an early-started per-token combine begins with a device-scope acquire fence
#endif
#ifndef AFD_COMBINE_EARLY
#define AFD_COMBINE_EARLY 1       // a combine right after another one of the same exchange starts at once
#endif
#ifndef AFD_COMBINE_SHARE
#define AFD_COMBINE_SHARE 1       // per-source segmented combines take an equal share of the SMs
#endif
#ifndef AFD_TOKEN_COMBINE_MIN
#define AFD_TOKEN_COMBINE_MIN 4  // x SMs: tokens from which the per-token combine is used
#endif
static_assert(kChunk <= (1 << kRankBits), "rank in chunk must fit its field");

// Every kernel of the library asks for the same split of each SM's unified
// L1 / shared memory. The kernels of one exchange overlap on the same SMs
// through programmatic dependent launch; when their preferred splits differ
// (the layout needs tens of KB of shared memory, the combines none), an
// SM cannot take blocks of the next kernel until it has drained and changed
// its split, which cost up to 6 us per round trip.
constexpr int kSharedCarveout = 50;  // percent of the maximum shared memory

constexpr int kErrRange = 5;    // AFD_ERR_ROUTE_RANGE
constexpr int kErrDup = 6;      // AFD_ERR_ROUTE_DUP
constexpr int kErrTimeout = 11; // AFD_ERR_TIMEOUT
constexpr int kDefaultWaitPolls = 1 << 22;  // see afd_set_wait_limit
// Rows up to this many bytes take the bulk-copy scatter (two row buffers per
// two-warp block: 33 KB of shared memory at the limit, under the 48 KB a
// launch gets without opting in). 2A2F round trip at T=2048: H7168 172.1 ->
// 163.8 us and H8192 196.2 -> 186.5 us against the register scatter.
constexpr int kBulkRowMax = 16384;
constexpr unsigned long long kNoError = ~0ull;

// The sticky route error: the smallest key wins, so the reported route is the
// first in (source, token, k) order. key = s << 56 | t << 16 | k << 8 | code.
__host__ __device__ inline unsigned long long route_error_key(int s, int t, int k, int code) {
  return ((unsigned long long)s << 56) | ((unsigned long long)(uint32_t)t << 16) |
         ((unsigned long long)k << 8) | (unsigned long long)code;
}

struct SourceDesc {
  const uint8_t* x;      // [T][row_bytes]
  const int64_t* ids;    // [T][K]
  const float* w;        // [T][K]
  const float* scale;    // FP8: scale(t, b) = scale[t * sst + b * ssb]
  int64_t sst, ssb;
  int32_t T;             // live tokens
  int32_t tok_off;       // first flattened token of this source
  int32_t x_device;      // x is device memory (not host memory mapped for the device)
  int32_t pad_;
};

// Everything the layout and scatter kernels of one exchange read or write.
struct DispatchParams {
  SourceDesc src[kMaxSources];
  int32_t A, F, E, Ef, K, alpha, bucket;
  int32_t row_bytes;     // 2H (BF16) or H (FP8)
  int32_t nscale;        // H / 128 for FP8, else 0
  int32_t total_tokens;  // sum of T
  int32_t layout_ctas;   // CTAs of the layout cluster (large path)
  int32_t x_device;      // 1 when every source's rows are in device memory (bulk copies allowed)
  int32_t wait_polls;    // polls of a bulk row load before the scatter gives up (AFD_ERR_TIMEOUT)
  int64_t R_arena;       // rows per worker arena
  // context scratch
  int32_t* route_tmp;    // [total_tokens][K]: the layout's route codes, (worker << 24) | row, or -1
  unsigned long long* err;
  // context outputs
  int32_t* starts;       // [E] aligned start of each expert (worker-local rows)
  int32_t* ends;         // [E] ends[] (worker-local)
  int32_t* hcounts;      // [E] aligned counts
  int2* routes;          // receipt [total_tokens][K]: {code, weight bits}
  int32_t* row_src;      // [F][R_arena]
  float* row_w;          // [F][R_arena]
  uint8_t* rows;         // [F][R_arena][row_bytes]
  float* row_scales;     // [F][R_arena][nscale]
};

struct CombineParams {
  const int2* routes[kMaxSources];   // receipt rows of each source, [T][K]
  uint16_t* out[kMaxSources];        // BF16 [T][out_stride]
  int64_t out_stride[kMaxSources];   // elements
  int32_t tok_off[kMaxSources];      // first flattened token of each source in this launch
  const uint16_t* reply[kMaxWorkers];// BF16 [rows][H] per worker
  int32_t A, K, H, total_tokens;
  int32_t mode;                      // AFD_COMBINE_*
  int32_t early;                     // nonzero: the previous kernel on the stream is a combine of
                                     // the same exchange (start at once, wait for it at the end;
                                     // launch_combine picks the form, afd_combine.cu)
  int32_t share;                     // combines of this exchange expected to run side by side
                                     // (one per source when each source collects on its own)
};


// Launchers (return the launch's cudaError_t).
bool dispatch_is_small(const DispatchParams& p);
int layout_ctas_for(int total_tokens, int sm_cap, int max_ctas);
cudaError_t launch_dispatch(const DispatchParams& p, int sm_cap, cudaStream_t stream);
cudaError_t launch_cached_scatter(const DispatchParams& p, int sm_cap, cudaStream_t stream);
cudaError_t launch_combine(const CombineParams& p, int sm_cap, cudaStream_t stream);
cudaError_t configure_dispatch_kernels(int* max_ctas);
// afd_l2_flush: writes vecs 16-byte vectors at `scratch`, then reads the next
// vecs, both with an L2 evict-last policy.
cudaError_t launch_l2_flush(uint4* scratch, int64_t vecs, cudaStream_t stream);
#ifndef AFD_PHASE_TIMERS
#define AFD_PHASE_TIMERS 0  // 1: the diagnostic build with %globaltimer stamps (afd_device.cuh)
#endif
constexpr int kStampKinds = 4;     // first dispatch kernel, scatter, waiting combine, early combine
constexpr int kStampBlocks = 4096;  // blocks recorded per kind
constexpr int kStampPoints = 8;     // points recorded per block
#if AFD_PHASE_TIMERS
// Phase-timer builds: copy out (and optionally zero) each translation unit's
// stamps, [2][kStampBlocks][kStampPoints] each.
cudaError_t read_dispatch_stamps(unsigned long long* host, bool clear);
cudaError_t read_combine_stamps(unsigned long long* host, bool clear);
#endif
cudaError_t configure_combine_kernels();

}  // namespace afd
