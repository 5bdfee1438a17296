/*
 * afd.h -- MoE token dispatch and combine between Attention sources and FFN
 * expert workers, on one GPU (C ABI of libafd.so).
 *
 * The calls follow the afdEP-comm "API contract" page (sections "Roles and
 * tensors" and "Graphs, streams and lifetime"): source_dispatch,
 * worker_receive, worker_reply, source_collect. On one GPU the A sources and
 * F workers are logical partitions of the same HBM: nothing crosses a device
 * or process boundary, and a call's "rank" is an index argument.
 *
 * One exchange:
 *   1. afd_source_dispatch(s) for every source s (any order). The last one
 *      enqueues the layout and scatter kernels.
 *   2. afd_worker_receive(f) for every worker f: expert-major rows, their
 *      weights, the device prefix sums ends[] and an opaque receipt.
 *   3. the caller's expert computes BF16 replies, then afd_worker_reply(f)
 *      with the receipt, for every worker.
 *   4. afd_source_collect(s) for every source: BF16 [T,H] summed over the
 *      selected experts, in original token order.
 * A context holds at most one exchange in flight; the next dispatch waits
 * (host-side check) until every source has collected the previous one.
 *
 * Conventions for every call:
 *   - Device pointers are addresses on the context's device; host pointers
 *     are noted as such. Every array is dense row-major unless a stride says
 *     otherwise.
 *   - Wherever a buffer argument below says "device", the call also takes
 *     managed memory and page-locked host memory (cudaHostAlloc /
 *     cudaHostRegister; the kernels then read or write it over the host link
 *     through its mapped device address, with no copy). Pageable host memory,
 *     memory of another device and pointers CUDA does not know are refused
 *     with AFD_ERR_ARG before anything is enqueued.
 *   - `stream` is a cudaStream_t of the context's device (NULL = the legacy
 *     default stream). Work is enqueued, never waited for, unless a call says
 *     it synchronizes. When a call uses a different stream from the previous
 *     call on the context, it first makes its stream wait for the previous
 *     call's work (an event), so roles may run on separate streams. No such
 *     wait crosses a stream-capture boundary: around a capture the caller
 *     orders the work (e.g. synchronizes before capturing).
 *   - Host-detected errors return at once and enqueue nothing.
 *   - The caller owns every pointer it passes; each must stay valid and
 *     unchanged until the GPU work that reads or writes it has completed.
 *   - The context owns the receive arenas, the receipts, the single-worker
 *     view inboxes and the pinned host counts; pointers it returns stay
 *     valid until afd_destroy, and their contents until the exchange's rules
 *     below say.
 *   - All calls are host-thread-unsafe on one context: serialize them.
 */
#ifndef AFD_H
#define AFD_H

#include <stdint.h>

#if defined(__GNUC__)
#define AFD_API __attribute__((visibility("default")))
#else
#define AFD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* afd_stream; /* a cudaStream_t */

typedef struct afd_ctx afd_ctx; /* opaque, owned by the library */

typedef enum afd_status {
  AFD_OK = 0,
  AFD_ERR_ARG = 1,          /* null pointer, size, shape or stride outside the contract */
  AFD_ERR_STATE = 2,        /* call out of exchange order, or repeated */
  AFD_ERR_BUCKET = 3,       /* T > bucket, bucket > capacity, or roles disagree on
                               bucket / read_host_counts within one exchange */
  AFD_ERR_RECEIPT = 4,      /* reply receipt, worker or row count differs from the receive */
  AFD_ERR_ROUTE_RANGE = 5,  /* device-detected top-k ID outside [-1, num_experts) */
  AFD_ERR_ROUTE_DUP = 6,    /* device-detected repeated ID within one token */
  AFD_ERR_CUDA = 7,         /* a CUDA runtime call failed (see afd_error_detail) */
  AFD_ERR_OOM = 8,          /* device or pinned allocation failed at create */
  AFD_ERR_CAPTURING = 9,    /* a host-synchronizing request on a capturing stream */
  AFD_ERR_UNSUPPORTED = 10, /* configuration outside what this build implements */
  AFD_ERR_TIMEOUT = 11      /* a bounded device-side wait gave up (reported like a route
                               error, through afd_get_error; the outputs are unspecified) */
} afd_status;

enum { AFD_BF16 = 0, AFD_FP8_E4M3 = 1 };

/* How the combine sums a token's reply rows (afd_config.combine_mode).
 * FUSED: one FP32 fused multiply-add chain over the routes in ascending k,
 *   one rounding to BF16.
 * TWO_STAGE: the pages' two-stage reduction (afdEP-comm design page,
 *   sections 6 and 19): each worker's routes give a BF16 partial (FMA chain
 *   in ascending k, one rounding); the partials are added in FP32 in the
 *   order of each worker's last route and rounded once. Equal to FUSED when
 *   F == 1.
 * TWO_STAGE_FP8: as TWO_STAGE, with each partial carried as E4M3 values and
 *   a shared power-of-two factor 2^e for every block of 128 of them (e the
 *   smallest integer >= -117 with amax <= 448 * 2^e): the lossy reply format
 *   of section 19. Each decoded value q * 2^e is rounded to FP32 before it is
 *   added, so a block whose amax is 248 * 2^120 or more decodes to infinity.
 * The two-stage modes need top_k <= 8. */
enum { AFD_COMBINE_FUSED = 0, AFD_COMBINE_TWO_STAGE = 1, AFD_COMBINE_TWO_STAGE_FP8 = 2 };

/* Fixed per context. "API contract", Roles and tensors: H divisible by 256,
 * top-k at most 32 and at most E, experts divide evenly over the workers (worker f owns
 * experts [f*E/F, (f+1)*E/F)). Limits of this build: A <= 64, F <= 64,
 * E <= 1024, and a worker arena below 2^24 rows. */
typedef struct afd_config {
  int32_t num_sources;      /* A >= 1 Attention sources */
  int32_t num_workers;      /* F >= 1 FFN workers */
  int32_t num_experts;      /* E, a multiple of F */
  int32_t top_k;            /* K, 1 <= K <= min(32, E) */
  int32_t hidden;           /* H, a multiple of 256 */
  int32_t capacity;         /* max tokens per source in one exchange (sizes the arenas) */
  int32_t expert_alignment; /* alpha >= 1: each expert's first row is a multiple of alpha */
  int32_t dtype;            /* AFD_BF16, or AFD_FP8_E4M3 (E4M3 rows + FP32 block-128 scales) */
  int32_t num_sms;          /* cap on the SMs the kernels spread over; 0 = every SM */
  int32_t combine_mode;     /* AFD_COMBINE_FUSED (0), _TWO_STAGE or _TWO_STAGE_FP8 */
} afd_config;

/* Creates a context on `device` and allocates its device arenas:
 *   rows      F x R_arena x row_bytes   (row_bytes = 2H for BF16, H for FP8)
 *   scales    F x R_arena x H/128 FP32  (FP8 only)
 *   inboxes   A x capacity x H BF16     (F == 1 only; see afd_source_collect)
 * with R_arena = align_up(A*capacity*min(K, E/F) + (E/F)*(alpha-1), alpha).
 * Returns AFD_ERR_ARG / AFD_ERR_UNSUPPORTED for a bad config, AFD_ERR_OOM if
 * an allocation fails (nothing is leaked), AFD_ERR_CUDA for a bad device.
 * "API contract": Buffer(group, config). */
AFD_API afd_status afd_create(const afd_config* config, int32_t device, afd_ctx** out);

/* Waits for the context's outstanding work, frees everything it owns.
 * NULL is accepted. Counterpart of Buffer.close() in the "API contract"
 * (Graphs, streams and lifetime). CUDA graphs that captured calls on this
 * context must be destroyed before it. */
AFD_API afd_status afd_destroy(afd_ctx* ctx);

/* Stages source `source` for the current exchange. "API contract", Roles and
 * tensors: source_dispatch(x, ids, weights, x_scale=None, *, bucket,
 * read_host_counts=False).
 *   x          device, [num_tokens, H]: BF16, or E4M3 bytes for AFD_FP8_E4M3
 *   ids        device int64 [num_tokens, K]; each ID in [0, E) or -1 (skip),
 *              unique within a token
 *   weights    device FP32 [num_tokens, K]; weight of the matching ID
 *   x_scale    device FP32 scales (FP8 only, else NULL): the scale of token t,
 *              128-column block b is x_scale[t*scale_stride_t +
 *              b*scale_stride_b] (strided views, e.g. a transposed [H/128, T]
 *              tensor, are allowed); strides are in elements
 *   num_tokens T, 0 <= T <= bucket (T = 0 sources are valid and contribute
 *              nothing; x/ids/weights may then be NULL)
 *   bucket     bucket <= capacity; every call of one exchange passes the same
 *   read_host_counts  0 or 1; every call of one exchange passes the same
 * When every source has staged, this call enqueues the exchange's layout and
 * scatter kernels on `stream`. Route checks run on the GPU: an invalid ID
 * makes the exchange's outputs unspecified and sets the context's sticky
 * route error (afd_get_error); it never traps the device.
 * Errors: AFD_ERR_STATE (source already staged, or the previous exchange is
 * not collected), AFD_ERR_BUCKET, AFD_ERR_ARG, AFD_ERR_CAPTURING
 * (read_host_counts on a capturing stream), AFD_ERR_CUDA. */
AFD_API afd_status afd_source_dispatch(afd_ctx* ctx, int32_t source, const void* x, const int64_t* ids,
                               const float* weights, const float* x_scale,
                               int64_t scale_stride_t, int64_t scale_stride_b,
                               int32_t num_tokens, int32_t bucket, int32_t read_host_counts,
                               afd_stream stream);

/* Dispatch that reuses the routing of the last exchange (its IDs, layout and
 * receipts) and moves only the rows: the decode-time routing reuse of
 * "DeepEP V2 ElasticBuffer first principles", section 4 (cached dispatch
 * skips the layout and any host synchronization). Every source of the
 * exchange must use this call (no mixing with afd_source_dispatch), with the
 * same num_tokens and bucket as in the last exchange whose dispatch ran the
 * layout; ends[], host counts, row_src and the receipts stay as they were.
 *   x, x_scale, strides, read_host_counts: as in afd_source_dispatch
 *   weights    device FP32 [num_tokens, K] new routing weights for the same
 *              IDs, or NULL to keep the previous exchange's weights
 * Errors: AFD_ERR_STATE (no layout to reuse, a different num_tokens/bucket,
 * or an exchange that mixes the two dispatch calls), plus those of
 * afd_source_dispatch. */
AFD_API afd_status afd_source_dispatch_cached(afd_ctx* ctx, int32_t source, const void* x,
                                              const float* weights, const float* x_scale,
                                              int64_t scale_stride_t, int64_t scale_stride_b,
                                              int32_t num_tokens, int32_t bucket,
                                              int32_t read_host_counts, afd_stream stream);

/* What a worker receives. Rows of local expert l (0 <= l < E/F) are
 * [align_up(ends[l-1], alpha), ends[l]) with ends[-1] = 0 ("API contract",
 * Roles and tensors). Inside an expert, rows follow source ascending, then
 * token ascending. Padding rows below align_up(ends[E/F-1], alpha) have
 * row_src -1 and weight +0; rows from there up to num_rows are unspecified,
 * and so are the bytes of every padding row. A consumer must treat only the
 * rows inside some [start, ends[l]) range as tokens. */
typedef struct afd_recv {
  void* rows;                 /* device [num_rows, H] BF16 or E4M3 bytes (context-owned) */
  float* row_scales;          /* device FP32 [num_rows, H/128] (FP8), else NULL */
  const float* weights;       /* device FP32 [num_rows]: routing weight of each row */
  const int32_t* row_src;     /* device int32 [num_rows]: (s*bucket + t)*K + k, or -1 */
  const int32_t* ends;        /* device int32 [E/F] receive prefix sums */
  const int32_t* host_counts; /* pinned host int32 [E/F] aligned counts
                                 align_up(count[l], alpha), or NULL */
  int64_t num_rows;           /* receive shape to hand back to afd_worker_reply */
  uint64_t receipt;           /* opaque; pass unchanged to afd_worker_reply */
} afd_recv;

/* Returns worker `worker`'s part of the current exchange. Launches no kernel.
 * read_host_counts = 0: num_rows is the conservative capacity
 * align_up(A*bucket*min(K, E/F) + (E/F)*(alpha-1), alpha) and the device
 * ends[] identify live rows; host_counts is NULL. read_host_counts = 1:
 * synchronizes `stream`, copies the aligned counts to pinned host memory and
 * sets num_rows to their sum (the exact receive shape); it then reports a
 * pending route error as AFD_ERR_ROUTE_*. This is the host-synchronizing
 * mode of the "API contract" (Graphs, streams and lifetime), meant for eager
 * callers that size their expert buffers exactly. Rows stay valid until the
 * next exchange's last afd_source_dispatch is enqueued.
 * Errors: AFD_ERR_STATE (no dispatched exchange, or worker already received),
 * AFD_ERR_BUCKET, AFD_ERR_CAPTURING, AFD_ERR_ARG, AFD_ERR_CUDA. */
AFD_API afd_status afd_worker_receive(afd_ctx* ctx, int32_t worker, int32_t bucket,
                              int32_t read_host_counts, afd_stream stream, afd_recv* out);

/* Hands worker `worker`'s BF16 replies back ("API contract": worker_reply).
 * The reply covers the whole receive shape, row for row; only rows that hold
 * a route are read.
 *   rows      device BF16 [num_rows, H], unweighted expert outputs; row r
 *             answers received row r. Padding rows are never read. It may be
 *             the received rows themselves (an identity expert, BF16 only).
 *             The library reads it until the combine of the exchange's last
 *             collected source has completed; it must stay unchanged until
 *             then.
 *   num_rows  must equal the afd_recv.num_rows of this worker's receive
 *   receipt   must equal the afd_recv.receipt of this worker's receive
 * The library applies each routing weight exactly once, in the combine,
 * which runs in afd_source_collect (one launch per source) or
 * afd_source_collect_all (one launch for all sources), for every F. This call
 * launches no kernel.
 * Errors: AFD_ERR_STATE, AFD_ERR_RECEIPT, AFD_ERR_ARG, AFD_ERR_CUDA. */
AFD_API afd_status afd_worker_reply(afd_ctx* ctx, int32_t worker, const void* rows, int64_t num_rows,
                            uint64_t receipt, afd_stream stream);

/* A view handed out by afd_source_collect. */
typedef struct afd_view {
  const void* data;   /* device BF16 [num_tokens, H] with row stride `row_stride` */
  int64_t row_stride; /* in elements */
  int32_t num_tokens;
  int32_t is_view;    /* 1: `data` is the context's inbox; 0: the result is in `out` */
} afd_view;

/* Source `source`'s result: out[t][h] = bf16(sum over k ascending of
 * w[t][k] * reply(k)[h]) accumulated with FP32 fused multiply-adds from +0
 * and rounded once to nearest-even; skipped (-1) routes add nothing; a token
 * with no valid route gives +0. Rows come back in the source's own token
 * order. Counterpart of source_collect(*, view=False) in the "API contract".
 *   out   device BF16 [T, H] (contiguous), T = the source's num_tokens; may be
 *         NULL only when view = 1 and F == 1
 *   view  1 asks for the single-worker view: with F == 1 the combine writes
 *         the context's inbox instead of `out`, and `view_out` points at it,
 *         read-only and valid until the next afd_source_dispatch on this
 *         context ("13. Single-FFN collect view" of the design page). With
 *         F > 1 the ordinary result is written to `out` and
 *         view_out->is_view = 0.
 *   view_out  host; filled on success (may be NULL when view = 0)
 * When the previous call on this context was a collect of the same exchange
 * that launched a combine on the same stream, this call's combine starts
 * without waiting for that one (both only read the replies) and completes
 * after it, so stream order still holds for whatever follows. Work enqueued on
 * the stream between the two calls must therefore not write the reply rows
 * or this source's `out`.
 * Errors: AFD_ERR_STATE (replies missing, or source already collected),
 * AFD_ERR_ARG, AFD_ERR_CUDA. */
AFD_API afd_status afd_source_collect(afd_ctx* ctx, int32_t source, void* out, int32_t view,
                              afd_stream stream, afd_view* view_out);

/* Every source's result at once: for each source s the same as
 * afd_source_collect(s, outs[s], view, ...), with one combine launch for all
 * sources (on one GPU the sources' combines are independent, so they can
 * share a launch). Every source must still be uncollected.
 *   outs   host array of A device pointers, BF16 [T_s, H] each; an entry may
 *          be NULL for a source with T = 0, or when view = 1 and F == 1
 *   view   as in afd_source_collect
 *   views  host array of A afd_view, filled on success; may be NULL
 * Errors: as afd_source_collect (nothing is enqueued on an error). */
AFD_API afd_status afd_source_collect_all(afd_ctx* ctx, void* const* outs, int32_t view,
                                          afd_stream stream, afd_view* views);

/* The sticky error found on the GPU. Synchronizes the context's device work
 * first. code = AFD_OK, AFD_ERR_ROUTE_RANGE or AFD_ERR_ROUTE_DUP (for these,
 * (source, token, k) is the invalid route that comes first in (source,
 * token, k) order among all exchanges since the last afd_clear_error), or
 * AFD_ERR_TIMEOUT (a bounded wait of the scatter's bulk copies gave up at
 * (source, token); k = 0; see afd_set_wait_limit). Any pointer may be NULL.
 * Not allowed while the context's last stream is capturing
 * (AFD_ERR_CAPTURING). */
AFD_API afd_status afd_get_error(afd_ctx* ctx, int32_t* code, int32_t* source, int32_t* token,
                         int32_t* k);

/* Sets how many times the scatter polls for each source row's bulk load
 * before it gives up (default 4,194,304, each poll possibly suspending the
 * thread for a while). A load that does not complete in time is reported
 * through afd_get_error as AFD_ERR_TIMEOUT at that row's (source, token); the
 * warp that gave up waits for the load still in flight (up to 2 s of GPU
 * time), moves no more rows but still writes every receipt, so the rest of
 * the exchange runs and its outputs are unspecified. 0 makes every first
 * wait give up at once: a way to exercise that error path. Applies to
 * dispatches enqueued after the call (a captured graph keeps the value it
 * was captured with).
 * Errors: AFD_ERR_ARG (polls < 0). */
AFD_API afd_status afd_set_wait_limit(afd_ctx* ctx, int32_t polls);

/* For benchmarks that start every step with a cold L2: writes the first half
 * of `scratch` and then reads the second half, 16 bytes at a time, both with
 * an L2 evict-last policy (the one the scatter's row stores use, which
 * ordinary writes and reads cannot evict). Afterwards L2 holds only clean
 * lines of the second half: every earlier line, whatever its priority, has
 * been evicted and, if dirty, written back. Enqueued on `stream`.
 *   scratch  device memory of `bytes` bytes, 16-byte aligned; its contents
 *            are overwritten
 *   bytes    a multiple of 32, at least twice the L2 size for a full flush
 * Errors: AFD_ERR_ARG (alignment or size), AFD_ERR_CUDA. */
AFD_API afd_status afd_l2_flush(void* scratch, int64_t bytes, afd_stream stream);

/* Diagnostic: the phase stamps of a library built with -DAFD_PHASE_TIMERS=1
 * (%globaltimer, ns). Synchronizes the device, then copies the stamps to
 * `host` as uint64 [4][4096][8]: [kind][block][point], 0 where nothing was
 * recorded; clear = 1 also zeroes them. Kinds: 0 the exchange's first
 * dispatch kernel (points 0 start, 1 dependency wait passed, 2 first IDs
 * marked, 3 counted, 4 cluster barrier passed, 5 counts of all CTAs read,
 * 6 scan done, 7 route codes written; the one-kernel dispatches record 0, 1
 * and 7), 1 the scatter (0 start, 1 wait passed, 2 first row in shared
 * memory, 3 all stores issued, 4 stores complete, 5 end), 2 a combine that
 * waits first and 3 an early-started combine (0 start, 1 wait passed or
 * ready to load, 2 sums stored, 3 end). The stamps are global to the process;
 * the last launch of a kind overwrites the earlier ones; blocks past 4096
 * are not recorded.
 *   host   host uint64 array of `count` >= 131072 elements
 * Errors: AFD_ERR_UNSUPPORTED when built without phase timers (whatever the
 * arguments), AFD_ERR_ARG, AFD_ERR_CUDA. */
AFD_API afd_status afd_phase_stamps(afd_ctx* ctx, uint64_t* host, int64_t count, int32_t clear);

/* Clears the sticky route error (enqueued on `stream`). */
AFD_API afd_status afd_clear_error(afd_ctx* ctx, afd_stream stream);

/* Abandons the current exchange (host state only; enqueued GPU work still
 * runs). Lets a caller recover after a failed call mid-exchange. */
AFD_API afd_status afd_reset_exchange(afd_ctx* ctx);

/* Static text for a status. */
AFD_API const char* afd_status_string(afd_status status);

/* Text of the last failure on this context (host check or CUDA error). */
AFD_API const char* afd_error_detail(const afd_ctx* ctx);

/* Receive arena rows per worker (R_arena above), for sizing reply buffers. */
AFD_API int64_t afd_arena_rows(const afd_ctx* ctx);

/* Receive shape for `bucket` with read_host_counts = 0. */
AFD_API int64_t afd_recv_rows_for_bucket(const afd_ctx* ctx, int32_t bucket);

/* Routing layout without allocation (no counterpart in the pages). Some
 * callers cannot call cudaMalloc: code that runs inside another framework's
 * memory pool or allocator hook, or a process whose device memory is fully
 * reserved up front. This call allocates nothing, through the CUDA runtime or
 * any library: its scratch (384 KiB) is a fixed device array inside
 * libafd, which every GPU that loads the library holds until the process
 * exits. It computes, for one source's routing, what the dispatch layout
 * computes: route checks, per-worker ends[] with expert_alignment padding,
 * and the row of every valid route (expert-major; inside an expert, token
 * order), without moving any payload.
 *   ids        device int64 [num_tokens, top_k]; IDs in [0, num_experts) or -1
 *   ends       device int32 [num_experts] out: per worker f, ends[f*E/F + l]
 *              is local expert l's end (same convention as afd_recv.ends)
 *   slots      device int32 [num_tokens, top_k] out: the route's row inside
 *              its worker (worker = ID / (E/F)), or -1 (skipped or invalid)
 *   error      device int32 [3] out: {code, token, k} of the first invalid
 *              route in (token, k) order (code AFD_ERR_ROUTE_RANGE or
 *              AFD_ERR_ROUTE_DUP), or {AFD_OK, -1, -1}
 * Limits: num_tokens <= 8192, top_k <= 32, num_tokens * top_k <= 65536,
 * num_experts <= 1024, and align_up(num_tokens * top_k + (E/F) *
 * (expert_alignment - 1), expert_alignment) <= INT32_MAX (the largest row
 * index of a worker must fit an int32); larger sizes return
 * AFD_ERR_UNSUPPORTED and enqueue nothing. Every buffer must be reachable from the current device (its
 * device memory, managed memory, or page-locked host memory); pageable host
 * memory or another device's memory returns AFD_ERR_ARG and enqueues
 * nothing. Work is enqueued on `stream` (the current device's).
 * The first call on a device looks up the scratch array's device address
 * (and sets a kernel attribute); make that first call before any stream
 * capture on that device. All calls on a device share the one scratch array:
 * calls whose GPU work overlaps (different streams without ordering) race and
 * give wrong results; order them. */
AFD_API afd_status afd_route_layout_noalloc(const int64_t* ids, int32_t num_tokens, int32_t top_k,
                                            int32_t num_experts, int32_t num_workers,
                                            int32_t expert_alignment, int32_t* ends,
                                            int32_t* slots, int32_t* error, afd_stream stream);

/* Library version, (major << 16) | minor. */
AFD_API int32_t afd_version(void);

#ifdef __cplusplus
}
#endif
#endif /* AFD_H */
