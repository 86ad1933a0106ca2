/*
 * mla_decode.h -- C ABI of libmla_decode: single-token decode attention for
 * multi-head latent attention (MLA) on one GB300 (sm_103a).
 *
 * The operation (kernelindex.com, amd-mixed-mla submissions 668813 "v0092a",
 * 695854 and 600081): every request b has 16 query heads q[b,h,0:576] that
 * share one latent KV head.  Over the request's tokens t (reached through
 * kv_indptr and a page table) the scores are
 *     s[h,t] = (1/sqrt(576)) * sum_{d<576} q[b,h,d] * k_t[d]
 * and the output is the softmax-weighted sum of the first 512 dims of k_t:
 *     out[b,h,:] = sum_t softmax_t(s[h,:]) * k_t[0:512],
 *     lse[b,h]   = ln sum_t exp(s[h,t]).
 * The KV row is stored bf16, fp8-e4m3 times one per-tensor fp32 kv_scale, or
 * MXFP4 (e2m1 nibbles, element 2i in the low nibble of byte i, one e8m0 scale
 * byte per 32 elements).  The work is cut into split-KV pieces whose partial
 * results are merged by their log-sum-exp weights (the stage-1 / stage-2
 * scheme of submission 668813's MXFP4 route and of aiter's
 * mla_decode_fwd / mla_reduce_v1 calls on all three pages).
 *
 * Conventions for every call:
 *   - Nothing throws and nothing falls back to the CPU: each call returns an
 *     mla_status.  A call that returns an error has launched nothing.
 *   - mla_decode_run never synchronises the stream and never reads device
 *     memory on the host.
 *   - Pointers named *_host are host memory; every other data pointer is
 *     device memory owned by the caller.  The plan object is owned by the
 *     library and released with mla_plan_destroy.
 *   - A plan is not thread-safe: mla_decode_run updates caches inside it
 *     (tensor maps, which workspace holds its table), so one plan must not
 *     be used by two host threads at the same time.  Different plans may.
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* mla_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer, bad indptr */
  MLA_ERR_UNSUPPORTED = 2,   /* valid but not implemented combination (dtype / page size) */
  MLA_ERR_WORKSPACE = 3,     /* workspace smaller than mla_plan_workspace_size(), or (from
                                mla_decode_check) holding another plan's table */
  MLA_ERR_CUDA = 4,          /* a CUDA runtime / driver call failed */
  MLA_ERR_DEVICE_TIMEOUT = 5 /* a device-side pipeline wait gave up (see mla_decode_check) */
} mla_status;

typedef enum {
  MLA_DTYPE_BF16 = 0,
  MLA_DTYPE_FP8_E4M3 = 1,   /* OCP e4m3fn, used with a per-tensor fp32 scale */
  MLA_DTYPE_MXFP4 = 2       /* KV only: 288 packed bytes + e8m0 scales per token */
} mla_dtype;

typedef struct mla_plan mla_plan;

#define MLA_MAX_Q_LEN 64   /* query tokens per request accepted by mla_decode_plan_q */

typedef struct {
  int32_t batch_size;
  int32_t page_size;
  int32_t num_ctas;          /* stage-1 grid size */
  int32_t num_items;         /* work items (request, token range) */
  int32_t num_partials;      /* split partial results written to the workspace */
  int32_t num_merge_jobs;    /* requests merged (or zero-filled) by stage 2 */
  int64_t total_tokens;
  int64_t total_tiles;       /* 128-token tiles over all requests */
  size_t workspace_bytes;
  int32_t q_len;             /* query tokens per request */
  int32_t unit_tokens;       /* tokens between possible cut points (mla_plan_options) */
  int32_t item_cost;         /* cost of an extra request in a CTA (balanced plan) */
  int32_t cluster_size;      /* 8: split requests are merged inside stage 1, in
                                thread-block clusters of that many CTAs (mla_plan_options
                                merge); 0: by stage 2 */
} mla_plan_info;

/*
 * mla_decode_plan -- build the work partition for one batch shape.
 *
 * Plays the role of aiter's get_mla_metadata_v1 on the pages (submission
 * 668813 cache builders; submission 600081 "v9" persistent path): it reads
 * only host arrays, so it causes no device synchronisation.
 *
 *   kv_indptr_host        [batch_size+1] int32, non-decreasing, in PAGES:
 *                         request b owns page-table entries
 *                         kv_indptr[b] .. kv_indptr[b+1]-1.  With
 *                         page_size == 1 this is a token offset.
 *   kv_last_page_len_host [batch_size] int32 tokens used in each request's
 *                         last page (1..page_size), or NULL for full pages.
 *   batch_size            >= 1.
 *   page_size             tokens per page, >= 1.  With a page table, a
 *                         multiple of 8 lets one TMA box copy 8 rows of a
 *                         page; other sizes (bf16 / fp8 KV) copy every row
 *                         on its own.  MXFP4 rows are loaded row by row
 *                         by the dequantising threads, for any page size.
 *   q_dtype               MLA_DTYPE_BF16 or MLA_DTYPE_FP8_E4M3.
 *   kv_dtype              MLA_DTYPE_BF16, MLA_DTYPE_FP8_E4M3 or MLA_DTYPE_MXFP4.
 *   num_splits            0: the planner balances 128-token tiles over the
 *                         CTAs (a request may be cut anywhere on a tile
 *                         boundary), counting each extra request a CTA
 *                         holds as half a tile; S > 0: every request is cut into S
 *                         contiguous ranges of ceil(tiles/S) tiles, one CTA
 *                         each, as the pages' fixed-split kernels do.
 *   num_sms               CTAs of the balanced plan; 0 = the SM count of the
 *                         current CUDA device.
 *   plan_out              receives the new plan (library-owned).
 * Errors: MLA_ERR_INVALID_ARG (null/negative/non-monotone input, bad
 * last-page length), MLA_ERR_UNSUPPORTED (dtype or page size combination not
 * implemented), MLA_ERR_CUDA (device query failed when num_sms == 0).
 */
mla_status mla_decode_plan(const int32_t* kv_indptr_host, const int32_t* kv_last_page_len_host,
                           int32_t batch_size, int32_t page_size, mla_dtype q_dtype,
                           mla_dtype kv_dtype, int32_t num_splits, int32_t num_sms,
                           mla_plan** plan_out);

/*
 * mla_decode_plan_q -- mla_decode_plan for q_len query tokens per request
 * (speculative or multi-token decode).  mla_decode_plan is this call with
 * q_len = 1.
 *
 * The pages run one query token per request (max_seqlen_qo = 1 in the
 * metadata calls of submission 668813, with the causal flag set) and name
 * four query tokens in the route selection of submission 695854.  The
 * reading implemented: the q_len query tokens are the last q_len positions
 * of each sequence, already in the KV cache, and attend causally, so that
 * query token t of a request with n tokens attends to its first
 * n - q_len + 1 + t tokens (none: out = 0, lse = -inf).
 *
 * q, out and lse then hold batch_size * q_len rows, row b * q_len + t for
 * query token t of request b ([batch, q_len, 16, ...] contiguous).  With an
 * even q_len and fp8 q and KV, query tokens 2p and 2p+1 share one pass over
 * the KV (32 q rows per tile).  Otherwise every query token is planned as its
 * own causal prefix.  The balanced plan gives each pass (pair or token) its
 * own group of CTAs, balanced over all requests, so that the passes over a
 * request's KV run side by side and all but one are served from L2.
 *
 * Arguments as for mla_decode_plan, plus q_len in [1, MLA_MAX_Q_LEN].
 * Errors: as mla_decode_plan; MLA_ERR_INVALID_ARG for q_len out of range or
 * batch_size * q_len * 16 above INT32_MAX.
 */
mla_status mla_decode_plan_q(const int32_t* kv_indptr_host, const int32_t* kv_last_page_len_host,
                             int32_t batch_size, int32_t q_len, int32_t page_size,
                             mla_dtype q_dtype, mla_dtype kv_dtype, int32_t num_splits,
                             int32_t num_sms, mla_plan** plan_out);

/*
 * Plan options (mla_decode_plan_ex, mla_decode_autotune).  All zero gives
 * the plan of mla_decode_plan with num_splits = 0 on every SM.
 *   num_splits   0: balanced plan; S > 0: every request cut into S ranges.
 *   num_sms      CTAs of a balanced plan; 0 = the SM count of the device.
 *   item_cost    balanced plan: what an extra request in a CTA costs, in
 *                half tiles (an epilogue before the next request's first
 *                tile); 0 = 1.  Larger values give fewer requests per CTA.
 *   unit_tokens  tokens between the planner's possible cut points: 128 (a
 *                whole tile; 0 means 128), 64 or 32.  Finer cuts spread small
 *                batches over more CTAs (each then loads only its rows).
 *   merge        0: when every CTA holds one item and every request is split
 *                over 8 consecutive CTAs (a small batch of equal lengths, one
 *                query token, bf16 or fp8 KV), each request's CTAs run as one
 *                thread-block cluster and merge its partials through
 *                distributed shared memory: no partials in the workspace, no
 *                stage-2 launch.  If the device cannot hold such a cluster,
 *                run falls back to stage 2.  1: always merge with stage 2.
 */
typedef struct {
  int32_t num_splits;
  int32_t num_sms;
  int32_t item_cost;
  int32_t unit_tokens;
  int32_t merge;
} mla_plan_options;

/*
 * mla_decode_plan_ex -- mla_decode_plan_q with plan options (NULL = all
 * zero).  Errors: as mla_decode_plan_q; MLA_ERR_INVALID_ARG for an item cost
 * outside [0, 64] or a unit other than 0, 32, 64, 128.
 */
mla_status mla_decode_plan_ex(const int32_t* kv_indptr_host, const int32_t* kv_last_page_len_host,
                              int32_t batch_size, int32_t q_len, int32_t page_size,
                              mla_dtype q_dtype, mla_dtype kv_dtype,
                              const mla_plan_options* options, mla_plan** plan_out);

/* One timed candidate of mla_decode_autotune: its options and the median
 * time of its timed calls in milliseconds (< 0: not timed, its workspace did
 * not fit). */
typedef struct {
  mla_plan_options options;
  float ms;
} mla_tune_result;

#define MLA_TUNE_IGNORE_CACHE 1   /* mla_decode_autotune flag: time even a shape seen before */

/*
 * mla_decode_autotune -- choose the plan of one batch shape by timing
 * candidate plans on the caller's inputs (the runtime autotune of the
 * earlier version of submission 600081: _time_fn / _aiter_best /
 * _best_for_shape).  The candidates are the default balanced plan (and,
 * when it merges inside clusters, the same plan merged by stage 2), item
 * costs 2 and 4, cut units of 64 and 32 tokens, the split count of the
 * pages' split tables for this (batch, length) if it has one, and one split
 * per request.  Every candidate runs once (uploading its table), then `reps`
 * calls (1 .. 1000) are timed one by one with CUDA events on `stream`; the
 * candidate with the smallest median time wins (mla_autotune_select), and
 * the winner is remembered for the shape (batch, query tokens, page size,
 * formats, total and largest request length, page table or not, device) for
 * the rest of the process: a later call for the same shape returns that
 * plan without timing unless flags has MLA_TUNE_IGNORE_CACHE.
 *
 * Arguments: the shape as for mla_decode_plan_q, the inputs and outputs as
 * for mla_decode_run (out and lse are overwritten by the timed calls).
 * workspace NULL: nothing runs; *workspace_needed receives the workspace the
 * largest candidate needs (the two-call pattern).  Otherwise candidates
 * whose workspace exceeds workspace_bytes are skipped.  results (up to
 * max_results, may be NULL with max_results 0) receive each candidate's
 * options and median time, *num_results their count (0 when the cached
 * choice was used).  *plan_out receives the chosen plan (library-owned,
 * release it with mla_plan_destroy).
 *
 * This call synchronises `stream` (it reads the timings and the device error
 * word) and is meant for a first call per shape, not for the timed path.
 * Errors: MLA_ERR_INVALID_ARG (arguments; a page outside the pool),
 * MLA_ERR_WORKSPACE (no candidate fits the workspace), MLA_ERR_CUDA,
 * MLA_ERR_DEVICE_TIMEOUT, and the errors of mla_decode_plan_ex and
 * mla_decode_run.
 */
mla_status mla_decode_autotune(const int32_t* kv_indptr_host,
                               const int32_t* kv_last_page_len_host, int32_t batch_size,
                               int32_t q_len, int32_t page_size, mla_dtype q_dtype,
                               mla_dtype kv_dtype, const void* q, const float* q_scale,
                               const void* kv, const float* kv_scale, const uint8_t* kv_e8m0,
                               int64_t kv_e8m0_row_stride, int64_t kv_pool_rows,
                               const int32_t* kv_indices, void* workspace,
                               size_t workspace_bytes, void* out, float* lse, int32_t reps,
                               int32_t flags, mla_stream_t stream, mla_tune_result* results,
                               int32_t max_results, int32_t* num_results,
                               size_t* workspace_needed, mla_plan** plan_out);

/*
 * The selection rule of mla_decode_autotune, on the host: ms holds
 * num_candidates x reps times (candidate-major); a candidate with a negative
 * or NaN time was not run and is skipped.  *best receives the candidate with
 * the smallest median (for an even reps, the mean of the middle two), the
 * first one on ties.  Errors: MLA_ERR_INVALID_ARG on bad arguments or when
 * no candidate was run.
 */
mla_status mla_autotune_select(const float* ms, int32_t num_candidates, int32_t reps,
                               int32_t* best);

/* Bytes of device workspace mla_decode_run needs for this plan (work table,
 * split partials, error word).  Errors: MLA_ERR_INVALID_ARG on NULL. */
mla_status mla_plan_workspace_size(const mla_plan* plan, size_t* bytes);

/* Summary numbers of a plan.  Errors: MLA_ERR_INVALID_ARG on NULL. */
mla_status mla_plan_get_info(const mla_plan* plan, mla_plan_info* info);

/*
 * Copies the host work table out for inspection: cta_indptr [num_ctas+1]
 * int32 (items of CTA i are cta_indptr[i] .. cta_indptr[i+1]-1) and items
 * [num_items][4] int32 = {request, first token, end token, partial slot or -1
 * for a request written directly}.  Either pointer may be NULL.
 */
mla_status mla_plan_get_work(const mla_plan* plan, int32_t* cta_indptr, int32_t* items);

void mla_plan_destroy(mla_plan* plan);

/*
 * mla_decode_run -- one decode call (stage-1 split kernel + stage-2 merge),
 * enqueued on `stream`.  The role of aiter's mla_decode_fwd on the pages.
 *
 *   q          [batch,16,576] contiguous, bf16 or e4m3 bytes (plan's q_dtype);
 *              16-byte aligned.  A plan made with q_len > 1 takes
 *              [batch,q_len,16,576] (and out / lse likewise).
 *   q_scale    device fp32 [1]; required when q is e4m3, ignored otherwise.
 *   kv         KV pool, kv_pool_rows rows of 576 bf16 / 576 e4m3 bytes /
 *              288 packed MXFP4 bytes, contiguous; row r of page p is
 *              p*page_size + r.  16-byte aligned.
 *   kv_scale   device fp32 [1]; required for e4m3 KV, ignored otherwise.
 *   kv_e8m0, kv_e8m0_row_stride
 *              MXFP4 only: e8m0 scale rows, 18 bytes used per row (the
 *              pages' [total_kv, 18] layout), row stride in bytes: even and
 *              >= 18, base 2-byte aligned (MLA_ERR_INVALID_ARG below 18,
 *              MLA_ERR_UNSUPPORTED if odd).  NULL / ignored for other KV types.
 *   kv_pool_rows  number of rows in the KV pool (bounds every access).
 *   kv_indices device int32 page table, indexed from kv_indptr; NULL = the
 *              identity table (request b's pages are kv_indptr[b]..; they
 *              must all lie inside the pool, else MLA_ERR_INVALID_ARG).
 *              Every entry must be a page inside the pool: an entry outside
 *              it is read as page 0 and reported by mla_decode_check.
 *   workspace, workspace_bytes
 *              device scratch of at least mla_plan_workspace_size() bytes,
 *              256-byte aligned.  The work table is copied into it on the
 *              first run with a given workspace pointer (one host-to-device
 *              copy on `stream`); afterwards runs only launch kernels.  A
 *              workspace belongs to one plan.  If the memory at that address
 *              was freed and reused for another plan's workspace (a caching
 *              allocator hands out the same address again), the kernels find
 *              the other plan's stamp in it, write nothing, and the next
 *              mla_decode_check returns MLA_ERR_WORKSPACE; the plan then
 *              uploads its table again on its next run.
 *   out        [batch,16,512] bf16, 16-byte aligned.
 *   lse        [batch,16] fp32 natural-log LSE of the scaled scores, or NULL.
 *              Empty requests give out = 0 and lse = -inf.
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_WORKSPACE, MLA_ERR_UNSUPPORTED,
 * MLA_ERR_CUDA (launch failure; the stream state is then the caller's).
 */
mla_status mla_decode_run(mla_plan* plan, const void* q, const float* q_scale, const void* kv,
                          const float* kv_scale, const uint8_t* kv_e8m0,
                          int64_t kv_e8m0_row_stride, int64_t kv_pool_rows,
                          const int32_t* kv_indices, void* workspace, size_t workspace_bytes,
                          void* out, float* lse, mla_stream_t stream);

/*
 * Synchronises `stream`, reads the workspace's device error word and clears
 * it.  Returns
 *   MLA_OK                  nothing went wrong since the last check;
 *   MLA_ERR_DEVICE_TIMEOUT  a kernel's bounded pipeline wait gave up;
 *   MLA_ERR_INVALID_ARG     a page-table entry pointed outside the pool (that
 *                           entry was read as page 0, so the outputs of its
 *                           request are wrong; nothing outside the pool was
 *                           touched);
 *   MLA_ERR_WORKSPACE       the workspace held another plan's table, so the
 *                           run wrote no output (see mla_decode_run);
 *   MLA_ERR_CUDA            a CUDA call failed.
 * workspace NULL checks the library's own array used by
 * mla_decode_run_noalloc on the current device instead (errors of a
 * no-allocation call are readable until the next such call on the device).
 */
mla_status mla_decode_check(const mla_plan* plan, void* workspace, mla_stream_t stream);

/*
 * mla_selftest_bounded_wait -- exercises the timeout path of the pipeline
 * waits on the GPU.  It launches one warp that waits, with the same bounded
 * wait every decode pipeline stage uses, on an mbarrier that nothing arrives
 * on, for limit_us microseconds (1 .. 1000000).  The workspace's device error
 * word is cleared first; the wait gives up and sets its producer bit, and the
 * kernel returns.  The next mla_decode_check then returns MLA_ERR_DEVICE_TIMEOUT and
 * clears the word; the CUDA context stays usable.  Enqueued on `stream`.
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_WORKSPACE, MLA_ERR_CUDA.
 */
mla_status mla_selftest_bounded_wait(const mla_plan* plan, void* workspace, size_t workspace_bytes,
                                     uint32_t limit_us, mla_stream_t stream);

/*
 * mla_decode_run_noalloc -- mla_decode_run without a caller-provided workspace.
 *
 * The pages have no counterpart of this call.  It is for callers that cannot
 * allocate device memory (a plug-in or C client inside a process whose
 * framework owns the device allocator, or code that must not allocate once
 * it runs): the library keeps a fixed 16 MiB workspace array in device global
 * memory, which every GPU that loads the library holds until the process
 * exits.  Inputs, outputs and their rules are those of mla_decode_run.
 *   - Plans needing more than 16 MiB (mla_plan_workspace_size) are rejected
 *     with MLA_ERR_WORKSPACE before anything is enqueued.
 *   - The first call on a device looks the array's address up
 *     (cudaGetSymbolAddress) with that device current.
 *   - Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.
 *   - Every call copies its plan's work table into the array (one
 *     host-to-device copy on `stream`), which also clears the error word.
 *   - Device-side errors of a call (a bounded wait that gave up, a page
 *     outside the pool) are read with mla_decode_check(plan, NULL, stream)
 *     before the next call on the device clears them.
 *   - All calls share the one array: calls that overlap on the GPU (other
 *     streams, other threads) race and corrupt each other; order them.
 * Errors: as mla_decode_run, plus MLA_ERR_WORKSPACE for an oversized plan
 * and MLA_ERR_CUDA if the array's address cannot be obtained.
 */
mla_status mla_decode_run_noalloc(mla_plan* plan, const void* q, const float* q_scale,
                                  const void* kv, const float* kv_scale, const uint8_t* kv_e8m0,
                                  int64_t kv_e8m0_row_stride, int64_t kv_pool_rows,
                                  const int32_t* kv_indices, void* out, float* lse,
                                  mla_stream_t stream);

/*
 * Optional instrumentation (the pages time their decode stages with CUDA
 * events, submission 695854, stage timings): when `before` / `after` are
 * non-NULL cudaEvent_t handles, every following mla_decode_run records
 * `before` on its stream just before the stage-1 launch and `after` just
 * after it.  Pass NULL, NULL to stop.  The events stay owned by the caller.
 * Errors: MLA_ERR_INVALID_ARG on a NULL plan.
 */
mla_status mla_plan_set_stage1_events(mla_plan* plan, void* before, void* after);

/* Static, human-readable name of a status code. */
const char* mla_status_string(mla_status status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */
