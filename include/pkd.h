/*
 * pkd -- batched GQA decode attention over a CSR-paged KV cache, for GB300
 * (sm_103a).  C ABI: plain pointers and sizes only.
 *
 * The problem (FlashInfer, in depth -- "The block-sparse page table",
 * "Plan and run: the inspector-executor split", "Load balancing with
 * split-KV"; FlashInfer 完全拆解 -- 页表就是一张块稀疏矩阵, 先切长 KV，再做
 * 最长任务优先分配, 固定指针比固定内容更重要, 在线 Softmax 为什么允许任意切块):
 *
 *   A batch of B requests, each with one query token.  Request i owns the
 *   pages indices[indptr[i] .. indptr[i+1]) of a page pool, in order; its
 *   last page holds last_page_len[i] tokens (1..P), so its KV length is
 *   l_i = P (n_i - 1) + last_page_len[i].  Each layer's cache is one tensor
 *   [num_pages][2][P][Hkv][D] (NHD; K at index 0, V at index 1).  For every
 *   request i and query head h (KV head h / g, g = Hq / Hkv):
 *       out[i][h] = softmax(q[i][h] . K^T / sqrt(D)) V
 *       lse[i][h] = log sum_t exp(q[i][h] . k_t / sqrt(D))   (natural log)
 *
 * Calls:
 *   pkd_plan  -- once per decode step, on the host: checks the table, splits
 *                long KV ranges into page-aligned chunks, assigns the work
 *                items to a fixed set of CTAs (longest first onto the least
 *                loaded), builds the reduction map, and copies the schedule
 *                into the fixed-address device workspace.
 *   pkd_run   -- once per layer: persistent decode kernel plus the merge of
 *                split chunks.  Stream-ordered, no host sync, no allocation,
 *                capturable in a CUDA graph.
 *   pkd_merge_states -- exact combination of two attention states.
 *
 * Conventions.  Every device pointer is a plain CUDA device address; every
 * stream argument is a cudaStream_t passed as void* (NULL = legacy default
 * stream).  The caller owns every buffer, the workspace included; the
 * library never allocates device memory.  Return values: PKD_OK (0) or a
 * negative PKD_E_* code; pkd_status_str() names it.  Nothing aborts.
 */
#ifndef PKD_H_
#define PKD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define PKD_OK 0
#define PKD_E_INVALID_ARG -1        /* null pointer, bad size, misaligned  */
#define PKD_E_BAD_TABLE -2          /* indptr / last_page_len / page id    */
#define PKD_E_UNSUPPORTED_SHAPE -3  /* D, Hq % Hkv, group size, Hkv        */
#define PKD_E_WORKSPACE_TOO_SMALL -4
#define PKD_E_NO_PLAN -5            /* run before any plan                  */
#define PKD_E_STALE_PLAN -6         /* run against another plan's epoch    */
#define PKD_E_CAPACITY -7           /* batch or page count above capacity  */
#define PKD_E_CUDA -8               /* a CUDA runtime call failed          */
#define PKD_E_DEVICE -9             /* the device reported an error word   */
#define PKD_E_SCRATCH_LIMIT -10     /* needs more than the static scratch   */

/* Device error word bits (pkd_last_device_error). */
#define PKD_DEV_ERR_TIMEOUT 1       /* a bounded wait gave up               */
#define PKD_DEV_ERR_BOUNDS 2        /* a schedule entry pointed out of range */

/* ---- configuration ----------------------------------------------------- */
typedef struct pkd_config {
    int32_t num_qo_heads;      /* Hq                                        */
    int32_t num_kv_heads;      /* Hkv, 1..8; Hq % Hkv == 0, g in {1,2,4,8}  */
    int32_t head_dim;          /* D; 128                                    */
    int32_t page_size;         /* P >= 1                                    */
    int32_t max_batch;         /* capacity: requests per plan               */
    int32_t max_num_pages;     /* capacity: page ids per plan (nnz)         */
    int32_t num_pages;         /* pool size; page ids must be < num_pages   */
    int32_t alpha;             /* per-item cost in tokens (cost = alpha +
                                  tokens); < 0 selects the default (32)     */
    int32_t min_chunk_tokens;  /* split floor in tokens; < 0 -> 256          */
    int32_t num_ctas;          /* persistent grid; 0 -> SMs x CTAs per SM    */
    uint32_t flags;            /* PKD_FLAG_* (0 = defaults)                 */
} pkd_config;

/* Consumer variant of the decode kernel.  By default the GQA group is folded
 * onto tensor cores (mma.sync m16n8k16, bf16 in / fp32 accumulate); the
 * CUDA-core variant (fp32 FMA) is kept for comparison.  These flags force
 * one; setting both is an error. */
#define PKD_FLAG_FMA_CONSUMER 1u
#define PKD_FLAG_MMA_CONSUMER 2u
/* Shared-prefix context (FlashInfer 完全拆解, Composable Format: a shared
 * prefix as an (R, 1) block so R queries reuse one read of its KV): plans made
 * with pkd_plan_shared give work items over blocks of R = 16 / g requests of
 * one group, run by a decode kernel whose tensor-core tile holds all R x g
 * query rows of a KV head.  Not combinable with PKD_FLAG_FMA_CONSUMER.  The
 * workspace then holds R partial-state slots per item. */
#define PKD_FLAG_SHARED_PREFIX 4u
/* FP8 cache: the KV cache holds E4M3 values (one byte per element, same NHD
 * shape) with a per-call scale for K and one for V (pkd_run_scaled): the
 * attended key is k_scale * K and the value v_scale * V ("FlashInfer 完全拆解",
 * performance section: E4M3 KV in vLLM; applicability table: low-precision KV
 * needs a scale contract).  Tensor-core consumer only; not combinable with
 * PKD_FLAG_SHARED_PREFIX. */
#define PKD_FLAG_KV_FP8 8u
/* KV producer.  When the page size is a multiple of 16 and the consumer is
 * the tensor-core one, the decode kernel copies 16 tokens of K (or V) of all
 * KV heads per TMA tensor copy (a 5-D tensor map over the NHD cache, 128-byte
 * shared-memory swizzle); otherwise it copies one token row (all KV heads) per
 * bulk copy.  This flag forces the token-row copies.  Combinable with every
 * other flag. */
#define PKD_FLAG_ROW_COPIES 16u
/* Chunk rule.  By default the split chunk is the closed-form work bound
 * ceil(sum_i l_i / N_CTA) rounded up to whole pages (its half and quarter
 * are tried too, the smallest predicted makespan wins).  With this flag the
 * chunk is the largest page multiple, not below min_chunk_tokens, whose split
 * still gives at least N_CTA work items (binary search; pyshine FlashInfer
 * tour, "Planning on the Host, Executing on the Device", where the prefill
 * planner searches the KV chunk this way). */
#define PKD_FLAG_CHUNK_SEARCH 64u
/* HND cache layout: kv is [num_pages][2][Hkv][P][D] -- within a page, each KV
 * head's P token rows are contiguous -- instead of NHD [num_pages][2][P][Hkv][D]
 * ("FlashInfer 完全拆解", section 接口层最容易踩的四个坑: NHD and HND order the
 * last three dimensions differently; low-precision KV may prefer HND).  Same
 * results as NHD for the same values.  With page tiles (page size a multiple
 * of 16) only the tensor map changes; token-row copies become one copy per
 * token and KV head.  Combinable with every other flag. */
#define PKD_FLAG_HND 32u
/* Dense shared-prefix kernel (with PKD_FLAG_SHARED_PREFIX; bf16 cache, page
 * size a multiple of 16).  A shared prefix is a dense contraction: up to
 * 128 / g requests of a group read the same pages, so their 128 query rows
 * of one KV head form one 128-row tile ("FlashInfer 完全拆解", Composable
 * Format).  Plans then cut groups into blocks of 128 / g requests and give
 * every (block, KV head, chunk) its own work item; the kernel runs S = Q K^T
 * and O += P V on the 5th-generation tensor cores (tcgen05.mma, accumulators
 * in tensor memory), streaming the head's page tiles with TMA.  Not
 * combinable with PKD_FLAG_FMA_CONSUMER, PKD_FLAG_KV_FP8 or
 * PKD_FLAG_ROW_COPIES. */
#define PKD_FLAG_DENSE_PREFIX 128u
/* Cascade context ("FlashInfer, in depth", "Prefill, masks and shared
 * prefixes" and "Cascades, Merges, and the Autotuner": attention once per
 * prefix level, then one merge; "FlashInfer 完全拆解", Composable Format).
 * Plans made with pkd_plan_cascade hold both levels of a decode step: the
 * shared-prefix level (work items over one KV head of a block of up to
 * 128 / g requests, as PKD_FLAG_DENSE_PREFIX) and every request's own suffix
 * (work items over a request's token range, all KV heads, as pkd_plan).
 * pkd_run then launches one kernel whose first CTAs run the prefix items on
 * the 5th-generation tensor cores and whose other CTAs run the suffix items
 * on the decode path, side by side, every item writing a partial state; one
 * merge folds each request's prefix and suffix states into out / lse.  The
 * planner splits the grid between the levels by a cost model.  bf16 cache,
 * page size a multiple of 16; combinable with PKD_FLAG_HND and
 * PKD_FLAG_MMA_CONSUMER only. */
#define PKD_FLAG_CASCADE 256u

typedef struct pkd_ctx pkd_ctx;
typedef struct pkd_graph pkd_graph;

/* Summary of the last plan (host-side copy). */
typedef struct pkd_plan_info {
    int32_t batch;
    int32_t num_ctas;
    int32_t chunk_tokens;      /* chosen chunk (page multiple)             */
    int32_t num_items;
    int32_t num_units;         /* split requests                            */
    int32_t num_slots;         /* partial states in the workspace           */
    int64_t total_tokens;      /* sum of l_i                                */
    int64_t makespan;          /* predicted max per-CTA cost                */
    int32_t nnz;               /* pages referenced                          */
    int32_t schedule_words;    /* int32 words pkd_plan_host writes          */
    int32_t page_tiles;        /* 1: the context's decode kernel copies KV in
                                  16-token page tiles (tensor map); 0: one
                                  copy per token row (pkd_plan /
                                  pkd_plan_shared fill it; pkd_plan_host
                                  leaves it 0)                              */
    int32_t prefix_ctas;       /* cascade plans: CTAs given the shared-prefix
                                  level (0 otherwise)                       */
    int32_t prefix_chunk_tokens; /* cascade plans: that level's chunk        */
} pkd_plan_info;

/* Bytes of device workspace needed for this configuration.  With
 * num_ctas == 0 the grid size is read from the current CUDA device.  Returns
 * 0 when the configuration is invalid or the device query fails. */
size_t pkd_workspace_bytes(const pkd_config *cfg);

/* Create a context over a caller-owned device workspace (at least
 * pkd_workspace_bytes(cfg) bytes, 256-byte aligned, kept alive and at the
 * same address for the context's life: the schedule lives at fixed offsets
 * inside it so that captured launches stay valid).  Allocates pinned host
 * staging and two events.  Errors: INVALID_ARG, UNSUPPORTED_SHAPE,
 * WORKSPACE_TOO_SMALL, CUDA. */
int pkd_create(const pkd_config *cfg, void *d_workspace, size_t workspace_bytes,
               pkd_ctx **out);

/* Destroy a context (synchronizes with its pending staging copies). */
void pkd_destroy(pkd_ctx *ctx);

/* Plan one decode step.  Host arrays (int32): indptr[batch + 1],
 * indices[indptr[batch]], last_page_len[batch].  They are copied into
 * pinned staging before the call returns, so the caller may reuse them at
 * once; the schedule reaches the workspace by two cudaMemcpyAsync on
 * `stream`, the body and then the header, which carries the plan's epoch
 * word ((epoch - 1) mod (2^31 - 1) + 1); staging is double-buffered and
 * fenced by events.  batch may be 0.
 * On success *epoch (if not NULL) receives the new plan epoch (>= 1).
 * Errors: INVALID_ARG, BAD_TABLE, CAPACITY, CUDA. */
int pkd_plan(pkd_ctx *ctx, const int32_t *indptr, const int32_t *indices,
             const int32_t *last_page_len, int32_t batch, void *stream,
             uint64_t *epoch);

/* Plan a shared-prefix level (needs a context created with
 * PKD_FLAG_SHARED_PREFIX).  Requests group_indptr[j] .. group_indptr[j+1]-1
 * (group_indptr[0] = 0, strictly increasing, batch = group_indptr[num_groups])
 * all attend over group j's pages indices[indptr[j] .. indptr[j+1]) with
 * last_page_len[j] -- a CSR table over groups.  pkd_run then returns, for
 * every request and query head, the attention state (out, lse) over its
 * group's pages, to be combined with the request's own suffix state by
 * pkd_merge_states (FlashInfer 完全拆解, Composable Format; FlashInfer, in
 * depth, "Prefill, masks and shared prefixes").  Errors: as pkd_plan. */
int pkd_plan_shared(pkd_ctx *ctx, const int32_t *group_indptr, int32_t num_groups,
                    const int32_t *indptr, const int32_t *indices,
                    const int32_t *last_page_len, void *stream, uint64_t *epoch);

/* Plan a cascade step (needs a context created with PKD_FLAG_CASCADE): the
 * shared-prefix level and every request's own suffix in one schedule.
 * Requests group_indptr[j] .. group_indptr[j+1]-1 (group_indptr[0] = 0,
 * strictly increasing, batch = group_indptr[num_groups]) share group j's
 * prefix pages p_indices[p_indptr[j] .. p_indptr[j+1]) with p_last[j] tokens
 * in the last one; request r's own pages are s_indices[s_indptr[r] ..
 * s_indptr[r+1]) with s_last[r] (every request has at least one suffix
 * token).  Request r attends over its prefix then its suffix: pkd_run
 * returns out / lse over both, merged ("FlashInfer, in depth", "Prefill,
 * masks and shared prefixes": the shared pages once for all queries, each
 * suffix separately, one LSE combine).  Host arrays, int32, copied before
 * the call returns.  The page capacity (max_num_pages) covers both tables.
 * Errors: INVALID_ARG, BAD_TABLE, CAPACITY, CUDA. */
int pkd_plan_cascade(pkd_ctx *ctx, const int32_t *group_indptr, int32_t num_groups,
                     const int32_t *p_indptr, const int32_t *p_indices, const int32_t *p_last,
                     const int32_t *s_indptr, const int32_t *s_indices, const int32_t *s_last,
                     void *stream, uint64_t *epoch);

/* Format advice for a shared-prefix step ("FlashInfer 完全拆解", Composable
 * Format 只在复用足够大时占优: splitting off the shared prefix pays only when
 * the reuse is large enough).  For the same tables as pkd_plan_cascade (page
 * ids are not needed), predicts the GPU time per layer of the cascade plan
 * and of the single format -- every request over its whole table, prefix
 * pages then its own, planned by pkd_plan -- from each planner's predicted
 * makespan and the KV bytes each reads, time = a + b x makespan + c x MB
 * (constants fitted on GB300 over the pages' grid of prefix length x batch
 * and shorter prefixes), and picks the faster.  Host only,
 * no CUDA call; cfg is the cascade context's configuration (flags
 * PKD_FLAG_CASCADE, num_ctas >= 2, the grid the plans would use). */
typedef struct pkd_format_advice {
    int32_t use_cascade;       /* 1: the cascade plan is predicted faster   */
    int32_t prefix_ctas;       /* the cascade plan's prefix CTAs            */
    int64_t cascade_makespan;  /* cascade planner, suffix-token units       */
    int64_t single_makespan;   /* plain planner over whole requests, tokens */
    float cascade_us;          /* predicted microseconds per layer          */
    float single_us;
} pkd_format_advice;
int pkd_advise_format(const pkd_config *cfg, const int32_t *group_indptr, int32_t num_groups,
                      const int32_t *p_indptr, const int32_t *p_last, const int32_t *s_indptr,
                      const int32_t *s_last, pkd_format_advice *advice);

/* Summary of the current plan.  Errors: INVALID_ARG, NO_PLAN. */
int pkd_get_plan_info(const pkd_ctx *ctx, pkd_plan_info *info);

/* Attention for one layer with the current plan.
 *   q    : device bf16 [batch][Hq][D], contiguous, 16-byte aligned
 *   kv   : device bf16 [num_pages][2][P][Hkv][D] (NHD), 16-byte aligned
 *   out  : device bf16 [batch][Hq][D]
 *   lse  : device fp32 [batch][Hq] or NULL (natural-log LSE of the scaled
 *          scores)
 * expect_epoch: 0 accepts any plan, and the schedule must be ordered before
 * the launch by `stream` (planned on it, or an event).  Otherwise it must
 * equal the current plan's epoch (STALE_PLAN otherwise), and the kernels
 * also wait on the device, before reading the schedule, until its header
 * holds that epoch's word: the plan may then be uploaded on another stream
 * with no event between the two (the upload must not wait for this run).
 * That wait is bounded (about 2 s); when it runs out the decode kernel
 * does no work and ORs PKD_DEV_ERR_TIMEOUT into the device error word
 * (pkd_last_device_error), and out / lse are undefined.  Captured
 * graphs take expect_epoch 0.  Launches the decode kernel and the merge
 * kernel on `stream`, with programmatic dependent launch: the decode kernel
 * may start while the previous kernel in the stream runs and reads q and
 * the KV cache at once, so a kernel that writes them ahead of it in the same
 * stream must not release its dependents before it completes (kernels
 * launched without the programmatic attribute, such as pkd_append_kv's,
 * never do), and q and kv must not alias the out / lse of an earlier run
 * still in the stream; out, lse and the partial states are written only
 * after the previous kernel completes.
 * Errors: INVALID_ARG, NO_PLAN, STALE_PLAN, CUDA. */
int pkd_run(pkd_ctx *ctx, const void *q, const void *kv, void *out, float *lse,
            uint64_t expect_epoch, void *stream);

/* pkd_run with scales: scores use k_scale * K and the output v_scale * V
 * (lse is the log-sum-exp of the scaled scores).  Required for an FP8 cache
 * (PKD_FLAG_KV_FP8; kv then holds E4M3 bytes, [num_pages][2][P][Hkv][D]);
 * for bf16 any finite scales are allowed, pkd_run is (1, 1).
 * Errors: as pkd_run; INVALID_ARG for a non-finite scale. */
int pkd_run_scaled(pkd_ctx *ctx, const void *q, const void *kv, void *out, float *lse,
                   float k_scale, float v_scale, uint64_t expect_epoch, void *stream);

/* merge_states: for each of n x heads rows,
 *   m = max(s_a, s_b), w_a = exp(s_a - m), w_b = exp(s_b - m),
 *   v = (w_a v_a + w_b v_b) / (w_a + w_b), s = m + log(w_a + w_b)
 * (FlashInfer 完全拆解, 在线 Softmax 为什么允许任意切块; FlashInfer, in
 * depth, "Load balancing with split-KV").  s = -inf marks an empty state;
 * two empty states give v = 0, s = -inf.
 *   v_a, v_b, v_out : device bf16 [n][heads][head_dim], 16-byte aligned
 *   s_a, s_b, s_out : device fp32 [n][heads]
 * head_dim must be a multiple of 8.  v_out may alias v_a or v_b, s_out may
 * alias s_a or s_b.  Errors: INVALID_ARG, CUDA. */
int pkd_merge_states(const void *v_a, const float *s_a, const void *v_b,
                     const float *s_b, void *v_out, float *s_out, int32_t n,
                     int32_t heads, int32_t head_dim, void *stream);

/* append_paged_kv_cache: write n new tokens' K and V rows into their page
 * slots (pyshine FlashInfer tour, "The Paged KV Cache Layer"; the slot rule is
 * the page table's, FlashInfer, in depth, "The block-sparse page table").
 * Token i belongs to request b = batch_indices[i] at 0-based position
 * pos = positions[i] of the request's length after the append; its K row goes
 * to kv[indices[indptr[b] + pos / P]][0][pos % P] and its V row to [...][1][...].
 *   k_new, v_new         : device bf16 [n][Hkv][D], 16-byte aligned
 *   batch_indices, positions : device int32 [n]
 *   indptr [batch + 1], indices [indptr[batch]], last_page_len [batch] :
 *                          device int32, the table after the append
 *   kv                   : device bf16 [num_pages][2][P][Hkv][D] (NHD)
 *   err                  : device int32 word or NULL
 * A token whose request, position (outside 0..len-1) or page id (outside the
 * pool) is out of range is skipped and PKD_DEV_ERR_BOUNDS is OR-ed into *err;
 * nothing is written outside the cache.  Stream-ordered, no host sync.
 * Errors: INVALID_ARG, CUDA. */
int pkd_append_kv(const void *k_new, const void *v_new, const int32_t *batch_indices,
                  const int32_t *positions, int32_t n, const int32_t *indptr,
                  const int32_t *indices, const int32_t *last_page_len, int32_t batch,
                  void *kv, int32_t num_pages, int32_t page_size, int32_t num_kv_heads,
                  int32_t head_dim, int32_t *err, void *stream);

/* pkd_append_kv for other caches.  flags: PKD_FLAG_HND (kv is
 * [num_pages][2][Hkv][P][D]; the token's row of head h goes to
 * kv[page][0 or 1][h][pos % P]) and/or PKD_FLAG_KV_FP8 (one byte per element:
 * k_new, v_new and kv hold E4M3 bytes, copied as given -- quantising is the
 * caller's).  head_dim * element bytes must be a multiple of 16.  Other flags:
 * INVALID_ARG.  pkd_append_kv is this with flags 0. */
int pkd_append_kv_ex(const void *k_new, const void *v_new, const int32_t *batch_indices,
                     const int32_t *positions, int32_t n, const int32_t *indptr,
                     const int32_t *indices, const int32_t *last_page_len, int32_t batch,
                     void *kv, int32_t num_pages, int32_t page_size, int32_t num_kv_heads,
                     int32_t head_dim, uint32_t flags, int32_t *err, void *stream);

/* pkd_append_kv_ex for every layer of a step in one launch: the layers share
 * the step's tokens and page table (batch_indices, positions, indptr,
 * indices, last_page_len, as in pkd_append_kv), and layer l's rows
 * k_new[l] / v_new[l] ([n][Hkv][D] each) go into cache kv[l].  k_new, v_new
 * and kv are HOST arrays of `layers` device pointers (1 <= layers <= 128),
 * read before the call returns; every layer's cache has the same shape and
 * flags.  Tokens outside the table are skipped in every layer and flagged
 * once in *err.  Errors: INVALID_ARG (as pkd_append_kv_ex, layers out of
 * range, a null or misaligned pointer), CUDA. */
int pkd_append_kv_layers(int32_t layers, const void *const *k_new, const void *const *v_new,
                         void *const *kv, const int32_t *batch_indices,
                         const int32_t *positions, int32_t n, const int32_t *indptr,
                         const int32_t *indices, const int32_t *last_page_len, int32_t batch,
                         int32_t num_pages, int32_t page_size, int32_t num_kv_heads,
                         int32_t head_dim, uint32_t flags, int32_t *err, void *stream);

/* Self-test of the device-side bounded waits (failure detection without a
 * GPU fault; FlashInfer, in depth, "Failure modes in production": errors come
 * back as status, never as a hang).  Launches one small kernel on `stream`
 * whose waits, on barriers nothing arrives on, use the same bounded wait as
 * the decode and prefix kernels: with mode 0 one wait runs out its limit
 * (about 2 s) and ORs PKD_DEV_ERR_TIMEOUT into *d_err; with mode 1 a second
 * waiter, started half a limit later, must stop on the first one's abort
 * flag instead of running out its own limit.  d_err (int32) and d_wait_ns
 * (2 x uint64: each wait's duration, 0 for a wait that was not run) are
 * device pointers owned by the caller, who zeroes *d_err and synchronizes
 * before reading them.  Errors: INVALID_ARG (mode not 0 or 1, null pointer),
 * CUDA (launch failed). */
int pkd_selftest_bounded_wait(int32_t mode, int32_t *d_err, unsigned long long *d_wait_ns,
                              void *stream);

/* Read and clear the context's device error word: the read and the reset
 * are ordered on `stream` after the work already in it, and the call waits
 * for `stream` only (work on other streams keeps running).  *dev_err
 * receives PKD_DEV_ERR_* bits (0 = none).  Errors: INVALID_ARG, CUDA. */
int pkd_last_device_error(pkd_ctx *ctx, void *stream, int32_t *dev_err);

/* Copy the schedule in the device workspace back to the host (test aid;
 * synchronizes `stream`).  Writes the same words pkd_plan_host produces. */
int pkd_read_schedule(pkd_ctx *ctx, int32_t *host_words, size_t max_words,
                      void *stream);

/* The planner alone, on the host, without CUDA: validates the table and
 * writes the schedule words for `num_ctas` CTAs into host_words (layout:
 * see pkd_schedule_layout).  cfg->num_ctas must be > 0.  Errors:
 * INVALID_ARG, BAD_TABLE, CAPACITY. */
int pkd_plan_host(const pkd_config *cfg, const int32_t *indptr,
                  const int32_t *indices, const int32_t *last_page_len,
                  int32_t batch, int32_t *host_words, size_t max_words,
                  pkd_plan_info *info);

/* pkd_plan_host for a shared-prefix plan (cfg->flags has
 * PKD_FLAG_SHARED_PREFIX; arguments as pkd_plan_shared). */
int pkd_plan_host_shared(const pkd_config *cfg, const int32_t *group_indptr,
                         int32_t num_groups, const int32_t *indptr, const int32_t *indices,
                         const int32_t *last_page_len, int32_t *host_words,
                         size_t max_words, pkd_plan_info *info);

/* pkd_plan_host for a cascade plan (cfg->flags has PKD_FLAG_CASCADE;
 * arguments as pkd_plan_cascade). */
int pkd_plan_host_cascade(const pkd_config *cfg, const int32_t *group_indptr,
                          int32_t num_groups, const int32_t *p_indptr,
                          const int32_t *p_indices, const int32_t *p_last,
                          const int32_t *s_indptr, const int32_t *s_indices,
                          const int32_t *s_last, int32_t *host_words, size_t max_words,
                          pkd_plan_info *info);

/* Word offsets of the schedule arrays (see pkd_plan_host):
 *   off[0] cta_indptr[num_ctas + 1]
 *   off[1] items[num_items][8] = {req, tok_begin, tok_end, dst_slot,
 *                                 first_page, n_req, slot_stride, 0}
 *          (items of CTA c are items[cta_indptr[c] .. cta_indptr[c+1]) in
 *          LPT order; the item covers requests req .. req + n_req - 1 (1
 *          without grouping); dst_slot -1 = write through to out/lse, else
 *          request req + i writes slot dst_slot + i * slot_stride;
 *          first_page = indptr[table row] + tok_begin / P, an index into
 *          page_list; cascade plans: prefix items have slot stride -1 and
 *          dst_slot = their chunk index, request req + i writing slot
 *          merge_indptr[req + i] + dst_slot; the page list holds the prefix
 *          table's indices, then the suffix table's)
 *   off[2] units[num_units][2] = {req, num_chunks}
 *   off[3] merge_indptr[num_units + 1]
 *   off[4] page_list[nnz]    (the CSR indices, unchanged)
 *   off[5] total words
 * Header words 0..31 hold: magic, batch, Hq, Hkv, D, P, num_ctas,
 * num_items, num_units, num_slots, chunk, alpha, nnz, makespan (clamped to
 * int32), split floor, requests per block, the most chunks of any split
 * request, the max_batch and max_num_pages the offsets were laid out for,
 * (cascade plans) the CTAs of the prefix level and its chunk, the plan's
 * epoch word (in a context's workspace; 0 in host-only plans), then zeros.
 * Errors: INVALID_ARG. */
int pkd_schedule_layout(const pkd_config *cfg, int64_t off[6]);

/* ---- CUDA-graph capture of a whole decode step ------------------------- */
/* Capture `layers` pkd_run calls (the current plan's workspace is read at
 * replay time, so re-planning between replays is allowed as long as batch
 * and capacities fit) into a graph.  Arrays of device pointers, one per
 * layer; kv_scales: NULL or host floats {k_scale, v_scale} per layer.  flags: PKD_GRAPH_TIMING records an event before and after each
 * layer's decode kernel, readable with pkd_graph_layer_times.
 * Errors: INVALID_ARG, NO_PLAN, CUDA. */
#define PKD_GRAPH_TIMING 1u
int pkd_graph_capture(pkd_ctx *ctx, int32_t layers, const void *const *q,
                      const void *const *kv, void *const *out,
                      float *const *lse, const float *kv_scales, uint32_t flags,
                      pkd_graph **graph);
/* pkd_graph_capture with the step's host I/O in the graph: q_host[l]
 * (page-locked host memory, the layer's [batch][Hq][D] bf16 queries) is
 * copied to q[l] before layer l runs, and out[l] / lse[l] are copied back to
 * out_host[l] / lse_host[l] (page-locked) after it.  The copies run on their
 * own captured streams: every layer's query copy may start when the graph
 * starts, and each layer's results leave while later layers compute.  Any of
 * q_host, out_host, lse_host may be NULL (no copy of that kind); lse_host
 * needs lse.  Sizes come from the plan current at capture (its batch).
 * Errors: INVALID_ARG, NO_PLAN, CUDA (also for host memory that is not
 * page-locked). */
int pkd_graph_capture_io(pkd_ctx *ctx, int32_t layers, const void *const *q,
                         const void *const *kv, void *const *out, float *const *lse,
                         const float *kv_scales, const void *const *q_host,
                         void *const *out_host, float *const *lse_host, uint32_t flags,
                         pkd_graph **graph);
/* Launch the captured step on `stream`.  Errors: INVALID_ARG, CUDA. */
int pkd_graph_launch(pkd_graph *graph, void *stream);
/* After the launch has completed: decode-kernel milliseconds per layer
 * (ms[layers]) of the most recent launch.  Errors: INVALID_ARG, CUDA. */
int pkd_graph_layer_times(pkd_graph *graph, float *ms);
void pkd_graph_destroy(pkd_graph *graph);

/* ---- allocation-free variant ------------------------------------------- */
/* No counterpart on the pages: this entry point exists for callers that may
 * not allocate device memory at all -- an engine whose allocator owns every
 * byte of the GPU and forbids libraries from calling cudaMalloc, a process
 * under a hard memory cap, or a plugin given no allocator.  Such callers
 * cannot provide the workspace that pkd_create needs.
 *
 * pkd_run_static_scratch runs one layer (decode kernel + merge of split
 * chunks, the same kernels as pkd_run) with the schedule and the partial
 * states in a static 32 MiB device array inside this library (held by every
 * GPU that loads the library until the process exits).  It calls no
 * allocator: no cudaMalloc / cudaFree / cudaMallocHost, no pkd_create.  Its
 * decode kernel copies KV one token row per bulk copy (the producer pkd_run
 * uses when page tiles are off), since it keeps no tensor maps.
 *   cfg            : the configuration (no flags but the consumer ones);
 *                    cfg->num_ctas must be > 0 and equal the value the
 *                    schedule was planned for
 *   schedule_words : host buffer written by pkd_plan_host(cfg, ...) for this
 *                    step (num_words = its length, >= page_list offset + nnz).
 *                    It is checked before use: planned for this cfg (shape,
 *                    CTA count, max_batch and max_num_pages, which fix the
 *                    word offsets), queues, requests, pages and partial-state
 *                    slots all in range.  It is copied with cudaMemcpyAsync
 *                    on `stream`; from pageable memory that copy is staged
 *                    before the call returns, from page-locked memory it is
 *                    asynchronous and the buffer must stay unchanged until
 *                    the stream has passed it.
 *   q, kv, out, lse: as for pkd_run
 * The whole layout for cfg (make sure max_batch / max_num_pages are not
 * larger than needed) must fit the 32 MiB array, else PKD_E_SCRATCH_LIMIT.
 * All calls share the array and it keeps the last call's contents (the
 * device error word is cleared at the start of each call); calls whose GPU
 * work overlaps race, so serialise them on one stream.  The first call on a
 * device sets the device up (looks up the array's address and the kernel
 * attribute) with that device current; make it before any stream capture.
 * Device-side errors (a page id outside the pool, a bounded wait that gave
 * up) land in the array's error word: read them with
 * pkd_static_scratch_last_error.
 * Errors: INVALID_ARG (null / misaligned pointer, schedule not matching cfg),
 * UNSUPPORTED_SHAPE, SCRATCH_LIMIT, CUDA. */
int pkd_run_static_scratch(const pkd_config *cfg, const int32_t *schedule_words,
                           size_t num_words, const void *q, const void *kv,
                           void *out, float *lse, void *stream);

/* Read and clear the device error word of the static array for the layout
 * of cfg (the word the last pkd_run_static_scratch call with this cfg
 * cleared and its kernels set): a stream-ordered read, then the reset, then
 * a wait for `stream` only.  Allocates nothing.  *dev_err receives
 * PKD_DEV_ERR_* bits (0 = none).  Errors: INVALID_ARG, UNSUPPORTED_SHAPE,
 * SCRATCH_LIMIT (cfg as for pkd_run_static_scratch), CUDA. */
int pkd_static_scratch_last_error(const pkd_config *cfg, void *stream, int32_t *dev_err);

/* Human-readable name of a status code. */
const char *pkd_status_str(int status);

/* Library version (major * 10000 + minor * 100 + patch). */
int pkd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKD_H_ */
