/*
 * psd.h - paged split-KV decode for one NVIDIA GB300 (sm_103a): the C ABI.
 *
 * Operations (mlxcel PR #1004, "compute shared prompt prefixes once per decode
 * batch"; ROCm ATOM PR #1701 section 3.2 for fp8 latent KV):
 *   paged_decode_partial  split-KV partial attention; one (V, LSE) row per work item
 *                         and query head, LSE in log2 units (Merge contract section)
 *   merge_states          log2-LSE merge of contiguous rows grouped by o_indptr
 *                         (Merge contract section)
 *   detect_shared_prefix  host: pick one subgroup sharing a whole-page prefix
 *                         (Detection section, Task item 1)
 *   build_cascade_plan    host: level-0 / level-1 work lists and merge groups
 *                         (Task item 2)
 *   cascade_decode        device: level 0 with KV-head-major stacked queries,
 *                         level 1, and the exact merge (Decomposition section)
 *
 * Conventions shared by every entry point
 *   - Every function returns psd_status; nothing throws or aborts across the ABI.
 *     On failure psd_last_error() returns a thread-local message.
 *   - "device" pointers are CUDA global memory on the context's device; "host"
 *     pointers are ordinary CPU memory.  All buffers are owned by the caller.  The
 *     decode, merge, planning and append entry points allocate no device memory:
 *     scratch lives in a caller-provided workspace sized by psd_workspace_bytes()
 *     (or, for cascade_decode_no_alloc, in the library's own fixed array).  The one
 *     exception is psd_autotune_tile, which allocates its L2-flush buffer once per
 *     context (freed by psd_destroy).
 *   - Device work is enqueued asynchronously on the caller's stream (NULL = the
 *     legacy default stream).  Host arrays passed in may be reused as soon as the
 *     call returns.
 *   - A batch of 0 requests is valid and does no device work; q and the outputs
 *     may then be NULL.
 *   - Host validation (shapes, page table, page ids < num_pages, alignment) runs
 *     before any launch and returns PSD_ERR_INVALID_ARG.  Kernels re-check page
 *     ids; a bad id or an expired bounded wait sets a flag in the workspace that
 *     psd_check_device_error() reports as PSD_ERR_DEVICE_FAULT.  No kernel traps.
 *
 * Layouts (row-major, innermost last)
 *   q        [B, Hq, Dqk]                 bf16
 *   k_pool   [num_pages, page_size, Hkv, Dqk]  bf16 or fp8-e4m3 codes
 *   v_pool   [num_pages, page_size, Hkv, Dv]   same dtype; or v_pool == k_pool with
 *            Hkv == 1 and Dv <= Dqk: V is the first Dv columns of the K rows (an MLA
 *            latent shared by K and V)
 *   partial  v [N, Hq, Dv] f32 normalised per row, lse [N, Hq] f32 (log2)
 *   page table (CSR): page_indptr [B+1], page_indices [nnz], last_page_len [B];
 *            request b has n_b = page_indptr[b+1]-page_indptr[b] >= 1 pages and
 *            L_b = (n_b - 1) * page_size + last_page_len[b] tokens,
 *            1 <= last_page_len[b] <= page_size.
 *   Query head h reads KV head h / (Hq / Hkv) (Decomposition section).
 *   fp8-e4m3 elements decode to code * k_scale (K) and code * v_scale (V).
 */
#ifndef PSD_H
#define PSD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *psd_stream_t; /* identical to cudaStream_t */

typedef enum {
  PSD_OK = 0,
  PSD_ERR_INVALID_ARG = 1,
  PSD_ERR_UNSUPPORTED = 2,
  PSD_ERR_CUDA = 3,
  PSD_ERR_DEVICE_FAULT = 4,
  PSD_ERR_WORKSPACE_TOO_SMALL = 5
} psd_status;

typedef enum { PSD_BF16 = 0, PSD_FP8_E4M3 = 1 } psd_dtype;

/* Why a cascade was not taken (Path attribution section: CascadeFailed(reason)). */
typedef enum {
  PSD_DECLINE_NONE = 0,                /* cascade taken */
  PSD_DECLINE_DISABLED = 1,            /* switched off by argument or environment */
  PSD_DECLINE_NO_SHARED_PAGES = 2,     /* no two multi-page requests share a first page */
  PSD_DECLINE_MEMBERS_BELOW_THRESHOLD = 3,
  PSD_DECLINE_SPAN_BELOW_THRESHOLD = 4 /* includes spans capped below the threshold */
} psd_decline_reason;

/* Device-fault flag bits written by kernels into the workspace's fault word (its
 * first 8 bytes, tagged with the call that wrote them; psd_check_device_error). */
enum {
  PSD_FAULT_PAGE_ID = 1,      /* a page id outside [0, num_pages) was skipped */
  PSD_FAULT_WAIT_TIMEOUT = 2, /* a bounded barrier wait gave up */
  PSD_FAULT_RANGE = 4         /* an index outside the range an operation accepts
                                 (a RoPE position past the cos/sin table) */
};

/* CSR page table (Detection section: PagedCsrView).  Host or device arrays. */
typedef struct {
  const int32_t *page_indptr;   /* [batch + 1] */
  const int32_t *page_indices;  /* [page_indptr[batch]] */
  const int32_t *last_page_len; /* [batch] */
  int32_t batch;
  int32_t page_size;
} psd_page_table;

/* One split-KV unit: a (request, page tile) pair (Decomposition section).
 *   q_index  request whose query rows are used; -1 = the stacked level-0 request
 *   page_off position in page_indices of the tile's first page
 *   n_tokens tokens in the tile (1..tile_tokens)
 *   out_row  partial row written (level 0: chunk index within the shared span) */
typedef struct {
  int32_t q_index;
  int32_t page_off;
  int32_t n_tokens;
  int32_t out_row;
} psd_work_item;

/* Problem description shared by paged_decode_partial and cascade_decode.
 * q and page_indices_dev may also be pinned host memory (cudaHostAlloc or
 * cudaHostRegister, same pointer on host and device).  The partial kernels then read
 * the query rows and page ids over the host link as they run.  No separate
 * host-to-device copy is needed, and a step reads each query row once per work item
 * and KV head.  The host must not write them until the call's stream work has
 * finished.  The MLA latent kernel loads q by TMA and takes device q only; with host
 * q it returns PSD_ERR_UNSUPPORTED before it launches. */
typedef struct {
  const void *q;                   /* [batch, Hq, Dqk] bf16, device or pinned host */
  const void *k_pool;              /* device [num_pages, page_size, Hkv, Dqk] */
  const void *v_pool;              /* device [num_pages, page_size, Hkv, Dv], or k_pool */
  const int32_t *page_indices_dev; /* the page table's page_indices, device or pinned host */
  int64_t num_page_indices;        /* length of page_indices_dev (nnz) */
  int64_t num_pages;
  int32_t batch, Hq, Hkv, Dqk, Dv, page_size;
  int32_t kv_dtype;                /* psd_dtype */
  float k_scale, v_scale;          /* fp8 dequant scales; ignored for bf16 */
  float sm_scale;                  /* softmax scale, e.g. 1/sqrt(Dqk) */
} psd_decode_args;

/* A decode plan: flat (num_members == 0) or two-level cascade.  The caller owns
 * every array and sets the capacities; psd_plan_capacity() gives them. */
typedef struct {
  /* capacities (in) */
  int32_t batch_capacity;      /* >= batch */
  int32_t item_capacity;       /* >= page_indptr[batch] (each item holds >= 1 page) */
  int32_t *members;            /* [batch_capacity] member requests, increasing */
  int32_t *member_row_base;    /* [batch_capacity] first merge row of each member */
  psd_work_item *l0_items;     /* [item_capacity] level-0 chunks of the shared span */
  psd_work_item *l1_items;     /* [item_capacity] level-1 (or flat) chunks */
  int32_t *o_indptr;           /* [batch_capacity + 1] final merge groups */
  /* results (out) */
  int32_t batch, page_size, tile_tokens;
  int32_t num_members, shared_pages, decline_reason;
  int32_t l0_num_items, l1_num_items;
  int32_t num_rows;            /* total partial rows = o_indptr[batch] */
} psd_cascade_plan;

/* Which path a cascade_decode call took (Path attribution section:
 * PagedDecodeOutcome::FusedCascade / CascadeFailed). */
typedef struct {
  int32_t path; /* 0 flat, 1 cascade */
  int32_t decline_reason;
  int32_t batch, members, shared_pages, shared_tokens;
  int32_t prefix_chunks, suffix_chunks;
} psd_cascade_stats;

/* In-context counters (Task item 5, without a metrics server).  lists_inline /
 * lists_uploaded count decode calls whose work lists travelled in the kernel
 * launches' parameters / by one host-to-device copy into the workspace. */
typedef struct {
  int64_t launches_flat, launches_cascade;
  int64_t cascade_shared_tokens, cascade_member_sequences, cascade_failures;
  int64_t lists_inline, lists_uploaded;
} psd_counters;

typedef struct psd_ctx psd_ctx;

/* ----------------------------------------------------------------- context */
/* Create a context bound to CUDA device `device` (queries SM count, loads the
 * driver's tensor-map encoder).  Host memory only.  Thread-compatible: one
 * context per thread, or external locking. */
psd_status psd_create(psd_ctx **ctx, int device);
psd_status psd_destroy(psd_ctx *ctx);
/* Which kernel computes partials on bf16 pools with separate K and V.  AUTO and
 * TENSOR_CORE: the 16-row-group tensor-core kernel (QK^T and PV as m16n8k16
 * MMAs; the stacked level-0 rows are split into groups of 16, or into 64-row
 * blocks that read each K/V tile once when those blocks fill a wave of the GPU).  CUDA_CORE: the
 * CUDA-core kernel wherever it applies (G <= 8 rows per KV head; warp-shuffle
 * reductions and f32x2 FMAs).  Both compute the same partials.  fp8 pools with
 * separate K and V (head dims 64, 128, 256) use the 64-row mma.sync kernel; the
 * fp8 MLA latent (128 heads over a 576-wide latent, V its first 512 columns) uses
 * the tcgen05 kernel, or the 64-row kernel when CUDA_CORE is selected. */
typedef enum { PSD_KERNEL_AUTO = 0, PSD_KERNEL_CUDA_CORE = 1, PSD_KERNEL_TENSOR_CORE = 2 } psd_partial_kernel;
psd_status psd_set_partial_kernel(psd_ctx *ctx, int32_t kind);
/* Which kernel computes the stacked level-0 rows of a cascade (mlxcel PR #1004,
 * Decomposition: the M members' G query heads of one KV head, KV-head major) on bf16
 * pools with separate K and V.  TCGEN05: a persistent kernel on the 5th-generation
 * tensor cores, one CTA per SM over (level-0 chunk, KV head, block of up to 128
 * stacked rows) tasks (head dims 64 and 128, page sizes that are multiples of 16, a
 * positive softmax scale), launched before level 1 on a second
 * stream.  MMA_SYNC: the 16-row-group tensor-core kernel, sharing one launch with
 * level 1.  AUTO (the default): TCGEN05 from 32 stacked rows per KV head where it
 * applies and level 0 holds at least two (chunk, KV head, 128-row) tasks per SM,
 * unless the CUDA-core partial kernel is selected.  Both compute the same
 * partials. */
typedef enum { PSD_LEVEL0_AUTO = 0, PSD_LEVEL0_MMA_SYNC = 1, PSD_LEVEL0_TCGEN05 = 2 } psd_level0_kernel;
psd_status psd_set_level0_kernel(psd_ctx *ctx, int32_t kind);
/* Kernel timing, for measurement: when enabled, paged_decode_partial and
 * cascade_decode record CUDA events around each kernel they launch, on the
 * stream that kernel runs on.  psd_get_kernel_times waits for the most recent
 * call's events and returns the level-0 partial, the level-1 (or flat) partial
 * and the merge kernel durations in milliseconds (0 for a kernel the call did not
 * launch; any pointer may be NULL).  Enabling creates the events (host-side CUDA
 * objects, no device memory). */
psd_status psd_set_timing(psd_ctx *ctx, int32_t enable);
/* Testing aid for the kernels' bounded waits (no counterpart on the pages).  With
 * from_tile >= 0, the 16-row-group tensor-core, CUDA-core, tcgen05 level-0 and MLA
 * partial kernels launched through this context issue no loads for any item's tiles
 * at index from_tile and later (16-token tiles of the tensor-core kernel, the
 * CUDA-core kernel's own ring tiles, the 64-token tiles of the tcgen05 kernels), so
 * their waits for those tiles run out after wait_limit_cycles (1e5 to 2e9 SM
 * cycles); each timed-out warp stops consuming tiles, the kernel completes, and the
 * call's fault word carries PSD_FAULT_WAIT_TIMEOUT for psd_check_device_error.
 * Every copy a kernel did issue is waited for before it exits, and the tcgen05
 * kernels free their tensor memory only after their issued MMAs have completed.
 * The streaming form of psd_merge_states copies no input row from index from_tile
 * of a CTA's range on; its output rows from the first one that needs such a row to
 * the end of the CTA's range read as NaN (v and LSE: a merge has no fault word).
 * Outputs of such a call are meaningless.  from_tile < 0 switches the aid off (the
 * default; the other kernels ignore it).  PSD_ERR_INVALID_ARG for a limit outside
 * the range. */
psd_status psd_test_withhold_loads(psd_ctx *ctx, int32_t from_tile, int64_t wait_limit_cycles);
psd_status psd_get_kernel_times(psd_ctx *ctx, float *level0_ms, float *partial_ms, float *merge_ms);
/* Thread-local message describing the last failure on this thread. */
const char *psd_last_error(void);
psd_status psd_get_counters(const psd_ctx *ctx, psd_counters *out);
/* Kill switch (Task item 4): reads PSD_CASCADE_ATTENTION; 0/false/off/no -> 0,
 * 1/true/on/yes -> 1, unset or anything else -> `fallback`. */
int32_t psd_cascade_env_enabled(int32_t fallback);

/* ------------------------------------------------------------ host planning */
/* Flat split-KV work list (Decomposition: one unit per (request, page tile)).
 * Request b gets ceil(L_b / tile_tokens) items; item c starts at page position
 * page_indptr[b] + c*tile_tokens/page_size and writes row o_indptr[b] + c.
 * host: host page table.  items: [item_capacity] host.  o_indptr: [batch+1] host.
 * tile_tokens must be a positive multiple of page_size. */
psd_status psd_split_plan(const psd_page_table *host, int32_t tile_tokens,
                          psd_work_item *items, int32_t item_capacity,
                          int32_t *num_items, int32_t *o_indptr);

/* Shared-prefix detection (Detection section; Task items 1 and 4; Left out /
 * unsure).  Requests with >= 2 pages are grouped by first page id; a group with
 * >= max(2, min_members) requests gets span = longest positional common page
 * prefix over all its members, capped at min(n_b) - 1 so no member's last page is
 * shared; spans >= max(1, min_shared_pages) compete on span * (members - 1), ties
 * to the group with the smallest first member.  Outputs (host): members [batch]
 * in increasing order, *num_members (0 on decline), *shared_pages,
 * *decline_reason (psd_decline_reason).  Deterministic and bit-exact. */
psd_status detect_shared_prefix(const psd_page_table *host, int32_t min_shared_pages,
                                int32_t min_members, int32_t *members,
                                int32_t *num_members, int32_t *shared_pages,
                                int32_t *decline_reason);

/* Cascade plan (Task item 2).  Level 0: the first shared_pages pages of members[0]
 * (identical pool pages for every member) split into tile_tokens chunks, items
 * with q_index -1 and out_row = chunk index.  Level 1: every request, members
 * starting after the span, non-members whole.  Merge group of request b: its
 * level-0 rows (members only; row member_row_base[m] + chunk) then its level-1
 * rows.  num_members == 0 gives the flat plan.  plan arrays are host memory. */
psd_status build_cascade_plan(const psd_page_table *host, const int32_t *members,
                              int32_t num_members, int32_t shared_pages,
                              int32_t tile_tokens, psd_cascade_plan *plan);

/* detect_shared_prefix + build_cascade_plan, or the flat plan with the decline
 * reason.  enable: 1 on, 0 off, -1 = psd_cascade_env_enabled(0). */
psd_status psd_plan_decode(const psd_page_table *host, int32_t tile_tokens, int32_t enable,
                           int32_t min_shared_pages, int32_t min_members,
                           psd_cascade_plan *plan);

/* Capacities a plan for this page table needs. */
psd_status psd_plan_capacity(const psd_page_table *host, int32_t *batch_capacity,
                             int32_t *item_capacity);

/* Plan cache (mlxcel PR #1004, Left out / unsure: detection re-runs per layer and
 * per step; a cascade-plan entry in the plan cache is the named follow-up).  The key
 * is everything psd_plan_decode reads: the resolved enable switch, both thresholds,
 * tile_tokens, page_size, batch and the full contents of page_indptr, page_indices
 * and last_page_len, since a split-KV plan depends on KV lengths as well as on the
 * page rows (FreeToken issue #750, Layer-major prefill for offloaded MoE, Attention
 * batching section: a cache keyed by rows alone was a bug).  A hit returns exactly
 * the plan psd_plan_decode would compute.
 *
 * The cache owns its plans: `capacity` entries in [1, 1024], least recently used
 * evicted.  It is host-only, allocates host memory only, and is not thread-safe (one
 * cache per thread).  psd_plan_cache_destroy(NULL) is a no-op. */
typedef struct psd_plan_cache psd_plan_cache;
psd_status psd_plan_cache_create(psd_plan_cache **cache, int32_t capacity);
psd_status psd_plan_cache_destroy(psd_plan_cache *cache);
/* Looks `host` up, planning it on a miss (same arguments and errors as
 * psd_plan_decode; an invalid table is rejected before its arrays are read).
 * *plan points into the cache and stays valid until the next lookup on this cache or
 * its destruction; *hit (nullable) is 1 when no planning ran. */
psd_status psd_plan_cache_lookup(psd_plan_cache *cache, const psd_page_table *host,
                                 int32_t tile_tokens, int32_t enable, int32_t min_shared_pages,
                                 int32_t min_members, const psd_cascade_plan **plan, int32_t *hit);
/* As psd_plan_cache_lookup, with a caller-kept generation number for the page table
 * (e.g. one per decode step, shared by every layer).  When generation >= 0 and an
 * entry was stored or last matched under the same generation with the same
 * tile_tokens, resolved enable, thresholds and batch, that entry is returned without
 * reading the table's arrays: O(1) instead of O(page ids).  The caller must change
 * the generation whenever any array of the table changes; reusing a generation for a
 * different table returns that generation's plan.  generation < 0 is
 * psd_plan_cache_lookup. */
psd_status psd_plan_cache_lookup_gen(psd_plan_cache *cache, int64_t generation,
                                     const psd_page_table *host, int32_t tile_tokens,
                                     int32_t enable, int32_t min_shared_pages, int32_t min_members,
                                     const psd_cascade_plan **plan, int32_t *hit);
/* Lookups answered from the cache, lookups that planned, and live entries (all nullable). */
psd_status psd_plan_cache_stats(const psd_plan_cache *cache, int64_t *hits, int64_t *misses,
                                int32_t *entries);

/* Workspace bytes for cascade_decode / paged_decode_partial: work lists and
 * merge groups for up to `num_items` items and `batch` requests, plus partial
 * rows `num_rows` x Hq x Dv (pass 0 rows for paged_decode_partial). */
size_t psd_workspace_bytes(int32_t batch, int32_t num_items, int64_t num_rows, int32_t Hq,
                           int32_t Dv);

/* ---------------------------------------------------------------- device ops */
/* Split-KV partial attention (Decomposition and Merge contract sections).
 * For every item i and query head h, over the item's tokens j:
 *   t_j = sm_scale * <q[item.q_index, h], k_j> * log2(e),  m = max_j t_j,
 *   l = sum_j 2^(t_j - m),  v_out[item.out_row, h] = sum_j 2^(t_j - m) v_j / l,
 *   lse_out[item.out_row, h] = m + log2(l).
 * One CTA owns all G = Hq/Hkv query heads of one KV head for one item, so each
 * K/V element is read from HBM once.  items: host [num_items] with q_index in
 * [0, batch).  v_out: device [out_rows, Hq, Dv] f32.  lse_out: device
 * [out_rows, Hq] f32.  workspace: device, >= psd_workspace_bytes(batch,
 * num_items, 0, Hq, Dv) bytes, 16-byte aligned. */
psd_status paged_decode_partial(psd_ctx *ctx, const psd_decode_args *args,
                                const psd_work_item *items, int32_t num_items,
                                float *v_out, float *lse_out, int64_t out_rows,
                                void *workspace, size_t workspace_bytes,
                                psd_stream_t stream);

/* Log2-LSE merge (Merge contract section).  For output row r and head h over rows
 * i in [o_indptr[r], o_indptr[r+1]):  M = max lse_i, w_i = 2^(lse_i - M),
 *   v_out = sum w_i v_i / sum w_i,  lse_out = M + log2(sum w_i).
 * A one-row group copies v and lse bit-exactly; an empty or all -inf group
 * gives 0 and -inf.  A row whose lse is -inf is an empty partial (no tokens): its
 * weight is zero and its v is not used, whatever it holds.  v_in device [N, H, D] f32, lse_in device [N, H] f32,
 * o_indptr_dev device [num_out + 1] int32 (non-decreasing), v_out device
 * [num_out, H, D] f32, lse_out device [num_out, H] f32 or NULL.  D % 4 == 0,
 * D <= 1024; all pointers 16-byte aligned. */
psd_status merge_states(psd_ctx *ctx, const float *v_in, const float *lse_in,
                        const int32_t *o_indptr_dev, int64_t num_out, int32_t H,
                        int32_t D, float *v_out, float *lse_out, psd_stream_t stream);

/* Two-level cascade decode (Decomposition section; Task item 2), or flat decode
 * when plan->num_members == 0.  Level 0 attends the shared span once with the
 * members' query heads stacked KV-head-major (h0 = kv*(M*G) + m*G + g); level 1
 * attends every request's remaining tokens; merge_states combines each member's
 * level-0 and level-1 rows (and passes a non-member's single chunk group through).
 * o: device [batch, Hq, Dv] f32.  lse: device [batch, Hq] f32 (log2) or NULL.
 * o and lse may instead be pinned host memory (cudaHostAlloc / cudaHostRegister,
 * same pointer on host and device): the merge kernel then stores the outputs into
 * host memory over the host link, and they are readable once the stream has
 * synchronised; no separate device-to-host copy is needed.
 * workspace: >= psd_workspace_bytes(batch, plan item total, plan->num_rows, Hq, Dv).
 * stats (host, nullable) receives which path ran.  The work lists reach the GPU in
 * the launches' parameters when they fit (16 KB of items, order and members, and
 * batch < 1024) and every launch's kernel takes them there (the bf16 16-row-group
 * tensor-core kernel, and the tcgen05 kernel for the stacked level-0 rows);
 * otherwise by one copy from pinned staging into the workspace. */
psd_status cascade_decode(psd_ctx *ctx, const psd_decode_args *args,
                          const psd_cascade_plan *plan, float *o, float *lse,
                          void *workspace, size_t workspace_bytes,
                          psd_cascade_stats *stats, psd_stream_t stream);

/* cascade_decode for callers that cannot allocate device memory.  No counterpart
 * on the source pages: it exists for callers that run inside another runtime's
 * memory pool or a plugin sandbox and may not call cudaMalloc (or any allocator)
 * when they decode, so they cannot hand cascade_decode a workspace.  This entry
 * point takes the same inputs and outputs but keeps all scratch (work lists, the
 * fault word, the partial rows) in one fixed 16 MiB array in the library's own
 * device memory, present on every GPU that loads the library until the process
 * exits.  It calls no allocating routine (no cudaMalloc/cudaFree, no pinned host
 * buffer).
 *   - Plans whose scratch (psd_workspace_bytes of the plan) exceeds 16 MiB are
 *     rejected with PSD_ERR_WORKSPACE_TOO_SMALL and a message naming both sizes.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is kept for the life of the
 *     process: do not reset the device (cudaDeviceReset) while using this entry
 *     point.
 *   - Every call on a device shares the one array, which keeps the last call's
 *     contents; each call clears the fault word itself.  Calls whose device work
 *     overlaps (other streams, unordered host threads) race on the array.
 *   - The work lists are laid out and ordered as cascade_decode lays them out
 *     (longest items first, both levels in one launch where one kernel serves
 *     them).  When the 16-row-group tensor-core kernel runs every launch and the
 *     lists fit in its launch parameters (up to about 800 items and 1023
 *     requests), they travel there and the call makes no host-to-device copy;
 *     otherwise one cudaMemcpyAsync from pageable host memory places them in the
 *     array.
 *   - fault_bits_dev (device int32, nullable) receives the call's PSD_FAULT_* bits.
 * Results equal cascade_decode's on the same plan. */
psd_status cascade_decode_no_alloc(psd_ctx *ctx, const psd_decode_args *args,
                                   const psd_cascade_plan *plan, float *o, float *lse,
                                   int32_t *fault_bits_dev, psd_cascade_stats *stats,
                                   psd_stream_t stream);

/* ------------------------------------------------- several and nested shared spans
 * An extension the pages scope out (mlxcel PR #1004: Task item 1 keeps to a single
 * shared level; Left out / unsure lists nested sharing, a system prompt common to
 * all plus a per-tenant sub-prefix, as not attempted because it needs another
 * level).  Planning rules:
 *   every first-page group that passes the thresholds becomes a segment (not only
 *   the one with the most saved reads); inside a segment [start, start + span) its
 *   members are grouped again by their page at start + span and each group gets the
 *   same rules from there (span over all its members, capped so no member's last
 *   page is shared, min_shared_pages, min_members), up to max_levels levels;
 *   segments are listed depth first, groups in order of their lowest batch index.
 * Each segment is one stacked level-0 request (M_s * G rows per KV head, KV-head
 * major); request b's final merge group holds its segments' chunk rows in segment
 * order, then its level-1 rows, which start after its deepest segment.  With
 * max_levels = 1 and one qualifying group the plan equals psd_plan_decode's. */
typedef struct {
  int32_t first_member; /* into members[] and member_row_base[] */
  int32_t num_members;
  int32_t start_page;   /* page position of the span in every member's page list */
  int32_t shared_pages;
  int32_t first_item;   /* into l0_items[] */
  int32_t num_items;
} psd_segment;

typedef struct {
  /* capacities (in): psd_plan_nested_capacity gives them */
  int32_t batch_capacity;   /* >= batch */
  int32_t entry_capacity;   /* >= batch * max_levels ((segment, member) entries) */
  int32_t segment_capacity; /* >= batch * max_levels */
  int32_t item_capacity;    /* >= page_indptr[batch] */
  psd_segment *segments;
  int32_t *members;         /* [entry_capacity] each segment's members, increasing */
  int32_t *member_row_base; /* [entry_capacity] first partial row of each entry */
  psd_work_item *l0_items;  /* [item_capacity] span chunks, by segment; out_row = chunk */
  psd_work_item *l1_items;  /* [item_capacity] */
  int32_t *o_indptr;        /* [batch_capacity + 1] */
  /* results (out) */
  int32_t batch, page_size, tile_tokens, max_levels;
  int32_t num_segments, num_entries, decline_reason;
  int32_t l0_num_items, l1_num_items;
  int32_t num_rows;
} psd_nested_plan;

psd_status psd_plan_nested_capacity(const psd_page_table *host, int32_t max_levels,
                                    int32_t *batch_capacity, int32_t *entry_capacity,
                                    int32_t *segment_capacity, int32_t *item_capacity);
/* max_levels in [1, 8]; enable as in psd_plan_decode.  No segment: the flat plan
 * with psd_plan_decode's decline reason. */
psd_status psd_plan_nested(const psd_page_table *host, int32_t tile_tokens, int32_t enable,
                           int32_t min_shared_pages, int32_t min_members, int32_t max_levels,
                           psd_nested_plan *plan);
/* Workspace bytes cascade_decode_nested needs for this plan. */
size_t psd_nested_workspace_bytes(const psd_nested_plan *plan, int32_t Hq, int32_t Dv);
/* Decode with a nested plan: one stacked level-0 launch per segment, level 1, one
 * merge (stats->members counts (segment, member) entries and shared_pages sums the
 * spans).  Same arguments, errors and fault word as cascade_decode. */
psd_status cascade_decode_nested(psd_ctx *ctx, const psd_decode_args *args,
                                 const psd_nested_plan *plan, float *o, float *lse,
                                 void *workspace, size_t workspace_bytes,
                                 psd_cascade_stats *stats, psd_stream_t stream);

/* ------------------------------------------------------------ chunk-size tuning
 * mlxcel PR #1004, Left out / unsure: the shape-bucketed kernel autotuner with the
 * cold-L2 benchmark methodology is not wired to either cascade geometry; both plans
 * use the heuristic chunk size.  psd_autotune_tile times cascade_decode for each
 * candidate tile_tokens on the caller's batch (psd_plan_decode with `enable` and the
 * thresholds): one untimed call, then `reps` timed calls, each preceded by a cold-L2
 * flush (a 256 MB write, then a 256 MB read of another region, so that L2 holds no
 * input and no dirty line; the context allocates the 512 MB buffer once), timed with
 * CUDA events on `stream`; the call is synchronous.  The candidate with the lowest mean
 * is recorded under the batch's shape bucket: (Hq, Hkv, Dqk, Dv, kv_dtype,
 * page_size, batch and total tokens each rounded up to a power of two, whether the
 * plan cascades).  Candidates must be positive multiples of page_size; o, lse and
 * the workspace are as for cascade_decode and must fit every candidate (the
 * smallest tile has the most partial rows).  ms_out (nullable, [n_tiles]) receives
 * the means.  Unlike the decode entry points this call allocates (the flush
 * buffer, once per context). */
psd_status psd_autotune_tile(psd_ctx *ctx, const psd_decode_args *args, const psd_page_table *host,
                             const int32_t *tiles, int32_t n_tiles, int32_t enable,
                             int32_t min_shared_pages, int32_t min_members, int32_t reps, float *o,
                             float *lse, void *workspace, size_t workspace_bytes, psd_stream_t stream,
                             int32_t *best_tile, float *ms_out);
/* The tile recorded for this batch's shape bucket by psd_autotune_tile on this
 * context, or default_tile when none was (or the arguments are invalid). */
int32_t psd_tuned_tile(psd_ctx *ctx, const psd_decode_args *args, const psd_page_table *host,
                       int32_t enable, int32_t min_shared_pages, int32_t min_members,
                       int32_t default_tile);

/* ---------------------------------------------------------------- RoPE + append
 * The step before decode: the new token of each request is roped and appended to
 * the paged pool (ROCm ATOM PR #1701, section 1 and 3.3: one fused kernel ropes
 * every query and the new token's rope part of K, concatenates the non-rope latent
 * with it, and writes the KV row only for the slots this rank owns; 3.2: fp8 KV
 * dequantises as code * scale).
 *
 * Per token t (pos = positions[t], r = rot_dim, frequencies i < r/2 with
 * c_i = cos_sin[pos][i], s_i = cos_sin[pos][r/2 + i]):
 *   q[t, h, q_rope_col + a_i], q[t, h, q_rope_col + b_i] are rotated in place for
 *   every head h, where (a_i, b_i) = (i, i + r/2) when neox, else (2i, 2i + 1):
 *   x' = x c_i - y s_i, y' = y c_i + x s_i in f32, each product rounded, then bf16;
 *   if slot_mapping[t] >= 0 (slot = page * page_size + position in page), for every
 *   KV head: k_pool[slot] = [k_nope[t] | rope(k_rope[t]) on its first r columns]
 *   and v_pool[slot] = v[t], stored as bf16, or for PSD_FP8_E4M3 as the saturating
 *   round-to-nearest-even E4M3 code of value / scale (k_scale for K, v_scale for V).
 * A position outside [0, max_position) leaves token t untouched and sets
 * PSD_FAULT_RANGE; a slot >= num_pages * page_size skips its KV write and sets
 * PSD_FAULT_PAGE_ID, both in *fault_dev (device int32, caller-owned, OR-ed).
 * num_tokens == 0 is a no-op (the pointers are not checked). */
typedef struct {
  void *q;                     /* device [T, Hq, Dq] bf16, roped in place (NULL iff Hq == 0) */
  int32_t Hq, Dq, q_rope_col;
  const void *k_nope;          /* device [T, Hkv, Dk_nope] bf16 (NULL iff Dk_nope == 0) */
  const void *k_rope;          /* device [T, Hkv, Dk_rope] bf16 */
  int32_t Hkv, Dk_nope, Dk_rope;
  const void *v;               /* device [T, Hkv, Dv] bf16 (NULL iff Dv == 0: V is in the K row) */
  int32_t Dv;
  int32_t rot_dim;             /* even, >= 2, <= Dk_rope, q_rope_col + rot_dim <= Dq */
  int32_t neox;                /* 1: pairs (i, i + r/2); 0: pairs (2i, 2i + 1) */
  const float *cos_sin;        /* device [max_position, rot_dim] f32 */
  int32_t max_position;
  const int32_t *positions;    /* device [T] */
  const int32_t *slot_mapping; /* device [T]; negative = not this rank's slot (no KV write) */
  int32_t num_tokens;          /* T */
  void *k_pool;                /* device [num_pages, page_size, Hkv, Dk_nope + Dk_rope] */
  void *v_pool;                /* device [num_pages, page_size, Hkv, Dv] (NULL iff Dv == 0) */
  int64_t num_pages;
  int32_t page_size;
  int32_t kv_dtype;            /* PSD_BF16 or PSD_FP8_E4M3 (both pools) */
  float k_scale, v_scale;      /* fp8 only: finite and > 0 */
  int32_t *fault_dev;          /* device int32 fault word */
} psd_rope_append_args;

psd_status rope_append_kv(psd_ctx *ctx, const psd_rope_append_args *args, psd_stream_t stream);

/* Synchronises `stream` and reads the workspace's fault word: PSD_OK, or
 * PSD_ERR_DEVICE_FAULT with the PSD_FAULT_* bits in *fault_bits (nullable).
 * The word (the workspace's first 8 bytes) is tagged with the call that wrote it:
 * only faults of this context's latest decode call on `workspace` are reported, so
 * nothing has to clear it between calls and a fresh workspace needs no
 * initialisation.  The context remembers its 64 most recently used workspaces;
 * an older one reads as clean.  A reported fault is cleared. */
psd_status psd_check_device_error(psd_ctx *ctx, void *workspace, psd_stream_t stream,
                                  int32_t *fault_bits);

#ifdef __cplusplus
}
#endif

#endif /* PSD_H */
