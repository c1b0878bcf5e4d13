/*
 * pagedattn.h -- C ABI of libpagedattn: paged decode attention on NVIDIA sm_103a (GB300).
 *
 * The operation ("[TIL] Optimizing paged attention", retepy.com, sections "Paged
 * Attention", "Data Layout" and "Baseline"): a decode step gives every sequence b of a
 * batch one query token with query_heads heads of head_dim elements. Its K/V history
 * lives in a paged cache. Token t of sequence b is stored in physical page
 * block_tables[b][t / page_size] at slot t % page_size. Query head h reads K/V head
 * h / (query_heads / kv_heads), i.e. consecutive query heads share a K/V head (GQA).
 * For each (b, h):
 *
 *     s_t    = scale * dot(query[b][h], key_cache[page(t)][slot(t)][kv(h)])   t < ctx[b]
 *     out    = sum_t softmax(s)_t * value_cache[page(t)][slot(t)][kv(h)]
 *
 * Data types and layouts (all row-major, C order):
 *   query          fp16  [batch][query_heads][head_dim]
 *   key_cache      fp16  [num_physical_pages][page_size][kv_heads][head_dim]
 *                        ([num_physical_pages][kv_heads][page_size][head_dim] with
 *                        cache_layout = PA_LAYOUT_HEAD_MAJOR)
 *   value_cache    fp16  same layout as key_cache
 *   block_tables   int32 [batch][max_pages_per_sequence]; only the first
 *                        ceil(context_lengths[b] / page_size) entries of row b are read
 *   context_lengths int32 [batch]
 *   out            fp32  [batch][query_heads][head_dim]; fully overwritten
 *
 * Ownership: every pointer argument is device memory owned by the caller; the library
 * neither retains nor frees it after the call returns. Calls are asynchronous on the
 * given CUDA stream (a cudaStream_t passed as void*; NULL = the legacy default
 * stream); no call synchronises the host or copies data to it, except
 * pa_get_device_error. Results are deterministic: the same inputs on the same GPU model
 * give bitwise-identical outputs (fixed work split, fixed merge order, no float atomics).
 *
 * Errors: host-side checks run before any launch and return a status without touching
 * the GPU. Device-side index problems (a needed block-table entry outside
 * [0, num_physical_pages), a context length outside [0, max_pages_per_sequence *
 * page_size]) are never read through: the offending page is skipped, the context is
 * clamped, and a flag is raised in the device error word (pa_get_device_error).
 * A context length of 0 yields an all-zero output row.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Shape of one decode step. The pages' "Problem" (section "Baseline"), plus the size of
 * the page pool so that page ids can be range-checked. */
typedef struct pa_problem_t {
  int32_t batch;                  /* sequences, >= 0 (0 is a no-op) */
  int32_t query_heads;            /* >= 1, a multiple of kv_heads */
  int32_t kv_heads;               /* >= 1 */
  int32_t head_dim;               /* 64, 128 or 256 */
  int32_t page_size;              /* tokens per page: a power of two in [8, 256] */
  int32_t max_pages_per_sequence; /* columns of block_tables, >= 1 */
  int32_t num_physical_pages;     /* pages in each cache, >= 1;
                                     num_physical_pages * page_size < 2^31 */
  int32_t cache_layout;           /* pa_cache_layout_t; 0 (the pages' layout) by default */
} pa_problem_t;

/* Layout of key_cache and value_cache. TOKEN_MAJOR is the layout of "[TIL] Optimizing paged
 * attention", section "Data Layout"; HEAD_MAJOR is the alternative that section "V2
 * (Vectorization)" proposes comparing, in which one K/V head's rows of a page are contiguous
 * (num_physical_pages * kv_heads < 2^31). */
typedef enum pa_cache_layout_t {
  PA_LAYOUT_TOKEN_MAJOR = 0, /* [num_physical_pages][page_size][kv_heads][head_dim] */
  PA_LAYOUT_HEAD_MAJOR = 1   /* [num_physical_pages][kv_heads][page_size][head_dim] */
} pa_cache_layout_t;

typedef enum pa_status_t {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, query_heads % kv_heads != 0,
                             non-finite scale, bad option value */
  PA_ERR_UNSUPPORTED = 2, /* head_dim or page_size outside the supported set, pool too big */
  PA_ERR_MISALIGNED = 3,  /* a tensor pointer is not 16-byte aligned (4 for int32 arrays) */
  PA_ERR_WORKSPACE = 4,   /* caller workspace too small, or allocating it failed */
  PA_ERR_CUDA = 5,        /* a CUDA runtime/driver call or a launch failed */
  PA_ERR_NO_DEVICE = 6    /* no usable sm_103a device is current */
} pa_status_t;

/* Bits of the device error word. */
#define PA_DEVERR_PAGE_ID 1u /* a needed block-table entry was outside the page pool */
#define PA_DEVERR_CONTEXT 2u /* a context length was < 0 or > max_pages*page_size */
#define PA_DEVERR_TIMEOUT 4u /* a pipeline wait ran past its time limit; output invalid */
#define PA_DEVERR_QUERY_START 8u /* pa_prefill: query offsets decreasing, past total_tokens,
                                   or more new tokens than context */

/* How work is split across the GPU. */
typedef enum pa_schedule_t {
  PA_SCHEDULE_AUTO = 0,    /* heuristic (pa_plan) */
  PA_SCHEDULE_SINGLE = 1,  /* one worker per (sequence, K/V head group), whole context,
                              final output written directly; no workspace */
  PA_SCHEDULE_BALANCED = 2 /* split-K: the concatenated K/V tiles of all sequences are cut
                              into equal contiguous ranges, one per worker; a worker
                              writes per-range (max, sum, partial output) for sequences it
                              shares with other workers, and those are merged by
                              log-sum-exp */
} pa_schedule_t;

/* Arithmetic of the group x token products. */
typedef enum pa_math_t {
  PA_MATH_AUTO = 0, /* heuristic (pa_plan) */
  PA_MATH_SIMT = 1, /* fp32 FMA on CUDA cores */
  PA_MATH_MMA = 2   /* fp16 x fp16 -> fp32 warp-level tensor-core tiles (m16n8k16) */
} pa_math_t;

/* Where the split-K merge runs (balanced schedule). */
typedef enum pa_combine_t {
  PA_COMBINE_AUTO = 0,  /* heuristic: KERNEL when workers >= units, else FUSED */
  PA_COMBINE_FUSED = 1, /* the worker holding a sequence's head group's first tiles merges
                           it once the other workers sharing it have published their
                           states (one launch per call) */
  PA_COMBINE_KERNEL = 2 /* a separate log-sum-exp combine kernel, 1 to 8 warps per (unit,
                           head) by contributor count, launched as a programmatic dependent
                           of the decode kernel */
} pa_combine_t;

typedef struct pa_options_t {
  int32_t schedule;    /* pa_schedule_t */
  int32_t math;        /* pa_math_t */
  int32_t combine;     /* pa_combine_t */
  int32_t workers;     /* balanced: number of warps that take K/V tiles (rounded up to a
                          multiple of the plan's group); 0 = as many as fit at once */
  int32_t stages;      /* K/V pipeline depth per worker; 0 = default */
  int32_t warps_per_cta; /* 0 = default */
  int32_t tile_tokens; /* tokens per K/V tile: 0 = default; 16 or 32 for head_dim 128 */
  int32_t test_flags;  /* 0, or PA_TEST_EXPIRE_WAITS (tests of failure detection only) */
} pa_options_t;

/* Test hook for the failure path: every warp's first K/V tile waits for 16 bytes that never
 * arrive, so its bounded wait runs out (after about a second), the call raises
 * PA_DEVERR_TIMEOUT and its outputs are invalid; the device stays usable, and the workspace
 * the call used needs no re-initialisation (see pa_workspace_init). */
#define PA_TEST_EXPIRE_WAITS 1

/* What pa_decode / pa_decode_ex will launch for a problem (filled by pa_plan). */
typedef struct pa_plan_t {
  int32_t schedule;       /* resolved pa_schedule_t */
  int32_t math;           /* resolved pa_math_t */
  int32_t combine;        /* resolved pa_combine_t */
  int32_t workers;        /* warps that process K/V tiles */
  int32_t warps_per_cta;
  int32_t ctas;
  int32_t stages;
  int32_t tile_tokens;    /* tokens per K/V tile */
  int32_t units;          /* batch * kv_heads * ceil(g / 8): (sequence, head group) units */
  int32_t heads_per_unit; /* query heads one warp serves with one K/V read (<= 8) */
  int32_t group;          /* warps per worker: they serve neighbouring units of a sequence
                             over the same tokens */
  int64_t smem_bytes;     /* dynamic shared memory per CTA */
  int64_t workspace_bytes;/* bytes pa_decode_ex needs for this plan */
} pa_plan_t;

/* Resolve the schedule/math heuristic for `problem` on a GPU with `sm_count` SMs.
 * Pure host logic (no GPU needed). The heuristic follows the context-split discussion
 * of the pages ("[TIL] Optimizing paged attention", section "V4 (Context-axis
 * parallelism)"; partition sizing against the SM count in the paged_attention_v2
 * notes): one worker per unit while the units alone fill the GPU several times over and
 * the longest possible context (max_pages_per_sequence * page_size) is short; otherwise
 * the balanced split-K schedule. options may be NULL (all AUTO). */
pa_status_t pa_plan(const pa_problem_t *problem, const pa_options_t *options, int32_t sm_count,
                    pa_plan_t *plan);

/* Bytes of device workspace pa_decode_ex needs for `problem` and `options` on the current
 * device (0 for the single-pass schedule). The workspace holds what the split-K schedule of
 * "[TIL] Optimizing paged attention", section "V4 (Context-axis parallelism)", writes
 * between its two phases -- per range the running maximum, the sum and the unnormalised
 * partial output -- plus one flag per range for the fused merge (the range's state is
 * published by writing the call's number into it).
 * That section leaves the buffer to the calling code; here the caller owns it
 * (pa_decode_ex), or the library does (pa_decode), or a static array (pa_decode_noalloc). */
pa_status_t pa_workspace_size(const pa_problem_t *problem, const pa_options_t *options,
                              size_t *bytes);

/* Zero a caller-owned workspace (cudaMemsetAsync on `stream`) -- the split-K buffer of
 * "[TIL] Optimizing paged attention", section "V4 (Context-axis parallelism)". Call it once
 * for every new buffer (also when a freed buffer's address comes back from the allocator):
 * the fused merge's flags must not start out holding arbitrary values. Between calls the
 * buffer must not be written by anyone else. Nothing needs resetting after a call, whether
 * it completed or its waits expired (PA_DEVERR_TIMEOUT): every call publishes its partial
 * states under a number of its own (unique within the process, never 0), so flags that
 * earlier calls left behind never match a later call's. */
pa_status_t pa_workspace_init(void *workspace, size_t workspace_bytes, void *stream);

/* One decode step with the heuristic's plan: the operation at the top of this file, as
 * "[TIL] Optimizing paged attention" defines it in sections "Paged Attention" (one query
 * token per sequence against its cached K/V) and "Baseline" (block-table gather, GQA head
 * mapping, scaled dot products, softmax, weighted sum of V; fp32 output). The split-K
 * workspace, when needed, is owned by the library: one grow-only buffer per device,
 * allocated on first need (the first call that needs it must not be inside stream
 * capture), released at process exit. Calls that use that buffer must not overlap in time
 * on different streams. query/key_cache/value_cache: fp16 device pointers; out: fp32
 * device pointer. Returns PA_OK once the work is queued on `stream`; host-side errors are
 * returned before anything is queued. */
pa_status_t pa_decode(const pa_problem_t *problem, const void *query, const void *key_cache,
                      const void *value_cache, const int32_t *block_tables,
                      const int32_t *context_lengths, float scale, float *out, void *stream);

/* pa_decode with explicit options and a caller-owned workspace of workspace_bytes
 * (>= pa_workspace_size; zeroed once by pa_workspace_init; 256-byte aligned). workspace may
 * be NULL when the plan needs none; a missing or short one is PA_ERR_WORKSPACE. Same
 * operation ("[TIL] Optimizing paged attention", sections "Paged Attention" and
 * "Baseline"); the options choose how the work is split ("V4 (Context-axis
 * parallelism)": one pass per sequence, or the context cut across workers and merged by
 * log-sum-exp) and which arithmetic computes the group x token products. Concurrent calls
 * must use distinct workspaces. */
pa_status_t pa_decode_ex(const pa_problem_t *problem, const void *query, const void *key_cache,
                         const void *value_cache, const int32_t *block_tables,
                         const int32_t *context_lengths, float scale, float *out,
                         const pa_options_t *options, void *workspace, size_t workspace_bytes,
                         void *stream);

/* Size of the fixed device scratch that pa_decode_noalloc uses (16 MiB). */
#define PA_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/* pa_decode for callers that must not allocate device memory -- no counterpart in the
 * paper; it exists for deployments, not for the method. A serving engine typically
 * reserves nearly all of HBM for its K/V page pool at start-up and allows no allocation
 * afterwards, and cudaMalloc/cudaFree synchronise the device, which a decode loop cannot
 * afford; code running inside such an engine may have no allocator at all. This call
 * never calls cudaMalloc, cudaFree or any allocating routine: when the heuristic's plan
 * needs split-K scratch, it uses a 16 MiB array compiled into the library
 * (PA_NOALLOC_SCRATCH_BYTES), which every GPU that loads the library holds until the
 * process exits. Arguments, layouts and results are those of pa_decode; the caller still
 * passes all inputs and the output.
 *  - A plan that needs more scratch than PA_NOALLOC_SCRATCH_BYTES (pa_plan reports it in
 *    workspace_bytes) is refused with PA_ERR_WORKSPACE before any launch.
 *  - The first call on each device looks up the array's device address (and may load the
 *    library's GPU code); make that first call before any stream capture begins.
 *  - Every call shares the one array per device and it keeps the previous call's contents
 *    (none of it needs clearing: each call publishes its partial states under a number of
 *    its own). Calls whose work overlaps on the GPU (other streams, other host threads)
 *    race on the array and give wrong results: serialise them. */
pa_status_t pa_decode_noalloc(const pa_problem_t *problem, const void *query,
                              const void *key_cache, const void *value_cache,
                              const int32_t *block_tables, const int32_t *context_lengths,
                              float scale, float *out, void *stream);

/* Split-K partial phase with a fixed number of splits per sequence, as in "[TIL]
 * Optimizing paged attention", section "V4 (Context-axis parallelism)": sequence b's
 * pages are cut into num_splits ranges of ceil(pages_b / num_splits) pages (the last
 * ranges may be short or empty); for each (b, split, query head) it writes
 *   partial_max [batch][num_splits][query_heads]           fp32: max_t s_t * log2(e)
 *   partial_sum [batch][num_splits][query_heads]           fp32: sum_t 2^(s_t log2 e - max)
 *   partial_out [batch][num_splits][query_heads][head_dim] fp32: sum_t 2^(..) * V_t,
 *                                                          not normalised
 * (an empty range writes max = -inf, sum = 0, out = 0). The maximum is in base-2 units
 * (scores times log2(e)). num_splits >= 1. math: pa_math_t (0 = AUTO). */
pa_status_t pa_split_kv_partial(const pa_problem_t *problem, const void *query,
                                const void *key_cache, const void *value_cache,
                                const int32_t *block_tables, const int32_t *context_lengths,
                                float scale, int32_t num_splits, int32_t math,
                                float *partial_max, float *partial_sum, float *partial_out,
                                void *stream);

/* Log-sum-exp combine of the arrays pa_split_kv_partial writes ("[TIL] Optimizing paged
 * attention", section "V4 (Context-axis parallelism)", merge kernel): splits with sum 0
 * are skipped, the rest are merged in split order and the result normalised into out
 * [batch][query_heads][head_dim] (0 where every split is empty). */
pa_status_t pa_split_kv_combine(const pa_problem_t *problem, int32_t num_splits,
                                const float *partial_max, const float *partial_sum,
                                const float *partial_out, float *out, void *stream);

/* Append one token per sequence to the paged caches: new_key[b][h][:] and new_value[b][h]
 * [:] (fp16, [batch][kv_heads][head_dim], 16-byte aligned) are written at token index
 * t = context_lengths[b] -- physical page block_tables[b][t / page_size], slot t % page_size,
 * in the problem's cache_layout. This is the cache write that precedes a decode step ("[TIL]
 * Optimizing paged attention", section "Paged Attention": the K and V of earlier tokens are
 * kept and reused); context_lengths holds the lengths before the append, and the caller
 * decodes with each length plus one afterwards. The page for index t must already be in
 * the block table. A sequence whose t is outside [0, max_pages_per_sequence * page_size) or
 * whose page id is outside the pool is skipped and flagged (PA_DEVERR_CONTEXT /
 * PA_DEVERR_PAGE_ID). Two sequences appending to the same (page, slot) race. */
pa_status_t pa_append_kv(const pa_problem_t *problem, const void *new_key, const void *new_value,
                         const int32_t *block_tables, const int32_t *context_lengths,
                         void *key_cache, void *value_cache, void *stream);

/* Causal multi-token (prefill) attention over the paged caches: the decode step of
 * section "Paged Attention" extended to several new tokens per sequence, computed
 * flash-style ("[TIL] Optimizing paged attention", section "Flash Attention": score
 * tiles, an online softmax and the weighted value sum, never materialising the score
 * matrix). Sequence b has n_b = query_start[b + 1] - query_start[b] new tokens whose K and V
 * are already in the cache (written before the call, e.g. by pa_append_kv or a bulk copy):
 * they are the last n_b of its context_lengths[b] tokens, so the j-th new token sits at
 * position p = context_lengths[b] - n_b + j and attends to tokens 0..p.
 *   query        fp16 [total_tokens][query_heads][head_dim], device, 16-byte aligned; row
 *                query_start[b] + j is the j-th new token of sequence b
 *   query_start  int32 [batch + 1], device, non-decreasing, query_start[0] = 0 and
 *                query_start[batch] <= total_tokens
 *   max_query_len  host int >= every n_b (sizes the grid; tokens past it are not computed)
 *   key_cache, value_cache, block_tables, context_lengths, scale  as for pa_decode
 *   out          fp32 [total_tokens][query_heads][head_dim], device, 16-byte aligned; rows of
 *                new tokens are written, other rows are left untouched
 *   options      may be NULL; only test_flags is read (other fields must be zero)
 * Supports head_dim 64, 128 and 256 and query_heads / kv_heads <= 128. A sequence with
 * inconsistent offsets is skipped and flagged (PA_DEVERR_QUERY_START), one with a context
 * length out of range likewise (PA_DEVERR_CONTEXT); a needed page id outside the pool is
 * flagged (PA_DEVERR_PAGE_ID) and its rows are invalid. Runs asynchronously on `stream`;
 * allocates nothing. */
pa_status_t pa_prefill(const pa_problem_t *problem, const void *query, const int32_t *query_start,
                       int64_t total_tokens, int32_t max_query_len, const void *key_cache,
                       const void *value_cache, const int32_t *block_tables,
                       const int32_t *context_lengths, float scale, float *out,
                       const pa_options_t *options, void *stream);

/* Read and clear the device error word of the current device (PA_DEVERR_* bits) after
 * the work queued on `stream` finishes. Synchronises `stream`. The word records the
 * preconditions of "[TIL] Optimizing paged attention", section "Paged Attention" (a
 * sequence's needed block-table entries name pages of the pool; its context fits its table
 * row) that a call found broken, and expired pipeline waits. *flags receives the bits;
 * PA_ERR_CUDA if the copy or the synchronisation failed.
 *
 * The library caches, per device, device addresses it looked up or allocated (this word,
 * the pa_decode workspace, the pa_decode_noalloc scratch). They belong to the device's
 * primary context: after cudaDeviceReset, or any other end of that context, they are stale,
 * so do not reset a device while the library is in use on it. */
pa_status_t pa_get_device_error(void *stream, uint32_t *flags);

/* Static description of a status code (library plumbing; the pages' launch functions return
 * nothing, section "Baseline"). Never NULL. */
const char *pa_status_string(pa_status_t status);

/* Library version as 10000 * major + 100 * minor + patch (library plumbing, no counterpart in
 * the pages). */
int32_t pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
