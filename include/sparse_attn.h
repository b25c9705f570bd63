/*
 * sparse_attn.h -- C ABI of the GB300 (sm_103a) query-guided block-sparse decode
 * attention library (libsparse_attn.so).
 *
 * One decode step (select, then compute: SGLang分层稀疏注意力技术解析与优化实践 §1.2, §2.2):
 *
 *   sparse_attn_build_meta   once per context: per-block key bounding box (min/max per
 *                            channel) and, when asked for, per-block key means.
 *   sparse_attn_select       per step: score every block of each (sequence, KV head) from
 *                            the metadata, keep the local window, take the top-k blocks
 *                            (optionally in two levels), emit ascending block ids.
 *   sparse_attn_decode       per step: exact softmax attention over the union of the
 *                            selected blocks' tokens.
 *   sparse_attn_diff         per step: diff against the previous step and an LRU slot
 *                            cache; reports hits, misses (with their slots), evictions.
 *
 * Conventions shared by every call
 * --------------------------------
 *  * All tensor pointers are DEVICE pointers into memory the caller owns.  The library
 *    never allocates or frees device memory and keeps no pointer after a call returns.
 *  * Calls are asynchronous on the given stream (a cudaStream_t; NULL = legacy default
 *    stream).  Only sparse_attn_get_device_error synchronises.  select, decode and diff
 *    are launched as programmatic dependents of the stream's previous kernel: they may
 *    be scheduled while it finishes, but read no memory before it has completed, so
 *    stream order is kept exactly.
 *  * "unit" = one (sequence b, KV head kvh) pair, index u = b * Hkv + kvh.
 *  * Query head h reads KV head h / (Hq / Hkv) (grouped-query attention).
 *  * Layouts (row-major, contiguous):
 *      q           [B, Hq, D]                      q_dtype
 *      k_pages,
 *      v_pages     [num_pages, Hkv, block_size, D] kv_dtype  (one page = one block)
 *      block_table [B, nb_cap] int32  logical block j of sequence b -> physical page;
 *                  nb_cap = ceil(capacity_tokens / block_size), = nb when capacity is 0
 *      kmin, kmax  [B, Hkv, nb_cap, D] kv_dtype  (min/max of stored values: exact)
 *      kmean       [B, Hkv, n_mean_cap, D] float  (mean over mean_block tokens)
 *      sel_ids     [B, Hkv, sel_stride] int32 ascending; sel_count [B, Hkv] int32
 *      out         [B, Hq, D] float
 *    with nb = ceil(n_tokens / block_size), sel_stride = sparse_attn_sel_stride(p),
 *    mean_block = two_level ? coarse_block : block_size, n_mean = ceil(n_tokens/mean_block);
 *    with capacity = capacity_tokens (or n_tokens when it is 0), nb_cap = ceil(capacity /
 *    block_size) and n_mean_cap = ceil(capacity / mean_block) are the rows allocated per
 *    sequence / unit, of which the first nb (n_mean) hold the current context.
 *    The last block may be partial (n_tokens not a multiple of block_size); its
 *    missing tokens are never read into any result.
 *  * Inputs must be finite.  Every pointer must be 16-byte aligned.
 *  * The workspace (`ws`, `ws_bytes` >= sparse_attn_workspace_size) holds scores,
 *    split-K partials, per-unit completion counters and a device error word.  Run
 *    sparse_attn_workspace_init once after allocating it.  Calls that share one
 *    workspace must be ordered on one stream.  sparse_attn_build_meta and
 *    sparse_attn_append_meta use only its first 256 bytes (the error word), so one
 *    workspace sized for any length serves them at every length.
 *
 * Status codes: 0 OK, 1 INVALID_ARG (null/misaligned pointer, bad size), 2 UNSUPPORTED
 * (a dtype / head_dim / block_size / group combination without a kernel), 3 CUDA_ERROR
 * (a launch failed), 4 DEVICE_BOUNDS (reported only by sparse_attn_get_device_error).
 * Argument checks happen on the host before any launch; an entry that fails them
 * launches nothing.  No call traps, asserts on the device or spins without a bound.
 */
#ifndef SPARSE_ATTN_H
#define SPARSE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* sparse_attn_stream; /* same type as cudaStream_t */

enum {
    SPARSE_ATTN_OK = 0,
    SPARSE_ATTN_INVALID_ARG = 1,
    SPARSE_ATTN_UNSUPPORTED = 2,
    SPARSE_ATTN_CUDA_ERROR = 3,
    SPARSE_ATTN_DEVICE_BOUNDS = 4
};

enum { SPARSE_ATTN_F32 = 0, SPARSE_ATTN_BF16 = 1 };
enum { SPARSE_ATTN_SCORE_QUEST = 0, SPARSE_ATTN_SCORE_MEAN = 1 };

/* Device error word bits (sparse_attn_get_device_error). */
enum {
    SPARSE_ATTN_ERR_PAGE = 1u << 0,      /* block_table entry outside [0, num_pages) */
    SPARSE_ATTN_ERR_SEL_ID = 1u << 1,    /* sel_ids / prev_ids entry outside [0, nb) */
    SPARSE_ATTN_ERR_SEL_COUNT = 1u << 2, /* sel_count outside [0, sel_stride] */
    SPARSE_ATTN_ERR_TIMEOUT = 1u << 3,   /* a bounded wait (async copy, tensor-core MMA
                                            completion, a selection published by another
                                            CTA) gave up after about a second */
    SPARSE_ATTN_ERR_SLOT = 1u << 4,      /* LRU state holds an id outside [-1, nb) */
    SPARSE_ATTN_ERR_CAPACITY = 1u << 5   /* a per-CTA work list overflowed (the host's
                                            launch limits exclude it; a set bit is a bug) */
};

/* Problem description.  Passed by pointer, read during the call, never retained.
 * Field names follow the sparse-attention config of 从HiSparse到QSA的移植实战 §3.1
 * (window size, coarse block, fine block, top_k_coarse, top_k_fine). */
typedef struct sparse_attn_params {
    int32_t batch;          /* B >= 0 (0: nothing to do) */
    int32_t num_q_heads;    /* Hq, a multiple of Hkv; Hq / Hkv in {1, 2, 4, 8} */
    int32_t num_kv_heads;   /* Hkv >= 1 */
    int32_t head_dim;       /* D in {64, 128} */
    int32_t n_tokens;       /* N >= 0 tokens cached per sequence */
    int32_t block_size;     /* tokens per page = per selection block: 8, 16, 32, 64 or 128 */
    int32_t num_pages;      /* pages in k_pages / v_pages (bounds for block_table) */
    int32_t window_tokens;  /* W >= 0: blocks holding any of the last W tokens are always kept */
    int32_t topk;           /* k >= 0 blocks (single level) or level-2 slices (two level) */
    int32_t two_level;      /* 0: single level; 1: coarse blocks, then slices */
    int32_t coarse_block;   /* tokens per coarse block (two level), a multiple of block_size */
    int32_t topk_coarse;    /* K1 >= 0 coarse blocks surviving level 1 */
    int32_t score_kind;     /* single level: SPARSE_ATTN_SCORE_QUEST or SPARSE_ATTN_SCORE_MEAN */
    int32_t kv_dtype;       /* SPARSE_ATTN_F32 or SPARSE_ATTN_BF16 for K/V pages and kmin/kmax */
    int32_t q_dtype;        /* SPARSE_ATTN_F32 or SPARSE_ATTN_BF16 */
    float softmax_scale;    /* <= 0: 1/sqrt(D) */
    int32_t num_reserve;    /* >= 0 reserve block ids per unit (sparse_attn_select_reserved);
                               0 for sparse_attn_select */
    int32_t num_queries;    /* Q: query vectors per sequence sharing one selection per KV
                               head (0 or 1: one decode query).  With Q > 1, q and out are
                               [B, Q, Hq, D] (query t of sequence b at row b * Q + t), the
                               selection scores are summed over the Q queries, and the KV
                               dtype must be bf16, single level */
    int32_t capacity_tokens;  /* 0, or >= n_tokens: kmin / kmax / kmean are allocated for a
                               context of this many tokens, [B, Hkv, ceil(capacity /
                               block_size), D] and [B, Hkv, ceil(capacity / mean block), D],
                               so the context can grow (sparse_attn_append_meta) without
                               moving them; 0 means capacity = n_tokens */
} sparse_attn_params;

/* Human-readable name of a status code (static storage). */
const char* sparse_attn_status_string(int status);

/* Blocks per sequence, nb = ceil(n_tokens / block_size); -1 on bad params. */
int32_t sparse_attn_num_blocks(const sparse_attn_params* p);

/* int32 entries per unit row of sel_ids (and of every diff list): the largest
 * selection possible, min(topk, candidates) + min(num_reserve, candidates) + window
 * blocks; -1 on bad params. */
int32_t sparse_attn_sel_stride(const sparse_attn_params* p);

/* k for a context of n_tokens in pages of block_size tokens, by the SparDA page's §3.2
 * rule of a kept fraction falling with the sequence length: every block when
 * n_tokens <= 8192, else max(1, floor(nb * r)) with r = 15% (n_tokens <= 16384),
 * 10% (<= 32768) and 5% beyond (the page lists 16K, 32K, 128K; a length between two
 * listed points takes the next point's ratio).  Host-only; -1 on a bad argument. */
int32_t sparse_attn_topk_for_length(int32_t n_tokens, int32_t block_size);

/* Bytes of workspace the calls below need for this problem.  When capacity_tokens >
 * n_tokens the size covers every context length up to capacity_tokens, so one
 * workspace serves a growing context. */
int sparse_attn_workspace_size(const sparse_attn_params* p, size_t* bytes);

/* Zero the workspace's counters and error word (stream-ordered).  Call once after
 * allocating a workspace, before its first use. */
int sparse_attn_workspace_init(void* ws, size_t ws_bytes, sparse_attn_stream stream);

/* Limit, in SM clock cycles, of the fused step's hand-off waits on this workspace:
 * sparse_attn_step's decode waits for the selections that other CTAs (or the select
 * kernel launched just before it) publish -- per unit of its range, or, when each CTA
 * decodes whole units, for the next unit in publication order.  0 (the value
 * sparse_attn_workspace_init leaves) selects the default of 2e9 cycles, about one
 * second at GB300 clocks; larger values are capped at it.  (Waits inside one CTA's
 * own pipeline -- copy and tensor-core completions -- always use the default.)  A wait
 * that runs out sets SPARSE_ATTN_ERR_TIMEOUT in the error word and the step goes on
 * with the selection as it finds it and returns, so the context stays usable; that
 * call's results are then unspecified (a unit may keep an earlier call's output), and
 * later calls are unaffected.
 * Stream-ordered; copies 8 bytes from host memory, so it cannot be captured into a
 * CUDA graph.  No counterpart in the pages: it exists to bound and to test the waits. */
int sparse_attn_workspace_set_wait_limit(void* ws, size_t ws_bytes, uint64_t cycles,
                                         sparse_attn_stream stream);

/* Per-block metadata from the paged keys.
 * Defines: Quest key bounding box -- for each unit, block j and channel d,
 *   kmin[j][d] = min_t K[t][d], kmax[j][d] = max_t K[t][d] over the block's tokens
 *   (SGLang分层稀疏注意力技术解析与优化实践 §3.1.2, the key bounding box);
 * and, when kmean != NULL, kmean[r][d] = mean of K[t][d] over the tokens of mean row r
 *   (SparDA page www.2kiu.com/news/4656707 §3.1, mean pooling; 从HiSparse到QSA的移植实战
 *   §2.2, the coarse-block summary).  kmean is required when two_level or score_kind ==
 *   MEAN, and may be NULL otherwise.
 * Reads k_pages through block_table; writes kmin, kmax (kv_dtype) and kmean (float). */
int sparse_attn_build_meta(const sparse_attn_params* p, const void* k_pages,
                           const int32_t* block_table, void* kmin, void* kmax, float* kmean,
                           void* ws, size_t ws_bytes, sparse_attn_stream stream);

/* Metadata after tokens were appended to the cache (SGLang page §2.2, the block
 * representation is kept current as the context grows; §3.1.1, incremental update
 * instead of a rebuild).  p describes the context after the append (n_tokens = N_new);
 * tokens [n_old, N_new) of every sequence are new and already in the pages.  Only the
 * rows holding new tokens are rebuilt from their tokens (with the rows sharing a
 * build run), so the result equals sparse_attn_build_meta at N_new bit for bit; the
 * other rows are left as they are.  0 <= n_old <= n_tokens. */
int sparse_attn_append_meta(const sparse_attn_params* p, int32_t n_old, const void* k_pages,
                            const int32_t* block_table, void* kmin, void* kmax, float* kmean,
                            void* ws, size_t ws_bytes, sparse_attn_stream stream);

/* Block selection for one decode query per query head.
 * Single level (SGLang page §3.1.2; SparDA page §3.2 fixed top-k):
 *   score[u][j] = sum over the group's heads h and channels d of
 *                 max(q_h[d] * kmin[j][d], q_h[d] * kmax[j][d])           (QUEST), or
 *               = sum over h of q_h . kmean[j]                           (MEAN);
 *   candidates are the blocks outside the window; the top k by (score desc, block id
 *   asc) are united with the window blocks (从HiSparse到QSA的移植实战 §2.2, third level).
 * Two level (从HiSparse到QSA的移植实战 §2.2, §3.1):
 *   level 1 ranks every coarse block by sum_h q_h . kmean[c] and keeps topk_coarse;
 *   level 2 ranks the non-window slices (blocks) inside the survivors by the Quest bound
 *   and keeps topk; the window blocks are added.
 * Scores are kept in fp32 (the HiSparse->QSA page's §5.1 shows fp16 block scores
 * mis-ranking the top-k boundary).
 * Writes sel_ids (ascending, sel_count[u] valid entries per row) and sel_count. */
int sparse_attn_select(const sparse_attn_params* p, const void* q, const void* kmin,
                       const void* kmax, const float* kmean, int32_t* sel_ids,
                       int32_t* sel_count, void* ws, size_t ws_bytes, sparse_attn_stream stream);

/* sparse_attn_select plus a reserve set (SparDA page §3.4: a small set of extra blocks
 * kept at random is added to every selection result).  reserve_ids: device int32
 * [units, p->num_reserve], drawn by the caller (this library draws no random numbers);
 * any order, repeats and window or top-k blocks allowed.  The output row is the union
 * of the top-k, the reserve blocks and the window, ascending without repeats, so
 * sel_count[u] varies with the overlap.  An id outside [0, nb) sets
 * SPARSE_ATTN_ERR_SEL_ID and is skipped.  num_reserve = 0 is sparse_attn_select. */
int sparse_attn_select_reserved(const sparse_attn_params* p, const void* q, const void* kmin,
                                const void* kmax, const float* kmean, const int32_t* reserve_ids,
                                int32_t* sel_ids, int32_t* sel_count, void* ws, size_t ws_bytes,
                                sparse_attn_stream stream);

/* Sparse decode attention (从HiSparse到QSA的移植实战 §3.3: iterate only the selected
 * blocks given as a compact index array; SGLang page §2.2, the attention stage that
 * follows the selection).
 *   out[b][h] = sum over tokens t of the selected blocks of unit (b, h / G) of
 *               softmax_t(softmax_scale * q_h . k_t) * v_t,
 * exactly, over those tokens only; an empty selection gives a zero row.
 * Out-of-range sel_ids / block_table entries set a device error bit and are skipped.
 * With num_queries > 1 every query row of a unit attends over the unit's selection:
 * bf16 queries run on the fifth-generation tensor cores with K/V loaded by the tensor
 * memory accelerator from the page pools (viewed as [num_pages * Hkv * block_size, D]
 * bf16 rows), fp32 queries on the warp-level tensor-core path. */
int sparse_attn_decode(const sparse_attn_params* p, const void* q, const void* k_pages,
                       const void* v_pages, const int32_t* block_table, const int32_t* sel_ids,
                       const int32_t* sel_count, float* out, void* ws, size_t ws_bytes,
                       sparse_attn_stream stream);

/* One decode step in a single launch: sparse_attn_select_reserved (num_reserve = 0
 * allowed, reserve_ids may then be NULL) followed by sparse_attn_decode, with the same
 * results bit for bit (SGLang page §1.2, select-then-compute as one step).  The
 * attention of a (sequence, KV head) unit starts as soon as that unit's selection is
 * written, not after the whole batch's.  sel_ids / sel_count are written as by the
 * select call.  Single-level selection, bf16 K/V and one query per sequence only
 * (SPARSE_ATTN_UNSUPPORTED otherwise, or when one CTA per SM cannot hold the problem:
 * then call the two entry points).  The launch is cooperative; a workspace must not be
 * shared by two concurrent steps. */
int sparse_attn_step(const sparse_attn_params* p, const void* q, const void* kmin, const void* kmax,
                     const float* kmean, const int32_t* reserve_ids, const void* k_pages,
                     const void* v_pages, const int32_t* block_table, int32_t* sel_ids,
                     int32_t* sel_count, float* out, void* ws, size_t ws_bytes, sparse_attn_stream stream);

/* Kernels one sparse_attn_step call launches on the current device: 1 (the single
 * cooperative launch), 2 (select, then decode as its programmatic dependent waiting per
 * unit; chosen when there are more (sequence, KV head) units than SMs or a CTA's share
 * would not fit), 0 (B = 0), or -1 when the problem is invalid or not supported by
 * sparse_attn_step.  Host-only. */
int32_t sparse_attn_step_launches(const sparse_attn_params* p);

/* Step-to-step diff and LRU slot cache (SGLang page §3.2: cache 2-4x top-k, LRU
 * eviction; steps a-d: diff against the previous step, find what is resident, load
 * the misses, update the index).  For each unit, with S = sel_ids row (ascending,
 * sel_count entries) and P = prev_ids row:
 *   new = S \ P, dropped = P \ S, hits = S blocks resident, misses = the others
 *   (all ascending).  Miss i (ascending) takes the lowest free slot (slot_block == -1)
 *   if any, else evicts the resident block NOT in S with the smallest
 *   (slot_last_use, block id); evict_ids[i'] / evict_slot[i'] list evictions in miss
 *   order.  Then slot_last_use = step for every block of S.
 * In/out state: slot_block, slot_last_use [B*Hkv, cache_slots] int32 (start: all -1).
 * Outputs: every list [B*Hkv, sel_stride] int32; counts [B*Hkv, 5] int32 =
 *   {hits, misses, evictions, new, dropped}.
 * Requires sel_stride <= cache_slots <= 1024. */
int sparse_attn_diff(const sparse_attn_params* p, int32_t step, const int32_t* sel_ids,
                     const int32_t* sel_count, const int32_t* prev_ids,
                     const int32_t* prev_count, int32_t cache_slots, int32_t* slot_block,
                     int32_t* slot_last_use, int32_t* hit_ids, int32_t* miss_ids,
                     int32_t* miss_slot, int32_t* evict_ids, int32_t* evict_slot,
                     int32_t* new_ids, int32_t* dropped_ids, int32_t* counts, void* ws,
                     size_t ws_bytes, sparse_attn_stream stream);

/* sparse_attn_diff that also writes this step's slot map in the same launch:
 * sel_slot[u][i] = the slot holding sel_ids[u][i] after the step (a hit keeps its slot,
 * a miss gets the slot it is placed in) -- what sparse_attn_slot_map would compute from
 * the updated slot_block.  sel_slot: [B*Hkv, sel_stride] int32; other arguments and
 * outputs as sparse_attn_diff.  When the diff refuses a unit (error bit set) its
 * sel_slot row is left as it was. */
int sparse_attn_diff_slots(const sparse_attn_params* p, int32_t step, const int32_t* sel_ids,
                           const int32_t* sel_count, const int32_t* prev_ids,
                           const int32_t* prev_count, int32_t cache_slots, int32_t* slot_block,
                           int32_t* slot_last_use, int32_t* hit_ids, int32_t* miss_ids,
                           int32_t* miss_slot, int32_t* evict_ids, int32_t* evict_slot,
                           int32_t* new_ids, int32_t* dropped_ids, int32_t* counts,
                           int32_t* sel_slot, void* ws, size_t ws_bytes, sparse_attn_stream stream);

/* ---- Slot pool: misses loaded from a host-resident store ("SGLang分层稀疏注意力技术解析与
 * 优化实践" §3.3 IO transfer: full KV cache page-first in pinned / host-registered
 * memory, zero-copy transfer of a step's misses batched over requests; §3.2 steps c-d:
 * load the misses into the claimed slots, then update the index).
 * The pool holds, per unit, cache_slots page tiles: pool_k / pool_v [B*Hkv, cache_slots,
 * block_size, D] in the KV dtype, owned by the caller; slot s of unit u holds the block
 * the diff's slot_block[u][s] names. */

/* sel_slot[u][i] = the slot of unit u holding sel_ids[u][i] (i < sel_count[u]), from
 * the slot_block state after sparse_attn_diff of this step; a selected block that is not
 * resident gets -1 and sets SPARSE_ATTN_ERR_SLOT.  sel_slot: [B*Hkv, sel_stride] int32. */
int sparse_attn_slot_map(const sparse_attn_params* p, const int32_t* sel_ids,
                         const int32_t* sel_count, const int32_t* slot_block, int32_t cache_slots,
                         int32_t* sel_slot, void* ws, size_t ws_bytes, sparse_attn_stream stream);

/* IO kernel: for every unit u and miss i < counts[u][1], copy the K and V tiles of
 * block miss_ids[u][i] (page block_table[b][miss_ids], KV head u % Hkv) from the host
 * store into slot miss_slot[u][i] of pool_k / pool_v, in one launch.  host_k_pages /
 * host_v_pages: [num_pages, Hkv, block_size, D] page-first, in pinned or
 * cudaHostRegister'ed host memory (read by the GPU in place) or in device memory;
 * unregistered host memory is INVALID_ARG.  miss_ids / miss_slot / counts as written by
 * sparse_attn_diff.  Out-of-range ids, slots or pages set an error bit and are skipped. */
int sparse_attn_load_misses(const sparse_attn_params* p, const void* host_k_pages,
                            const void* host_v_pages, const int32_t* block_table,
                            const int32_t* miss_ids, const int32_t* miss_slot, const int32_t* counts,
                            int32_t cache_slots, void* pool_k, void* pool_v, void* ws,
                            size_t ws_bytes, sparse_attn_stream stream);

/* sparse_attn_decode reading K/V through the slot pool: the tokens of selected block
 * sel_ids[u][i] come from slot sel_slot[u][i] of unit u's pool (the page table and the
 * page pools are not read).  Same output and error rules as sparse_attn_decode. */
int sparse_attn_decode_slots(const sparse_attn_params* p, const void* q, const void* pool_k,
                             const void* pool_v, int32_t cache_slots, const int32_t* sel_ids,
                             const int32_t* sel_slot, const int32_t* sel_count, float* out,
                             void* ws, size_t ws_bytes, sparse_attn_stream stream);

/* sparse_attn_load_misses and sparse_attn_decode_slots in one launch, so that the
 * miss transfer overlaps the attention over the resident blocks ("SGLang分层稀疏注意力
 * 技术解析与优化实践" §3.3: the IO is hidden behind compute).  Loader CTAs copy each
 * unit's misses (miss_ids / miss_slot / counts as written by sparse_attn_diff) from the
 * host store into the pool exactly as sparse_attn_load_misses does, while the decode
 * CTAs attend to every unit's resident blocks first and to its missed blocks last, after
 * waiting (bounded, see sparse_attn_workspace_set_wait_limit) for the unit's loads.
 * sel_slot must come from sparse_attn_slot_map after this step's diff (miss slots
 * included).  The pool ends as after sparse_attn_load_misses; the output equals
 * sparse_attn_load_misses + sparse_attn_decode_slots up to the fp32 rounding of the
 * changed order (bit for bit for a unit without misses).  When no SM is left for
 * loaders the misses are loaded first, in their own launch.  bf16 K/V only (else
 * UNSUPPORTED); host memory rules as sparse_attn_load_misses; other arguments as
 * sparse_attn_decode_slots. */
int sparse_attn_decode_slots_io(const sparse_attn_params* p, const void* q, void* pool_k, void* pool_v,
                                int32_t cache_slots, const int32_t* sel_ids, const int32_t* sel_slot,
                                const int32_t* sel_count, const void* host_k_pages,
                                const void* host_v_pages, const int32_t* block_table,
                                const int32_t* miss_ids, const int32_t* miss_slot, const int32_t* counts,
                                float* out, void* ws, size_t ws_bytes, sparse_attn_stream stream);

/* Synchronise `stream`, copy the device error word to *flags (SPARSE_ATTN_ERR_* bits)
 * and clear it.  Returns SPARSE_ATTN_DEVICE_BOUNDS when any bit was set. */
int sparse_attn_get_device_error(void* ws, size_t ws_bytes, sparse_attn_stream stream,
                                 uint32_t* flags);

/* Block selection without a caller-provided workspace.
 *
 * The pages have no counterpart to this entry point; it exists for callers that
 * cannot allocate device memory: code that runs where cudaMalloc is forbidden or
 * unsafe (inside another framework's allocator or stream-ordered memory pool,
 * inside a host callback, in a plugin whose host owns every device allocation), or
 * a process whose device memory is entirely reserved by someone else's pool.
 *
 * Same inputs, outputs and results as sparse_attn_select for single-level
 * selection (two_level must be 0).  The scratch it needs -- error word, per-unit
 * completion counters and the fp32 score rows -- lives in a fixed array of
 * SPARSE_ATTN_NOALLOC_SCRATCH_BYTES inside the library, which every device that
 * loads the library keeps until the process exits.  Nothing is allocated and no
 * allocating library routine is called.
 *
 * - A problem whose scratch (256 B + 3 counter rows + units x candidates x 4 B,
 *   each part rounded up to 256 B) exceeds the array returns
 *   SPARSE_ATTN_UNSUPPORTED before any launch; two_level = 1 does too.
 * - The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any stream
 *   capture.
 * - Every call shares the one array: the counters are cleared at the start of each
 *   call (stream-ordered), but calls whose execution overlaps on the GPU -- on
 *   different streams, or from different host threads -- race on it and must be
 *   serialised by the caller.
 * - Device-side error bits of a call stay in the private array (select has no
 *   data-dependent indexing; only a timed-out copy wait could set one); read them
 *   with sparse_attn_select_noalloc_device_error.
 * - The cached address belongs to the device's context: after a cudaDeviceReset of
 *   that device the process must not call this entry point again. */
#define SPARSE_ATTN_NOALLOC_SCRATCH_BYTES (4u << 20)
int sparse_attn_select_noalloc(const sparse_attn_params* p, const void* q, const void* kmin,
                               const void* kmax, const float* kmean, int32_t* sel_ids,
                               int32_t* sel_count, sparse_attn_stream stream);

/* Error word of sparse_attn_select_noalloc's private scratch on the current device:
 * synchronise `stream`, copy the word to *flags (SPARSE_ATTN_ERR_* bits set by the
 * noalloc calls since the last one started) and clear it.  Returns
 * SPARSE_ATTN_DEVICE_BOUNDS when any bit was set.  Allocates nothing; the same
 * first-call and no-overlap rules as sparse_attn_select_noalloc apply. */
int sparse_attn_select_noalloc_device_error(sparse_attn_stream stream, uint32_t* flags);

#ifdef __cplusplus
}
#endif
#endif /* SPARSE_ATTN_H */
