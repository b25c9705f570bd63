/*
 * Plain fp64 CPU oracle for query-guided block-sparse decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this code: only the test suite, the smoke check and the CPU-baseline leg
 * of the benchmark use it.  It shares no header, helper or constant with the
 * CUDA library.
 *
 * Every routine is a direct, slow statement of one step of the method:
 *
 *   build_meta      per-block key bounding box (min/max per channel) and per-block
 *                   key mean.  Bounding box: "SGLang分层稀疏注意力技术解析与优化实践"
 *                   §3.1.2 (Quest: per-block, per-dimension key min/max).  Mean:
 *                   SparDA page (www.2kiu.com/news/4656707) §3.1 (mean pooling of the
 *                   block's tokens as its representative vector) and
 *                   "从HiSparse到QSA的移植实战" §2.2 (coarse-block summary vector).
 *   quest_scores    sum over the GQA group and the channels of
 *                   max(q_d * min_d, q_d * max_d): the upper bound of q.k over a
 *                   block's bounding box (SGLang page §3.1.2, "geometric relevance").
 *   mean_scores     sum over the group of q . mean(K_block) (SparDA page §3.1).
 *   select          top-k by (score desc, block id asc) over the non-window blocks,
 *                   united with the local window, emitted in ascending id order
 *                   (SparDA page §3.2 fixed top-k; HiSparse->QSA page §2.2 window).
 *   select_two_level  coarse 1024-token blocks ranked by the mean score, top K1
 *                   survive; their 64-token slices ranked by the Quest bound,
 *                   top K2 plus the window (HiSparse->QSA page §2.2, §3.1).
 *   decode          exact softmax attention over the union of the selected tokens
 *                   only (HiSparse->QSA page §3.3; SGLang page §1.2 select-then-compute).
 *   lru_step        step-to-step diff and LRU slot cache (SGLang page §3.2, steps a-d).
 *   union_reserve   a selection united with a reserve set of extra blocks drawn at
 *                   random by the caller (SparDA page §3.4: a small randomly kept
 *                   "reserve set" added to the selection result).
 *   topk_for_length k from the context length: no compression up to 8K tokens, then
 *                   15% / 10% / 5% of the blocks up to 16K / 32K / beyond (SparDA page
 *                   §3.2, sparsity ratio by sequence length; k = max(1, floor(nb * r))).
 *
 * Readings where the pages are silent are listed in the repository's design notes
 * and restated at each routine.  All arithmetic is double precision; stored bf16 /
 * fp32 inputs are widened exactly.
 *
 * Status: every routine returns 0 on success and a negative value on a bad argument.
 */
#ifndef SPARSE_ATTN_ORACLE_H
#define SPARSE_ATTN_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int batch;          /* B */
    int num_q_heads;    /* Hq */
    int num_kv_heads;   /* Hkv; Hq is a multiple of Hkv, head h reads KV head h / (Hq/Hkv) */
    int head_dim;       /* D */
    int n_tokens;       /* N, tokens cached per sequence */
    int block_size;     /* tokens per page = per selection block */
    int num_pages;      /* pages in the K/V pools */
    int window_tokens;  /* W, the last W tokens are always attended */
    int topk;           /* k blocks (single level) or K2 slices (two level) */
    int two_level;      /* 0 / 1 */
    int coarse_block;   /* tokens per coarse block (two level) */
    int topk_coarse;    /* K1 */
    int score_kind;     /* 0 = Quest bound, 1 = block mean */
    int kv_bf16;        /* 1: K/V stored as bfloat16, 0: float32 */
    int q_bf16;         /* 1: q stored as bfloat16, 0: float32 */
    double softmax_scale; /* <= 0 means 1/sqrt(D) */
} oracle_problem;

int oracle_num_blocks(const oracle_problem* p);
int oracle_first_window_block(const oracle_problem* p);
int oracle_mean_block(const oracle_problem* p);     /* tokens averaged per kmean row */
int oracle_num_mean_rows(const oracle_problem* p);  /* kmean rows per unit */

/* kmin, kmax: [B, Hkv, nb, D]; kmean: [B, Hkv, oracle_num_mean_rows, D] or NULL. */
int oracle_build_meta(const oracle_problem* p, const void* k_pages, const int32_t* block_table,
                      double* kmin, double* kmax, double* kmean);

/* Scores of units [unit_begin, unit_end) (unit = b * Hkv + kvh).
 * quest: out [units_total, nb]; mean: out [units_total, rows]. */
int oracle_quest_scores(const oracle_problem* p, int unit_begin, int unit_end, const void* q,
                        const double* kmin, const double* kmax, double* scores);
int oracle_mean_scores(const oracle_problem* p, int unit_begin, int unit_end, const void* q,
                       const double* kmean, int rows, double* scores);

/* Single-level selection from precomputed per-block scores [units_total, nb].
 * sel_ids: [units_total, sel_stride] ascending; sel_count: [units_total]. */
int oracle_select(const oracle_problem* p, int unit_begin, int unit_end, const double* scores,
                  int32_t* sel_ids, int32_t* sel_count, int sel_stride);

/* Two-level selection.  coarse_scores [units, n_coarse] and slice_scores [units, nb]
 * (NaN where a slice is not a level-2 candidate) are written for the caller's
 * near-tie checks; survivors [units, topk_coarse] ascending, n_survivors [units]. */
int oracle_select_two_level(const oracle_problem* p, int unit_begin, int unit_end, const void* q,
                            const double* kmin, const double* kmax, const double* kmean,
                            double* coarse_scores, double* slice_scores,
                            int32_t* survivors, int32_t* n_survivors,
                            int32_t* sel_ids, int32_t* sel_count, int sel_stride);

/* Level 2 only, given the survivors (ascending coarse ids) of each unit. */
int oracle_select_level2(const oracle_problem* p, int unit_begin, int unit_end, const void* q,
                         const double* kmin, const double* kmax,
                         const int32_t* survivors, const int32_t* n_survivors, int surv_stride,
                         double* slice_scores, int32_t* sel_ids, int32_t* sel_count,
                         int sel_stride);

/* Union of each unit's selection (ascending ids, sel_count[u] of them) with its
 * n_reserve reserve block ids (any order; duplicates and window ids allowed), written
 * ascending without duplicates to out_ids [units, out_stride] / out_count.  A reserve
 * id outside [0, nb) is an error (-5). */
int oracle_union_reserve(const oracle_problem* p, int unit_begin, int unit_end,
                         const int32_t* sel_ids, const int32_t* sel_count, int sel_stride,
                         const int32_t* reserve, int n_reserve,
                         int32_t* out_ids, int32_t* out_count, int out_stride);

/* k for a context of n_tokens in blocks of block_size tokens: every block when
 * n_tokens <= 8192, else max(1, floor(nb * r)) with r = 15% (n_tokens <= 16384),
 * 10% (<= 32768), 5% (beyond).  Negative on a bad argument. */
int oracle_topk_for_length(int n_tokens, int block_size);

/* out: [B, Hq, D]; only the heads of units [unit_begin, unit_end) are written. */
int oracle_decode(const oracle_problem* p, int unit_begin, int unit_end, const void* q,
                  const void* k_pages, const void* v_pages, const int32_t* block_table,
                  const int32_t* sel_ids, const int32_t* sel_count, int sel_stride,
                  double* out);

/* One decode step of the diff + LRU slot cache for n_units independent units.
 * counts: [n_units, 5] = hits, misses, evictions, new, dropped.
 * Lists: [n_units, out_stride]. */
int oracle_lru_step(int n_units, int step, int cache_slots,
                    const int32_t* cur_ids, const int32_t* cur_count, int cur_stride,
                    const int32_t* prev_ids, const int32_t* prev_count, int prev_stride,
                    int32_t* slot_block, int32_t* slot_last_use,
                    int32_t* hit_ids, int32_t* miss_ids, int32_t* miss_slot,
                    int32_t* evict_ids, int32_t* evict_slot,
                    int32_t* new_ids, int32_t* dropped_ids, int out_stride,
                    int32_t* counts);

#ifdef __cplusplus
}
#endif
#endif
