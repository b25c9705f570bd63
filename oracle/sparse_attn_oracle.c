/*
 * Plain fp64 CPU oracle for query-guided block-sparse decode attention.
 * TEST INFRASTRUCTURE ONLY -- see sparse_attn_oracle.h for scope and citations.
 *
 * Written for a reader checking it against the pages by eye: one loop nest per
 * formula, no blocking, no fusion, no reordering beyond what the definition says.
 */
#include "sparse_attn_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- inputs -- */

/* Exact value of one stored element (bfloat16 is the top half of an IEEE float). */
static double load_value(const void* base, size_t index, int is_bf16)
{
    if (is_bf16) {
        uint16_t half = ((const uint16_t*)base)[index];
        uint32_t bits = (uint32_t)half << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float*)base)[index];
}

static int check_problem(const oracle_problem* p)
{
    if (!p) return -1;
    if (p->batch < 0 || p->num_q_heads <= 0 || p->num_kv_heads <= 0 || p->head_dim <= 0) return -1;
    if (p->num_q_heads % p->num_kv_heads != 0) return -1;
    if (p->n_tokens < 0 || p->block_size <= 0 || p->window_tokens < 0 || p->topk < 0) return -1;
    if (p->two_level && (p->coarse_block <= 0 || p->coarse_block % p->block_size != 0 ||
                         p->topk_coarse < 0)) return -1;
    return 0;
}

int oracle_num_blocks(const oracle_problem* p)
{
    return (p->n_tokens + p->block_size - 1) / p->block_size;
}

/* Reading: the window is the last W tokens of the context; a block belongs to the
 * window when it holds any of them.  W = 0 means no window. */
int oracle_first_window_block(const oracle_problem* p)
{
    int nb = oracle_num_blocks(p);
    if (p->window_tokens <= 0) return nb;
    int first_token = p->n_tokens - p->window_tokens;
    if (first_token < 0) first_token = 0;
    return first_token / p->block_size;
}

int oracle_mean_block(const oracle_problem* p)
{
    return p->two_level ? p->coarse_block : p->block_size;
}

int oracle_num_mean_rows(const oracle_problem* p)
{
    int mb = oracle_mean_block(p);
    return (p->n_tokens + mb - 1) / mb;
}

static int tokens_in_block(const oracle_problem* p, int j)
{
    int start = j * p->block_size;
    int n = p->n_tokens - start;
    return n < p->block_size ? n : p->block_size;
}

static size_t kv_index(const oracle_problem* p, int page, int kvh, int t, int d)
{
    return (((size_t)page * p->num_kv_heads + kvh) * p->block_size + t) * p->head_dim + d;
}

/* Query element d of query head h of sequence b. */
static double q_value(const oracle_problem* p, const void* q, int b, int h, int d)
{
    size_t idx = ((size_t)b * p->num_q_heads + h) * p->head_dim + d;
    return load_value(q, idx, p->q_bf16);
}

/* ------------------------------------------------------------ build_meta -- */

/* Per block j and channel d: min and max of K over the block's tokens (the Quest
 * key bounding box), and the mean of K over each mean-row's tokens. */
int oracle_build_meta(const oracle_problem* p, const void* k_pages, const int32_t* block_table,
                      double* kmin, double* kmax, double* kmean)
{
    if (check_problem(p)) return -1;
    const int nb = oracle_num_blocks(p), D = p->head_dim, Hkv = p->num_kv_heads;
    for (int b = 0; b < p->batch; ++b)
        for (int kvh = 0; kvh < Hkv; ++kvh)
            for (int j = 0; j < nb; ++j) {
                int page = block_table[(size_t)b * nb + j];
                if (page < 0 || page >= p->num_pages) return -2;
                int nt = tokens_in_block(p, j);
                for (int d = 0; d < D; ++d) {
                    double lo = INFINITY, hi = -INFINITY;
                    for (int t = 0; t < nt; ++t) {
                        double x = load_value(k_pages, kv_index(p, page, kvh, t, d), p->kv_bf16);
                        if (x < lo) lo = x;
                        if (x > hi) hi = x;
                    }
                    size_t o = (((size_t)b * Hkv + kvh) * nb + j) * D + d;
                    kmin[o] = lo;
                    kmax[o] = hi;
                }
            }

    if (kmean) {
        const int mb = oracle_mean_block(p), rows = oracle_num_mean_rows(p);
        for (int b = 0; b < p->batch; ++b)
            for (int kvh = 0; kvh < Hkv; ++kvh)
                for (int r = 0; r < rows; ++r) {
                    int t0 = r * mb, t1 = t0 + mb;
                    if (t1 > p->n_tokens) t1 = p->n_tokens;
                    for (int d = 0; d < D; ++d) {
                        double sum = 0.0;
                        for (int tok = t0; tok < t1; ++tok) {
                            int j = tok / p->block_size, t = tok % p->block_size;
                            int page = block_table[(size_t)b * nb + j];
                            sum += load_value(k_pages, kv_index(p, page, kvh, t, d), p->kv_bf16);
                        }
                        kmean[(((size_t)b * Hkv + kvh) * rows + r) * D + d] = sum / (double)(t1 - t0);
                    }
                }
    }
    return 0;
}

/* ---------------------------------------------------------------- scores -- */

/* Quest bound, summed over the query heads that share KV head kvh (GQA). */
int oracle_quest_scores(const oracle_problem* p, int unit_begin, int unit_end, const void* q,
                        const double* kmin, const double* kmax, double* scores)
{
    if (check_problem(p)) return -1;
    const int nb = oracle_num_blocks(p), D = p->head_dim, Hkv = p->num_kv_heads;
    const int G = p->num_q_heads / Hkv;
    for (int u = unit_begin; u < unit_end; ++u) {
        int b = u / Hkv, kvh = u % Hkv;
        for (int j = 0; j < nb; ++j) {
            const double* lo = kmin + ((size_t)u * nb + j) * D;
            const double* hi = kmax + ((size_t)u * nb + j) * D;
            double s = 0.0;
            for (int g = 0; g < G; ++g) {
                int h = kvh * G + g;
                for (int d = 0; d < D; ++d) {
                    double qd = q_value(p, q, b, h, d);
                    double a = qd * lo[d], c = qd * hi[d];
                    s += (a > c) ? a : c;
                }
            }
            scores[(size_t)u * nb + j] = s;
        }
    }
    return 0;
}

/* Sum over the group of q_h . mean(K over the row's tokens). */
int oracle_mean_scores(const oracle_problem* p, int unit_begin, int unit_end, const void* q,
                       const double* kmean, int rows, double* scores)
{
    if (check_problem(p)) return -1;
    const int D = p->head_dim, Hkv = p->num_kv_heads, G = p->num_q_heads / Hkv;
    for (int u = unit_begin; u < unit_end; ++u) {
        int b = u / Hkv, kvh = u % Hkv;
        for (int r = 0; r < rows; ++r) {
            const double* m = kmean + ((size_t)u * rows + r) * D;
            double s = 0.0;
            for (int g = 0; g < G; ++g)
                for (int d = 0; d < D; ++d) s += q_value(p, q, b, kvh * G + g, d) * m[d];
            scores[(size_t)u * rows + r] = s;
        }
    }
    return 0;
}

/* ------------------------------------------------------------- selection -- */

typedef struct {
    double score;
    int32_t id;
} scored_id;

/* Order: higher score first; on equal scores the lower block id first. */
static int by_score_desc_id_asc(const void* x, const void* y)
{
    const scored_id* a = (const scored_id*)x;
    const scored_id* b = (const scored_id*)y;
    if (a->score > b->score) return -1;
    if (a->score < b->score) return 1;
    return (a->id > b->id) - (a->id < b->id);
}

static int by_int_asc(const void* x, const void* y)
{
    int32_t a = *(const int32_t*)x, b = *(const int32_t*)y;
    return (a > b) - (a < b);
}

/* Keep the first min(k, n) candidates in (score desc, id asc) order; returns how
 * many were kept and writes their ids (unordered) to out. */
static int top_k(scored_id* cand, int n, int k, int32_t* out)
{
    qsort(cand, (size_t)n, sizeof *cand, by_score_desc_id_asc);
    int keep = k < n ? k : n;
    for (int i = 0; i < keep; ++i) out[i] = cand[i].id;
    return keep;
}

int oracle_select(const oracle_problem* p, int unit_begin, int unit_end, const double* scores,
                  int32_t* sel_ids, int32_t* sel_count, int sel_stride)
{
    if (check_problem(p)) return -1;
    const int nb = oracle_num_blocks(p), wfirst = oracle_first_window_block(p);
    if (sel_stride < (p->topk < wfirst ? p->topk : wfirst) + (nb - wfirst)) return -3;
    scored_id* cand = (scored_id*)malloc(sizeof(scored_id) * (size_t)(nb > 0 ? nb : 1));
    if (!cand) return -4;
    for (int u = unit_begin; u < unit_end; ++u) {
        int32_t* out = sel_ids + (size_t)u * sel_stride;
        /* candidates: every block outside the window (the window is added in full) */
        for (int j = 0; j < wfirst; ++j) {
            cand[j].score = scores[(size_t)u * nb + j];
            cand[j].id = j;
        }
        int n = top_k(cand, wfirst, p->topk, out);
        for (int j = wfirst; j < nb; ++j) out[n++] = j;
        qsort(out, (size_t)n, sizeof *out, by_int_asc);
        sel_count[u] = n;
    }
    free(cand);
    return 0;
}

/* SparDA page §3.4: the selection result is extended by a reserve set of blocks kept
 * at random; the union is taken as sets and emitted in ascending id order. */
int oracle_union_reserve(const oracle_problem* p, int unit_begin, int unit_end,
                         const int32_t* sel_ids, const int32_t* sel_count, int sel_stride,
                         const int32_t* reserve, int n_reserve,
                         int32_t* out_ids, int32_t* out_count, int out_stride)
{
    if (check_problem(p) || n_reserve < 0) return -1;
    const int nb = oracle_num_blocks(p);
    int32_t* all = (int32_t*)malloc(sizeof(int32_t) * (size_t)(sel_stride + n_reserve + 1));
    if (!all) return -4;
    for (int u = unit_begin; u < unit_end; ++u) {
        int n = 0;
        for (int i = 0; i < sel_count[u]; ++i) all[n++] = sel_ids[(size_t)u * sel_stride + i];
        for (int i = 0; i < n_reserve; ++i) {
            const int32_t j = reserve[(size_t)u * n_reserve + i];
            if (j < 0 || j >= nb) {
                free(all);
                return -5;
            }
            all[n++] = j;
        }
        qsort(all, (size_t)n, sizeof *all, by_int_asc);
        int m = 0;   /* drop repeats of the sorted list */
        for (int i = 0; i < n; ++i)
            if (m == 0 || all[i] != all[m - 1]) all[m++] = all[i];
        if (m > out_stride) {
            free(all);
            return -3;
        }
        for (int i = 0; i < m; ++i) out_ids[(size_t)u * out_stride + i] = all[i];
        out_count[u] = m;
    }
    free(all);
    return 0;
}

/* SparDA page §3.2: the kept fraction falls with the sequence length -- none dropped
 * up to 8K tokens, 15% at 16K, 10% at 32K, 5% at 128K; lengths between two listed
 * points take the next listed point's ratio, and k = max(1, floor(nb * ratio)) as in
 * the page's decode sketch (§3.4), in integer arithmetic. */
int oracle_topk_for_length(int n_tokens, int block_size)
{
    if (n_tokens < 0 || block_size < 1) return -1;
    const long long nb = ((long long)n_tokens + block_size - 1) / block_size;
    if (n_tokens <= 8192) return (int)nb;
    const long long percent = n_tokens <= 16384 ? 15 : (n_tokens <= 32768 ? 10 : 5);
    const long long k = nb * percent / 100;
    return (int)(k > 1 ? k : 1);
}

int oracle_select_level2(const oracle_problem* p, int unit_begin, int unit_end, const void* q,
                         const double* kmin, const double* kmax,
                         const int32_t* survivors, const int32_t* n_survivors, int surv_stride,
                         double* slice_scores, int32_t* sel_ids, int32_t* sel_count,
                         int sel_stride)
{
    if (check_problem(p) || !p->two_level) return -1;
    const int nb = oracle_num_blocks(p), wfirst = oracle_first_window_block(p);
    const int D = p->head_dim, Hkv = p->num_kv_heads, G = p->num_q_heads / Hkv;
    const int per_coarse = p->coarse_block / p->block_size;
    scored_id* cand = (scored_id*)malloc(sizeof(scored_id) * (size_t)(nb > 0 ? nb : 1));
    if (!cand) return -4;
    for (int u = unit_begin; u < unit_end; ++u) {
        int b = u / Hkv, kvh = u % Hkv;
        for (int j = 0; j < nb; ++j) slice_scores[(size_t)u * nb + j] = NAN;
        int n = 0;
        for (int i = 0; i < n_survivors[u]; ++i) {
            int c = survivors[(size_t)u * surv_stride + i];
            for (int s = 0; s < per_coarse; ++s) {
                int j = c * per_coarse + s;
                if (j >= nb || j >= wfirst) continue;   /* window slices are added in full */
                const double* lo = kmin + ((size_t)u * nb + j) * D;
                const double* hi = kmax + ((size_t)u * nb + j) * D;
                double sc = 0.0;
                for (int g = 0; g < G; ++g)
                    for (int d = 0; d < D; ++d) {
                        double qd = q_value(p, q, b, kvh * G + g, d);
                        double a = qd * lo[d], e = qd * hi[d];
                        sc += (a > e) ? a : e;
                    }
                slice_scores[(size_t)u * nb + j] = sc;
                cand[n].score = sc;
                cand[n].id = j;
                ++n;
            }
        }
        int32_t* out = sel_ids + (size_t)u * sel_stride;
        int m = top_k(cand, n, p->topk, out);
        if (sel_stride < m + (nb - wfirst)) { free(cand); return -3; }
        for (int j = wfirst; j < nb; ++j) out[m++] = j;
        qsort(out, (size_t)m, sizeof *out, by_int_asc);
        sel_count[u] = m;
    }
    free(cand);
    return 0;
}

int oracle_select_two_level(const oracle_problem* p, int unit_begin, int unit_end, const void* q,
                            const double* kmin, const double* kmax, const double* kmean,
                            double* coarse_scores, double* slice_scores,
                            int32_t* survivors, int32_t* n_survivors,
                            int32_t* sel_ids, int32_t* sel_count, int sel_stride)
{
    if (check_problem(p) || !p->two_level) return -1;
    const int rows = oracle_num_mean_rows(p);   /* coarse blocks per unit */
    int rc = oracle_mean_scores(p, unit_begin, unit_end, q, kmean, rows, coarse_scores);
    if (rc) return rc;
    scored_id* cand = (scored_id*)malloc(sizeof(scored_id) * (size_t)(rows > 0 ? rows : 1));
    if (!cand) return -4;
    /* Level 1: every coarse block is a candidate, the window region included. */
    for (int u = unit_begin; u < unit_end; ++u) {
        for (int c = 0; c < rows; ++c) {
            cand[c].score = coarse_scores[(size_t)u * rows + c];
            cand[c].id = c;
        }
        int32_t* surv = survivors + (size_t)u * p->topk_coarse;
        int n = top_k(cand, rows, p->topk_coarse, surv);
        qsort(surv, (size_t)n, sizeof *surv, by_int_asc);
        n_survivors[u] = n;
    }
    free(cand);
    /* Level 2: the slices inside the survivors. */
    return oracle_select_level2(p, unit_begin, unit_end, q, kmin, kmax, survivors, n_survivors,
                                p->topk_coarse, slice_scores, sel_ids, sel_count, sel_stride);
}

/* ---------------------------------------------------------------- decode -- */

/* o_h = sum_t softmax_t(scale * q_h . k_t) v_t over the tokens of the selected
 * blocks only.  An empty selection yields a zero output. */
int oracle_decode(const oracle_problem* p, int unit_begin, int unit_end, const void* q,
                  const void* k_pages, const void* v_pages, const int32_t* block_table,
                  const int32_t* sel_ids, const int32_t* sel_count, int sel_stride,
                  double* out)
{
    if (check_problem(p)) return -1;
    const int nb = oracle_num_blocks(p), D = p->head_dim, Hkv = p->num_kv_heads;
    const int G = p->num_q_heads / Hkv, bs = p->block_size;
    const double scale = p->softmax_scale > 0 ? p->softmax_scale : 1.0 / sqrt((double)D);
    const size_t max_tokens = (size_t)(sel_stride > 0 ? sel_stride : 1) * bs;
    double* logit = (double*)malloc(sizeof(double) * max_tokens);
    int* tok_page = (int*)malloc(sizeof(int) * max_tokens);
    int* tok_slot = (int*)malloc(sizeof(int) * max_tokens);
    if (!logit || !tok_page || !tok_slot) { free(logit); free(tok_page); free(tok_slot); return -4; }

    for (int u = unit_begin; u < unit_end; ++u) {
        int b = u / Hkv, kvh = u % Hkv;
        int count = sel_count[u];
        if (count < 0 || count > sel_stride) { free(logit); free(tok_page); free(tok_slot); return -2; }
        /* the token set T: every valid token of every selected block */
        size_t n = 0;
        for (int i = 0; i < count; ++i) {
            int j = sel_ids[(size_t)u * sel_stride + i];
            if (j < 0 || j >= nb) { free(logit); free(tok_page); free(tok_slot); return -2; }
            int page = block_table[(size_t)b * nb + j];
            if (page < 0 || page >= p->num_pages) { free(logit); free(tok_page); free(tok_slot); return -2; }
            int nt = tokens_in_block(p, j);
            for (int t = 0; t < nt; ++t) {
                tok_page[n] = page;
                tok_slot[n] = t;
                ++n;
            }
        }
        for (int g = 0; g < G; ++g) {
            int h = kvh * G + g;
            double* o = out + ((size_t)b * p->num_q_heads + h) * D;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            if (n == 0) continue;
            double m = -INFINITY;
            for (size_t i = 0; i < n; ++i) {
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += q_value(p, q, b, h, d) *
                           load_value(k_pages, kv_index(p, tok_page[i], kvh, tok_slot[i], d), p->kv_bf16);
                logit[i] = scale * dot;
                if (logit[i] > m) m = logit[i];
            }
            double denom = 0.0;
            for (size_t i = 0; i < n; ++i) {
                double w = exp(logit[i] - m);
                denom += w;
                for (int d = 0; d < D; ++d)
                    o[d] += w * load_value(v_pages, kv_index(p, tok_page[i], kvh, tok_slot[i], d), p->kv_bf16);
            }
            for (int d = 0; d < D; ++d) o[d] /= denom;
        }
    }
    free(logit);
    free(tok_page);
    free(tok_slot);
    return 0;
}

/* ------------------------------------------------------------- diff + LRU -- */

static int contains_id(const int32_t* a, int n, int32_t x)
{
    for (int i = 0; i < n; ++i)
        if (a[i] == x) return 1;
    return 0;
}

/* For one unit, with request set S_t (ascending) and the previous step's S_{t-1}:
 *   new = S_t \ S_{t-1}, dropped = S_{t-1} \ S_t          (ascending ids)
 *   hits = S_t blocks already resident, misses = the rest (ascending ids)
 *   each miss, in ascending id order, takes the lowest free slot if one exists,
 *   otherwise evicts the resident block NOT in S_t with the smallest
 *   (last_use, block id); then every block of S_t gets last_use = t.
 * Cold start: all slots free (slot_block = -1). */
int oracle_lru_step(int n_units, int step, int cache_slots,
                    const int32_t* cur_ids, const int32_t* cur_count, int cur_stride,
                    const int32_t* prev_ids, const int32_t* prev_count, int prev_stride,
                    int32_t* slot_block, int32_t* slot_last_use,
                    int32_t* hit_ids, int32_t* miss_ids, int32_t* miss_slot,
                    int32_t* evict_ids, int32_t* evict_slot,
                    int32_t* new_ids, int32_t* dropped_ids, int out_stride,
                    int32_t* counts)
{
    if (n_units < 0 || cache_slots <= 0) return -1;
    for (int u = 0; u < n_units; ++u) {
        const int32_t* S = cur_ids + (size_t)u * cur_stride;
        const int32_t* P = prev_ids + (size_t)u * prev_stride;
        int ns = cur_count[u], np = prev_count[u];
        if (ns < 0 || ns > cur_stride || np < 0 || np > prev_stride || ns > out_stride ||
            np > out_stride || ns > cache_slots) return -2;
        int32_t* blk = slot_block + (size_t)u * cache_slots;
        int32_t* last = slot_last_use + (size_t)u * cache_slots;
        int32_t* o_hit = hit_ids + (size_t)u * out_stride;
        int32_t* o_miss = miss_ids + (size_t)u * out_stride;
        int32_t* o_mslot = miss_slot + (size_t)u * out_stride;
        int32_t* o_evict = evict_ids + (size_t)u * out_stride;
        int32_t* o_eslot = evict_slot + (size_t)u * out_stride;
        int32_t* o_new = new_ids + (size_t)u * out_stride;
        int32_t* o_drop = dropped_ids + (size_t)u * out_stride;
        int n_hit = 0, n_miss = 0, n_evict = 0, n_new = 0, n_drop = 0;

        /* (a) difference against the previous step */
        for (int i = 0; i < ns; ++i)
            if (!contains_id(P, np, S[i])) o_new[n_new++] = S[i];
        for (int i = 0; i < np; ++i)
            if (!contains_id(S, ns, P[i])) o_drop[n_drop++] = P[i];

        /* (b) what is already on the GPU */
        for (int i = 0; i < ns; ++i) {
            int resident = 0;
            for (int s = 0; s < cache_slots; ++s)
                if (blk[s] == S[i]) resident = 1;
            if (resident) o_hit[n_hit++] = S[i];
            else o_miss[n_miss++] = S[i];
        }

        /* (c) place each miss: a free slot, else the least recently used block
         * that this step does not need */
        for (int i = 0; i < n_miss; ++i) {
            int slot = -1;
            for (int s = 0; s < cache_slots && slot < 0; ++s)
                if (blk[s] < 0) slot = s;
            if (slot < 0) {
                for (int s = 0; s < cache_slots; ++s) {
                    if (contains_id(S, ns, blk[s])) continue;
                    if (slot < 0 || last[s] < last[slot] ||
                        (last[s] == last[slot] && blk[s] < blk[slot]))
                        slot = s;
                }
                if (slot < 0) return -5;   /* cannot happen while |S_t| <= slots */
                o_evict[n_evict] = blk[slot];
                o_eslot[n_evict] = slot;
                ++n_evict;
            }
            blk[slot] = o_miss[i];
            o_mslot[i] = slot;
        }

        /* (d) recency update for everything this step uses */
        for (int s = 0; s < cache_slots; ++s)
            if (blk[s] >= 0 && contains_id(S, ns, blk[s])) last[s] = step;

        int32_t* c = counts + (size_t)u * 5;
        c[0] = n_hit;
        c[1] = n_miss;
        c[2] = n_evict;
        c[3] = n_new;
        c[4] = n_drop;
    }
    return 0;
}
