// extern "C" entry points of libsparse_attn: argument checks, problem geometry,
// workspace carve-up and kernel launches.  No entry allocates device memory.
#include <math.h>
#include <string.h>

#include "sa_internal.h"

namespace sa {
namespace {

constexpr int kMaxCandidates = 16384;   // per-unit selection keys staged in shared memory

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// 0 on success, else a status code; fills g.
int make_geometry(const sparse_attn_params* p, Geometry* g)
{
    if (!p || !g) return SPARSE_ATTN_INVALID_ARG;
    memset(g, 0, sizeof *g);
    if (p->batch < 0 || p->num_q_heads < 1 || p->num_kv_heads < 1 || p->head_dim < 1 ||
        p->n_tokens < 0 || p->block_size < 1 || p->num_pages < 0 || p->window_tokens < 0 ||
        p->topk < 0 || p->topk_coarse < 0 || p->num_reserve < 0 || p->num_queries < 0 ||
        (p->capacity_tokens != 0 && p->capacity_tokens < p->n_tokens))
        return SPARSE_ATTN_INVALID_ARG;
    if (p->num_q_heads % p->num_kv_heads != 0) return SPARSE_ATTN_INVALID_ARG;
    if (p->two_level != 0 && p->two_level != 1) return SPARSE_ATTN_INVALID_ARG;
    if (p->score_kind != SPARSE_ATTN_SCORE_QUEST && p->score_kind != SPARSE_ATTN_SCORE_MEAN)
        return SPARSE_ATTN_INVALID_ARG;
    if ((p->kv_dtype != SPARSE_ATTN_F32 && p->kv_dtype != SPARSE_ATTN_BF16) ||
        (p->q_dtype != SPARSE_ATTN_F32 && p->q_dtype != SPARSE_ATTN_BF16))
        return SPARSE_ATTN_INVALID_ARG;
    if (!(p->softmax_scale == p->softmax_scale) || isinf(p->softmax_scale)) return SPARSE_ATTN_INVALID_ARG;

    const int G = p->num_q_heads / p->num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return SPARSE_ATTN_UNSUPPORTED;
    if (p->head_dim != 64 && p->head_dim != 128) return SPARSE_ATTN_UNSUPPORTED;
    const int bs = p->block_size;
    if (bs != 8 && bs != 16 && bs != 32 && bs != 64 && bs != 128) return SPARSE_ATTN_UNSUPPORTED;
    const bool kv_bf16 = p->kv_dtype == SPARSE_ATTN_BF16;
    if (!decode_supported(p->head_dim, kv_bf16, bs, G)) return SPARSE_ATTN_UNSUPPORTED;

    g->B = p->batch;
    g->Hq = p->num_q_heads;
    g->Hkv = p->num_kv_heads;
    g->G = G;
    g->D = p->head_dim;
    g->N = p->n_tokens;
    g->bs = bs;
    g->nb = (p->n_tokens + bs - 1) / bs;
    g->num_pages = p->num_pages;
    if (g->nb > kMaxCandidates) return SPARSE_ATTN_UNSUPPORTED;
    if (g->B > 0 && g->nb > 0 && g->num_pages < 1) return SPARSE_ATTN_INVALID_ARG;
    if (p->window_tokens > 0) {
        int first_tok = p->n_tokens - p->window_tokens;
        if (first_tok < 0) first_tok = 0;
        g->win_first = first_tok / bs;
    } else {
        g->win_first = g->nb;
    }
    g->win_count = g->nb - g->win_first;
    g->n_cand = g->win_first;
    g->topk = p->topk;
    g->n_reserve = p->num_reserve;
    g->Q = p->num_queries > 1 ? p->num_queries : 1;
    if (g->Q > 1 && (p->two_level != 0 || !kv_bf16)) return SPARSE_ATTN_UNSUPPORTED;
    if ((long long)g->Q * G > (1 << 20)) return SPARSE_ATTN_UNSUPPORTED;
    const int k_max = p->topk < g->n_cand ? p->topk : g->n_cand;
    const int r_max = p->num_reserve < g->n_cand ? p->num_reserve : g->n_cand;
    const int stride = k_max + r_max + g->win_count;
    g->sel_stride = stride > 0 ? stride : 1;
    g->kv_bf16 = kv_bf16;
    g->q_bf16 = p->q_dtype == SPARSE_ATTN_BF16;
    g->two_level = p->two_level != 0;
    g->score_kind = p->score_kind;
    if (g->two_level) {
        if (p->coarse_block < bs || p->coarse_block % bs != 0) return SPARSE_ATTN_INVALID_ARG;
        g->coarse_block = p->coarse_block;
        g->per_coarse = p->coarse_block / bs;
        g->n_coarse = (p->n_tokens + p->coarse_block - 1) / p->coarse_block;
        g->topk_coarse = p->topk_coarse;
        if (g->n_coarse > kMaxCandidates) return SPARSE_ATTN_UNSUPPORTED;
        if ((long long)g->topk_coarse * g->per_coarse > kMaxCandidates) return SPARSE_ATTN_UNSUPPORTED;
        g->mean_block = p->coarse_block;
    } else {
        g->mean_block = bs;
    }
    g->n_mean = (p->n_tokens + g->mean_block - 1) / g->mean_block;
    const long long cap = p->capacity_tokens > 0 ? p->capacity_tokens : p->n_tokens;
    g->nb_cap = int((cap + bs - 1) / bs);
    g->n_mean_cap = int((cap + g->mean_block - 1) / g->mean_block);
    const float scale = p->softmax_scale > 0.f ? p->softmax_scale : 1.0f / sqrtf(float(p->head_dim));
    g->scale_log2 = scale * 1.4426950408889634f;
    return SPARSE_ATTN_OK;
}

int status_of(cudaError_t e) { return e == cudaSuccess ? SPARSE_ATTN_OK : SPARSE_ATTN_CUDA_ERROR; }

}  // namespace

int num_sms()
{
    static std::atomic<int> cached[64];   // zero-initialised (static storage)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

WorkspaceLayout workspace_layout(const Geometry& g)
{
    WorkspaceLayout L{};
    const size_t units = size_t(g.units());
    int cols = g.n_cand;
    if (g.two_level) {
        cols = g.n_coarse;
        if (g.topk_coarse * g.per_coarse > cols) cols = g.topk_coarse * g.per_coarse;
    }
    L.score_cols = cols > 0 ? cols : 1;
    L.blocks_per_split = decode_blocks_per_item(g.D, g.kv_bf16, g.bs);
    L.max_splits = (g.sel_stride + L.blocks_per_split - 1) / L.blocks_per_split;
    if (L.max_splits < 1) L.max_splits = 1;
    const size_t heads = size_t(g.B) * g.Hq * g.Q;   // query rows (Q queries per sequence)
    const size_t dec_cells = units * size_t(g.Q > 1 ? mq_row_tiles(g.Q, g.G) : 1);

    size_t off = 0;
    // one 256-byte header: error word, the select kernel's work counters (4-11), the
    // fused step's publish-queue counters (12-23), the wait limit (24-31) and the fused
    // step's epoch and completion count (32-39)
    L.err = 0;
    L.sel_work = 4;
    L.sel_done = 8;
    L.dec_work = 12;
    L.dec_done = 16;
    off = 256;
    L.sel_counters = off;     off = align256(off + units * sizeof(uint32_t));
    L.dec_counters = off;     off = align256(off + dec_cells * sizeof(uint32_t));
    L.l1_counters = off;      off = align256(off + units * sizeof(uint32_t));
    L.ready = off;            off = align256(off + units * sizeof(uint32_t));
    L.queue = off;            off = align256(off + units * sizeof(uint32_t));
    L.scores = off;           off = align256(off + units * L.score_cols * sizeof(float));
    L.survivors = off;        off = align256(off + units * size_t(g.topk_coarse > 0 ? g.topk_coarse : 1) * sizeof(int32_t));
    L.n_survivors = off;      off = align256(off + units * sizeof(int32_t));
    L.part_m = off;           off = align256(off + heads * L.max_splits * sizeof(float));
    L.part_l = off;           off = align256(off + heads * L.max_splits * sizeof(float));
    L.part_o = off;           off = align256(off + heads * L.max_splits * size_t(g.D) * sizeof(float));
    L.total = off;
    return L;
}

}  // namespace sa

using namespace sa;

extern "C" {

const char* sparse_attn_status_string(int status)
{
    switch (status) {
        case SPARSE_ATTN_OK: return "ok";
        case SPARSE_ATTN_INVALID_ARG: return "invalid argument";
        case SPARSE_ATTN_UNSUPPORTED: return "unsupported configuration";
        case SPARSE_ATTN_CUDA_ERROR: return "CUDA launch error";
        case SPARSE_ATTN_DEVICE_BOUNDS: return "device-side bounds error";
        default: return "unknown status";
    }
}

int32_t sparse_attn_num_blocks(const sparse_attn_params* p)
{
    Geometry g;
    return make_geometry(p, &g) == SPARSE_ATTN_OK ? g.nb : -1;
}

int32_t sparse_attn_sel_stride(const sparse_attn_params* p)
{
    Geometry g;
    return make_geometry(p, &g) == SPARSE_ATTN_OK ? g.sel_stride : -1;
}

int sparse_attn_workspace_size(const sparse_attn_params* p, size_t* bytes)
{
    if (!bytes) return SPARSE_ATTN_INVALID_ARG;
    Geometry g;
    int st = make_geometry(p, &g);
    if (st) return st;
    size_t total = workspace_layout(g).total;
    if (p->capacity_tokens > p->n_tokens) {
        // Every length up to the capacity: each term of the layout grows with the
        // length except the window's block count, which alternates between two values
        // as the window slides over block boundaries; bound that one separately.
        sparse_attn_params pc = *p;
        pc.n_tokens = p->capacity_tokens;
        Geometry gc;
        st = make_geometry(&pc, &gc);
        if (st) return st;
        if (p->window_tokens > 0) {
            int win_max = (p->window_tokens + gc.bs - 1) / gc.bs + 1;
            if (win_max > gc.nb) win_max = gc.nb;
            const int k_max = gc.topk < gc.n_cand ? gc.topk : gc.n_cand;
            const int r_max = gc.n_reserve < gc.n_cand ? gc.n_reserve : gc.n_cand;
            if (k_max + r_max + win_max > gc.sel_stride) gc.sel_stride = k_max + r_max + win_max;
        }
        const size_t tc = workspace_layout(gc).total;
        if (tc > total) total = tc;
    }
    *bytes = total;
    return SPARSE_ATTN_OK;
}

int sparse_attn_workspace_init(void* ws, size_t ws_bytes, sparse_attn_stream stream)
{
    if (!ws || !aligned(ws, 256) || ws_bytes < 256) return SPARSE_ATTN_INVALID_ARG;
    return status_of(cudaMemsetAsync(ws, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream)));
}

int sparse_attn_workspace_set_wait_limit(void* ws, size_t ws_bytes, uint64_t cycles, sparse_attn_stream stream)
{
    if (!ws || !aligned(ws, 256) || ws_bytes < 256) return SPARSE_ATTN_INVALID_ARG;
    // pageable source: the runtime stages the 8 bytes before returning
    const unsigned long long v = cycles;
    return status_of(cudaMemcpyAsync(static_cast<char*>(ws) + kHdrWaitLimitByte, &v, sizeof v,
                                     cudaMemcpyHostToDevice, reinterpret_cast<cudaStream_t>(stream)));
}

static int meta_common(const sparse_attn_params* p, int32_t first_token, const void* k_pages,
                       const int32_t* block_table, void* kmin, void* kmax, float* kmean, void* ws,
                       size_t ws_bytes, sparse_attn_stream stream)
{
    Geometry g;
    int st = make_geometry(p, &g);
    if (st) return st;
    if (first_token < 0 || first_token > g.N) return SPARSE_ATTN_INVALID_ARG;
    const WorkspaceLayout L = workspace_layout(g);
    // the metadata kernels touch only the header's error word
    if (!ws || !aligned(ws, 256) || ws_bytes < 256) return SPARSE_ATTN_INVALID_ARG;
    const bool need_mean = g.two_level || g.score_kind == SPARSE_ATTN_SCORE_MEAN;
    if (need_mean && !kmean) return SPARSE_ATTN_INVALID_ARG;
    if (g.units() > 0 && g.nb > 0) {
        if (!k_pages || !block_table || !kmin || !kmax) return SPARSE_ATTN_INVALID_ARG;
        if (!aligned(k_pages, 16) || !aligned(kmin, 16) || !aligned(kmax, 16) ||
            !aligned(block_table, 4) || (kmean && !aligned(kmean, 16)))
            return SPARSE_ATTN_INVALID_ARG;
    }
    if (first_token == g.N && first_token > 0) return SPARSE_ATTN_OK;   // nothing appended
    char* w = static_cast<char*>(ws);
    return status_of(launch_build_meta(g, k_pages, block_table, kmin, kmax, need_mean ? kmean : nullptr,
                                       reinterpret_cast<uint32_t*>(w + L.err), first_token,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

int sparse_attn_build_meta(const sparse_attn_params* p, const void* k_pages,
                           const int32_t* block_table, void* kmin, void* kmax, float* kmean,
                           void* ws, size_t ws_bytes, sparse_attn_stream stream)
{
    return meta_common(p, 0, k_pages, block_table, kmin, kmax, kmean, ws, ws_bytes, stream);
}

int sparse_attn_append_meta(const sparse_attn_params* p, int32_t n_old, const void* k_pages,
                            const int32_t* block_table, void* kmin, void* kmax, float* kmean,
                            void* ws, size_t ws_bytes, sparse_attn_stream stream)
{
    return meta_common(p, n_old, k_pages, block_table, kmin, kmax, kmean, ws, ws_bytes, stream);
}

static int select_common(const sparse_attn_params* p, const void* q, const void* kmin,
                         const void* kmax, const float* kmean, const int32_t* reserve_ids,
                         int32_t* sel_ids, int32_t* sel_count, void* ws, size_t ws_bytes,
                         sparse_attn_stream stream)
{
    Geometry g;
    int st = make_geometry(p, &g);
    if (st) return st;
    if (g.n_reserve > 0 && g.units() > 0 && (!reserve_ids || !aligned(reserve_ids, 4)))
        return SPARSE_ATTN_INVALID_ARG;
    const WorkspaceLayout L = workspace_layout(g);
    if (!ws || !aligned(ws, 256) || ws_bytes < L.total) return SPARSE_ATTN_INVALID_ARG;
    if (g.units() > 0) {
        if (!q || !sel_ids || !sel_count || !aligned(q, 16) || !aligned(sel_ids, 4) ||
            !aligned(sel_count, 4))
            return SPARSE_ATTN_INVALID_ARG;
        const bool need_mean = g.two_level || g.score_kind == SPARSE_ATTN_SCORE_MEAN;
        const bool need_box = g.two_level || g.score_kind == SPARSE_ATTN_SCORE_QUEST;
        if (g.nb > 0) {
            if (need_mean && (!kmean || !aligned(kmean, 16))) return SPARSE_ATTN_INVALID_ARG;
            if (need_box && (!kmin || !kmax || !aligned(kmin, 16) || !aligned(kmax, 16)))
                return SPARSE_ATTN_INVALID_ARG;
        }
    }
    return status_of(launch_select(g, L, static_cast<char*>(ws), q, kmin, kmax, kmean, reserve_ids, sel_ids,
                                   sel_count, reinterpret_cast<cudaStream_t>(stream)));
}

int sparse_attn_select(const sparse_attn_params* p, const void* q, const void* kmin,
                       const void* kmax, const float* kmean, int32_t* sel_ids,
                       int32_t* sel_count, void* ws, size_t ws_bytes, sparse_attn_stream stream)
{
    if (p && p->num_reserve != 0) return SPARSE_ATTN_INVALID_ARG;   // use sparse_attn_select_reserved
    return select_common(p, q, kmin, kmax, kmean, nullptr, sel_ids, sel_count, ws, ws_bytes, stream);
}

int sparse_attn_select_reserved(const sparse_attn_params* p, const void* q, const void* kmin,
                                const void* kmax, const float* kmean, const int32_t* reserve_ids,
                                int32_t* sel_ids, int32_t* sel_count, void* ws, size_t ws_bytes,
                                sparse_attn_stream stream)
{
    return select_common(p, q, kmin, kmax, kmean, reserve_ids, sel_ids, sel_count, ws, ws_bytes, stream);
}

int32_t sparse_attn_topk_for_length(int32_t n_tokens, int32_t block_size)
{
    if (n_tokens < 0 || block_size < 1) return -1;
    const long long nb = ((long long)n_tokens + block_size - 1) / block_size;
    if (n_tokens <= 8192) return int32_t(nb);                 // short contexts keep every block
    const long long percent = n_tokens <= 16384 ? 15 : (n_tokens <= 32768 ? 10 : 5);
    const long long k = nb * percent / 100;
    return int32_t(k > 1 ? k : 1);
}

int sparse_attn_decode(const sparse_attn_params* p, const void* q, const void* k_pages,
                       const void* v_pages, const int32_t* block_table, const int32_t* sel_ids,
                       const int32_t* sel_count, float* out, void* ws, size_t ws_bytes,
                       sparse_attn_stream stream)
{
    Geometry g;
    int st = make_geometry(p, &g);
    if (st) return st;
    const WorkspaceLayout L = workspace_layout(g);
    if (!ws || !aligned(ws, 256) || ws_bytes < L.total) return SPARSE_ATTN_INVALID_ARG;
    if (g.units() > 0) {
        if (!q || !out || !sel_ids || !sel_count || !aligned(q, 16) || !aligned(out, 16) ||
            !aligned(sel_ids, 4) || !aligned(sel_count, 4))
            return SPARSE_ATTN_INVALID_ARG;
        if (g.nb > 0 && (!k_pages || !v_pages || !block_table || !aligned(k_pages, 16) ||
                         !aligned(v_pages, 16) || !aligned(block_table, 4)))
            return SPARSE_ATTN_INVALID_ARG;
    }
    if (g.Q > 1)
        return status_of(launch_decode_mq(g, L, static_cast<char*>(ws), q, k_pages, v_pages, block_table,
                                          sel_ids, sel_count, out, reinterpret_cast<cudaStream_t>(stream)));
    return status_of(launch_decode(g, L, static_cast<char*>(ws), q, k_pages, v_pages, block_table,
                                   sel_ids, sel_count, out, nullptr, 0, reinterpret_cast<cudaStream_t>(stream)));
}

int32_t sparse_attn_step_launches(const sparse_attn_params* p)
{
    Geometry g;
    if (make_geometry(p, &g) != SPARSE_ATTN_OK || !step_supported(g)) return -1;
    return step_launches(g, workspace_layout(g));
}

int sparse_attn_step(const sparse_attn_params* p, const void* q, const void* kmin, const void* kmax,
                     const float* kmean, const int32_t* reserve_ids, const void* k_pages,
                     const void* v_pages, const int32_t* block_table, int32_t* sel_ids,
                     int32_t* sel_count, float* out, void* ws, size_t ws_bytes, sparse_attn_stream stream)
{
    Geometry g;
    int st = make_geometry(p, &g);
    if (st) return st;
    if (!step_supported(g)) return SPARSE_ATTN_UNSUPPORTED;
    if (g.n_reserve > 0 && g.units() > 0 && (!reserve_ids || !aligned(reserve_ids, 4)))
        return SPARSE_ATTN_INVALID_ARG;
    const WorkspaceLayout L = workspace_layout(g);
    if (!ws || !aligned(ws, 256) || ws_bytes < L.total) return SPARSE_ATTN_INVALID_ARG;
    if (g.units() > 0) {
        if (!q || !out || !sel_ids || !sel_count || !aligned(q, 16) || !aligned(out, 16) ||
            !aligned(sel_ids, 4) || !aligned(sel_count, 4))
            return SPARSE_ATTN_INVALID_ARG;
        if (g.nb > 0) {
            const bool mean = g.score_kind == SPARSE_ATTN_SCORE_MEAN;
            if (mean && (!kmean || !aligned(kmean, 16))) return SPARSE_ATTN_INVALID_ARG;
            if (!mean && (!kmin || !kmax || !aligned(kmin, 16) || !aligned(kmax, 16)))
                return SPARSE_ATTN_INVALID_ARG;
            if (!k_pages || !v_pages || !block_table || !aligned(k_pages, 16) || !aligned(v_pages, 16) ||
                !aligned(block_table, 4))
                return SPARSE_ATTN_INVALID_ARG;
        }
    }
    const cudaError_t e = launch_step(g, L, static_cast<char*>(ws), q, kmin, kmax, kmean, reserve_ids, k_pages,
                                      v_pages, block_table, sel_ids, sel_count, out,
                                      reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return SPARSE_ATTN_UNSUPPORTED;
    return status_of(e);
}

static int diff_impl(const sparse_attn_params* p, int32_t step, const int32_t* sel_ids,
                     const int32_t* sel_count, const int32_t* prev_ids,
                     const int32_t* prev_count, int32_t cache_slots, int32_t* slot_block,
                     int32_t* slot_last_use, int32_t* hit_ids, int32_t* miss_ids,
                     int32_t* miss_slot, int32_t* evict_ids, int32_t* evict_slot,
                     int32_t* new_ids, int32_t* dropped_ids, int32_t* counts, int32_t* sel_slot,
                     void* ws, size_t ws_bytes, sparse_attn_stream stream)
{
    Geometry g;
    int st = make_geometry(p, &g);
    if (st) return st;
    const WorkspaceLayout L = workspace_layout(g);
    if (!ws || !aligned(ws, 256) || ws_bytes < L.total) return SPARSE_ATTN_INVALID_ARG;
    if (cache_slots < 1 || cache_slots > 1024 || g.sel_stride > cache_slots) return SPARSE_ATTN_INVALID_ARG;
    if (g.units() > 0) {
        const void* ptrs[] = {sel_ids, sel_count, prev_ids, prev_count, slot_block, slot_last_use,
                              hit_ids, miss_ids, miss_slot, evict_ids, evict_slot, new_ids,
                              dropped_ids, counts};
        for (const void* ptr : ptrs)
            if (!ptr || !aligned(ptr, 4)) return SPARSE_ATTN_INVALID_ARG;
    }
    char* w = static_cast<char*>(ws);
    return status_of(launch_diff(g, step, sel_ids, sel_count, prev_ids, prev_count, cache_slots,
                                 slot_block, slot_last_use, hit_ids, miss_ids, miss_slot, evict_ids,
                                 evict_slot, new_ids, dropped_ids, counts,
                                 reinterpret_cast<uint32_t*>(w + L.err),
                                 reinterpret_cast<cudaStream_t>(stream), sel_slot));
}

int sparse_attn_diff(const sparse_attn_params* p, int32_t step, const int32_t* sel_ids,
                     const int32_t* sel_count, const int32_t* prev_ids,
                     const int32_t* prev_count, int32_t cache_slots, int32_t* slot_block,
                     int32_t* slot_last_use, int32_t* hit_ids, int32_t* miss_ids,
                     int32_t* miss_slot, int32_t* evict_ids, int32_t* evict_slot,
                     int32_t* new_ids, int32_t* dropped_ids, int32_t* counts, void* ws,
                     size_t ws_bytes, sparse_attn_stream stream)
{
    return diff_impl(p, step, sel_ids, sel_count, prev_ids, prev_count, cache_slots, slot_block, slot_last_use,
                     hit_ids, miss_ids, miss_slot, evict_ids, evict_slot, new_ids, dropped_ids, counts, nullptr, ws,
                     ws_bytes, stream);
}

int sparse_attn_diff_slots(const sparse_attn_params* p, int32_t step, const int32_t* sel_ids,
                           const int32_t* sel_count, const int32_t* prev_ids, const int32_t* prev_count,
                           int32_t cache_slots, int32_t* slot_block, int32_t* slot_last_use, int32_t* hit_ids,
                           int32_t* miss_ids, int32_t* miss_slot, int32_t* evict_ids, int32_t* evict_slot,
                           int32_t* new_ids, int32_t* dropped_ids, int32_t* counts, int32_t* sel_slot, void* ws,
                           size_t ws_bytes, sparse_attn_stream stream)
{
    if (!sel_slot || !aligned(sel_slot, 4)) return SPARSE_ATTN_INVALID_ARG;
    return diff_impl(p, step, sel_ids, sel_count, prev_ids, prev_count, cache_slots, slot_block, slot_last_use,
                     hit_ids, miss_ids, miss_slot, evict_ids, evict_slot, new_ids, dropped_ids, counts, sel_slot, ws,
                     ws_bytes, stream);
}

int sparse_attn_get_device_error(void* ws, size_t ws_bytes, sparse_attn_stream stream, uint32_t* flags)
{
    if (!ws || !flags || !aligned(ws, 256) || ws_bytes < 256) return SPARSE_ATTN_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, ws, sizeof word, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, sizeof word, s);
    if (e != cudaSuccess) return SPARSE_ATTN_CUDA_ERROR;
    *flags = word;
    return word ? SPARSE_ATTN_DEVICE_BOUNDS : SPARSE_ATTN_OK;
}

// ---- slot pool: misses from a host-resident store, decode through the slots ----
// A device-accessible address for a caller buffer that may be pinned / registered host
// memory (page-first K/V store) or device memory; null for unregistered host memory.
static const void* device_view(const void* ptr)
{
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return ptr;
    if (at.type == cudaMemoryTypeHost) return at.devicePointer;
    return nullptr;
}

int sparse_attn_slot_map(const sparse_attn_params* p, const int32_t* sel_ids, const int32_t* sel_count,
                         const int32_t* slot_block, int32_t cache_slots, int32_t* sel_slot, void* ws,
                         size_t ws_bytes, sparse_attn_stream stream)
{
    Geometry g;
    int st = make_geometry(p, &g);
    if (st) return st;
    const WorkspaceLayout L = workspace_layout(g);
    if (!ws || !aligned(ws, 256) || ws_bytes < L.total) return SPARSE_ATTN_INVALID_ARG;
    if (cache_slots < 1 || cache_slots > 1024 || g.sel_stride > cache_slots) return SPARSE_ATTN_INVALID_ARG;
    if (g.units() > 0 && (!sel_ids || !sel_count || !slot_block || !sel_slot || !aligned(sel_ids, 4) ||
                          !aligned(sel_count, 4) || !aligned(slot_block, 4) || !aligned(sel_slot, 4)))
        return SPARSE_ATTN_INVALID_ARG;
    return status_of(launch_slot_map(g, sel_ids, sel_count, slot_block, cache_slots, sel_slot,
                                     reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + L.err),
                                     reinterpret_cast<cudaStream_t>(stream)));
}

int sparse_attn_load_misses(const sparse_attn_params* p, const void* host_k_pages, const void* host_v_pages,
                            const int32_t* block_table, const int32_t* miss_ids, const int32_t* miss_slot,
                            const int32_t* counts, int32_t cache_slots, void* pool_k, void* pool_v, void* ws,
                            size_t ws_bytes, sparse_attn_stream stream)
{
    Geometry g;
    int st = make_geometry(p, &g);
    if (st) return st;
    const WorkspaceLayout L = workspace_layout(g);
    if (!ws || !aligned(ws, 256) || ws_bytes < L.total) return SPARSE_ATTN_INVALID_ARG;
    if (cache_slots < 1 || cache_slots > 1024 || g.sel_stride > cache_slots) return SPARSE_ATTN_INVALID_ARG;
    if (g.units() == 0 || g.nb == 0) return SPARSE_ATTN_OK;
    const void* hk = host_k_pages ? device_view(host_k_pages) : nullptr;
    const void* hv = host_v_pages ? device_view(host_v_pages) : nullptr;
    if (!hk || !hv || !aligned(hk, 16) || !aligned(hv, 16) || !block_table || !miss_ids || !miss_slot ||
        !counts || !pool_k || !pool_v || !aligned(pool_k, 16) || !aligned(pool_v, 16) ||
        !aligned(block_table, 4) || !aligned(miss_ids, 4) || !aligned(miss_slot, 4) || !aligned(counts, 4))
        return SPARSE_ATTN_INVALID_ARG;
    return status_of(launch_load_misses(g, hk, hv, block_table, miss_ids, miss_slot, counts, cache_slots,
                                        pool_k, pool_v,
                                        reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + L.err),
                                        reinterpret_cast<cudaStream_t>(stream)));
}

int sparse_attn_decode_slots(const sparse_attn_params* p, const void* q, const void* pool_k,
                             const void* pool_v, int32_t cache_slots, const int32_t* sel_ids,
                             const int32_t* sel_slot, const int32_t* sel_count, float* out, void* ws,
                             size_t ws_bytes, sparse_attn_stream stream)
{
    Geometry g;
    int st = make_geometry(p, &g);
    if (st) return st;
    const WorkspaceLayout L = workspace_layout(g);
    if (!ws || !aligned(ws, 256) || ws_bytes < L.total) return SPARSE_ATTN_INVALID_ARG;
    if (cache_slots < 1 || cache_slots > 1024 || g.sel_stride > cache_slots) return SPARSE_ATTN_INVALID_ARG;
    if (g.Q > 1) return SPARSE_ATTN_UNSUPPORTED;
    if (g.units() > 0) {
        if (!q || !out || !sel_ids || !sel_slot || !sel_count || !aligned(q, 16) || !aligned(out, 16) ||
            !aligned(sel_ids, 4) || !aligned(sel_slot, 4) || !aligned(sel_count, 4))
            return SPARSE_ATTN_INVALID_ARG;
        if (g.nb > 0 && (!pool_k || !pool_v || !aligned(pool_k, 16) || !aligned(pool_v, 16)))
            return SPARSE_ATTN_INVALID_ARG;
    }
    return status_of(launch_decode(g, L, static_cast<char*>(ws), q, pool_k, pool_v, nullptr, sel_ids,
                                   sel_count, out, sel_slot, cache_slots,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

int sparse_attn_decode_slots_io(const sparse_attn_params* p, const void* q, void* pool_k, void* pool_v,
                                int32_t cache_slots, const int32_t* sel_ids, const int32_t* sel_slot,
                                const int32_t* sel_count, const void* host_k_pages, const void* host_v_pages,
                                const int32_t* block_table, const int32_t* miss_ids, const int32_t* miss_slot,
                                const int32_t* counts, float* out, void* ws, size_t ws_bytes,
                                sparse_attn_stream stream)
{
    Geometry g;
    int st = make_geometry(p, &g);
    if (st) return st;
    const WorkspaceLayout L = workspace_layout(g);
    if (!ws || !aligned(ws, 256) || ws_bytes < L.total) return SPARSE_ATTN_INVALID_ARG;
    if (cache_slots < 1 || cache_slots > 1024 || g.sel_stride > cache_slots) return SPARSE_ATTN_INVALID_ARG;
    if (g.Q > 1) return SPARSE_ATTN_UNSUPPORTED;
    if (!g.kv_bf16) return SPARSE_ATTN_UNSUPPORTED;
    if (g.units() == 0) return SPARSE_ATTN_OK;
    if (!q || !out || !sel_ids || !sel_slot || !sel_count || !aligned(q, 16) || !aligned(out, 16) ||
        !aligned(sel_ids, 4) || !aligned(sel_slot, 4) || !aligned(sel_count, 4))
        return SPARSE_ATTN_INVALID_ARG;
    if (g.nb == 0)   // nothing selected: the plain slot decode writes the zero output
        return status_of(launch_decode(g, L, static_cast<char*>(ws), q, pool_k, pool_v, nullptr, sel_ids, sel_count,
                                       out, sel_slot, cache_slots, reinterpret_cast<cudaStream_t>(stream)));
    const void* hk = host_k_pages ? device_view(host_k_pages) : nullptr;
    const void* hv = host_v_pages ? device_view(host_v_pages) : nullptr;
    if (!hk || !hv || !aligned(hk, 16) || !aligned(hv, 16) || !block_table || !miss_ids || !miss_slot || !counts ||
        !pool_k || !pool_v || !aligned(pool_k, 16) || !aligned(pool_v, 16) || !aligned(block_table, 4) ||
        !aligned(miss_ids, 4) || !aligned(miss_slot, 4) || !aligned(counts, 4))
        return SPARSE_ATTN_INVALID_ARG;
    const SlotIo io{hk, hv, miss_ids, miss_slot, counts};
    return status_of(launch_decode(g, L, static_cast<char*>(ws), q, pool_k, pool_v, block_table, sel_ids, sel_count,
                                   out, sel_slot, cache_slots, reinterpret_cast<cudaStream_t>(stream), nullptr, &io));
}

// ---- selection for callers that cannot allocate device memory ---------------
// The scratch lives in this file-scope array; host code needs its device address,
// looked up once per device (cudaGetSymbolAddress) with that device current.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SPARSE_ATTN_NOALLOC_SCRATCH_BYTES];

// Two host threads making the first call on a device at once both look the address up
// and store the same value (atomic slots, no data race).  The address belongs to the
// device's current context: after a cudaDeviceReset the cached value is stale, so a
// process that resets a device must not call sparse_attn_select_noalloc on it again.
static void* noalloc_scratch_address(int* status)
{
    static std::atomic<void*> cached[64];   // zero-initialised (static storage)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *status = SPARSE_ATTN_CUDA_ERROR;
        return nullptr;
    }
    void* ptr = cached[dev].load(std::memory_order_acquire);
    if (ptr == nullptr) {
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
            *status = SPARSE_ATTN_CUDA_ERROR;
            return nullptr;
        }
        cached[dev].store(ptr, std::memory_order_release);
    }
    *status = SPARSE_ATTN_OK;
    return ptr;
}

int sparse_attn_select_noalloc(const sparse_attn_params* p, const void* q, const void* kmin,
                               const void* kmax, const float* kmean, int32_t* sel_ids,
                               int32_t* sel_count, sparse_attn_stream stream)
{
    Geometry g;
    int st = make_geometry(p, &g);
    if (st) return st;
    if (g.two_level || g.n_reserve != 0) return SPARSE_ATTN_UNSUPPORTED;
    const WorkspaceLayout L = workspace_layout(g);
    // select touches the header, the counter rows and the score rows only
    const size_t need = L.scores + size_t(g.units()) * L.score_cols * sizeof(float);
    if (need > SPARSE_ATTN_NOALLOC_SCRATCH_BYTES) return SPARSE_ATTN_UNSUPPORTED;
    if (g.units() > 0) {
        if (!q || !sel_ids || !sel_count || !aligned(q, 16) || !aligned(sel_ids, 4) ||
            !aligned(sel_count, 4))
            return SPARSE_ATTN_INVALID_ARG;
        const bool need_mean = g.score_kind == SPARSE_ATTN_SCORE_MEAN;
        if (g.nb > 0) {
            if (need_mean && (!kmean || !aligned(kmean, 16))) return SPARSE_ATTN_INVALID_ARG;
            if (!need_mean && (!kmin || !kmax || !aligned(kmin, 16) || !aligned(kmax, 16)))
                return SPARSE_ATTN_INVALID_ARG;
        }
    }
    char* ws = static_cast<char*>(noalloc_scratch_address(&st));
    if (st) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // error word and completion counters must start at zero; scores need no clearing
    if (cudaMemsetAsync(ws, 0, L.scores, s) != cudaSuccess) return SPARSE_ATTN_CUDA_ERROR;
    return status_of(launch_select(g, L, ws, q, kmin, kmax, kmean, nullptr, sel_ids, sel_count, s));
}

int sparse_attn_select_noalloc_device_error(sparse_attn_stream stream, uint32_t* flags)
{
    if (!flags) return SPARSE_ATTN_INVALID_ARG;
    int st = SPARSE_ATTN_OK;
    void* ws = noalloc_scratch_address(&st);
    if (st) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, ws, sizeof word, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, sizeof word, s);
    if (e != cudaSuccess) return SPARSE_ATTN_CUDA_ERROR;
    *flags = word;
    return word ? SPARSE_ATTN_DEVICE_BOUNDS : SPARSE_ATTN_OK;
}

}  // extern "C"
