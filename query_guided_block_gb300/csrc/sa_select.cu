// Query-guided block selection: score every candidate block from its metadata, then
// a per-(sequence, KV head) top-k united with the local window.
//
// Scoring ("SGLang分层稀疏注意力技术解析与优化实践" §3.1.2, the bound of q.k over a block's
// key bounding box), summed over the query heads of a GQA group:
//     s(j) = sum_h sum_d max(q_h[d] * min_j[d], q_h[d] * max_j[d]).
// Since min_j <= max_j, max(q*lo, q*hi) = max(q,0)*hi + min(q,0)*lo, and the sum over
// heads folds into two D-vectors computed once per CTA:
//     P[d] = sum_h max(q_h[d], 0),  Nn[d] = sum_h min(q_h[d], 0),
//     s(j) = P . max_j + Nn . min_j.
// So a G-head group costs two FMAs per metadata element pair, whatever G is, and the
// kernel streams the metadata at HBM rate.  Mean scoring (SparDA page §3.1; HiSparse->QSA
// page §2.2 level 1) is s(j) = (sum_h q_h) . mean_j.  Scores are fp32 (HiSparse->QSA §5.1).
//
// Selection (SparDA page §3.2 fixed top-k; HiSparse->QSA §2.2 window level): the k
// largest scores by (score desc, block id asc), plus the window blocks, ascending.
//
// Work split: a persistent grid streams chunks of metadata rows through a multi-stage
// bulk-copy pipeline (see the kernel below); a half-warp (D = 128, bf16) scores one
// row from shared memory.  Scores go to an L2-resident workspace row.  The CTA that
// scores a unit's last chunk (device-scope counter, no waiting) runs a radix select
// over the unit's order-preserving uint32 keys in shared memory: four 8-bit digit
// passes with warp-aggregated shared-memory histograms, early exit once a digit bin
// holds exactly the remaining count, then a stable tie rule (lower id first) and an
// ordered compaction by warp ballots.
#include "sa_select_body.cuh"

namespace sa {
namespace {

template <int KIND, bool MBF16, int D>
__global__ void __launch_bounds__(kSelThreads) select_kernel(SelectArgs a, uint32_t* ready)
{
    select_body<KIND, MBF16, D>(a, ready);
}

template <int KIND, bool MBF16, int D>
cudaError_t launch_select_t(const SelectArgs& a0, int units, uint32_t* ready, cudaStream_t s)
{
    SelectArgs a = a0;
    set_chunking<KIND, MBF16, D>(a, units);
    const size_t keys_bytes = size_t(kSelThreads) * key_tile(a.n_cand) * sizeof(uint32_t);
    // two CTAs per SM when they fit: dynamic stages + keys, plus static (histogram) and
    // the per-CTA reservation
    constexpr size_t kStatic = 13 * 1024;
    a.stages = (2 * (3 * size_t(kStageBytes) + keys_bytes + kStatic) <= size_t(kSmemPerSm)) ? 3 : 2;
    const size_t smem = size_t(a.stages) * kStageBytes + keys_bytes;
    static bool configured = false;   // once per instantiation, before any graph capture
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(select_kernel<KIND, MBF16, D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(2 * kStageBytes + kMaxSelectKeys * sizeof(uint32_t)));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int per_sm = (2 * (smem + kStatic) <= size_t(kSmemPerSm)) ? 2 : 1;
    int ctas = num_sms() * per_sm;
    if (ctas > a.total_chunks) ctas = a.total_chunks;
    return launch_after_previous(select_kernel<KIND, MBF16, D>, dim3(unsigned(ctas)), dim3(kSelThreads), smem, s, a,
                                 ready);
}

cudaError_t dispatch_select(const SelectArgs& a, int kind, bool mbf16, int D, int units,
                            cudaStream_t s, uint32_t* ready = nullptr)
{
    if (kind == KIND_MEAN) {
        return D == 128 ? launch_select_t<KIND_MEAN, false, 128>(a, units, ready, s)
                        : launch_select_t<KIND_MEAN, false, 64>(a, units, ready, s);
    }
    if (D == 128) {
        return mbf16 ? launch_select_t<KIND_QUEST, true, 128>(a, units, ready, s)
                     : launch_select_t<KIND_QUEST, false, 128>(a, units, ready, s);
    }
    return mbf16 ? launch_select_t<KIND_QUEST, true, 64>(a, units, ready, s)
                 : launch_select_t<KIND_QUEST, false, 64>(a, units, ready, s);
}

}  // namespace

cudaError_t launch_select(const Geometry& g, const WorkspaceLayout& L, char* ws, const void* q,
                          const void* kmin, const void* kmax, const float* kmean,
                          const int32_t* reserve_ids, int32_t* sel_ids, int32_t* sel_count,
                          cudaStream_t s, uint32_t* ready)
{
    const int units = g.units();
    if (units == 0) return cudaSuccess;
    SelectArgs a = select_args_base(g, L, ws, q, kmin, kmax, kmean);
    if (!g.two_level) {
        set_single_level(a, g, reserve_ids, sel_ids, sel_count);
        const int kind = g.score_kind == SPARSE_ATTN_SCORE_MEAN ? KIND_MEAN : KIND_QUEST;
        return dispatch_select(a, kind, g.kv_bf16, g.D, units, s, ready);
    }

    // ---- two level: level 1 over coarse blocks (mean score, no window) ----
    int32_t* surv = reinterpret_cast<int32_t*>(ws + L.survivors);
    int32_t* n_surv = reinterpret_cast<int32_t*>(ws + L.n_survivors);
    SelectArgs l1 = a;
    l1.rows = g.n_coarse;
    l1.row_stride = g.n_mean_cap;
    l1.via_survivors = 0;
    l1.row_limit = g.n_coarse;
    l1.n_cand = g.n_coarse;
    l1.groups = 1;
    l1.group_rows = g.n_coarse;
    l1.k = g.topk_coarse;
    l1.win_first = 0;
    l1.win_count = 0;
    l1.reserve = nullptr;
    l1.n_reserve = 0;
    l1.out_ids = surv;
    l1.out_stride = g.topk_coarse > 0 ? g.topk_coarse : 1;
    l1.out_count = n_surv;
    l1.counters = reinterpret_cast<uint32_t*>(ws + L.l1_counters);
    if (l1.n_cand == 0) { l1.n_cand = 1; l1.group_rows = 1; l1.row_limit = 0; }
    cudaError_t e = dispatch_select(l1, KIND_MEAN, false, g.D, units, s);
    if (e != cudaSuccess) return e;

    // ---- level 2: Quest bound over the survivors' slices, plus the window ----
    SelectArgs l2 = a;
    l2.rows = g.nb;
    l2.row_stride = g.nb_cap;
    l2.via_survivors = 1;
    l2.surv = surv;
    l2.n_surv = n_surv;
    l2.surv_stride = l1.out_stride;
    l2.per_coarse = g.per_coarse;
    l2.row_limit = g.win_first;
    l2.groups = g.topk_coarse;
    l2.group_rows = g.per_coarse;
    l2.n_cand = g.topk_coarse * g.per_coarse;
    l2.k = g.topk;
    l2.win_first = g.win_first;
    l2.win_count = g.win_count;
    l2.reserve = reserve_ids;
    l2.n_reserve = g.n_reserve;
    l2.out_ids = sel_ids;
    l2.out_stride = g.sel_stride;
    l2.out_count = sel_count;
    if (l2.n_cand == 0) {
        l2.groups = 1; l2.group_rows = 1; l2.n_cand = 1; l2.row_limit = 0; l2.via_survivors = 0;
    }
    return dispatch_select(l2, KIND_QUEST, g.kv_bf16, g.D, units, s);
}

}  // namespace sa
