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
// Work split: the candidates of a unit are cut into `splits` slices, one CTA each.  A
// half-warp (D = 128, bf16) covers one metadata row with 16-byte loads; four rows per
// half-warp are in flight.  Scores go to an L2-resident workspace row.  The CTA that
// completes a unit last (device-scope counter, no waiting) runs a radix select over
// the unit's order-preserving uint32 keys in shared memory: four 8-bit digit passes
// with warp-aggregated shared-memory histograms, early exit once a digit bin holds
// exactly the remaining count, then a stable tie rule (lower id first) and an ordered
// compaction by warp ballots.
#include "sa_common.cuh"
#include "sa_internal.h"

namespace sa {
namespace {

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kScoreUnroll = 4;
constexpr int kMaxSelectKeys = 16384;   // candidates per unit held in shared memory

enum { KIND_QUEST = 0, KIND_MEAN = 1 };

struct SelectArgs {
    const void* q;
    int q_bf16;
    const void* kmin;    // QUEST: [units, rows, D] metadata dtype
    const void* kmax;
    const float* kmean;  // MEAN:  [units, rows, D] fp32
    int rows;            // metadata rows per unit
    int Hkv, G;
    int Hq;
    // candidates: c in [0, n_cand); direct (c is the row) or via level-1 survivors
    int via_survivors;
    const int32_t* surv;     // [units, surv_stride], ascending coarse ids
    const int32_t* n_surv;   // [units]
    int surv_stride;
    int per_coarse;          // rows per coarse block
    int row_limit;           // rows >= row_limit are not candidates (window / past end)
    int n_cand;
    int cand_per_cta;
    int splits;
    // selection
    int k;
    int win_first, win_count;
    int32_t* out_ids;
    int out_stride;
    int32_t* out_count;
    // workspace
    float* scores;           // [units, n_cand]
    uint32_t* counters;      // [units]
    uint32_t* err;
};

// Row id of candidate c of unit u, or -1 when c is not a candidate.
__device__ __forceinline__ int candidate_row(const SelectArgs& a, int u, int c)
{
    if (c >= a.n_cand) return -1;
    if (!a.via_survivors) return c;
    const int i = c / a.per_coarse;
    if (i >= a.n_surv[u]) return -1;
    const int row = a.surv[size_t(u) * a.surv_stride + i] * a.per_coarse + (c - i * a.per_coarse);
    return row < a.row_limit ? row : -1;
}

// ------------------------------------------------------------- top-k ----
// Runs in one CTA.  keys[0..n) hold order keys (0 = not a candidate).
__device__ void topk_and_emit(const SelectArgs& a, int u, uint32_t* keys, int n, int n_valid)
{
    __shared__ uint32_t hist[256];
    __shared__ uint32_t s_bin, s_above, s_binc;
    __shared__ int s_wtot[kSelWarps];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int k_eff = min(a.k, n_valid);
    int32_t* out = a.out_ids + size_t(u) * a.out_stride;

    uint32_t prefix = 0, mask = 0;
    int krem = k_eff;
    bool all_of_prefix = false;
    for (int pass = 0; pass < 4 && k_eff > 0; ++pass) {
        const int shift = 24 - 8 * pass;
        if (tid < 256) hist[tid] = 0;
        __syncthreads();
        for (int base = 0; base < n; base += kSelThreads) {
            const int c = base + tid;
            const uint32_t key = c < n ? keys[c] : 0u;
            const bool match = c < n && key != 0u && (key & mask) == prefix;
            const uint32_t bin = match ? ((key >> shift) & 255u) : 256u;
            const uint32_t peers = __match_any_sync(kFullMask, bin);
            if (match && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
        }
        __syncthreads();
        if (warp == 0) {
            uint32_t cnt[8], sum = 0;
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                cnt[r] = hist[255 - 8 * lane - r];
                sum += cnt[r];
            }
            uint32_t inc = sum;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                uint32_t t = __shfl_up_sync(kFullMask, inc, off);
                if (lane >= off) inc += t;
            }
            const uint32_t hit = __ballot_sync(kFullMask, inc >= uint32_t(krem));
            if (lane == __ffs(hit) - 1) {
                uint32_t above = inc - sum;
                for (int r = 0; r < 8; ++r) {
                    if (above + cnt[r] >= uint32_t(krem)) {
                        s_bin = 255 - 8 * lane - r;
                        s_above = above;
                        s_binc = cnt[r];
                        break;
                    }
                    above += cnt[r];
                }
            }
        }
        __syncthreads();
        krem -= int(s_above);
        prefix |= s_bin << shift;
        mask |= 255u << shift;
        if (int(s_binc) == krem) {
            all_of_prefix = true;   // every key with this prefix is selected
            break;
        }
    }
    // Threshold rule:  all_of_prefix: (key & mask) >= prefix
    //                  otherwise:      key > T, or key == T among the first krem (by id)
    const uint32_t T = prefix;
    const bool need_ties = k_eff > 0 && !all_of_prefix;

    // Each warp owns a contiguous chunk of candidates, read lane-interleaved, so ballot
    // order is candidate order.
    const int chunk = ((n + kSelWarps * 32 - 1) / (kSelWarps * 32)) * 32;
    const int c0 = warp * chunk, c1 = min(n, c0 + chunk);

    int eq_base = 0;
    if (need_ties) {
        int eq = 0;
        for (int c = c0 + lane; c - lane < c1; c += 32) {
            const bool e = c < c1 && keys[c] == T;
            eq += __popc(__ballot_sync(kFullMask, e));
        }
        if (lane == 0) s_wtot[warp] = eq;
        __syncthreads();
        for (int w = 0; w < warp; ++w) eq_base += s_wtot[w];
        __syncthreads();
    }
    auto selected = [&](int c, int eq_rank) -> bool {
        const uint32_t key = keys[c];
        if (k_eff == 0 || key == 0u) return false;
        if (all_of_prefix) return (key & mask) >= prefix;
        return key > T || (key == T && eq_rank < krem);
    };
    // count per warp
    int cnt = 0;
    {
        int eq_run = eq_base;
        for (int c = c0 + lane; c - lane < c1; c += 32) {
            const bool in = c < c1;
            const bool e = in && need_ties && keys[c] == T;
            const uint32_t eb = __ballot_sync(kFullMask, e);
            const int rank = eq_run + __popc(eb & lanemask_lt());
            const bool s = in && selected(c, rank);
            cnt += __popc(__ballot_sync(kFullMask, s));
            eq_run += __popc(eb);
        }
    }
    if (lane == 0) s_wtot[warp] = cnt;
    __syncthreads();
    int pos = 0;
    for (int w = 0; w < warp; ++w) pos += s_wtot[w];
    {
        int eq_run = eq_base;
        for (int c = c0 + lane; c - lane < c1; c += 32) {
            const bool in = c < c1;
            const bool e = in && need_ties && keys[c] == T;
            const uint32_t eb = __ballot_sync(kFullMask, e);
            const int rank = eq_run + __popc(eb & lanemask_lt());
            const bool s = in && selected(c, rank);
            const uint32_t sb = __ballot_sync(kFullMask, s);
            if (s) out[pos + __popc(sb & lanemask_lt())] = candidate_row(a, u, c);
            pos += __popc(sb);
            eq_run += __popc(eb);
        }
    }
    for (int i = tid; i < a.win_count; i += kSelThreads) out[k_eff + i] = a.win_first + i;
    if (tid == 0) a.out_count[u] = k_eff + a.win_count;
}

// ------------------------------------------------------------- kernel ---
template <int KIND, bool MBF16, int D>
__global__ void __launch_bounds__(kSelThreads) select_kernel(SelectArgs a)
{
    extern __shared__ uint32_t keys[];
    __shared__ bool s_last;

    constexpr int ESZ = (KIND == KIND_QUEST && MBF16) ? 2 : 4;
    constexpr int EPL = 16 / ESZ;
    constexpr int LPR = D / EPL;
    constexpr int RPW = 32 / LPR;
    constexpr int ROWS_PER_PASS = kSelWarps * RPW;

    const int u = blockIdx.x / a.splits;
    const int split = blockIdx.x - u * a.splits;
    const int b = u / a.Hkv, kvh = u - b * a.Hkv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sub = lane % LPR, rsub = lane / LPR;
    const int d0 = sub * EPL;

    // query coefficients for this lane's channels
    float cp[EPL], cn[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) { cp[e] = 0.f; cn[e] = 0.f; }
    for (int g = 0; g < a.G; ++g) {
        const size_t qrow = (size_t(b) * a.Hq + size_t(kvh) * a.G + g) * D + d0;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            const float x = load_q(a.q, qrow + e, a.q_bf16 != 0);
            if constexpr (KIND == KIND_QUEST) {
                cp[e] += fmaxf(x, 0.f);
                cn[e] += fminf(x, 0.f);
            } else {
                cp[e] += x;
            }
        }
    }

    // score this CTA's candidates
    const int cbeg = split * a.cand_per_cta;
    const int cend = min(a.n_cand, cbeg + a.cand_per_cta);
    float* srow = a.scores + size_t(u) * a.n_cand;
    const char* hi_base;
    const char* lo_base;
    if constexpr (KIND == KIND_QUEST) {
        hi_base = reinterpret_cast<const char*>(a.kmax) + size_t(u) * a.rows * D * ESZ + d0 * ESZ;
        lo_base = reinterpret_cast<const char*>(a.kmin) + size_t(u) * a.rows * D * ESZ + d0 * ESZ;
    } else {
        hi_base = reinterpret_cast<const char*>(a.kmean) + size_t(u) * a.rows * D * 4 + d0 * 4;
        lo_base = hi_base;
    }
    for (int base = cbeg + warp * RPW; base < cend; base += ROWS_PER_PASS * kScoreUnroll) {
        uint4 vh[kScoreUnroll], vl[kScoreUnroll];
        int row[kScoreUnroll];
#pragma unroll
        for (int i = 0; i < kScoreUnroll; ++i) {
            const int c = base + i * ROWS_PER_PASS + rsub;
            row[i] = c < cend ? candidate_row(a, u, c) : -1;
            if (row[i] >= 0) {
                vh[i] = ld_stream16(hi_base + size_t(row[i]) * D * ESZ);
                if constexpr (KIND == KIND_QUEST) vl[i] = ld_stream16(lo_base + size_t(row[i]) * D * ESZ);
            } else {
                vh[i] = make_uint4(0, 0, 0, 0);
                vl[i] = make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int i = 0; i < kScoreUnroll; ++i) {
            float fh[EPL], s = 0.f;
            unpack16<ESZ == 2>(vh[i], fh);
            if constexpr (KIND == KIND_QUEST) {
                float fl[EPL];
                unpack16<ESZ == 2>(vl[i], fl);
#pragma unroll
                for (int e = 0; e < EPL; ++e) s = fmaf(cp[e], fh[e], fmaf(cn[e], fl[e], s));
            } else {
#pragma unroll
                for (int e = 0; e < EPL; ++e) s = fmaf(cp[e], fh[e], s);
            }
#pragma unroll
            for (int m = LPR / 2; m >= 1; m >>= 1) s += __shfl_xor_sync(kFullMask, s, m);
            const int c = base + i * ROWS_PER_PASS + rsub;
            if (sub == 0 && c < cend) srow[c] = row[i] >= 0 ? s : -INFINITY;
        }
    }

    // the last CTA of this unit selects
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const uint32_t done = atomicAdd(&a.counters[u], 1u);
        s_last = (done == uint32_t(a.splits - 1));
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (tid == 0) a.counters[u] = 0u;   // every split of this launch has arrived

    int n_valid = 0;
    for (int base = 0; base < a.n_cand; base += kSelThreads) {
        const int c = base + tid;
        bool valid = false;
        if (c < a.n_cand) {
            valid = candidate_row(a, u, c) >= 0;
            keys[c] = valid ? order_key(__ldcg(srow + c)) : 0u;
        }
        n_valid += __syncthreads_count(valid);
    }
    topk_and_emit(a, u, keys, a.n_cand, n_valid);
}

template <int KIND, bool MBF16, int D>
cudaError_t launch_select_t(const SelectArgs& a, int units, cudaStream_t s)
{
    const size_t smem = size_t(a.n_cand) * sizeof(uint32_t);
    static bool configured = false;   // once per instantiation, before any graph capture
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(select_kernel<KIND, MBF16, D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(kMaxSelectKeys * sizeof(uint32_t)));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    select_kernel<KIND, MBF16, D><<<dim3(unsigned(units * a.splits)), kSelThreads, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t dispatch_select(const SelectArgs& a, int kind, bool mbf16, int D, int units,
                            cudaStream_t s)
{
    if (kind == KIND_MEAN) {
        return D == 128 ? launch_select_t<KIND_MEAN, false, 128>(a, units, s)
                        : launch_select_t<KIND_MEAN, false, 64>(a, units, s);
    }
    if (D == 128) {
        return mbf16 ? launch_select_t<KIND_QUEST, true, 128>(a, units, s)
                     : launch_select_t<KIND_QUEST, false, 128>(a, units, s);
    }
    return mbf16 ? launch_select_t<KIND_QUEST, true, 64>(a, units, s)
                 : launch_select_t<KIND_QUEST, false, 64>(a, units, s);
}

// Candidates per CTA: enough CTAs to cover the GPU several times over, each streaming
// between 16 KB and 256 KB of metadata.
int pick_cand_per_cta(long long units, int n_cand, int row_bytes)
{
    const long long total = units * (long long)n_cand * row_bytes;
    long long target = total / (4 * 152);
    if (target < 16 * 1024) target = 16 * 1024;
    if (target > 256 * 1024) target = 256 * 1024;
    long long per = target / row_bytes;
    if (per < 32) per = 32;
    if (per > n_cand) per = n_cand;
    return int(per > 0 ? per : 1);
}

}  // namespace

cudaError_t launch_select(const Geometry& g, const WorkspaceLayout& L, char* ws, const void* q,
                          const void* kmin, const void* kmax, const float* kmean,
                          int32_t* sel_ids, int32_t* sel_count, cudaStream_t s)
{
    const int units = g.units();
    if (units == 0) return cudaSuccess;
    uint32_t* err = reinterpret_cast<uint32_t*>(ws + L.err);
    const int meta_esz = g.kv_bf16 ? 2 : 4;

    SelectArgs a{};
    a.q = q;
    a.q_bf16 = g.q_bf16;
    a.kmin = kmin;
    a.kmax = kmax;
    a.kmean = kmean;
    a.Hkv = g.Hkv;
    a.G = g.G;
    a.Hq = g.Hq;
    a.err = err;
    a.scores = reinterpret_cast<float*>(ws + L.scores);

    if (!g.two_level) {
        a.rows = g.nb;
        a.via_survivors = 0;
        a.row_limit = g.win_first;
        a.n_cand = g.n_cand;
        a.k = g.topk;
        a.win_first = g.win_first;
        a.win_count = g.win_count;
        a.out_ids = sel_ids;
        a.out_stride = g.sel_stride;
        a.out_count = sel_count;
        a.counters = reinterpret_cast<uint32_t*>(ws + L.sel_counters);
        if (g.score_kind == SPARSE_ATTN_SCORE_MEAN) {
            a.kmean = kmean;
            a.cand_per_cta = pick_cand_per_cta(units, a.n_cand, g.D * 4);
        } else {
            a.cand_per_cta = pick_cand_per_cta(units, a.n_cand, 2 * g.D * meta_esz);
        }
        if (a.n_cand == 0) {
            // no candidates: a single pass that only emits the window
            a.cand_per_cta = 1;
            a.splits = 1;
        } else {
            a.splits = (a.n_cand + a.cand_per_cta - 1) / a.cand_per_cta;
        }
        const int kind = g.score_kind == SPARSE_ATTN_SCORE_MEAN ? KIND_MEAN : KIND_QUEST;
        return dispatch_select(a, kind, g.kv_bf16, g.D, units, s);
    }

    // ---- two level: level 1 over coarse blocks (mean score, no window) ----
    int32_t* surv = reinterpret_cast<int32_t*>(ws + L.survivors);
    int32_t* n_surv = reinterpret_cast<int32_t*>(ws + L.n_survivors);
    SelectArgs l1 = a;
    l1.rows = g.n_coarse;
    l1.via_survivors = 0;
    l1.row_limit = g.n_coarse;
    l1.n_cand = g.n_coarse;
    l1.k = g.topk_coarse;
    l1.win_first = 0;
    l1.win_count = 0;
    l1.out_ids = surv;
    l1.out_stride = g.topk_coarse > 0 ? g.topk_coarse : 1;
    l1.out_count = n_surv;
    l1.counters = reinterpret_cast<uint32_t*>(ws + L.l1_counters);
    l1.cand_per_cta = pick_cand_per_cta(units, l1.n_cand, g.D * 4);
    if (l1.n_cand == 0) { l1.cand_per_cta = 1; l1.splits = 1; }
    else l1.splits = (l1.n_cand + l1.cand_per_cta - 1) / l1.cand_per_cta;
    cudaError_t e = dispatch_select(l1, KIND_MEAN, false, g.D, units, s);
    if (e != cudaSuccess) return e;

    // ---- level 2: Quest bound over the survivors' slices, plus the window ----
    SelectArgs l2 = a;
    l2.rows = g.nb;
    l2.via_survivors = 1;
    l2.surv = surv;
    l2.n_surv = n_surv;
    l2.surv_stride = l1.out_stride;
    l2.per_coarse = g.per_coarse;
    l2.row_limit = g.win_first;
    l2.n_cand = g.topk_coarse * g.per_coarse;
    l2.k = g.topk;
    l2.win_first = g.win_first;
    l2.win_count = g.win_count;
    l2.out_ids = sel_ids;
    l2.out_stride = g.sel_stride;
    l2.out_count = sel_count;
    l2.counters = reinterpret_cast<uint32_t*>(ws + L.sel_counters);
    l2.cand_per_cta = pick_cand_per_cta(units, l2.n_cand, 2 * g.D * meta_esz);
    if (l2.n_cand == 0) { l2.cand_per_cta = 1; l2.splits = 1; }
    else l2.splits = (l2.n_cand + l2.cand_per_cta - 1) / l2.cand_per_cta;
    return dispatch_select(l2, KIND_QUEST, g.kv_bf16, g.D, units, s);
}

}  // namespace sa
