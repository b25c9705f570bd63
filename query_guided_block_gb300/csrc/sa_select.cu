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
#include <type_traits>

#include "sa_select_body.cuh"

namespace sa {
namespace {

template <int KIND, bool MBF16, int D>
__global__ void __launch_bounds__(kSelThreads) select_kernel(SelectArgs a, uint32_t* ready)
{
    select_body<KIND, MBF16, D>(a, ready);
}

// The warp-slab streaming of the fused step as a select kernel of its own (one CTA per
// SM, the CTA's query coefficients summed before any copy is in flight).
template <int KIND, bool MBF16, int D>
__global__ void __launch_bounds__(kSelThreads, 1) select_warps_kernel(SelectArgs a, uint32_t* ready)
{
    select_body_warps<KIND, MBF16, D>(a, ready);
}

template <int KIND, bool MBF16, int D>
cudaError_t launch_select_warps_t(const SelectArgs& a0, int units, uint32_t* ready, cudaStream_t s)
{
    using WS = SlabSelShape<KIND, MBF16, D>;
    SelectArgs a = a0;
    set_slab_chunking<KIND, MBF16, D>(a, units);
    const size_t keys = size_t(kSelThreads) * key_tile(a.n_cand) * sizeof(uint32_t);
    const size_t smem = WS::RING_BYTES > keys ? WS::RING_BYTES : keys;
    static std::atomic<unsigned long long> configured{0};   // devices set up
    const cudaError_t cfg = once_per_device(configured, [&]() -> cudaError_t {
        return cudaFuncSetAttribute(select_warps_kernel<KIND, MBF16, D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(WS::RING_BYTES));
    });
    if (cfg != cudaSuccess) return cfg;
    int ctas = num_sms();
    if (ctas > a.total_chunks) ctas = a.total_chunks;
    // a CTA records the units it completes in a fixed list
    const long long per_cta = ((long long)a.total_chunks + ctas - 1) / ctas;
    if (per_cta / a.chunks_per_unit + 2 > kSlabSelMaxUnits) return cudaErrorNotSupported;
    return launch_after_previous(select_warps_kernel<KIND, MBF16, D>, dim3(unsigned(ctas)), dim3(kSelThreads), smem, s,
                                 a, ready);
}

// Several queries per sequence (many query rows per unit, one coefficient sum per unit
// change) with no more units than SMs: the warp-slab kernel, whose CTAs sum their
// units' coefficients before streaming (mq_128k select 86.5 -> 76.6 us); otherwise the
// two-CTA-per-SM streaming kernel, which ranks the units two CTAs at a time.
template <int KIND, bool MBF16, int D>
cudaError_t launch_select_t(const SelectArgs& a0, int units, uint32_t* ready, cudaStream_t s)
{
    if (a0.Q > 1 && units <= num_sms()) {
        const cudaError_t e = launch_select_warps_t<KIND, MBF16, D>(a0, units, ready, s);
        if (e != cudaErrorNotSupported) return e;
    }
    SelectArgs a = a0;
    set_chunking<KIND, MBF16, D>(a, units);
    const size_t keys_bytes = size_t(kSelThreads) * key_tile(a.n_cand) * sizeof(uint32_t);
    // two CTAs per SM when they fit: dynamic stages + keys, plus static (histogram) and
    // the per-CTA reservation
    constexpr size_t kStatic = 13 * 1024;
    a.stages = (2 * (3 * size_t(kStageBytes) + keys_bytes + kStatic) <= size_t(kSmemPerSm)) ? 3 : 2;
    const size_t smem = size_t(a.stages) * kStageBytes + keys_bytes;
    static std::atomic<unsigned long long> configured{0};   // devices set up
    const cudaError_t cfg = once_per_device(configured, [&]() -> cudaError_t {
        return cudaFuncSetAttribute(select_kernel<KIND, MBF16, D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(2 * kStageBytes + kMaxSelectKeys * sizeof(uint32_t)));
    });
    if (cfg != cudaSuccess) return cfg;
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

// ------------------------------------------------------ two-level, per unit ---
// Both levels of one (sequence, KV head) unit in one CTA (HiSparse->QSA page §2.2 and
// §3.1: coarse-block mean scores, top K1 coarse blocks, Quest bound over their slices,
// top K2 slices plus the window).  A unit's two levels are a short dependent chain over
// little data (the 256K workload reads 128 KB of means and 384 KB of slice bounds per
// unit), so one CTA per unit runs the chain without any cross-CTA hand-off: the
// scores go straight into shared-memory keys (no score row in global memory), and the
// rows are read with 16-byte loads, kRowsInFlight rows per lane group in flight.  The
// per-row arithmetic (each lane's fma chain over its channels, then the same xor
// butterfly over the row's lanes) and the query-coefficient sums are those of the
// streaming select kernel, so the scores are the same bits.
constexpr int kRowsInFlight = 8;

// Score `nrows` candidate rows into keys[0, nrows): row_of(c) gives the metadata row of
// candidate c or -1.  Returns (via shared memory, after a barrier) the valid count and
// the key range.
template <int KIND, bool MBF16, int D, typename RowOf>
__device__ __forceinline__ int score_rows_to_keys(const SelectArgs& a, int u, uint32_t* keys, int nrows,
                                                  const float (&cp)[SelectShape<KIND, MBF16, D>::EPL],
                                                  const float (&cn)[SelectShape<KIND, MBF16, D>::EPL],
                                                  RowOf row_of, uint32_t& key_lo, uint32_t& key_hi)
{
    using SS = SelectShape<KIND, MBF16, D>;
    constexpr int EPL = SS::EPL, LPR = SS::LPR, RPW = SS::RPW, R = kRowsInFlight;
    constexpr int ROWS_PER_WARP = RPW * R;
    __shared__ int s_count;
    __shared__ uint32_t s_lo, s_hi;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sub = lane % LPR, rsub = lane / LPR;
    if (tid == 0) {
        s_count = 0;
        s_lo = 0xffffffffu;
        s_hi = 0u;
    }
    __syncthreads();
    const char* hi_src = reinterpret_cast<const char*>(KIND == KIND_QUEST ? a.kmax : (const void*)a.kmean);
    const char* lo_src = reinterpret_cast<const char*>(a.kmin);
    const size_t unit_off = size_t(u) * a.row_stride;
    int mine = 0;
    uint32_t lo = 0xffffffffu, hi = 0u;
    for (int base = warp * ROWS_PER_WARP; base < nrows; base += kSelWarps * ROWS_PER_WARP) {
        int row[R];
        uint4 vh[R], vl[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int c = base + rsub * R + r;
            row[r] = c < nrows ? row_of(c) : -1;
            if (row[r] >= 0) {
                const size_t off = (unit_off + row[r]) * SS::ROW_BYTES + sub * 16;
                vh[r] = ld_stream16(hi_src + off);
                if constexpr (KIND == KIND_QUEST) vl[r] = ld_stream16(lo_src + off);
            }
        }
        float part[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float acc = 0.f;
            if (row[r] >= 0) {
                float fh[EPL];
                unpack16<SS::ESZ == 2>(vh[r], fh);
                if constexpr (KIND == KIND_QUEST) {
                    float fl[EPL];
                    unpack16<SS::ESZ == 2>(vl[r], fl);
#pragma unroll
                    for (int e = 0; e < EPL; ++e) acc = fmaf(cp[e], fh[e], fmaf(cn[e], fl[e], acc));
                } else {
#pragma unroll
                    for (int e = 0; e < EPL; ++e) acc = fmaf(cp[e], fh[e], acc);
                }
            }
            part[r] = acc;
        }
        group_reduce_transposed<R, LPR>(part, lane);
        constexpr int OUT = R >= LPR ? R / LPR : 1;
        constexpr int SPREAD = R >= LPR ? 1 : LPR / R;
        if (sub % SPREAD == 0) {
#pragma unroll
            for (int i = 0; i < OUT; ++i) {
                const int r = R >= LPR ? sub * (R / LPR) + i : sub / SPREAD;
                const int c = base + rsub * R + r;
                if (c < nrows) {
                    const bool ok = row_of(c) >= 0;
                    const uint32_t key = order_key(part[i]);
                    keys[c] = ok ? key : 0u;
                    if (ok) {
                        lo = min(lo, key);
                        hi = max(hi, key);
                        ++mine;
                    }
                }
            }
        }
    }
    for (int c = nrows + tid; c < kSelThreads * key_tile(nrows); c += kSelThreads) keys[c] = 0u;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        mine += __shfl_xor_sync(kFullMask, mine, off);
        lo = min(lo, __shfl_xor_sync(kFullMask, lo, off));
        hi = max(hi, __shfl_xor_sync(kFullMask, hi, off));
    }
    if (lane == 0) {
        atomicAdd(&s_count, mine);
        atomicMin(&s_lo, lo);
        atomicMax(&s_hi, hi);
    }
    __syncthreads();
    key_lo = s_lo;
    key_hi = s_hi;
    return s_count;
}

// Query coefficients of unit u in the streaming kernel's order: thread t sums channel
// t mod D over rows t / D, t / D + 256 / D, ... (quest: max(q, 0) and min(q, 0); mean: q),
// the partials go through shared memory and each lane adds its channels' partials.
template <int KIND, int EPL, int D>
__device__ __forceinline__ void unit_coefficients(const SelectArgs& a, int u, int d0, float (&cp)[EPL],
                                                  float (&cn)[EPL])
{
    constexpr int RSTEP = kSelThreads / D;
    __shared__ float s_part[2][kSelThreads];
    const int tid = threadIdx.x;
    const int b = u / a.Hkv, kvh = u - (u / a.Hkv) * a.Hkv;
    const int dch = tid % D;
    const int rows = a.Q * a.G;
    float pp = 0.f, nn = 0.f;
    for (int r = tid / D; r < rows; r += RSTEP) {
        const int t = r / a.G, g = r - t * a.G;
        const float x = load_q(a.q, ((size_t(b) * a.Q + t) * a.Hq + size_t(kvh) * a.G + g) * D + dch, a.q_bf16 != 0);
        if constexpr (KIND == KIND_QUEST) {
            pp += fmaxf(x, 0.f);
            nn += fminf(x, 0.f);
        } else {
            pp += x;
        }
    }
    __syncthreads();   // a previous call's partials have been read
    s_part[0][tid] = pp;
    s_part[1][tid] = nn;
    __syncthreads();
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        float sp = 0.f, sn = 0.f;
#pragma unroll
        for (int k2 = 0; k2 < RSTEP; ++k2) {
            sp += s_part[0][d0 + e + k2 * D];
            sn += s_part[1][d0 + e + k2 * D];
        }
        cp[e] = sp;
        cn[e] = sn;
    }
}

template <bool MBF16, int D>
__global__ void __launch_bounds__(kSelThreads) select_two_level_kernel(SelectArgs l1, SelectArgs l2)
{
    using S1 = SelectShape<KIND_MEAN, false, D>;
    using S2 = SelectShape<KIND_QUEST, MBF16, D>;
    extern __shared__ __align__(16) uint32_t keys[];
    __shared__ int s_surv[kSelThreads];
    __shared__ int s_nsurv;
    const int u = blockIdx.x;
    const int lane = threadIdx.x & 31;
    grid_dependency_wait();   // inputs and workspace may come from the previous kernel
    allow_dependents_early();

    // ---- level 1: mean score of every coarse block, top K1 ----
    {
        float cp[S1::EPL], cn[S1::EPL];
        unit_coefficients<KIND_MEAN, S1::EPL, D>(l1, u, (lane % S1::LPR) * S1::EPL, cp, cn);
        uint32_t klo, khi;
        const int n_valid = score_rows_to_keys<KIND_MEAN, false, D>(
            l1, u, keys, l1.n_cand, cp, cn, [&](int c) { return c < l1.row_limit ? c : -1; }, klo, khi);
        topk_and_emit(l1, u, keys, l1.n_cand, n_valid, klo, khi);
    }
    __syncthreads();   // survivors written (global, this CTA)
    if (threadIdx.x == 0) s_nsurv = min(l1.out_count[u], l2.groups);
    for (int i = threadIdx.x; i < l2.groups; i += kSelThreads)
        s_surv[i] = l1.out_ids[size_t(u) * l1.out_stride + i];
    __syncthreads();

    // ---- level 2: Quest bound over the survivors' slices, top K2 plus the window ----
    {
        float cp[S2::EPL], cn[S2::EPL];
        unit_coefficients<KIND_QUEST, S2::EPL, D>(l2, u, (lane % S2::LPR) * S2::EPL, cp, cn);
        const int nsurv = s_nsurv, per = l2.per_coarse, limit = l2.row_limit;
        auto row_of = [&](int c) -> int {
            const int i = c / per;
            if (i >= nsurv) return -1;
            const int row = s_surv[i] * per + (c - i * per);
            return row < limit ? row : -1;
        };
        uint32_t klo, khi;
        const int n_valid = score_rows_to_keys<KIND_QUEST, MBF16, D>(l2, u, keys, l2.n_cand, cp, cn, row_of, klo, khi);
        topk_and_emit(l2, u, keys, l2.n_cand, n_valid, klo, khi, l2.via_survivors ? s_surv : nullptr, nsurv);
    }
}

// ------------------------------------------- two-level, a cluster per unit ---
// The same two levels with P CTAs per unit, one thread-block cluster each, when the
// units alone would leave most SMs idle (the 256K workload has 64 units on 152 SMs).
// Each CTA scores its 1/P of the unit's coarse rows, then of the survivors' slices,
// into a scratch area of its own shared memory and stores the keys into CTA 0's key
// array (distributed shared memory), with its (valid count, key range) in CTA 0's
// per-rank slots.  After a cluster barrier CTA 0 runs the top-k on the whole key array:
// level 1's survivors go to global memory, a second barrier makes them visible to the
// cluster, and level 2's selection is emitted by CTA 0 alone.  Candidate numbering,
// scores and the top-k are those of the one-CTA kernel, so the selection is the same.
constexpr int kMaxClusterRanks = 8;
// keys (up to kMaxSelectKeys) and a share's scratch keys (P >= 2: at most half of them)
constexpr size_t kTwoLevelSmemMax = (kMaxSelectKeys + kMaxSelectKeys / 2) * sizeof(uint32_t);

template <bool MBF16, int D>
__global__ void __launch_bounds__(kSelThreads) select_two_level_cluster_kernel(SelectArgs l1, SelectArgs l2, int P,
                                                                             int scratch_off)
{
    using S1 = SelectShape<KIND_MEAN, false, D>;
    using S2 = SelectShape<KIND_QUEST, MBF16, D>;
    extern __shared__ __align__(16) uint32_t keys[];
    uint32_t* scratch = keys + scratch_off;           // this CTA's share, before it moves to CTA 0
    __shared__ uint32_t s_stat[kMaxClusterRanks][3];  // CTA 0: per rank (valid count, key lo, key hi)
    __shared__ int s_surv[kSelThreads];
    __shared__ int s_nsurv;
    const uint32_t rank = cluster_ctarank();
    const int u = int(blockIdx.x) / P;
    const int tid = threadIdx.x, lane = tid & 31;
    const uint32_t keys0 = cluster_map(smem_u32(keys), 0);
    const uint32_t stat0 = cluster_map(smem_u32(&s_stat[0][0]), 0);
    grid_dependency_wait();   // inputs and workspace may come from the previous kernel
    allow_dependents_early();

    // this CTA's share [c0, c1) of n candidates: score into scratch, move to CTA 0
    auto score_share = [&](const SelectArgs& a, auto kind_tag, const auto& cp, const auto& cn, int n, auto row_of) {
        constexpr int KIND = decltype(kind_tag)::value;
        const int c0 = int((long long)n * rank / P), c1 = int((long long)n * (rank + 1) / P);
        constexpr bool MB = KIND == KIND_QUEST ? MBF16 : false;
        uint32_t lo = 0xffffffffu, hi = 0u;
        const int nv = score_rows_to_keys<KIND, MB, D>(a, u, scratch, c1 - c0, cp, cn,
                                                       [&](int i) { return row_of(c0 + i); }, lo, hi);
        for (int i = tid; i < c1 - c0; i += kSelThreads) st_cluster_u32(keys0 + uint32_t(c0 + i) * 4u, scratch[i]);
        if (tid == 0) {
            st_cluster_u32(stat0 + rank * 12u, uint32_t(nv));
            st_cluster_u32(stat0 + rank * 12u + 4u, lo);
            st_cluster_u32(stat0 + rank * 12u + 8u, hi);
        }
        cluster_sync_all();   // CTA 0 holds every key of the level
    };
    // CTA 0: zero the padding past n, combine the ranks' statistics
    auto gather = [&](int n, int& n_valid, uint32_t& lo, uint32_t& hi) {
        for (int c = n + tid; c < kSelThreads * key_tile(n); c += kSelThreads) keys[c] = 0u;
        n_valid = 0;
        lo = 0xffffffffu;
        hi = 0u;
        for (int r = 0; r < P; ++r) {
            n_valid += int(s_stat[r][0]);
            if (s_stat[r][0] > 0u) {
                lo = min(lo, s_stat[r][1]);
                hi = max(hi, s_stat[r][2]);
            }
        }
        __syncthreads();
    };

    // ---- level 1: mean score of every coarse block, top K1 ----
    {
        float cp[S1::EPL], cn[S1::EPL];
        unit_coefficients<KIND_MEAN, S1::EPL, D>(l1, u, (lane % S1::LPR) * S1::EPL, cp, cn);
        score_share(l1, std::integral_constant<int, KIND_MEAN>(), cp, cn, l1.n_cand,
                    [&](int c) { return c < l1.row_limit ? c : -1; });
        if (rank == 0) {
            int n_valid;
            uint32_t lo, hi;
            gather(l1.n_cand, n_valid, lo, hi);
            topk_and_emit(l1, u, keys, l1.n_cand, n_valid, lo, hi);
        }
        cluster_sync_all();   // survivors (global, written by CTA 0) visible to the cluster
    }
    if (tid == 0) s_nsurv = min(__ldcg(l1.out_count + u), l2.groups);
    for (int i = tid; i < l2.groups; i += kSelThreads) s_surv[i] = __ldcg(l1.out_ids + size_t(u) * l1.out_stride + i);
    __syncthreads();

    // ---- level 2: Quest bound over the survivors' slices, top K2 plus the window ----
    {
        float cp[S2::EPL], cn[S2::EPL];
        unit_coefficients<KIND_QUEST, S2::EPL, D>(l2, u, (lane % S2::LPR) * S2::EPL, cp, cn);
        const int nsurv = s_nsurv, per = l2.per_coarse, limit = l2.row_limit;
        score_share(l2, std::integral_constant<int, KIND_QUEST>(), cp, cn, l2.n_cand, [&](int c) -> int {
            const int i = c / per;
            if (i >= nsurv) return -1;
            const int row = s_surv[i] * per + (c - i * per);
            return row < limit ? row : -1;
        });
        if (rank == 0) {
            int n_valid;
            uint32_t lo, hi;
            gather(l2.n_cand, n_valid, lo, hi);
            topk_and_emit(l2, u, keys, l2.n_cand, n_valid, lo, hi, l2.via_survivors ? s_surv : nullptr, nsurv);
        }
    }
}

// CTAs per unit for the cluster kernel: a power of two up to 4 that keeps about two
// CTAs per SM; 1 selects the one-CTA kernel.
inline int two_level_ranks(int units)
{
    const int sms = num_sms();
    int P = 1;
    while (P < 4 && (long long)units * P * 2 <= 2LL * sms) P *= 2;
    return P;
}

template <bool MBF16, int D>
cudaError_t launch_two_level_cluster_t(const SelectArgs& l1, const SelectArgs& l2, int units, int P, cudaStream_t s)
{
    const int n = l1.n_cand > l2.n_cand ? l1.n_cand : l2.n_cand;
    const int keys_n = kSelThreads * key_tile(n);
    const int share = (n + P - 1) / P;
    const int scratch_n = kSelThreads * key_tile(share);
    const size_t smem = size_t(keys_n + scratch_n) * sizeof(uint32_t);
    if (smem > kTwoLevelSmemMax) return cudaErrorInvalidValue;
    static std::atomic<unsigned long long> configured{0};   // devices set up
    const cudaError_t cfg = once_per_device(configured, [&]() -> cudaError_t {
        return cudaFuncSetAttribute(select_two_level_cluster_kernel<MBF16, D>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    int(kTwoLevelSmemMax));
    });
    if (cfg != cudaSuccess) return cfg;
    return launch_clusters_after_previous(select_two_level_cluster_kernel<MBF16, D>, dim3(unsigned(units * P)),
                                          dim3(kSelThreads), smem, unsigned(P), s, l1, l2, P, keys_n);
}

template <bool MBF16, int D>
cudaError_t launch_two_level_t(const SelectArgs& l1, const SelectArgs& l2, int units, cudaStream_t s)
{
    const int P = two_level_ranks(units);
    if (P > 1) return launch_two_level_cluster_t<MBF16, D>(l1, l2, units, P, s);
    const int n = l1.n_cand > l2.n_cand ? l1.n_cand : l2.n_cand;
    const size_t smem = size_t(kSelThreads) * key_tile(n) * sizeof(uint32_t);
    static std::atomic<unsigned long long> configured{0};   // devices set up
    const cudaError_t cfg = once_per_device(configured, [&]() -> cudaError_t {
        return cudaFuncSetAttribute(select_two_level_kernel<MBF16, D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(kMaxSelectKeys * sizeof(uint32_t)));
    });
    if (cfg != cudaSuccess) return cfg;
    return launch_after_previous(select_two_level_kernel<MBF16, D>, dim3(unsigned(units)), dim3(kSelThreads), smem,
                                 s, l1, l2);
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
    if (l2.groups <= kSelThreads) {   // both levels of a unit in one CTA
        if (g.D == 128)
            return g.kv_bf16 ? launch_two_level_t<true, 128>(l1, l2, units, s)
                             : launch_two_level_t<false, 128>(l1, l2, units, s);
        return g.kv_bf16 ? launch_two_level_t<true, 64>(l1, l2, units, s)
                         : launch_two_level_t<false, 64>(l1, l2, units, s);
    }
    // more survivors than a CTA holds: the streaming kernel, one launch per level
    cudaError_t e = dispatch_select(l1, KIND_MEAN, false, g.D, units, s);
    if (e != cudaSuccess) return e;
    return dispatch_select(l2, KIND_QUEST, g.kv_bf16, g.D, units, s);
}

}  // namespace sa
