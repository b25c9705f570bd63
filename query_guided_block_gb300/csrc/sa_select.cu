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
#include "sa_common.cuh"
#include "sa_internal.h"

namespace sa {
namespace {

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kMaxStages = 3;             // chunks in flight per CTA (2 or 3, set at launch)
constexpr int kStageBytes = 32 * 1024;    // metadata bytes per chunk
constexpr int kMaxSelectKeys = 16384;     // candidates per unit held in shared memory

enum { KIND_QUEST = 0, KIND_MEAN = 1 };

struct SelectArgs {
    const void* q;
    int q_bf16;
    const void* kmin;    // QUEST: [units, rows, D] metadata dtype
    const void* kmax;
    const float* kmean;  // MEAN:  [units, rows, D] fp32
    int rows;            // metadata rows per unit (the context's)
    int row_stride;      // metadata rows allocated per unit (capacity)
    int Hkv, G;
    int Hq;
    int Q;               // query vectors per sequence; the coefficients sum over all of them
    // candidates: c in [0, n_cand); direct (c is the row) or via level-1 survivors
    int via_survivors;
    const int32_t* surv;     // [units, surv_stride], ascending coarse ids
    const int32_t* n_surv;   // [units]
    int surv_stride;
    int per_coarse;          // rows per coarse block
    int row_limit;           // rows >= row_limit are not candidates (window / past end)
    int n_cand;              // candidate slots per unit = groups * group_rows
    int groups, group_rows;  // candidate slots come in groups of contiguous rows
    int chunks_per_group, chunks_per_unit, total_chunks;
    int stages;
    // selection
    int k;
    int win_first, win_count;
    const int32_t* reserve;  // [units, n_reserve] extra block ids united with the top-k (or null)
    int n_reserve;
    int32_t* out_ids;
    int out_stride;
    int32_t* out_count;
    // workspace
    float* scores;           // [units, n_cand]
    uint32_t* counters;      // [units] scored slots
    uint32_t* err;
};

// Row id of candidate c of unit u, or -1 when c is not a candidate.
__device__ __forceinline__ int candidate_row(const SelectArgs& a, int u, int c)
{
    if (c >= a.n_cand) return -1;
    if (!a.via_survivors) return c < a.row_limit ? c : -1;
    const int i = c / a.per_coarse;
    if (i >= a.n_surv[u]) return -1;
    const int row = a.surv[size_t(u) * a.surv_stride + i] * a.per_coarse + (c - i * a.per_coarse);
    return row < a.row_limit ? row : -1;
}

// ------------------------------------------------------------- top-k ----
// Runs in one CTA.  keys[0..n) hold order keys (0 = not a candidate); candidate order
// is block-id order.  Finds the k-th candidate (T, cT) in (key desc, index asc) order;
// the selection is then {c : key > T, or key == T and c <= cT}.
//
// Radix passes take 11-bit digits below the common prefix of the candidates' keys
// (2048-bin shared-memory histograms).  As soon as the boundary bin holds at most
// kGather candidates they are gathered and ranked directly; if it holds exactly the
// remaining count, every key of that bin is in.
__device__ void topk_and_emit(const SelectArgs& a, int u, uint32_t* keys, int n, int n_valid)
{
    constexpr int kBins = 2048;
    constexpr int kBinsPerThread = kBins / kSelThreads;
    constexpr int kGather = kSelThreads;
    __shared__ uint32_t hist[kBins];
    __shared__ uint32_t s_bin, s_above, s_binc, s_lo, s_hi, s_T;
    __shared__ int s_cT, s_ng;
    __shared__ uint32_t g_key[kGather];
    __shared__ int g_idx[kGather];
    __shared__ int s_wtot[kSelWarps];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int k_eff = min(a.k, n_valid);
    int32_t* out = a.out_ids + size_t(u) * a.out_stride;

    // mode 0: none / all candidates; 1: (key & mask) >= prefix; 2: threshold (T, cT)
    int mode = 0;
    uint32_t prefix = 0, mask = 0, T = 0;
    int cT = -1;
    int krem = k_eff;
    if (k_eff > 0 && k_eff < n_valid) {
        if (tid == 0) { s_lo = 0xffffffffu; s_hi = 0u; }
        __syncthreads();
        uint32_t lo = 0xffffffffu, hi = 0u;
        for (int c = tid; c < n; c += kSelThreads) {
            const uint32_t key = keys[c];
            if (key) { lo = min(lo, key); hi = max(hi, key); }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            lo = min(lo, __shfl_xor_sync(kFullMask, lo, off));
            hi = max(hi, __shfl_xor_sync(kFullMask, hi, off));
        }
        if (lane == 0) { atomicMin(&s_lo, lo); atomicMax(&s_hi, hi); }
        __syncthreads();
        lo = s_lo;
        hi = s_hi;
        int low_bits = (lo == hi) ? 0 : 32 - __clz(lo ^ hi);
        mask = low_bits >= 32 ? 0u : ~((1u << low_bits) - 1u);
        prefix = hi & mask;
        uint32_t binc = uint32_t(n_valid);   // candidates matching the current prefix
        while (true) {
            if (binc <= uint32_t(kGather) || low_bits == 0) break;
            const int w = min(11, low_bits);
            const int shift = low_bits - w;
            const uint32_t dmask = (1u << w) - 1u;
#pragma unroll
            for (int i = 0; i < kBinsPerThread; ++i) hist[tid + i * kSelThreads] = 0u;
            __syncthreads();
            for (int c = tid; c < n; c += kSelThreads) {
                const uint32_t key = keys[c];
                if (key != 0u && (key & mask) == prefix) atomicAdd(&hist[(key >> shift) & dmask], 1u);
            }
            __syncthreads();
            // thread t owns bins 2047-8t .. 2040-8t (descending); scan from the top
            uint32_t cnt[kBinsPerThread], sum = 0;
#pragma unroll
            for (int r = 0; r < kBinsPerThread; ++r) {
                cnt[r] = hist[kBins - 1 - kBinsPerThread * tid - r];
                sum += cnt[r];
            }
            uint32_t inc = sum;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t t = __shfl_up_sync(kFullMask, inc, off);
                if (lane >= off) inc += t;
            }
            if (lane == 31) s_wtot[warp] = int(inc);
            __syncthreads();
            for (int wv = 0; wv < warp; ++wv) inc += uint32_t(s_wtot[wv]);
            const uint32_t before = inc - sum;
            if (before < uint32_t(krem) && inc >= uint32_t(krem)) {
                uint32_t above = before;
                for (int r = 0; r < kBinsPerThread; ++r) {
                    if (above + cnt[r] >= uint32_t(krem)) {
                        s_bin = uint32_t(kBins - 1 - kBinsPerThread * tid - r);
                        s_above = above;
                        s_binc = cnt[r];
                        break;
                    }
                    above += cnt[r];
                }
            }
            __syncthreads();
            krem -= int(s_above);
            prefix |= s_bin << shift;
            mask |= dmask << shift;
            low_bits = shift;
            binc = s_binc;
            __syncthreads();   // s_wtot / s_bin are rewritten below
            if (int(binc) == krem) break;
        }
        if (int(binc) == krem) {
            mode = 1;   // the whole boundary bin is in
        } else if (binc <= uint32_t(kGather)) {
            // gather the boundary candidates and rank them by (key desc, index asc)
            if (tid == 0) s_ng = 0;
            __syncthreads();
            for (int c = tid; c < n; c += kSelThreads) {
                const uint32_t key = keys[c];
                if (key != 0u && (key & mask) == prefix) {
                    const int slot = atomicAdd(&s_ng, 1);
                    g_key[slot] = key;
                    g_idx[slot] = c;
                }
            }
            __syncthreads();
            const int ng = s_ng;
            if (tid < ng) {
                const uint32_t mk = g_key[tid];
                const int mi = g_idx[tid];
                int rank = 0;
                for (int j = 0; j < ng; ++j)
                    rank += (g_key[j] > mk) || (g_key[j] == mk && g_idx[j] < mi);
                if (rank == krem - 1) { s_T = mk; s_cT = mi; }
            }
            __syncthreads();
            mode = 2;
            T = s_T;
            cT = s_cT;
        } else {
            // more than kGather candidates share every key bit: ties on one key value;
            // the krem lowest indices among them are in (ordered count over indices)
            const int chunk = ((n + kSelWarps * 32 - 1) / (kSelWarps * 32)) * 32;
            const int c0 = warp * chunk, c1 = min(n, c0 + chunk);
            int eq = 0;
            for (int c = c0 + lane; c - lane < c1; c += 32) {
                const bool e = c < c1 && keys[c] == prefix;
                eq += __popc(__ballot_sync(kFullMask, e));
            }
            if (lane == 0) s_wtot[warp] = eq;
            __syncthreads();
            int run = 0;
            for (int wv = 0; wv < warp; ++wv) run += s_wtot[wv];
            for (int c = c0 + lane; c - lane < c1; c += 32) {
                const bool e = c < c1 && keys[c] == prefix;
                const uint32_t eb = __ballot_sync(kFullMask, e);
                if (e && run + __popc(eb & lanemask_lt()) == krem - 1) s_cT = c;
                run += __popc(eb);
            }
            __syncthreads();
            mode = 2;
            T = prefix;
            cT = s_cT;
        }
    } else if (k_eff > 0) {
        mode = 1;   // every candidate (mask = prefix = 0)
    }

    auto selected = [&](int c) -> bool {
        const uint32_t key = keys[c];
        if (mode == 0 || key == 0u) return false;
        if (mode == 1) return (key & mask) >= prefix;
        return key > T || (key == T && c <= cT);
    };
    if (a.n_reserve > 0) {
        // Reserve set (SparDA page §3.4): the top-k rows and the unit's reserve blocks
        // outside the window are marked in a bitmap over block ids (the histogram's
        // storage, free now), then emitted in ascending order, then the window.
        uint32_t* bits = hist;
        const int nw = (a.rows + 31) >> 5;   // <= kBins words: rows <= 16384
        for (int i = tid; i < nw; i += kSelThreads) bits[i] = 0u;
        __syncthreads();
        for (int c = tid; c < n; c += kSelThreads)
            if (selected(c)) {
                const int r = candidate_row(a, u, c);
                atomicOr(&bits[r >> 5], 1u << (r & 31));
            }
        for (int i = tid; i < a.n_reserve; i += kSelThreads) {
            const int j = a.reserve[size_t(u) * a.n_reserve + i];
            if (j < 0 || j >= a.rows) raise_error(a.err, SPARSE_ATTN_ERR_SEL_ID);
            else if (j < a.win_first) atomicOr(&bits[j >> 5], 1u << (j & 31));
        }
        __syncthreads();
        const int per = (nw + kSelThreads - 1) / kSelThreads;   // words per thread, in order
        const int w0 = min(nw, tid * per), w1 = min(nw, w0 + per);
        int cnt = 0;
        for (int w = w0; w < w1; ++w) cnt += __popc(bits[w]);
        int inc = cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int t = __shfl_up_sync(kFullMask, inc, off);
            if (lane >= off) inc += t;
        }
        if (lane == 31) s_wtot[warp] = inc;
        __syncthreads();
        int pos = inc - cnt, total = 0;
        for (int wv = 0; wv < kSelWarps; ++wv) {
            pos += wv < warp ? s_wtot[wv] : 0;
            total += s_wtot[wv];
        }
        for (int w = w0; w < w1; ++w)
            for (uint32_t m = bits[w]; m; m &= m - 1) out[pos++] = w * 32 + (__ffs(m) - 1);
        for (int i = tid; i < a.win_count; i += kSelThreads) out[total + i] = a.win_first + i;
        if (tid == 0) a.out_count[u] = total + a.win_count;
        return;
    }
    // Each warp owns a contiguous chunk of candidates, read lane-interleaved, so ballot
    // order is candidate order.
    const int chunk = ((n + kSelWarps * 32 - 1) / (kSelWarps * 32)) * 32;
    const int c0 = warp * chunk, c1 = min(n, c0 + chunk);
    int cnt = 0;
    for (int c = c0 + lane; c - lane < c1; c += 32)
        cnt += __popc(__ballot_sync(kFullMask, c < c1 && selected(c)));
    if (lane == 0) s_wtot[warp] = cnt;
    __syncthreads();
    int pos = 0;
    for (int wv = 0; wv < warp; ++wv) pos += s_wtot[wv];
    for (int c = c0 + lane; c - lane < c1; c += 32) {
        const bool sl = c < c1 && selected(c);
        const uint32_t sb = __ballot_sync(kFullMask, sl);
        if (sl) out[pos + __popc(sb & lanemask_lt())] = candidate_row(a, u, c);
        pos += __popc(sb);
    }
    for (int i = tid; i < a.win_count; i += kSelThreads) out[k_eff + i] = a.win_first + i;
    if (tid == 0) a.out_count[u] = k_eff + a.win_count;
}

// Unit u's scores -> order keys in shared memory (0 for slots that are not
// candidates); returns the number of candidates.  Loads are issued in batches of
// independent requests so the L2 latency is paid once per batch, not per element.
__device__ int load_keys(const SelectArgs& a, int u, uint32_t* keys, int* s_count)
{
    constexpr int kBatch = 16;   // 4096 candidates: one round trip
    const float* row = a.scores + size_t(u) * a.n_cand;
    int mine = 0;
    for (int base = threadIdx.x; base < a.n_cand; base += kSelThreads * kBatch) {
        float x[kBatch];
        bool ok[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int c = base + i * kSelThreads;
            ok[i] = c < a.n_cand && candidate_row(a, u, c) >= 0;
            x[i] = ok[i] ? __ldcg(row + c) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int c = base + i * kSelThreads;
            if (c < a.n_cand) keys[c] = ok[i] ? order_key(x[i]) : 0u;
            mine += ok[i];
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mine += __shfl_xor_sync(kFullMask, mine, off);
    if ((threadIdx.x & 31) == 0) atomicAdd(s_count, mine);
    __syncthreads();
    return *s_count;
}

// ------------------------------------------------------------- kernel ---
// Persistent streaming kernel.  The candidates of every unit are cut into chunks of
// contiguous metadata rows (<= kStageBytes per chunk), numbered unit-major; CTA i
// owns an equal contiguous range of chunk ids, so it crosses a unit boundary once or
// twice and needs no per-chunk synchronisation with other CTAs.  The CTA keeps
// kStages chunks in flight with 1-D bulk async copies (complete_tx on one mbarrier per
// stage; a stage's copies are issued by different warps); all threads score from
// shared memory.  When a CTA finishes its segment of a
// unit it adds the segment's slot count to the unit's counter; the CTA that completes
// the count runs the unit's top-k.  Nothing waits on another CTA.
template <int KIND, bool MBF16, int D>
struct SelectShape {
    static constexpr int ESZ = (KIND == KIND_QUEST && MBF16) ? 2 : 4;
    static constexpr int EPL = 16 / ESZ;
    static constexpr int LPR = D / EPL;
    static constexpr int RPW = 32 / LPR;
    static constexpr int ROW_BYTES = D * ESZ;
    static constexpr int ARRAYS = KIND == KIND_QUEST ? 2 : 1;
    static constexpr int ROWS = kStageBytes / (ARRAYS * ROW_BYTES);   // rows per chunk
    static constexpr int R = ROWS / (kSelWarps * RPW);                 // rows per lane group
    static_assert(R >= 1 && ROWS % (kSelWarps * RPW) == 0, "chunk rows must split over the warps");
};

struct ChunkInfo {
    int u, cand0, row0, nrows, nslots;
};

__device__ __forceinline__ ChunkInfo chunk_info(const SelectArgs& a, int cid, int rows_per_chunk)
{
    ChunkInfo c;
    c.u = cid / a.chunks_per_unit;
    const int rem = cid - c.u * a.chunks_per_unit;
    const int grp = rem / a.chunks_per_group;
    const int slot0 = (rem - grp * a.chunks_per_group) * rows_per_chunk;
    c.nslots = min(rows_per_chunk, a.group_rows - slot0);
    c.cand0 = grp * a.group_rows + slot0;
    if (a.via_survivors) {
        if (grp >= a.n_surv[c.u]) {
            c.row0 = 0;
            c.nrows = 0;
            return c;
        }
        c.row0 = a.surv[size_t(c.u) * a.surv_stride + grp] * a.per_coarse + slot0;
    } else {
        c.row0 = slot0;
    }
    c.nrows = max(0, min(c.nslots, a.row_limit - c.row0));
    return c;
}

template <int KIND, bool MBF16, int D>
__global__ void __launch_bounds__(kSelThreads) select_kernel(SelectArgs a)
{
    using SS = SelectShape<KIND, MBF16, D>;
    constexpr int EPL = SS::EPL, LPR = SS::LPR, RPW = SS::RPW, ROWS = SS::ROWS, R = SS::R;
    extern __shared__ __align__(128) unsigned char smem[];
    const int stages = a.stages;
    uint32_t* keys = reinterpret_cast<uint32_t*>(smem + stages * kStageBytes);
    __shared__ __align__(8) uint64_t full[kMaxStages];
    __shared__ int s_topk_unit, s_nvalid;
    __shared__ float s_coef[2][kSelThreads];   // per-thread partial sums of the query coefficients

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sub = lane % LPR, rsub = lane / LPR;
    const int d0 = sub * EPL;
    const int row_group = warp * RPW + rsub;            // rows row_group*R .. +R-1 of a chunk
    const char* hi_src = reinterpret_cast<const char*>(KIND == KIND_QUEST ? a.kmax : (const void*)a.kmean);
    const char* lo_src = reinterpret_cast<const char*>(a.kmin);
    const int c_begin = int((long long)a.total_chunks * blockIdx.x / gridDim.x);
    const int c_end = int((long long)a.total_chunks * (blockIdx.x + 1) / gridDim.x);

    // Copies issued by one thread complete one after another, so each stage's copies
    // come from different warps (lane 0): stage s, array a -> warp (2 s + a) mod 8.
    auto issue = [&](int cid, int array) {
        const int s = (cid - c_begin) % stages;
        const ChunkInfo c = chunk_info(a, cid, ROWS);
        const uint32_t bytes = uint32_t(c.nrows) * SS::ROW_BYTES;
        if (array == 0) mbar_arrive_expect_tx(&full[s], bytes * SS::ARRAYS);
        if (bytes) {
            const size_t off = (size_t(c.u) * a.row_stride + c.row0) * SS::ROW_BYTES;
            unsigned char* dst = smem + s * kStageBytes;
            if (array == 0) bulk_copy_g2s(dst, hi_src + off, bytes, &full[s]);
            else bulk_copy_g2s(dst + ROWS * SS::ROW_BYTES, lo_src + off, bytes, &full[s]);
        }
    };
    auto issue_mine = [&](int cid) {   // every warp's lane 0
        const int s = (cid - c_begin) % stages;
        for (int arr = 0; arr < SS::ARRAYS; ++arr)
            if ((s * SS::ARRAYS + arr) % kSelWarps == warp) issue(cid, arr);
    };

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    allow_dependents_early();
    grid_dependency_wait();   // inputs and workspace may come from the previous kernel
    __syncthreads();
    if (lane == 0)
        for (int cid = c_begin; cid < c_end && cid < c_begin + stages; ++cid) issue_mine(cid);

    int cur_u = -1;
    uint32_t seg_slots = 0;
    float cp[EPL], cn[EPL];
    for (int cid = c_begin; cid < c_end; ++cid) {
        const int k = cid - c_begin;
        const int s = k % stages;
        const uint32_t parity = uint32_t(k / stages) & 1u;
        const ChunkInfo c = chunk_info(a, cid, ROWS);
        if (c.u != cur_u) {   // query coefficients of this unit (uniform across the CTA)
            // The CTA sums the unit's Q x G query rows per channel together: thread t takes
            // channel t mod D of rows t / D, t / D + 256 / D, ... (coalesced loads), the
            // 256 / D partial sums of a channel meet in shared memory.
            cur_u = c.u;
            const int b = c.u / a.Hkv, kvh = c.u - (c.u / a.Hkv) * a.Hkv;
            constexpr int RSTEP = kSelThreads / D;
            const int dch = tid % D;
            const int rows = a.Q * a.G;
            float pp = 0.f, nn = 0.f;
#pragma unroll 8
            for (int r = tid / D; r < rows; r += RSTEP) {
                const int t = r / a.G, g = r - t * a.G;
                const float x = load_q(a.q, ((size_t(b) * a.Q + t) * a.Hq + size_t(kvh) * a.G + g) * D + dch,
                                       a.q_bf16 != 0);
                if constexpr (KIND == KIND_QUEST) {
                    pp += fmaxf(x, 0.f);
                    nn += fminf(x, 0.f);
                } else {
                    pp += x;
                }
            }
            s_coef[0][tid] = pp;
            s_coef[1][tid] = nn;
            __syncthreads();
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                float sp = 0.f, sn = 0.f;
#pragma unroll
                for (int k2 = 0; k2 < RSTEP; ++k2) {
                    sp += s_coef[0][d0 + e + k2 * D];
                    sn += s_coef[1][d0 + e + k2 * D];
                }
                cp[e] = sp;
                cn[e] = sn;
            }
        }
        if (!mbar_wait_bounded(&full[s], parity, kWaitCycles)) raise_error(a.err, SPARSE_ATTN_ERR_TIMEOUT);

        // R rows per lane group, partial dots summed over the group's LPR lanes at once
        const unsigned char* hi = smem + s * kStageBytes + d0 * SS::ESZ;
        const unsigned char* lo = hi + ROWS * SS::ROW_BYTES;
        float part[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int row = row_group * R + r;
            float fh[EPL], acc = 0.f;
            unpack16<SS::ESZ == 2>(*reinterpret_cast<const uint4*>(hi + row * SS::ROW_BYTES), fh);
            if constexpr (KIND == KIND_QUEST) {
                float fl[EPL];
                unpack16<SS::ESZ == 2>(*reinterpret_cast<const uint4*>(lo + row * SS::ROW_BYTES), fl);
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc = fmaf(cp[e], fh[e], fmaf(cn[e], fl[e], acc));
            } else {
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc = fmaf(cp[e], fh[e], acc);
            }
            part[r] = acc;
        }
        group_reduce_transposed<R, LPR>(part, lane);
        {
            constexpr int OUT = R >= LPR ? R / LPR : 1;
            constexpr int SPREAD = R >= LPR ? 1 : LPR / R;
            float* srow = a.scores + size_t(c.u) * a.n_cand + c.cand0;
            if (sub % SPREAD == 0) {
#pragma unroll
                for (int i = 0; i < OUT; ++i) {
                    const int r = R >= LPR ? sub * (R / LPR) + i : sub / SPREAD;
                    const int row = row_group * R + r;
                    if (row < c.nrows) srow[row] = part[i];
                }
            }
        }
        seg_slots += uint32_t(c.nslots);
        __syncthreads();   // stage s fully read; this chunk's scores written
        if (lane == 0 && cid + stages < c_end) issue_mine(cid + stages);

        // end of this CTA's segment of unit c.u: report it; the completing CTA selects
        const bool seg_end = cid + 1 == c_end || (cid + 1) / a.chunks_per_unit != c.u;
        if (seg_end) {
            if (tid == 0) {
                const uint32_t before = atomic_add_acq_rel_u32(&a.counters[c.u], seg_slots);
                s_topk_unit = (before + seg_slots == uint32_t(a.n_cand)) ? c.u : -1;
            }
            seg_slots = 0;
            __syncthreads();
            const int tu = s_topk_unit;
            if (tu >= 0) {
                if (tid == 0) {
                    a.counters[tu] = 0u;   // every slot of this unit is scored
                    s_nvalid = 0;
                }
                __syncthreads();
                const int n_valid = load_keys(a, tu, keys, &s_nvalid);
                topk_and_emit(a, tu, keys, a.n_cand, n_valid);
                __syncthreads();
            }
        }
    }
}

template <int KIND, bool MBF16, int D>
cudaError_t launch_select_t(const SelectArgs& a0, int units, cudaStream_t s)
{
    using SS = SelectShape<KIND, MBF16, D>;
    SelectArgs a = a0;
    a.chunks_per_group = (a.group_rows + SS::ROWS - 1) / SS::ROWS;
    a.chunks_per_unit = a.groups * a.chunks_per_group;
    a.total_chunks = units * a.chunks_per_unit;
    const size_t keys_bytes = size_t(a.n_cand) * sizeof(uint32_t);
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
    return launch_after_previous(select_kernel<KIND, MBF16, D>, dim3(unsigned(ctas)), dim3(kSelThreads), smem, s, a);
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

}  // namespace

cudaError_t launch_select(const Geometry& g, const WorkspaceLayout& L, char* ws, const void* q,
                          const void* kmin, const void* kmax, const float* kmean,
                          const int32_t* reserve_ids, int32_t* sel_ids, int32_t* sel_count,
                          cudaStream_t s)
{
    const int units = g.units();
    if (units == 0) return cudaSuccess;
    SelectArgs a{};
    a.q = q;
    a.q_bf16 = g.q_bf16;
    a.kmin = kmin;
    a.kmax = kmax;
    a.kmean = kmean;
    a.Hkv = g.Hkv;
    a.G = g.G;
    a.Hq = g.Hq;
    a.Q = g.Q;
    a.err = reinterpret_cast<uint32_t*>(ws + L.err);
    a.scores = reinterpret_cast<float*>(ws + L.scores);
    a.counters = reinterpret_cast<uint32_t*>(ws + L.sel_counters);

    if (!g.two_level) {
        a.rows = g.nb;
        a.row_stride = g.score_kind == SPARSE_ATTN_SCORE_MEAN ? g.n_mean_cap : g.nb_cap;
        a.via_survivors = 0;
        a.row_limit = g.win_first;
        a.n_cand = g.n_cand;
        a.groups = 1;
        a.group_rows = g.n_cand;
        a.k = g.topk;
        a.win_first = g.win_first;
        a.win_count = g.win_count;
        a.reserve = reserve_ids;
        a.n_reserve = g.n_reserve;
        a.out_ids = sel_ids;
        a.out_stride = g.sel_stride;
        a.out_count = sel_count;
        if (a.n_cand == 0) {
            // no candidates: one slot-free pass that only emits the window
            a.group_rows = 1;
            a.n_cand = 1;
            a.row_limit = 0;
        }
        const int kind = g.score_kind == SPARSE_ATTN_SCORE_MEAN ? KIND_MEAN : KIND_QUEST;
        return dispatch_select(a, kind, g.kv_bf16, g.D, units, s);
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
