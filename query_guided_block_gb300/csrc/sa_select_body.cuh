// Device side of block selection (scoring stream, radix top-k, emission), shared by
// the select kernels and the fused step kernel.  The design notes are in sa_select.cu.
#pragma once

#include "sa_common.cuh"
#include "sa_internal.h"

namespace sa {
namespace {

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kMaxStages = 5;             // chunks in flight per CTA (set at launch)
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
    int unit_ranges;         // warp-slab select: CTA c streams unit c's chunks (no more units than CTAs)
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
// Keys per thread in the top-k passes: thread t owns keys [t * key_tile(n), (t + 1) *
// key_tile(n)) and reads them four at a time; the key array is zero-padded to
// kSelThreads * key_tile(n) entries.
__host__ __device__ constexpr int key_tile(int n)
{
    return ((n + kSelThreads * 4 - 1) / (kSelThreads * 4)) * 4;
}

// Runs in one CTA.  keys[0..n) hold order keys (0 = not a candidate); candidate order
// is block-id order.  Finds the k-th candidate (T, cT) in (key desc, index asc) order;
// the selection is then {c : key > T, or key == T and c <= cT}.
//
// Radix passes take 11-bit digits below the common prefix of the candidates' keys
// (2048-bin shared-memory histograms).  As soon as the boundary bin holds at most
// kGather candidates they are gathered and ranked directly; if it holds exactly the
// remaining count, every key of that bin is in.  key_lo / key_hi: the smallest and
// largest key among the n_valid candidates (from load_keys).
__device__ void topk_and_emit(const SelectArgs& a, int u, uint32_t* keys, int n, int n_valid,
                              uint32_t key_lo, uint32_t key_hi, const int* surv_smem = nullptr, int n_surv_smem = 0)
{
    // candidate -> block id; with the level-1 survivors already in shared memory the
    // emission does not go back to global memory for them (same mapping as candidate_row)
    auto row_of = [&](int c) -> int {
        if (surv_smem == nullptr) return candidate_row(a, u, c);
        if (c >= a.n_cand) return -1;
        const int i = c / a.per_coarse;
        if (i >= n_surv_smem) return -1;
        const int row = surv_smem[i] * a.per_coarse + (c - i * a.per_coarse);
        return row < a.row_limit ? row : -1;
    };
    constexpr int kBins = 2048;
    constexpr int kBinsPerThread = kBins / kSelThreads;
    constexpr int kGather = kSelThreads;
    constexpr int kGatherDirect = 64;   // ranked directly without a radix pass
    __shared__ uint32_t hist[kBins];
    __shared__ uint32_t s_bin, s_above, s_binc, s_T;
    __shared__ int s_cT, s_ng;
    __shared__ uint32_t g_key[kGather];
    __shared__ int g_idx[kGather];
    __shared__ int s_wtot[kSelWarps];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int k_eff = min(a.k, n_valid);
    int32_t* out = a.out_ids + size_t(u) * a.out_stride;
    const int kpt = key_tile(n);
    const uint32_t* my_keys = keys + tid * kpt;      // 16-byte aligned: kpt is a multiple of 4

    // mode 0: none / all candidates; 1: (key & mask) >= prefix; 2: threshold (T, cT)
    int mode = 0;
    uint32_t prefix = 0, mask = 0, T = 0;
    int cT = -1;
    int krem = k_eff;
    if (k_eff > 0 && k_eff < n_valid) {
        const uint32_t lo = key_lo, hi = key_hi;
        int low_bits = (lo == hi) ? 0 : 32 - __clz(lo ^ hi);
        mask = low_bits >= 32 ? 0u : ~((1u << low_bits) - 1u);
        prefix = hi & mask;
        uint32_t binc = uint32_t(n_valid);   // candidates matching the current prefix
        // Gather the boundary candidates once they fit the gather buffer, but take at
        // least one radix pass first unless they are few: ranking a full buffer is
        // quadratic in the candidates.
        int passes = 0;
        while (true) {
            if (low_bits == 0 || (binc <= uint32_t(kGather) && (passes > 0 || binc <= uint32_t(kGatherDirect)))) break;
            ++passes;
            const int w = min(11, low_bits);
            const int shift = low_bits - w;
            const uint32_t dmask = (1u << w) - 1u;
#pragma unroll
            for (int i = 0; i < kBinsPerThread; ++i) hist[tid + i * kSelThreads] = 0u;
            __syncthreads();
            for (int i = 0; i < kpt; i += 4) {
                const uint4 v = *reinterpret_cast<const uint4*>(my_keys + i);
                const uint32_t kk[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (kk[e] != 0u && (kk[e] & mask) == prefix) atomicAdd(&hist[(kk[e] >> shift) & dmask], 1u);
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
            for (int i = 0; i < kpt; i += 4) {
                const uint4 v = *reinterpret_cast<const uint4*>(my_keys + i);
                const uint32_t kk[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (kk[e] != 0u && (kk[e] & mask) == prefix) {
                        const int slot = atomicAdd(&s_ng, 1);
                        g_key[slot] = kk[e];
                        g_idx[slot] = tid * kpt + i + e;
                    }
                }
            }
            __syncthreads();
            const int ng = s_ng;
            if (tid < ng) {
                const uint32_t mk = g_key[tid];
                const int mi = g_idx[tid];
                int rank = 0;
#pragma unroll 8
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

    auto selected_key = [&](uint32_t key, int c) -> bool {
        if (mode == 0 || key == 0u) return false;
        if (mode == 1) return (key & mask) >= prefix;
        return key > T || (key == T && c <= cT);
    };
    auto selected = [&](int c) -> bool { return selected_key(keys[c], c); };
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
                const int r = row_of(c);
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
    // Thread t owns candidates [t * kpt, (t + 1) * kpt): count its selected ones, find
    // its offset by a scan over the threads (thread order is candidate order), then
    // write their rows in order.  Each pass reads its keys four at a time.
    int cnt = 0;
    for (int i = 0; i < kpt; i += 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(my_keys + i);
        const uint32_t kk[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) cnt += selected_key(kk[e], tid * kpt + i + e);
    }
    int inc = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(kFullMask, inc, off);
        if (lane >= off) inc += t;
    }
    if (lane == 31) s_wtot[warp] = inc;
    __syncthreads();
    int pos = inc - cnt;
    for (int wv = 0; wv < warp; ++wv) pos += s_wtot[wv];
    for (int i = 0; i < kpt && cnt > 0; i += 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(my_keys + i);
        const uint32_t kk[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = tid * kpt + i + e;
            if (selected_key(kk[e], c)) {
                out[pos++] = row_of(c);
                --cnt;
            }
        }
    }
    for (int i = tid; i < a.win_count; i += kSelThreads) out[k_eff + i] = a.win_first + i;
    if (tid == 0) a.out_count[u] = k_eff + a.win_count;
}

// Unit u's scores -> order keys in shared memory (0 for slots that are not
// candidates, and for the padding up to kSelThreads * key_tile(n_cand) entries);
// returns the number of candidates and the smallest and largest key.  Loads are issued in batches of
// independent requests so the L2 latency is paid once per batch, not per element.
__device__ int load_keys(const SelectArgs& a, int u, uint32_t* keys, uint32_t& key_lo, uint32_t& key_hi)
{
    constexpr int kBatch = 16;   // 4096 candidates: one round trip
    __shared__ int s_count;
    __shared__ uint32_t s_lo, s_hi;
    if (threadIdx.x == 0) {
        s_count = 0;
        s_lo = 0xffffffffu;
        s_hi = 0u;
    }
    __syncthreads();
    const float* row = a.scores + size_t(u) * a.n_cand;
    int mine = 0;
    uint32_t lo = 0xffffffffu, hi = 0u;
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
            const uint32_t key = order_key(x[i]);
            if (c < a.n_cand) keys[c] = ok[i] ? key : 0u;
            if (ok[i]) {
                lo = min(lo, key);
                hi = max(hi, key);
            }
            mine += ok[i];
        }
    }
    for (int c = a.n_cand + threadIdx.x; c < kSelThreads * key_tile(a.n_cand); c += kSelThreads) keys[c] = 0u;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        mine += __shfl_xor_sync(kFullMask, mine, off);
        lo = min(lo, __shfl_xor_sync(kFullMask, lo, off));
        hi = max(hi, __shfl_xor_sync(kFullMask, hi, off));
    }
    if ((threadIdx.x & 31) == 0) {
        atomicAdd(&s_count, mine);
        atomicMin(&s_lo, lo);
        atomicMax(&s_hi, hi);
    }
    __syncthreads();
    key_lo = s_lo;
    key_hi = s_hi;
    return s_count;
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

// One CTA's share of a select launch: CTA blockIdx.x of gridDim.x streams its
// contiguous range of chunks; the CTA completing a unit ranks and emits it.  With
// `ready` set, that CTA then publishes the step's flag value in ready[u] (release) once
// the unit's ids and count are written, for a decode in the same grid or in the kernel
// launched after this one.  Returns that value (0 without `ready`).
template <int KIND, bool MBF16, int D>
__device__ __forceinline__ uint32_t select_body(const SelectArgs& a, uint32_t* ready)
{
    using SS = SelectShape<KIND, MBF16, D>;
    constexpr int EPL = SS::EPL, LPR = SS::LPR, RPW = SS::RPW, ROWS = SS::ROWS, R = SS::R;
    extern __shared__ __align__(128) unsigned char smem[];
    const int stages = a.stages;
    uint32_t* keys = reinterpret_cast<uint32_t*>(smem + stages * kStageBytes);
    __shared__ __align__(8) uint64_t full[kMaxStages];
    __shared__ int s_topk_unit;
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
    grid_dependency_wait();   // inputs and workspace may come from the previous kernel
    // the step's flag value, read before any dependent kernel may start (that kernel
    // reads the same epoch word, which only a finishing step changes)
    const uint32_t flag_value = ready != nullptr ? step_flag_value(a.err) : 0u;
    // Only now may a dependent kernel start: whatever ran before this one has finished,
    // so a dependent that skips its own wait (waiting on ready flags instead) still
    // sees every earlier write.
    allow_dependents_early();
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
                if (tid == 0) a.counters[tu] = 0u;   // every slot of this unit is scored
                uint32_t klo, khi;
                const int n_valid = load_keys(a, tu, keys, klo, khi);
                topk_and_emit(a, tu, keys, a.n_cand, n_valid, klo, khi);
                __syncthreads();
                if (ready != nullptr && tid == 0) {
                    __threadfence();
                    st_release_gpu(&ready[tu], flag_value);
                }
            }
        }
    }
    return flag_value;
}


// ---------------------------------------------- warp-independent streaming ---
// The same scores as select_body, without a CTA-wide step per chunk: the CTA's chunk
// range is cut into 8 KB slabs (both arrays of ROWS metadata rows) and warp w streams
// slabs w, w + 8, ... through its own kSlabSelStages-deep ring filled by its lanes'
// 16-byte cp.async copies, so a warp waits only on its own copies.  Each warp sums its
// unit's query coefficients itself (the same partial-sum order as the CTA-wide sum, so
// the scores are bit-identical) and, at the end of its part of a unit, adds its slot
// count to the unit's counter.  A warp that completes a unit records it; when every
// warp of the CTA has finished streaming, the CTA ranks and emits the units it
// completed, with the keys in the freed rings, and publishes each one in ready[].
constexpr int kSlabSelBytes = 8 * 1024;
constexpr int kSlabSelStages = 3;
constexpr int kSlabSelMaxUnits = 64;   // units one CTA may complete in a launch
constexpr int kSlabSelCoefUnits = 4;   // units whose query coefficients the CTA sums up front

template <int KIND, bool MBF16, int D>
struct SlabSelShape {
    using SS = SelectShape<KIND, MBF16, D>;
    static constexpr int ROWS = kSlabSelBytes / (SS::ARRAYS * SS::ROW_BYTES);   // rows per slab
    static constexpr int R = ROWS / SS::RPW;                                    // rows per lane group
    static constexpr int CPL = ROWS * SS::ROW_BYTES / (16 * 32);                // copies per lane per array
    static constexpr size_t RING_BYTES = size_t(kSelWarps) * kSlabSelStages * kSlabSelBytes;
    static_assert(R >= 1 && ROWS % SS::RPW == 0 && CPL >= 1 && (ROWS * SS::ROW_BYTES) % 512 == 0,
                  "a slab must split evenly over the lanes");
};

template <int KIND, bool MBF16, int D>
__device__ __forceinline__ uint32_t select_body_warps(const SelectArgs& a, uint32_t* ready,
                                                      uint32_t* queue = nullptr, int* kept = nullptr)
{
    using SS = SelectShape<KIND, MBF16, D>;
    using WS = SlabSelShape<KIND, MBF16, D>;
    constexpr int EPL = SS::EPL, LPR = SS::LPR, ROWS = WS::ROWS, R = WS::R;
    constexpr int S = kSlabSelStages;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_done[kSlabSelMaxUnits];
    __shared__ int s_ndone;
    __shared__ float s_cf[kSlabSelCoefUnits][2][kSelThreads];   // per-thread partial coefficient sums

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sub = lane % LPR, rsub = lane / LPR;
    const int d0 = sub * EPL;
    const char* hi_src = reinterpret_cast<const char*>(KIND == KIND_QUEST ? a.kmax : (const void*)a.kmean);
    const char* lo_src = reinterpret_cast<const char*>(a.kmin);
    // CTA c's chunks: an equal share, or with unit_ranges all of unit c's (so each CTA
    // completes exactly one unit)
    const int n_units_all = a.chunks_per_unit > 0 ? a.total_chunks / a.chunks_per_unit : 0;
    const int c_begin = a.unit_ranges ? min(int(blockIdx.x), n_units_all) * a.chunks_per_unit
                                      : int((long long)a.total_chunks * blockIdx.x / gridDim.x);
    const int c_end = a.unit_ranges ? min(int(blockIdx.x) + 1, n_units_all) * a.chunks_per_unit
                                    : int((long long)a.total_chunks * (blockIdx.x + 1) / gridDim.x);
    const int n_mine = c_end - c_begin > warp ? (c_end - c_begin - warp + kSelWarps - 1) / kSelWarps : 0;
    const uint32_t ring = smem_u32(smem) + uint32_t(warp) * (S * kSlabSelBytes);

    if (tid == 0) s_ndone = 0;
    grid_dependency_wait();   // inputs and workspace may come from the previous kernel
    const uint32_t flag_value = ready != nullptr ? step_flag_value(a.err) : 0u;   // see select_body
    allow_dependents_early();

    // Query coefficients of the first kSlabSelCoefUnits units of the range, summed by
    // the whole CTA before any copy is in flight (a load queued behind a warp's copies
    // waits for them): thread t takes channel t mod D of rows t / D, t / D + 256 / D, ...
    const int u_first = c_begin < c_end ? chunk_info(a, c_begin, ROWS).u : 0;
    const int n_units = c_begin < c_end ? chunk_info(a, c_end - 1, ROWS).u - u_first + 1 : 0;
    {
        constexpr int RSTEP = kSelThreads / D;
        const int dch = tid % D;
        const int rows = a.Q * a.G;
        for (int i = 0; i < min(n_units, kSlabSelCoefUnits); ++i) {
            const int u = u_first + i;
            const int b = u / a.Hkv, kvh = u - (u / a.Hkv) * a.Hkv;
            float pp = 0.f, nn = 0.f;
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
            s_cf[i][0][tid] = pp;
            s_cf[i][1][tid] = nn;
        }
    }
    __syncthreads();

    // slab k of this warp is chunk c_begin + warp + 8 k; rows past the chunk's end are
    // not copied (their stale values are never written out)
    auto issue = [&](int k, int st) {
        const ChunkInfo c = chunk_info(a, c_begin + warp + k * kSelWarps, ROWS);
        const size_t off = (size_t(c.u) * a.row_stride + c.row0) * SS::ROW_BYTES;
        const uint32_t nbytes = uint32_t(c.nrows) * SS::ROW_BYTES;
        const uint32_t dst = ring + uint32_t(st) * kSlabSelBytes;
#pragma unroll
        for (int arr = 0; arr < SS::ARRAYS; ++arr) {
            const char* src = (arr == 0 ? hi_src : lo_src) + off;
#pragma unroll
            for (int i = 0; i < WS::CPL; ++i) {
                const uint32_t byte = uint32_t(lane + i * 32) * 16;
                if (byte < nbytes) cp_async_16_zfill(dst + arr * (ROWS * SS::ROW_BYTES) + byte, src + byte, 16u);
            }
        }
    };
    // this unit's query coefficients, summed in the CTA-wide kernel's order: partial
    // sums over rows r, r + 256 / D, ... for r = 0 .. 256 / D - 1, then the partials
    float cp[EPL], cn[EPL];
    auto coefficients = [&](int u) {
        constexpr int RSTEP = kSelThreads / D;
        if (u - u_first < kSlabSelCoefUnits) {
            const int i = u - u_first;
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                float sp = 0.f, sn = 0.f;
#pragma unroll
                for (int k2 = 0; k2 < RSTEP; ++k2) {
                    sp += s_cf[i][0][d0 + e + k2 * D];
                    sn += s_cf[i][1][d0 + e + k2 * D];
                }
                cp[e] = sp;
                cn[e] = sn;
            }
            return;
        }
        constexpr int BATCH = 8;   // query rows whose channel vectors are loaded together
        static_assert(BATCH % RSTEP == 0, "a batch must hold whole row classes");
        const int b = u / a.Hkv, kvh = u - (u / a.Hkv) * a.Hkv;
        const int rows = a.Q * a.G;
        float pp[RSTEP][EPL], nn[RSTEP][EPL];
#pragma unroll
        for (int k2 = 0; k2 < RSTEP; ++k2)
#pragma unroll
            for (int e = 0; e < EPL; ++e) pp[k2][e] = nn[k2][e] = 0.f;
        for (int r0 = 0; r0 < rows; r0 += BATCH) {
            float x[BATCH][EPL];
#pragma unroll
            for (int j = 0; j < BATCH; ++j) {
                const int r = r0 + j;
                if (r < rows) {
                    const int t = r / a.G, g = r - t * a.G;
                    load_q_vec<EPL>(a.q, ((size_t(b) * a.Q + t) * a.Hq + size_t(kvh) * a.G + g) * D + d0,
                                    a.q_bf16 != 0, x[j]);
                }
            }
#pragma unroll
            for (int j = 0; j < BATCH; ++j) {
                if (r0 + j < rows) {
#pragma unroll
                    for (int e = 0; e < EPL; ++e) {
                        if constexpr (KIND == KIND_QUEST) {
                            pp[j % RSTEP][e] += fmaxf(x[j][e], 0.f);
                            nn[j % RSTEP][e] += fminf(x[j][e], 0.f);
                        } else {
                            pp[j % RSTEP][e] += x[j][e];
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            float sp = 0.f, sn = 0.f;
#pragma unroll
            for (int k2 = 0; k2 < RSTEP; ++k2) {
                sp += pp[k2][e];
                sn += nn[k2][e];
            }
            cp[e] = sp;
            cn[e] = sn;
        }
    };
    // this warp's part of unit u is scored: count it; the warp completing the unit
    // records it for the CTA
    auto report = [&](int u, uint32_t n) {
        __threadfence();   // this lane's score stores, before the count that publishes them
        __syncwarp();
        if (lane == 0) {
            const uint32_t before = atomic_add_acq_rel_u32(&a.counters[u], n);
            if (before + n == uint32_t(a.n_cand)) {
                a.counters[u] = 0u;   // every slot of this unit is scored
                const int i = atomicAdd(&s_ndone, 1);
                if (i < kSlabSelMaxUnits) s_done[i] = u;
                else raise_error(a.err, SPARSE_ATTN_ERR_CAPACITY);
            }
        }
        __syncwarp();
    };

#pragma unroll
    for (int k = 0; k < S - 1; ++k) {
        if (k < n_mine) issue(k, k);
        cp_async_commit();
    }
    int cur_u = -1;
    uint32_t seg_slots = 0;
    for (int k = 0; k < n_mine; ++k) {
        cp_async_wait_group<S - 2>();   // this lane's copies of slab k are done
        __syncwarp();                   // ... and every lane's; the stage read last is free
        if (k + S - 1 < n_mine) issue(k + S - 1, (k + S - 1) % S);
        cp_async_commit();
        const ChunkInfo c = chunk_info(a, c_begin + warp + k * kSelWarps, ROWS);
        if (c.u != cur_u) {
            if (cur_u >= 0) report(cur_u, seg_slots);
            cur_u = c.u;
            seg_slots = 0;
            coefficients(c.u);
        }
        const unsigned char* hi = smem + size_t(warp * S + k % S) * kSlabSelBytes + d0 * SS::ESZ;
        const unsigned char* lo = hi + ROWS * SS::ROW_BYTES;
        float part[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int row = rsub * R + r;
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
                    const int row = rsub * R + r;
                    if (row < c.nrows) srow[row] = part[i];
                }
            }
        }
        seg_slots += uint32_t(c.nslots);
    }
    if (cur_u >= 0) report(cur_u, seg_slots);
    cp_async_wait_group<0>();
    __syncthreads();   // every warp is done streaming; the rings are free

    uint32_t* keys = reinterpret_cast<uint32_t*>(smem);
    const int nd = min(s_ndone, kSlabSelMaxUnits);
    for (int i = 0; i < nd; ++i) {
        const int u = s_done[i];
        uint32_t klo, khi;
        const int n_valid = load_keys(a, u, keys, klo, khi);
        topk_and_emit(a, u, keys, a.n_cand, n_valid, klo, khi);
        __syncthreads();
        if (queue != nullptr) {
            // queue mode: the CTA keeps its first unit (*kept) and queues the others
            // (append, publish the position), then counts the unit as ranked (after
            // its queue entry: a count of every unit means the queue is complete)
            if (tid == 0) {
                if (i == 0) {
                    *kept = u;
                } else {
                    const int slot = int(atomicAdd(header_word(a.err, kHdrQueueTail), 1u));
                    queue[slot] = uint32_t(u);
                    __threadfence();
                    st_release_gpu(&ready[slot], flag_value);
                }
                red_add_release_gpu(header_word(a.err, kHdrRanked), 1u);
            }
        } else if (ready != nullptr && tid == 0) {
            __threadfence();
            st_release_gpu(&ready[u], flag_value);
        }
    }
    return flag_value;
}

// Arguments common to every select launch of a problem.
inline SelectArgs select_args_base(const Geometry& g, const WorkspaceLayout& L, char* ws, const void* q,
                                   const void* kmin, const void* kmax, const float* kmean)
{
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
    return a;
}

// Single-level selection: every block before the window is a candidate row.
inline void set_single_level(SelectArgs& a, const Geometry& g, const int32_t* reserve_ids,
                             int32_t* sel_ids, int32_t* sel_count)
{
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
}

// Chunk geometry of a launch over `units` units.
template <int KIND, bool MBF16, int D>
inline void set_chunking(SelectArgs& a, int units)
{
    using SS = SelectShape<KIND, MBF16, D>;
    a.chunks_per_group = (a.group_rows + SS::ROWS - 1) / SS::ROWS;
    a.chunks_per_unit = a.groups * a.chunks_per_group;
    a.total_chunks = units * a.chunks_per_unit;
}

// Chunk geometry of a warp-slab launch over `units` units.
template <int KIND, bool MBF16, int D>
inline void set_slab_chunking(SelectArgs& a, int units)
{
    constexpr int ROWS = SlabSelShape<KIND, MBF16, D>::ROWS;
    a.chunks_per_group = (a.group_rows + ROWS - 1) / ROWS;
    a.chunks_per_unit = a.groups * a.chunks_per_group;
    a.total_chunks = units * a.chunks_per_unit;
}

}  // namespace
}  // namespace sa
