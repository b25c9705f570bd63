// Step-to-step diff and LRU slot cache ("SGLang分层稀疏注意力技术解析与优化实践" §3.2).
//
// The page describes: adjacent decode steps share 80-90% of their top-k; the GPU keeps
// a cache 2-4x the top-k with LRU eviction; per step (a) diff the current set against
// the previous one, (b) find what is already resident, (c) load the misses, (d) update
// the index.  The rules are sequential ("each miss in ascending id takes the lowest
// free slot, else evicts the least recently used block the step does not need"); they
// have a closed form that a warp evaluates in parallel:
//   * misses never free a slot, so miss i takes free_slot[i] while free slots last,
//   * then victim[i - n_free], where victims are the resident blocks not requested this
//     step sorted by (last_use, block id) -- requested blocks cannot become victims,
//     so later misses never see earlier placements as candidates.
// One warp per (sequence, KV head) unit; the unit's slot table lives in shared memory.
#include "sa_common.cuh"
#include "sa_internal.h"

namespace sa {
namespace {

constexpr int kDiffWarps = 4;

struct DiffArgs {
    const int32_t *sel_ids, *sel_count, *prev_ids, *prev_count;
    int32_t *slot_block, *slot_last_use;
    int32_t *hit_ids, *miss_ids, *miss_slot, *evict_ids, *evict_slot, *new_ids, *dropped_ids;
    int32_t* counts;
    uint32_t* err;
    int units, stride, C, nb, step;
    int32_t* sel_slot;   // optional [units, stride]: each selected block's slot after the step
};

__device__ __forceinline__ bool find_sorted(const int* a, int n, int x, int* pos)
{
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] < x) lo = mid + 1;
        else hi = mid;
    }
    *pos = lo;
    return lo < n && a[lo] == x;
}

// Ordered compaction: lanes holding `flag` append `value` to dst in lane/iteration order.
__device__ __forceinline__ int append_ordered(bool flag, int value, int* dst, int run, int lane)
{
    const uint32_t bal = __ballot_sync(kFullMask, flag);
    if (flag) dst[run + __popc(bal & lanemask_lt())] = value;
    return run + __popc(bal);
}

__global__ void __launch_bounds__(kDiffWarps * 32) diff_kernel(DiffArgs a)
{
    extern __shared__ int dsm[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int u = blockIdx.x * kDiffWarps + warp;
    if (u >= a.units) return;
    allow_dependents_early();
    grid_dependency_wait();   // inputs and slot state may come from the previous kernel
    const int W = a.stride, C = a.C;
    int* S = dsm + warp * (3 * W + 5 * C);
    int* P = S + W;
    int* hit_slot = P + W;       // slot holding S[i], or -1
    int* blk = hit_slot + W;     // slot -> block
    int* last = blk + C;         // slot -> last use
    int* is_hit = last + C;      // slot holds a requested block
    int* freel = is_hit + C;     // free slots, ascending
    int* victim = freel + C;     // eviction order

    int ns = a.sel_count[u], np = a.prev_count[u];
    bool bad = ns < 0 || ns > W || ns > C || np < 0 || np > W;
    if (bad) ns = np = 0;
    const size_t row = size_t(u) * W;
    for (int i = lane; i < ns; i += 32) S[i] = a.sel_ids[row + i];
    for (int i = lane; i < np; i += 32) P[i] = a.prev_ids[row + i];
    for (int s = lane; s < C; s += 32) {
        blk[s] = a.slot_block[size_t(u) * C + s];
        last[s] = a.slot_last_use[size_t(u) * C + s];
        is_hit[s] = 0;
    }
    for (int i = lane; i < ns; i += 32) hit_slot[i] = -1;
    __syncwarp();
    // validate: ids in range and strictly ascending; slot contents in [-1, nb)
    bool bad_ids = false, bad_slot = false;
    for (int i = lane; i < ns; i += 32)
        bad_ids |= S[i] < 0 || S[i] >= a.nb || (i > 0 && S[i - 1] >= S[i]);
    for (int i = lane; i < np; i += 32)
        bad_ids |= P[i] < 0 || P[i] >= a.nb || (i > 0 && P[i - 1] >= P[i]);
    for (int s = lane; s < C; s += 32) bad_slot |= blk[s] < -1 || blk[s] >= a.nb;
    bad_ids = __any_sync(kFullMask, bad_ids);
    bad_slot = __any_sync(kFullMask, bad_slot);
    int32_t* cnt = a.counts + size_t(u) * 5;
    if (bad || bad_ids || bad_slot) {
        if (lane == 0) {
            raise_error(a.err, bad ? SPARSE_ATTN_ERR_SEL_COUNT
                               : bad_ids ? SPARSE_ATTN_ERR_SEL_ID : SPARSE_ATTN_ERR_SLOT);
        }
        if (lane < 5) cnt[lane] = 0;
        return;   // state left untouched
    }

    // (a) diff against the previous step
    int n_new = 0, n_drop = 0;
    for (int base = 0; base < ns; base += 32) {
        const int i = base + lane;
        int pos;
        const bool f = i < ns && !find_sorted(P, np, S[i], &pos);
        n_new = append_ordered(f, i < ns ? S[i] : 0, a.new_ids + row, n_new, lane);
    }
    for (int base = 0; base < np; base += 32) {
        const int i = base + lane;
        int pos;
        const bool f = i < np && !find_sorted(S, ns, P[i], &pos);
        n_drop = append_ordered(f, i < np ? P[i] : 0, a.dropped_ids + row, n_drop, lane);
    }

    // (b) what is resident
    for (int s = lane; s < C; s += 32) {
        int pos;
        if (blk[s] >= 0 && find_sorted(S, ns, blk[s], &pos)) {
            hit_slot[pos] = s;
            is_hit[s] = 1;
        }
    }
    __syncwarp();
    int n_hit = 0, n_miss = 0, n_free = 0;
    for (int base = 0; base < ns; base += 32) {
        const int i = base + lane;
        const bool in = i < ns;
        const bool h = in && hit_slot[i] >= 0;
        n_hit = append_ordered(h, in ? S[i] : 0, a.hit_ids + row, n_hit, lane);
        n_miss = append_ordered(in && !h, in ? S[i] : 0, a.miss_ids + row, n_miss, lane);
    }
    for (int base = 0; base < C; base += 32) {
        const int s = base + lane;
        n_free = append_ordered(s < C && blk[s] < 0, s, freel, n_free, lane);
    }
    // (c) eviction order among resident, unrequested blocks: rank by (last use, id)
    const int need = n_miss > n_free ? n_miss - n_free : 0;
    for (int i = lane; i < need; i += 32) victim[i] = -1;
    __syncwarp();
    if (need > 0) {
        for (int s = lane; s < C; s += 32) {
            if (blk[s] < 0 || is_hit[s]) continue;
            int rank = 0;
            for (int t = 0; t < C; ++t) {
                if (blk[t] < 0 || is_hit[t]) continue;
                rank += (last[t] < last[s]) || (last[t] == last[s] && blk[t] < blk[s]);
            }
            if (rank < need) victim[rank] = s;
        }
    }
    __syncwarp();
    // A slot table holding one block twice leaves a rank unfilled: refuse it untouched.
    bool hole = false;
    for (int i = lane; i < need; i += 32) hole |= victim[i] < 0 || victim[i] >= C;
    if (__any_sync(kFullMask, hole)) {
        if (lane == 0) raise_error(a.err, SPARSE_ATTN_ERR_SLOT);
        if (lane < 5) cnt[lane] = 0;
        return;
    }
    // placements (misses are read back from the output list written above)
    const int32_t* misses = a.miss_ids + row;
    for (int i = lane; i < n_miss; i += 32) {
        const int slot = i < n_free ? freel[i] : victim[i - n_free];
        a.miss_slot[row + i] = slot;
        if (i >= n_free) {
            a.evict_ids[row + (i - n_free)] = blk[slot];
            a.evict_slot[row + (i - n_free)] = slot;
        }
    }
    __syncwarp();
    // (d) index update: place misses, stamp every requested block
    for (int i = lane; i < n_miss; i += 32) {
        const int slot = i < n_free ? freel[i] : victim[i - n_free];
        a.slot_block[size_t(u) * C + slot] = misses[i];
        a.slot_last_use[size_t(u) * C + slot] = a.step;
    }
    for (int i = lane; i < ns; i += 32)
        if (hit_slot[i] >= 0) a.slot_last_use[size_t(u) * C + hit_slot[i]] = a.step;
    if (a.sel_slot != nullptr) {
        // the slot map of the step: a hit keeps its slot; the r-th miss (selection order)
        // takes the r-th placement above
        int run = 0;
        for (int base = 0; base < ns; base += 32) {
            const int i = base + lane;
            const bool miss = i < ns && hit_slot[i] < 0;
            const uint32_t bal = __ballot_sync(kFullMask, miss);
            if (i < ns) {
                const int r = run + __popc(bal & lanemask_lt());
                a.sel_slot[row + i] = miss ? (r < n_free ? freel[r] : victim[r - n_free]) : hit_slot[i];
            }
            run += __popc(bal);
        }
    }
    if (lane == 0) {
        cnt[0] = n_hit;
        cnt[1] = n_miss;
        cnt[2] = n_miss > n_free ? n_miss - n_free : 0;
        cnt[3] = n_new;
        cnt[4] = n_drop;
    }
}

}  // namespace

cudaError_t launch_diff(const Geometry& g, int step, const int32_t* sel_ids,
                        const int32_t* sel_count, const int32_t* prev_ids,
                        const int32_t* prev_count, int cache_slots, int32_t* slot_block,
                        int32_t* slot_last_use, int32_t* hit_ids, int32_t* miss_ids,
                        int32_t* miss_slot, int32_t* evict_ids, int32_t* evict_slot,
                        int32_t* new_ids, int32_t* dropped_ids, int32_t* counts, uint32_t* err,
                        cudaStream_t s, int32_t* sel_slot)
{
    const int units = g.units();
    if (units == 0) return cudaSuccess;
    DiffArgs a{sel_ids, sel_count, prev_ids, prev_count, slot_block, slot_last_use,
               hit_ids, miss_ids, miss_slot, evict_ids, evict_slot, new_ids, dropped_ids,
               counts, err, units, g.sel_stride, cache_slots, g.nb, step, sel_slot};
    const size_t smem = size_t(kDiffWarps) * (3 * size_t(g.sel_stride) + 5 * size_t(cache_slots)) * sizeof(int);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(diff_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(smem));
        if (e != cudaSuccess) return e;
    }
    return launch_after_previous(diff_kernel, dim3(unsigned((units + kDiffWarps - 1) / kDiffWarps)),
                                 dim3(kDiffWarps * 32), smem, s, a);
}

}  // namespace sa
