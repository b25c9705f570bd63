// Device side of the bf16 decode (warp-independent slabs on tensor cores) and the unit
// merge, shared by the decode kernels and the fused step kernel.  The design notes are
// in sa_decode.cu.
#pragma once

#include "sa_common.cuh"
#include "sa_internal.h"

namespace sa {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kItemKBytes = 16 * 1024;     // K bytes per item (V the same)
constexpr int kMaxRangeBlocks = 1024;      // page lookups a CTA caches in shared memory
constexpr int kDecSmemLimit = 224 * 1024;  // dynamic shared memory a decode CTA may use

struct DecodeArgs {
    const void* q;
    int q_bf16;
    const void* k_pages;
    const void* v_pages;
    const int32_t* block_table;
    const int32_t* sel_ids;
    const int32_t* sel_count;
    float* out;
    int Hq, Hkv, nb, bs, N, num_pages, sel_stride;
    int bt_stride;           // block_table row length (capacity in blocks)
    // slot mode (slot_C > 0): K/V come from a per-unit slot pool [units * slot_C, bs, D]
    // through sel_slot [units, sel_stride] instead of block_table and the page pools
    const int32_t* sel_slot;
    int slot_C;
    int page_heads;          // KV heads per page: Hkv, or 1 in slot mode
    int blocks_per_item, items_per_unit, total_items, units;
    int stages;
    float scale_log2;
    float* part_m;   // [B*Hq, items_per_unit]
    float* part_l;
    float* part_o;   // [B*Hq, items_per_unit, D]
    uint32_t* counters;
    uint32_t* err;
};

// The CTA that completed unit u merges the unit's partials.  A unit's segments start
// at its first item and at every CTA range start inside it; each segment wrote one
// (m, l, o) partial at the slot of its first item, so segment i of a unit whose first
// item lies in CTA c0 sits at slot max(start(c0 + i), x0) - x0.  Segments are taken
// kMergeChunk at a time, and within a chunk every load is issued before any is used:
// each thread loads the o values of its outputs and a share of the (m, l) pairs, the
// pairs go through shared memory, and the outputs are combined against the running
// maximum (rescaled when a later chunk raises it).
constexpr int kMergeChunk = 8;
constexpr int kMergeOut = 4;                   // outputs per thread: G * D <= 4 * kDecThreads

__device__ void merge_unit(const DecodeArgs& a, int u, int G, int D)
{
    __shared__ float s_pm[8][kMergeChunk], s_pl[8][kMergeChunk];
    const int tid = threadIdx.x;
    const int b = u / a.Hkv, kvh = u - (u / a.Hkv) * a.Hkv;
    const size_t head0 = size_t(b) * a.Hq + size_t(kvh) * G;
    const int ipu = a.items_per_unit;
    const long long x0 = (long long)u * ipu, x1 = x0 + ipu;
    const long long T = a.total_items, C = gridDim.x;
    if (tid == 0) a.counters[u] = 0u;
    long long c0 = x0 * C / T;                                   // CTA holding item x0
    while (c0 + 1 < C && (T * (c0 + 1)) / C <= x0) ++c0;
    while (c0 > 0 && (T * c0) / C > x0) --c0;
    long long c1 = (x1 * C + T - 1) / T;                         // first CTA starting at or after x1
    while (c1 > c0 + 1 && (T * (c1 - 1)) / C >= x1) --c1;
    while (c1 < C && (T * c1) / C < x1) ++c1;
    const int nseg = int(c1 - c0);
    auto slot = [&](int i) -> int { return int(max((T * (c0 + i)) / C, x0) - x0); };

    float num[kMergeOut], den[kMergeOut], mrun[kMergeOut];
#pragma unroll
    for (int r = 0; r < kMergeOut; ++r) num[r] = den[r] = 0.f, mrun[r] = -INFINITY;
    for (int base = 0; base < nseg; base += kMergeChunk) {
        const int n = min(kMergeChunk, nseg - base);
        float ov[kMergeOut][kMergeChunk];
#pragma unroll
        for (int r = 0; r < kMergeOut; ++r) {
            const int i = tid + r * kDecThreads;
            const int g = i / D, d = i - (i / D) * D;
#pragma unroll
            for (int e = 0; e < kMergeChunk; ++e)
                ov[r][e] = (i < G * D && e < n) ? __ldcg(a.part_o + ((head0 + g) * ipu + slot(base + e)) * D + d) : 0.f;
        }
        if (tid < G * kMergeChunk) {
            const int g = tid / kMergeChunk, e = tid - g * kMergeChunk;
            float pm = -INFINITY, pl = 0.f;
            if (e < n) {
                pm = __ldcg(a.part_m + (head0 + g) * ipu + slot(base + e));
                pl = __ldcg(a.part_l + (head0 + g) * ipu + slot(base + e));
            }
            s_pm[g][e] = pm;
            s_pl[g][e] = pl;
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < kMergeOut; ++r) {
            const int i = tid + r * kDecThreads;
            if (i >= G * D) break;
            const int g = i / D;
            float mx = mrun[r];
#pragma unroll
            for (int e = 0; e < kMergeChunk; ++e) mx = fmaxf(mx, s_pm[g][e]);
            if (mx == -INFINITY) continue;                       // nothing valid yet
            const float resc = mrun[r] == -INFINITY ? 0.f : fast_exp2(mrun[r] - mx);
            float nu = num[r] * resc, de = den[r] * resc;
#pragma unroll
            for (int e = 0; e < kMergeChunk; ++e) {
                const float pm = s_pm[g][e];
                if (pm == -INFINITY) continue;                   // empty segment (or past n)
                const float w = fast_exp2(pm - mx);
                nu = fmaf(w, ov[r][e], nu);
                de = fmaf(w, s_pl[g][e], de);
            }
            num[r] = nu;
            den[r] = de;
            mrun[r] = mx;
        }
        __syncthreads();                                         // s_pm / s_pl reused
    }
#pragma unroll
    for (int r = 0; r < kMergeOut; ++r) {
        const int i = tid + r * kDecThreads;
        if (i >= G * D) break;
        a.out[head0 * D + i] = den[r] > 0.f ? num[r] / den[r] : 0.f;
    }
}

// ---------------------------------------------------------------------------
// bf16 K/V slabs (the job-based decode of sa_job_decode.cuh): warps stream 16-token
// slabs independently, contractions on tensor cores.
//   * Each warp runs its own ring of slabs in shared memory, filled with 16-byte
//     cp.async copies (global -> shared, L2 only) issued by its own lanes, so a warp
//     waits only on its own copies (cp.async.wait_group + __syncwarp).  Rows without a
//     token (empty block slots, the tail past the context) are zero-filled by the copy.
//   * Layout per slab: K then V, each token row split into 64-channel halves of
//     128-byte rows with the 16-byte chunk index XOR-ed with the row index mod 8, so
//     the 8-row ldmatrix reads are conflict-free.
//   * S = q K^T with mma.sync m16n8k16 (bf16 in, fp32 accumulate): A rows 0..7 are the
//     G query heads, columns the 8 tokens of a tile.  An fp32 query is split into
//     bf16 hi + lo; the lo part rides in A rows 8..15, so one MMA yields both halves
//     of the dot and the score is c0 + c2.
//   * Online softmax on the accumulator fragments: a head's row lives in the 4 lanes
//     of a quad, so the slab maximum takes two shuffles; the running sum stays per
//     lane until the segment ends.
//   * O += P V with the score fragments reused as the A operand (the C layout of two
//     8-token tiles is the A layout of one 16-token k-step).  P is carried as bf16
//     hi (rows 0..7) + lo (rows 8..15): the weights keep ~16 mantissa bits at the cost
//     of no extra MMA, and each output is c0 + c2 of its accumulator.
//   * At the end of a job every warp writes its (m, l, o) to the ring stage it has just
//     freed; the CTA combines the 8 into the job's partial.
constexpr int kSlabTokens = 16;
constexpr int kRowBytes = 128;   // one 64-channel half of a token row

template <int D>
struct SlabShape {
    static constexpr int HALVES = D / 64;
    static constexpr int HALF_BYTES = kSlabTokens * kRowBytes;       // 2 KB
    static constexpr int TENSOR_BYTES = HALVES * HALF_BYTES;        // K (or V) of a slab
    static constexpr int SLAB_BYTES = 2 * TENSOR_BYTES;             // 8 KB (D 128) / 4 KB (D 64)
    static constexpr int STAGES = D == 128 ? 3 : 6;                 // 192 KB of rings per CTA
    static constexpr int CPR = D / 8;                               // 16-byte chunks per token row
    static constexpr int RPI = 32 / CPR;                            // rows one warp copy covers
    static constexpr int CP_ITERS = kSlabTokens / RPI;
    static constexpr int DT = D / 8;                                // 8-channel tiles
    static_assert(8 * D * 4 <= SLAB_BYTES, "a warp's flushed G x D outputs must fit one stage");
};

__device__ __forceinline__ uint32_t swz(uint32_t half_base, int token, int chunk)
{
    return half_base + uint32_t(token) * kRowBytes + uint32_t((chunk ^ (token & 7)) << 4);
}

// Arguments of a decode launch (split-K partials and counters in the workspace).
inline DecodeArgs decode_args(const Geometry& g, const WorkspaceLayout& L, char* ws, const void* q,
                              const void* k_pages, const void* v_pages, const int32_t* block_table,
                              const int32_t* sel_ids, const int32_t* sel_count, float* out,
                              const int32_t* sel_slot, int slot_C)
{
    DecodeArgs a{};
    a.sel_slot = sel_slot;
    a.slot_C = slot_C;
    a.page_heads = slot_C > 0 ? 1 : g.Hkv;
    a.q = q;
    a.q_bf16 = g.q_bf16;
    a.k_pages = k_pages;
    a.v_pages = v_pages;
    a.block_table = block_table;
    a.sel_ids = sel_ids;
    a.sel_count = sel_count;
    a.out = out;
    a.Hq = g.Hq;
    a.Hkv = g.Hkv;
    a.nb = g.nb;
    a.bs = g.bs;
    a.N = g.N;
    a.num_pages = g.num_pages;
    a.bt_stride = g.nb_cap;
    a.sel_stride = g.sel_stride;
    a.blocks_per_item = L.blocks_per_split;
    a.items_per_unit = L.max_splits;
    a.units = g.units();
    a.total_items = g.units() * L.max_splits;
    a.scale_log2 = g.scale_log2;
    a.part_m = reinterpret_cast<float*>(ws + L.part_m);
    a.part_l = reinterpret_cast<float*>(ws + L.part_l);
    a.part_o = reinterpret_cast<float*>(ws + L.part_o);
    a.counters = reinterpret_cast<uint32_t*>(ws + L.dec_counters);
    a.err = reinterpret_cast<uint32_t*>(ws + L.err);
    return a;
}

}  // namespace
}  // namespace sa
