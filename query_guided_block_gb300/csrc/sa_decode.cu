// Sparse decode attention over the selected blocks only.
//
// "从HiSparse到QSA的移植实战" §3.3: the attention kernel walks a compact array of selected
// block indices and never reads unselected KV; HBM bandwidth is the bound.  SparDA page
// (www.2kiu.com/news/4656707) §5.3: skip unselected pages inside the kernel rather than
// gathering them into a temporary buffer first.  The softmax is exact over the union of
// the selected tokens (SGLang page §1.2 "select-then-compute").
//
// Design: a persistent grid streams "items" (a few selected blocks, ~64 tokens, of one
// (sequence, KV head) unit) through a kStages-deep shared-memory pipeline.
//   * Items are numbered unit-major; CTA i owns an equal contiguous range, so it sees
//     one or two unit boundaries and no CTA ever waits on another.
//   * At start the CTA resolves, for its whole range, selected id -> page through the
//     page table into shared memory (bounds-checked), so the producer thread issues
//     copies without touching global memory.
//   * kStages items stay in flight: per item, 1-D bulk async copies (cp.async.bulk) of
//     each (page, KV head) K tile and V tile -- block_size x D contiguous -- complete
//     on the stage's `full` mbarrier; warps release the stage on its `empty` mbarrier.
//     Copies from one issuing thread complete one after another, so each item's copies
//     are issued by different warps.
//   * QK^T in fp32: a key row is covered by LPR lanes with one 16-byte shared load
//     each; the G heads' partial dots are summed across the row's lanes with the
//     transposed halving reduction.  Per head, warps keep the running max / sum of an
//     online softmax (exp2, scores pre-scaled by scale * log2 e); PV accumulates in
//     registers, rescaled when the max moves.
//   * At the end of its segment of a unit, the CTA reduces its accumulators across
//     warps and writes one (m, l, o) partial; the CTA that completes a unit's item
//     count merges the unit's partials (log-sum-exp) into fp32 outputs.
// GQA tiles are G x tokens: far too narrow for a tensor-core tile to pay (>= 64 rows),
// and the kernel is HBM-bound at ~2 FMA per byte, so the contraction stays on FMA units.

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
    int blocks_per_item, items_per_unit, total_items, units;
    int stages;
    float scale_log2;
    float* part_m;   // [B*Hq, items_per_unit]
    float* part_l;
    float* part_o;   // [B*Hq, items_per_unit, D]
    uint32_t* counters;
    uint32_t* err;
};

template <int D, bool BF16, int G>
struct DecodeShape {
    static constexpr int ESZ = BF16 ? 2 : 4;
    static constexpr int EPL = 16 / ESZ;
    static constexpr int LPR = D / EPL;
    static constexpr int RPW = 32 / LPR;
    static constexpr int ROW_BYTES = D * ESZ;
    static constexpr int ITEM_TOKENS = kItemKBytes / ROW_BYTES;       // at block_size <= this
    static constexpr int R0 = 16 / G;
    static constexpr int R1 = ITEM_TOKENS / (kDecWarps * RPW);
    static constexpr int R = R0 < R1 ? R0 : R1;                      // rows per lane group
    static constexpr int V = R * G;                                  // partial dots per lane
    static constexpr int ROWS_PER_BATCH = kDecWarps * RPW * R;
    static_assert(ITEM_TOKENS % ROWS_PER_BATCH == 0, "item must split evenly over the warps");
    // the cross-warp reduction at a segment end reuses the item's stage buffer
    static_assert(kDecWarps * G * D * 4 <= 2 * ITEM_TOKENS * ROW_BYTES, "reduction must fit a stage");
};

size_t decode_fixed_smem(int G, int item_tokens)
{
    return size_t(2) * G * item_tokens * sizeof(float) + size_t(2) * kMaxRangeBlocks * sizeof(int);
}

// The CTA that completed unit u merges the unit's partials.  A unit's segments start
// at its first item and at every CTA range start inside it; each segment wrote one
// (m, l, o) partial at the slot of its first item.
__device__ void merge_unit(const DecodeArgs& a, int u, int G, int D)
{
    if (threadIdx.x == 0) a.counters[u] = 0u;
    const int b = u / a.Hkv, kvh = u - (u / a.Hkv) * a.Hkv;
    const size_t head0 = size_t(b) * a.Hq + size_t(kvh) * G;
    const int ipu = a.items_per_unit;
    const int x0 = u * ipu, x1 = x0 + ipu;
    const long long T = a.total_items, C = gridDim.x;
    int c0 = int((long long)x0 * C / T);                         // CTA holding item x0
    while (c0 + 1 < C && (T * (c0 + 1)) / C <= x0) ++c0;
    while (c0 > 0 && (T * c0) / C > x0) --c0;
    for (int i = threadIdx.x; i < G * D; i += kDecThreads) {
        const int g = i / D, d = i - g * D;
        const size_t h = head0 + g;
        float mx = -INFINITY;
        for (long long c = c0; c < C && (T * c) / C < x1; ++c) {
            const int slot = int(max((T * c) / C, (long long)x0) - x0);
            mx = fmaxf(mx, __ldcg(a.part_m + h * ipu + slot));
        }
        float num = 0.f, den = 0.f;
        if (mx != -INFINITY) {
            for (long long c = c0; c < C && (T * c) / C < x1; ++c) {
                const int slot = int(max((T * c) / C, (long long)x0) - x0);
                const float ms = __ldcg(a.part_m + h * ipu + slot);
                if (ms == -INFINITY) continue;
                const float wgt = fast_exp2(ms - mx);
                den = fmaf(wgt, __ldcg(a.part_l + h * ipu + slot), den);
                num = fmaf(wgt, __ldcg(a.part_o + (h * ipu + slot) * D + d), num);
            }
        }
        a.out[h * D + d] = den > 0.f ? num / den : 0.f;
    }
}

template <int D, bool BF16, int G>
__global__ void __launch_bounds__(kDecThreads, 2) decode_kernel(DecodeArgs a)
{
    using S = DecodeShape<D, BF16, G>;
    constexpr int EPL = S::EPL, LPR = S::LPR, RPW = S::RPW, R = S::R, V = S::V;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sub = lane % LPR, rsub = lane / LPR;
    const int bpi = a.blocks_per_item;
    const int item_tokens = bpi * a.bs;
    const uint32_t tile_bytes = uint32_t(a.bs) * S::ROW_BYTES;
    const size_t stage_bytes = size_t(2) * item_tokens * S::ROW_BYTES;

    extern __shared__ __align__(128) unsigned char smem[];
    float* s_s = reinterpret_cast<float*>(smem + a.stages * stage_bytes);   // [G][item_tokens]
    float* p_s = s_s + G * item_tokens;                                     // [item_tokens][G]
    int* blk_page = reinterpret_cast<int*>(p_s + G * item_tokens);          // [range blocks]
    int* blk_valid = blk_page + kMaxRangeBlocks;
    __shared__ __align__(8) uint64_t full[4], empty[4];
    __shared__ float s_alpha[G], s_m[G], s_l[G];
    __shared__ int s_counts[64];
    __shared__ int s_merge_unit;

    const int i_begin = int((long long)a.total_items * blockIdx.x / gridDim.x);
    const int i_end = int((long long)a.total_items * (blockIdx.x + 1) / gridDim.x);
    if (i_begin >= i_end) return;
    const int u_lo = i_begin / a.items_per_unit;
    const int u_hi = (i_end - 1) / a.items_per_unit;

    // ---- resolve the range: counts, selected ids -> pages ---------------------
    for (int u = u_lo + tid; u <= u_hi; u += kDecThreads) {
        int count = a.sel_count[u];
        if (count < 0 || count > a.sel_stride) {
            raise_error(a.err, SPARSE_ATTN_ERR_SEL_COUNT);
            count = count < 0 ? 0 : a.sel_stride;
        }
        s_counts[u - u_lo] = count;
    }
    __syncthreads();
    const int n_range_blocks = (i_end - i_begin) * bpi;
    for (int e = tid; e < n_range_blocks; e += kDecThreads) {
        const int item = i_begin + e / bpi;
        const int u = item / a.items_per_unit;
        const int slot = (item - u * a.items_per_unit) * bpi + e % bpi;
        int page = -1, valid = 0;
        if (slot < s_counts[u - u_lo]) {
            const int j = a.sel_ids[size_t(u) * a.sel_stride + slot];
            if (j < 0 || j >= a.nb) {
                raise_error(a.err, SPARSE_ATTN_ERR_SEL_ID);
            } else {
                const int b = u / a.Hkv;
                const int p = a.block_table[size_t(b) * a.nb + j];
                if (p < 0 || p >= a.num_pages) {
                    raise_error(a.err, SPARSE_ATTN_ERR_PAGE);
                } else {
                    page = p;
                    valid = min(a.bs, a.N - j * a.bs);
                }
            }
        }
        blk_page[e] = page;
        blk_valid[e] = valid;
    }
    if (tid == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kDecWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    const char* kbase = reinterpret_cast<const char*>(a.k_pages);
    const char* vbase = reinterpret_cast<const char*>(a.v_pages);
    // Copies issued by one thread complete one after another, so an item's 2 * bpi
    // copies (K and V tile of each block) are spread over the warps: copy i of the item
    // in stage s is issued by warp (s * 2 bpi + i) mod 8; the owner of copy 0 also posts
    // the stage's expected byte count.
    auto issue_mine = [&](int item) {   // every warp's lane 0
        const int k = item - i_begin;
        const int s = k % a.stages;
        unsigned char* kd = smem + s * stage_bytes;
        unsigned char* vd = kd + size_t(item_tokens) * S::ROW_BYTES;
        const int u = item / a.items_per_unit;
        const size_t head_off = size_t(u % a.Hkv) * tile_bytes;
        const size_t page_stride = size_t(a.Hkv) * tile_bytes;
        for (int i = 0; i < 2 * bpi; ++i) {
            if ((s * 2 * bpi + i) % kDecWarps != warp) continue;
            if (i == 0) {
                uint32_t nbytes = 0;
                for (int j = 0; j < bpi; ++j) nbytes += blk_page[k * bpi + j] >= 0 ? tile_bytes : 0u;
                mbar_arrive_expect_tx(&full[s], 2 * nbytes);
            }
            const int j = i >> 1;
            const int page = blk_page[k * bpi + j];
            if (page < 0) continue;
            if ((i & 1) == 0)
                bulk_copy_g2s(kd + size_t(j) * tile_bytes, kbase + page * page_stride + head_off, tile_bytes, &full[s]);
            else
                bulk_copy_g2s(vd + size_t(j) * tile_bytes, vbase + page * page_stride + head_off, tile_bytes, &full[s]);
        }
    };
    if (lane == 0)
        for (int item = i_begin; item < i_end && item < i_begin + a.stages; ++item) issue_mine(item);

    // running state of the current unit segment
    float qr[G][EPL];
    float acc[G][EPL];
    float m_run = -INFINITY, l_run = 0.f;      // per head, kept by warp g (replicated in its lanes)
    int cur_u = -1, seg_first = 0;

    for (int item = i_begin; item < i_end; ++item) {
        const int k = item - i_begin;
        const int s = k % a.stages;
        const uint32_t parity = uint32_t(k / a.stages) & 1u;
        const int u = item / a.items_per_unit;
        if (u != cur_u) {
            cur_u = u;
            seg_first = item;
            const int b = u / a.Hkv, kvh = u - (u / a.Hkv) * a.Hkv;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const size_t qrow = (size_t(b) * a.Hq + size_t(kvh) * G + g) * D + sub * EPL;
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    qr[g][e] = load_q(a.q, qrow + e, a.q_bf16 != 0) * a.scale_log2;
                    acc[g][e] = 0.f;
                }
            }
            m_run = -INFINITY;
            l_run = 0.f;
        }
        const unsigned char* ks = smem + s * stage_bytes;
        const unsigned char* vs = ks + size_t(item_tokens) * S::ROW_BYTES;
        if (!mbar_wait_bounded(&full[s], parity, kWaitCycles)) raise_error(a.err, SPARSE_ATTN_ERR_TIMEOUT);

        // ---- S = q K^T over the item's tokens -------------------------------
        for (int t_base = 0; t_base < item_tokens; t_base += S::ROWS_PER_BATCH) {
            const int t0 = t_base + ((warp * RPW) + rsub) * R;
            float v[V];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float kf[EPL];
                unpack16<BF16>(*reinterpret_cast<const uint4*>(ks + size_t(t0 + r) * S::ROW_BYTES + sub * 16), kf);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float d = 0.f;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) d = fmaf(qr[g][e], kf[e], d);
                    v[r * G + g] = d;
                }
            }
            group_reduce_transposed<V, LPR>(v, lane);
            constexpr int OUT = V >= LPR ? V / LPR : 1;
            constexpr int SPREAD = V >= LPR ? 1 : LPR / V;
            if (sub % SPREAD == 0) {
#pragma unroll
                for (int i = 0; i < OUT; ++i) {
                    const int idx = V >= LPR ? sub * (V / LPR) + i : sub / SPREAD;
                    const int r = idx / G, g = idx - (idx / G) * G;
                    const int t = t0 + r;
                    const int blk = t / a.bs;
                    const bool ok = (t - blk * a.bs) < blk_valid[k * bpi + blk];
                    s_s[g * item_tokens + t] = ok ? v[i] : -INFINITY;
                }
            }
        }
        __syncthreads();

        // ---- online softmax statistics: warp g owns head g ---------------------
        if (warp < G) {
            const int g = warp;
            float mi = -INFINITY;
            for (int t = lane; t < item_tokens; t += 32) mi = fmaxf(mi, s_s[g * item_tokens + t]);
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) mi = fmaxf(mi, __shfl_xor_sync(kFullMask, mi, off));
            const float m_new = fmaxf(m_run, mi);
            const float alpha = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - m_new);
            float li = 0.f;
            for (int t = lane; t < item_tokens; t += 32) {
                const float x = s_s[g * item_tokens + t];
                const float p = (x == -INFINITY) ? 0.f : fast_exp2(x - m_new);
                p_s[t * G + g] = p;
                li += p;
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) li += __shfl_xor_sync(kFullMask, li, off);
            l_run = l_run * alpha + li;
            m_run = m_new;
            if (lane == 0) s_alpha[g] = alpha;
        }
        __syncthreads();

        // ---- O += P V ----------------------------------------------------------
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float al = s_alpha[g];
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[g][e] *= al;
        }
        for (int t = warp * RPW + rsub; t < item_tokens; t += kDecWarps * RPW) {
            const int blk = t / a.bs;
            if ((t - blk * a.bs) >= blk_valid[k * bpi + blk]) continue;
            float vf[EPL];
            unpack16<BF16>(*reinterpret_cast<const uint4*>(vs + size_t(t) * S::ROW_BYTES + sub * 16), vf);
            float p[G];
            if constexpr (G % 4 == 0) {
#pragma unroll
                for (int g = 0; g < G; g += 4) {
                    const float4 pv = *reinterpret_cast<const float4*>(p_s + t * G + g);
                    p[g] = pv.x; p[g + 1] = pv.y; p[g + 2] = pv.z; p[g + 3] = pv.w;
                }
            } else {
#pragma unroll
                for (int g = 0; g < G; ++g) p[g] = p_s[t * G + g];
            }
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc[g][e] = fmaf(p[g], vf[e], acc[g][e]);
        }
        const bool seg_end = item + 1 == i_end || (item + 1) / a.items_per_unit != u;
        if (seg_end) {
            // ---- end of this CTA's segment of unit u: one partial ---------------
#pragma unroll
            for (int m = LPR; m < 32; m <<= 1)
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int e = 0; e < EPL; ++e) acc[g][e] += __shfl_xor_sync(kFullMask, acc[g][e], m);
            __syncthreads();   // every warp is done with this stage: reduce through it
            float* red = reinterpret_cast<float*>(smem + s * stage_bytes);   // [warps][G][D]
            if (rsub == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int e = 0; e < EPL; ++e) red[(warp * G + g) * D + sub * EPL + e] = acc[g][e];
            }
            if (warp < G && lane == 0) { s_m[warp] = m_run; s_l[warp] = l_run; }
            __syncthreads();
            const int b = u / a.Hkv, kvh = u - (u / a.Hkv) * a.Hkv;
            const size_t head0 = size_t(b) * a.Hq + size_t(kvh) * G;
            const int slot = seg_first - u * a.items_per_unit;
            const int ipu = a.items_per_unit;
            for (int i = tid; i < G * D; i += kDecThreads) {
                const int g = i / D, d = i - g * D;
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < kDecWarps; ++w) sum += red[(w * G + g) * D + d];
                a.part_o[((head0 + g) * ipu + slot) * D + d] = sum;
            }
            // the segment's partial lives at the slot of its first item
            if (tid < G) {
                a.part_m[(head0 + tid) * ipu + slot] = s_m[tid];
                a.part_l[(head0 + tid) * ipu + slot] = s_l[tid];
            }
            __syncthreads();   // the stage buffer is free again
            if (tid == 0) {
                const uint32_t n = uint32_t(item - seg_first + 1);
                const uint32_t before = atomic_add_acq_rel_u32(&a.counters[u], n);
                s_merge_unit = before + n == uint32_t(ipu) ? u : -1;
            }
        }
        // release the stage; its issuing warps refill it with the item kStages ahead
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&empty[s]);
            const int nxt = item + a.stages;
            bool mine = false;
            for (int i = 0; i < 2 * bpi; ++i) mine |= (s * 2 * bpi + i) % kDecWarps == warp;
            if (nxt < i_end && mine) {
                if (!mbar_wait_bounded(&empty[s], parity, kWaitCycles)) raise_error(a.err, SPARSE_ATTN_ERR_TIMEOUT);
                issue_mine(nxt);
            }
        }
        if (!seg_end) continue;
        __syncthreads();
        if (s_merge_unit < 0) continue;

        merge_unit(a, u, G, D);
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// bf16 K/V: the same persistent item pipeline, with the GQA contractions on tensor
// cores.  Staging: every thread issues 16-byte cp.async copies (global -> shared,
// L2 only) of its share of the item's K and V rows into a 128-byte-swizzled layout --
// each token row split into 64-channel halves of 128-byte rows, the 16-byte chunk index
// XOR-ed with the row index mod 8 -- so the 8-row ldmatrix accesses below are
// conflict-free.  Rows that carry no token (empty block slots, the tail past the
// context) are zero-filled by the copy itself.  Per-thread copies never stall the
// issuing warp the way a bulk copy issued per page tile did (measured: ~0.8 us per issue
// with 4-8 KB page tiles).  kDecStages - 1 items stay in flight.
//   S = Q K^T : mma.sync m16n8k16, rows = the G query heads (padded to 16),
//               columns = 8 tokens per tile, warps split the item's tokens;
//   O += P V  : rows = heads, columns = 8 channels per tile, k = 16 tokens,
//               warps split the head dimension, so no cross-warp reduction;
//               P enters as a bf16 hi + lo pair (two MMAs), so the weights keep
//               ~16 mantissa bits; accumulation is fp32 throughout.
// A bf16 query is exact in the MMA; an fp32 query is split into hi + lo too.
constexpr int kRowBytes = 128;   // one 64-channel half of a token row
constexpr int kDecStages = 3;

__device__ __forceinline__ uint32_t swz(uint32_t half_base, int token, int chunk)
{
    // 128-byte swizzle: the 16-byte chunk index is XOR-ed with the row index mod 8
    return half_base + uint32_t(token) * kRowBytes + uint32_t((chunk ^ (token & 7)) << 4);
}

template <int D, int G, bool QSPLIT>
__global__ void __launch_bounds__(kDecThreads, 2) decode_mma_kernel(DecodeArgs a)
{
    constexpr int HALVES = D / 64;
    constexpr int DT = D / 8;                      // 8-channel tiles
    constexpr int DT_PER_WARP = DT / kDecWarps;    // 2 (D = 128) or 1 (D = 64)
    constexpr int CPR = D / 8;                     // 16-byte chunks per token row
    static_assert(DT % kDecWarps == 0, "channel tiles must split over the warps");
    static_assert(G <= 8, "query rows live in the first 8 MMA rows");

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g4 = lane >> 2, t4 = lane & 3;       // MMA fragment coordinates
    const int bpi = a.blocks_per_item;
    const int item_tokens = bpi * a.bs;
    const uint32_t half_bytes = uint32_t(item_tokens) * kRowBytes;
    const uint32_t stage_bytes = 2u * HALVES * half_bytes;
    const int p_pitch = item_tokens + 8;           // bf16 elements per P row (bank spread)

    extern __shared__ __align__(128) unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // swizzle pattern repeats every 1024 bytes
    unsigned char* smem = smem_raw + (base - raw);
    uint16_t* p_s = reinterpret_cast<uint16_t*>(smem + kDecStages * stage_bytes);   // [2][G][p_pitch]
    int* blk_page = reinterpret_cast<int*>(p_s + 2 * G * p_pitch + 8);         // [range blocks]
    int* blk_valid = blk_page + kMaxRangeBlocks;
    __shared__ float red_m[kDecWarps][8], red_l[kDecWarps][8];   // per-warp max / sum per head
    __shared__ int s_counts[64];
    __shared__ int s_merge_unit;

    const int i_begin = int((long long)a.total_items * blockIdx.x / gridDim.x);
    const int i_end = int((long long)a.total_items * (blockIdx.x + 1) / gridDim.x);
    if (i_begin >= i_end) return;
    const int u_lo = i_begin / a.items_per_unit;
    const int u_hi = (i_end - 1) / a.items_per_unit;

    // ---- resolve the range: counts, selected ids -> pages ---------------------
    for (int u = u_lo + tid; u <= u_hi; u += kDecThreads) {
        int count = a.sel_count[u];
        if (count < 0 || count > a.sel_stride) {
            raise_error(a.err, SPARSE_ATTN_ERR_SEL_COUNT);
            count = count < 0 ? 0 : a.sel_stride;
        }
        s_counts[u - u_lo] = count;
    }
    __syncthreads();
    const int n_range_blocks = (i_end - i_begin) * bpi;
    for (int e = tid; e < n_range_blocks; e += kDecThreads) {
        const int item = i_begin + e / bpi;
        const int u = item / a.items_per_unit;
        const int slot = (item - u * a.items_per_unit) * bpi + e % bpi;
        int page = -1, valid = 0;
        if (slot < s_counts[u - u_lo]) {
            const int j = a.sel_ids[size_t(u) * a.sel_stride + slot];
            if (j < 0 || j >= a.nb) {
                raise_error(a.err, SPARSE_ATTN_ERR_SEL_ID);
            } else {
                const int p = a.block_table[size_t(u / a.Hkv) * a.nb + j];
                if (p < 0 || p >= a.num_pages) {
                    raise_error(a.err, SPARSE_ATTN_ERR_PAGE);
                } else {
                    page = p;
                    valid = min(a.bs, a.N - j * a.bs);
                }
            }
        }
        blk_page[e] = page;
        blk_valid[e] = valid;
    }
    __syncthreads();

    // Stage an item: K then V rows of its tokens, 16-byte chunks.  Thread tid always
    // copies chunk c = tid % CPR of tokens tid / CPR + i * (256 / CPR); the swizzle term
    // (c ^ token) & 7 is therefore constant per thread.
    const char* kbase = reinterpret_cast<const char*>(a.k_pages);
    const char* vbase = reinterpret_cast<const char*>(a.v_pages);
    constexpr int TSTEP = kDecThreads / CPR;
    const int cp_c = tid % CPR, cp_t0 = tid / CPR;
    const int bs_shift = __ffs(a.bs) - 1;
    const uint32_t cp_dst0 = (cp_c >> 3) * half_bytes + uint32_t(cp_t0) * kRowBytes +
                             uint32_t(((cp_c & 7) ^ (cp_t0 & 7)) << 4);
    const int n_per_tensor = item_tokens / TSTEP;
    auto issue_item = [&](int item) {   // every thread
        const int k = item - i_begin;
        const uint32_t kd = base + (k % kDecStages) * stage_bytes + cp_dst0;
        const uint32_t vd = kd + HALVES * half_bytes;
        const size_t head_rows = size_t((item / a.items_per_unit) % a.Hkv) * a.bs;
        for (int i = 0; i < n_per_tensor; ++i) {
            const int t = cp_t0 + i * TSTEP;
            const int j = t >> bs_shift, r = t & (a.bs - 1);
            const int page = blk_page[k * bpi + j];
            const bool ok = page >= 0 && r < blk_valid[k * bpi + j];
            const size_t off = ok ? ((size_t(page) * a.Hkv * a.bs + head_rows + r) * (D * 2) + cp_c * 16) : 0;
            const uint32_t bytes = ok ? 16u : 0u;
            cp_async_16_zfill(kd + uint32_t(i * TSTEP) * kRowBytes, kbase + off, bytes);
            cp_async_16_zfill(vd + uint32_t(i * TSTEP) * kRowBytes, vbase + off, bytes);
        }
    };
    for (int kk = 0; kk < kDecStages - 1; ++kk) {
        if (i_begin + kk < i_end) issue_item(i_begin + kk);
        cp_async_commit();
    }

    // query A-fragments (rows g4 < G), per 16-channel k-step: a0 = (g4, 2t4..), a2 = (g4, 2t4+8..)
    uint32_t qa0[D / 16], qa2[D / 16];                       // bf16 (hi) part
    uint32_t qb0[QSPLIT ? D / 16 : 1], qb2[QSPLIT ? D / 16 : 1];  // lo part (fp32 query)
    float acc[DT_PER_WARP][4];
    float m_run = -INFINITY, l_run = 0.f;   // head g4's running statistics (all warps agree)
    int cur_u = -1, seg_first = 0;

    for (int item = i_begin; item < i_end; ++item) {
        const int k = item - i_begin;
        const int s = k % kDecStages;
        const int u = item / a.items_per_unit;
        if (u != cur_u) {
            cur_u = u;
            seg_first = item;
            const int b = u / a.Hkv, kvh = u - (u / a.Hkv) * a.Hkv;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                float f[4] = {0.f, 0.f, 0.f, 0.f};
                if (g4 < G) {
                    const size_t qrow = (size_t(b) * a.Hq + size_t(kvh) * G + g4) * D + ks * 16 + 2 * t4;
                    f[0] = load_q(a.q, qrow, a.q_bf16 != 0);
                    f[1] = load_q(a.q, qrow + 1, a.q_bf16 != 0);
                    f[2] = load_q(a.q, qrow + 8, a.q_bf16 != 0);
                    f[3] = load_q(a.q, qrow + 9, a.q_bf16 != 0);
                }
                qa0[ks] = pack_bf16x2(f[0], f[1]);
                qa2[ks] = pack_bf16x2(f[2], f[3]);
                if constexpr (QSPLIT) {   // remainder after bf16 rounding
                    qb0[ks] = pack_bf16x2(f[0] - bf16_lo(qa0[ks]), f[1] - bf16_hi(qa0[ks]));
                    qb2[ks] = pack_bf16x2(f[2] - bf16_lo(qa2[ks]), f[3] - bf16_hi(qa2[ks]));
                }
            }
#pragma unroll
            for (int j = 0; j < DT_PER_WARP; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
            m_run = -INFINITY;
            l_run = 0.f;
        }
        const uint32_t ks_base = base + s * stage_bytes;
        const uint32_t vs_base = ks_base + HALVES * half_bytes;
        // this item's copies (this thread's) are done; after the barrier everyone's are,
        // and every thread has finished the previous item, whose stage is refilled now
        cp_async_wait_group<kDecStages - 2>();
        __syncthreads();
        if (item + kDecStages - 1 < i_end) issue_item(item + kDecStages - 1);
        cp_async_commit();

        // ---- S = q K^T: warp w takes token tiles w, w + 8, ...; softmax on the fragments
        constexpr int NT_MAX = 4;                  // token tiles per warp (item <= 256 tokens)
        const int nt_per_warp = item_tokens / (8 * kDecWarps);
        float sv[NT_MAX][2];
        float wmax = -INFINITY;
#pragma unroll
        for (int q = 0; q < NT_MAX; ++q) {
            sv[q][0] = sv[q][1] = -INFINITY;
            if (q >= nt_per_warp) continue;
            const int n0 = (warp + q * kDecWarps) * 8;
            float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kp = 0; kp < D / 32; ++kp) {   // two 16-channel k-steps per ldmatrix.x4
                const int ch = kp * 4 + (lane >> 3);       // 8-channel chunk of this lane's matrix
                const uint32_t addr = swz(ks_base + (ch >> 3) * half_bytes, n0 + (lane & 7), ch & 7);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(addr, b0, b1, b2, b3);
                mma_bf16_16816(c, qa0[2 * kp], 0u, qa2[2 * kp], 0u, b0, b1);
                mma_bf16_16816(c, qa0[2 * kp + 1], 0u, qa2[2 * kp + 1], 0u, b2, b3);
                if constexpr (QSPLIT) {
                    mma_bf16_16816(c, qb0[2 * kp], 0u, qb2[2 * kp], 0u, b0, b1);
                    mma_bf16_16816(c, qb0[2 * kp + 1], 0u, qb2[2 * kp + 1], 0u, b2, b3);
                }
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = n0 + 2 * t4 + e;
                const int j = t >> bs_shift;
                const bool ok = (t & (a.bs - 1)) < blk_valid[k * bpi + j];
                sv[q][e] = ok ? c[e] * a.scale_log2 : -INFINITY;
                wmax = fmaxf(wmax, sv[q][e]);
            }
        }
        // per-head max over the warp's tokens (the 4 lanes of a fragment row), then the CTA
        wmax = fmaxf(wmax, __shfl_xor_sync(kFullMask, wmax, 1));
        wmax = fmaxf(wmax, __shfl_xor_sync(kFullMask, wmax, 2));
        if (t4 == 0) red_m[warp][g4] = wmax;
        __syncthreads();
        float alpha = 0.f;
        {
            float mi = -INFINITY;
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) mi = fmaxf(mi, red_m[w][g4]);
            const float m_new = fmaxf(m_run, mi);
            alpha = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - m_new);
            float wsum = 0.f;
            if (g4 < G) {
#pragma unroll
                for (int q = 0; q < NT_MAX; ++q) {
                    if (q >= nt_per_warp) continue;
                    const int t = (warp + q * kDecWarps) * 8 + 2 * t4;
                    float p[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        p[e] = (sv[q][e] == -INFINITY) ? 0.f : fast_exp2(sv[q][e] - m_new);
                        wsum += p[e];
                    }
                    const uint32_t hi = pack_bf16x2(p[0], p[1]);
                    const uint32_t lo = pack_bf16x2(p[0] - bf16_lo(hi), p[1] - bf16_hi(hi));
                    *reinterpret_cast<uint32_t*>(p_s + g4 * p_pitch + t) = hi;
                    *reinterpret_cast<uint32_t*>(p_s + (G + g4) * p_pitch + t) = lo;
                }
            }
            wsum += __shfl_xor_sync(kFullMask, wsum, 1);
            wsum += __shfl_xor_sync(kFullMask, wsum, 2);
            if (t4 == 0) red_l[warp][g4] = wsum;
            m_run = m_new;
        }
        __syncthreads();
        {
            float li = 0.f;
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) li += red_l[w][g4];
            l_run = l_run * alpha + li;
        }

        // ---- O += P V: warp w owns channel tiles w * DT_PER_WARP .. ---------------
        {
            const float al = g4 < G ? alpha : 0.f;
#pragma unroll
            for (int j = 0; j < DT_PER_WARP; ++j) {
                acc[j][0] *= al;
                acc[j][1] *= al;
            }
            const uint32_t* p32 = reinterpret_cast<const uint32_t*>(p_s);
            for (int kk = 0; kk < item_tokens / 16; ++kk) {
                const int k0 = kk * 16;
                uint32_t ah0 = 0, ah2 = 0, al0 = 0, al2 = 0;
                if (g4 < G) {
                    ah0 = p32[(g4 * p_pitch + k0 + 2 * t4) >> 1];
                    ah2 = p32[(g4 * p_pitch + k0 + 8 + 2 * t4) >> 1];
                    al0 = p32[((G + g4) * p_pitch + k0 + 2 * t4) >> 1];
                    al2 = p32[((G + g4) * p_pitch + k0 + 8 + 2 * t4) >> 1];
                }
#pragma unroll
                for (int jp = 0; jp < DT_PER_WARP; jp += 2) {
                    // matrices: (tokens k0.., ch c), (tokens k0+8.., ch c), (k0.., c+1), (k0+8.., c+1)
                    const int mtx = lane >> 3;
                    const int tok = k0 + (mtx & 1) * 8 + (lane & 7);
                    const int chunk = (warp * DT_PER_WARP + jp) + (mtx >> 1);
                    const uint32_t addr = swz(vs_base + (chunk >> 3) * half_bytes, tok, chunk & 7);
                    uint32_t r0, r1, r2 = 0, r3 = 0;
                    if constexpr (DT_PER_WARP >= 2) ldsm_x4_trans(addr, r0, r1, r2, r3);
                    else ldsm_x2_trans(addr, r0, r1);   // lanes 0..15 address the two matrices
                    mma_bf16_16816(acc[jp], ah0, 0u, ah2, 0u, r0, r1);
                    mma_bf16_16816(acc[jp], al0, 0u, al2, 0u, r0, r1);
                    if constexpr (DT_PER_WARP >= 2) {
                        mma_bf16_16816(acc[jp + 1], ah0, 0u, ah2, 0u, r2, r3);
                        mma_bf16_16816(acc[jp + 1], al0, 0u, al2, 0u, r2, r3);
                    }
                }
            }
        }

        const bool seg_end = item + 1 == i_end || (item + 1) / a.items_per_unit != u;
        if (seg_end) {
            // ---- end of this CTA's segment of unit u: one partial (no reduction) --
            const int b = u / a.Hkv, kvh = u - (u / a.Hkv) * a.Hkv;
            const size_t head0 = size_t(b) * a.Hq + size_t(kvh) * G;
            const int slot = seg_first - u * a.items_per_unit;
            const int ipu = a.items_per_unit;
            if (g4 < G) {
#pragma unroll
                for (int j = 0; j < DT_PER_WARP; ++j) {
                    const int ch = (warp * DT_PER_WARP + j) * 8 + 2 * t4;
                    float* dst = a.part_o + ((head0 + g4) * ipu + slot) * D + ch;
                    *reinterpret_cast<float2*>(dst) = make_float2(acc[j][0], acc[j][1]);
                }
            }
            if (warp == 0 && t4 == 0 && g4 < G) {
                a.part_m[(head0 + g4) * ipu + slot] = m_run;
                a.part_l[(head0 + g4) * ipu + slot] = l_run;
            }
            __syncthreads();
            if (tid == 0) {
                const uint32_t n = uint32_t(item - seg_first + 1);
                const uint32_t before = atomic_add_acq_rel_u32(&a.counters[u], n);
                s_merge_unit = before + n == uint32_t(ipu) ? u : -1;
            }
        }
        if (!seg_end) continue;
        __syncthreads();
        if (s_merge_unit < 0) continue;
        merge_unit(a, u, G, D);
        __syncthreads();
    }
    cp_async_wait_group<0>();
}

template <int D, bool BF16, int G>
cudaError_t launch_decode_t(DecodeArgs a, cudaStream_t s)
{
    using S = DecodeShape<D, BF16, G>;
    const int item_tokens = a.blocks_per_item * a.bs;
    const size_t stage = size_t(2) * item_tokens * S::ROW_BYTES;
    const size_t fixed = decode_fixed_smem(G, item_tokens);
    a.stages = (2 * (3 * stage + fixed + 1024) <= size_t(kSmemPerSm)) ? 3 : 2;
    const size_t smem = a.stages * stage + fixed;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, BF16, G>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmemLimit);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int per_sm = (2 * (smem + 1024) <= size_t(kSmemPerSm)) ? 2 : 1;
    long long ctas = (long long)num_sms() * per_sm;
    // every CTA's range must fit its shared-memory page cache
    const long long min_ctas = ((long long)a.total_items * a.blocks_per_item + kMaxRangeBlocks - 1) / kMaxRangeBlocks;
    if (ctas < min_ctas) ctas = min_ctas;
    // ... and touch at most 64 units
    const long long min_ctas_units = (a.units + 61) / 62;
    if (ctas < min_ctas_units) ctas = min_ctas_units;
    if (ctas > a.total_items) ctas = a.total_items;
    decode_kernel<D, BF16, G><<<dim3(unsigned(ctas)), kDecThreads, smem, s>>>(a);
    return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t dispatch_group(const DecodeArgs& a, int G, cudaStream_t s)
{
    switch (G) {
        case 1: return launch_decode_t<D, BF16, 1>(a, s);
        case 2: return launch_decode_t<D, BF16, 2>(a, s);
        case 4: return launch_decode_t<D, BF16, 4>(a, s);
        case 8: return launch_decode_t<D, BF16, 8>(a, s);
        default: return cudaErrorInvalidValue;
    }
}


// ---- tensor-core path (bf16 K/V) ----------------------------------------------
size_t mma_fixed_smem(int G, int item_tokens)
{
    return 1024 /* alignment slack */ + size_t(2) * G * (item_tokens + 8) * sizeof(uint16_t) + 32 +
           size_t(2) * kMaxRangeBlocks * sizeof(int);
}

template <int D, int G, bool QSPLIT>
cudaError_t launch_decode_mma_t(DecodeArgs a, cudaStream_t s)
{
    const int item_tokens = a.blocks_per_item * a.bs;
    const size_t stage = size_t(2) * item_tokens * D * 2;
    const size_t smem = kDecStages * stage + mma_fixed_smem(G, item_tokens);
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<D, G, QSPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kDecSmemLimit);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int per_sm = (2 * (smem + 1024) <= size_t(kSmemPerSm)) ? 2 : 1;
    long long ctas = (long long)num_sms() * per_sm;
    const long long min_ctas = ((long long)a.total_items * a.blocks_per_item + kMaxRangeBlocks - 1) / kMaxRangeBlocks;
    if (ctas < min_ctas) ctas = min_ctas;
    const long long min_ctas_units = (a.units + 61) / 62;
    if (ctas < min_ctas_units) ctas = min_ctas_units;
    if (ctas > a.total_items) ctas = a.total_items;
    decode_mma_kernel<D, G, QSPLIT><<<dim3(unsigned(ctas)), kDecThreads, smem, s>>>(a);
    return cudaGetLastError();
}

template <int D, bool QSPLIT>
cudaError_t dispatch_mma(const DecodeArgs& a, int G, const void* k_pages, const void* v_pages, cudaStream_t s)
{
    switch (G) {
        case 1: return launch_decode_mma_t<D, 1, QSPLIT>(a, s);
        case 2: return launch_decode_mma_t<D, 2, QSPLIT>(a, s);
        case 4: return launch_decode_mma_t<D, 4, QSPLIT>(a, s);
        case 8: return launch_decode_mma_t<D, 8, QSPLIT>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int decode_blocks_per_item(int D, bool kv_bf16, int block_size)
{
    const int item_tokens = kItemKBytes / (D * (kv_bf16 ? 2 : 4));
    return item_tokens >= block_size ? item_tokens / block_size : 1;
}

bool decode_supported(int D, bool kv_bf16, int block_size, int G)
{
    const int bpi = decode_blocks_per_item(D, kv_bf16, block_size);
    const int item_tokens = bpi * block_size;
    const size_t stage = size_t(2) * item_tokens * D * (kv_bf16 ? 2 : 4);
    if (kv_bf16) return 3 * stage + mma_fixed_smem(G, item_tokens) <= size_t(kDecSmemLimit);
    return 2 * stage + decode_fixed_smem(G, item_tokens) <= size_t(kDecSmemLimit);
}

cudaError_t launch_decode(const Geometry& g, const WorkspaceLayout& L, char* ws, const void* q,
                          const void* k_pages, const void* v_pages, const int32_t* block_table,
                          const int32_t* sel_ids, const int32_t* sel_count, float* out,
                          cudaStream_t s)
{
    const int units = g.units();
    if (units == 0) return cudaSuccess;
    DecodeArgs a{};
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
    a.sel_stride = g.sel_stride;
    a.blocks_per_item = L.blocks_per_split;
    a.items_per_unit = L.max_splits;
    a.units = units;
    a.total_items = units * L.max_splits;
    a.scale_log2 = g.scale_log2;
    a.part_m = reinterpret_cast<float*>(ws + L.part_m);
    a.part_l = reinterpret_cast<float*>(ws + L.part_l);
    a.part_o = reinterpret_cast<float*>(ws + L.part_o);
    a.counters = reinterpret_cast<uint32_t*>(ws + L.dec_counters);
    a.err = reinterpret_cast<uint32_t*>(ws + L.err);
    if (g.kv_bf16) {   // tensor-core path
        if (g.q_bf16)
            return g.D == 128 ? dispatch_mma<128, false>(a, g.G, k_pages, v_pages, s)
                              : dispatch_mma<64, false>(a, g.G, k_pages, v_pages, s);
        return g.D == 128 ? dispatch_mma<128, true>(a, g.G, k_pages, v_pages, s)
                          : dispatch_mma<64, true>(a, g.G, k_pages, v_pages, s);
    }
    return g.D == 128 ? dispatch_group<128, false>(a, g.G, s) : dispatch_group<64, false>(a, g.G, s);
}

}  // namespace sa
