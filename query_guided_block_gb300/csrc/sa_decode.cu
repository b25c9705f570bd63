// Sparse decode attention over the selected blocks only.
//
// "从HiSparse到QSA的移植实战" §3.3: the attention kernel walks a compact array of selected
// block indices and never reads unselected KV; HBM bandwidth is the bound.  SparDA page
// (www.2kiu.com/news/4656707) §5.3: skip unselected pages inside the kernel rather than
// gathering them into a temporary buffer first.  The softmax is exact over the union of
// the selected tokens (SGLang page §1.2 "select-then-compute").
//
// Design: a persistent grid over "items" (a few selected blocks, 64-128 tokens, of one
// (sequence, KV head) unit), numbered unit-major; CTA i owns an equal contiguous range,
// so it sees one or two unit boundaries and no CTA ever waits on another.  At start the
// CTA resolves, for its whole range, selected id -> page through the page table into
// shared memory (bounds-checked).  At the end of its segment of a unit the CTA writes
// one (m, l, o) partial; the CTA that completes a unit's item count merges the unit's
// partials (log-sum-exp) into fp32 outputs.
//   * bf16 K/V (the fast path, decode_mma_kernel below): warps stream 16-token slabs
//     independently through per-warp cp.async rings and do QK^T and PV on tensor cores
//     (mma.sync m16n8k16, fp32 accumulate) with the softmax on the fragments.
//   * fp32 K/V (decode_kernel): items through a CTA-wide bulk-copy pipeline, dots on
//     FMA units with the G heads' partial sums reduced across a key row's lanes.

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
    allow_dependents_early();
    grid_dependency_wait();   // inputs and workspace may come from the previous kernel

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
            } else if (a.slot_C > 0) {
                const int sl = a.sel_slot[size_t(u) * a.sel_stride + slot];
                if (sl < 0 || sl >= a.slot_C) {
                    raise_error(a.err, SPARSE_ATTN_ERR_SLOT);
                } else {
                    page = u * a.slot_C + sl;
                    valid = min(a.bs, a.N - j * a.bs);
                }
            } else {
                const int b = u / a.Hkv;
                const int p = a.block_table[size_t(b) * a.bt_stride + j];
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
        const size_t head_off = a.slot_C > 0 ? 0 : size_t(u % a.Hkv) * tile_bytes;
        const size_t page_stride = size_t(a.page_heads) * tile_bytes;
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
    return launch_after_previous(decode_kernel<D, BF16, G>, dim3(unsigned(ctas)), dim3(kDecThreads), smem, s, a);
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

// ---------------------------------------------------------------------------
// bf16 K/V: warps stream 16-token slabs independently, contractions on tensor cores.
//   * The CTA owns the same contiguous item range as above; its items are cut into
//     16-token slabs and warp w takes slabs w, w + 8, ... of the range.  Each warp runs
//     its own kSlabStages-deep ring of slabs in shared memory, filled with 16-byte
//     cp.async copies (global -> shared, L2 only) issued by its own lanes, so a warp
//     waits only on its own copies (cp.async.wait_group + __syncwarp) and the CTA never
//     synchronises inside a unit.  Rows without a token (empty block slots, the tail
//     past the context) are zero-filled by the copy.
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
//   * At the end of the CTA's segment of a unit every warp writes its (m, l, o) to the
//     ring stage it has just freed; the CTA combines the 8 into one partial and the
//     completing CTA merges the unit, as on the fp32 path.
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
    static constexpr size_t RING_BYTES = size_t(kDecWarps) * STAGES * SLAB_BYTES;
    static_assert(8 * D * 4 <= SLAB_BYTES, "a warp's flushed G x D outputs must fit one stage");
};

__device__ __forceinline__ uint32_t swz(uint32_t half_base, int token, int chunk)
{
    return half_base + uint32_t(token) * kRowBytes + uint32_t((chunk ^ (token & 7)) << 4);
}

template <int D>
constexpr size_t slab_smem_bytes()
{
    return 1024 /* alignment slack */ + SlabShape<D>::RING_BYTES + size_t(2) * kMaxRangeBlocks * sizeof(int);
}

template <int D, int G, bool QSPLIT>
__global__ void __launch_bounds__(kDecThreads, 1) decode_mma_kernel(DecodeArgs a)
{
    using SS = SlabShape<D>;
    constexpr int S = SS::STAGES;
    constexpr int DT = SS::DT;
    static_assert(G <= 8, "query rows live in the first 8 MMA rows");

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g4 = lane >> 2, t4 = lane & 3;       // MMA fragment coordinates
    const int bpi = a.blocks_per_item;
    const int ipu = a.items_per_unit;
    const int item_tokens = bpi * a.bs;            // a power of two >= 64
    const int spi_shift = __ffs(item_tokens / kSlabTokens) - 1;
    const int spi_mask = (1 << spi_shift) - 1;
    const int bs_shift = __ffs(a.bs) - 1;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // swizzle pattern repeats every 1024 bytes
    unsigned char* smem = smem_raw + (base - raw);
    const uint32_t ring = base + uint32_t(warp) * (S * SS::SLAB_BYTES);
    int* blk_page = reinterpret_cast<int*>(smem + SS::RING_BYTES);
    int* blk_valid = blk_page + kMaxRangeBlocks;
    __shared__ float s_m[kDecWarps][8], s_l[kDecWarps][8];
    __shared__ int s_flush[kDecWarps];             // byte offset of each warp's flushed (o)
    __shared__ int s_merge_unit;

    const int i_begin = int((long long)a.total_items * blockIdx.x / gridDim.x);
    const int i_end = int((long long)a.total_items * (blockIdx.x + 1) / gridDim.x);
    if (i_begin >= i_end) return;
    const int u_lo = i_begin / ipu;
    const int u_hi = (i_end - 1) / ipu;
    allow_dependents_early();
    grid_dependency_wait();   // inputs and workspace may come from the previous kernel

    // query A fragments: rows g4 < G; the lo part of an fp32 query in rows 8..15.  A bf16
    // query's pair (2 t4, 2 t4 + 1) is one aligned 32-bit word, loaded straight into the
    // fragment, so the load latency is paid at the first MMA rather than here.
    uint32_t qa[D / 16][4];
    auto load_qfrag = [&](int u) {
        const size_t head0 = size_t(u / a.Hkv) * a.Hq + size_t(u % a.Hkv) * G;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const size_t qrow = (head0 + g4) * D + ks * 16 + 2 * t4;
            if constexpr (!QSPLIT) {
                const uint32_t* q32 = reinterpret_cast<const uint32_t*>(a.q);
                qa[ks][0] = g4 < G ? __ldg(q32 + qrow / 2) : 0u;
                qa[ks][2] = g4 < G ? __ldg(q32 + qrow / 2 + 4) : 0u;
                qa[ks][1] = qa[ks][3] = 0u;
            } else {
                const float2* q64 = reinterpret_cast<const float2*>(a.q);
                const float2 f0 = g4 < G ? __ldg(q64 + qrow / 2) : make_float2(0.f, 0.f);
                const float2 f2 = g4 < G ? __ldg(q64 + qrow / 2 + 4) : make_float2(0.f, 0.f);
                qa[ks][0] = pack_bf16x2(f0.x, f0.y);
                qa[ks][2] = pack_bf16x2(f2.x, f2.y);
                qa[ks][1] = pack_bf16x2(f0.x - bf16_lo(qa[ks][0]), f0.y - bf16_hi(qa[ks][0]));
                qa[ks][3] = pack_bf16x2(f2.x - bf16_lo(qa[ks][2]), f2.y - bf16_hi(qa[ks][2]));
            }
        }
    };
    load_qfrag(u_lo);

    // ---- resolve the range: selected ids -> pages (two dependent loads) --------
    const int n_range_blocks = (i_end - i_begin) * bpi;
    for (int e = tid; e < n_range_blocks; e += kDecThreads) {
        const int item = i_begin + e / bpi;
        const int u = item / ipu;
        const int slot = (item - u * ipu) * bpi + e % bpi;
        int count = a.sel_count[u];
        const int j = slot < a.sel_stride ? a.sel_ids[size_t(u) * a.sel_stride + slot] : -1;
        if (count < 0 || count > a.sel_stride) {
            raise_error(a.err, SPARSE_ATTN_ERR_SEL_COUNT);
            count = count < 0 ? 0 : a.sel_stride;
        }
        int page = -1, valid = 0;
        if (slot < count) {
            if (j < 0 || j >= a.nb) {
                raise_error(a.err, SPARSE_ATTN_ERR_SEL_ID);
            } else if (a.slot_C > 0) {
                const int sl = a.sel_slot[size_t(u) * a.sel_stride + slot];
                if (sl < 0 || sl >= a.slot_C) {
                    raise_error(a.err, SPARSE_ATTN_ERR_SLOT);
                } else {
                    page = u * a.slot_C + sl;
                    valid = min(a.bs, a.N - j * a.bs);
                }
            } else {
                const int p = a.block_table[size_t(u / a.Hkv) * a.bt_stride + j];
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

    // Stage slab s of the range into this warp's stage st: lane copies chunk cp_c of
    // slab rows cp_r, cp_r + RPI, ...; a warp instruction covers RPI whole token rows.
    const char* kbase = reinterpret_cast<const char*>(a.k_pages);
    const char* vbase = reinterpret_cast<const char*>(a.v_pages);
    const int cp_c = lane % SS::CPR, cp_r = lane / SS::CPR;
    const int n_slabs = (i_end - i_begin) << spi_shift;
    auto issue_slab = [&](int s, int st) {
        const int k = s >> spi_shift;                                  // item within the range
        const int t0 = (s & spi_mask) * kSlabTokens;                  // first token in the item
        const size_t head_rows = a.slot_C > 0 ? 0 : size_t(((i_begin + k) / ipu) % a.Hkv) * a.bs;
        const uint32_t kd = ring + uint32_t(st) * SS::SLAB_BYTES + uint32_t(cp_c >> 3) * SS::HALF_BYTES;
        const uint32_t vd = kd + SS::TENSOR_BYTES;
#pragma unroll
        for (int i = 0; i < SS::CP_ITERS; ++i) {
            const int tr = cp_r + i * SS::RPI;                         // row within the slab
            const int t = t0 + tr;
            const int e = k * bpi + (t >> bs_shift), r = t & (a.bs - 1);
            const bool ok = r < blk_valid[e];                          // 0 for an empty slot
            const size_t off = ok ? ((size_t(blk_page[e]) * a.page_heads * a.bs + head_rows + r) * (D * 2) + cp_c * 16) : 0;
            const uint32_t so = uint32_t(tr) * kRowBytes + uint32_t(((cp_c & 7) ^ (tr & 7)) << 4);
            cp_async_16_zfill(kd + so, kbase + off, ok ? 16u : 0u);
            cp_async_16_zfill(vd + so, vbase + off, ok ? 16u : 0u);
        }
    };
#pragma unroll
    for (int kk = 0; kk < S - 1; ++kk) {
        const int s = warp + kk * kDecWarps;
        if (s < n_slabs) issue_slab(s, kk);
        cp_async_commit();
    }

    int my = 0;                                    // slabs this warp has consumed
    for (int u = u_lo; u <= u_hi; ++u) {
        const int seg_i0 = max(i_begin, u * ipu), seg_i1 = min(i_end, (u + 1) * ipu);
        const int se = (seg_i1 - i_begin) << spi_shift;
        const int b = u / a.Hkv, kvh = u - (u / a.Hkv) * a.Hkv;
        const size_t head0 = size_t(b) * a.Hq + size_t(kvh) * G;

        float acc[DT][4];
#pragma unroll
        for (int j = 0; j < DT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
        float m_run = -INFINITY, l_run = 0.f;      // head g4: running max (quad-uniform), lane sum

        for (int s = warp + my * kDecWarps; s < se; s += kDecWarps, ++my) {
            cp_async_wait_group<S - 2>();          // this lane's copies of slab s are done
            __syncwarp();                          // ... and every lane's; stage my - 1 is free
            {
                const int nx = s + (S - 1) * kDecWarps;
                if (nx < n_slabs) issue_slab(nx, (my + S - 1) % S);
                cp_async_commit();
            }
            const uint32_t kst = ring + uint32_t(my % S) * SS::SLAB_BYTES;
            const uint32_t vst = kst + SS::TENSOR_BYTES;

            // ---- S = q K^T over the slab's two 8-token tiles ----------------------
            float c[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                c[nt][0] = c[nt][1] = c[nt][2] = c[nt][3] = 0.f;
#pragma unroll
                for (int kp = 0; kp < D / 32; ++kp) {   // two 16-channel k-steps per ldmatrix.x4
                    const int ch = kp * 4 + (lane >> 3);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(swz(kst + uint32_t(ch >> 3) * SS::HALF_BYTES, nt * 8 + (lane & 7), ch & 7), b0, b1, b2, b3);
                    mma_bf16_16816(c[nt], qa[2 * kp][0], qa[2 * kp][1], qa[2 * kp][2], qa[2 * kp][3], b0, b1);
                    mma_bf16_16816(c[nt], qa[2 * kp + 1][0], qa[2 * kp + 1][1], qa[2 * kp + 1][2], qa[2 * kp + 1][3], b2, b3);
                }
            }
            // ---- online softmax on the fragments ----------------------------------
            const int k = s >> spi_shift;
            const int tb = (s & spi_mask) * kSlabTokens + 2 * t4;
            float sc[2][2];
            float mx = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int t = tb + nt * 8 + e;
                    const bool ok = (t & (a.bs - 1)) < blk_valid[k * bpi + (t >> bs_shift)];
                    sc[nt][e] = ok ? (c[nt][e] + c[nt][e + 2]) * a.scale_log2 : -INFINITY;
                    mx = fmaxf(mx, sc[nt][e]);
                }
            mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 2));
            const float m_new = fmaxf(m_run, mx);
            const float alpha = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - m_new);
            m_run = m_new;
            float p[2][2];
            float psum = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    p[nt][e] = (sc[nt][e] == -INFINITY) ? 0.f : fast_exp2(sc[nt][e] - m_new);
                    psum += p[nt][e];
                }
            l_run = fmaf(l_run, alpha, psum);
            const uint32_t ph0 = pack_bf16x2(p[0][0], p[0][1]);
            const uint32_t ph2 = pack_bf16x2(p[1][0], p[1][1]);
            const uint32_t pl0 = pack_bf16x2(p[0][0] - bf16_lo(ph0), p[0][1] - bf16_hi(ph0));
            const uint32_t pl2 = pack_bf16x2(p[1][0] - bf16_lo(ph2), p[1][1] - bf16_hi(ph2));

            // ---- O += P V: all D channels, k = the slab's 16 tokens ---------------
#pragma unroll
            for (int j = 0; j < DT; ++j) {
                acc[j][0] *= alpha;
                acc[j][1] *= alpha;
                acc[j][2] *= alpha;
                acc[j][3] *= alpha;
            }
#pragma unroll
            for (int jp = 0; jp < DT; jp += 2) {
                // matrices: (tokens 0..7, chunk jp), (8..15, jp), (0..7, jp + 1), (8..15, jp + 1)
                const int mtx = lane >> 3;
                const int chunk = jp + (mtx >> 1);
                uint32_t r0, r1, r2, r3;
                ldsm_x4_trans(swz(vst + uint32_t(chunk >> 3) * SS::HALF_BYTES, (mtx & 1) * 8 + (lane & 7), chunk & 7),
                              r0, r1, r2, r3);
                mma_bf16_16816(acc[jp], ph0, pl0, ph2, pl2, r0, r1);
                mma_bf16_16816(acc[jp + 1], ph0, pl0, ph2, pl2, r2, r3);
            }
        }

        if (u < u_hi) load_qfrag(u + 1);           // in flight across the combine below

        // ---- end of the CTA's segment of unit u: combine the warps ---------------
        l_run += __shfl_xor_sync(kFullMask, l_run, 1);
        l_run += __shfl_xor_sync(kFullMask, l_run, 2);
        {
            const int free_off = int((warp * S + (my + S - 1) % S) * SS::SLAB_BYTES);
            float* ob = reinterpret_cast<float*>(smem + free_off);
            if (g4 < G) {
#pragma unroll
                for (int j = 0; j < DT; ++j)
                    *reinterpret_cast<float2*>(ob + g4 * D + j * 8 + 2 * t4) =
                        make_float2(acc[j][0] + acc[j][2], acc[j][1] + acc[j][3]);
                if (t4 == 0) {
                    s_m[warp][g4] = m_run;
                    s_l[warp][g4] = l_run;
                }
            }
            if (lane == 0) s_flush[warp] = free_off;
        }
        __syncthreads();
        const int slot = seg_i0 - u * ipu;
        for (int i = tid; i < G * D; i += kDecThreads) {
            const int g = i / D, d = i - g * D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, s_m[w][g]);
            float o = 0.f, l = 0.f;
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) {
                const float mw = s_m[w][g];
                if (mw == -INFINITY) continue;     // a warp without a token here wrote nothing useful
                const float wt = fast_exp2(mw - M);
                o = fmaf(wt, reinterpret_cast<const float*>(smem + s_flush[w])[g * D + d], o);
                l = fmaf(wt, s_l[w][g], l);
            }
            const size_t ps = (head0 + g) * ipu + slot;
            a.part_o[ps * D + d] = o;
            if (d == 0) {
                a.part_m[ps] = M;
                a.part_l[ps] = l;
            }
        }
        __syncthreads();                           // partials written; flush stages free again
        if (tid == 0) {
            const uint32_t n = uint32_t(seg_i1 - seg_i0);
            const uint32_t before = atomic_add_acq_rel_u32(&a.counters[u], n);
            s_merge_unit = before + n == uint32_t(ipu) ? u : -1;
        }
        __syncthreads();
        if (s_merge_unit >= 0) {
            merge_unit(a, u, G, D);
            __syncthreads();
        }
    }
    cp_async_wait_group<0>();
}

template <int D, int G, bool QSPLIT>
cudaError_t launch_decode_mma_t(DecodeArgs a, cudaStream_t s)
{
    constexpr size_t smem = slab_smem_bytes<D>();
    static_assert(smem <= size_t(kDecSmemLimit), "slab rings must fit a CTA");
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<D, G, QSPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kDecSmemLimit);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    long long ctas = num_sms();                    // one CTA (8 independent warps) per SM
    const long long min_ctas = ((long long)a.total_items * a.blocks_per_item + kMaxRangeBlocks - 1) / kMaxRangeBlocks;
    if (ctas < min_ctas) ctas = min_ctas;
    const long long min_ctas_units = (a.units + 61) / 62;
    if (ctas < min_ctas_units) ctas = min_ctas_units;
    if (ctas > a.total_items) ctas = a.total_items;
    return launch_after_previous(decode_mma_kernel<D, G, QSPLIT>, dim3(unsigned(ctas)), dim3(kDecThreads), smem, s, a);
}

template <int D, bool QSPLIT>
cudaError_t dispatch_mma(const DecodeArgs& a, int G, cudaStream_t s)
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
    if (kv_bf16) return item_tokens % kSlabTokens == 0;   // slab rings have a fixed size
    return 2 * stage + decode_fixed_smem(G, item_tokens) <= size_t(kDecSmemLimit);
}

cudaError_t launch_decode(const Geometry& g, const WorkspaceLayout& L, char* ws, const void* q,
                          const void* k_pages, const void* v_pages, const int32_t* block_table,
                          const int32_t* sel_ids, const int32_t* sel_count, float* out,
                          const int32_t* sel_slot, int slot_C, cudaStream_t s)
{
    const int units = g.units();
    if (units == 0) return cudaSuccess;
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
            return g.D == 128 ? dispatch_mma<128, false>(a, g.G, s) : dispatch_mma<64, false>(a, g.G, s);
        return g.D == 128 ? dispatch_mma<128, true>(a, g.G, s) : dispatch_mma<64, true>(a, g.G, s);
    }
    return g.D == 128 ? dispatch_group<128, false>(a, g.G, s) : dispatch_group<64, false>(a, g.G, s);
}

}  // namespace sa
