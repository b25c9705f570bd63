// Sparse decode attention over the selected blocks only.
//
// "从HiSparse到QSA的移植实战" §3.3: the attention kernel walks a compact array of selected
// block indices and never reads unselected KV; HBM bandwidth is the bound.  SparDA page
// (www.2kiu.com/news/4656707) §5.3: skip unselected pages inside the kernel rather than
// gathering them into a temporary buffer first.  The softmax is exact over the union of
// the selected tokens (SGLang page §1.2: select, then compute).
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

#include "sa_decode_body.cuh"

namespace sa {
namespace {

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
    static std::atomic<unsigned long long> configured{0};   // devices set up
    const cudaError_t cfg = once_per_device(configured, [&]() -> cudaError_t {
        return cudaFuncSetAttribute(decode_kernel<D, BF16, G>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmemLimit);
    });
    if (cfg != cudaSuccess) return cfg;
    const int per_sm = (2 * (smem + 1024) <= size_t(kSmemPerSm)) ? 2 : 1;
    long long ctas = (long long)num_sms() * per_sm;
    // every CTA's range must fit its shared-memory page cache
    const long long min_ctas = ((long long)a.total_items * a.blocks_per_item + kMaxRangeBlocks - 1) / kMaxRangeBlocks;
    if (ctas < min_ctas) ctas = min_ctas;
    // ... and touch at most 64 units
    const long long min_ctas_units = (a.units + 61) / 62;
    if (ctas < min_ctas_units) ctas = min_ctas_units;
    if (ctas > a.total_items) ctas = a.total_items;
    DecodeArgs args = a;
    args.ranges = int(ctas);   // this kernel's ranges: one per CTA of its own grid
    return launch_after_previous(decode_kernel<D, BF16, G>, dim3(unsigned(ctas)), dim3(kDecThreads), smem, s, args);
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


// With `ready` set the kernel runs behind a select kernel that publishes each unit's
// selection: it skips the grid-wide wait and waits per unit instead, so its CTAs
// start on SMs as the select kernel's CTAs leave them.
template <int D, int G, bool QSPLIT, bool IO>
__global__ void __launch_bounds__(kDecThreads, 1) decode_mma_kernel(DecodeArgs a, uint32_t* ready)
{
    allow_dependents_early();
    if (ready == nullptr) {
        grid_dependency_wait();   // inputs and workspace may come from the previous kernel
        decode_mma_body<D, G, QSPLIT, IO>(a, nullptr, 0u);
        return;
    }
    // behind the step's select kernel: the same flag value as it publishes
    const uint32_t flag_value = step_flag_value(a.err);
    decode_mma_body<D, G, QSPLIT, IO>(a, ready, flag_value);
    finish_step(a.err, flag_value);
}

// Loader CTA: copy the misses (K and V tiles) of units [u0, u1) from the host store into
// their pool slots, then publish io_flags[u] for each.  The whole share is one batch --
// miss counts, then every miss's ids and pages, then every tile, each step with all its
// loads in flight -- so the latency is paid a few times per CTA, not per unit.
// `scratch`: dynamic shared memory for (u1 - u0) + 1 counts and 2 offsets per miss.
__device__ void load_misses_for_units(const DecodeArgs& a, int u0, int u1, int D, uint32_t flag_value,
                                      unsigned char* scratch, size_t scratch_bytes)
{
    constexpr int kInFlight = 8;
    __shared__ int s_total;
    const int tid = threadIdx.x;
    const int nu = u1 - u0;
    int* first = reinterpret_cast<int*>(scratch);                        // [nu + 1] prefix of counts
    long long* offs = reinterpret_cast<long long*>(scratch + ((size_t(nu + 1) * sizeof(int) + 15) & ~size_t(15)));
    const long long max_misses = (long long)((scratch + scratch_bytes) - reinterpret_cast<unsigned char*>(offs)) / 16;
    const size_t tile = size_t(a.bs) * D * 2;
    if (nu <= 0) return;
    for (int i = tid; i < nu; i += kDecThreads) {
        int n = a.io_counts[size_t(u0 + i) * 5 + 1];
        if (n < 0 || n > a.sel_stride) {
            raise_error(a.err, SPARSE_ATTN_ERR_SEL_COUNT);
            n = n < 0 ? 0 : a.sel_stride;
        }
        first[i + 1] = n;
    }
    __syncthreads();
    if (tid == 0) {   // a few hundred units at most: a serial prefix is cheap
        first[0] = 0;
        for (int i = 0; i < nu; ++i) first[i + 1] += first[i];
        if (first[nu] > max_misses) raise_error(a.err, SPARSE_ATTN_ERR_SEL_COUNT);   // host sizing prevents it
        s_total = int(min((long long)first[nu], max_misses));
    }
    __syncthreads();
    const int total = s_total;
    for (int m = tid; m < total; m += kDecThreads) {
        int lo = 0, hi = nu;   // the unit holding miss m: first[lo] <= m < first[lo + 1]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (first[mid] <= m) lo = mid;
            else hi = mid;
        }
        const int u = u0 + lo, i = m - first[lo];
        const int b = u / a.Hkv, kvh = u - (u / a.Hkv) * a.Hkv;
        const int j = a.io_miss_ids[size_t(u) * a.sel_stride + i];
        const int sl = a.io_miss_slot[size_t(u) * a.sel_stride + i];
        long long so = -1, dst = 0;
        if (j < 0 || j >= a.nb || sl < 0 || sl >= a.slot_C) {
            raise_error(a.err, j < 0 || j >= a.nb ? SPARSE_ATTN_ERR_SEL_ID : SPARSE_ATTN_ERR_SLOT);
        } else {
            const int p = a.block_table[size_t(b) * a.bt_stride + j];
            if (p < 0 || p >= a.num_pages) {
                raise_error(a.err, SPARSE_ATTN_ERR_PAGE);
            } else {
                so = (long long)((size_t(p) * a.Hkv + kvh) * tile);
                dst = (long long)((size_t(u) * a.slot_C + sl) * tile);
            }
        }
        offs[2 * m] = so;
        offs[2 * m + 1] = dst;
    }
    __syncthreads();
    const long long n16 = (long long)(tile / 16);
    const long long elems = n16 * total;                    // per tensor
    char* pk = const_cast<char*>(static_cast<const char*>(a.k_pages));
    char* pv = const_cast<char*>(static_cast<const char*>(a.v_pages));
    for (long long base = 0; base < 2 * elems; base += (long long)kDecThreads * kInFlight) {
        uint4 v[kInFlight];
#pragma unroll
        for (int r = 0; r < kInFlight; ++r) {
            const long long f = base + (long long)r * kDecThreads + tid;
            if (f < 2 * elems) {
                const long long g = f < elems ? f : f - elems;
                const int m = int(g / n16);
                if (offs[2 * m] >= 0) v[r] = ld_stream16((f < elems ? a.io_host_k : a.io_host_v) + offs[2 * m] + (g - m * n16) * 16);
            }
        }
#pragma unroll
        for (int r = 0; r < kInFlight; ++r) {
            const long long f = base + (long long)r * kDecThreads + tid;
            if (f < 2 * elems) {
                const long long g = f < elems ? f : f - elems;
                const int m = int(g / n16);
                if (offs[2 * m] >= 0)
                    *reinterpret_cast<uint4*>((f < elems ? pk : pv) + offs[2 * m + 1] + (g - m * n16) * 16) = v[r];
            }
        }
    }
    __syncthreads();   // every tile of the share is written
    for (int i = tid; i < nu; i += kDecThreads) {
        __threadfence();
        st_release_gpu(a.io_flags + u0 + i, flag_value);
    }
}

// The slot decode with the step's misses loaded in the same cooperative grid: CTAs
// below a.ranges decode (a unit's missed blocks last), the others load the misses of an
// equal share of the units.  Every CTA is resident, the loaders wait on nothing, so each
// wait ends.
template <int D, int G, bool QSPLIT>
__global__ void __launch_bounds__(kDecThreads, 1) decode_io_kernel(DecodeArgs a)
{
    const uint32_t flag_value = step_flag_value(a.err);
    if (int(blockIdx.x) < a.ranges) {
        decode_mma_body<D, G, QSPLIT, true>(a, nullptr, flag_value);
    } else {
        extern __shared__ __align__(16) unsigned char io_scratch[];   // the rings this CTA does not use
        const int L = int(blockIdx.x) - a.ranges;
        const int u0 = int((long long)a.units * L / a.io_loaders), u1 = int((long long)a.units * (L + 1) / a.io_loaders);
        load_misses_for_units(a, u0, u1, D, flag_value, io_scratch, slab_smem_bytes_io<D>());
    }
    finish_step(a.err, flag_value);
}

template <int D, int G, bool QSPLIT>
cudaError_t launch_decode_io_t(DecodeArgs a, cudaStream_t s)
{
    constexpr size_t smem = slab_smem_bytes_io<D>();
    static_assert(smem <= size_t(kDecSmemLimit), "slab rings must fit a CTA");
    static std::atomic<unsigned long long> configured{0};   // devices set up
    const cudaError_t cfg = once_per_device(configured, [&]() -> cudaError_t {
        return cudaFuncSetAttribute(decode_io_kernel<D, G, QSPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kDecSmemLimit);
    });
    if (cfg != cudaSuccess) return cfg;
    cudaLaunchConfig_t c = {};
    c.gridDim = dim3(unsigned(a.ranges + a.io_loaders));
    c.blockDim = dim3(kDecThreads);
    c.dynamicSmemBytes = smem;
    c.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // all CTAs resident: the decode's waits end
    attr[0].val.cooperative = 1;
    c.attrs = attr;
    c.numAttrs = 1;
    return cudaLaunchKernelEx(&c, decode_io_kernel<D, G, QSPLIT>, a);
}

template <int D, int G, bool QSPLIT>
cudaError_t launch_decode_mma_t(DecodeArgs a, uint32_t* ready, cudaStream_t s)
{
    if (a.io_host_k != nullptr) return launch_decode_io_t<D, G, QSPLIT>(a, s);
    static_assert(slab_smem_bytes<D>() <= size_t(kDecSmemLimit), "slab rings must fit a CTA");
    constexpr size_t smem = slab_smem_bytes<D>();
    static std::atomic<unsigned long long> configured{0};   // devices set up
    const cudaError_t cfg = once_per_device(configured, [&]() -> cudaError_t {
        return cudaFuncSetAttribute(decode_mma_kernel<D, G, QSPLIT, false>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kDecSmemLimit);
    });
    if (cfg != cudaSuccess) return cfg;
    const unsigned ctas = unsigned(a.ranges);       // one CTA (8 independent warps) per range
    return launch_after_previous(decode_mma_kernel<D, G, QSPLIT, false>, dim3(ctas), dim3(kDecThreads), smem, s, a,
                                 ready);
}

template <int D, bool QSPLIT>
cudaError_t dispatch_mma(const DecodeArgs& a, int G, uint32_t* ready, cudaStream_t s)
{
    switch (G) {
        case 1: return launch_decode_mma_t<D, 1, QSPLIT>(a, ready, s);
        case 2: return launch_decode_mma_t<D, 2, QSPLIT>(a, ready, s);
        case 4: return launch_decode_mma_t<D, 4, QSPLIT>(a, ready, s);
        case 8: return launch_decode_mma_t<D, 8, QSPLIT>(a, ready, s);
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
                          const int32_t* sel_slot, int slot_C, cudaStream_t s, uint32_t* ready,
                          const SlotIo* io)
{
    const int units = g.units();
    if (units == 0) return cudaSuccess;
    DecodeArgs a = decode_args(g, L, ws, q, k_pages, v_pages, block_table, sel_ids, sel_count, out,
                               sel_slot, slot_C);
    if (io != nullptr) {
        if (!g.kv_bf16 || slot_C < 1) return cudaErrorNotSupported;
        const int loaders = num_sms() - a.ranges < 32 ? num_sms() - a.ranges : 32;
        // a loader's share must fit its shared memory: counts, then two offsets per miss
        const long long per = loaders > 0 ? (units + loaders - 1) / loaders : 0;
        const size_t need = size_t(per + 1) * sizeof(int) + 16 + size_t(per) * g.sel_stride * 16;
        const size_t have = g.D == 128 ? slab_smem_bytes_io<128>() : slab_smem_bytes_io<64>();
        if (loaders < 1 || need > have) {   // the misses first, in their own launch
            const cudaError_t e = launch_load_misses(g, io->host_k, io->host_v, block_table, io->miss_ids,
                                                     io->miss_slot, io->counts, slot_C, const_cast<void*>(k_pages),
                                                     const_cast<void*>(v_pages), a.err, s);
            if (e != cudaSuccess) return e;
        } else {
            a.io_host_k = static_cast<const char*>(io->host_k);
            a.io_host_v = static_cast<const char*>(io->host_v);
            a.io_miss_ids = io->miss_ids;
            a.io_miss_slot = io->miss_slot;
            a.io_counts = io->counts;
            a.io_flags = reinterpret_cast<uint32_t*>(ws + L.ready);
            a.io_loaders = loaders;
        }
    }
    if (g.kv_bf16) {   // tensor-core path
        if (g.q_bf16)
            return g.D == 128 ? dispatch_mma<128, false>(a, g.G, ready, s) : dispatch_mma<64, false>(a, g.G, ready, s);
        return g.D == 128 ? dispatch_mma<128, true>(a, g.G, ready, s) : dispatch_mma<64, true>(a, g.G, ready, s);
    }
    return g.D == 128 ? dispatch_group<128, false>(a, g.G, s) : dispatch_group<64, false>(a, g.G, s);
}

}  // namespace sa
