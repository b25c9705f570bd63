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
constexpr int kBarDecoders = 1;            // named barrier of the kDecThreads decoding threads

// Barrier of the CTA's kDecThreads decoding threads (threads 0 .. kDecThreads - 1): the
// whole CTA in the decode kernels, the worker warps (not the control warp) in the fused
// step kernel.
__device__ __forceinline__ void decoder_barrier()
{
    asm volatile("bar.sync %0, %1;" ::"n"(kBarDecoders), "n"(kDecThreads) : "memory");
}

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
    // slot mode with the step's misses loaded in the same launch (io_host_k != null):
    // loader CTAs copy unit u's misses (io_miss_ids[u][0 .. io_counts[u][1]), ascending,
    // into pool slots io_miss_slot[u][...]) from the host store -- page block_table[b][j],
    // KV head u % Hkv -- and publish io_flags[u] = the launch's flag value; the decode
    // takes a unit's missed blocks last and waits (bounded) for that flag before them
    const char* io_host_k;
    const char* io_host_v;
    const int32_t* io_miss_ids;
    const int32_t* io_miss_slot;
    const int32_t* io_counts;
    uint32_t* io_flags;
    int io_loaders;          // CTAs ranges .. ranges + io_loaders - 1 load misses
    int blocks_per_item, items_per_unit, total_items, units;
    int ranges;              // CTAs 0 .. ranges - 1 own contiguous item ranges (<= the grid)
    int stages;
    float scale_log2;
    float* part_m;   // [B*Hq, items_per_unit]
    float* part_l;
    float* part_o;   // [B*Hq, items_per_unit, D]
    uint32_t* counters;
    uint32_t* err;
};

// The CTA that completed unit u merges the unit's partials.  A unit's segments start
// at its first item and at every range start inside it (range c = items
// [T c / R, T (c + 1) / R) of the T items, R = a.ranges); each segment wrote one
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
    const long long T = a.total_items, C = a.ranges;
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
        decoder_barrier();
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
        decoder_barrier();                                       // s_pm / s_pl reused
    }
#pragma unroll
    for (int r = 0; r < kMergeOut; ++r) {
        const int i = tid + r * kDecThreads;
        if (i >= G * D) break;
        a.out[head0 * D + i] = den[r] > 0.f ? num[r] / den[r] : 0.f;
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

// With misses read from the host in the same pass: one more int per cached block (its
// host page, or -1).
template <int D>
constexpr size_t slab_smem_bytes_io()
{
    return slab_smem_bytes<D>() + size_t(kMaxRangeBlocks) * sizeof(int);
}

// Items [i_begin, i_end) of a decode launch, by one CTA.  With `ready` set, the CTA
// first waits (bounded) until ready[u] == flag_value for every unit of the range (the
// selection may still be running in this grid or in the select kernel before this one).
template <int D, int G, bool QSPLIT, bool IO = false>
__device__ __forceinline__ void decode_mma_items(const DecodeArgs& a, uint32_t* ready, uint32_t flag_value,
                                                 int i_begin, int i_end)
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
    int* blk_host = blk_valid + kMaxRangeBlocks;   // only with IO (slab_smem_bytes_io)
    constexpr bool io = IO;
    __shared__ float s_m[kDecWarps][8], s_l[kDecWarps][8];
    __shared__ int s_flush[kDecWarps];             // byte offset of each warp's flushed (o)
    __shared__ int s_merge_unit;

    if (i_begin >= i_end) return;
    const int u_lo = i_begin / ipu;
    const int u_hi = (i_end - 1) / ipu;

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
    if (ready != nullptr) {   // selections published by other CTAs (acquire)
        const long long wait_cycles = handoff_wait_limit(a.err);
        for (int u = u_lo + tid; u <= u_hi; u += kDecThreads)
            if (!wait_flag_bounded(ready + u, flag_value, wait_cycles)) raise_error(a.err, SPARSE_ATTN_ERR_TIMEOUT);
        __threadfence();
        decoder_barrier();
    }
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
        int page = -1, valid = 0, host = -1;
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
                    if (io) {   // a miss of this step: its host page
                        int n_miss = a.io_counts[size_t(u) * 5 + 1];
                        n_miss = n_miss < 0 ? 0 : min(n_miss, a.sel_stride);
                        const int32_t* mids = a.io_miss_ids + size_t(u) * a.sel_stride;
                        int lo = 0, hi = n_miss;   // first index with mids[index] >= j
                        while (lo < hi) {
                            const int mid = (lo + hi) >> 1;
                            if (mids[mid] < j) lo = mid + 1;
                            else hi = mid;
                        }
                        if (lo < n_miss && mids[lo] == j) host = 1;
                    }
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
        if (io) blk_host[e] = host;
    }
    decoder_barrier();
    if constexpr (IO) {
        // a unit's missed blocks last (stable within hits and within misses), so their
        // load overlaps the attention over the unit's resident blocks; the rings are
        // free yet and hold the copy
        int* tmp = reinterpret_cast<int*>(smem);
        for (int e = tid; e < n_range_blocks; e += kDecThreads) {
            tmp[3 * e] = blk_page[e];
            tmp[3 * e + 1] = blk_valid[e];
            tmp[3 * e + 2] = blk_host[e];
        }
        decoder_barrier();
        for (int e = tid; e < n_range_blocks; e += kDecThreads) {
            const int u = (i_begin + e / bpi) / ipu;
            const int e0 = max(0, u * ipu - i_begin) * bpi;                  // the unit's first block here
            const int e1 = min(n_range_blocks, ((u + 1) * ipu - i_begin) * bpi);
            int before = 0, total = 0;                                      // misses before e / in all
            for (int f = e0; f < e1; ++f) {
                const int m = tmp[3 * f + 2] >= 0;
                total += m;
                before += (f < e) & m;
            }
            const bool miss = tmp[3 * e + 2] >= 0;
            const int pos = e0 + (miss ? (e1 - e0 - total) + before : (e - e0) - before);
            blk_page[pos] = tmp[3 * e];
            blk_valid[pos] = tmp[3 * e + 1];
            blk_host[pos] = tmp[3 * e + 2];
        }
        decoder_barrier();
    }

    // Stage slab s of the range into this warp's stage st: lane copies chunk cp_c of
    // slab rows cp_r, cp_r + RPI, ...; a warp instruction covers RPI whole token rows.
    // Before the first slab of a unit that holds a block missed this step, the warp
    // waits (bounded, acquire) until the loaders have put the unit's misses in the pool.
    int io_unit_ready = -1;
    const char* kbase = reinterpret_cast<const char*>(a.k_pages);
    const char* vbase = reinterpret_cast<const char*>(a.v_pages);
    const int cp_c = lane % SS::CPR, cp_r = lane / SS::CPR;
    const int n_slabs = (i_end - i_begin) << spi_shift;
    auto issue_slab = [&](int s, int st) {
        const int k = s >> spi_shift;                                  // item within the range
        const int t0 = (s & spi_mask) * kSlabTokens;                  // first token in the item
        if constexpr (IO) {
            const int su = (i_begin + k) / ipu;
            if (su != io_unit_ready && (blk_host[k * bpi + (t0 >> bs_shift)] >= 0 ||
                                        blk_host[k * bpi + ((t0 + kSlabTokens - 1) >> bs_shift)] >= 0)) {
                if (!wait_flag_bounded(a.io_flags + su, flag_value, handoff_wait_limit(a.err)))
                    raise_error(a.err, SPARSE_ATTN_ERR_TIMEOUT);
                __syncwarp();
                io_unit_ready = su;
            }
        }
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
        decoder_barrier();
        // a segment holding the whole unit is its result: no partial, no merge (the
        // merge of one partial gives the same bits)
        const bool whole = seg_i0 == u * ipu && seg_i1 == (u + 1) * ipu;
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
            if (whole) {
                a.out[head0 * D + i] = l > 0.f ? o / l : 0.f;
                continue;
            }
            const size_t ps = (head0 + g) * ipu + slot;
            a.part_o[ps * D + d] = o;
            if (d == 0) {
                a.part_m[ps] = M;
                a.part_l[ps] = l;
            }
        }
        decoder_barrier();                           // partials written; flush stages free again
        if (whole) continue;
        if (tid == 0) {
            const uint32_t n = uint32_t(seg_i1 - seg_i0);
            const uint32_t before = atomic_add_acq_rel_u32(&a.counters[u], n);
            s_merge_unit = before + n == uint32_t(ipu) ? u : -1;
        }
        decoder_barrier();
        if (s_merge_unit >= 0) {
            merge_unit(a, u, G, D);
            decoder_barrier();
        }
    }
    cp_async_wait_group<0>();
}


// One CTA's share of a decode launch: range blockIdx.x of a.ranges (none beyond).
template <int D, int G, bool QSPLIT, bool IO = false>
__device__ __forceinline__ void decode_mma_body(const DecodeArgs& a, uint32_t* ready, uint32_t flag_value)
{
    if (int(blockIdx.x) >= a.ranges) return;
    const int i_begin = int((long long)a.total_items * blockIdx.x / a.ranges);
    const int i_end = int((long long)a.total_items * (blockIdx.x + 1) / a.ranges);
    decode_mma_items<D, G, QSPLIT, IO>(a, ready, flag_value, i_begin, i_end);
}

// Item ranges of a bf16 decode launch (one per CTA).  By default one per SM (more when
// a range would overflow a CTA's page cache or touch more than 62 units, never more
// than there are items): the units are then cut across CTA boundaries and merged.
// When whole units, or equal parts of units, fill at least 80% of the SMs, the ranges
// follow the unit boundaries instead: with units <= SMs each unit is split into
// SMs / units equal parts (one part: the segment is the result, no partial and no
// merge); with more units than SMs each range holds the same number of whole units.
// An SM streams about as fast as the HBM share of a full grid allows, so leaving a few
// SMs idle costs less than the split units' partials, merges and segment ends.
inline int decode_ranges(int units, int items_per_unit, int blocks_per_item, int sms)
{
    const long long T = (long long)units * items_per_unit;
    long long R = sms;
    const long long min_ctas = (T * blocks_per_item + kMaxRangeBlocks - 1) / kMaxRangeBlocks;
    const long long min_units = (units + 61) / 62;
    if (R < min_ctas) R = min_ctas;
    if (R < min_units) R = min_units;
    if (R > T) R = T;
    long long aligned = 0;
    if (units > 0 && units <= sms) {
        aligned = (long long)units * (sms / units);
    } else if (units > sms) {
        const long long per = (units + sms - 1) / sms;
        if (units % per == 0) aligned = units / per;
    }
    if (aligned > 0 && 5 * aligned >= 4LL * sms && aligned >= min_ctas && aligned >= min_units && aligned <= T)
        R = aligned;
    return int(R < 1 ? 1 : R);
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
    a.ranges = decode_ranges(g.units(), L.max_splits, L.blocks_per_split, num_sms());   // bf16 path
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
