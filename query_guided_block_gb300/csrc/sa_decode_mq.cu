// Multi-query sparse attention: Q query vectors per sequence share one selection per
// KV head ("从HiSparse到QSA的移植实战" §1.1, §4.3: the long-context prefill setting, where
// many queries read the same selected blocks), so Q K^T over a unit's Q x G query rows is
// a dense contraction.  Same exact softmax over the selected tokens as the one-query
// decode; the output is [B, Q, Hq, D] fp32.
//
// Design (FlashAttention-2 style, tensor cores via mma.sync m16n8k16, bf16 in / fp32
// accumulate):
//   * CTA = (unit, tile of 64 query rows, split of the unit's selected tokens); 4 warps
//     own 16 rows each.  Row r of a unit is (query t = r / G, head g = r % G).
//   * The split's selected tokens are streamed in 64-token K/V tiles through a 3-stage
//     cp.async ring (128-byte XOR swizzle, rows without a token zero-filled); one CTA
//     barrier per tile, amortised over 16 x 64 x D of work per warp.
//   * Per tile and warp: S = Q K^T (8 token groups x D/16 k-steps), the online softmax
//     on the accumulator fragments (row max across the quad), then O += P V with the
//     score fragments reused as the A operand; P is carried as bf16 hi + lo (two MMAs),
//     an fp32 query as bf16 hi + lo too.
//   * Each split writes (m, l, o) per row; the CTA completing a (unit, row tile) merges
//     the splits (log-sum-exp).  One split writes the output directly.
#include "sa_common.cuh"
#include "sa_internal.h"
#include "sa_tcgen05.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

namespace sa {
namespace {

constexpr int kMqThreads = 128;
constexpr int kMqWarps = 4;
constexpr int kMqRows = 64;          // query rows per CTA
constexpr int kMqTile = 64;          // tokens per K/V tile
constexpr int kMqStages = 3;
constexpr int kMqMaxBlocks = 1024;   // page lookups per split held in shared memory
constexpr int kMqMaxSplits = 16;     // token splits of one (unit, row tile)
constexpr int kRowB = 128;           // bytes of one 64-channel half of a token row

struct MqArgs {
    const void* q;
    int q_bf16;
    const void* k_pages;
    const void* v_pages;
    const int32_t* block_table;
    const int32_t* sel_ids;
    const int32_t* sel_count;
    float* out;
    int Hq, Hkv, G, Q, R, nb, bs, N, num_pages, sel_stride;
    int bt_stride;       // block_table row length (capacity in blocks)
    int row_tiles, nsplit, max_splits;
    float scale_log2;
    float* part_m;    // [units * R, max_splits]
    float* part_l;
    float* part_o;    // [units * R, max_splits, D]
    uint32_t* counters;   // [units * row_tiles]
    uint32_t* err;
};

__device__ __forceinline__ uint32_t swz(uint32_t half_base, int token, int chunk)
{
    return half_base + uint32_t(token) * kRowB + uint32_t((chunk ^ (token & 7)) << 4);
}

// The CTA completing a (unit, row tile) merges its splits' (m, l, o) into the output:
// weights per (row, split) once into shared memory, then each output reads its splits'
// partials, eight outputs at a time.
template <int D>
__device__ void mq_merge(const MqArgs& a, int u, int rt)
{
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int b = u / a.Hkv, kvh = u - b * a.Hkv;
    auto head_of = [&](int r) -> size_t {   // q / out row of unit row r
        const int t = r / a.G, g = r - (r / a.G) * a.G;
        return (size_t(b) * a.Q + t) * a.Hq + size_t(kvh) * a.G + g;
    };
    __shared__ float s_w[kMqRows][kMqMaxSplits], s_den[kMqRows];
    const int rows = min(kMqRows, a.R - rt * kMqRows);
    for (int rr = tid; rr < rows; rr += nthr) {
        const size_t pr0 = (size_t(u) * a.R + rt * kMqRows + rr) * a.max_splits;
        float M = -INFINITY;
        for (int s2 = 0; s2 < a.nsplit; ++s2) M = fmaxf(M, __ldcg(a.part_m + pr0 + s2));
        float den = 0.f;
        for (int s2 = 0; s2 < a.nsplit; ++s2) {
            const float ms = __ldcg(a.part_m + pr0 + s2);
            const float w = (ms == -INFINITY || M == -INFINITY) ? 0.f : fast_exp2(ms - M);
            s_w[rr][s2] = w;
            den = fmaf(w, __ldcg(a.part_l + pr0 + s2), den);
        }
        s_den[rr] = den;
    }
    __syncthreads();
    const int n_out = rows * D;
    for (int i0 = tid; i0 < n_out; i0 += nthr * 8) {
        float num[8];
#pragma unroll
        for (int k2 = 0; k2 < 8; ++k2) num[k2] = 0.f;
        for (int s2 = 0; s2 < a.nsplit; ++s2) {
            float v[8];
#pragma unroll
            for (int k2 = 0; k2 < 8; ++k2) {
                const int i = i0 + k2 * nthr;
                const int rr = i / D, d = i - (i / D) * D;
                v[k2] = (i < n_out && s_w[min(rr, kMqRows - 1)][s2] > 0.f)
                            ? __ldcg(a.part_o + ((size_t(u) * a.R + rt * kMqRows + rr) * a.max_splits + s2) * D + d)
                            : 0.f;
            }
#pragma unroll
            for (int k2 = 0; k2 < 8; ++k2) {
                const int i = i0 + k2 * nthr;
                if (i < n_out) num[k2] = fmaf(s_w[i / D][s2], v[k2], num[k2]);
            }
        }
#pragma unroll
        for (int k2 = 0; k2 < 8; ++k2) {
            const int i = i0 + k2 * nthr;
            if (i >= n_out) continue;
            const int rr = i / D, d = i - (i / D) * D;
            const float den = s_den[rr];
            a.out[head_of(rt * kMqRows + rr) * D + d] = den > 0.f ? num[k2] / den : 0.f;
        }
    }
}

template <int D, bool QSPLIT>
__global__ void __launch_bounds__(kMqThreads, 2) decode_mq_kernel(MqArgs a)
{
    constexpr int HALVES = D / 64;
    constexpr int HALF_BYTES = kMqTile * kRowB;               // 8 KB
    constexpr int TENSOR_BYTES = HALVES * HALF_BYTES;
    constexpr int STAGE_BYTES = 2 * TENSOR_BYTES;
    constexpr int DT = D / 8;
    constexpr int CPR = D / 8;                                // 16-byte chunks per token row
    constexpr int CP_PER_THREAD = kMqTile * CPR / kMqThreads;
    static_assert(kMqTile * CPR % kMqThreads == 0, "tile copy must split over the threads");

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g4 = lane >> 2, t4 = lane & 3;
    const int sp = blockIdx.x % a.nsplit;
    const int rt = (blockIdx.x / a.nsplit) % a.row_tiles;
    const int u = blockIdx.x / (a.nsplit * a.row_tiles);
    const int b = u / a.Hkv, kvh = u - b * a.Hkv;
    const int bs_shift = __ffs(a.bs) - 1;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char* smem = smem_raw + (base - raw);
    int* blk_page = reinterpret_cast<int*>(smem + kMqStages * STAGE_BYTES);
    int* blk_valid = blk_page + kMqMaxBlocks;
    __shared__ int s_merge;

    allow_dependents_early();
    grid_dependency_wait();   // inputs and workspace may come from the previous kernel

    // ---- the split's tiles and the blocks they touch --------------------------
    int count = a.sel_count[u];
    if (count < 0 || count > a.sel_stride) {
        if (tid == 0) raise_error(a.err, SPARSE_ATTN_ERR_SEL_COUNT);
        count = count < 0 ? 0 : a.sel_stride;
    }
    const int ntok = count * a.bs;
    const int tiles = (ntok + kMqTile - 1) / kMqTile;
    const int t0 = int((long long)tiles * sp / a.nsplit), t1 = int((long long)tiles * (sp + 1) / a.nsplit);
    const int blk0 = (t0 * kMqTile) >> bs_shift;
    const int blk1 = min(count, ((t1 * kMqTile - 1) >> bs_shift) + 1);
    const int nblk = t1 > t0 ? blk1 - blk0 : 0;
    for (int e = tid; e < nblk; e += kMqThreads) {
        const int slot = blk0 + e;
        int page = -1, valid = 0;
        const int j = a.sel_ids[size_t(u) * a.sel_stride + slot];
        if (j < 0 || j >= a.nb) {
            raise_error(a.err, SPARSE_ATTN_ERR_SEL_ID);
        } else {
            const int p = a.block_table[size_t(b) * a.bt_stride + j];
            if (p < 0 || p >= a.num_pages) {
                raise_error(a.err, SPARSE_ATTN_ERR_PAGE);
            } else {
                page = p;
                valid = min(a.bs, a.N - j * a.bs);
            }
        }
        if (e < kMqMaxBlocks) {
            blk_page[e] = page;
            blk_valid[e] = valid;
        }
    }
    __syncthreads();

    // ---- staging: thread copies chunk cp_c of tile rows cp_r + i * (128 / CPR) -------
    const char* kbase = reinterpret_cast<const char*>(a.k_pages);
    const char* vbase = reinterpret_cast<const char*>(a.v_pages);
    const int cp_c = tid % CPR, cp_r = tid / CPR;
    constexpr int ROWS_PER_PASS = kMqThreads / CPR;
    auto issue_tile = [&](int tile, int st) {
        const uint32_t kd = base + uint32_t(st) * STAGE_BYTES + uint32_t(cp_c >> 3) * HALF_BYTES;
        const uint32_t vd = kd + TENSOR_BYTES;
#pragma unroll
        for (int i = 0; i < CP_PER_THREAD; ++i) {
            const int tr = cp_r + i * ROWS_PER_PASS;                // row in the tile
            const int gi = tile * kMqTile + tr;                     // selected-token index
            const int e = (gi >> bs_shift) - blk0, r = gi & (a.bs - 1);
            const bool ok = gi < ntok && e >= 0 && e < min(nblk, kMqMaxBlocks) && r < blk_valid[max(0, min(e, kMqMaxBlocks - 1))];
            const size_t off = ok ? ((size_t(blk_page[e]) * a.Hkv * a.bs + size_t(kvh) * a.bs + r) * (D * 2) + cp_c * 16) : 0;
            const uint32_t so = uint32_t(tr) * kRowB + uint32_t(((cp_c & 7) ^ (tr & 7)) << 4);
            cp_async_16_zfill(kd + so, kbase + off, ok ? 16u : 0u);
            cp_async_16_zfill(vd + so, vbase + off, ok ? 16u : 0u);
        }
    };
#pragma unroll
    for (int kk = 0; kk < kMqStages - 1; ++kk) {
        if (t0 + kk < t1) issue_tile(t0 + kk, kk);
        cp_async_commit();
    }

    // ---- query A fragments: rows r_lo = row g4, r_hi = row g4 + 8 of the warp ----------
    const int r_lo = rt * kMqRows + warp * 16 + g4, r_hi = r_lo + 8;
    auto head_of = [&](int r) -> size_t {   // q / out row of unit row r
        const int t = r / a.G, g = r - (r / a.G) * a.G;
        return (size_t(b) * a.Q + t) * a.Hq + size_t(kvh) * a.G + g;
    };
    uint32_t qa[D / 16][4], qb[QSPLIT ? D / 16 : 1][4];
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        float f[2][4];
#pragma unroll
        for (int hrow = 0; hrow < 2; ++hrow) {
            const int r = hrow ? r_hi : r_lo;
            const size_t qrow = r < a.R ? head_of(r) * D + ks * 16 + 2 * t4 : 0;
            f[hrow][0] = r < a.R ? load_q(a.q, qrow, a.q_bf16 != 0) : 0.f;
            f[hrow][1] = r < a.R ? load_q(a.q, qrow + 1, a.q_bf16 != 0) : 0.f;
            f[hrow][2] = r < a.R ? load_q(a.q, qrow + 8, a.q_bf16 != 0) : 0.f;
            f[hrow][3] = r < a.R ? load_q(a.q, qrow + 9, a.q_bf16 != 0) : 0.f;
        }
        qa[ks][0] = pack_bf16x2(f[0][0], f[0][1]);
        qa[ks][1] = pack_bf16x2(f[1][0], f[1][1]);
        qa[ks][2] = pack_bf16x2(f[0][2], f[0][3]);
        qa[ks][3] = pack_bf16x2(f[1][2], f[1][3]);
        if constexpr (QSPLIT) {
            qb[ks][0] = pack_bf16x2(f[0][0] - bf16_lo(qa[ks][0]), f[0][1] - bf16_hi(qa[ks][0]));
            qb[ks][1] = pack_bf16x2(f[1][0] - bf16_lo(qa[ks][1]), f[1][1] - bf16_hi(qa[ks][1]));
            qb[ks][2] = pack_bf16x2(f[0][2] - bf16_lo(qa[ks][2]), f[0][3] - bf16_hi(qa[ks][2]));
            qb[ks][3] = pack_bf16x2(f[1][2] - bf16_lo(qa[ks][3]), f[1][3] - bf16_hi(qa[ks][3]));
        }
    }

    float acc[DT][4];
#pragma unroll
    for (int j = 0; j < DT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};   // rows g4, g4 + 8

    for (int tile = t0; tile < t1; ++tile) {
        const int k = tile - t0;
        cp_async_wait_group<kMqStages - 2>();
        __syncthreads();                     // tile k staged by everyone; stage k - 1 is free
        if (tile + kMqStages - 1 < t1) issue_tile(tile + kMqStages - 1, (k + kMqStages - 1) % kMqStages);
        cp_async_commit();
        const uint32_t kst = base + uint32_t(k % kMqStages) * STAGE_BYTES;
        const uint32_t vst = kst + TENSOR_BYTES;

        // S = Q K^T: 8 groups of 8 tokens
        float c[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            c[nt][0] = c[nt][1] = c[nt][2] = c[nt][3] = 0.f;
#pragma unroll
            for (int kp = 0; kp < D / 32; ++kp) {
                const int ch = kp * 4 + (lane >> 3);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(swz(kst + uint32_t(ch >> 3) * HALF_BYTES, nt * 8 + (lane & 7), ch & 7), b0, b1, b2, b3);
                mma_bf16_16816(c[nt], qa[2 * kp][0], qa[2 * kp][1], qa[2 * kp][2], qa[2 * kp][3], b0, b1);
                mma_bf16_16816(c[nt], qa[2 * kp + 1][0], qa[2 * kp + 1][1], qa[2 * kp + 1][2], qa[2 * kp + 1][3], b2, b3);
                if constexpr (QSPLIT) {
                    mma_bf16_16816(c[nt], qb[2 * kp][0], qb[2 * kp][1], qb[2 * kp][2], qb[2 * kp][3], b0, b1);
                    mma_bf16_16816(c[nt], qb[2 * kp + 1][0], qb[2 * kp + 1][1], qb[2 * kp + 1][2], qb[2 * kp + 1][3], b2, b3);
                }
            }
        }
        // online softmax: scale, mask tokens that do not exist, row max over the quad
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int gi = tile * kMqTile + nt * 8 + 2 * t4 + e;
                const int eb = (gi >> bs_shift) - blk0, r = gi & (a.bs - 1);
                const bool ok = gi < ntok && eb >= 0 && eb < min(nblk, kMqMaxBlocks) &&
                                r < blk_valid[max(0, min(eb, kMqMaxBlocks - 1))];
                c[nt][e] = ok ? c[nt][e] * a.scale_log2 : -INFINITY;
                c[nt][e + 2] = ok ? c[nt][e + 2] * a.scale_log2 : -INFINITY;
                mx[0] = fmaxf(mx[0], c[nt][e]);
                mx[1] = fmaxf(mx[1], c[nt][e + 2]);
            }
        float alpha[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(kFullMask, mx[h], 1));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(kFullMask, mx[h], 2));
            const float m_new = fmaxf(m_run[h], mx[h]);
            alpha[h] = (m_run[h] == -INFINITY) ? 0.f : fast_exp2(m_run[h] - m_new);
            m_run[h] = m_new;
        }
        float psum[2] = {0.f, 0.f};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int h = e >> 1;
                c[nt][e] = (c[nt][e] == -INFINITY) ? 0.f : fast_exp2(c[nt][e] - m_run[h]);
                psum[h] += c[nt][e];
            }
        l_run[0] = fmaf(l_run[0], alpha[0], psum[0]);
        l_run[1] = fmaf(l_run[1], alpha[1], psum[1]);
#pragma unroll
        for (int j = 0; j < DT; ++j) {
            acc[j][0] *= alpha[0];
            acc[j][1] *= alpha[0];
            acc[j][2] *= alpha[1];
            acc[j][3] *= alpha[1];
        }
        // O += P V, k = 16 tokens per step; P from the score fragments, bf16 hi + lo
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const float* p0 = c[2 * kk];
            const float* p1 = c[2 * kk + 1];
            const uint32_t h0 = pack_bf16x2(p0[0], p0[1]), h1 = pack_bf16x2(p0[2], p0[3]);
            const uint32_t h2 = pack_bf16x2(p1[0], p1[1]), h3 = pack_bf16x2(p1[2], p1[3]);
            const uint32_t l0 = pack_bf16x2(p0[0] - bf16_lo(h0), p0[1] - bf16_hi(h0));
            const uint32_t l1 = pack_bf16x2(p0[2] - bf16_lo(h1), p0[3] - bf16_hi(h1));
            const uint32_t l2 = pack_bf16x2(p1[0] - bf16_lo(h2), p1[1] - bf16_hi(h2));
            const uint32_t l3 = pack_bf16x2(p1[2] - bf16_lo(h3), p1[3] - bf16_hi(h3));
#pragma unroll
            for (int jp = 0; jp < DT; jp += 2) {
                const int mtx = lane >> 3;
                const int chunk = jp + (mtx >> 1);
                uint32_t r0, r1, r2, r3;
                ldsm_x4_trans(swz(vst + uint32_t(chunk >> 3) * HALF_BYTES, kk * 16 + (mtx & 1) * 8 + (lane & 7), chunk & 7),
                              r0, r1, r2, r3);
                mma_bf16_16816(acc[jp], h0, h1, h2, h3, r0, r1);
                mma_bf16_16816(acc[jp], l0, l1, l2, l3, r0, r1);
                mma_bf16_16816(acc[jp + 1], h0, h1, h2, h3, r2, r3);
                mma_bf16_16816(acc[jp + 1], l0, l1, l2, l3, r2, r3);
            }
        }
    }
    cp_async_wait_group<0>();

    // ---- the split's (m, l, o), or the output itself when there is one split ----------
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        l_run[h] += __shfl_xor_sync(kFullMask, l_run[h], 1);
        l_run[h] += __shfl_xor_sync(kFullMask, l_run[h], 2);
    }
    if (a.nsplit == 1) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = h ? r_hi : r_lo;
            if (r >= a.R) continue;
            const float inv = l_run[h] > 0.f ? 1.f / l_run[h] : 0.f;
            float* dst = a.out + head_of(r) * D + 2 * t4;
#pragma unroll
            for (int j = 0; j < DT; ++j)
                *reinterpret_cast<float2*>(dst + j * 8) = make_float2(acc[j][2 * h] * inv, acc[j][2 * h + 1] * inv);
        }
        return;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int r = h ? r_hi : r_lo;
        if (r >= a.R) continue;
        const size_t pr = (size_t(u) * a.R + r) * a.max_splits + sp;
        float* dst = a.part_o + pr * D + 2 * t4;
#pragma unroll
        for (int j = 0; j < DT; ++j)
            *reinterpret_cast<float2*>(dst + j * 8) = make_float2(acc[j][2 * h], acc[j][2 * h + 1]);
        if (t4 == 0) {
            a.part_m[pr] = m_run[h];
            a.part_l[pr] = l_run[h];
        }
    }
    __syncthreads();
    if (tid == 0) {
        const uint32_t before = atomic_add_acq_rel_u32(&a.counters[size_t(u) * a.row_tiles + rt], 1u);
        s_merge = before + 1 == uint32_t(a.nsplit);
        if (s_merge) a.counters[size_t(u) * a.row_tiles + rt] = 0u;
    }
    __syncthreads();
    if (!s_merge) return;
    mq_merge<D>(a, u, rt);
}

// ------------------------------------------------------------------ tcgen05 ---
// The same attention on the fifth-generation tensor cores (bf16 queries).  Six warps
// with fixed roles; per 64-token tile k of the split:
//   load (warp 4, one thread, running ahead on its own)  the tile's K and V arrive by
//       TMA: one 2-D box (64 channels x up to 64 tokens of one KV head of one page) per
//       selected block and 64-channel half, written with the 128-byte swizzle by the
//       tensor map and counted on the stage's mbarrier; a stage is refilled once the
//       MMAs that read it have completed (a per-stage mbarrier);
//   S(k) = Q K^T (warp 6, one thread)  tcgen05.mma (M = 128, N = 64, K = D) into tensor
//       memory, three S buffers, issued two tiles ahead; A holds the 64 query rows twice
//       (rows r and r + 64), so S lanes 64..127 repeat lanes 0..63;
//   softmax (warps 0-3)  thread = (query row, half of the tile's columns): warps 0-1 take
//       columns 0..31 from lanes 0..63, warps 2-3 columns 32..63 from lanes 64..127; the
//       two halves of a row exchange their maxima through a named barrier, then apply
//       the online softmax with a lazy reference (the maximum used for exp2 moves, and O
//       is rescaled in tensor memory, only when the running maximum grows by more than
//       kLazy, so P <= 2^kLazy) and write P as bf16: hi in row r, the remainder lo in
//       row r + 64 of one 128-row A tile;
//   O += P V (warp 5, one thread)  tcgen05.mma (M = 128, N = D, K = 64), B = the V tile read
//       MN-major; O rows r and r + 64 hold the hi and lo products and add up at the end.
//       Warp 5 also builds each tile's token-validity mask two tiles ahead and zeroes
//       the V rows of tokens that are not selected (a box reads whole blocks).
// The two MMA groups of a tile are issued by two threads at once (each commits its own
// group): O += P(k) V(k) by warp 5 and S(k + 2) by warp 6; S(k) is complete before O(k)
// is issued (the softmax waited for it), so O(k)'s completion frees the stage.  Every
// group completes on an mbarrier (three for S, one for O, one per staging stage for
// loaded and for free) and every wait is bounded; warps 0-3, 5 and 6 meet once per
// tile, the loader never waits on them.
constexpr float kLazy = 8.f;   // log2 growth of the row maximum before O is rescaled
constexpr int kTcThreads = 224;

template <int D>
struct MqTcShape {
    static constexpr int T = 64;                            // tokens per tile
    static constexpr int HALVES = D / 64;
    static constexpr int KV_HALF = T * kRowB;               // 8 KB: 64 tokens x 128 B
    static constexpr int KV_TENSOR = HALVES * KV_HALF;
    static constexpr int STAGE_BYTES = 2 * KV_TENSOR;       // K then V
    static constexpr int STAGES = 4;
    static constexpr int Q_HALF = 128 * kRowB;              // 128 rows x 128 B
    static constexpr int Q_BYTES = HALVES * Q_HALF;
    static constexpr int P_BYTES = 128 * kRowB;             // 128 rows x 64 tokens bf16
    static constexpr int OFF_Q = 0, OFF_P = Q_BYTES;
    static constexpr int OFF_KV = OFF_P + P_BYTES;
    static constexpr int OFF_BLK = OFF_KV + STAGES * STAGE_BYTES;
    static constexpr size_t SMEM = 1024 + size_t(OFF_BLK) + size_t(2) * kMqMaxBlocks * sizeof(int);
};

__device__ __forceinline__ void named_barrier(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    decode_mq_tc_kernel(MqArgs a, const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        int box_rows)
{
    using SH = MqTcShape<D>;
    constexpr int T = SH::T, STAGES = SH::STAGES;
    constexpr int CPR = D / 8;                              // 16-byte chunks per token row
    constexpr uint32_t S_COL = 0, O_COL = 256, TMEM_COLS = 512;   // S buffers at 0, 64, 128
    constexpr uint32_t IDESC_S = idesc_bf16_f32(128, T, false);
    constexpr uint32_t IDESC_O = idesc_bf16_f32(128, D, true);
    static_assert(O_COL + D <= TMEM_COLS, "S and O must fit the allocation");
    constexpr int LOADER = 4 * 32, ISSUER = 5 * 32, ISSUER_S = 6 * 32;   // single-thread roles

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sp = blockIdx.x % a.nsplit;
    const int rt = (blockIdx.x / a.nsplit) % a.row_tiles;
    const int u = blockIdx.x / (a.nsplit * a.row_tiles);
    const int b = u / a.Hkv, kvh = u - b * a.Hkv;
    const int bs_shift = __ffs(a.bs) - 1;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;           // swizzle atoms: 1024-byte aligned
    unsigned char* smem = smem_raw + (base - raw);
    int* blk_page = reinterpret_cast<int*>(smem + SH::OFF_BLK);
    int* blk_valid = blk_page + kMqMaxBlocks;
    __shared__ __align__(8) uint64_t bar_s[3], bar_o, bar_kv[STAGES], bar_free[STAGES];
    __shared__ uint32_t s_tmem;
    __shared__ uint32_t s_mask[3][2];                        // valid tokens of a tile (64 bits)
    __shared__ float s_mx[2][64];                            // per-half row maxima
    __shared__ float s_l[64];                                // row sums of the second half
    __shared__ int s_merge;

    allow_dependents_early();
    grid_dependency_wait();   // inputs and workspace may come from the previous kernel

    if (warp == 0) {
        tmem_alloc(&s_tmem, TMEM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bar_s[i], 1);
        mbar_init(&bar_o, 1);
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&bar_kv[i], 1);
            mbar_init(&bar_free[i], 1);
        }
        fence_mbar_init();
    }

    // ---- the split's tiles and the blocks they touch --------------------------
    int count = a.sel_count[u];
    if (count < 0 || count > a.sel_stride) {
        if (tid == 0) raise_error(a.err, SPARSE_ATTN_ERR_SEL_COUNT);
        count = count < 0 ? 0 : a.sel_stride;
    }
    const int ntok = count * a.bs;
    const int tiles = (ntok + T - 1) / T;
    const int t0 = int((long long)tiles * sp / a.nsplit), t1 = int((long long)tiles * (sp + 1) / a.nsplit);
    const int blk0 = (t0 * T) >> bs_shift;
    const int blk1 = min(count, ((t1 * T - 1) >> bs_shift) + 1);
    const int nblk = t1 > t0 ? blk1 - blk0 : 0;
    for (int e = tid; e < nblk; e += kTcThreads) {
        const int slot = blk0 + e;
        int page = -1, valid = 0;
        const int j = a.sel_ids[size_t(u) * a.sel_stride + slot];
        if (j < 0 || j >= a.nb) {
            raise_error(a.err, SPARSE_ATTN_ERR_SEL_ID);
        } else {
            const int p = a.block_table[size_t(b) * a.bt_stride + j];
            if (p < 0 || p >= a.num_pages) {
                raise_error(a.err, SPARSE_ATTN_ERR_PAGE);
            } else {
                page = p;
                valid = min(a.bs, a.N - j * a.bs);
            }
        }
        if (e < kMqMaxBlocks) {
            blk_page[e] = page;
            blk_valid[e] = valid;
        }
    }

    // ---- query rows 0..63 of the tile (zero past R), repeated in rows 64..127 --------
    auto head_of = [&](int r) -> size_t {   // q / out row of unit row r
        const int t = r / a.G, g = r - (r / a.G) * a.G;
        return (size_t(b) * a.Q + t) * a.Hq + size_t(kvh) * a.G + g;
    };
    for (int i = tid; i < 64 * CPR; i += kTcThreads) {
        const int row = i / CPR, c = i - (i / CPR) * CPR;
        const int r = rt * kMqRows + row;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r < a.R) v = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.q) + head_of(r) * D) + c);
        const int off = (c >> 3) * SH::Q_HALF + (((c & 7) ^ (row & 7)) << 4);
        *reinterpret_cast<uint4*>(smem + SH::OFF_Q + off + row * kRowB) = v;
        *reinterpret_cast<uint4*>(smem + SH::OFF_Q + off + (row + 64) * kRowB) = v;
    }
    fence_proxy_async_smem();   // Q, before the tensor core reads it
    tc_fence_before_sync();
    __syncthreads();            // page lookups, barriers and tensor memory ready
    tc_fence_after_sync();
    const uint32_t tmem = s_tmem;

    auto token_ok = [&](int gi) -> bool {
        const int e = (gi >> bs_shift) - blk0, r = gi & (a.bs - 1);
        return gi < ntok && e >= 0 && e < min(nblk, kMqMaxBlocks) && r < blk_valid[max(0, min(e, kMqMaxBlocks - 1))];
    };
    auto box_ok = [&](int gi) -> bool {
        const int e = (gi >> bs_shift) - blk0;
        return gi < ntok && e >= 0 && e < min(nblk, kMqMaxBlocks) && blk_page[e] >= 0;
    };
    // the loader thread: the tile's boxes into stage st, counted on bar_kv[st]
    auto load_tile = [&](int tile, int st) {
        const uint32_t kst = base + SH::OFF_KV + uint32_t(st) * SH::STAGE_BYTES;
        const int g0 = tile * T;
        uint32_t bytes = 0;
        for (int r0 = 0; r0 < T; r0 += box_rows)
            if (box_ok(g0 + r0)) bytes += uint32_t(box_rows) * kRowB * SH::HALVES * 2;
        mbar_arrive_expect_tx(&bar_kv[st], bytes);
        for (int r0 = 0; r0 < T; r0 += box_rows) {
            const int gi = g0 + r0;
            if (!box_ok(gi)) continue;
            const int e = (gi >> bs_shift) - blk0;
            const int y = (blk_page[e] * a.Hkv + kvh) * a.bs + (gi & (a.bs - 1));
#pragma unroll
            for (int h = 0; h < SH::HALVES; ++h) {
                const uint32_t off = uint32_t(h) * SH::KV_HALF + uint32_t(r0) * kRowB;
                tma_load_2d(smem + (kst - base) + off, &kmap, h * 64, y, &bar_kv[st]);
                tma_load_2d(smem + (kst - base) + SH::KV_TENSOR + off, &vmap, h * 64, y, &bar_kv[st]);
            }
        }
    };
    // warp 5: 64-bit validity mask of a tile (two tokens per lane)
    auto write_mask = [&](int k) {
        const int g0 = (t0 + k) * T;
        const uint32_t m0 = __ballot_sync(kFullMask, token_ok(g0 + lane));
        const uint32_t m1 = __ballot_sync(kFullMask, token_ok(g0 + 32 + lane));
        if (lane == 0) {
            s_mask[k % 3][0] = m0;
            s_mask[k % 3][1] = m1;
        }
    };
    // Descriptors differ from their operand's base only in the start-address field
    // (bits 0-13, in 16-byte units); every operand lies in this CTA's shared memory, so
    // adding an offset >> 4 never carries out of the field.
    const uint64_t q_desc = smem_desc_sw128(base + SH::OFF_Q, 16, 1024);
    const uint64_t p_desc = smem_desc_sw128(base + SH::OFF_P, 16, 1024);
    const uint64_t k_desc0 = smem_desc_sw128(base + SH::OFF_KV, 16, 1024);
    const uint64_t v_desc0 = smem_desc_sw128(base + SH::OFF_KV + SH::KV_TENSOR, SH::KV_HALF, 1024);
    auto issue_s = [&](int k) {   // S(k) = Q K^T into S buffer k mod 3
        const uint64_t kd = k_desc0 + uint64_t((uint32_t(k % STAGES) * SH::STAGE_BYTES) >> 4);
        const uint32_t d_tmem = tmem + S_COL + uint32_t(k % 3) * T;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = uint32_t(ks & 3) * 32;
            umma_bf16(d_tmem, q_desc + ((uint32_t(ks >> 2) * SH::Q_HALF + off) >> 4),
                      kd + ((uint32_t(ks >> 2) * SH::KV_HALF + off) >> 4), IDESC_S, ks > 0 ? 1u : 0u);
        }
        umma_commit(&bar_s[k % 3]);
    };
    auto issue_o = [&](int k) {   // O += P(k) V(k), P hi in rows 0..63 and lo in rows 64..127
        const uint64_t vd = v_desc0 + uint64_t((uint32_t(k % STAGES) * SH::STAGE_BYTES) >> 4);
#pragma unroll
        for (int kk = 0; kk < T / 16; ++kk)
            umma_bf16(tmem + O_COL, p_desc + ((uint32_t(kk) * 32) >> 4), vd + ((uint32_t(kk) * 16 * kRowB) >> 4), IDESC_O,
                      (k > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&bar_o);
        umma_commit(&bar_free[k % STAGES]);   // stage k mod STAGES may be refilled
    };
    auto wait_kv = [&](int k) {   // tile k's boxes have landed
        if (!mbar_wait_bounded(&bar_kv[k % STAGES], uint32_t(k / STAGES) & 1u, kWaitCycles))
            raise_error(a.err, SPARSE_ATTN_ERR_TIMEOUT);
    };

    const int ntiles = t1 - t0;
    if (tid == LOADER)
        for (int k = 0; k < STAGES - 1 && k < ntiles; ++k) load_tile(t0 + k, k);
    if (warp == 5) {
        if (ntiles > 0) write_mask(0);
        if (ntiles > 1) write_mask(1);
    }
    if (tid == ISSUER_S) {
        for (int k = 0; k < 2 && k < ntiles; ++k) {
            wait_kv(k);
            issue_s(k);
        }
    }
    __syncthreads();   // masks of tiles 0 and 1

    const uint32_t lane_base = uint32_t(32 * (warp & 3)) << 16;   // this warp's tensor-memory lanes
    const int row = (32 * warp + lane) & 63;                      // softmax warps: the query row
    const int half = warp >> 1;                                  // softmax warps: column half
    float m_ref = -INFINITY, l_run = 0.f;                        // reference maximum, half-row sum
    for (int k = 0; k < ntiles; ++k) {
        if (warp < 4) {
            if (!mbar_wait_bounded(&bar_s[k % 3], uint32_t(k / 3) & 1u, kWaitCycles))
                raise_error(a.err, SPARSE_ATTN_ERR_TIMEOUT);
            tc_fence_after_sync();
            uint32_t sv[32];
            tmem_ld32(tmem + lane_base + S_COL + uint32_t(k % 3) * T + uint32_t(half) * 32, sv);
            tmem_wait_ld();
            const uint32_t mk = s_mask[k % 3][half];
            float x[32];
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                x[j] = ((mk >> j) & 1u) ? __uint_as_float(sv[j]) * a.scale_log2 : -INFINITY;
                mx = fmaxf(mx, x[j]);
            }
            s_mx[half][row] = mx;
            named_barrier(1 + (warp & 1), 64);   // the other half of these rows
            mx = fmaxf(s_mx[0][row], s_mx[1][row]);
            bool rescale = false;
            float alpha = 1.f;
            if (mx > m_ref + kLazy || (m_ref == -INFINITY && mx != -INFINITY)) {
                alpha = m_ref == -INFINITY ? 0.f : fast_exp2(m_ref - mx);
                m_ref = mx;
                rescale = true;
            }
            // O += P(k - 1) V(k - 1) is done: P and O are free
            if (k > 0 && !mbar_wait_bounded(&bar_o, uint32_t(k - 1) & 1u, kWaitCycles))
                raise_error(a.err, SPARSE_ATTN_ERR_TIMEOUT);
            tc_fence_after_sync();
            if (k > 0 && __any_sync(kFullMask, rescale)) {   // this warp's O rows (lazy)
                const float al = rescale ? alpha : 1.f;
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t ov[32];
                    tmem_ld32(tmem + lane_base + O_COL + c0, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * al);
                    tmem_st32(tmem + lane_base + O_COL + c0, ov);
                }
                tmem_wait_st();
            }
            if (rescale) l_run *= alpha;
            float psum = 0.f;
            unsigned char* ph = smem + SH::OFF_P + row * kRowB;
            unsigned char* pl = smem + SH::OFF_P + (row + 64) * kRowB;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    const int j = c * 8 + 2 * e2;
                    const float p0 = x[j] == -INFINITY ? 0.f : fast_exp2(x[j] - m_ref);
                    const float p1 = x[j + 1] == -INFINITY ? 0.f : fast_exp2(x[j + 1] - m_ref);
                    psum += p0 + p1;
                    hw[e2] = pack_bf16x2(p0, p1);
                    lw[e2] = pack_bf16x2(p0 - bf16_lo(hw[e2]), p1 - bf16_hi(hw[e2]));
                }
                const int slot = ((half * 4 + c) ^ (row & 7)) << 4;   // row and row + 64 share row & 7
                *reinterpret_cast<uint4*>(ph + slot) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4*>(pl + slot) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
            l_run += psum;
            fence_proxy_async_smem();   // P(k), before the tensor core reads it
        } else if (warp == 5) {
            if (k + 2 < ntiles) write_mask(k + 2);
            // zero V rows of tile k whose token is not selected (boxes read whole blocks)
            const uint32_t m0 = s_mask[k % 3][0], m1 = s_mask[k % 3][1];
            if ((m0 & m1) != 0xffffffffu) {
                wait_kv(k);
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    if (((hr ? m1 : m0) >> lane) & 1u) continue;
                    const int tr = hr * 32 + lane;
#pragma unroll
                    for (int h = 0; h < SH::HALVES; ++h)
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            *reinterpret_cast<uint4*>(smem + SH::OFF_KV + (k % STAGES) * SH::STAGE_BYTES + SH::KV_TENSOR +
                                                      h * SH::KV_HALF + tr * kRowB + c * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
        } else if (warp == 4) {
            // the loader: tile k + STAGES - 1 into the stage tile k - 1 used, once the
            // MMAs reading it are done
            if (tid == LOADER && k + STAGES - 1 < ntiles) {
                if (k > 0 && !mbar_wait_bounded(&bar_free[(k - 1) % STAGES], uint32_t((k - 1) / STAGES) & 1u, kWaitCycles))
                    raise_error(a.err, SPARSE_ATTN_ERR_TIMEOUT);
                load_tile(t0 + k + STAGES - 1, (k + STAGES - 1) % STAGES);
            }
            continue;   // the loader does not meet the others
        }
        tc_fence_before_sync();
        named_barrier(3, kTcThreads - 32);   // warps 0-3, 5 and 6
        tc_fence_after_sync();
        if (tid == ISSUER) {
            wait_kv(k);        // already complete: the tensor core reads V(k) after this thread saw it land
            issue_o(k);
        } else if (tid == ISSUER_S && k + 2 < ntiles) {
            wait_kv(k + 2);
            issue_s(k + 2);
        }
    }
    if (ntiles > 0 && !mbar_wait_bounded(&bar_o, uint32_t(ntiles - 1) & 1u, kWaitCycles))
        raise_error(a.err, SPARSE_ATTN_ERR_TIMEOUT);
    tc_fence_after_sync();

    // ---- epilogue: O[r] + O[r + 64], the lo rows and second-half sums via shared memory ----
    float* lo_rows = reinterpret_cast<float*>(smem + SH::OFF_KV);   // [64][D], the free ring
    if (warp == 2 || warp == 3) {
        s_l[row] = l_run;
        if (ntiles > 0) {
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t ov[32];
                tmem_ld32(tmem + lane_base + O_COL + c0, ov);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) lo_rows[row * D + ((c0 + j + lane) & (D - 1))] = __uint_as_float(ov[j]);
            }
        }
    }
    __syncthreads();
    const int r_unit = rt * kMqRows + row;
    if (warp < 2) {
        const float lsum = l_run + s_l[row];
        const bool have = r_unit < a.R;
        float* dst = nullptr;
        float inv = 1.f;
        if (have) {
            if (a.nsplit == 1) {
                dst = a.out + head_of(r_unit) * D;
                inv = lsum > 0.f ? 1.f / lsum : 0.f;
            } else {
                const size_t pr = (size_t(u) * a.R + r_unit) * a.max_splits + sp;
                dst = a.part_o + pr * D;
                a.part_m[pr] = m_ref;
                a.part_l[pr] = lsum;
            }
        }
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t ov[32];
            if (ntiles > 0) {
                tmem_ld32(tmem + lane_base + O_COL + c0, ov);
                tmem_wait_ld();
            }
            if (have) {
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    float o4[4];
#pragma unroll
                    for (int e2 = 0; e2 < 4; ++e2) {
                        const int d = c0 + j + e2;
                        o4[e2] = ntiles > 0 ? (__uint_as_float(ov[j + e2]) + lo_rows[row * D + ((d + lane) & (D - 1))]) * inv
                                            : 0.f;
                    }
                    *reinterpret_cast<float4*>(dst + c0 + j) = make_float4(o4[0], o4[1], o4[2], o4[3]);
                }
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
    if (a.nsplit == 1) return;
    if (tid == 0) {
        const uint32_t before = atomic_add_acq_rel_u32(&a.counters[size_t(u) * a.row_tiles + rt], 1u);
        s_merge = before + 1 == uint32_t(a.nsplit);
        if (s_merge) a.counters[size_t(u) * a.row_tiles + rt] = 0u;
    }
    __syncthreads();
    if (!s_merge) return;
    mq_merge<D>(a, u, rt);
}

// A 2-D tensor map over a page pool viewed as [num_pages * Hkv * bs rows, D bf16]: boxes
// of 64 channels x box_rows tokens, 128-byte swizzle (the layout the MMAs read).
inline cudaError_t encode_pool_map(CUtensorMap* map, const void* pool, int D, long long rows, int box_rows)
{
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
            return cudaErrorNotSupported;
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const cuuint64_t dims[2] = {cuuint64_t(D), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(D) * 2};
    const cuuint32_t box[2] = {64u, cuuint32_t(box_rows)};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D>
cudaError_t launch_mq_tc_t(const MqArgs& a, int units, int num_pages, cudaStream_t s)
{
    const size_t smem = MqTcShape<D>::SMEM;
    static std::atomic<unsigned long long> configured{0};   // devices set up
    const cudaError_t cfg = once_per_device(configured, [&]() -> cudaError_t {
        return cudaFuncSetAttribute(decode_mq_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(smem));
    });
    if (cfg != cudaSuccess) return cfg;
    const int box_rows = a.bs < MqTcShape<D>::T ? a.bs : MqTcShape<D>::T;
    const long long rows = (long long)num_pages * a.Hkv * a.bs;
    CUtensorMap kmap, vmap;
    cudaError_t e = encode_pool_map(&kmap, a.k_pages, D, rows, box_rows);
    if (e != cudaSuccess) return e;
    e = encode_pool_map(&vmap, a.v_pages, D, rows, box_rows);
    if (e != cudaSuccess) return e;
    const unsigned grid = unsigned(size_t(units) * a.row_tiles * a.nsplit);
    return launch_after_previous(decode_mq_tc_kernel<D>, dim3(grid), dim3(kTcThreads), smem, s, a, kmap, vmap, box_rows);
}

template <int D, bool QSPLIT>
cudaError_t launch_mq_t(const MqArgs& a, int units, cudaStream_t s)
{
    constexpr int STAGE_BYTES = 2 * (D / 64) * kMqTile * kRowB;
    constexpr size_t smem = 1024 + size_t(kMqStages) * STAGE_BYTES + size_t(2) * kMqMaxBlocks * sizeof(int);
    static std::atomic<unsigned long long> configured{0};   // devices set up
    const cudaError_t cfg = once_per_device(configured, [&]() -> cudaError_t {
        return cudaFuncSetAttribute(decode_mq_kernel<D, QSPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(smem));
    });
    if (cfg != cudaSuccess) return cfg;
    const unsigned grid = unsigned(size_t(units) * a.row_tiles * a.nsplit);
    return launch_after_previous(decode_mq_kernel<D, QSPLIT>, dim3(grid), dim3(kMqThreads), smem, s, a);
}

}  // namespace

int mq_row_tiles(int Q, int G) { return (Q * G + kMqRows - 1) / kMqRows; }

cudaError_t launch_decode_mq(const Geometry& g, const WorkspaceLayout& L, char* ws, const void* q,
                             const void* k_pages, const void* v_pages, const int32_t* block_table,
                             const int32_t* sel_ids, const int32_t* sel_count, float* out, cudaStream_t s)
{
    const int units = g.units();
    if (units == 0) return cudaSuccess;
    MqArgs a{};
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
    a.G = g.G;
    a.Q = g.Q;
    a.R = g.Q * g.G;
    a.nb = g.nb;
    a.bs = g.bs;
    a.N = g.N;
    a.num_pages = g.num_pages;
    a.bt_stride = g.nb_cap;
    a.sel_stride = g.sel_stride;
    a.row_tiles = mq_row_tiles(g.Q, g.G);
    a.max_splits = L.max_splits;
    // splits of the selected tokens: about two CTAs per SM, at least enough for each
    // split's blocks to fit the page cache, at most the workspace's partial slots
    const int tiles = (g.sel_stride * g.bs + kMqTile - 1) / kMqTile;
    const long long cells = (long long)units * a.row_tiles;
    // bf16 queries run on tcgen05 (one CTA per SM: at most one wave of splits); fp32
    // queries on mma.sync (two CTAs per SM)
    const bool tc = g.q_bf16 != 0;
    long long ns = tc ? (num_sms() >= cells ? num_sms() / cells : 1) : (2LL * num_sms() + cells - 1) / cells;
    const long long ns_min = (g.sel_stride + (kMqMaxBlocks - 16) - 1) / (kMqMaxBlocks - 16);
    if (ns < ns_min) ns = ns_min;
    if (ns > tiles) ns = tiles > 0 ? tiles : 1;
    if (ns > L.max_splits) ns = L.max_splits;
    if (ns > kMqMaxSplits) ns = kMqMaxSplits;
    if (ns < ns_min) return cudaErrorInvalidValue;   // the workspace cannot hold enough splits
    a.nsplit = int(ns);
    a.scale_log2 = g.scale_log2;
    a.part_m = reinterpret_cast<float*>(ws + L.part_m);
    a.part_l = reinterpret_cast<float*>(ws + L.part_l);
    a.part_o = reinterpret_cast<float*>(ws + L.part_o);
    a.counters = reinterpret_cast<uint32_t*>(ws + L.dec_counters);
    a.err = reinterpret_cast<uint32_t*>(ws + L.err);
    if (tc) return g.D == 128 ? launch_mq_tc_t<128>(a, units, g.num_pages, s) : launch_mq_tc_t<64>(a, units, g.num_pages, s);
    return g.D == 128 ? launch_mq_t<128, true>(a, units, s) : launch_mq_t<64, true>(a, units, s);
}

}  // namespace sa
