// Sparse decode attention over the selected blocks only.
//
// "从HiSparse到QSA的移植实战" §3.3: the attention kernel walks a compact array of selected
// block indices and never reads unselected KV; HBM bandwidth is the bound.  SparDA page
// (www.2kiu.com/news/4656707) §5.3: skip unselected pages inside the kernel rather than
// gathering them into a temporary buffer first.  The softmax is exact over the union of
// the selected tokens (SGLang page §1.2 "select-then-compute").
//
// Design (one CTA = one split of one (sequence, KV head) unit, all G query heads):
//   1. read this split's slice of sel_ids, map block -> page through block_table;
//   2. one thread issues 1-D bulk async copies (cp.async.bulk) of each selected
//      (page, KV head) K tile and V tile -- each tile is block_size x D contiguous -- into
//      shared memory, completing on two mbarriers (K first, so QK^T overlaps the V copy);
//   3. QK^T in fp32: a key row is covered by LPR lanes with one 16-byte shared load each;
//      per-row partial dots of all G heads are summed across the row's lanes with the
//      transposed halving reduction;
//   4. per-head max / exp2 / sum for the split (scores pre-scaled by scale*log2 e);
//   5. PV in fp32: lanes own D-slices, warps own tokens, reduced through shared memory;
//   6. write the split's (m, l, o) partial; the CTA finishing a unit last merges the
//      unit's partials (log-sum-exp) and writes fp32 outputs.  No CTA waits on another.
// GQA tiles are G x tokens: far too narrow for a tensor-core tile to pay (>= 64 rows), and
// the kernel is HBM-bound at ~2 FMA per byte, so the contraction stays on FMA units.
#include "sa_common.cuh"
#include "sa_internal.h"

namespace sa {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kStageBytes = 64 * 1024;   // K + V tiles staged per CTA
constexpr int kMaxBlocksPerSplit = 32;   // 256 tokens / 8-token blocks

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
    int blocks_per_split, max_splits;
    float scale_log2;
    float* part_m;   // [B*Hq, max_splits]
    float* part_l;
    float* part_o;   // [B*Hq, max_splits, D]
    uint32_t* counters;
    uint32_t* err;
};

template <int D, bool BF16>
struct DecodeShape {
    static constexpr int ESZ = BF16 ? 2 : 4;
    static constexpr int EPL = 16 / ESZ;
    static constexpr int LPR = D / EPL;
    static constexpr int RPW = 32 / LPR;
    static constexpr int TPS = kStageBytes / (2 * D * ESZ);   // tokens per split
    static constexpr int ROW_BYTES = D * ESZ;
};

template <int D, bool BF16, int G>
__global__ void __launch_bounds__(kDecThreads, 2) decode_kernel(DecodeArgs a)
{
    using S = DecodeShape<D, BF16>;
    constexpr int EPL = S::EPL, LPR = S::LPR, RPW = S::RPW, TPS = S::TPS;
    constexpr int R = (16 / G) < (TPS / (kDecWarps * RPW)) ? (16 / G) : (TPS / (kDecWarps * RPW));
    constexpr int V = R * G;                        // partial dots per lane per batch
    constexpr int ROWS_PER_BATCH = kDecWarps * RPW * R;
    static_assert(TPS % ROWS_PER_BATCH == 0, "token tile must split evenly");
    static_assert(8 * G * D * 4 <= TPS * S::ROW_BYTES, "reduction buffer must fit the K region");

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* k_s = smem;
    unsigned char* v_s = smem + TPS * S::ROW_BYTES;
    float* s_s = reinterpret_cast<float*>(v_s + TPS * S::ROW_BYTES);   // [G][TPS]
    float* p_s = s_s + G * TPS;                                       // [TPS][G]
    __shared__ __align__(8) uint64_t bar_k, bar_v;
    __shared__ int blk_page[kMaxBlocksPerSplit];
    __shared__ int blk_valid[kMaxBlocksPerSplit];     // valid tokens per staged block
    __shared__ int s_nblk, s_count;
    __shared__ float s_m[G], s_l[G];
    __shared__ bool s_last;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int splits = a.max_splits;
    const int u = blockIdx.x / splits;
    const int split = blockIdx.x - u * splits;
    const int b = u / a.Hkv, kvh = u - b * a.Hkv;
    const int bps = a.blocks_per_split;

    // ---- 1. this split's blocks ---------------------------------------
    if (tid == 0) {
        int count = a.sel_count[u];
        if (count < 0 || count > a.sel_stride) {
            raise_error(a.err, SPARSE_ATTN_ERR_SEL_COUNT);
            count = count < 0 ? 0 : a.sel_stride;
        }
        s_count = count;
        const int first = split * bps;
        int n = min(bps, count - first);
        if (n < 0) n = 0;
        s_nblk = n;
        mbar_init(&bar_k, 1);
        mbar_init(&bar_v, 1);
        fence_mbar_init();
    }
    __syncthreads();
    const int nblk = s_nblk;
    if (tid < bps) {
        int page = -1, valid = 0;
        if (tid < nblk) {
            const int j = a.sel_ids[size_t(u) * a.sel_stride + split * bps + tid];
            if (j < 0 || j >= a.nb) {
                raise_error(a.err, SPARSE_ATTN_ERR_SEL_ID);
            } else {
                const int p = a.block_table[size_t(b) * a.nb + j];
                if (p < 0 || p >= a.num_pages) {
                    raise_error(a.err, SPARSE_ATTN_ERR_PAGE);
                } else {
                    page = p;
                    valid = min(a.bs, a.N - j * a.bs);
                }
            }
        }
        blk_page[tid] = page;
        blk_valid[tid] = valid;
    }
    __syncthreads();

    if (nblk > 0) {
        // ---- 2. stage K and V tiles --------------------------------------
        const uint32_t tile_bytes = uint32_t(a.bs) * S::ROW_BYTES;
        if (tid == 0) {
            uint32_t nbytes = 0;
            for (int i = 0; i < nblk; ++i) nbytes += blk_page[i] >= 0 ? tile_bytes : 0u;
            const size_t head_off = size_t(kvh) * tile_bytes;
            const size_t page_stride = size_t(a.Hkv) * tile_bytes;
            mbar_arrive_expect_tx(&bar_k, nbytes);
            for (int i = 0; i < nblk; ++i)
                if (blk_page[i] >= 0)
                    bulk_copy_g2s(k_s + size_t(i) * tile_bytes,
                                  reinterpret_cast<const char*>(a.k_pages) + blk_page[i] * page_stride + head_off,
                                  tile_bytes, &bar_k);
            mbar_arrive_expect_tx(&bar_v, nbytes);
            for (int i = 0; i < nblk; ++i)
                if (blk_page[i] >= 0)
                    bulk_copy_g2s(v_s + size_t(i) * tile_bytes,
                                  reinterpret_cast<const char*>(a.v_pages) + blk_page[i] * page_stride + head_off,
                                  tile_bytes, &bar_v);
        }

        // q for this lane's channels, pre-scaled into the log2 domain
        const int sub = lane % LPR, rsub = lane / LPR;
        float qr[G][EPL];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const size_t qrow = (size_t(b) * a.Hq + size_t(kvh) * G + g) * D + sub * EPL;
#pragma unroll
            for (int e = 0; e < EPL; ++e) qr[g][e] = load_q(a.q, qrow + e, a.q_bf16 != 0) * a.scale_log2;
        }

        if (!mbar_wait_bounded(&bar_k, 0, kWaitCycles)) raise_error(a.err, SPARSE_ATTN_ERR_TIMEOUT);

        // ---- 3. S = q K^T for the staged tokens ----------------------------
        const int ntok = nblk * a.bs;
        for (int t_base = 0; t_base < ntok; t_base += ROWS_PER_BATCH) {
            const int t0 = t_base + ((warp * RPW) + rsub) * R;
            float v[V];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float kf[EPL];
                unpack16<BF16>(*reinterpret_cast<const uint4*>(k_s + size_t(t0 + r) * S::ROW_BYTES + sub * 16), kf);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float acc = 0.f;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) acc = fmaf(qr[g][e], kf[e], acc);
                    v[r * G + g] = acc;
                }
            }
            group_reduce_transposed<V, LPR>(v, lane);
            if constexpr (V >= LPR) {
#pragma unroll
                for (int i = 0; i < V / LPR; ++i) {
                    const int idx = sub * (V / LPR) + i;
                    const int r = idx / G, g = idx - (idx / G) * G;
                    const int t = t0 + r;
                    const int blk = t / a.bs;
                    const bool ok = t < ntok && (t - blk * a.bs) < blk_valid[blk];
                    s_s[g * TPS + t] = ok ? v[i] : -INFINITY;
                }
            } else {
                if (sub % (LPR / V) == 0) {
                    const int idx = sub / (LPR / V);
                    const int r = idx / G, g = idx - (idx / G) * G;
                    const int t = t0 + r;
                    const int blk = t / a.bs;
                    const bool ok = t < ntok && (t - blk * a.bs) < blk_valid[blk];
                    s_s[g * TPS + t] = ok ? v[0] : -INFINITY;
                }
            }
        }
        __syncthreads();

        // ---- 4. per-head split softmax statistics ---------------------------
        for (int g = warp; g < G; g += kDecWarps) {
            float m = -INFINITY;
            for (int t = lane; t < ntok; t += 32) m = fmaxf(m, s_s[g * TPS + t]);
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFullMask, m, off));
            float l = 0.f;
            for (int t = lane; t < ntok; t += 32) {
                const float x = s_s[g * TPS + t];
                const float p = (m == -INFINITY || x == -INFINITY) ? 0.f : fast_exp2(x - m);
                p_s[t * G + g] = p;
                l += p;
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) l += __shfl_xor_sync(kFullMask, l, off);
            if (lane == 0) { s_m[g] = m; s_l[g] = l; }
        }
        if (!mbar_wait_bounded(&bar_v, 0, kWaitCycles)) raise_error(a.err, SPARSE_ATTN_ERR_TIMEOUT);
        __syncthreads();

        // ---- 5. O = P V ------------------------------------------------------
        float acc[G][EPL];
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[g][e] = 0.f;
        for (int t = warp * RPW + rsub; t < ntok; t += kDecWarps * RPW) {
            const int blk = t / a.bs;
            if ((t - blk * a.bs) >= blk_valid[blk]) continue;
            float vf[EPL];
            unpack16<BF16>(*reinterpret_cast<const uint4*>(v_s + size_t(t) * S::ROW_BYTES + sub * 16), vf);
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
#pragma unroll
        for (int m = LPR; m < 32; m <<= 1)
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc[g][e] += __shfl_xor_sync(kFullMask, acc[g][e], m);
        float* red = reinterpret_cast<float*>(k_s);   // K tiles are no longer needed
        if (rsub == 0) {
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int e = 0; e < EPL; ++e) red[(warp * G + g) * D + sub * EPL + e] = acc[g][e];
        }
        __syncthreads();

        // ---- 6. split partial -------------------------------------------------
        const size_t head0 = size_t(b) * a.Hq + size_t(kvh) * G;
        for (int i = tid; i < G * D; i += kDecThreads) {
            const int g = i / D, d = i - g * D;
            float o = 0.f;
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) o += red[(w * G + g) * D + d];
            a.part_o[((head0 + g) * splits + split) * D + d] = o;
        }
        if (tid < G) {
            a.part_m[(head0 + tid) * splits + split] = s_m[tid];
            a.part_l[(head0 + tid) * splits + split] = s_l[tid];
        }
    }

    // ---- merge, by whichever CTA completes this unit last ----------------------
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(&a.counters[u], 1u) == uint32_t(splits - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (tid == 0) a.counters[u] = 0u;
    const int used = (s_count + bps - 1) / bps;
    const size_t head0 = size_t(b) * a.Hq + size_t(kvh) * G;
    for (int i = tid; i < G * D; i += kDecThreads) {
        const int g = i / D, d = i - g * D;
        const size_t h = head0 + g;
        float mx = -INFINITY;
        for (int sp = 0; sp < used; ++sp) mx = fmaxf(mx, __ldcg(a.part_m + h * splits + sp));
        float num = 0.f, den = 0.f;
        if (mx != -INFINITY) {
            for (int sp = 0; sp < used; ++sp) {
                const float ms = __ldcg(a.part_m + h * splits + sp);
                if (ms == -INFINITY) continue;
                const float w = fast_exp2(ms - mx);
                den = fmaf(w, __ldcg(a.part_l + h * splits + sp), den);
                num = fmaf(w, __ldcg(a.part_o + (h * splits + sp) * D + d), num);
            }
        }
        a.out[h * D + d] = den > 0.f ? num / den : 0.f;
    }
}

template <int D, bool BF16, int G>
cudaError_t launch_decode_t(const DecodeArgs& a, int units, cudaStream_t s)
{
    using S = DecodeShape<D, BF16>;
    const size_t smem = size_t(2) * S::TPS * S::ROW_BYTES + size_t(2) * G * S::TPS * sizeof(float);
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, BF16, G>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    decode_kernel<D, BF16, G><<<dim3(unsigned(units * a.max_splits)), kDecThreads, smem, s>>>(a);
    return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t dispatch_group(const DecodeArgs& a, int G, int units, cudaStream_t s)
{
    switch (G) {
        case 1: return launch_decode_t<D, BF16, 1>(a, units, s);
        case 2: return launch_decode_t<D, BF16, 2>(a, units, s);
        case 4: return launch_decode_t<D, BF16, 4>(a, units, s);
        case 8: return launch_decode_t<D, BF16, 8>(a, units, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int decode_tokens_per_split(int D, bool kv_bf16)
{
    return kStageBytes / (2 * D * (kv_bf16 ? 2 : 4));
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
    a.blocks_per_split = L.blocks_per_split;
    a.max_splits = L.max_splits;
    a.scale_log2 = g.scale_log2;
    a.part_m = reinterpret_cast<float*>(ws + L.part_m);
    a.part_l = reinterpret_cast<float*>(ws + L.part_l);
    a.part_o = reinterpret_cast<float*>(ws + L.part_o);
    a.counters = reinterpret_cast<uint32_t*>(ws + L.dec_counters);
    a.err = reinterpret_cast<uint32_t*>(ws + L.err);
    if (g.D == 128)
        return g.kv_bf16 ? dispatch_group<128, true>(a, g.G, units, s)
                         : dispatch_group<128, false>(a, g.G, units, s);
    return g.kv_bf16 ? dispatch_group<64, true>(a, g.G, units, s)
                     : dispatch_group<64, false>(a, g.G, units, s);
}

}  // namespace sa
