// Per-block key metadata: Quest bounding box (min / max per channel) and block means.
//
// "SGLang分层稀疏注意力技术解析与优化实践" §3.1.2: each KV block keeps, per key dimension,
// the minimum and maximum over its tokens.  SparDA page (www.2kiu.com/news/4656707) §3.1
// and "从HiSparse到QSA的移植实战" §2.2: a block (or coarse block) is summarised by the mean
// of its keys.
//
// Mapping: one warp walks a run of consecutive logical blocks of one (sequence, KV head)
// unit.  A key row of D elements is covered by LPR lanes with one 16-byte load each
// (coalesced, 32/LPR rows per warp instruction); min/max/sum stay in registers and
// are combined across the row groups of the warp with xor shuffles.  min/max of bf16
// values are bf16 values, so the stored bounding box is exact.  Means accumulate in
// fp32.  HBM traffic: the keys once, plus the metadata written.
#include "sa_common.cuh"
#include "sa_internal.h"

namespace sa {
namespace {

constexpr int kMetaWarps = 8;
constexpr int kMetaRunNoMean = 4;   // blocks per warp when no mean is needed

struct MetaArgs {
    const void* k_pages;
    const int32_t* block_table;
    void* kmin;
    void* kmax;
    float* kmean;
    uint32_t* err;
    int Hkv, bs, N, nb, num_pages, D;
    int bt_stride;        // block_table row length (capacity in blocks)
    int run_blocks;       // logical blocks per warp run (= mean row when kmean is built)
    int runs_per_unit;    // runs of the context
    int run_first;        // first run to (re)build: 0, or the run holding the first appended token
    int row_stride;       // kmin / kmax rows per unit (capacity)
    int mean_stride;      // kmean rows per unit (capacity)
    long long total_runs; // units * (runs_per_unit - run_first)
};

template <int D, bool BF16>
__global__ void __launch_bounds__(kMetaWarps * 32) build_meta_kernel(MetaArgs a)
{
    constexpr int ESZ = BF16 ? 2 : 4;
    constexpr int EPL = 16 / ESZ;      // elements per lane
    constexpr int LPR = D / EPL;       // lanes per key row
    constexpr int RPW = 32 / LPR;      // rows per warp instruction
    static_assert(LPR >= 1 && LPR <= 32 && 32 % LPR == 0, "bad lane split");

    const int lane = threadIdx.x & 31;
    const long long run = (long long)blockIdx.x * kMetaWarps + (threadIdx.x >> 5);
    if (run >= a.total_runs) return;
    allow_dependents_early();
    grid_dependency_wait();   // K pages (e.g. just appended) may come from the previous kernel
    const int live = a.runs_per_unit - a.run_first;
    const int u = int(run / live);
    const int r = a.run_first + int(run % live);
    const int b = u / a.Hkv, kvh = u % a.Hkv;
    const int sub = lane % LPR, rsub = lane / LPR;

    const char* kbase = reinterpret_cast<const char*>(a.k_pages);
    const size_t tile_bytes = size_t(a.bs) * D * ESZ;

    float sum[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) sum[e] = 0.f;
    int tokens = 0;

    const int j0 = r * a.run_blocks;
    const int j1 = min(a.nb, j0 + a.run_blocks);
    for (int j = j0; j < j1; ++j) {
        const int page = a.block_table[size_t(b) * a.bt_stride + j];
        if (page < 0 || page >= a.num_pages) {
            if (lane == 0) raise_error(a.err, SPARSE_ATTN_ERR_PAGE);
            continue;
        }
        const int nt = min(a.bs, a.N - j * a.bs);
        tokens += nt;
        const char* tile = kbase + (size_t(page) * a.Hkv + kvh) * tile_bytes + sub * 16;
        float lo[EPL], hi[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) { lo[e] = __int_as_float(0x7f800000); hi[e] = -lo[e]; }

        // rows rsub, rsub + RPW, ... ; four loads in flight per lane
        int t = rsub;
        for (; t + 3 * RPW < nt; t += 4 * RPW) {
            uint4 v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                v[i] = ld_stream16(tile + size_t(t + i * RPW) * D * ESZ);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float f[EPL];
                unpack16<BF16>(v[i], f);
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    lo[e] = fminf(lo[e], f[e]);
                    hi[e] = fmaxf(hi[e], f[e]);
                    sum[e] += f[e];
                }
            }
        }
        for (; t < nt; t += RPW) {
            float f[EPL];
            unpack16<BF16>(ld_stream16(tile + size_t(t) * D * ESZ), f);
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                lo[e] = fminf(lo[e], f[e]);
                hi[e] = fmaxf(hi[e], f[e]);
                sum[e] += f[e];
            }
        }
        // combine the row groups of this warp
#pragma unroll
        for (int m = LPR; m < 32; m <<= 1) {
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                lo[e] = fminf(lo[e], __shfl_xor_sync(kFullMask, lo[e], m));
                hi[e] = fmaxf(hi[e], __shfl_xor_sync(kFullMask, hi[e], m));
            }
        }
        if (rsub == 0) {
            const size_t row = (size_t(u) * a.row_stride + j) * D + sub * EPL;
            uint4 wlo, whi;
            if constexpr (BF16) {
                wlo.x = f32_to_bf16_bits_exact(lo[0]) | (f32_to_bf16_bits_exact(lo[1]) << 16);
                wlo.y = f32_to_bf16_bits_exact(lo[2]) | (f32_to_bf16_bits_exact(lo[3]) << 16);
                wlo.z = f32_to_bf16_bits_exact(lo[4]) | (f32_to_bf16_bits_exact(lo[5]) << 16);
                wlo.w = f32_to_bf16_bits_exact(lo[6]) | (f32_to_bf16_bits_exact(lo[7]) << 16);
                whi.x = f32_to_bf16_bits_exact(hi[0]) | (f32_to_bf16_bits_exact(hi[1]) << 16);
                whi.y = f32_to_bf16_bits_exact(hi[2]) | (f32_to_bf16_bits_exact(hi[3]) << 16);
                whi.z = f32_to_bf16_bits_exact(hi[4]) | (f32_to_bf16_bits_exact(hi[5]) << 16);
                whi.w = f32_to_bf16_bits_exact(hi[6]) | (f32_to_bf16_bits_exact(hi[7]) << 16);
                *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.kmin) + row) = wlo;
                *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.kmax) + row) = whi;
            } else {
                wlo = make_uint4(__float_as_uint(lo[0]), __float_as_uint(lo[1]),
                                 __float_as_uint(lo[2]), __float_as_uint(lo[3]));
                whi = make_uint4(__float_as_uint(hi[0]), __float_as_uint(hi[1]),
                                 __float_as_uint(hi[2]), __float_as_uint(hi[3]));
                *reinterpret_cast<uint4*>(reinterpret_cast<float*>(a.kmin) + row) = wlo;
                *reinterpret_cast<uint4*>(reinterpret_cast<float*>(a.kmax) + row) = whi;
            }
        }
    }

    if (a.kmean != nullptr) {
#pragma unroll
        for (int m = LPR; m < 32; m <<= 1) {
#pragma unroll
            for (int e = 0; e < EPL; ++e) sum[e] += __shfl_xor_sync(kFullMask, sum[e], m);
        }
        if (rsub == 0 && tokens > 0) {
            const float inv = 1.0f / float(tokens);
            float* dst = a.kmean + (size_t(u) * a.mean_stride + r) * D + sub * EPL;
#pragma unroll
            for (int e = 0; e < EPL; e += 4)
                *reinterpret_cast<float4*>(dst + e) =
                    make_float4(sum[e] * inv, sum[e + 1] * inv, sum[e + 2] * inv, sum[e + 3] * inv);
        }
    }
}

template <int D, bool BF16>
cudaError_t launch_meta_t(const MetaArgs& a, cudaStream_t s)
{
    const long long ctas = (a.total_runs + kMetaWarps - 1) / kMetaWarps;
    if (ctas == 0) return cudaSuccess;
    return launch_after_previous(build_meta_kernel<D, BF16>, dim3(unsigned(ctas)), dim3(kMetaWarps * 32), 0, s, a);
}

}  // namespace

cudaError_t launch_build_meta(const Geometry& g, const void* k_pages, const int32_t* block_table,
                              void* kmin, void* kmax, float* kmean, uint32_t* err, int first_token,
                              cudaStream_t s)
{
    MetaArgs a{};
    a.k_pages = k_pages;
    a.block_table = block_table;
    a.kmin = kmin;
    a.kmax = kmax;
    a.kmean = kmean;
    a.err = err;
    a.Hkv = g.Hkv;
    a.bs = g.bs;
    a.N = g.N;
    a.nb = g.nb;
    a.num_pages = g.num_pages;
    a.bt_stride = g.nb_cap;
    a.D = g.D;
    // A mean row is a whole number of blocks: one warp owns exactly one mean row.
    // Without means an append rebuilds single blocks (min / max are exact, so the
    // grouping of blocks into runs does not change a bit of the result).
    a.run_blocks = kmean ? g.mean_block / g.bs : (first_token > 0 ? 1 : kMetaRunNoMean);
    a.runs_per_unit = (g.nb + a.run_blocks - 1) / a.run_blocks;
    // rows holding tokens >= first_token are rebuilt from their tokens; earlier rows keep
    // their values (their tokens have not changed)
    a.run_first = min(a.runs_per_unit, (first_token / g.bs) / a.run_blocks);
    a.row_stride = g.nb_cap;
    a.mean_stride = g.n_mean_cap;
    a.total_runs = (long long)g.units() * (a.runs_per_unit - a.run_first);
    if (g.D == 128) return g.kv_bf16 ? launch_meta_t<128, true>(a, s) : launch_meta_t<128, false>(a, s);
    return g.kv_bf16 ? launch_meta_t<64, true>(a, s) : launch_meta_t<64, false>(a, s);
}

}  // namespace sa
