// Miss loading into a per-unit slot pool, and the slot map the decode reads through.
//
// "SGLang分层稀疏注意力技术解析与优化实践" §3.3 (IO transfer): the full KV cache stays in
// page-first layout in pinned, host-registered memory; the GPU keeps a slot pool; the
// blocks a step misses are transferred zero-copy, batched over requests, so that the
// IO per step stays small.  §3.2 (Sparse Diff Kernel, steps c-d): load the misses into
// the claimed slots, then update the index.
//
// GB300 design: the GPU reads the host store directly (NVLink-C2C, zero copy), one
// launch for every miss of every unit: each warp moves one K or V page tile (bs x D
// contiguous) with 16-byte loads, eight in flight per lane.  The slot map is one warp
// per unit matching the selected ids against the unit's slot_block row in shared
// memory.
#include "sa_common.cuh"
#include "sa_internal.h"

namespace sa {
namespace {

constexpr int kIoThreads = 256;
constexpr int kSlotMapWarps = 8;

struct IoArgs {
    const char* host_k;      // [num_pages, Hkv, bs, D], device-accessible host memory
    const char* host_v;
    const int32_t* block_table;
    const int32_t* miss_ids;     // [units, stride]
    const int32_t* miss_slot;
    const int32_t* counts;       // [units, 5]: misses at [1]
    char* pool_k;                // [units, C, bs, D]
    char* pool_v;
    int units, Hkv, nb, num_pages, stride, C;
    int bt_stride;               // block_table row length (capacity in blocks)
    size_t tile_bytes;           // bs * D * element size
    uint32_t* err;
};

// One CTA per (unit, tensor): the unit's misses are resolved to (source tile, slot) in
// one batch, then their tiles are copied as one flat range of 16-byte elements, sixteen
// loads in flight per thread, so a step's few misses per unit cost about one host round
// trip.
constexpr int kIoInFlight = 16;

__global__ void __launch_bounds__(kIoThreads) load_misses_kernel(IoArgs a)
{
    extern __shared__ long long io_tiles[];   // [2][stride]: source offset (-1: skip), dest offset
    const int tid = threadIdx.x;
    const int u = blockIdx.x >> 1, t = blockIdx.x & 1;
    allow_dependents_early();
    grid_dependency_wait();   // diff outputs may come from the previous kernel
    int n = a.counts[size_t(u) * 5 + 1];
    if (n < 0 || n > a.stride) {
        if (tid == 0) raise_error(a.err, SPARSE_ATTN_ERR_SEL_COUNT);
        n = n < 0 ? 0 : a.stride;
    }
    if (n == 0) return;
    long long* src_off = io_tiles;
    long long* dst_off = io_tiles + a.stride;
    const int b = u / a.Hkv, kvh = u - b * a.Hkv;
    for (int i = tid; i < n; i += kIoThreads) {
        const int j = a.miss_ids[size_t(u) * a.stride + i];
        const int s = a.miss_slot[size_t(u) * a.stride + i];
        long long so = -1;
        if (j < 0 || j >= a.nb || s < 0 || s >= a.C) {
            if (t == 0) raise_error(a.err, j < 0 || j >= a.nb ? SPARSE_ATTN_ERR_SEL_ID : SPARSE_ATTN_ERR_SLOT);
        } else {
            const int page = a.block_table[size_t(b) * a.bt_stride + j];
            if (page < 0 || page >= a.num_pages) {
                if (t == 0) raise_error(a.err, SPARSE_ATTN_ERR_PAGE);
            } else {
                so = (long long)((size_t(page) * a.Hkv + kvh) * a.tile_bytes);
            }
        }
        src_off[i] = so;
        dst_off[i] = (long long)((size_t(u) * a.C + (s >= 0 && s < a.C ? s : 0)) * a.tile_bytes);
    }
    __syncthreads();
    const char* src = t ? a.host_v : a.host_k;
    char* dst = t ? a.pool_v : a.pool_k;
    const long long n16 = (long long)(a.tile_bytes / 16);
    const long long total = n16 * n;
    for (long long base = 0; base < total; base += (long long)kIoThreads * kIoInFlight) {
        uint4 v[kIoInFlight];
#pragma unroll
        for (int r = 0; r < kIoInFlight; ++r) {
            const long long f = base + (long long)r * kIoThreads + tid;
            if (f < total) {
                const int m = int(f / n16);
                const long long so = src_off[m];
                if (so >= 0) v[r] = ld_stream16(src + so + (f - m * n16) * 16);
            }
        }
#pragma unroll
        for (int r = 0; r < kIoInFlight; ++r) {
            const long long f = base + (long long)r * kIoThreads + tid;
            if (f < total) {
                const int m = int(f / n16);
                if (src_off[m] >= 0) *reinterpret_cast<uint4*>(dst + dst_off[m] + (f - m * n16) * 16) = v[r];
            }
        }
    }
}

struct SlotMapArgs {
    const int32_t* sel_ids;
    const int32_t* sel_count;
    const int32_t* slot_block;   // [units, C]
    int32_t* sel_slot;           // [units, stride]
    int units, stride, C, nb;
    uint32_t* err;
};

// Warp per unit: the unit's selected ids (ascending) go to shared memory; each lane
// takes slots lane, lane + 32, ... and binary-searches its slot's block among them.
__global__ void __launch_bounds__(kSlotMapWarps * 32) slot_map_kernel(SlotMapArgs a)
{
    extern __shared__ int sm_ids[];   // [kSlotMapWarps][stride]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int u = blockIdx.x * kSlotMapWarps + warp;
    if (u >= a.units) return;
    allow_dependents_early();
    grid_dependency_wait();
    int* ids = sm_ids + warp * a.stride;
    int n = a.sel_count[u];
    if (n < 0 || n > a.stride) {
        if (lane == 0) raise_error(a.err, SPARSE_ATTN_ERR_SEL_COUNT);
        n = n < 0 ? 0 : a.stride;
    }
    for (int i = lane; i < n; i += 32) {
        ids[i] = a.sel_ids[size_t(u) * a.stride + i];
        a.sel_slot[size_t(u) * a.stride + i] = -1;
    }
    __syncwarp();
    for (int s = lane; s < a.C; s += 32) {
        const int j = a.slot_block[size_t(u) * a.C + s];
        if (j < 0) continue;
        int lo = 0, hi = n;                 // first index with ids[index] >= j
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (ids[mid] < j) lo = mid + 1;
            else hi = mid;
        }
        if (lo < n && ids[lo] == j) a.sel_slot[size_t(u) * a.stride + lo] = s;
    }
    __syncwarp();
    // a selected block with no slot was not made resident by the diff
    for (int i = lane; i < n; i += 32)
        if (a.sel_slot[size_t(u) * a.stride + i] < 0) raise_error(a.err, SPARSE_ATTN_ERR_SLOT);
}

}  // namespace

cudaError_t launch_load_misses(const Geometry& g, const void* host_k, const void* host_v,
                               const int32_t* block_table, const int32_t* miss_ids,
                               const int32_t* miss_slot, const int32_t* counts, int cache_slots,
                               void* pool_k, void* pool_v, uint32_t* err, cudaStream_t s)
{
    const int units = g.units();
    if (units == 0) return cudaSuccess;
    IoArgs a{};
    a.host_k = static_cast<const char*>(host_k);
    a.host_v = static_cast<const char*>(host_v);
    a.block_table = block_table;
    a.miss_ids = miss_ids;
    a.miss_slot = miss_slot;
    a.counts = counts;
    a.pool_k = static_cast<char*>(pool_k);
    a.pool_v = static_cast<char*>(pool_v);
    a.units = units;
    a.Hkv = g.Hkv;
    a.nb = g.nb;
    a.num_pages = g.num_pages;
    a.bt_stride = g.nb_cap;
    a.stride = g.sel_stride;
    a.C = cache_slots;
    a.tile_bytes = size_t(g.bs) * g.D * (g.kv_bf16 ? 2 : 4);
    a.err = err;
    const size_t smem = size_t(2) * g.sel_stride * sizeof(long long);
    return launch_after_previous(load_misses_kernel, dim3(unsigned(2 * units)), dim3(kIoThreads), smem, s, a);
}

cudaError_t launch_slot_map(const Geometry& g, const int32_t* sel_ids, const int32_t* sel_count,
                            const int32_t* slot_block, int cache_slots, int32_t* sel_slot,
                            uint32_t* err, cudaStream_t s)
{
    const int units = g.units();
    if (units == 0) return cudaSuccess;
    SlotMapArgs a{sel_ids, sel_count, slot_block, sel_slot, units, g.sel_stride, cache_slots, g.nb, err};
    const size_t smem = size_t(kSlotMapWarps) * g.sel_stride * sizeof(int);
    return launch_after_previous(slot_map_kernel, dim3(unsigned((units + kSlotMapWarps - 1) / kSlotMapWarps)),
                                 dim3(kSlotMapWarps * 32), smem, s, a);
}

}  // namespace sa
