// Host-side launcher interface between the C ABI (sa_api.cu) and the kernel files.
// Every launcher assumes its arguments were validated by the ABI layer and returns a
// cudaError_t from the launch.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "sparse_attn.h"

namespace sa {

// Derived, validated problem geometry.
struct Geometry {
    int B, Hq, Hkv, G, D, N, bs, nb, num_pages;
    int win_first, win_count;      // window blocks [win_first, nb)
    int n_cand;                    // single-level candidates = win_first
    int sel_stride;                // ids per unit row
    bool kv_bf16, q_bf16;
    bool two_level;
    int coarse_block, per_coarse, n_coarse, topk_coarse;
    int mean_block, n_mean;        // kmean rows per unit
    int nb_cap, n_mean_cap;        // metadata rows allocated per unit (capacity_tokens)
    int topk;
    int n_reserve;                 // reserve block ids per unit (0: none)
    int Q;                         // query vectors per sequence sharing a selection (>= 1)
    int score_kind;
    float scale_log2;              // softmax_scale * log2(e)
    int units() const { return B * Hkv; }
};

// Workspace carve-up (byte offsets from the workspace base, each 256-byte aligned).
struct WorkspaceLayout {
    size_t err;            // uint32 error word (header words: see sa_common.cuh kHdr*)
    size_t sel_work;       // uint32 next chunk id (select kernels)
    size_t sel_done;       // uint32 finished CTAs (select kernels)
    size_t dec_work;       // uint32 (header) fused step: selections published so far
    size_t dec_done;       // uint32 (header) fused step: decode tickets taken so far
    size_t sel_counters;   // uint32 [units]
    size_t dec_counters;   // uint32 [units]
    size_t l1_counters;    // uint32 [units] (two-level, level 1)
    size_t ready;          // uint32 [units] (fused step: unit's selection published, or the
                           // queue entry at that position filled)
    size_t queue;          // uint32 [units] (fused step: units in the order they were published)
    size_t scores;         // float [units, score_cols]
    size_t survivors;      // int32 [units, topk_coarse] (two-level)
    size_t n_survivors;    // int32 [units]
    size_t part_m;         // float [B*Hq, max_splits]
    size_t part_l;         // float [B*Hq, max_splits]
    size_t part_o;         // float [B*Hq, max_splits, D]
    size_t total;
    int score_cols;        // candidates per unit row of the score buffer
    int max_splits;        // decode work items (split-K slices) per unit
    int blocks_per_split;  // selected blocks per decode work item
};

WorkspaceLayout workspace_layout(const Geometry& g);

// Byte offset of the wait-limit word in the workspace header (kHdrWaitLimit on the
// device side).
constexpr size_t kHdrWaitLimitByte = 24;

// Streaming multiprocessors of the current device (cached per device).
int num_sms();

// Runs a kernel's one-time host set-up (function attributes such as its dynamic
// shared-memory limit) once for each device it is launched on: the attributes belong to
// that device's context, so a process driving several GPUs sets each one up.  `done` is
// a bit mask over device ordinals 0..63 (beyond that the set-up runs on every call).
// Two host threads may both run `setup` for one device; it only sets attributes, so
// that is harmless.  A cudaDeviceReset discards the attributes but not this mask: a
// process that resets a device and then calls the library again gets launch errors.
template <typename Setup>
inline cudaError_t once_per_device(std::atomic<unsigned long long>& done, Setup setup)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool tracked = dev >= 0 && dev < 64;
    const unsigned long long bit = tracked ? (1ull << dev) : 0ull;
    if (tracked && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = setup();
    if (e == cudaSuccess && tracked) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}
constexpr int kSmemPerSm = 228 * 1024;

// Selected blocks per decode work item, and whether a (D, dtype, block, group)
// combination fits the decode kernel's shared-memory pipeline.
int decode_blocks_per_item(int D, bool kv_bf16, int block_size);
bool decode_supported(int D, bool kv_bf16, int block_size, int G);

cudaError_t launch_build_meta(const Geometry& g, const void* k_pages, const int32_t* block_table,
                              void* kmin, void* kmax, float* kmean, uint32_t* err, int first_token,
                              cudaStream_t s);

cudaError_t launch_select(const Geometry& g, const WorkspaceLayout& L, char* ws, const void* q,
                          const void* kmin, const void* kmax, const float* kmean,
                          const int32_t* reserve_ids, int32_t* sel_ids, int32_t* sel_count,
                          cudaStream_t s, uint32_t* ready = nullptr);   // publish ready[u] per unit

// Slot-pool decode reading the step's misses from the host store in the same pass.
struct SlotIo {
    const void* host_k;          // [num_pages, Hkv, bs, D], device-readable
    const void* host_v;
    const int32_t* miss_ids;     // [units, sel_stride], ascending per unit
    const int32_t* miss_slot;    // [units, sel_stride]: the pool slot of each miss
    const int32_t* counts;       // [units, 5]: misses at [1]
};

cudaError_t launch_decode(const Geometry& g, const WorkspaceLayout& L, char* ws, const void* q,
                          const void* k_pages, const void* v_pages, const int32_t* block_table,
                          const int32_t* sel_ids, const int32_t* sel_count, float* out,
                          const int32_t* sel_slot, int slot_C, cudaStream_t s,
                          uint32_t* ready = nullptr,    // bf16 K/V only: wait per unit on ready[]
                          const SlotIo* io = nullptr);  // bf16 K/V, slot mode only
// Multi-query attention (sa_decode_mq.cu): Q query vectors per sequence, one selection.
int mq_row_tiles(int Q, int G);
cudaError_t launch_decode_mq(const Geometry& g, const WorkspaceLayout& L, char* ws, const void* q,
                             const void* k_pages, const void* v_pages, const int32_t* block_table,
                             const int32_t* sel_ids, const int32_t* sel_count, float* out, cudaStream_t s);
// Slot pool (sa_io.cu): the misses' K/V tiles from a host-resident page-first store
// into their slots, and each selected block's slot.
cudaError_t launch_load_misses(const Geometry& g, const void* host_k, const void* host_v,
                               const int32_t* block_table, const int32_t* miss_ids,
                               const int32_t* miss_slot, const int32_t* counts, int cache_slots,
                               void* pool_k, void* pool_v, uint32_t* err, cudaStream_t s);
cudaError_t launch_slot_map(const Geometry& g, const int32_t* sel_ids, const int32_t* sel_count,
                            const int32_t* slot_block, int cache_slots, int32_t* sel_slot,
                            uint32_t* err, cudaStream_t s);

// Fused step (sa_step.cu): select then decode in one cooperative persistent launch,
// single-level selection, bf16 K/V, one query per sequence.  cudaErrorNotSupported
// when the problem does not fit one CTA per SM.
bool step_supported(const Geometry& g);
int step_launches(const Geometry& g, const WorkspaceLayout& L);   // kernels one step launches
cudaError_t launch_step(const Geometry& g, const WorkspaceLayout& L, char* ws, const void* q,
                        const void* kmin, const void* kmax, const float* kmean,
                        const int32_t* reserve_ids, const void* k_pages, const void* v_pages,
                        const int32_t* block_table, int32_t* sel_ids, int32_t* sel_count, float* out,
                        cudaStream_t s);
cudaError_t launch_step_d64(const Geometry& g, const WorkspaceLayout& L, char* ws, const void* q,
                            const void* kmin, const void* kmax, const float* kmean,
                            const int32_t* reserve_ids, const void* k_pages, const void* v_pages,
                            const int32_t* block_table, int32_t* sel_ids, int32_t* sel_count, float* out,
                            cudaStream_t s);

cudaError_t launch_diff(const Geometry& g, int step, const int32_t* sel_ids,
                        const int32_t* sel_count, const int32_t* prev_ids,
                        const int32_t* prev_count, int cache_slots, int32_t* slot_block,
                        int32_t* slot_last_use, int32_t* hit_ids, int32_t* miss_ids,
                        int32_t* miss_slot, int32_t* evict_ids, int32_t* evict_slot,
                        int32_t* new_ids, int32_t* dropped_ids, int32_t* counts, uint32_t* err,
                        cudaStream_t s, int32_t* sel_slot = nullptr);   // also the slot map

}  // namespace sa
