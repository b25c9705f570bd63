// The fused step kernel (select phase, then decode phase, in one cooperative grid)
// and its launcher, instantiated per head dimension by sa_step.cu (D = 128) and
// sa_step_d64.cu (D = 64).  The design notes are in sa_step.cu.
#pragma once

#include "sa_decode_body.cuh"
#include "sa_select_body.cuh"

namespace sa {
namespace {

static_assert(kSelThreads == kDecThreads, "both phases run on the same CTA shape");

// When every decode range is one whole unit, the CTA that ranks a unit decodes it
// straight after (the selection is its own: no hand-off, no wait).  A CTA that ranks
// more than one unit keeps the first and queues the others: it appends each to a queue
// and publishes the position (ready[position] = the step's flag value, release), and
// the CTAs that rank nothing take tickets and decode the queued units in order.  A
// ticket holder waits (bounded) until its position is published, or until every unit
// is ranked and the queue ends before it.  Otherwise CTA c decodes range c once its
// units are published.  A unit's result comes from the same per-unit code either way,
// so the bits do not depend on which CTA computes it.
template <int KIND, int D, int G, bool QSPLIT>
__global__ void __launch_bounds__(kDecThreads, 1) step_kernel(SelectArgs sa_args, DecodeArgs da, uint32_t* ready,
                                                              uint32_t* queue)
{
    __shared__ int s_unit;
    const bool by_queue = da.ranges == da.units;
    if (threadIdx.x == 0) s_unit = -1;
    const uint32_t flag_value =
        select_body_warps<KIND, KIND == KIND_QUEST, D>(sa_args, ready, by_queue ? queue : nullptr, &s_unit);
    __syncthreads();   // select's rings and keys are reused as the decode rings
    if (by_queue) {
        const int kept = s_unit;
        if (kept >= 0) {
            decode_mma_items<D, G, QSPLIT>(da, nullptr, 0u, kept * da.items_per_unit, (kept + 1) * da.items_per_unit);
        } else {
            const long long wait_cycles = handoff_wait_limit(da.err);
            uint32_t* tail = header_word(da.err, kHdrQueueTail);
            uint32_t* ranked = header_word(da.err, kHdrRanked);
            while (true) {
                if (threadIdx.x == 0) {
                    const uint32_t t = atomicAdd(header_word(da.err, kHdrQueueHead), 1u);
                    int u = -1;
                    const long long t0 = clock64();
                    while (true) {
                        if (ld_acquire_gpu(ready + min(t, uint32_t(da.units - 1))) == flag_value && t < uint32_t(da.units)) {
                            const int v = int(__ldcg(queue + t));
                            if (v >= 0 && v < da.units) u = v;
                            else raise_error(da.err, SPARSE_ATTN_ERR_TIMEOUT);
                            break;
                        }
                        // every unit ranked and the queue ends before t: nothing for this ticket
                        if (ld_acquire_gpu(ranked) >= uint32_t(da.units) && ld_acquire_gpu(tail) <= t) break;
                        if (clock64() - t0 > wait_cycles) {
                            raise_error(da.err, SPARSE_ATTN_ERR_TIMEOUT);
                            break;
                        }
                        __nanosleep(32);
                    }
                    s_unit = u;
                    __threadfence();
                }
                __syncthreads();
                const int u = s_unit;
                __syncthreads();   // s_unit is rewritten by the next ticket
                if (u < 0) break;
                decode_mma_items<D, G, QSPLIT>(da, nullptr, 0u, u * da.items_per_unit, (u + 1) * da.items_per_unit);
                __syncthreads();   // the next unit reuses the rings and the page cache
            }
        }
    } else {
        decode_mma_body<D, G, QSPLIT>(da, ready, flag_value);
    }
    finish_step(da.err, flag_value);
}

template <int KIND, int D, int G, bool QSPLIT>
cudaError_t launch_step_t(const SelectArgs& sa_args, const DecodeArgs& da, uint32_t* ready, uint32_t* queue, int ctas,
                          cudaStream_t s)
{
    constexpr size_t smem = slab_smem_bytes<D>();
    static_assert(smem >= SlabSelShape<KIND, KIND == KIND_QUEST, D>::RING_BYTES &&
                      smem >= kMaxSelectKeys * sizeof(uint32_t),
                  "select rings and keys must fit the decode rings");
    auto kernel = step_kernel<KIND, D, G, QSPLIT>;
    static std::atomic<unsigned long long> configured{0};   // devices set up
    const cudaError_t set_up = once_per_device(configured, [&]() -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kDecThreads, smem);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) return cudaErrorNotSupported;
        return cudaSuccess;
    });
    if (set_up != cudaSuccess) return set_up;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(ctas));
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // all CTAs resident: the decode waits end
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, sa_args, da, ready, queue);
}

template <int KIND, int D, bool QSPLIT>
cudaError_t dispatch_step_g(const SelectArgs& sa_args, const DecodeArgs& da, uint32_t* ready, uint32_t* queue, int ctas, int G,
                            cudaStream_t s)
{
    switch (G) {
        case 1: return launch_step_t<KIND, D, 1, QSPLIT>(sa_args, da, ready, queue, ctas, s);
        case 2: return launch_step_t<KIND, D, 2, QSPLIT>(sa_args, da, ready, queue, ctas, s);
        case 4: return launch_step_t<KIND, D, 4, QSPLIT>(sa_args, da, ready, queue, ctas, s);
        case 8: return launch_step_t<KIND, D, 8, QSPLIT>(sa_args, da, ready, queue, ctas, s);
        default: return cudaErrorInvalidValue;
    }
}

// CTAs of the fused grid: one per SM, fewer when there are fewer decode items; 0 when
// the decode ranges (those of the decode kernel, so both give the same bits) need more
// CTAs than that.
int step_ctas(const Geometry& g, const WorkspaceLayout& L)
{
    const long long items = (long long)g.units() * L.max_splits;
    long long ctas = num_sms();
    if (ctas > items) ctas = items;
    if (ctas < 1) return 0;
    const int ranges = decode_ranges(g.units(), L.max_splits, L.blocks_per_split, num_sms());
    return ranges > ctas ? 0 : int(ctas);
}

// CTAs of the single-launch step, or 0 when the problem runs as two kernels: the grid
// must hold every decode range (step_ctas), each CTA may complete at most
// kSlabSelMaxUnits units, and there must be no more units than CTAs (a CTA runs the
// top-ks of the units it completes one after another, while the select kernel, two
// CTAs per SM, runs them side by side).
template <int D>
int step_single_ctas(const Geometry& g, const WorkspaceLayout& L)
{
    const int units = g.units();
    const int ctas = step_ctas(g, L);
    if (ctas == 0 || units > ctas) return 0;
    const int rows = g.score_kind == SPARSE_ATTN_SCORE_MEAN ? SlabSelShape<KIND_MEAN, false, D>::ROWS
                                                           : SlabSelShape<KIND_QUEST, true, D>::ROWS;
    const long long chunks_per_unit = ((g.n_cand > 0 ? g.n_cand : 1) + rows - 1) / rows;
    const long long per_cta = (units * chunks_per_unit + ctas - 1) / ctas;
    if (per_cta / chunks_per_unit + 2 > kSlabSelMaxUnits) return 0;
    return ctas;
}

template <int D>
cudaError_t launch_step_impl(const Geometry& g, const WorkspaceLayout& L, char* ws, const void* q,
                             const void* kmin, const void* kmax, const float* kmean,
                             const int32_t* reserve_ids, const void* k_pages, const void* v_pages,
                             const int32_t* block_table, int32_t* sel_ids, int32_t* sel_count,
                             float* out, cudaStream_t s)
{
    const int units = g.units();
    if (units == 0) return cudaSuccess;
    const int ctas = step_single_ctas<D>(g, L);
    if (ctas == 0) return cudaErrorNotSupported;
    const bool mean = g.score_kind == SPARSE_ATTN_SCORE_MEAN;

    SelectArgs sa_args = select_args_base(g, L, ws, q, kmin, kmax, kmean);
    set_single_level(sa_args, g, reserve_ids, sel_ids, sel_count);
    if (mean) set_slab_chunking<KIND_MEAN, false, D>(sa_args, units);
    else set_slab_chunking<KIND_QUEST, true, D>(sa_args, units);
    DecodeArgs da = decode_args(g, L, ws, q, k_pages, v_pages, block_table, sel_ids, sel_count, out, nullptr, 0);
    // with whole-unit decode ranges every CTA up to the unit count streams one unit,
    // ranks it and decodes it
    sa_args.unit_ranges = da.ranges == da.units ? 1 : 0;
    uint32_t* ready = reinterpret_cast<uint32_t*>(ws + L.ready);
    uint32_t* queue = reinterpret_cast<uint32_t*>(ws + L.queue);

    const bool qs = !g.q_bf16;
    if (mean)
        return qs ? dispatch_step_g<KIND_MEAN, D, true>(sa_args, da, ready, queue, ctas, g.G, s)
                  : dispatch_step_g<KIND_MEAN, D, false>(sa_args, da, ready, queue, ctas, g.G, s);
    return qs ? dispatch_step_g<KIND_QUEST, D, true>(sa_args, da, ready, queue, ctas, g.G, s)
              : dispatch_step_g<KIND_QUEST, D, false>(sa_args, da, ready, queue, ctas, g.G, s);
}

}  // namespace
}  // namespace sa
