// Fused decode step: block selection and sparse attention in one persistent launch.
//
// "SGLang分层稀疏注意力技术解析与优化实践" §1.2 (select-then-compute) runs selection and
// the attention over the selected tokens as two stages of one decode step.  Here both
// stages run in one cooperative grid, one CTA (eight worker warps and a control warp)
// per SM, arranged so that HBM stays busy across the hand-off between them:
//   1. streaming: the metadata slabs are listed unit by unit and cut into groups of
//      four; worker warp W scores groups W, W + NW, ... (NW worker warps in the grid),
//      so units complete one after another through the whole phase rather than all at
//      its end; the warp whose count completes a unit puts it on a device-wide queue
//      and keeps streaming;
//   2. ranking: control warps take queue positions as they come free and rank each unit
//      on their own (bisection over the key values, lower block id first on ties),
//      write the selection and publish ready[u] = the step's number (release) -- while
//      the workers of every CTA go on streaming, so only the last units' ranking is
//      exposed;
//   3. decode: once its workers have streamed their groups, the CTA runs the decode
//      kernel's warp-slab attention over its own contiguous range of decode items,
//      waiting (bounded, acquire) only for the units of that range.
// Nothing in the grid waits on a CTA that is not resident (cooperative launch), every
// wait is bounded, and the last CTA to finish advances the step epoch.  Problems the
// control warp cannot rank on chip (more than kRankMaxKeys candidates) or whose decode
// ranges do not fit one CTA per SM run as the select kernel followed by the decode
// kernel, launched as its programmatic dependent and waiting per unit on the same flags.
#include "sa_step_kernel.cuh"

namespace sa {

bool step_supported(const Geometry& g)
{
    return g.kv_bf16 && !g.two_level && g.Q == 1 && decode_supported(g.D, g.kv_bf16, g.bs, g.G);
}

int step_launches(const Geometry& g, const WorkspaceLayout& L)
{
    if (g.units() == 0) return 0;
    const int single = g.D == 64 ? step_single_ctas<64>(g, L) : step_single_ctas<128>(g, L);
    return single > 0 ? 1 : 2;
}

// Select and decode for one step.  The single cooperative launch when its grid holds
// the problem (one CTA per SM); otherwise the two kernels, the decode launched behind
// the select and waiting per unit on the published selections.
cudaError_t launch_step(const Geometry& g, const WorkspaceLayout& L, char* ws, const void* q,
                        const void* kmin, const void* kmax, const float* kmean,
                        const int32_t* reserve_ids, const void* k_pages, const void* v_pages,
                        const int32_t* block_table, int32_t* sel_ids, int32_t* sel_count, float* out,
                        cudaStream_t s)
{
    cudaError_t e = g.D == 64
        ? launch_step_d64(g, L, ws, q, kmin, kmax, kmean, reserve_ids, k_pages, v_pages, block_table, sel_ids,
                          sel_count, out, s)
        : launch_step_impl<128>(g, L, ws, q, kmin, kmax, kmean, reserve_ids, k_pages, v_pages, block_table,
                                sel_ids, sel_count, out, s);
    if (e != cudaErrorNotSupported) return e;
    uint32_t* ready = reinterpret_cast<uint32_t*>(ws + L.ready);
    e = launch_select(g, L, ws, q, kmin, kmax, kmean, reserve_ids, sel_ids, sel_count, s, ready);
    if (e != cudaSuccess) return e;
    return launch_decode(g, L, ws, q, k_pages, v_pages, block_table, sel_ids, sel_count, out, nullptr, 0, s, ready);
}

}  // namespace sa
