// Fused decode step: block selection and sparse attention in one persistent launch.
//
// "SGLang分层稀疏注意力技术解析与优化实践" §1.2 (select-then-compute) runs selection and
// the attention over the selected tokens as two stages of one decode step.  Here both
// stages run in a single cooperative grid of one CTA (8 warps) per SM:
//   1. select phase: every warp streams its own 8 KB metadata slabs through a private
//      cp.async ring and scores them (the select kernel's arithmetic, so the scores are
//      the same bits); the warp completing a unit records it, and once the CTA has
//      finished streaming it ranks and emits its completed units, publishing
//      ready[u] = 1 (device-scope release) for each;
//   2. decode phase: the decode kernel's warp-independent tensor-core attention; each
//      CTA waits (bounded, acquire) only for the units of its own item range instead of
//      for the whole selection, and the CTA merging a unit clears ready[u].
// The select phase never waits on another CTA and a cooperative launch keeps every CTA
// resident, so each wait of the decode phase ends.  Shared memory: the select rings and
// keys alias the decode rings (a barrier separates the phases).  Problems whose grid
// does not fit this shape run as the select kernel followed by the decode kernel,
// launched as its programmatic dependent and waiting per unit on the same flags.
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
