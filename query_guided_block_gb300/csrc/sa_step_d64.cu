// Fused step kernel instantiations for head dimension 64 (a translation unit of its
// own so that the two head dimensions compile in parallel).
#include "sa_step_kernel.cuh"

namespace sa {

cudaError_t launch_step_d64(const Geometry& g, const WorkspaceLayout& L, char* ws, const void* q,
                            const void* kmin, const void* kmax, const float* kmean,
                            const int32_t* reserve_ids, const void* k_pages, const void* v_pages,
                            const int32_t* block_table, int32_t* sel_ids, int32_t* sel_count, float* out,
                            cudaStream_t s)
{
    return launch_step_impl<64>(g, L, ws, q, kmin, kmax, kmean, reserve_ids, k_pages, v_pages, block_table,
                                sel_ids, sel_count, out, s);
}

}  // namespace sa
