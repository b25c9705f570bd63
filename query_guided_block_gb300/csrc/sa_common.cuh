// Device-side helpers shared by the sm_103a kernels of libsparse_attn.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sa_internal.h"
#include "sparse_attn.h"

namespace sa {

constexpr uint32_t kFullMask = 0xffffffffu;
constexpr int kWarp = 32;

// ------------------------------------------------------------ error word --
__device__ __forceinline__ void raise_error(uint32_t* err, uint32_t bit) { atomicOr(err, bit); }

// --------------------------------------------------------- element loads --
// bfloat16 is the upper half of an IEEE-754 binary32, so widening is a shift.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// 16 bytes -> 8 floats (bf16) or 4 floats (fp32).
template <bool BF16>
__device__ __forceinline__ void unpack16(const uint4& v, float* f)
{
    if constexpr (BF16) {
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
        f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
        f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    } else {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    }
}

// Streaming 16-byte load that does not allocate in L1 (data read exactly once).
__device__ __forceinline__ uint4 ld_stream16(const void* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Load one element of a q vector stored as bf16 or fp32 (runtime dtype).
__device__ __forceinline__ float load_q(const void* q, size_t idx, bool bf16)
{
    if (bf16) {
        uint16_t h = reinterpret_cast<const uint16_t*>(q)[idx];
        return __uint_as_float(uint32_t(h) << 16);
    }
    return reinterpret_cast<const float*>(q)[idx];
}

// N consecutive query elements from element idx (16-byte aligned for N = 8 bf16 or
// 4 fp32; 8-byte for 4 bf16), widened to fp32.
template <int N>
__device__ __forceinline__ void load_q_vec(const void* q, size_t idx, bool bf16, float* out)
{
    static_assert(N == 4 || N == 8, "4 or 8 elements");
    if (bf16) {
        const uint16_t* p = reinterpret_cast<const uint16_t*>(q) + idx;
        if constexpr (N == 8) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
            unpack16<true>(v, out);
        } else {
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
            out[0] = bf16_lo(v.x); out[1] = bf16_hi(v.x);
            out[2] = bf16_lo(v.y); out[3] = bf16_hi(v.y);
        }
    } else {
        const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(q) + idx);
#pragma unroll
        for (int i = 0; i < N / 4; ++i) {
            const float4 v = __ldg(p + i);
            out[4 * i] = v.x; out[4 * i + 1] = v.y; out[4 * i + 2] = v.z; out[4 * i + 3] = v.w;
        }
    }
}

// Round-trip of a float that holds a bf16 value back to its 16-bit pattern (exact).
__device__ __forceinline__ uint32_t f32_to_bf16_bits_exact(float x) { return __float_as_uint(x) >> 16; }

// ------------------------------------------------------ ordering of keys --
// Monotone map float -> uint32: a > b  <=>  key(a) > key(b) for non-NaN values.
// Finite scores never map to 0, which marks "not a candidate".
__device__ __forceinline__ uint32_t order_key(float f)
{
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ------------------------------------------------------- warp utilities --
__device__ __forceinline__ uint32_t lanemask_lt()
{
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ int warp_inclusive_scan(int v, int lane)
{
#pragma unroll
    for (int off = 1; off < kWarp; off <<= 1) {
        int t = __shfl_up_sync(kFullMask, v, off);
        if (lane >= off) v += t;
    }
    return v;
}

// Sum each of V values held by a lane over the groups of L consecutive lanes
// (L a power of two <= 32, xor-aligned).  "Transposed" halving: at every step a lane
// keeps half of its values and trades the other half with its partner, so reducing
// V values costs V - V/L shuffles instead of V * log2(L).  Afterwards lane
// (lane % L) holds, in v[0 .. max(1, V/L) - 1], the totals of value indices
//   (lane % L) * (V / L) + r            when V >= L, or
//   (lane % L) / (L / V)                when V <  L (one value, replicated).
template <int V, int L>
__device__ __forceinline__ void group_reduce_transposed(float (&v)[V], int lane)
{
    int n = V;
#pragma unroll
    for (int m = L / 2; m >= 1; m >>= 1) {
        if (n > 1) {
            const bool upper = (lane & m) != 0;
            const int half = n / 2;
#pragma unroll
            for (int i = 0; i < V / 2; ++i) {
                if (i < half) {
                    float send = upper ? v[i] : v[i + half];
                    float keep = upper ? v[i + half] : v[i];
                    v[i] = keep + __shfl_xor_sync(kFullMask, send, m);
                }
            }
            n = half;
        } else {
            v[0] += __shfl_xor_sync(kFullMask, v[0], m);
        }
    }
}

// --------------------------------------------------- mbarrier / bulk copy --
__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// 1-D bulk async copy global -> this CTA's shared memory, completion counted in bytes
// on `bar`.  Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of `bar` to complete, giving up after about `max_cycles`
// SM clocks.  Returns false on time-out (the caller records an error).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  long long max_cycles)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > max_cycles) return false;
    }
    return true;
}

// 2-D tiled bulk tensor copy (TMA) global -> this CTA's shared memory.  x is the
// innermost coordinate (elements; x * element size must be a multiple of 16 bytes),
// y the row; completion counted in bytes on `bar`.  `tmap` is the generic address of a
// CUtensorMap kernel parameter.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// 16-byte asynchronous copy global -> shared (L2 only); src_bytes < 16 zero-fills the
// rest (0: the source is not read at all).
__device__ __forceinline__ void cp_async_16_zfill(uint32_t dst, const void* src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait_group()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later async-proxy
// (bulk copy) writes to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------- warp-level MMA (bf16) --
// Four 8x8 b16 matrices from shared memory; lane i supplies the row address of row
// (i % 8) of matrix (i / 8).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D += A (16x16 bf16, row) * B (16x8 bf16, col), fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x2_trans(uint32_t addr, uint32_t& r0, uint32_t& r1)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
}

// Device-scope counter add with release (this CTA's writes, ordered before it by a
// CTA barrier) and acquire (other CTAs' writes, when this add completes a count).
__device__ __forceinline__ uint32_t atomic_add_acq_rel_u32(uint32_t* p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Programmatic dependent launch.  A kernel launched with launch_after_previous() may
// start while the previous kernel on the stream is still running; it must call
// grid_dependency_wait() before its first global-memory access, which returns once the
// previous kernel has completed and its writes are visible.  Kernels that call
// allow_dependents_early() let the next such kernel be scheduled before they finish.
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void allow_dependents_early()
{
    asm volatile("griddepcontrol.launch_dependents;" :::);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_after_previous(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                        cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// The same, in thread-block clusters of `cluster` consecutive CTAs.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_clusters_after_previous(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                                 unsigned cluster, cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---------------------------------------------------- thread-block clusters --
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster: arrive (release) and wait (acquire), so
// memory written before the barrier (shared memory of any CTA of the cluster, global
// memory) is visible to every thread of the cluster after it.
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address, in the shared-memory window of CTA `rank` of this cluster, of the variable
// at local shared address `local`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t local, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Two floats -> bf16x2 (round to nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// About one second at GB300 clocks: far beyond any legitimate copy latency.
constexpr long long kWaitCycles = 2000000000LL;


// Device-scope flag hand-off between CTAs of one grid: the writer publishes with a
// release store (after a fence that covers its CTA's writes), the reader polls with
// acquire loads.
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Device-scope release reduction (no value returned, so the thread does not wait for
// it): every earlier memory operation of this thread is ordered before the add.
__device__ __forceinline__ void red_add_release_gpu(uint32_t* p, uint32_t v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Wait until *flag == want, giving up after about `max_cycles` SM clocks (false).
__device__ __forceinline__ bool wait_flag_bounded(const uint32_t* flag, uint32_t want, long long max_cycles)
{
    if (ld_acquire_gpu(flag) == want) return true;
    const long long t0 = clock64();
    while (ld_acquire_gpu(flag) != want) {
        if (clock64() - t0 > max_cycles) return false;
        __nanosleep(32);
    }
    return true;
}

// Workspace header words (byte offsets from the workspace base; the error word is at 0).
constexpr int kHdrWaitLimit = int(kHdrWaitLimitByte);   // uint64: wait limit in SM clocks, 0 = kWaitCycles
constexpr int kHdrStepEpoch = 32;   // uint32: fused steps completed on this workspace
constexpr int kHdrStepDone = 36;    // uint32: CTAs of the running step that have finished
constexpr int kHdrQueueTail = 12;   // uint32: fused step: selections published to the queue
constexpr int kHdrQueueHead = 16;   // uint32: fused step: decode tickets taken
constexpr int kHdrRanked = 20;      // uint32: fused step: units ranked (queued or kept)

__device__ __forceinline__ uint32_t* header_word(uint32_t* err, int byte)
{
    return reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(err) + byte);
}

// The limit of the fused step's hand-off waits (a unit's selection published by another
// CTA, or by the select kernel launched just before), read once from the workspace
// header (`err` is the workspace base).  0 selects kWaitCycles; larger values are capped
// at it.  Waits inside a CTA's own pipeline (copy and MMA completions, the workers'
// wait for their control warp) always use kWaitCycles.
__device__ __forceinline__ long long handoff_wait_limit(const uint32_t* err)
{
    const unsigned long long v =
        __ldcg(reinterpret_cast<const unsigned long long*>(reinterpret_cast<const char*>(err) + kHdrWaitLimit));
    return (v == 0 || v > (unsigned long long)kWaitCycles) ? kWaitCycles : (long long)v;
}

// Per-unit hand-off of the fused step.  A step numbered E + 1 (E = the epoch word when
// it starts) publishes unit u's selection by storing E + 1 in ready[u]; its decode waits
// for that value.  Flags left by an earlier step (E or less, even one written late by a
// step whose waits ran out) never match, so no flag ever needs clearing.  The value 0
// (a fresh workspace) is skipped when the counter wraps.
__device__ __forceinline__ uint32_t step_flag_value(uint32_t* err)
{
    const uint32_t next = ld_acquire_gpu(header_word(err, kHdrStepEpoch)) + 1u;
    return next == 0u ? 1u : next;
}

// The end of one CTA's share of the launch that completes a step (the fused kernel, or
// the decode kernel behind the step's select kernel): the last CTA of the grid to
// finish resets the completion count and the publish queue's counters for the next
// step and stores the step's number as the new epoch.  After the kernel boundary every
// later launch sees them.
__device__ __forceinline__ void finish_step(uint32_t* err, uint32_t step_value)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        uint32_t* done = header_word(err, kHdrStepDone);
        if (atomic_add_acq_rel_u32(done, 1u) + 1u == gridDim.x) {
            *done = 0u;
            *header_word(err, kHdrQueueTail) = 0u;   // every CTA is past its publishes and tickets
            *header_word(err, kHdrQueueHead) = 0u;
            *header_word(err, kHdrRanked) = 0u;
            st_release_gpu(header_word(err, kHdrStepEpoch), step_value);
        }
    }
}

// exp2 on the special-function unit (PTX ex2.approx.ftz.f32; about 2 ulp).
__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace sa
