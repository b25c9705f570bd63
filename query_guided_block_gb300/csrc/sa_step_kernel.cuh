// The fused step kernel (selection and attention of one decode step in one cooperative
// grid) and its launcher, instantiated per head dimension by sa_step.cu (D = 128) and
// sa_step_d64.cu (D = 64).  The design notes are in sa_step.cu.
#pragma once

#include <limits.h>

#include "sa_decode_body.cuh"
#include "sa_select_body.cuh"

namespace sa {
namespace {

constexpr int kWorkerWarps = kDecWarps;                   // stream, then decode
constexpr int kCtlWarp = kWorkerWarps;                    // the control warp follows the workers
constexpr int kStepThreads = (kWorkerWarps + 1) * 32;
constexpr int kRankMaxKeys = 4096;   // candidates per unit the control warp ranks on chip
constexpr int kRankMaxRows = 8192;   // blocks per unit its reserve-set bitmap covers
constexpr int kRankList = 256;       // candidates kept once the k-th key is bracketed this tightly
constexpr int kGroupSlabs = 4;       // consecutive slabs of one unit a worker warp takes per visit

static_assert(kSlabSelStages * kSlabSelBytes == SlabShape<128>::STAGES * SlabShape<128>::SLAB_BYTES &&
                  kSlabSelStages * kSlabSelBytes == SlabShape<64>::STAGES * SlabShape<64>::SLAB_BYTES,
              "a worker warp's ring serves its select slabs and then its decode slabs");
constexpr int kWarpRingBytes = kSlabSelStages * kSlabSelBytes;
constexpr size_t kStepRingBytes = size_t(kWorkerWarps) * kWarpRingBytes;

// Dynamic shared memory of the fused kernel: alignment slack, worker rings, the decode
// range's page cache and the control warp's key row.
constexpr size_t kStepPageCacheBytes = size_t(2) * kMaxRangeBlocks * sizeof(int);
constexpr size_t step_smem_bytes()
{
    return 1024 + kStepRingBytes + kStepPageCacheBytes + size_t(kRankMaxKeys) * sizeof(uint32_t);
}

// The control warp's ranking scratch and the workers' streaming count (static shared memory).
struct RankSync {
    uint32_t list_key[kRankList];  // bracketed candidates (index order); reserve-set bitmap
    uint32_t list_idx[kRankList];
};

// Fused-step arguments beyond select and decode: the step's hand-off in the workspace.
struct StepArgs {
    uint32_t* ready;               // [units] flag value once a unit's selection is written
    unsigned long long* queue;     // [units] completed units: (flag value << 32) | (unit + 1)
    uint32_t* head;                // queue entries claimed by control warps
    uint32_t* tail;                // queue entries pushed by worker warps
    int units;
};

__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_gpu_u64(const unsigned long long* p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu_u64(unsigned long long* p, unsigned long long v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// ------------------------------------------------------------- streaming ---
// The slab list is unit-major and cut into groups of kGroupSlabs consecutive slabs of
// one unit.  Worker warp W (of NW = 8 per CTA x the grid) takes groups W, W + NW, ..., so
// every warp works near the same point of the list and units complete one after
// another through the whole phase instead of all at its end.  Per group the warp forms
// its unit's two coefficient vectors (the same partial-sum order as the select kernel,
// so the scores are the same bits; the query rows of the next group are loaded one group
// ahead), scores the group's slabs from its cp.async ring (the copy sequence runs
// across groups), stores the scores and adds the group's slot count to the unit's
// counter (release).  The warp whose count completes a unit resets the counter and
// queues the unit device-wide; the count's result is looked at one group later, so its
// round trip overlaps the next group.
template <int KIND, int D, int G, bool QSPLIT>
__device__ __forceinline__ void worker_stream(const SelectArgs& a, const StepArgs& st, uint32_t flag_value, unsigned char* ring_ptr,
                              uint32_t ring)
{
    using SS = SelectShape<KIND, KIND == KIND_QUEST, D>;
    using WS = SlabSelShape<KIND, KIND == KIND_QUEST, D>;
    constexpr int EPL = SS::EPL, LPR = SS::LPR, ROWS = WS::ROWS, R = WS::R;
    constexpr int S = kSlabSelStages;
    constexpr int RSTEP = kSelThreads / D;   // query-row classes of the select kernel's sum
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane % LPR, rsub = lane / LPR;
    const int d0 = sub * EPL;
    const char* hi_src = reinterpret_cast<const char*>(KIND == KIND_QUEST ? a.kmax : (const void*)a.kmean);
    const char* lo_src = reinterpret_cast<const char*>(a.kmin);
    const int W = blockIdx.x * kWorkerWarps + warp;
    const int NW = gridDim.x * kWorkerWarps;
    const int spu = a.chunks_per_unit;                         // slabs per unit
    const int gpu = (spu + kGroupSlabs - 1) / kGroupSlabs;      // groups per unit
    const int total_groups = st.units * gpu;
    const int n_groups = W < total_groups ? (total_groups - 1 - W) / NW + 1 : 0;

    // this warp's slab sequence: group gi = W + m * NW covers slabs [first, first + n)
    auto group_slabs = [&](int m, int& cid0, int& n) {
        const int gi = W + m * NW;
        const int u = gi / gpu, k = gi - u * gpu;
        cid0 = u * spu + k * kGroupSlabs;
        n = min(kGroupSlabs, spu - k * kGroupSlabs);
    };
    // copy slab number `i` of the sequence (group m, slab j of it) into stage st_
    int iss_m = 0, iss_j = 0;                                   // next slab to issue
    auto issue_next = [&](int st_) {
        if (iss_m >= n_groups) return;
        int cid0, n;
        group_slabs(iss_m, cid0, n);
        const ChunkInfo c = chunk_info(a, cid0 + iss_j, ROWS);
        const size_t off = (size_t(c.u) * a.row_stride + c.row0) * SS::ROW_BYTES;
        const uint32_t nbytes = uint32_t(c.nrows) * SS::ROW_BYTES;
        const uint32_t dst = ring + uint32_t(st_) * kSlabSelBytes;
#pragma unroll
        for (int arr = 0; arr < SS::ARRAYS; ++arr) {
            const char* src = (arr == 0 ? hi_src : lo_src) + off;
#pragma unroll
            for (int i = 0; i < WS::CPL; ++i) {
                const uint32_t byte = uint32_t(lane + i * 32) * 16;
                if (byte < nbytes) cp_async_16_zfill(dst + arr * (ROWS * SS::ROW_BYTES) + byte, src + byte, 16u);
            }
        }
        if (++iss_j == n) {
            iss_j = 0;
            ++iss_m;
        }
    };
    // query rows of a unit for this lane's channels (raw; converted when used)
    float qx[G][EPL];
    auto load_q_rows = [&](int m) {
        if (m >= n_groups) return;
        int cid0, n;
        group_slabs(m, cid0, n);
        const int u = cid0 / spu;
        const size_t qb = (size_t(u / a.Hkv) * a.Hq + size_t(u % a.Hkv) * G) * D + d0;
#pragma unroll
        for (int g = 0; g < G; ++g) load_q_vec<EPL>(a.q, qb + size_t(g) * D, !QSPLIT, qx[g]);
    };
    auto push = [&](int u) {   // lane 0: every slot of unit u is scored
        a.counters[u] = 0u;
        const uint32_t idx = atomicAdd(st.tail, 1u);
        if (idx < uint32_t(st.units))
            st_release_gpu_u64(st.queue + idx, (static_cast<unsigned long long>(flag_value) << 32) | uint32_t(u + 1));
        else
            raise_error(a.err, SPARSE_ATTN_ERR_CAPACITY);
    };

    load_q_rows(0);
#pragma unroll
    for (int k = 0; k < S - 1; ++k) {
        issue_next(k);
        cp_async_commit();
    }
    int pend_u = -1;
    uint32_t pend_old = 0, pend_n = 0;
    int slab = 0;   // slabs consumed so far (ring position)
    for (int m = 0; m < n_groups; ++m) {
        int cid0, n;
        group_slabs(m, cid0, n);
        const int u = cid0 / spu;
        // the unit's coefficient vectors for this lane's channels, then the next group's rows
        float cp[EPL], cn[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            float sp = 0.f, sn = 0.f;
#pragma unroll
            for (int k2 = 0; k2 < RSTEP; ++k2) {
                float pp = 0.f, nn = 0.f;
#pragma unroll
                for (int r = k2; r < G; r += RSTEP) {
                    if constexpr (KIND == KIND_QUEST) {
                        pp += fmaxf(qx[r][e], 0.f);
                        nn += fminf(qx[r][e], 0.f);
                    } else {
                        pp += qx[r][e];
                    }
                }
                sp += pp;
                sn += nn;
            }
            cp[e] = sp;
            cn[e] = sn;
        }
        load_q_rows(m + 1);
        uint32_t slots = 0;
        for (int j = 0; j < n; ++j, ++slab) {
            cp_async_wait_group<S - 2>();   // this lane's copies of this slab are done
            __syncwarp();                   // ... and every lane's; the stage read last is free
            issue_next((slab + S - 1) % S);
            cp_async_commit();
            const ChunkInfo c = chunk_info(a, cid0 + j, ROWS);
            const unsigned char* hi = ring_ptr + size_t(slab % S) * kSlabSelBytes + d0 * SS::ESZ;
            const unsigned char* lo = hi + ROWS * SS::ROW_BYTES;
            float part[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int row = rsub * R + r;
                float fh[EPL], acc = 0.f;
                unpack16<SS::ESZ == 2>(*reinterpret_cast<const uint4*>(hi + row * SS::ROW_BYTES), fh);
                if constexpr (KIND == KIND_QUEST) {
                    float fl[EPL];
                    unpack16<SS::ESZ == 2>(*reinterpret_cast<const uint4*>(lo + row * SS::ROW_BYTES), fl);
#pragma unroll
                    for (int e = 0; e < EPL; ++e) acc = fmaf(cp[e], fh[e], fmaf(cn[e], fl[e], acc));
                } else {
#pragma unroll
                    for (int e = 0; e < EPL; ++e) acc = fmaf(cp[e], fh[e], acc);
                }
                part[r] = acc;
            }
            group_reduce_transposed<R, LPR>(part, lane);
            {
                constexpr int OUT = R >= LPR ? R / LPR : 1;
                constexpr int SPREAD = R >= LPR ? 1 : LPR / R;
                float* srow = a.scores + size_t(c.u) * a.n_cand + c.cand0;
                if (sub % SPREAD == 0) {
#pragma unroll
                    for (int i = 0; i < OUT; ++i) {
                        const int r = R >= LPR ? sub * (R / LPR) + i : sub / SPREAD;
                        const int row = rsub * R + r;
                        if (row < c.nrows) srow[row] = part[i];
                    }
                }
            }
            slots += uint32_t(c.nslots);
        }
        __syncwarp();   // every lane's scores before lane 0's release count
        if (lane == 0) {
            const uint32_t old = atomic_add_acq_rel_u32(&a.counters[u], slots);
            if (pend_u >= 0 && pend_old + pend_n == uint32_t(a.n_cand)) push(pend_u);
            pend_u = u;
            pend_old = old;
            pend_n = slots;
        }
    }
    if (lane == 0 && pend_u >= 0 && pend_old + pend_n == uint32_t(a.n_cand)) push(pend_u);
    cp_async_wait_group<0>();
    __syncwarp();
}

// --------------------------------------------------------------- ranking ---
// The control warp ranks one completed unit exactly, without shared-memory atomics
// (scores of a unit cluster, so histogram bins would collide):
//   * the unit's scores come from L2 into shared memory as order keys (0: none);
//   * the k-th largest key T is found by bisection over key values, each probe a
//     count of keys >= t (every lane counts its keys, one warp reduction); once the
//     keys >= the lower bracket are at most kRankList they are gathered in index order
//     and the remaining probes count only them;
//   * the selection is {key > T} plus, among keys == T, the lowest indices up to k
//     (lower block id first), emitted in ascending order by ballots, then the window;
//     with a reserve set the top-k rows and the reserve blocks go through a bitmap.
// The unit is then published (fence + release store of the step's flag value).
__device__ __forceinline__ void rank_unit(const SelectArgs& a, int u, uint32_t* keys, RankSync& rs,
                                          uint32_t* ready, uint32_t flag_value)
{
    const int lane = threadIdx.x & 31;
    const uint32_t lt = lanemask_lt();
    // single-level selection: candidate c is block row c when c < row_limit (the kernel
    // parameters are read once, into registers)
    const int n = a.n_cand;
    const int lim = min(a.n_cand, a.row_limit);
    const int n128 = (n + 127) & ~127;
    const int k_req = a.k, rows = a.rows, win_first = a.win_first, win_count = a.win_count;
    const int n_reserve = a.n_reserve;
    const int32_t* reserve = a.reserve;
    uint32_t* err = a.err;
    int32_t* out = a.out_ids + size_t(u) * a.out_stride;
    int32_t* out_count = a.out_count;
    const float* row = a.scores + size_t(u) * a.n_cand;
    for (int c = lane; c < n; c += 32) cp_async_4(smem_u32(keys + c), row + c);
    cp_async_commit();
    cp_async_wait_group<0>();
    __syncwarp();
    uint32_t lo = 0xffffffffu, hi = 0u;
    int nv = 0;
#pragma unroll 8
    for (int c = lane; c < n128; c += 32) {
        uint32_t key = 0u;
        if (c < lim) key = order_key(__uint_as_float(keys[c]));
        keys[c] = key;
        if (key) {
            lo = min(lo, key);
            hi = max(hi, key);
            ++nv;
        }
    }
    nv = __reduce_add_sync(kFullMask, nv);
    lo = __reduce_min_sync(kFullMask, lo);
    hi = __reduce_max_sync(kFullMask, hi);
    __syncwarp();
    const int k_eff = min(k_req, nv);
    const uint4* keys4 = reinterpret_cast<const uint4*>(keys);
    auto count_all = [&](uint32_t t) -> int {   // keys >= t (t > 0)
        int c = 0;
#pragma unroll 8
        for (int i = lane; i < n128 / 4; i += 32) {
            const uint4 v = keys4[i];
            c += (v.x >= t) + (v.y >= t) + (v.z >= t) + (v.w >= t);
        }
        return __reduce_add_sync(kFullMask, c);
    };
    int nl = 0;   // gathered candidates (0: not gathered)
    auto count_list = [&](uint32_t t) -> int {
        int c = 0;
#pragma unroll 8
        for (int i = lane; i < nl; i += 32) c += rs.list_key[i] >= t;
        return __reduce_add_sync(kFullMask, c);
    };
    auto gather = [&](uint32_t t) {   // keys >= t into the list, index order
        int run = 0;
#pragma unroll 4
        for (int c0 = 0; c0 < n128; c0 += 32) {
            const uint32_t key = keys[c0 + lane];
            const bool in = key >= t && key != 0u;
            const uint32_t b = __ballot_sync(kFullMask, in);
            if (in) {
                rs.list_key[run + __popc(b & lt)] = key;
                rs.list_idx[run + __popc(b & lt)] = uint32_t(c0 + lane);
            }
            run += __popc(b);
        }
        __syncwarp();
        nl = run;
    };

    bool all = k_eff > 0 && k_eff >= nv;   // every candidate
    uint32_t T = 0xffffffffu;
    int cT = -1;
    if (k_eff > 0 && !all) {
        // bisection: count(>= tl) >= k_eff > count(>= th + 1)
        uint32_t tl = lo, th = hi;
        int cnt_l = nv;
        while (tl < th) {
            const uint32_t mid = tl + ((th - tl) >> 1) + 1u;
            const int c = nl > 0 ? count_list(mid) : count_all(mid);
            if (c >= k_eff) {
                tl = mid;
                cnt_l = c;
            } else {
                th = mid - 1u;
            }
            if (nl == 0 && cnt_l <= kRankList) gather(tl);
        }
        T = tl;
        if (nl == 0 && cnt_l <= kRankList) gather(T);
        // among keys == T, the lowest indices fill the remaining places
        const int above = T == 0xffffffffu ? 0 : (nl > 0 ? count_list(T + 1u) : count_all(T + 1u));
        const int krem = k_eff - above;
        int run = 0, hit = -1;
        const int limit = nl > 0 ? nl : n128;
        for (int c0 = 0; c0 < limit; c0 += 32) {
            const int p = c0 + lane;
            const uint32_t key = nl > 0 ? (p < nl ? rs.list_key[p] : 0u) : keys[p];
            const bool e = key == T;
            const uint32_t b = __ballot_sync(kFullMask, e);
            if (e && run + __popc(b & lt) == krem - 1) hit = nl > 0 ? int(rs.list_idx[p]) : p;
            run += __popc(b);
        }
        cT = __reduce_max_sync(kFullMask, hit);
    }
    auto selected = [&](uint32_t key, int c) -> bool {
        if (key == 0u || k_eff == 0) return false;
        if (all) return true;
        return key > T || (key == T && c <= cT);
    };

    int total = 0;
    if (n_reserve > 0) {
        // Reserve set (SparDA page §3.4): top-k rows and reserve blocks outside the window
        // marked in a bitmap over block ids, emitted in ascending order
        __syncwarp();   // the gathered list is not used past here; its storage holds the bitmap
        uint32_t* bits = rs.list_key;        // <= kRankList words: rows <= kRankMaxRows
        const int nw = (rows + 31) >> 5;
        for (int i = lane; i < nw; i += 32) bits[i] = 0u;
        __syncwarp();
        for (int c = lane; c < lim; c += 32)
            if (selected(keys[c], c)) atomicOr(&bits[c >> 5], 1u << (c & 31));
        for (int i = lane; i < n_reserve; i += 32) {
            const int j = reserve[size_t(u) * n_reserve + i];
            if (j < 0 || j >= rows) raise_error(err, SPARSE_ATTN_ERR_SEL_ID);
            else if (j < win_first) atomicOr(&bits[j >> 5], 1u << (j & 31));
        }
        __syncwarp();
        for (int w0 = 0; w0 < nw; w0 += 32) {
            const int w = w0 + lane;
            const uint32_t m = w < nw ? bits[w] : 0u;
            const int cnt = __popc(m);
            int inc = cnt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int t = __shfl_up_sync(kFullMask, inc, off);
                if (lane >= off) inc += t;
            }
            int pos = total + inc - cnt;
            for (uint32_t mm = m; mm; mm &= mm - 1) out[pos++] = w * 32 + (__ffs(mm) - 1);
            total += __shfl_sync(kFullMask, inc, 31);
        }
    } else if (nl > 0 && !all) {
        for (int c0 = 0; c0 < nl; c0 += 32) {   // every selected key is in the list
            const int p = c0 + lane;
            const bool sel = p < nl && selected(rs.list_key[p], int(rs.list_idx[p]));
            const uint32_t b = __ballot_sync(kFullMask, sel);
            if (sel) out[total + __popc(b & lt)] = int(rs.list_idx[p]);
            total += __popc(b);
        }
    } else {
        for (int c0 = 0; c0 < n128; c0 += 32) {
            const int c = c0 + lane;
            const bool sel = c < lim && selected(keys[c], c);
            const uint32_t b = __ballot_sync(kFullMask, sel);
            if (sel) out[total + __popc(b & lt)] = c;
            total += __popc(b);
        }
    }
    for (int i = lane; i < win_count; i += 32) out[total + i] = win_first + i;
    if (lane == 0) out_count[u] = total + win_count;
    __syncwarp();
    if (lane == 0) {
        __threadfence();
        st_release_gpu(&ready[u], flag_value);
    }
    __syncwarp();
}

// ----------------------------------------------------------------- kernel ---
template <int KIND, int D, int G, bool QSPLIT>
__global__ void __launch_bounds__(kStepThreads, 1) step_kernel(SelectArgs sa_args, DecodeArgs da, StepArgs st)
{
    static_assert(SlabShape<D>::RING_BYTES == kStepRingBytes, "the decode rings are the streaming rings");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;   // the decode swizzle repeats every 1024 bytes
    unsigned char* smem = smem_raw + (base - raw);
    uint32_t* keys = reinterpret_cast<uint32_t*>(smem + kStepRingBytes + kStepPageCacheBytes);
    __shared__ RankSync rs;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    grid_dependency_wait();   // inputs and workspace may come from the previous kernel
    const uint32_t flag_value = step_flag_value(sa_args.err);

    if (warp == kCtlWarp) {
        // control warp: rank completed units taken from the device-wide queue (whichever
        // control warp is free takes the next position)
        int claim = -1;               // queue position this warp ranks once it is filled
        long long idle_since = -1;    // no progress since then (bounded like every wait)
        while (true) {
            if (claim < 0) {
                uint32_t h = 0;
                if (lane == 0) h = atomicAdd(st.head, 1u);
                h = __shfl_sync(kFullMask, h, 0);
                if (h >= uint32_t(st.units)) break;   // every position is taken
                claim = int(h);
                idle_since = -1;
            }
            unsigned long long v = 0;
            if (lane == 0) v = ld_acquire_gpu_u64(st.queue + claim);
            v = __shfl_sync(kFullMask, v, 0);
            __syncwarp();
            if (uint32_t(v >> 32) == flag_value) {
                rank_unit(sa_args, int(uint32_t(v)) - 1, keys, rs, st.ready, flag_value);
                claim = -1;
                continue;
            }
            const long long now = clock64();
            if (idle_since < 0) idle_since = now;
            if (now - idle_since > kWaitCycles) {
                if (lane == 0) raise_error(sa_args.err, SPARSE_ATTN_ERR_TIMEOUT);
                break;
            }
            __nanosleep(128);
        }
    } else {
        const uint32_t ring = base + uint32_t(warp) * kWarpRingBytes;
        worker_stream<KIND, D, G, QSPLIT>(sa_args, st, flag_value, smem + size_t(warp) * kWarpRingBytes, ring);
        decode_mma_body<D, G, QSPLIT>(da, st.ready, flag_value);   // waits per unit on the published selections
    }
    finish_step(sa_args.err, flag_value);
}

template <int KIND, int D, int G, bool QSPLIT>
cudaError_t launch_step_t(const SelectArgs& sa_args, const DecodeArgs& da, const StepArgs& st, int ctas,
                          cudaStream_t s)
{
    constexpr size_t smem = step_smem_bytes();
    auto kernel = step_kernel<KIND, D, G, QSPLIT>;
    static std::atomic<unsigned long long> configured{0};   // devices set up
    const cudaError_t set_up = once_per_device(configured, [&]() -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kStepThreads, smem);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) return cudaErrorNotSupported;
        return cudaSuccess;
    });
    if (set_up != cudaSuccess) return set_up;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(ctas));
    cfg.blockDim = dim3(kStepThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // all CTAs resident: every wait on another CTA ends
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, sa_args, da, st);
}

template <int KIND, int D, bool QSPLIT>
cudaError_t dispatch_step_g(const SelectArgs& sa_args, const DecodeArgs& da, const StepArgs& st, int ctas, int G,
                            cudaStream_t s)
{
    switch (G) {
        case 1: return launch_step_t<KIND, D, 1, QSPLIT>(sa_args, da, st, ctas, s);
        case 2: return launch_step_t<KIND, D, 2, QSPLIT>(sa_args, da, st, ctas, s);
        case 4: return launch_step_t<KIND, D, 4, QSPLIT>(sa_args, da, st, ctas, s);
        case 8: return launch_step_t<KIND, D, 8, QSPLIT>(sa_args, da, st, ctas, s);
        default: return cudaErrorInvalidValue;
    }
}

// CTAs of the single-launch step (one per SM, fewer when there are fewer decode items),
// or 0 when the problem runs as two kernels: the control warp holds at most
// kRankMaxKeys candidate keys of a unit (and a bitmap of kRankMaxRows blocks for a
// reserve set), and every CTA's decode range must fit its page cache and touch at most
// 62 units -- the decode kernel's own grid is then the same, so both cut the decode
// into the same partials and give the same bits.
template <int D>
int step_single_ctas(const Geometry& g, const WorkspaceLayout& L)
{
    const int units = g.units();
    if (units == 0 || g.n_cand > kRankMaxKeys) return 0;
    if (g.n_reserve > 0 && g.nb > kRankMaxRows) return 0;
    const long long items = (long long)units * L.max_splits;
    long long ctas = num_sms();
    if (ctas > items) ctas = items;
    const long long min_ctas = (items * L.blocks_per_split + kMaxRangeBlocks - 1) / kMaxRangeBlocks;
    const long long min_ctas_units = (units + 61) / 62;
    if (ctas < 1 || ctas < min_ctas || ctas < min_ctas_units) return 0;
    return int(ctas);
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
    StepArgs st{};
    st.ready = reinterpret_cast<uint32_t*>(ws + L.ready);
    st.queue = reinterpret_cast<unsigned long long*>(ws + L.rank_queue);
    st.head = reinterpret_cast<uint32_t*>(ws + L.err + kHdrRankHeadByte);
    st.tail = reinterpret_cast<uint32_t*>(ws + L.err + kHdrRankTailByte);
    st.units = units;

    const bool qs = !g.q_bf16;
    if (mean)
        return qs ? dispatch_step_g<KIND_MEAN, D, true>(sa_args, da, st, ctas, g.G, s)
                  : dispatch_step_g<KIND_MEAN, D, false>(sa_args, da, st, ctas, g.G, s);
    return qs ? dispatch_step_g<KIND_QUEST, D, true>(sa_args, da, st, ctas, g.G, s)
              : dispatch_step_g<KIND_QUEST, D, false>(sa_args, da, st, ctas, g.G, s);
}

}  // namespace
}  // namespace sa
