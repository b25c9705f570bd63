// The fused step kernel (selection and attention of one decode step in one cooperative
// grid) and its launcher, instantiated per head dimension by sa_step.cu (D = 128) and
// sa_step_d64.cu (D = 64).  The design notes are in sa_step.cu.
#pragma once

#include <limits.h>

#include "sa_job_decode.cuh"
#include "sa_select_body.cuh"

namespace sa {
namespace {

constexpr int kRankMaxKeys = 4096;   // candidates per unit the control warp ranks on chip
constexpr int kRankMaxRows = 8192;   // blocks per unit its reserve-set bitmap covers
constexpr int kRankQueue = 256;      // units one CTA's worker warps may complete in a step
constexpr int kRankBins = 256;       // 8-bit radix digits

static_assert(kSlabSelStages * kSlabSelBytes == SlabShape<128>::STAGES * SlabShape<128>::SLAB_BYTES &&
                  kSlabSelStages * kSlabSelBytes == SlabShape<64>::STAGES * SlabShape<64>::SLAB_BYTES,
              "a worker warp's ring serves its select slabs and then its decode slabs");
constexpr int kWarpRingBytes = kSlabSelStages * kSlabSelBytes;
constexpr size_t kStepRingBytes = size_t(kWorkerWarps) * kWarpRingBytes;

// Dynamic shared memory of the fused kernel: alignment slack, worker rings, the decode
// job descriptors and the control warp's key row.
constexpr size_t step_smem_bytes()
{
    return 1024 + kStepRingBytes + size_t(kJobRing) * sizeof(JobDesc) + size_t(kRankMaxKeys) * sizeof(uint32_t);
}

// Worker -> control-warp hand-off of completed units (static shared memory).
struct RankSync {
    int q[kRankQueue];        // unit + 1 of each completed unit, in push order (0: not yet stored)
    int tail;                 // pushes so far
    int stream_done;          // worker warps that finished streaming
    uint32_t hist[kRankBins]; // radix histogram; gather list; reserve-set bitmap
};

__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// ------------------------------------------------------------- streaming ---
// Worker warp W (of NW = 8 per CTA x the grid) scores the 8 KB metadata slabs W, W + NW,
// W + 2 NW, ... of the unit-major slab list, so every warp works near the same point of
// the list and units complete one after another through the whole phase instead of
// all at its end.  Per slab the warp forms its unit's two coefficient vectors from the
// query (the same partial-sum order as the select kernel, so the scores are the same
// bits), scores the rows from its cp.async ring, stores them and adds the slab's slot
// count to the unit's counter (release); the warp whose count completes a unit resets
// the counter and queues the unit for the control warp.  A count's result is looked at
// one slab later, so its round trip overlaps the next slab.
template <int KIND, int D, int G>
__device__ void worker_stream(const SelectArgs& a, RankSync& rs, unsigned char* ring_ptr, uint32_t ring)
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
    const int n_mine = W < a.total_chunks ? (a.total_chunks - 1 - W) / NW + 1 : 0;

    auto issue = [&](int k, int st) {
        if (k >= n_mine) return;
        const ChunkInfo c = chunk_info(a, W + k * NW, ROWS);
        const size_t off = (size_t(c.u) * a.row_stride + c.row0) * SS::ROW_BYTES;
        const uint32_t nbytes = uint32_t(c.nrows) * SS::ROW_BYTES;
        const uint32_t dst = ring + uint32_t(st) * kSlabSelBytes;
#pragma unroll
        for (int arr = 0; arr < SS::ARRAYS; ++arr) {
            const char* src = (arr == 0 ? hi_src : lo_src) + off;
#pragma unroll
            for (int i = 0; i < WS::CPL; ++i) {
                const uint32_t byte = uint32_t(lane + i * 32) * 16;
                if (byte < nbytes) cp_async_16_zfill(dst + arr * (ROWS * SS::ROW_BYTES) + byte, src + byte, 16u);
            }
        }
    };
    auto push = [&](int u) {   // lane 0: every slot of unit u is scored
        a.counters[u] = 0u;
        const int idx = atomicAdd(&rs.tail, 1);
        if (idx < kRankQueue) st_release_cta_shared(&rs.q[idx], u + 1);
        else raise_error(a.err, SPARSE_ATTN_ERR_CAPACITY);
    };

#pragma unroll
    for (int k = 0; k < S - 1; ++k) {
        issue(k, k);
        cp_async_commit();
    }
    int pend_u = -1;
    uint32_t pend_old = 0, pend_n = 0;
    for (int k = 0; k < n_mine; ++k) {
        cp_async_wait_group<S - 2>();   // this lane's copies of slab k are done
        __syncwarp();                   // ... and every lane's; the stage read last is free
        issue(k + S - 1, (k + S - 1) % S);
        cp_async_commit();
        const ChunkInfo c = chunk_info(a, W + k * NW, ROWS);

        // the unit's coefficient vectors for this lane's channels
        float cp[EPL], cn[EPL];
        {
            float x[G][EPL];
            const size_t qb = (size_t(c.u / a.Hkv) * a.Hq + size_t(c.u % a.Hkv) * G) * D + d0;
#pragma unroll
            for (int g = 0; g < G; ++g) load_q_vec<EPL>(a.q, qb + size_t(g) * D, a.q_bf16 != 0, x[g]);
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                float sp = 0.f, sn = 0.f;
#pragma unroll
                for (int k2 = 0; k2 < RSTEP; ++k2) {
                    float pp = 0.f, nn = 0.f;
#pragma unroll
                    for (int r = k2; r < G; r += RSTEP) {
                        if constexpr (KIND == KIND_QUEST) {
                            pp += fmaxf(x[r][e], 0.f);
                            nn += fminf(x[r][e], 0.f);
                        } else {
                            pp += x[r][e];
                        }
                    }
                    sp += pp;
                    sn += nn;
                }
                cp[e] = sp;
                cn[e] = sn;
            }
        }
        const unsigned char* hi = ring_ptr + size_t(k % S) * kSlabSelBytes + d0 * SS::ESZ;
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
        __syncwarp();   // every lane's scores before lane 0's release count
        if (lane == 0) {
            const uint32_t old = atomic_add_acq_rel_u32(&a.counters[c.u], uint32_t(c.nslots));
            if (pend_u >= 0 && pend_old + pend_n == uint32_t(a.n_cand)) push(pend_u);
            pend_u = c.u;
            pend_old = old;
            pend_n = uint32_t(c.nslots);
        }
    }
    if (lane == 0 && pend_u >= 0 && pend_old + pend_n == uint32_t(a.n_cand)) push(pend_u);
    cp_async_wait_group<0>();
    __syncwarp();
    if (lane == 0) {
        __threadfence_block();
        atomicAdd(&rs.stream_done, 1);
    }
}

// --------------------------------------------------------------- ranking ---
// The control warp ranks one completed unit: its scores come from L2 into shared
// memory as order keys, an 8-bit radix select below the keys' common prefix narrows
// the k-th key to a bin of at most 32 (gathered and ranked directly) or to exact ties,
// and the selection {key > T, or key == T and index <= cT} (lower block id first) is
// emitted in ascending order by ballots, then the window; with a reserve set the top-k
// rows and the reserve blocks go through a bitmap first.  The unit is then published
// (fence + release store of the step's flag value).
__device__ void rank_unit(const SelectArgs& a, int u, uint32_t* keys, RankSync& rs, uint32_t* ready,
                          uint32_t flag_value)
{
    const int lane = threadIdx.x & 31;
    const uint32_t lt = lanemask_lt();
    const int n = a.n_cand;
    const int n32 = (n + 31) & ~31;
    const float* row = a.scores + size_t(u) * a.n_cand;
    for (int c = lane; c < n; c += 32) cp_async_4(smem_u32(keys + c), row + c);
    cp_async_commit();
    cp_async_wait_group<0>();
    __syncwarp();
    uint32_t lo = 0xffffffffu, hi = 0u;
    int nv = 0;
    for (int c = lane; c < n32; c += 32) {
        uint32_t key = 0u;
        if (c < n && candidate_row(a, u, c) >= 0) key = order_key(__uint_as_float(keys[c]));
        keys[c] = key;
        if (key) {
            lo = min(lo, key);
            hi = max(hi, key);
            ++nv;
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        nv += __shfl_xor_sync(kFullMask, nv, off);
        lo = min(lo, __shfl_xor_sync(kFullMask, lo, off));
        hi = max(hi, __shfl_xor_sync(kFullMask, hi, off));
    }
    __syncwarp();
    const int k_eff = min(a.k, nv);

    // mode 0: none; 1: (key & mask) >= prefix; 2: threshold (T, cT)
    int mode = 0;
    uint32_t prefix = 0u, mask = 0u, T = 0u;
    int cT = -1;
    if (k_eff > 0 && k_eff < nv) {
        int krem = k_eff;
        int low_bits = (lo == hi) ? 0 : 32 - __clz(lo ^ hi);
        mask = low_bits >= 32 ? 0u : ~((1u << low_bits) - 1u);
        prefix = hi & mask;
        uint32_t binc = uint32_t(nv);   // candidates matching the current prefix
        while (low_bits > 0 && binc > 32u && int(binc) != krem) {
            const int w = min(8, low_bits);
            const int shift = low_bits - w;
            const uint32_t dmask = (1u << w) - 1u;
            for (int i = lane; i < kRankBins; i += 32) rs.hist[i] = 0u;
            __syncwarp();
            for (int c = lane; c < n32; c += 32) {
                const uint32_t key = keys[c];
                if (key != 0u && (key & mask) == prefix) atomicAdd(&rs.hist[(key >> shift) & dmask], 1u);
            }
            __syncwarp();
            // lane l holds bins 255 - 8l .. 248 - 8l (descending); find the krem-th key
            uint32_t cnt[8], sum = 0u;
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                cnt[r] = rs.hist[kRankBins - 1 - 8 * lane - r];
                sum += cnt[r];
            }
            uint32_t inc = sum;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t t = __shfl_up_sync(kFullMask, inc, off);
                if (lane >= off) inc += t;
            }
            const uint32_t before = inc - sum;
            const bool mine = before < uint32_t(krem) && inc >= uint32_t(krem);
            uint32_t bin = 0u, above = 0u, bc = 0u;
            if (mine) {
                uint32_t acc = before;
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    if (acc + cnt[r] >= uint32_t(krem)) {
                        bin = uint32_t(kRankBins - 1 - 8 * lane - r);
                        above = acc;
                        bc = cnt[r];
                        break;
                    }
                    acc += cnt[r];
                }
            }
            const int src = __ffs(__ballot_sync(kFullMask, mine)) - 1;
            bin = __shfl_sync(kFullMask, bin, src);
            above = __shfl_sync(kFullMask, above, src);
            bc = __shfl_sync(kFullMask, bc, src);
            krem -= int(above);
            prefix |= bin << shift;
            mask |= dmask << shift;
            low_bits = shift;
            binc = bc;
            __syncwarp();   // the histogram is rewritten next pass
        }
        if (int(binc) == krem) {
            mode = 1;   // the whole boundary bin is in
        } else if (binc <= 32u) {
            // gather the boundary candidates (index order) and rank them by (key desc, index asc)
            uint32_t* g = rs.hist;   // keys at [0, 32), indices at [32, 64)
            int ng = 0;
            for (int c0 = 0; c0 < n32; c0 += 32) {
                const int c = c0 + lane;
                const uint32_t key = keys[c];
                const bool in = key != 0u && (key & mask) == prefix;
                const uint32_t b = __ballot_sync(kFullMask, in);
                if (in) {
                    const int slot = ng + __popc(b & lt);
                    g[slot] = key;
                    g[32 + slot] = uint32_t(c);
                }
                ng += __popc(b);
            }
            __syncwarp();
            const uint32_t mk = lane < ng ? g[lane] : 0u;
            const int mi = lane < ng ? int(g[32 + lane]) : INT_MAX;
            int rank = 0;
            for (int jj = 0; jj < ng; ++jj) {
                const uint32_t kj = __shfl_sync(kFullMask, mk, jj);
                const int ij = __shfl_sync(kFullMask, mi, jj);
                rank += (kj > mk) || (kj == mk && ij < mi);
            }
            const bool kth = lane < ng && rank == krem - 1;
            const int src = __ffs(__ballot_sync(kFullMask, kth)) - 1;
            T = __shfl_sync(kFullMask, mk, src);
            cT = __shfl_sync(kFullMask, mi, src);
            mode = 2;
            __syncwarp();
        } else {
            // more than 32 candidates share every key bit: the krem lowest indices are in
            T = prefix;
            int run = 0, hit = -1;
            for (int c0 = 0; c0 < n32; c0 += 32) {
                const int c = c0 + lane;
                const bool e = keys[c] == prefix;
                const uint32_t b = __ballot_sync(kFullMask, e);
                if (e && run + __popc(b & lt) == krem - 1) hit = c;
                run += __popc(b);
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) hit = max(hit, __shfl_xor_sync(kFullMask, hit, off));
            cT = hit;
            mode = 2;
        }
    } else if (k_eff > 0) {
        mode = 1;   // every candidate (mask = prefix = 0)
    }

    auto selected = [&](uint32_t key, int c) -> bool {
        if (mode == 0 || key == 0u) return false;
        if (mode == 1) return (key & mask) >= prefix;
        return key > T || (key == T && c <= cT);
    };
    int32_t* out = a.out_ids + size_t(u) * a.out_stride;
    int total = 0;
    if (a.n_reserve > 0) {
        // Reserve set (SparDA page §3.4): top-k rows and reserve blocks outside the window
        // marked in a bitmap over block ids, emitted in ascending order
        uint32_t* bits = rs.hist;
        const int nw = (a.rows + 31) >> 5;   // <= kRankBins words: rows <= kRankMaxRows
        for (int i = lane; i < nw; i += 32) bits[i] = 0u;
        __syncwarp();
        for (int c = lane; c < n; c += 32)
            if (selected(keys[c], c)) {
                const int r = candidate_row(a, u, c);
                atomicOr(&bits[r >> 5], 1u << (r & 31));
            }
        for (int i = lane; i < a.n_reserve; i += 32) {
            const int j = a.reserve[size_t(u) * a.n_reserve + i];
            if (j < 0 || j >= a.rows) raise_error(a.err, SPARSE_ATTN_ERR_SEL_ID);
            else if (j < a.win_first) atomicOr(&bits[j >> 5], 1u << (j & 31));
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
    } else {
        for (int c0 = 0; c0 < n32; c0 += 32) {
            const int c = c0 + lane;
            const bool sel = c < n && selected(keys[c], c);
            const uint32_t b = __ballot_sync(kFullMask, sel);
            if (sel) out[total + __popc(b & lt)] = candidate_row(a, u, c);
            total += __popc(b);
        }
    }
    for (int i = lane; i < a.win_count; i += 32) out[total + i] = a.win_first + i;
    if (lane == 0) a.out_count[u] = total + a.win_count;
    __syncwarp();
    if (lane == 0) {
        __threadfence();
        st_release_gpu(&ready[u], flag_value);
    }
    __syncwarp();
}

// ----------------------------------------------------------------- kernel ---
template <int KIND, int D, int G, bool QSPLIT>
__global__ void __launch_bounds__(kJobThreads, 1)
    step_kernel(SelectArgs sa_args, DecodeArgs da, JobArgs ja, uint32_t* ready)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;   // the decode swizzle repeats every 1024 bytes
    unsigned char* smem = smem_raw + (base - raw);
    JobDesc* desc = reinterpret_cast<JobDesc*>(smem + kStepRingBytes);
    uint32_t* keys = reinterpret_cast<uint32_t*>(smem + kStepRingBytes + size_t(kJobRing) * sizeof(JobDesc));
    __shared__ JobSync js;
    __shared__ RankSync rs;

    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) {
        js.consumed = 0;
        js.merge_unit = -1;
        js.avail = -1;
        js.end_job = INT_MAX;
        js.abort = 0;
        js.workers_done = 0;
        rs.tail = 0;
        rs.stream_done = 0;
    }
    for (int i = tid; i < kRankQueue; i += kJobThreads) rs.q[i] = 0;
    if (tid < kJobRing) desc[tid].seq = 0;
    grid_dependency_wait();   // inputs and workspace may come from the previous kernel
    const uint32_t flag_value = step_flag_value(sa_args.err);
    const long long wait_cycles = wait_limit(sa_args.err);
    __syncthreads();

    if (warp == kCtlWarp) {
        // control warp: rank the units this CTA's workers complete, feed decode jobs
        JobFeeder f{0, 0, 0, -1, false};
        int head = 0;
        long long idle_since = -1;   // no progress since then (bounded like every wait)
        while (true) {
            if (head < kRankQueue) {
                const int v = ld_acquire_cta_shared(&rs.q[head]);
                if (v != 0) {
                    rank_unit(sa_args, v - 1, keys, rs, ready, flag_value);
                    ++head;
                    idle_since = -1;
                    continue;
                }
            }
            if (feeder_step<D, G, QSPLIT>(f, da, ja, desc, js, ready, flag_value, wait_cycles)) {
                idle_since = -1;
                continue;
            }
            if (ld_acquire_cta_shared(&rs.stream_done) == kWorkerWarps &&
                head >= min(ld_acquire_cta_shared(&rs.tail), kRankQueue) &&
                (f.ended || ld_acquire_cta_shared(&js.workers_done) != 0))
                break;
            const long long now = clock64();
            if (idle_since < 0) idle_since = now;
            if (now - idle_since > 2 * wait_cycles) {
                if ((threadIdx.x & 31) == 0) raise_error(sa_args.err, SPARSE_ATTN_ERR_TIMEOUT);
                break;
            }
            __nanosleep(64);
        }
    } else {
        const uint32_t ring = base + uint32_t(warp) * kWarpRingBytes;
        worker_stream<KIND, D, G>(sa_args, rs, smem + size_t(warp) * kWarpRingBytes, ring);
        worker_decode<D, G, QSPLIT>(da, ja, desc, js, smem, ring, wait_cycles);
    }
    finish_jobs(sa_args.err, true, flag_value);
}

template <int KIND, int D, int G, bool QSPLIT>
cudaError_t launch_step_t(const SelectArgs& sa_args, const DecodeArgs& da, const JobArgs& ja, uint32_t* ready,
                          int ctas, cudaStream_t s)
{
    constexpr size_t smem = step_smem_bytes();
    auto kernel = step_kernel<KIND, D, G, QSPLIT>;
    static std::atomic<unsigned long long> configured{0};   // devices set up
    const cudaError_t set_up = once_per_device(configured, [&]() -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kJobThreads, smem);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) return cudaErrorNotSupported;
        return cudaSuccess;
    });
    if (set_up != cudaSuccess) return set_up;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(ctas));
    cfg.blockDim = dim3(kJobThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // all CTAs resident: every wait on another CTA ends
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, sa_args, da, ja, ready);
}

template <int KIND, int D, bool QSPLIT>
cudaError_t dispatch_step_g(const SelectArgs& sa_args, const DecodeArgs& da, const JobArgs& ja, uint32_t* ready,
                            int ctas, int G, cudaStream_t s)
{
    switch (G) {
        case 1: return launch_step_t<KIND, D, 1, QSPLIT>(sa_args, da, ja, ready, ctas, s);
        case 2: return launch_step_t<KIND, D, 2, QSPLIT>(sa_args, da, ja, ready, ctas, s);
        case 4: return launch_step_t<KIND, D, 4, QSPLIT>(sa_args, da, ja, ready, ctas, s);
        case 8: return launch_step_t<KIND, D, 8, QSPLIT>(sa_args, da, ja, ready, ctas, s);
        default: return cudaErrorInvalidValue;
    }
}

// CTAs of the single-launch step (one per SM), or 0 when the problem runs as two
// kernels: the control warp holds at most kRankMaxKeys candidate keys of a unit (and
// a bitmap of kRankMaxRows blocks for a reserve set), and the units a CTA's workers can
// complete must fit its queue.
template <int D>
int step_single_ctas(const Geometry& g)
{
    const int units = g.units();
    if (units == 0 || g.n_cand > kRankMaxKeys) return 0;
    if (g.n_reserve > 0 && g.nb > kRankMaxRows) return 0;
    const int rows = g.score_kind == SPARSE_ATTN_SCORE_MEAN ? SlabSelShape<KIND_MEAN, false, D>::ROWS
                                                           : SlabSelShape<KIND_QUEST, true, D>::ROWS;
    const long long slabs = (long long)units * (((g.n_cand > 0 ? g.n_cand : 1) + rows - 1) / rows);
    const long long ctas = num_sms();
    const long long per_warp = (slabs + ctas * kWorkerWarps - 1) / (ctas * kWorkerWarps);
    if (per_warp * kWorkerWarps > kRankQueue) return 0;
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
    const int ctas = step_single_ctas<D>(g);
    if (ctas == 0) return cudaErrorNotSupported;
    const bool mean = g.score_kind == SPARSE_ATTN_SCORE_MEAN;

    SelectArgs sa_args = select_args_base(g, L, ws, q, kmin, kmax, kmean);
    set_single_level(sa_args, g, reserve_ids, sel_ids, sel_count);
    if (mean) set_slab_chunking<KIND_MEAN, false, D>(sa_args, units);
    else set_slab_chunking<KIND_QUEST, true, D>(sa_args, units);
    DecodeArgs da = decode_args(g, L, ws, q, k_pages, v_pages, block_table, sel_ids, sel_count, out, nullptr, 0);
    const JobArgs ja = job_args(g, L, ws);
    uint32_t* ready = reinterpret_cast<uint32_t*>(ws + L.ready);

    const bool qs = !g.q_bf16;
    if (mean)
        return qs ? dispatch_step_g<KIND_MEAN, D, true>(sa_args, da, ja, ready, ctas, g.G, s)
                  : dispatch_step_g<KIND_MEAN, D, false>(sa_args, da, ja, ready, ctas, g.G, s);
    return qs ? dispatch_step_g<KIND_QUEST, D, true>(sa_args, da, ja, ready, ctas, g.G, s)
              : dispatch_step_g<KIND_QUEST, D, false>(sa_args, da, ja, ready, ctas, g.G, s);
}

}  // namespace
}  // namespace sa
