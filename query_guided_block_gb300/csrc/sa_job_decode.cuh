// Job-based bf16 decode: eight worker warps stream K/V slabs on tensor cores, a control
// warp hands them resolved jobs.  Shared by the decode kernel and the fused step kernel.
//
// Exact softmax attention over the selected tokens ("从HiSparse到QSA的移植实战" §3.3: the
// kernel walks the selected block ids and reads only their KV; SGLang page §1.2: select,
// then compute) cut into jobs: job k of unit u is its selection slots [k*J, (k+1)*J) with
// J = 256 / block_size, i.e. 256 tokens.  A job always produces one (m, l, o) partial
// at slot k, whoever runs it, and the unit's jobs are merged in slot order, so the
// result does not depend on which CTA ran which job.
//
//   * Control warp (the feeder): takes job tickets from a device-wide counter (so CTAs
//     that run faster take more jobs), waits without blocking for the unit's selection
//     when a select runs in the same grid or just before (ready flags), and resolves the
//     job's slots -> selected block -> page (bounds-checked) into a descriptor ring in
//     shared memory, kJobRing jobs ahead of the workers, with the unit's bf16 query rows.
//   * Worker warp w runs slabs w and w + 8 of every job (16 tokens each) through its own
//     cp.async ring of slabs; its copy sequence runs across job boundaries, so the next
//     job's tokens are already in flight while a job ends.  S = q K^T and O += P V use
//     mma.sync m16n8k16 with the softmax on the fragments (the layout notes are in
//     sa_decode_body.cuh).
//   * At the end of a job the eight warps combine their (m, l, o) through shared memory
//     (two worker-only named barriers per job), write the job's partial and count it;
//     the count's result is looked at one job later, so its round trip overlaps the next
//     job, and the CTA that counted a unit's last job merges the unit (log-sum-exp over
//     its jobs, slot order).
#pragma once

#include "sa_decode_body.cuh"

namespace sa {
namespace {

constexpr int kJobSlabs = 16;                         // 16-token slabs per job
constexpr int kJobTokens = kJobSlabs * kSlabTokens;   // 256
constexpr int kJobMaxBlocks = kJobTokens / 8;         // blocks of a job at the smallest block size
constexpr int kWorkerWarps = 8;
constexpr int kWorkerThreads = kWorkerWarps * 32;
constexpr int kCtlWarp = kWorkerWarps;                // the control warp follows the workers
constexpr int kJobThreads = kWorkerThreads + 32;
constexpr int kJobRing = 8;                           // descriptors resolved ahead of the workers
constexpr int kJobBatch = 4;                          // jobs the feeder resolves side by side
constexpr int kJobQWords = 256;                       // a unit's bf16 query rows when G * D <= 512
constexpr int kJobEnd = -1;
constexpr int kBarWorkers = 1;                        // named barrier of the 256 worker threads
static_assert(kJobSlabs == 2 * kWorkerWarps, "two slabs per worker warp and job");

struct JobDesc {
    int seq;                  // local job number + 1 once filled (stored last, release)
    int unit;                 // kJobEnd: no more jobs
    int k;                    // job index within the unit
    int pad;
    int page[kJobMaxBlocks];  // page (or pool tile) of each of the job's blocks, -1 if none
    int valid[kJobMaxBlocks]; // tokens of that block (0 for an empty slot)
    uint32_t q[kJobQWords];   // the unit's query rows (bf16 queries with G * D <= 512)
};

// Whether the descriptor carries the unit's query rows (else the workers read them from
// global memory at the start of each job).
template <int D, int G, bool QSPLIT>
__host__ __device__ constexpr bool job_q_in_desc()
{
    return !QSPLIT && G * D / 2 <= kJobQWords;
}

// Bytes of dynamic shared memory the decode part needs: 1 KB alignment slack, the
// worker rings, the descriptor ring.
template <int D>
constexpr size_t job_decode_smem_bytes()
{
    return 1024 + size_t(kWorkerWarps) * SlabShape<D>::STAGES * SlabShape<D>::SLAB_BYTES +
           size_t(kJobRing) * sizeof(JobDesc);
}

__device__ __forceinline__ void worker_barrier()
{
    asm volatile("bar.sync %0, %1;" ::"n"(kBarWorkers), "n"(kWorkerThreads) : "memory");
}

__device__ __forceinline__ int ld_acquire_cta_shared(const int* p)
{
    int v;
    asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_cta_shared(int* p, int v)
{
    asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

// State the control warp and the workers share (static shared memory of the kernel).
struct JobSync {
    int consumed;             // jobs the workers have combined (worker thread 0 stores)
    int merge_unit;           // unit whose last job this CTA just counted, or -1
    int avail;                // descriptors the workers may read: local jobs [0, avail]
    int end_job;              // local job number of the end marker once seen (else large)
    int abort;                // a descriptor wait ran out: the workers stop
    int workers_done;         // the workers have left their job loop
    float m[kWorkerWarps][8], l[kWorkerWarps][8];
    int flush[kWorkerWarps];
};

// Arguments of the job scheme beyond DecodeArgs.
struct JobArgs {
    int job_blocks;           // selected blocks per job (256 / block_size)
    int jobs_per_unit;
    int total_jobs;
    int part_stride;          // partial slots per query head in the workspace (>= jobs_per_unit)
    uint32_t* ticket;         // device-wide next-job counter (workspace header)
};

// --------------------------------------------------------------- control warp --
// Feeder: produces descriptors for the CTA's jobs in order (local job j -> slot
// j % kJobRing).  Jobs come from the device-wide counter in batches of up to kJobBatch
// consecutive jobs (the next batch's ticket is taken while the current one resolves);
// a batch is resolved side by side, one group of 32 / kJobBatch lanes per job, so its
// chain of dependent loads (counts and ids, then the page table) is paid once per batch.
// step() does one non-blocking piece of work and reports whether it made progress; it
// never waits on another CTA, so the control warp can interleave it with the selection
// work of the fused step.
struct JobFeeder {
    int produced;             // descriptors filled
    int state;                // 0: need a batch, 1: selections not yet published, 2: resolve
    int first, count;         // the batch being resolved: jobs [first, first + count)
    int next;                 // start of the next batch (ticket taken ahead), -1 if none yet
    long long t0;             // first time a selection was found unpublished
    bool ended;
};

__device__ __forceinline__ JobFeeder feeder_init() { return JobFeeder{0, 0, 0, 0, -1, -1, false}; }

template <int D, int G, bool QSPLIT>
__device__ bool feeder_step(JobFeeder& f, const DecodeArgs& a, const JobArgs& ja, JobDesc* desc, const JobSync& js,
                            const uint32_t* ready, uint32_t flag_value, long long wait_cycles)
{
    const int lane = threadIdx.x & 31;
    // jobs per batch: one lane group (32 / batch lanes) per job must cover its blocks
    const int batch = ja.job_blocks <= 32 / kJobBatch ? kJobBatch : (ja.job_blocks <= 16 ? 2 : 1);
    if (f.ended) return false;
    const int room = kJobRing - (f.produced - *reinterpret_cast<const volatile int*>(&js.consumed));
    if (f.state == 0) {
        if (room < batch) return false;
        int t = f.next;
        if (t < 0) {
            if (lane == 0) t = int(atomicAdd(ja.ticket, uint32_t(batch)));
            t = __shfl_sync(kFullMask, t, 0);
        }
        if (t >= ja.total_jobs) {   // no more jobs: the end marker
            JobDesc& d = desc[f.produced % kJobRing];
            if (lane == 0) {
                d.unit = kJobEnd;
                d.k = 0;
                st_release_cta_shared(&d.seq, f.produced + 1);
            }
            __syncwarp();
            f.ended = true;
            return true;
        }
        f.first = t;
        f.count = min(batch, ja.total_jobs - t);
        // the next batch's ticket, in flight while this one resolves
        int nt = 0;
        if (lane == 0) nt = int(atomicAdd(ja.ticket, uint32_t(batch)));
        f.next = __shfl_sync(kFullMask, nt, 0);
        f.state = ready != nullptr ? 1 : 2;
        f.t0 = -1;
        return true;
    }
    if (f.state == 1) {   // the batch's units' selections, published by a select of this step
        int ok = 1;
        if (lane < f.count) ok = ld_acquire_gpu(ready + (f.first + lane) / ja.jobs_per_unit) == flag_value;
        ok = __all_sync(kFullMask, ok);
        __syncwarp();
        if (!ok) {
            const long long now = clock64();
            if (f.t0 < 0) f.t0 = now;
            if (now - f.t0 <= wait_cycles) return false;
            if (lane == 0) raise_error(a.err, SPARSE_ATTN_ERR_TIMEOUT);
        }
        f.state = 2;
        return true;
    }
    // resolve: lane group g handles job first + g; its lane e, slot k * J + e -> block -> page
    const int per = 32 / batch;
    const int g = lane / per, e = lane - g * per;
    const int t = f.first + g;
    const bool live = g < f.count;
    const int u = live ? t / ja.jobs_per_unit : 0;
    const int k = live ? t - u * ja.jobs_per_unit : 0;
    int page = -1, valid = 0;
    if (live && e < ja.job_blocks) {
        int count = a.sel_count[u];
        if (count < 0 || count > a.sel_stride) {
            if (e == 0) raise_error(a.err, SPARSE_ATTN_ERR_SEL_COUNT);
            count = count < 0 ? 0 : a.sel_stride;
        }
        const int slot = k * ja.job_blocks + e;
        if (slot < count) {
            const int j = a.sel_ids[size_t(u) * a.sel_stride + slot];
            if (j < 0 || j >= a.nb) {
                raise_error(a.err, SPARSE_ATTN_ERR_SEL_ID);
            } else if (a.slot_C > 0) {
                const int sl = a.sel_slot[size_t(u) * a.sel_stride + slot];
                if (sl < 0 || sl >= a.slot_C) {
                    raise_error(a.err, SPARSE_ATTN_ERR_SLOT);
                } else {
                    page = u * a.slot_C + sl;
                    valid = min(a.bs, a.N - j * a.bs);
                }
            } else {
                const int p = a.block_table[size_t(u / a.Hkv) * a.bt_stride + j];
                if (p < 0 || p >= a.num_pages) {
                    raise_error(a.err, SPARSE_ATTN_ERR_PAGE);
                } else {
                    page = p;
                    valid = min(a.bs, a.N - j * a.bs);
                }
            }
        }
    }
    for (int b = 0; b < f.count; ++b) {   // every descriptor of the batch: all of its block entries
        JobDesc& d = desc[(f.produced + b) % kJobRing];
        for (int x = lane; x < kJobMaxBlocks; x += 32) {
            const int src = b * per + x;   // lane holding entry x of job b (when x < per)
            const int pg = __shfl_sync(kFullMask, page, src & 31);
            const int vd = __shfl_sync(kFullMask, valid, src & 31);
            d.page[x] = x < per ? pg : -1;
            d.valid[x] = x < per ? vd : 0;
        }
        if constexpr (job_q_in_desc<D, G, QSPLIT>()) {   // the unit's G query rows are contiguous
            const int ub = (f.first + b) / ja.jobs_per_unit;
            const size_t head0 = size_t(ub / a.Hkv) * a.Hq + size_t(ub % a.Hkv) * G;
            const uint4* q4 = reinterpret_cast<const uint4*>(reinterpret_cast<const uint32_t*>(a.q) + head0 * D / 2);
            uint4* dq = reinterpret_cast<uint4*>(d.q);
            for (int w = lane; w < G * D / 8; w += 32) dq[w] = __ldg(q4 + w);
        }
    }
    __syncwarp();
    if (lane == 0) {
        for (int b = 0; b < f.count; ++b) {
            JobDesc& d = desc[(f.produced + b) % kJobRing];
            const int tb = f.first + b;
            d.unit = tb / ja.jobs_per_unit;
            d.k = tb - d.unit * ja.jobs_per_unit;
            st_release_cta_shared(&d.seq, f.produced + b + 1);
        }
    }
    __syncwarp();
    f.produced += f.count;
    f.state = 0;
    return true;
}

// ------------------------------------------------------------------- workers --
// The CTA that counted unit u's last job merges its jobs' partials (slot order): each
// thread loads the o values of its outputs and a share of the (m, l) pairs, kMergeChunk
// jobs at a time with every load of a chunk issued before any is used.
__device__ void merge_jobs(const DecodeArgs& a, const JobArgs& ja, int u, int G, int D)
{
    __shared__ float s_pm[8][kMergeChunk], s_pl[8][kMergeChunk];
    const int tid = threadIdx.x;
    const int b = u / a.Hkv, kvh = u - (u / a.Hkv) * a.Hkv;
    const size_t head0 = size_t(b) * a.Hq + size_t(kvh) * G;
    const int ps = ja.part_stride, nseg = ja.jobs_per_unit;
    if (tid == 0) a.counters[u] = 0u;
    float num[kMergeOut], den[kMergeOut], mrun[kMergeOut];
#pragma unroll
    for (int r = 0; r < kMergeOut; ++r) num[r] = den[r] = 0.f, mrun[r] = -INFINITY;
    for (int base = 0; base < nseg; base += kMergeChunk) {
        const int n = min(kMergeChunk, nseg - base);
        float ov[kMergeOut][kMergeChunk];
#pragma unroll
        for (int r = 0; r < kMergeOut; ++r) {
            const int i = tid + r * kWorkerThreads;
            const int g = i / D, d = i - (i / D) * D;
#pragma unroll
            for (int e = 0; e < kMergeChunk; ++e)
                ov[r][e] = (i < G * D && e < n) ? __ldcg(a.part_o + ((head0 + g) * ps + base + e) * D + d) : 0.f;
        }
        if (tid < G * kMergeChunk) {
            const int g = tid / kMergeChunk, e = tid - g * kMergeChunk;
            float pm = -INFINITY, pl = 0.f;
            if (e < n) {
                pm = __ldcg(a.part_m + (head0 + g) * ps + base + e);
                pl = __ldcg(a.part_l + (head0 + g) * ps + base + e);
            }
            s_pm[g][e] = pm;
            s_pl[g][e] = pl;
        }
        worker_barrier();
#pragma unroll
        for (int r = 0; r < kMergeOut; ++r) {
            const int i = tid + r * kWorkerThreads;
            if (i >= G * D) break;
            const int g = i / D;
            float mx = mrun[r];
#pragma unroll
            for (int e = 0; e < kMergeChunk; ++e) mx = fmaxf(mx, s_pm[g][e]);
            if (mx == -INFINITY) continue;                       // nothing valid yet
            const float resc = mrun[r] == -INFINITY ? 0.f : fast_exp2(mrun[r] - mx);
            float nu = num[r] * resc, de = den[r] * resc;
#pragma unroll
            for (int e = 0; e < kMergeChunk; ++e) {
                const float pm = s_pm[g][e];
                if (pm == -INFINITY) continue;                   // empty job (or past n)
                const float w = fast_exp2(pm - mx);
                nu = fmaf(w, ov[r][e], nu);
                de = fmaf(w, s_pl[g][e], de);
            }
            num[r] = nu;
            den[r] = de;
            mrun[r] = mx;
        }
        worker_barrier();                                        // s_pm / s_pl reused
    }
#pragma unroll
    for (int r = 0; r < kMergeOut; ++r) {
        const int i = tid + r * kWorkerThreads;
        if (i >= G * D) break;
        a.out[head0 * D + i] = den[r] > 0.f ? num[r] / den[r] : 0.f;
    }
}

// Descriptor window of the workers: thread 0 of the workers waits (bounded) until the
// descriptors of local jobs up to j_hi are filled, or the end marker shows up, and
// publishes how far the workers may read; callers put a worker barrier after it, so
// every worker warp takes the same decisions (no warp can stop at a named barrier that
// another warp never reaches).
__device__ void sync_job_window(const DecodeArgs& a, JobDesc* desc, JobSync& js, int j_hi, long long wait_cycles)
{
    if (threadIdx.x != 0) return;
    int x = js.avail + 1;
    for (; x <= j_hi && js.end_job > x && !js.abort; ++x) {
        const JobDesc& d = desc[x % kJobRing];
        if (ld_acquire_cta_shared(&d.seq) != x + 1) {
            const long long t0 = clock64();
            while (ld_acquire_cta_shared(&d.seq) != x + 1) {
                if (clock64() - t0 > wait_cycles) {
                    raise_error(a.err, SPARSE_ATTN_ERR_TIMEOUT);
                    js.abort = 1;
                    break;
                }
                __nanosleep(64);
            }
            if (js.abort) break;
        }
        if (d.unit == kJobEnd) {
            js.end_job = x;
            break;
        }
        js.avail = x;
    }
}

// One worker warp's share of the CTA's jobs, until the feeder's end marker.  `ring` is
// the shared-memory address of this warp's slab ring, `smem` the generic pointer of the
// (1 KB aligned) dynamic shared-memory base the ring offsets are taken from.
template <int D, int G, bool QSPLIT>
__device__ void worker_decode(const DecodeArgs& a, const JobArgs& ja, JobDesc* desc, JobSync& js,
                              unsigned char* smem, uint32_t ring, long long wait_cycles)
{
    using SS = SlabShape<D>;
    constexpr int S = SS::STAGES;
    constexpr int DT = SS::DT;
    constexpr int H = S / 2;   // jobs the copies run ahead of the job being computed
    static_assert(H + 1 + kJobBatch <= kJobRing, "the copies' descriptors and a batch must fit the ring");
    static_assert(G <= 8, "query rows live in the first 8 MMA rows");
    static_assert(8 * D * 4 <= SS::SLAB_BYTES, "a warp's G x D outputs must fit one stage");

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g4 = lane >> 2, t4 = lane & 3;
    const int bs_shift = __ffs(a.bs) - 1;
    const char* kbase = reinterpret_cast<const char*>(a.k_pages);
    const char* vbase = reinterpret_cast<const char*>(a.v_pages);
    const int cp_c = lane % SS::CPR, cp_r = lane / SS::CPR;
    const uint32_t ring_off = ring - smem_u32(smem);

    // the window of readable descriptors: jobs [0, avail], none at or past end_job
    sync_job_window(a, desc, js, H, wait_cycles);
    worker_barrier();
    int avail = js.avail, end_job = js.end_job;
    bool abort = js.abort != 0;

    // slab i of this warp: job i / 2, slab warp + 8 (i % 2) of the job
    auto issue_slab = [&](int i, int st) {
        const int j = i >> 1;
        if (j > avail || j >= end_job || abort) return;   // never consumed
        const JobDesc& d = desc[j % kJobRing];
        const int t0 = (warp + (i & 1) * kWorkerWarps) * kSlabTokens;   // first token in the job
        const size_t head_rows = a.slot_C > 0 ? 0 : size_t(d.unit % a.Hkv) * a.bs;
        const uint32_t kd = ring + uint32_t(st) * SS::SLAB_BYTES + uint32_t(cp_c >> 3) * SS::HALF_BYTES;
        const uint32_t vd = kd + SS::TENSOR_BYTES;
#pragma unroll
        for (int i2 = 0; i2 < SS::CP_ITERS; ++i2) {
            const int tr = cp_r + i2 * SS::RPI;                        // row within the slab
            const int t = t0 + tr;
            const int e = t >> bs_shift, r = t & (a.bs - 1);
            const bool ok = r < d.valid[e];
            const size_t off = ok ? ((size_t(d.page[e]) * a.page_heads * a.bs + head_rows + r) * (D * 2) + cp_c * 16) : 0;
            const uint32_t so = uint32_t(tr) * kRowBytes + uint32_t(((cp_c & 7) ^ (tr & 7)) << 4);
            cp_async_16_zfill(kd + so, kbase + off, ok ? 16u : 0u);
            cp_async_16_zfill(vd + so, vbase + off, ok ? 16u : 0u);
        }
    };

    uint32_t qa[D / 16][4];
    auto load_qfrag = [&](const JobDesc& d) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            if constexpr (job_q_in_desc<D, G, QSPLIT>()) {
                const int w = (g4 * D + ks * 16 + 2 * t4) / 2;
                qa[ks][0] = g4 < G ? d.q[w] : 0u;
                qa[ks][2] = g4 < G ? d.q[w + 4] : 0u;
                qa[ks][1] = qa[ks][3] = 0u;
            } else if constexpr (!QSPLIT) {
                const size_t head0 = size_t(d.unit / a.Hkv) * a.Hq + size_t(d.unit % a.Hkv) * G;
                const uint32_t* q32 = reinterpret_cast<const uint32_t*>(a.q);
                const size_t qrow = (head0 + g4) * D + ks * 16 + 2 * t4;
                qa[ks][0] = g4 < G ? __ldg(q32 + qrow / 2) : 0u;
                qa[ks][2] = g4 < G ? __ldg(q32 + qrow / 2 + 4) : 0u;
                qa[ks][1] = qa[ks][3] = 0u;
            } else {
                const size_t head0 = size_t(d.unit / a.Hkv) * a.Hq + size_t(d.unit % a.Hkv) * G;
                const size_t qrow = (head0 + g4) * D + ks * 16 + 2 * t4;
                const float2* q64 = reinterpret_cast<const float2*>(a.q);
                const float2 f0 = g4 < G ? __ldg(q64 + qrow / 2) : make_float2(0.f, 0.f);
                const float2 f2 = g4 < G ? __ldg(q64 + qrow / 2 + 4) : make_float2(0.f, 0.f);
                qa[ks][0] = pack_bf16x2(f0.x, f0.y);
                qa[ks][2] = pack_bf16x2(f2.x, f2.y);
                qa[ks][1] = pack_bf16x2(f0.x - bf16_lo(qa[ks][0]), f0.y - bf16_hi(qa[ks][0]));
                qa[ks][3] = pack_bf16x2(f2.x - bf16_lo(qa[ks][2]), f2.y - bf16_hi(qa[ks][2]));
            }
        }
    };

#pragma unroll
    for (int kk = 0; kk < S - 1; ++kk) {
        issue_slab(kk, kk);
        cp_async_commit();
    }

    float acc[DT][4];
    float m_run = -INFINITY, l_run = 0.f;
    int pend_u = -1;          // thread 0: unit of the last counted job and the count before it
    uint32_t pend_old = 0u;
    for (int j = 0; j <= avail && j < end_job && !abort; ++j) {
        const JobDesc& d = desc[j % kJobRing];
        load_qfrag(d);
#pragma unroll
        for (int jj = 0; jj < DT; ++jj) acc[jj][0] = acc[jj][1] = acc[jj][2] = acc[jj][3] = 0.f;
        m_run = -INFINITY;
        l_run = 0.f;
        for (int half = 0; half < 2; ++half) {
            const int i = 2 * j + half;
            cp_async_wait_group<S - 2>();   // this lane's copies of slab i are done
            __syncwarp();                   // ... and every lane's; the stage read last is free
            issue_slab(i + S - 1, (i + S - 1) % S);
            cp_async_commit();
            const uint32_t kst = ring + uint32_t(i % S) * SS::SLAB_BYTES;
            const uint32_t vst = kst + SS::TENSOR_BYTES;

            // ---- S = q K^T over the slab's two 8-token tiles -----------------------
            float c[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                c[nt][0] = c[nt][1] = c[nt][2] = c[nt][3] = 0.f;
#pragma unroll
                for (int kp = 0; kp < D / 32; ++kp) {
                    const int ch = kp * 4 + (lane >> 3);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(swz(kst + uint32_t(ch >> 3) * SS::HALF_BYTES, nt * 8 + (lane & 7), ch & 7), b0, b1, b2, b3);
                    mma_bf16_16816(c[nt], qa[2 * kp][0], qa[2 * kp][1], qa[2 * kp][2], qa[2 * kp][3], b0, b1);
                    mma_bf16_16816(c[nt], qa[2 * kp + 1][0], qa[2 * kp + 1][1], qa[2 * kp + 1][2], qa[2 * kp + 1][3],
                                   b2, b3);
                }
            }
            // ---- online softmax on the fragments ------------------------------------
            const int tb = (warp + half * kWorkerWarps) * kSlabTokens + 2 * t4;
            float sc[2][2];
            float mx = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int t = tb + nt * 8 + e;
                    const bool ok = (t & (a.bs - 1)) < d.valid[t >> bs_shift];
                    sc[nt][e] = ok ? (c[nt][e] + c[nt][e + 2]) * a.scale_log2 : -INFINITY;
                    mx = fmaxf(mx, sc[nt][e]);
                }
            mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 2));
            const float m_new = fmaxf(m_run, mx);
            const float alpha = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - m_new);
            m_run = m_new;
            float p[2][2];
            float psum = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    p[nt][e] = (sc[nt][e] == -INFINITY) ? 0.f : fast_exp2(sc[nt][e] - m_new);
                    psum += p[nt][e];
                }
            l_run = fmaf(l_run, alpha, psum);
            const uint32_t ph0 = pack_bf16x2(p[0][0], p[0][1]);
            const uint32_t ph2 = pack_bf16x2(p[1][0], p[1][1]);
            const uint32_t pl0 = pack_bf16x2(p[0][0] - bf16_lo(ph0), p[0][1] - bf16_hi(ph0));
            const uint32_t pl2 = pack_bf16x2(p[1][0] - bf16_lo(ph2), p[1][1] - bf16_hi(ph2));

            // ---- O += P V: all D channels, k = the slab's 16 tokens -----------------
#pragma unroll
            for (int jj = 0; jj < DT; ++jj) {
                acc[jj][0] *= alpha;
                acc[jj][1] *= alpha;
                acc[jj][2] *= alpha;
                acc[jj][3] *= alpha;
            }
#pragma unroll
            for (int jp = 0; jp < DT; jp += 2) {
                const int mtx = lane >> 3;
                const int chunk = jp + (mtx >> 1);
                uint32_t r0, r1, r2, r3;
                ldsm_x4_trans(swz(vst + uint32_t(chunk >> 3) * SS::HALF_BYTES, (mtx & 1) * 8 + (lane & 7), chunk & 7),
                              r0, r1, r2, r3);
                mma_bf16_16816(acc[jp], ph0, pl0, ph2, pl2, r0, r1);
                mma_bf16_16816(acc[jp + 1], ph0, pl0, ph2, pl2, r2, r3);
            }
        }

        // ---- end of job j: combine the eight warps into the job's partial -----------
        l_run += __shfl_xor_sync(kFullMask, l_run, 1);
        l_run += __shfl_xor_sync(kFullMask, l_run, 2);
        {
            const int free_off = int(ring_off) + ((2 * j + 1) % S) * SS::SLAB_BYTES;   // the stage just read
            float* ob = reinterpret_cast<float*>(smem + free_off);
            if (g4 < G) {
#pragma unroll
                for (int jj = 0; jj < DT; ++jj)
                    *reinterpret_cast<float2*>(ob + g4 * D + jj * 8 + 2 * t4) =
                        make_float2(acc[jj][0] + acc[jj][2], acc[jj][1] + acc[jj][3]);
                if (t4 == 0) {
                    js.m[warp][g4] = m_run;
                    js.l[warp][g4] = l_run;
                }
            }
            if (lane == 0) js.flush[warp] = free_off;
        }
        const int u = d.unit, k = d.k;
        worker_barrier();   // the flushes are written; descriptor j is not read again
        if (tid == 0) {
            st_release_cta_shared(&js.consumed, j + 1);
            // the previous job's count, issued one job ago: did it complete a unit?
            js.merge_unit = (pend_u >= 0 && pend_old + 1u == uint32_t(ja.jobs_per_unit)) ? pend_u : -1;
            sync_job_window(a, desc, js, j + 1 + H, wait_cycles);
        }
        {
            const size_t head0 = size_t(u / a.Hkv) * a.Hq + size_t(u % a.Hkv) * G;
            for (int o = tid; o < G * D; o += kWorkerThreads) {
                const int g = o / D, dd = o - g * D;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kWorkerWarps; ++w) M = fmaxf(M, js.m[w][g]);
                float ov = 0.f, lv = 0.f;
#pragma unroll
                for (int w = 0; w < kWorkerWarps; ++w) {
                    const float mw = js.m[w][g];
                    if (mw == -INFINITY) continue;   // a warp without a token here wrote nothing useful
                    const float wt = fast_exp2(mw - M);
                    ov = fmaf(wt, reinterpret_cast<const float*>(smem + js.flush[w])[g * D + dd], ov);
                    lv = fmaf(wt, js.l[w][g], lv);
                }
                const size_t ps = (head0 + g) * ja.part_stride + k;
                a.part_o[ps * D + dd] = ov;
                if (dd == 0) {
                    a.part_m[ps] = M;
                    a.part_l[ps] = lv;
                }
            }
        }
        worker_barrier();   // partial written, flush stages free; window and merge decision published
        if (tid == 0) {     // count the job (release); its result is looked at one job later
            pend_old = atomic_add_acq_rel_u32(&a.counters[u], 1u);
            pend_u = u;
        }
        avail = js.avail;
        end_job = js.end_job;
        abort = js.abort != 0;
        const int mu = js.merge_unit;
        if (mu >= 0) {
            merge_jobs(a, ja, mu, G, D);
            worker_barrier();
        }
    }
    // the last job's count
    if (tid == 0) js.merge_unit = (pend_u >= 0 && pend_old + 1u == uint32_t(ja.jobs_per_unit)) ? pend_u : -1;
    worker_barrier();
    if (js.merge_unit >= 0) merge_jobs(a, ja, js.merge_unit, G, D);
    cp_async_wait_group<0>();
    if (tid == 0) st_release_cta_shared(&js.workers_done, 1);
}

// Job arguments of a decode over `units` units.
inline JobArgs job_args(const Geometry& g, const WorkspaceLayout& L, char* ws)
{
    JobArgs j{};
    j.job_blocks = L.job_blocks;
    j.jobs_per_unit = L.jobs_per_unit;
    j.total_jobs = g.units() * L.jobs_per_unit;
    j.part_stride = L.max_splits;
    j.ticket = reinterpret_cast<uint32_t*>(ws + L.dec_work);
    return j;
}

}  // namespace
}  // namespace sa
