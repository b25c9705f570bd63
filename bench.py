#!/usr/bin/env python3
"""Benchmark: sparse decode queries/s and achieved HBM GB/s on one GB300 (or N replicas).

One step = one pass of the hot path over one batch of decode queries:
select (score every block from its metadata + top-k + window) and decode (exact
softmax attention over the selected blocks), plus the diff/LRU step for the
multi-step workload.  Inputs are resident in HBM when the timed region starts.

Headline (stateless workloads): the K steps run back to back between one pair of
CUDA events on the launching stream, alternating between two independent instances
of the workload (another seed, separate buffers).  Each step touches several times
the L2's capacity and the step before it touched only the other instance, so no step
finds its inputs in the L2.  Beside it, each step is also timed between its own
events with the L2 flushed before it (a buffer of twice the L2 size written and then
read back, so the L2 holds only clean lines of unrelated data); that time carries
the event pair's own cost (~2 us on a GB300) and gives the per-step distribution and
the per-kernel breakdown.  The slot-cache workload carries state from step to step
and is timed per step, flushed, only.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on the host cores

Prints one JSON line (rank 0).  Under torchrun (N > 1) every rank runs an
independent replica of the workload on its own GPU (the path has no exchange
step); `value` is the sum over ranks of the queries processed divided by the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import dataclasses
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse decode queries/s and achieved HBM GB/s (% of peak) at 128K ctx, 1 GB300"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
DEFAULT_WORKLOAD = "gqa_128k"


# --------------------------------------------------------------- helpers --

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate_max(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over the process group (identity without one)."""
    if world <= 1 or not torch.distributed.is_initialized():
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1 and torch.distributed.is_initialized():
        torch.distributed.barrier()


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_digest(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


_CSRC = "query_guided_block_gb300/csrc/"
KERNEL_SOURCES = {
    "select": [_CSRC + f for f in ("sa_select.cu", "sa_select_body.cuh", "sa_common.cuh")],
    "decode": [_CSRC + f for f in ("sa_decode.cu", "sa_decode_body.cuh", "sa_common.cuh")],
    "step": [_CSRC + f for f in ("sa_step.cu", "sa_step_kernel.cuh", "sa_select_body.cuh", "sa_decode_body.cuh",
                                 "sa_common.cuh")],
    "decode_mq": [_CSRC + f for f in ("sa_decode_mq.cu", "sa_tcgen05.cuh", "sa_common.cuh")],
}


def recorded_traffic(kernel: str, workload: str, sources: str = ""):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel source (else None).  `sources` names the kernel's source files when
    they differ from `kernel`'s (the multi-query decode)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)\s+source_sha:\s*([0-9a-f]+)", text)
    if not m:
        return None
    if m.group(2) != source_digest(KERNEL_SOURCES[sources or kernel]):
        return None
    return float(m.group(1))


class ClockSampler:
    """nvidia-smi samples taken while the timed region runs."""

    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 50):
        self.rows = []
        self.proc = None
        self.err = None
        self.thread = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception as e:  # no nvidia-smi
            self.err = str(e)

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        if self.err or not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": self.err or "no samples"}
        inside = [r for t, r in self.rows if t0 <= t <= t1]
        note = "samples inside the timed region"
        if not inside:
            # region shorter than the sampling interval: nearest samples around it
            near = sorted(self.rows, key=lambda tr: min(abs(tr[0] - t0), abs(tr[0] - t1)))[:3]
            inside = [r for _, r in near]
            note = "timed region shorter than the sampling interval; nearest samples"
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in inside if num(r[0]) is not None]
        mx = [num(r[1]) for r in inside if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4)
                          if len(r) > 4 + i and r[4 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "note": note,
                "power_w_max": max((num(r[2]) or 0.0) for r in inside)}


# ------------------------------------------------------ algorithmic bytes --

def algorithmic_bytes(w, sel_count: torch.Tensor, sel_ids: torch.Tensor):
    """Bytes the method must move per launch (see the design notes):
    select: q + candidate metadata (min/max at the KV width; fp32 means) + ids out;
    decode: q + K/V of the selected tokens + their page-table entries + ids + out."""
    import numpy as np
    esz = 2 if w.kv_dtype == torch.bfloat16 else 4
    qsz = 2 if w.q_dtype == torch.bfloat16 else 4
    B, Hq, Hkv, D, bs, N = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, w.n_tokens
    nb = w.num_blocks
    units = B * Hkv
    Qn = max(1, w.num_queries)
    q_bytes = B * Qn * Hq * D * qsz
    win_first = (max(0, N - w.window_tokens) // bs) if w.window_tokens > 0 else nb
    cnt = sel_count.detach().cpu().numpy().reshape(-1).astype(np.int64)
    ids_bytes = int(cnt.sum()) * 4 + units * 4
    if w.two_level:
        n_coarse = -(-N // w.coarse_block)
        per = w.coarse_block // bs
        meta = units * n_coarse * D * 4 + units * min(w.topk_coarse * per, win_first) * 2 * D * esz
    elif w.score == "mean":
        meta = units * win_first * D * 4
    else:
        meta = units * win_first * 2 * D * esz
    select_bytes = q_bytes + meta + ids_bytes
    # selected tokens (the last block may be partial)
    tokens = int(cnt.sum()) * bs
    tail = N - (nb - 1) * bs if nb else bs
    if tail != bs:
        ids = sel_ids.detach().cpu().numpy().reshape(units, -1)
        holds_last = sum(int((ids[u, : cnt[u]] == nb - 1).any()) for u in range(units))
        tokens -= holds_last * (bs - tail)
    decode_bytes = q_bytes + tokens * 2 * D * esz + int(cnt.sum()) * 4 * 2 + units * 4 + B * Qn * Hq * D * 4
    # tensor work of the decode: S = q K^T and O = P V over the selected tokens
    decode_flops = 4.0 * tokens * Qn * (Hq // Hkv) * D   # each unit's tokens meet Q x G query rows
    return {"select": select_bytes, "decode": decode_bytes, "decode_flops": decode_flops}


# ------------------------------------------------------------- GPU arm --

def select_launches(w):
    """Kernel launches of one sparse_attn_select call: one, except a two-level selection
    with more than 256 level-1 survivors, which runs one launch per level."""
    return 2 if (w.two_level and w.topk_coarse > 256) else 1


def run_gpu_arm(args):
    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    from query_guided_block_gb300 import binding as Bn
    from query_guided_block_gb300.build import build
    from query_guided_block_gb300.decoder import SlotCache, SlotPool, SparseDecoder
    from query_guided_block_gb300.workloads import WORKLOADS, make_inputs

    if rank == 0 or world == 1:
        build()
    barrier(world)
    build()
    Bn.lib()

    w = WORKLOADS[args.workload]
    if args.batch:
        w = dataclasses.replace(w, batch=args.batch)
    inp = make_inputs(w, dev)
    p = Bn.params_for(w)
    dec = SparseDecoder(p, dev)
    multi_q = inp.get("queries_per_seq", 1) > 1    # q is [B, Q, Hq, D]: one step's queries
    q_all = inp["q"] if (inp["q"].dim() == 4 and not multi_q) else inp["q"].unsqueeze(0)
    q_static = q_all[0].clone()
    kp, vp, bt = inp["k_pages"], inp["v_pages"], inp["block_table"]
    cache = SlotCache(dec, w.cache_slots) if w.cache_slots else None
    stream = torch.cuda.current_stream()
    # --io: K/V come from a pinned host store through the slot pool (misses loaded each step)
    io = bool(args.io and cache)
    if args.io and not cache:
        raise SystemExit("--io needs a workload with an LRU slot cache (lru_64k)")
    pool = SlotPool(cache) if io else None
    host_k = kp.cpu().pin_memory() if io else None
    host_v = vp.cpu().pin_memory() if io else None
    miss_total = torch.zeros((), dtype=torch.int64, device=dev) if io else None

    # metadata (prefill-time), timed on its own
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dec.build_meta(kp, bt)
    torch.cuda.synchronize()
    e0.record()
    dec.build_meta(kp, bt)
    e1.record()
    torch.cuda.synchronize()
    meta_ms = e0.elapsed_time(e1)
    esz = 2 if w.kv_dtype == torch.bfloat16 else 4
    meta_bytes = kp.numel() * esz + dec.metadata_bytes() + bt.numel() * 4

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    flush_sum = torch.empty((), dtype=torch.int64, device=dev)

    class _Flush:   # write a 2x-L2 buffer, then read it back: the L2 ends clean
        def zero_(self):
            flush_buf.zero_()
            torch.sum(flush_buf.view(torch.int64), dim=0, out=flush_sum)

        def numel(self):
            return flush_buf.numel()
    flush = _Flush()

    # one appended token per sequence (a decode step's metadata upkeep), L2 flushed before each
    app_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(10)]
    for a_, b_ in app_ev:
        flush.zero_()
        a_.record(stream)
        dec.append_meta(w.n_tokens - 1, kp, bt)
        b_.record(stream)
    torch.cuda.synchronize()
    append_ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in app_ev[3:])
    # rows holding the new token are rebuilt with the other rows of their build run
    run_blocks = (w.coarse_block // w.block_size if w.two_level else 1) if dec.kmean is not None else 1
    nb_all = -(-w.n_tokens // w.block_size)
    run_start = ((w.n_tokens - 1) // w.block_size) // run_blocks * run_blocks
    reread = w.batch * w.num_kv_heads * (min(nb_all, run_start + run_blocks) - run_start)
    append_bytes = reread * w.block_size * w.head_dim * esz * (1 + 2 / w.block_size)
    step_counter = [0]

    reserve = inp.get("reserve_ids")   # random reserve set, drawn with the inputs
    # The step as a user calls it: sparse_attn_step (one cooperative launch, or select
    # followed by a decode that waits per unit) where it covers the problem, else the
    # select and decode calls.
    step_launches = -1 if (io or args.two_launch) else Bn.sparse_attn_step_launches(p)
    use_step = step_launches > 0
    serial_io = bool(io and args.io_serial)
    launches_per_step = ((step_launches if use_step else 1 + select_launches(w)) + (1 if cache else 0)
                         + (2 if serial_io else 0))

    def io_phase():   # diff, misses in from the host store, slot map (or: diff writing the slot map)
        if serial_io:
            cache.diff(step_counter[0])
            pool.load_misses(host_k, host_v, bt)
            pool.slot_map()
        else:
            cache.diff(step_counter[0], sel_slot=pool.sel_slot)

    def io_decode(q):   # attention through the slot pool; the misses read in the same pass
        if serial_io:
            pool.decode(q)
        else:
            pool.decode_io(q, host_k, host_v, bt)

    def one_step(q):
        if use_step:
            dec.step_fused(q, kp, vp, bt, reserve)
            if cache:
                cache.diff(step_counter[0])
        else:
            dec.select(q, reserve)
            if io:
                io_phase()
                io_decode(q)
            else:
                dec.decode(q, kp, vp, bt)
                if cache:
                    cache.diff(step_counter[0])
        if cache:
            cache.advance()
            step_counter[0] += 1

    for i in range(args.warmup):
        q = q_all[i % q_all.shape[0]] if cache else q_static
        one_step(q)
    torch.cuda.synchronize()
    if dec.device_error() != 0:
        raise RuntimeError("device error during warm-up")

    K = args.steps
    # Headline timing (stateless workloads): the K steps back to back between one pair of
    # events, alternating between two independent instances of the workload (another
    # seed, separate buffers).  A step touches several times the L2's capacity and the
    # step before it touched only the other instance, so no step finds its inputs in
    # the L2, and no flush or event runs between the steps.  The slot-cache workloads
    # carry state from step to step and are timed per step with the L2 flushed instead.
    block = not cache
    inst = []
    if block:
        inp2 = make_inputs(dataclasses.replace(w, seed=w.seed + 1), dev)
        dec2 = SparseDecoder(p, dev)
        dec2.build_meta(inp2["k_pages"], inp2["block_table"])
        q2_all = inp2["q"] if (inp2["q"].dim() == 4 and not multi_q) else inp2["q"].unsqueeze(0)
        inst = [(dec, q_static, kp, vp, bt, reserve),
                (dec2, q2_all[0].clone(), inp2["k_pages"], inp2["v_pages"], inp2["block_table"],
                 inp2.get("reserve_ids"))]
        del inp2, q2_all

    def inst_step(j):
        d, q_, k_, v_, b_, r_ = inst[j]
        if use_step:
            d.step_fused(q_, k_, v_, b_, r_)
        else:
            d.select(q_, r_)
            d.decode(q_, k_, v_, b_)

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    sampler = ClockSampler(dev.index) if (rank == 0 or world == 1) else None
    time.sleep(0.2 if sampler else 0)
    block_ms_local = None
    if block:
        for i in range(max(args.warmup, 4)):
            inst_step(i & 1)
        torch.cuda.synchronize()
        if dec.device_error() != 0 or inst[1][0].device_error() != 0:
            raise RuntimeError("device error during the second instance's warm-up")
        blk0, blk1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        t_start = time.time()
        blk0.record(stream)
        for i in range(K):
            inst_step(i & 1)
        blk1.record(stream)
        torch.cuda.synchronize()
        block_ms_local = blk0.elapsed_time(blk1)
    # per-step timing: each step between its own events, the L2 flushed before it
    # (the headline for the slot-cache workloads; the per-step distribution otherwise)
    barrier(world)
    torch.cuda.synchronize()
    if not block:
        t_start = time.time()
    for i in range(K):
        flush.zero_()
        q = q_all[(args.warmup + i) % q_all.shape[0]] if cache else q_static
        a, b, c, d = ev[i]
        a.record(stream)
        if use_step:                 # a step b [diff d]: no event between kernels that has no work to time
            dec.step_fused(q, kp, vp, bt, reserve)
            b.record(stream)
            if cache:
                cache.diff(step_counter[0])
                d.record(stream)
                cache.advance()
                step_counter[0] += 1
            continue
        dec.select(q, reserve)
        b.record(stream)
        if io:                       # a select b diff (+ misses) + map c decode (+ misses) d
            io_phase()
            c.record(stream)
            io_decode(q)
            d.record(stream)
            miss_total.add_(cache.counts[:, 1].sum())
        else:                        # a select b decode c diff d
            dec.decode(q, kp, vp, bt)
            c.record(stream)
            if cache:
                cache.diff(step_counter[0])
            d.record(stream)
        if cache:
            cache.advance()
            step_counter[0] += 1
    torch.cuda.synchronize()
    barrier(world)
    t_end = time.time()
    clocks = sampler.summary(t_start, t_end) if sampler else None
    if sampler:
        sampler.stop()
    flags = dec.device_error() | (inst[1][0].device_error() if block else 0)
    if flags:
        raise RuntimeError(f"device error flags 0x{flags:x}")

    step_ms = [e[0].elapsed_time(e[3] if (cache or not use_step) else e[1]) for e in ev]
    if use_step:
        fused_ms = [e[0].elapsed_time(e[1]) for e in ev]
        # breakdown: the select and decode calls timed on their own after the timed region
        bk = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
               torch.cuda.Event(enable_timing=True)) for _ in range(min(K, 100) + 3)]
        for a, b, c in bk:   # the first three calls are warm-up (a kernel's first launch loads it)
            flush.zero_()
            a.record(stream)
            dec.select(q_static if not cache else q_all[0], reserve)
            b.record(stream)
            dec.decode(q_static if not cache else q_all[0], kp, vp, bt)
            c.record(stream)
        torch.cuda.synchronize()
        sel_ms = [a.elapsed_time(b) for a, b, c in bk[3:]]
        dec_ms = [b.elapsed_time(c) for a, b, c in bk[3:]]
    else:
        sel_ms = [e[0].elapsed_time(e[1]) for e in ev]
        dec_ms = [e[2].elapsed_time(e[3]) if io else e[1].elapsed_time(e[2]) for e in ev]
    flushed_ms_per_step = aggregate_max(sum(step_ms), world, dev) / K
    total_ms_local = block_ms_local if block else sum(step_ms)
    total_ms = aggregate_max(total_ms_local, world, dev)
    queries = w.batch * w.num_q_heads * max(1, w.num_queries)
    value = world * queries * K / (total_ms / 1e3)
    ms_per_step = total_ms / K

    nbytes = algorithmic_bytes(w, dec.sel_count, dec.sel_ids)
    peak, peak_kind = hbm_peak()
    sel_avg, dec_avg = statistics.mean(sel_ms), statistics.mean(dec_ms)
    kern = {
        "select": {"ms": sel_avg, "bytes": nbytes["select"], "gbs": nbytes["select"] / sel_avg / 1e6,
                   "launches_per_step": select_launches(w)},
        "decode": {"ms": dec_avg, "bytes": nbytes["decode"], "gbs": nbytes["decode"] / dec_avg / 1e6,
                   "tflops": nbytes["decode_flops"] / dec_avg / 1e9, "launches_per_step": 1},
    }
    if io:
        io_ms = statistics.mean([e[1].elapsed_time(e[2]) for e in ev])
        io_bytes = float(miss_total.item()) * 2 * pool.tile_bytes() / K
        if serial_io:
            kern["diff_io"] = {"ms": io_ms, "misses_bytes": io_bytes, "host_read_gbs": io_bytes / io_ms / 1e6,
                               "launches_per_step": 3,
                               "note": "diff + miss tiles read from pinned host memory + slot map"}
        else:
            kern["diff_io"] = {"ms": io_ms, "misses_bytes": io_bytes, "launches_per_step": 1,
                               "note": "diff writing the slot map (sparse_attn_diff_slots); the miss tiles "
                                       "are read from pinned host memory inside the decode's launch "
                                       "(sparse_attn_decode_slots_io)"}
    elif cache:
        kern["diff"] = {"ms": statistics.mean([(e[1] if use_step else e[2]).elapsed_time(e[3]) for e in ev]),
                        "launches_per_step": 1}
    step_bytes = nbytes["select"] + nbytes["decode"]
    if use_step:
        st_flushed = statistics.mean(fused_ms)
        st_avg = ms_per_step if block else st_flushed
        kern["step"] = {"ms": st_avg, "ms_per_step_events_flushed": st_flushed,
                        "bytes": step_bytes, "gbs": step_bytes / st_avg / 1e6,
                        "launches_per_step": step_launches,
                        "note": "sparse_attn_step: " + ("one cooperative launch (select phase, then decode "
                                "phase waiting per unit)" if step_launches == 1 else
                                "select kernel, then decode as its dependent waiting per unit")}
        kern["select"]["note"] = kern["decode"]["note"] = "separate call, timed after the timed region"
    dominant = "step" if use_step else ("select" if sel_avg >= dec_avg else "decode")
    dk = kern[dominant]
    step_gbs = step_bytes / (ms_per_step / 1e3) / 1e9
    traffic = recorded_traffic(dominant, w.name, "decode_mq" if (multi_q and dominant == "decode") else "")
    roofline = {"bound": "hbm", "kernel": dominant, "achieved": dk["gbs"], "peak": peak,
                "unit": "GB/s", "frac": dk["gbs"] / peak, "traffic": traffic,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6.8 TB/s"}

    # end to end: pinned host q in, fp32 out back to pinned host, every step
    q_host = q_static.cpu().pin_memory()
    out_host = torch.empty(dec.out.shape, dtype=dec.out.dtype).pin_memory()
    q_dev = torch.empty_like(q_static)
    res_host = reserve.cpu().pin_memory() if reserve is not None else None
    res_dev = torch.empty_like(reserve) if reserve is not None else None
    if block:
        # the K steps back to back, alternating instances as in the headline; every step
        # uploads its instance's queries from pinned host memory and reads its output
        # back.  Uploads and downloads run on streams of their own, ordered by events:
        # step i waits for its upload and for the download of the step before it on the
        # same instance (which last wrote that output); the upload for step i waits for
        # that earlier step to finish reading the queries.  So step i's copies overlap
        # the neighbouring steps, and the region ends after the last download.
        hosts = [(q_host, q_dev, res_host, res_dev, out_host)]
        d1, q1, _, _, _, r1 = inst[1]
        hosts.append((q1.cpu().pin_memory(), torch.empty_like(q1),
                      r1.cpu().pin_memory() if r1 is not None else None,
                      torch.empty_like(r1) if r1 is not None else None,
                      torch.empty(d1.out.shape, dtype=d1.out.dtype).pin_memory()))
        up_s, down_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        uploaded = [torch.cuda.Event() for _ in range(2)]
        stepped = [torch.cuda.Event() for _ in range(2)]
        downloaded = [torch.cuda.Event() for _ in range(2)]
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        ea.record(stream)
        up_s.wait_event(ea)
        down_s.wait_event(ea)
        for i in range(K):
            j = i & 1
            qh, qd, rh, rd, oh = hosts[j]
            d_, _, k_, v_, b_, _ = inst[j]
            with torch.cuda.stream(up_s):
                if i >= 2:
                    up_s.wait_event(stepped[j])
                qd.copy_(qh, non_blocking=True)
                if rh is not None:
                    rd.copy_(rh, non_blocking=True)
                uploaded[j].record(up_s)
            stream.wait_event(uploaded[j])
            if i >= 2:
                stream.wait_event(downloaded[j])
            if use_step:
                d_.step_fused(qd, k_, v_, b_, rd)
            else:
                d_.select(qd, rd)
                d_.decode(qd, k_, v_, b_)
            stepped[j].record(stream)
            with torch.cuda.stream(down_s):
                down_s.wait_event(stepped[j])
                oh.copy_(d_.out, non_blocking=True)
                downloaded[j].record(down_s)
        stream.wait_event(downloaded[0])
        stream.wait_event(downloaded[1])
        eb.record(stream)
        torch.cuda.synchronize()
        e2e_ms = aggregate_max(ea.elapsed_time(eb), world, dev)
    else:
        e2e_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        torch.cuda.synchronize()
        for i in range(K):
            flush.zero_()
            a, b = e2e_ev[i]
            a.record(stream)
            q_dev.copy_(q_host, non_blocking=True)
            if reserve is not None:
                res_dev.copy_(res_host, non_blocking=True)
            if use_step:
                dec.step_fused(q_dev, kp, vp, bt, res_dev if reserve is not None else None)
                out_host.copy_(dec.out, non_blocking=True)
                b.record(stream)
                continue
            dec.select(q_dev, res_dev if reserve is not None else None)
            if io:
                io_phase()
                io_decode(q_dev)
                cache.advance()
                step_counter[0] += 1
            else:
                dec.decode(q_dev, kp, vp, bt)
            out_host.copy_(dec.out, non_blocking=True)
            b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = aggregate_max(sum(a.elapsed_time(b) for a, b in e2e_ev), world, dev)
    e2e = {"value": world * queries * K / (e2e_ms / 1e3), "unit": "queries/s",
           "h2d_bytes_per_step": q_host.numel() * q_host.element_size() +
                                 (res_host.numel() * 4 if res_host is not None else 0),
           "d2h_bytes_per_step": out_host.numel() * out_host.element_size(),
           "ms_per_step": e2e_ms / K}

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, inp, dev, args.cpu_seconds)

    # the other single-GPU workloads, measured in this process after the headline
    other = None
    if args.other_workloads and args.workload == DEFAULT_WORKLOAD and not args.batch and not io:
        del inp, dec, cache
        kp = vp = bt = q_all = q_static = None
        inst = hosts = None
        torch.cuda.empty_cache()
        other = {}
        for name in OTHER_WORKLOADS:
            other[name] = measure_other_workload(name, dev, args.other_steps, max(3, min(args.warmup, 10)),
                                                 flush, peak)

    result = {
        "metric": METRIC,
        "value": value,
        "unit": "queries/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        # each step between its own events with the L2 flushed before it (mean max over
        # ranks; median and 90th percentile of this rank): each such step also carries
        # the event pair's own ~2 us
        "ms_per_step_events_flushed": flushed_ms_per_step,
        "ms_per_step_events_flushed_p50": statistics.median(step_ms),
        "ms_per_step_events_flushed_p90": sorted(step_ms)[int(0.9 * (len(step_ms) - 1))],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.kv_dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded; planted relevant blocks)",
        "config": {"workload": w.name + ("+io" if io else ""), "batch": w.batch, "q_heads": w.num_q_heads,
                   "kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "context": w.n_tokens,
                   "block_size": w.block_size, "topk_blocks": w.topk,
                   "window_tokens": w.window_tokens, "two_level": w.two_level,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": ("inputs larger than L2: two independent instances of the workload alternate, "
                          f"each step touches {step_bytes / 2**20:.0f} MB against a {l2 >> 20} MB L2, and the step "
                          "before it touched only the other instance"
                          if block else
                          f"flushed before every step ({flush.numel() >> 20} MB written then read back, "
                          "outside the step events)"),
                   "step": (f"sparse_attn_step ({step_launches} launch{'es' if step_launches > 1 else ''})"
                            if use_step else
                            ("sparse_attn_select + diff + load_misses + slot_map + decode_slots" if serial_io else
                             "sparse_attn_select + diff_slots + decode_slots_io (misses loaded in the decode's "
                             "launch)")
                            if io else "sparse_attn_select + sparse_attn_decode"),
                   "timing": ("CUDA events on the launching stream around the K steps back to back (value, "
                              "ms_per_step, e2e); per call around each step with the L2 flushed before it "
                              "(ms_per_step_events_flushed*, kernels)"
                              if block else "CUDA events per call on the launching stream")},
        "hbm_gbs": step_gbs,
        "hbm_frac_of_measured": step_gbs / peak,
        "hbm_frac_of_nominal_8tbs": step_gbs / NOMINAL_HBM_GBS,
        "step_bytes": step_bytes,
        "roofline": roofline,
        "kernels": kern,
        "build_meta": {"ms": meta_ms, "gbs": meta_bytes / meta_ms / 1e6, "bytes": meta_bytes},
        "append_meta": {"ms": append_ms, "tokens_appended_per_sequence": 1, "blocks_rebuilt": reread,
                        "bytes": append_bytes,
                        "note": "sparse_attn_append_meta(n-1 -> n); launch-latency bound"},
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "other_workloads": other,
    }
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ------------------------------------------------------- other workloads --

OTHER_WORKLOADS = ("mha_32k", "two_level_256k", "lru_64k")


def measure_other_workload(name, dev, steps, warmup, flush, peak):
    """One more workload timed the way the headline is: the step a user calls
    (sparse_attn_step where it covers the problem, else select + decode), plus the
    diff against the LRU slot cache for the multi-step workload.  Stateless workloads:
    the steps back to back between one pair of events, alternating between two
    independent instances; the slot-cache workload: CUDA events around each step with
    the L2 flushed before it.  The per-step flushed time is reported for both."""
    from query_guided_block_gb300 import binding as Bn
    from query_guided_block_gb300.decoder import SlotCache, SparseDecoder
    from query_guided_block_gb300.workloads import WORKLOADS, make_inputs

    w = WORKLOADS[name]
    inp = make_inputs(w, dev)
    p = Bn.params_for(w)
    dec = SparseDecoder(p, dev)
    kp, vp, bt = inp["k_pages"], inp["v_pages"], inp["block_table"]
    dec.build_meta(kp, bt)
    cache = SlotCache(dec, w.cache_slots) if w.cache_slots else None
    q_all = inp["q"] if inp["q"].dim() == 4 else inp["q"].unsqueeze(0)
    launches = Bn.sparse_attn_step_launches(p)
    use_step = launches > 0
    stream = torch.cuda.current_stream()
    counter = [0]
    block = not cache
    insts = [(dec, q_all, kp, vp, bt)]
    if block:
        inp2 = make_inputs(dataclasses.replace(w, seed=w.seed + 1), dev)
        dec2 = SparseDecoder(p, dev)
        dec2.build_meta(inp2["k_pages"], inp2["block_table"])
        q2 = inp2["q"] if inp2["q"].dim() == 4 else inp2["q"].unsqueeze(0)
        insts.append((dec2, q2, inp2["k_pages"], inp2["v_pages"], inp2["block_table"]))
        del inp2, q2

    def one_step(i, j=0):
        d, qa, k_, v_, b_ = insts[j]
        q = qa[i % qa.shape[0]]
        if use_step:
            d.step_fused(q, k_, v_, b_)
        else:
            d.select(q)
            d.decode(q, k_, v_, b_)
        if cache:
            cache.diff(counter[0])
            cache.advance()
        counter[0] += 1

    for i in range(warmup):
        one_step(i, i % len(insts))
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i, (a, b) in enumerate(ev):
        flush.zero_()
        a.record(stream)
        one_step(warmup + i)
        b.record(stream)
    torch.cuda.synchronize()
    ms_flushed = statistics.mean(a.elapsed_time(b) for a, b in ev)
    ms = ms_flushed
    if block:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(steps):
            one_step(warmup + i, i & 1)
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / steps
    flags = 0
    for d_, *_ in insts:
        flags |= d_.device_error()
    if flags:
        raise RuntimeError(f"{name}: device error flags 0x{flags:x}")
    nbytes = algorithmic_bytes(w, dec.sel_count, dec.sel_ids)
    step_bytes = nbytes["select"] + nbytes["decode"]
    gbs = step_bytes / ms / 1e6
    per_step = (f"sparse_attn_step ({launches} launch{'es' if launches > 1 else ''})" if use_step
                else "sparse_attn_select + sparse_attn_decode") + (" + sparse_attn_diff" if cache else "")
    out = {"ms_per_step": ms, "ms_per_step_events_flushed": ms_flushed,
           "value": w.batch * w.num_q_heads / (ms / 1e3), "unit": "queries/s",
           "steps": steps, "warmup": warmup, "step": per_step, "step_bytes": step_bytes,
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak},
           "config": {"batch": w.batch, "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads,
                      "head_dim": w.head_dim, "context": w.n_tokens, "block_size": w.block_size,
                      "topk_blocks": w.topk, "window_tokens": w.window_tokens, "two_level": w.two_level,
                      "cache_slots": w.cache_slots,
                      "timing": ("steps back to back, two instances alternating (inputs larger than L2)" if block
                                 else "per step, L2 flushed before each")},
           "gpu_launches": (launches if use_step else 1 + select_launches(w)) * steps +
                           (steps if cache else 0)}
    del inp, dec, cache, insts
    torch.cuda.empty_cache()
    return out


# -------------------------------------------------------------- CPU arms --

def oracle_sample(w, inp, seqs):
    """Host copies of the sequences `seqs` with their metadata built by the oracle
    (not timed)."""
    import dataclasses
    import oracle
    from query_guided_block_gb300.workloads import gather_sequences
    host = gather_sequences(inp, seqs, "cpu")
    ws = dataclasses.replace(w, batch=len(seqs))
    p = oracle.problem(batch=ws.batch, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                       head_dim=w.head_dim, n_tokens=w.n_tokens, block_size=w.block_size,
                       num_pages=host["k_pages"].shape[0], window_tokens=w.window_tokens,
                       topk=w.topk, two_level=w.two_level, coarse_block=w.coarse_block,
                       topk_coarse=w.topk_coarse, score_kind=w.score,
                       kv_bf16=w.kv_dtype == torch.bfloat16, q_bf16=w.q_dtype == torch.bfloat16)
    need_mean = w.two_level or w.score == "mean"
    kmin, kmax, kmean = oracle.build_meta(p, host["k_pages"], host["block_table"], with_mean=need_mean)
    q = host["q"] if host["q"].dim() == 3 else host["q"][0]
    arrays = {k: oracle.host_array(v) for k, v in host.items()}
    arrays["q"] = oracle.host_array(q)
    return p, arrays, kmin, kmax, kmean


def oracle_unit_step(p, a, kmin, kmax, kmean, u):
    """The oracle's select + decode for one unit."""
    import oracle
    rng = (u, u + 1)
    if p.two_level:
        r = oracle.select_two_level(p, a["q"], kmin, kmax, kmean, units=rng)
        ids, cnt = r["sel_ids"], r["sel_count"]
    else:
        if p.score_kind == 1:
            sc = oracle.mean_scores(p, a["q"], kmean, units=rng)
        else:
            sc = oracle.quest_scores(p, a["q"], kmin, kmax, units=rng)
        ids, cnt = oracle.select(p, sc, units=rng)
    if "reserve_ids" in a:   # the reserve set joins the selection
        ids, cnt = oracle.union_reserve(p, ids, cnt, a["reserve_ids"].reshape(p.units, -1), units=rng)
    oracle.decode(p, a["q"], a["k_pages"], a["v_pages"], a["block_table"], ids, cnt, units=rng)


def cpu_baseline(w, inp, dev, seconds):
    seqs = sorted({0, w.batch - 1})
    p, a, kmin, kmax, kmean = oracle_sample(w, inp, seqs)
    units = list(range(p.units))
    threads = min(len(units), os.cpu_count() or 1)
    done, t0 = 0, time.time()
    with cf.ThreadPoolExecutor(threads) as ex:
        while True:
            list(ex.map(lambda u: oracle_unit_step(p, a, kmin, kmax, kmean, u), units))
            done += len(units)
            if time.time() - t0 >= seconds:
                break
    dt = time.time() - t0
    return {"value": done * w.group / dt, "unit": "queries/s", "cores": threads, "kind": "oracle",
            "sample": f"select+decode of {len(units)} units (sequences {seqs} of {w.batch}, all KV "
                      f"heads) repeated {done // len(units)}x over {dt:.1f} s; fp64 C oracle, "
                      f"one unit per thread"}


def run_reference_arm(args):
    """The fp64 oracle timed on the host cores, same workload / metric / unit."""
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return
    import oracle
    from query_guided_block_gb300.workloads import WORKLOADS, make_inputs
    oracle.build()
    from query_guided_block_gb300.workloads import scaled
    w = WORKLOADS[args.workload]
    # the same workload drawn on the host for two sequences (the oracle never needs more)
    ws = scaled(w, name=w.name, batch=min(2, w.batch))
    inp = make_inputs(ws, "cpu")
    seqs = list(range(ws.batch))
    p, a, kmin, kmax, kmean = oracle_sample(ws, inp, seqs)
    del inp
    threads = min(p.units, os.cpu_count() or 1)
    per_step_units = list(range(threads))           # one unit per thread per step

    def step():
        with cf.ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda u: oracle_unit_step(p, a, kmin, kmax, kmean, u), per_step_units))

    for _ in range(args.warmup):
        step()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = len(per_step_units) * w.group * args.steps / total
    sample = (f"each step: oracle select+decode of {len(per_step_units)} units (one per thread) "
              f"of sequences {seqs}")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "queries/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; planted relevant blocks)",
        "config": {"workload": w.name, "batch": w.batch, "q_heads": w.num_q_heads,
                   "kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "context": w.n_tokens},
        "cpu_baseline": {"value": value, "unit": "queries/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch (smaller profiling cases)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--two-launch", action="store_true",
                    help="time the separate select and decode calls instead of sparse_attn_step")
    ap.add_argument("--io", action="store_true",
                    help="LRU workloads: K/V read through the slot pool, misses loaded each step "
                         "from a pinned host store")
    ap.add_argument("--io-serial", action="store_true",
                    help="with --io: load the misses in their own launch before the decode")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-other-workloads", dest="other_workloads", action="store_false",
                    help="skip timing mha_32k, two_level_256k and lru_64k after the headline")
    ap.add_argument("--other-steps", type=int, default=200)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    if args.impl == "reference":
        run_reference_arm(args)
    else:
        run_gpu_arm(args)


if __name__ == "__main__":
    main()
