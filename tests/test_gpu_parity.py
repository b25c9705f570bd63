"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Tolerances (from the problem statement): selected ids, diff / LRU outputs and the
min/max bounding box are bit-exact (selection up to swaps among candidates whose
oracle scores lie within 1e-5 relative of the k-th score); attention output within
2e-3 max-abs for bf16 KV and 1e-5 for fp32 KV; block means (fp32 accumulation vs fp64)
within the error bound of fp32 summation over the row's tokens (tests.parity.check_means),
and exact on keys whose fp32 sums are exact.
"""
import concurrent.futures as cf
import dataclasses
import os

import numpy as np
import pytest
import torch

import oracle
from query_guided_block_gb300 import binding as B
from query_guided_block_gb300.build import build
from query_guided_block_gb300.decoder import SparseDecoder
from query_guided_block_gb300.workloads import WORKLOADS, Workload, make_inputs
from tests.parity import (ATOL, as_np, bf16_bits_to_f64, check_means, check_selection, check_two_level,
                          oracle_meta, sub_problem, sub_workload)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build()
    B.lib()


def run_gpu(w, inp, params=None):
    p = params or B.params_for(w)
    dec = SparseDecoder(p)
    dec.build_meta(inp["k_pages"], inp["block_table"])
    q = inp["q"] if inp["q"].dim() == 3 else inp["q"][0]
    dec.select(q, inp.get("reserve_ids"))
    dec.decode(q, inp["k_pages"], inp["v_pages"], inp["block_table"])
    flags = dec.device_error()
    assert flags == 0, f"device error flags 0x{flags:x}"
    return dec


def compare_all(w, inp, dec, seqs=None):
    """Full comparison of metadata, selection and output on sequences `seqs`."""
    seqs = list(range(w.batch)) if seqs is None else list(seqs)
    host = sub_problem(w, inp, seqs)
    ws = sub_workload(w, len(seqs))
    p, (kmin, kmax, kmean) = oracle_meta(ws, host)
    Hkv = w.num_kv_heads
    rows = [s * Hkv + h for s in seqs for h in range(Hkv)]
    # metadata: exact box, close means
    gmin = bf16_bits_to_f64(dec.kmin[seqs])
    gmax = bf16_bits_to_f64(dec.kmax[seqs])
    assert np.array_equal(gmin, kmin) and np.array_equal(gmax, kmax)
    if kmean is not None:
        check_means(as_np(dec.kmean[seqs]), kmean, host, ws,
                    w.coarse_block if w.two_level else w.block_size)
    gids = as_np(dec.sel_ids).reshape(w.units, -1)[rows]
    gcnt = as_np(dec.sel_count).reshape(-1)[rows]
    hq = host["q"] if host["q"].dim() == 3 else host["q"][0]
    reserve = as_np(host["reserve_ids"]).reshape(ws.units, -1) if w.num_reserve else None
    if w.two_level:
        check_two_level(ws, p, hq, kmin, kmax, kmean, gids, gcnt, units=range(ws.units),
                        reserve=reserve)
    else:
        if w.score == "mean":
            scores = oracle.mean_scores(p, hq, kmean)
        else:
            scores = oracle.quest_scores(p, hq, kmin, kmax)
        oid, ocnt = oracle.select(p, scores)
        if reserve is not None:   # SparDA page §3.4: the reserve set joins the selection
            oid, ocnt = oracle.union_reserve(p, oid, ocnt, reserve)
        check_selection(gids, gcnt, oid, ocnt, scores, w.topk, p.first_window_block())
    # attention on the GPU's own selection
    out = oracle.decode(p, hq, host["k_pages"], host["v_pages"], host["block_table"], gids, gcnt)
    got = as_np(dec.out[seqs]).astype(np.float64)
    err = np.abs(got - out).max() if out.size else 0.0
    assert err <= ATOL[w.kv_dtype], f"max abs error {err}"
    return err


def seq_chunks(batch, threads=None):
    """Sequences cut into about four chunks per host thread (at least one sequence each)."""
    threads = threads or max(1, min(8, (os.cpu_count() or 2) // 2))
    per = max(1, -(-batch // (4 * threads)))
    return [list(range(s, min(batch, s + per))) for s in range(0, batch, per)], threads


def compare_every_unit(w, inp, dec, threads=None, check=None):
    """compare_all (or `check`) over every sequence of the instance, a chunk of
    sequences at a time, the chunks spread over host threads (the oracle's ctypes calls
    release the interpreter lock).  Returns the worst attention error."""
    check = check or compare_all
    chunks, threads = seq_chunks(w.batch, threads)
    with cf.ThreadPoolExecutor(min(threads, len(chunks))) as ex:
        errs = list(ex.map(lambda c: check(w, inp, dec, seqs=c), chunks))
    return max(errs) if errs else 0.0


def _w(**kw):
    base = dict(name="gpu_small", batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128,
                n_tokens=5000, block_size=64, window_tokens=300, topk=9)
    base.update(kw)
    return Workload(**base)


# ------------------------------------------------------------- small cases --

def test_tiny_config_exact():
    w = WORKLOADS["tiny_fp32_4k"]
    inp = make_inputs(w, "cuda")
    dec = run_gpu(w, inp)
    compare_all(w, inp, dec)


SMALL = [
    dict(head_dim=128, num_q_heads=8, kv_dtype=torch.bfloat16, block_size=64),
    dict(head_dim=128, num_q_heads=8, kv_dtype=torch.bfloat16, block_size=32, planted_per_unit=5),
    dict(head_dim=64, num_q_heads=16, kv_dtype=torch.bfloat16, block_size=16),
    dict(head_dim=128, num_q_heads=2, kv_dtype=torch.float32, q_dtype=torch.float32, block_size=32),
    dict(head_dim=64, num_q_heads=4, kv_dtype=torch.float32, q_dtype=torch.bfloat16, block_size=8,
         n_tokens=3001),
    dict(head_dim=128, num_q_heads=2, kv_dtype=torch.bfloat16, block_size=128, n_tokens=9000,
         window_tokens=0),
    dict(head_dim=128, num_q_heads=8, kv_dtype=torch.bfloat16, score="mean", block_size=64),
    dict(head_dim=64, num_q_heads=8, kv_dtype=torch.float32, q_dtype=torch.float32, score="mean",
         block_size=32, n_tokens=4097),
    dict(head_dim=128, num_q_heads=8, kv_dtype=torch.bfloat16, q_dtype=torch.float32, block_size=64,
         n_tokens=5001),
    dict(head_dim=64, num_q_heads=16, kv_dtype=torch.bfloat16, q_dtype=torch.float32, block_size=128,
         n_tokens=3333, window_tokens=200),
]


@pytest.mark.parametrize("cfg", SMALL, ids=[str(i) for i in range(len(SMALL))])
def test_small_matrix(cfg):
    w = _w(**cfg)
    inp = make_inputs(w, "cuda")
    dec = run_gpu(w, inp)
    compare_all(w, inp, dec)


@pytest.mark.parametrize("cfg", [
    dict(score="mean", block_size=64, n_tokens=5000),
    dict(score="mean", block_size=32, n_tokens=4097, kv_dtype=torch.float32, q_dtype=torch.float32,
         head_dim=64, num_q_heads=8),
    dict(two_level=True, block_size=64, n_tokens=40000, coarse_block=1024, topk_coarse=6, topk=12,
         window_tokens=512, planted_per_unit=0),
], ids=["block_means", "fp32_ragged", "coarse_means"])
def test_block_means_exact_on_quantised_keys(cfg):
    """Keys on the grid m / 64, |m| <= 128 (exact in bf16): every fp32 partial sum of up
    to 1024 of them is a multiple of 2^-6 below 2^11 in magnitude (17 significant bits),
    so the kernel's fp32 sum is exact whatever its order.  A row's mean is then
    fl(S * fl(1/n)): exact when n is a power of two, within two roundings (2u relative)
    otherwise.  A wrong divisor (n + 1 for n) is off by about 1/n relative and fails."""
    w = _w(**cfg)
    inp = make_inputs(w, "cuda")
    k = inp["k_pages"].float()
    inp["k_pages"] = (torch.clamp(torch.round(k * 64), -128, 128) / 64).to(inp["k_pages"].dtype)
    dec = run_gpu(w, inp)
    host = sub_problem(w, inp, range(w.batch))
    _, (_, _, kmean) = oracle_meta(w, host)
    mb = w.coarse_block if w.two_level else w.block_size
    n = np.minimum(mb, w.n_tokens - np.arange(kmean.shape[2]) * mb)
    gm = as_np(dec.kmean).astype(np.float64)[:, :, : kmean.shape[2]]
    pow2 = (n & (n - 1)) == 0
    assert pow2.any()
    assert np.array_equal(gm[:, :, pow2], kmean[:, :, pow2]), "power-of-two rows must be exact"
    err = np.abs(gm[:, :, ~pow2] - kmean[:, :, ~pow2])
    assert (err <= 2.0 ** -23 * np.abs(kmean[:, :, ~pow2]) * (1 + 1e-9)).all(), "ragged rows beyond 2u"
    compare_all(w, inp, dec)


@pytest.mark.parametrize("n_tokens,topk,window", [(40000, 12, 512), (33000, 5, 1000), (70001, 20, 0)])
def test_two_level_small(n_tokens, topk, window):
    w = _w(n_tokens=n_tokens, block_size=64, window_tokens=window, topk=topk, two_level=True,
           coarse_block=1024, topk_coarse=6, planted_per_unit=10)
    inp = make_inputs(w, "cuda")
    dec = run_gpu(w, inp)
    compare_all(w, inp, dec)


def test_two_level_many_survivors():
    """More level-1 survivors than one CTA keeps (300 > 256 coarse blocks): the two levels
    run as two launches of the streaming select kernel."""
    w = _w(n_tokens=40000, block_size=32, window_tokens=300, topk=20, two_level=True,
           coarse_block=64, topk_coarse=300, planted_per_unit=6)
    inp = make_inputs(w, "cuda")
    dec = run_gpu(w, inp)
    compare_all(w, inp, dec)


@pytest.mark.parametrize("cfg", [
    dict(n_tokens=20000, block_size=32, topk=10, num_reserve=7, planted_per_unit=4),
    dict(n_tokens=9001, block_size=64, topk=3, num_reserve=40, window_tokens=700),
    dict(n_tokens=7000, block_size=16, topk=0, num_reserve=5, head_dim=64, num_q_heads=16),
    dict(n_tokens=60000, block_size=64, topk=9, num_reserve=6, two_level=True, coarse_block=1024,
         topk_coarse=5, planted_per_unit=8),
], ids=["single", "many", "k0", "two_level"])
def test_reserve_set(cfg):
    """Selection united with a caller-drawn reserve set (SparDA page §3.4); the drawn
    ids are overwritten so that repeats, window blocks and top-k blocks all occur."""
    w = _w(**cfg)
    inp = make_inputs(w, "cuda")
    r = inp["reserve_ids"]
    nb, wf = w.num_blocks, (max(0, w.n_tokens - w.window_tokens) // w.block_size
                            if w.window_tokens else w.num_blocks)
    r[..., 0] = r[..., 1]                        # a repeat
    r[..., 2] = nb - 1                           # a window block (or the last block)
    if w.planted_per_unit:
        r[..., 3] = inp["planted"][..., 0].to(torch.int32)   # very likely a top-k block
    dec = run_gpu(w, inp)
    compare_all(w, inp, dec)
    cnt = as_np(dec.sel_count).reshape(-1)
    assert cnt.max() <= dec.sel_stride


def test_reserve_id_out_of_range_sets_the_error_bit():
    w = _w(n_tokens=8192, block_size=64, topk=4, num_reserve=3)
    inp = make_inputs(w, "cuda")
    inp["reserve_ids"][0, 0, 1] = w.num_blocks      # outside [0, nb): reported and skipped
    dec = SparseDecoder(B.params_for(w))
    dec.build_meta(inp["k_pages"], inp["block_table"])
    dec.select(inp["q"], inp["reserve_ids"])
    assert dec.device_error() & B.ERR_SEL_ID
    ids = as_np(dec.sel_ids)[0, 0, : as_np(dec.sel_count)[0, 0]]
    assert w.num_blocks not in ids.tolist() and (np.diff(ids) > 0).all()


def test_ties_go_to_the_lower_block_id():
    """Logical blocks that share one physical page have identical scores."""
    w = _w(n_tokens=64 * 64, block_size=64, window_tokens=128, topk=7, num_q_heads=4,
           num_kv_heads=2)
    inp = make_inputs(w, "cuda")
    bt = inp["block_table"]
    # blocks 3, 10, 17, ... all point at one page; 5 more at another
    bt[:, 3::7] = bt[:, 3:4]
    bt[:, 5:40:9] = bt[:, 5:6]
    dec = run_gpu(w, inp)
    compare_all(w, inp, dec)
    # and the exact-tie members picked are the lowest ids of their tie group
    host = sub_problem(w, inp, range(w.batch))
    p, (kmin, kmax, _) = oracle_meta(w, host)
    sc = oracle.quest_scores(p, host["q"], kmin, kmax)
    ids = as_np(dec.sel_ids).reshape(w.units, -1)
    cnt = as_np(dec.sel_count).reshape(-1)
    for u in range(w.units):
        sel = set(ids[u, : cnt[u]].tolist())
        for j in sel:
            if j >= p.first_window_block():
                continue
            for i in range(j):
                if sc[u, i] == sc[u, j]:
                    assert i in sel, f"unit {u}: tie {i} < {j} not taken first"


@pytest.mark.parametrize("case", ["dense", "k_zero", "window_only_all", "no_window", "short"])
def test_degenerate_selections(case):
    kw = {"dense": dict(topk=10 ** 6), "k_zero": dict(topk=0),
          "window_only_all": dict(window_tokens=10 ** 6, topk=3),
          "no_window": dict(window_tokens=0, topk=4),
          "short": dict(n_tokens=37, block_size=16, window_tokens=20, topk=1)}[case]
    w = _w(**kw)
    inp = make_inputs(w, "cuda")
    dec = run_gpu(w, inp)
    compare_all(w, inp, dec)
    if case in ("dense", "window_only_all"):
        assert np.all(as_np(dec.sel_count) == w.num_blocks)


def test_empty_inputs():
    # zero context: nothing to select, zero output
    w = _w(n_tokens=0)
    p = B.params_for(w)
    dec = SparseDecoder(p)
    q = torch.randn(w.batch, w.num_q_heads, w.head_dim, device="cuda").to(w.q_dtype)
    dec.out.fill_(7.0)
    dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(1, dtype=torch.int32, device="cuda")
    dec.select(q)
    dec.decode(q, dummy, dummy, bt)
    assert dec.device_error() == 0
    assert np.all(as_np(dec.sel_count) == 0)
    assert np.all(as_np(dec.out) == 0)
    # zero batch: every entry point is a no-op
    p0 = B.params_for(dataclasses.replace(w, batch=0, n_tokens=100))
    dec0 = SparseDecoder(p0)
    dec0.select(q)
    dec0.decode(q, dummy, dummy, bt)
    assert dec0.device_error() == 0


def test_largest_block_count():
    """16384 blocks per unit: the largest selection the top-k stage holds on chip."""
    w = _w(batch=1, num_q_heads=2, num_kv_heads=1, n_tokens=16384 * 8, block_size=8,
           window_tokens=64, topk=100, planted_per_unit=20)
    inp = make_inputs(w, "cuda")
    dec = run_gpu(w, inp)
    compare_all(w, inp, dec)


# ----------------------------------------------------------- full sizes ----

@pytest.mark.parametrize("name", ["mha_32k", "gqa_128k", "two_level_256k", "reserve_128k"])
def test_full_size_every_unit(name):
    """The full configuration in the launch configuration the benchmark times; every
    sequence and KV head is checked against the oracle in full."""
    w = WORKLOADS[name]
    inp = make_inputs(w, "cuda")
    dec = run_gpu(w, inp)
    compare_every_unit(w, inp, dec)
    # workload sanity: planted blocks are found (the query points at them)
    if w.planted_per_unit and not w.two_level:
        ids = as_np(dec.sel_ids).reshape(w.units, -1)
        cnt = as_np(dec.sel_count).reshape(-1)
        planted = as_np(inp["planted"]).reshape(w.units, -1)
        hit = np.mean([np.isin(planted[u], ids[u, : cnt[u]]).mean() for u in range(w.units)])
        assert hit > 0.95, f"planted-block recall {hit:.3f}"
    del inp
    torch.cuda.empty_cache()
