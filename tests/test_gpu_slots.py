"""Slot pool fed from a host-resident store ("SGLang分层稀疏注意力技术解析与优化实践" §3.3
IO transfer, §3.2 steps c-d), through the C ABI:

* after each step's diff, the misses are copied from pinned host memory into their slots;
* decoding through the slot map equals decoding through the page table bit for bit
  (same kernel, same values, same order) and matches the oracle on the GPU's selection;
* every pool tile holds exactly the page tile of the block its slot names.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
from query_guided_block_gb300 import binding as B
from query_guided_block_gb300.build import build
from query_guided_block_gb300.decoder import SlotCache, SlotPool, SparseDecoder
from query_guided_block_gb300.workloads import WORKLOADS, make_inputs, scaled
from tests.parity import ATOL, as_np, oracle_meta, sub_problem, sub_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build()
    B.lib()


def _run_steps(w, inp, store_k, store_v, steps, check_oracle_at=()):
    p = B.params_for(w)
    dec = SparseDecoder(p)
    dec.build_meta(inp["k_pages"], inp["block_table"])
    cache = SlotCache(dec, w.cache_slots)
    pool = SlotPool(cache)
    out_pages = torch.empty_like(dec.out)
    for t in range(steps):
        q = inp["q"][t]
        dec.select(q)
        cache.diff(t)
        pool.load_misses(store_k, store_v, inp["block_table"])
        pool.slot_map()
        pool.decode(q)
        dec.decode(q, inp["k_pages"], inp["v_pages"], inp["block_table"], out=out_pages)
        torch.cuda.synchronize()
        assert dec.device_error() == 0
        assert torch.equal(dec.out, out_pages), f"step {t}: slot decode differs from page decode"
        _check_pool(w, inp, cache, pool, t)
        if t in check_oracle_at:
            _check_oracle(w, inp, dec, t)
        cache.advance()
    return dec, cache, pool


def _check_pool(w, inp, cache, pool, t):
    """Every resident slot holds its block's K and V tiles exactly."""
    blk = as_np(cache.slot_block)
    bt = inp["block_table"].long()
    rng = np.random.default_rng(t)
    for u in rng.choice(w.units, size=min(6, w.units), replace=False):
        b, h = divmod(int(u), w.num_kv_heads)
        for s in np.nonzero(blk[u] >= 0)[0][:12]:
            page = int(bt[b, int(blk[u, s])])
            assert torch.equal(pool.pool_k[u, s], inp["k_pages"][page, h])
            assert torch.equal(pool.pool_v[u, s], inp["v_pages"][page, h])


def _check_oracle(w, inp, dec, t):
    seqs = [0, w.batch - 1]
    host = sub_problem(w, inp, seqs)
    ws = sub_workload(w, len(seqs))
    p, _ = oracle_meta(ws, host)
    rows = [s * w.num_kv_heads + h for s in seqs for h in range(w.num_kv_heads)]
    gids = as_np(dec.sel_ids).reshape(w.units, -1)[rows]
    gcnt = as_np(dec.sel_count).reshape(-1)[rows]
    ref = oracle.decode(p, host["q"][t], host["k_pages"], host["v_pages"], host["block_table"], gids, gcnt)
    got = as_np(dec.out[seqs]).astype(np.float64)
    assert np.abs(got - ref).max() <= ATOL[w.kv_dtype]


def _small():
    return scaled(WORKLOADS["lru_64k"], batch=3, n_tokens=16384 + 100, steps=8, cache_slots=64)


def test_slot_decode_from_pinned_host_store():
    w = _small()
    inp = make_inputs(w, "cuda")
    hk = inp["k_pages"].cpu().pin_memory()
    hv = inp["v_pages"].cpu().pin_memory()
    _run_steps(w, inp, hk, hv, w.steps, check_oracle_at=(0, w.steps - 1))


def test_slot_decode_from_device_store():
    w = scaled(_small(), steps=3)
    inp = make_inputs(w, "cuda")
    _run_steps(w, inp, inp["k_pages"], inp["v_pages"], w.steps)


def test_full_size_slot_pool():
    """lru_64k (B32, 65536 tokens, 128 slots per KV head), 4 steps from pinned memory."""
    w = scaled(WORKLOADS["lru_64k"], steps=4, name="lru_64k")
    inp = make_inputs(w, "cuda")
    hk = inp["k_pages"].cpu().pin_memory()
    hv = inp["v_pages"].cpu().pin_memory()
    _run_steps(w, inp, hk, hv, w.steps, check_oracle_at=(w.steps - 1,))


def test_selected_block_not_resident_is_reported():
    w = scaled(_small(), steps=1)
    inp = make_inputs(w, "cuda")
    dec = SparseDecoder(B.params_for(w))
    dec.build_meta(inp["k_pages"], inp["block_table"])
    cache = SlotCache(dec, w.cache_slots)
    pool = SlotPool(cache)
    dec.select(inp["q"][0])
    pool.slot_map()                      # no diff: nothing is resident yet
    assert dec.device_error() & B.ERR_SLOT
    assert (as_np(pool.sel_slot)[:, 0] == -1).all()


def test_unregistered_host_store_is_rejected():
    w = scaled(_small(), steps=1)
    inp = make_inputs(w, "cuda")
    dec = SparseDecoder(B.params_for(w))
    cache = SlotCache(dec, w.cache_slots)
    pool = SlotPool(cache)
    pageable = np.zeros(inp["k_pages"].numel() * 2 // 4 + 4, dtype=np.float32)   # plain host memory
    ptr = C.c_void_p(pageable.ctypes.data)
    rc = B.lib().sparse_attn_load_misses(
        C.byref(dec.p), ptr, ptr, B._ptr(inp["block_table"]), B._ptr(cache.lists["miss_ids"]),
        B._ptr(cache.lists["miss_slot"]), B._ptr(cache.counts), w.cache_slots,
        B._ptr(pool.pool_k), B._ptr(pool.pool_v), B._ptr(dec.ws), dec.ws_bytes, None)
    assert rc == B.INVALID_ARG


def _check_same_pool_and_output(w, pool_a, pool_b, out_a, out_b, counts, t):
    """The pools end equal; outputs are the same bits for units without misses (same
    order) and equal up to fp32 rounding of the reordered sum for the others (the fused
    pass attends to a unit's missed blocks last)."""
    assert torch.equal(pool_a.pool_k, pool_b.pool_k) and torch.equal(pool_a.pool_v, pool_b.pool_v), f"step {t}"
    g = w.num_q_heads // w.num_kv_heads
    oa = out_a.reshape(w.units, g, -1)
    ob = out_b.reshape(w.units, g, -1)
    clean = counts[:, 1] == 0
    assert torch.equal(oa[clean], ob[clean]), f"step {t}: a unit without misses changed"
    assert torch.allclose(oa, ob, rtol=1e-5, atol=1e-6), f"step {t}: {float((oa - ob).abs().max())}"


@pytest.mark.parametrize("store", ["pinned", "device"])
def test_fused_miss_load_equals_load_then_decode(store):
    """sparse_attn_decode_slots_io (misses loaded in the decode's own launch) against
    load_misses + decode_slots over drifting steps, ragged last block included."""
    w = _small()
    inp = make_inputs(w, "cuda")
    if store == "pinned":
        hk, hv = inp["k_pages"].cpu().pin_memory(), inp["v_pages"].cpu().pin_memory()
    else:
        hk, hv = inp["k_pages"], inp["v_pages"]
    p = B.params_for(w)
    runs = []
    for _ in range(2):
        dec = SparseDecoder(p)
        dec.build_meta(inp["k_pages"], inp["block_table"])
        cache = SlotCache(dec, w.cache_slots)
        runs.append((dec, cache, SlotPool(cache)))
    (da, ca, pa), (db, cb, pb) = runs
    misses = 0
    for t in range(w.steps):
        q = inp["q"][t]
        for dec, cache, pool in runs:   # run b: the diff writes the slot map itself
            dec.select(q)
            cache.diff(t, sel_slot=pool.sel_slot if pool is pb else None)
        pa.load_misses(hk, hv, inp["block_table"])
        pa.slot_map()
        pa.decode(q)
        pb.decode_io(q, hk, hv, inp["block_table"])
        torch.cuda.synchronize()
        assert da.device_error() == 0 and db.device_error() == 0
        assert torch.equal(ca.counts, cb.counts)
        assert torch.equal(pa.sel_slot, pb.sel_slot), f"step {t}: the diff's slot map differs"
        misses += int(cb.counts[:, 1].sum())
        _check_same_pool_and_output(w, pa, pb, da.out, db.out, cb.counts, t)
        for _, cache, _ in runs:
            cache.advance()
    assert misses > 0


def test_fused_miss_load_full_size():
    """lru_64k at full size, 3 steps from pinned memory: the fused pass against the
    two-launch path on every output and every slot."""
    w = scaled(WORKLOADS["lru_64k"], steps=3, name="lru_64k")
    inp = make_inputs(w, "cuda")
    hk, hv = inp["k_pages"].cpu().pin_memory(), inp["v_pages"].cpu().pin_memory()
    p = B.params_for(w)
    runs = []
    for _ in range(2):
        dec = SparseDecoder(p)
        dec.build_meta(inp["k_pages"], inp["block_table"])
        cache = SlotCache(dec, w.cache_slots)
        runs.append((dec, cache, SlotPool(cache)))
    (da, ca, pa), (db, cb, pb) = runs
    for t in range(w.steps):
        q = inp["q"][t]
        for dec, cache, pool in runs:
            dec.select(q)
            cache.diff(t, sel_slot=pool.sel_slot if pool is pb else None)
        pa.load_misses(hk, hv, inp["block_table"])
        pa.slot_map()
        pa.decode(q)
        pb.decode_io(q, hk, hv, inp["block_table"])
        torch.cuda.synchronize()
        assert da.device_error() == 0 and db.device_error() == 0
        _check_same_pool_and_output(w, pa, pb, da.out, db.out, cb.counts, t)
        for _, cache, _ in runs:
            cache.advance()
