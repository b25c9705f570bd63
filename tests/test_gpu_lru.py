"""Consecutive decode steps: select + decode + diff/LRU on the GPU against the oracle.

The oracle's LRU is fed the GPU's own selections, so a waived near-tie swap in one
step cannot cascade into the cache comparison; every diff list, every count and the
whole slot state are then compared bit for bit at every step.
"""

import numpy as np
import pytest
import torch

import oracle
from query_guided_block_gb300 import binding as B
from query_guided_block_gb300.build import build
from query_guided_block_gb300.decoder import SlotCache, SparseDecoder
from query_guided_block_gb300.workloads import WORKLOADS, make_inputs, scaled
from tests.parity import ATOL, as_np, check_selection, oracle_meta, sub_problem, sub_workload

pytestmark = pytest.mark.gpu

LISTS = {"hit_ids": 0, "miss_ids": 1, "miss_slot": 1, "evict_ids": 2, "evict_slot": 2,
         "new_ids": 3, "dropped_ids": 4}


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available()
    build()
    B.lib()


def _compare_step(cache, r, units):
    gc = as_np(cache.counts)
    assert np.array_equal(gc, r["counts"]), "counts differ"
    for name, ci in LISTS.items():
        g = as_np(cache.lists[name])
        for u in range(units):
            n = r["counts"][u, ci]
            assert np.array_equal(g[u, :n], r[name][u, :n]), f"{name} unit {u}"


def run_steps(w, steps, check_seqs, check_steps, resume_at=None):
    inp = make_inputs(w, "cuda")
    p = B.params_for(w)
    dec = SparseDecoder(p)
    dec.build_meta(inp["k_pages"], inp["block_table"])
    cache = SlotCache(dec, w.cache_slots)
    U, C, W = w.units, w.cache_slots, dec.sel_stride
    blk = np.full((U, C), -1, np.int32)
    last = np.full((U, C), -1, np.int32)
    prev = np.full((U, W), -1, np.int32)
    prev_n = np.zeros(U, np.int32)

    host = sub_problem(w, inp, check_seqs)
    ws = sub_workload(w, len(check_seqs))
    po, (kmin, kmax, _) = oracle_meta(ws, host)
    rows = [s * w.num_kv_heads + h for s in check_seqs for h in range(w.num_kv_heads)]
    overlaps, hit_rates, saved = [], [], None
    for t in range(steps):
        q = inp["q"][t]
        if resume_at is not None and t == resume_at:
            saved = (cache.slot_block.clone(), cache.slot_last_use.clone(),
                     cache.prev_ids.clone(), cache.prev_count.clone())
        dec.select(q)
        dec.decode(q, inp["k_pages"], inp["v_pages"], inp["block_table"])
        cache.diff(t)
        assert dec.device_error() == 0
        gids = as_np(dec.sel_ids).reshape(U, W)
        gcnt = as_np(dec.sel_count).reshape(U)
        r = oracle.lru_step(t, C, gids, gcnt, prev, prev_n, blk, last)
        _compare_step(cache, r, U)
        assert np.array_equal(as_np(cache.slot_block), blk)
        assert np.array_equal(as_np(cache.slot_last_use), last)
        if t > 0:
            overlaps.append(np.mean((gcnt - r["counts"][:, 3]) / gcnt))
            hit_rates.append(np.mean(r["counts"][:, 0] / gcnt))
        if t in check_steps:
            hq = host["q"][t]
            sc = oracle.quest_scores(po, hq, kmin, kmax)
            oid, ocnt = oracle.select(po, sc)
            check_selection(gids[rows], gcnt[rows], oid, ocnt, sc, w.topk, po.first_window_block())
            out = oracle.decode(po, hq, host["k_pages"], host["v_pages"], host["block_table"],
                                gids[rows], gcnt[rows])
            err = np.abs(as_np(dec.out[check_seqs]).astype(np.float64) - out).max()
            assert err <= ATOL[w.kv_dtype]
        cache.advance()
        prev, prev_n = gids.copy(), gcnt.copy()
    return dec, cache, inp, saved, overlaps, hit_rates


def test_lru_scaled_with_checkpoint_resume():
    w = scaled(WORKLOADS["lru_64k"], batch=3, n_tokens=16384 + 100, steps=24, cache_slots=64,
               topk=24, window_tokens=500)
    steps = w.steps
    dec, cache, inp, saved, _, _ = run_steps(w, steps, check_seqs=[0, 2],
                                             check_steps={0, 11, steps - 1}, resume_at=12)
    final = [t.clone() for t in (cache.slot_block, cache.slot_last_use)]
    # resume from the copy taken at step 12 and replay: bit-identical state
    cache.slot_block.copy_(saved[0])
    cache.slot_last_use.copy_(saved[1])
    cache.prev_ids.copy_(saved[2])
    cache.prev_count.copy_(saved[3])
    for t in range(12, steps):
        dec.select(inp["q"][t])
        cache.diff(t)
        cache.advance()
    assert torch.equal(cache.slot_block, final[0]) and torch.equal(cache.slot_last_use, final[1])


def test_lru_full_64_steps():
    """All 64 steps of the 64K configuration: LRU state and lists bit-exact at every
    step on every unit; selection and attention of every unit against the oracle at
    every eighth step and the last."""
    w = WORKLOADS["lru_64k"]
    _, _, _, _, overlaps, hit_rates = run_steps(w, w.steps, check_seqs=list(range(w.batch)),
                                                check_steps=set(range(0, w.steps, 8)) | {w.steps - 1})
    # workload sanity (reported by the pages as 80-90% for real queries): drifting queries
    # keep most of the set from one step to the next
    assert np.mean(overlaps) > 0.5
    assert np.mean(hit_rates) >= np.mean(overlaps) - 1e-9
