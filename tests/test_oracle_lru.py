"""Pins for the oracle's step-to-step diff and LRU slot cache.

The oracle keeps per-slot timestamps and scans slots.  The cross-check below is a
separate textbook formulation: a recency list (OrderedDict, least recent first)
plus a heap of free slot numbers.  Blocks used at the same step are appended in
ascending id order, so list order equals (last use, block id) order -- the
eviction order the diff step defines ("SGLang分层稀疏注意力技术解析与优化实践",
§3.2: a GPU cache 2-4x the top-k, LRU eviction, diff against the previous step,
hits, misses, index update).
"""
import heapq
from collections import OrderedDict

import numpy as np
import pytest

import oracle


class TextbookLRU:
    def __init__(self, slots):
        self.slots = slots
        self.free = list(range(slots))
        heapq.heapify(self.free)
        self.where = {}                 # block -> slot
        self.recency = OrderedDict()    # block -> None, least recent first

    def step(self, request, previous):
        req = sorted(request)
        need = set(req)
        new = [b for b in req if b not in set(previous)]
        dropped = [b for b in sorted(previous) if b not in need]
        hits = [b for b in req if b in self.where]
        misses = [b for b in req if b not in self.where]
        placed, evicted = [], []
        for m in misses:
            if self.free:
                slot = heapq.heappop(self.free)
            else:
                victim = next(b for b in self.recency if b not in need)
                slot = self.where.pop(victim)
                del self.recency[victim]
                evicted.append((victim, slot))
            self.where[m] = slot
            placed.append(slot)
        for b in req:                   # ascending: ties in recency go to the lower id
            self.recency.pop(b, None)
            self.recency[b] = None
        return dict(new=new, dropped=dropped, hits=hits, misses=misses, miss_slot=placed,
                    evicted=evicted)


def _drift_sets(rng, n_steps, universe, size, move):
    cur = sorted(rng.choice(universe, size, replace=False).tolist())
    out = [cur]
    for _ in range(n_steps - 1):
        keep = rng.choice(cur, size - move, replace=False).tolist()
        pool = [b for b in range(universe) if b not in keep]
        cur = sorted(keep + rng.choice(pool, move, replace=False).tolist())
        out.append(cur)
    return out


def _run_oracle(sets_per_unit, slots):
    n_units = len(sets_per_unit)
    steps = len(sets_per_unit[0])
    width = max(len(s) for unit in sets_per_unit for s in unit)
    blk = np.full((n_units, slots), -1, np.int32)
    last = np.full((n_units, slots), -1, np.int32)
    prev = np.full((n_units, width), -1, np.int32)
    prev_n = np.zeros(n_units, np.int32)
    results = []
    for t in range(steps):
        cur = np.full((n_units, width), -1, np.int32)
        cur_n = np.zeros(n_units, np.int32)
        for u in range(n_units):
            s = sets_per_unit[u][t]
            cur[u, : len(s)] = s
            cur_n[u] = len(s)
        r = oracle.lru_step(t, slots, cur, cur_n, prev, prev_n, blk, last)
        results.append((r, blk.copy(), last.copy()))
        prev, prev_n = cur, cur_n
    return results


@pytest.mark.parametrize("seed,slots,size,move,universe",
                         [(0, 16, 5, 1, 40), (1, 8, 8, 3, 30), (2, 128, 40, 6, 1024),
                          (3, 12, 4, 4, 20), (4, 40, 40, 10, 200)])
def test_lru_matches_textbook_formulation(seed, slots, size, move, universe):
    rng = np.random.default_rng(seed)
    n_units, steps = 3, 30
    sets = [_drift_sets(rng, steps, universe, size, move) for _ in range(n_units)]
    got = _run_oracle(sets, slots)
    for u in range(n_units):
        ref = TextbookLRU(slots)
        prev = []
        for t in range(steps):
            want = ref.step(sets[u][t], prev)
            prev = sets[u][t]
            r, blk, _ = got[t]
            c = r["counts"][u]
            assert list(r["new_ids"][u, : c[3]]) == want["new"]
            assert list(r["dropped_ids"][u, : c[4]]) == want["dropped"]
            assert list(r["hit_ids"][u, : c[0]]) == want["hits"]
            assert list(r["miss_ids"][u, : c[1]]) == want["misses"]
            assert list(r["miss_slot"][u, : c[1]]) == want["miss_slot"]
            assert list(zip(r["evict_ids"][u, : c[2]], r["evict_slot"][u, : c[2]])) == want["evicted"]
            # the slot map itself
            assert {int(b): s for s, b in enumerate(blk[u]) if b >= 0} == ref.where


def test_lru_invariants():
    rng = np.random.default_rng(11)
    slots, size = 24, 10
    sets = [_drift_sets(rng, 40, 100, size, 3) for _ in range(4)]
    got = _run_oracle(sets, slots)
    for t, (r, blk, last) in enumerate(got):
        for u in range(4):
            hits, misses, ev, new, dropped = r["counts"][u]
            assert hits + misses == size
            resident_prev = np.count_nonzero(got[t - 1][1][u] >= 0) if t else 0
            assert ev == max(0, misses - (slots - resident_prev))
            assert set(sets[u][t]) <= set(blk[u][blk[u] >= 0].tolist())
            assert np.count_nonzero(blk[u] >= 0) <= slots
            assert all(last[u][s] == t for s in range(slots) if blk[u][s] in sets[u][t])
            assert new == len(set(sets[u][t]) - set(sets[u][t - 1] if t else []))


def test_lru_big_cache_never_evicts_and_constant_set_always_hits():
    rng = np.random.default_rng(5)
    sets = [_drift_sets(rng, 25, 50, 12, 4)]
    got = _run_oracle(sets, 50)
    assert all(r["counts"][0][2] == 0 for r, _, _ in got)
    const = [[list(range(3, 40, 3))] * 10]
    got = _run_oracle(const, 16)
    for t, (r, _, _) in enumerate(got):
        h, m, e, n, d = r["counts"][0]
        assert (h, m, e) == ((0, 13, 0) if t == 0 else (13, 0, 0))
        assert (n, d) == ((13, 0) if t == 0 else (0, 0))


def test_lru_checkpoint_resume_is_bit_identical():
    rng = np.random.default_rng(9)
    slots, size = 32, 10
    sets = _drift_sets(rng, 64, 300, size, 3)
    straight = _run_oracle([sets], slots)
    # 32 steps, copy the state out, continue from the copy
    first = _run_oracle([sets[:32]], slots)
    _, blk, last = first[-1]
    blk, last = blk.copy(), last.copy()
    prev = np.array([sets[31]], np.int32)
    prev_n = np.array([size], np.int32)
    for t in range(32, 64):
        cur = np.array([sets[t]], np.int32)
        r = oracle.lru_step(t, slots, cur, np.array([size], np.int32), prev, prev_n, blk, last)
        r0, blk0, last0 = straight[t]
        for key in r:
            assert np.array_equal(r[key], r0[key]), key
        assert np.array_equal(blk, blk0) and np.array_equal(last, last0)
        prev = cur


def test_lru_rejects_request_larger_than_cache():
    blk = np.full((1, 4), -1, np.int32)
    last = np.full((1, 4), -1, np.int32)
    cur = np.arange(5, dtype=np.int32).reshape(1, 5)
    with pytest.raises(ValueError):
        oracle.lru_step(0, 4, cur, np.array([5], np.int32), cur, np.array([0], np.int32), blk, last)
