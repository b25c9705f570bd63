"""Pins for the oracle's selection variants (SparDA page §3.2 sparsity ratio by length,
§3.4 reserve set), checked against the page's stated points and against plain Python
set semantics."""
import json
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def test_topk_for_length_matches_the_pages_points():
    g = json.load(open(os.path.join(HERE, "golden", "sparsity_by_length.json")))
    for c in g["cases"]:
        assert oracle.topk_for_length(c["n_tokens"], c["block_size"]) == c["k"], c


def test_topk_for_length_is_monotone_within_each_ratio_band():
    # inside one band the kept count never decreases with length; at a band edge the
    # ratio drops, so k may fall (8K -> 8K + 1 keeps 15% instead of everything)
    for lo, hi in ((8193, 16384), (16385, 32768), (32769, 300000)):
        ks = [oracle.topk_for_length(n, 64) for n in range(lo, hi, 997)]
        assert all(a <= b for a, b in zip(ks, ks[1:]))


def test_topk_for_length_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.topk_for_length(-1, 64)
    with pytest.raises(ValueError):
        oracle.topk_for_length(1024, 0)


def _selection(p, rng):
    """A valid selection (ascending top-k ids below the window, then the window)."""
    nb, wf = p.num_blocks, p.first_window_block()
    stride = p.sel_stride()
    ids = np.full((p.units, stride), -1, np.int32)
    cnt = np.zeros(p.units, np.int32)
    for u in range(p.units):
        top = sorted(rng.choice(wf, size=min(p.topk, wf), replace=False).tolist()) if wf else []
        row = top + list(range(wf, nb))
        ids[u, :len(row)] = row
        cnt[u] = len(row)
    return ids, cnt


@pytest.mark.parametrize("seed", range(6))
def test_union_reserve_equals_set_union(seed):
    rng = np.random.default_rng(seed)
    p = oracle.problem(batch=2, num_q_heads=4, num_kv_heads=2, head_dim=64,
                       n_tokens=int(rng.integers(64, 2000)), block_size=32, num_pages=64,
                       window_tokens=int(rng.integers(0, 200)), topk=int(rng.integers(0, 12)))
    ids, cnt = _selection(p, rng)
    n_res = int(rng.integers(0, 9))
    # reserve ids anywhere in [0, nb): duplicates, window ids and top-k ids included
    res = rng.integers(0, p.num_blocks, size=(p.units, n_res)).astype(np.int32)
    if n_res >= 2:
        res[:, 1] = res[:, 0]
    out, ocnt = oracle.union_reserve(p, ids, cnt, res)
    for u in range(p.units):
        want = sorted(set(ids[u, :cnt[u]].tolist()) | set(res[u].tolist()))
        assert out[u, :ocnt[u]].tolist() == want


def test_union_reserve_without_reserve_is_the_selection():
    rng = np.random.default_rng(7)
    p = oracle.problem(batch=1, num_q_heads=2, num_kv_heads=2, head_dim=64, n_tokens=1024,
                       block_size=64, num_pages=16, window_tokens=128, topk=4)
    ids, cnt = _selection(p, rng)
    out, ocnt = oracle.union_reserve(p, ids, cnt, np.zeros((p.units, 0), np.int32))
    assert (ocnt == cnt).all()
    for u in range(p.units):
        assert (out[u, :cnt[u]] == ids[u, :cnt[u]]).all()


def test_union_reserve_rejects_ids_outside_the_context():
    rng = np.random.default_rng(8)
    p = oracle.problem(batch=1, num_q_heads=2, num_kv_heads=2, head_dim=64, n_tokens=512,
                       block_size=64, num_pages=8, window_tokens=64, topk=2)
    ids, cnt = _selection(p, rng)
    with pytest.raises(ValueError):
        oracle.union_reserve(p, ids, cnt, np.full((p.units, 1), p.num_blocks, np.int32))
