"""Pins for the fp64 CPU oracle: each check ties it to something other than itself.

What pins what:
  * build_meta      -- numpy min / max / mean over tokens gathered through the page table
                       independently; tokens past the context end are poisoned and must
                       not leak in.
  * Quest score     -- the bound property (score >= q.k for every key of the block), the
                       bound being attained when a key sits on the box corner, and the
                       block-size-1 case where it collapses to the exact logit.
  * mean score      -- linearity: q . mean(K) == mean over tokens of q . k.
  * selection       -- brute force over every k-subset on tiny inputs (ties included), the
                       window always present, numpy's stable argsort when bs == 1.
  * decode          -- all blocks selected == dense softmax attention from torch's
                       scaled_dot_product_attention in fp64; any subset == dense attention
                       over the gathered subset; one token -> its value; q == 0 -> mean.
  * two-level       -- K1 covering every coarse block == single-level Quest; coarse block ==
                       slice -> the survivors themselves; survivors == brute-force top-K1.
LRU pins live in test_oracle_lru.py.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from query_guided_block_gb300.workloads import Workload, make_inputs
from tests.conftest import oracle_problem_for


def _small(name="pin", **kw):
    base = dict(name=name, batch=2, num_q_heads=4, num_kv_heads=2, head_dim=16,
                n_tokens=300, block_size=16, window_tokens=40, topk=5,
                kv_dtype=torch.float32, q_dtype=torch.float32)
    base.update(kw)
    return Workload(**base)


def _logical_kv(w, pages, block_table):
    """[B, Hkv, N, D] float64 keys in token order, gathered independently of the oracle."""
    x = oracle.host_array(pages)
    if x.dtype == np.uint16:
        x = (x.astype(np.uint32) << 16).view(np.float32)
    x = x.astype(np.float64)
    bt = np.asarray(block_table)
    B, nb, bs = w.batch, w.num_blocks, w.block_size
    out = np.empty((B, w.num_kv_heads, nb * bs, w.head_dim))
    for b in range(B):
        g = x[bt[b]]                                  # [nb, Hkv, bs, D]
        out[b] = g.transpose(1, 0, 2, 3).reshape(w.num_kv_heads, nb * bs, w.head_dim)
    return out[:, :, : w.n_tokens]


def _q64(q):
    x = oracle.host_array(q)
    if x.dtype == np.uint16:
        x = (x.astype(np.uint32) << 16).view(np.float32)
    return x.astype(np.float64)


def _poison_tail(w, inp):
    """Write huge values into the page slots past the context end."""
    tail = w.n_tokens % w.block_size
    if tail == 0:
        return
    for b in range(w.batch):
        page = int(inp["block_table"][b, w.num_blocks - 1])
        inp["k_pages"][page, :, tail:] = 1e30
        inp["v_pages"][page, :, tail:] = -1e30


# --------------------------------------------------------------- metadata --

@pytest.mark.parametrize("kv", [torch.float32, torch.bfloat16])
def test_meta_is_blockwise_min_max_and_mean(kv):
    w = _small(kv_dtype=kv, q_dtype=kv, score="mean")
    inp = make_inputs(w)
    _poison_tail(w, inp)
    p = oracle_problem_for(w)
    kmin, kmax, kmean = oracle.build_meta(p, inp["k_pages"], inp["block_table"], with_mean=True)
    K = _logical_kv(w, inp["k_pages"], inp["block_table"])
    for j in range(w.num_blocks):
        seg = K[:, :, j * w.block_size: (j + 1) * w.block_size]
        assert np.array_equal(kmin[:, :, j], seg.min(axis=2))
        assert np.array_equal(kmax[:, :, j], seg.max(axis=2))
        np.testing.assert_allclose(kmean[:, :, j], seg.mean(axis=2), rtol=0, atol=1e-13)
    assert np.abs(kmax).max() < 1e29, "tokens past the context end leaked into the metadata"


def test_coarse_mean_rows():
    w = _small(two_level=True, coarse_block=64, topk_coarse=2)
    inp = make_inputs(w)
    p = oracle_problem_for(w)
    _, _, kmean = oracle.build_meta(p, inp["k_pages"], inp["block_table"], with_mean=True)
    K = _logical_kv(w, inp["k_pages"], inp["block_table"])
    rows = math.ceil(w.n_tokens / 64)
    assert kmean.shape[2] == rows
    for r in range(rows):
        np.testing.assert_allclose(kmean[:, :, r], K[:, :, r * 64:(r + 1) * 64].mean(axis=2),
                                   rtol=0, atol=1e-13)


# ------------------------------------------------------------ Quest score --

@pytest.mark.parametrize("G,kv", [(1, torch.float32), (2, torch.float32), (4, torch.bfloat16)])
def test_quest_bound_dominates_every_key(G, kv):
    w = _small(num_q_heads=2 * G, num_kv_heads=2, kv_dtype=kv, q_dtype=kv)
    inp = make_inputs(w)
    p = oracle_problem_for(w)
    kmin, kmax, _ = oracle.build_meta(p, inp["k_pages"], inp["block_table"])
    s = oracle.quest_scores(p, inp["q"], kmin, kmax).reshape(w.batch, w.num_kv_heads, -1)
    K = _logical_kv(w, inp["k_pages"], inp["block_table"])
    q = _q64(inp["q"]).reshape(w.batch, w.num_kv_heads, G, w.head_dim)
    qk = np.einsum("bhgd,bhtd->bht", q, K)             # group-summed q.k per token
    for j in range(w.num_blocks):
        best = qk[:, :, j * w.block_size:(j + 1) * w.block_size].max(axis=2)
        assert np.all(s[:, :, j] >= best - 1e-9 * np.abs(best))


def test_quest_bound_attained_at_box_corner():
    """When a key of the block sits on the corner the query points to, score == q.k."""
    rng = np.random.default_rng(7)
    D, bs = 8, 4
    for trial in range(20):
        q = rng.standard_normal(D)
        keys = rng.standard_normal((bs, D))
        lo, hi = keys.min(0), keys.max(0)
        corner = np.where(q >= 0, hi, lo)
        keys[rng.integers(bs)] = corner               # still inside the same box
        pages = keys.reshape(1, 1, bs, D).astype(np.float32)
        p = oracle.problem(1, 1, 1, D, bs, bs, 1, 0, 1, kv_bf16=False, q_bf16=False)
        kmin, kmax, _ = oracle.build_meta(p, pages, np.zeros((1, 1), np.int32))
        qa = q.astype(np.float32).reshape(1, 1, D)
        s = oracle.quest_scores(p, qa, kmin, kmax)[0, 0]
        want = float(qa[0, 0].astype(np.float64) @ corner.astype(np.float32).astype(np.float64))
        assert s == pytest.approx(want, rel=1e-12, abs=1e-12)
        # and any other key strictly inside gives at most that value
        assert s >= (qa[0, 0].astype(np.float64) @ keys.astype(np.float32).astype(np.float64).T).max() - 1e-12


@pytest.mark.parametrize("G", [1, 4])
def test_quest_block_size_one_is_exact_logit_and_argsort_topk(G):
    w = _small(num_q_heads=2 * G, num_kv_heads=2, block_size=1, n_tokens=97, window_tokens=5,
               topk=11)
    inp = make_inputs(w)
    p = oracle_problem_for(w)
    kmin, kmax, _ = oracle.build_meta(p, inp["k_pages"], inp["block_table"])
    s = oracle.quest_scores(p, inp["q"], kmin, kmax)
    K = _logical_kv(w, inp["k_pages"], inp["block_table"])
    q = _q64(inp["q"]).reshape(w.batch, w.num_kv_heads, G, w.head_dim)
    logit = np.einsum("bhgd,bhtd->bht", q, K).reshape(w.units, -1)
    np.testing.assert_allclose(s, logit, rtol=1e-12, atol=1e-12)
    ids, cnt = oracle.select(p, s)
    nwin = 5
    for u in range(w.units):
        cand = logit[u, : w.n_tokens - nwin]
        order = np.argsort(-cand, kind="stable")[: w.topk]
        want = np.sort(np.concatenate([order, np.arange(w.n_tokens - nwin, w.n_tokens)]))
        assert cnt[u] == len(want)
        assert np.array_equal(ids[u, : cnt[u]], want)


def test_mean_score_is_linear_in_tokens():
    w = _small(score="mean", num_q_heads=8, num_kv_heads=2)
    inp = make_inputs(w)
    p = oracle_problem_for(w)
    _, _, kmean = oracle.build_meta(p, inp["k_pages"], inp["block_table"], with_mean=True)
    s = oracle.mean_scores(p, inp["q"], kmean).reshape(w.batch, w.num_kv_heads, -1)
    K = _logical_kv(w, inp["k_pages"], inp["block_table"])
    q = _q64(inp["q"]).reshape(w.batch, w.num_kv_heads, 4, w.head_dim)
    per_token = np.einsum("bhgd,bhtd->bht", q, K)
    for j in range(w.num_blocks):
        want = per_token[:, :, j * w.block_size:(j + 1) * w.block_size].mean(axis=2)
        np.testing.assert_allclose(s[:, :, j], want, rtol=1e-11, atol=1e-11)


# -------------------------------------------------------------- selection --

def _precedes(a, b, score):
    """a comes before b in (score desc, id asc) order."""
    return score[a] > score[b] or (score[a] == score[b] and a < b)


@pytest.mark.parametrize("seed", range(12))
def test_selection_equals_bruteforce_definition(seed):
    rng = np.random.default_rng(seed)
    nb = int(rng.integers(3, 13))
    bs = 4
    W = int(rng.integers(0, 3)) * bs
    k = int(rng.integers(0, nb + 2))
    p = oracle.problem(1, 1, 1, 4, nb * bs, bs, nb, W, k, kv_bf16=False, q_bf16=False)
    score = rng.integers(-3, 4, size=nb).astype(np.float64)   # many exact ties
    ids, cnt = oracle.select(p, score.reshape(1, nb))
    wf = nb - W // bs
    cand = list(range(wf))
    keep = min(k, wf)
    winners = []
    for S in itertools.combinations(cand, keep):
        rest = [c for c in cand if c not in S]
        if all(_precedes(a, b, score) for a in S for b in rest):
            winners.append(S)
    assert len(winners) == 1
    want = sorted(list(winners[0]) + list(range(wf, nb)))
    assert cnt[0] == len(want)
    assert list(ids[0, : cnt[0]]) == want


@pytest.mark.parametrize("N,bs,W", [(300, 16, 40), (257, 32, 33), (64, 16, 1000), (100, 10, 0)])
def test_window_always_selected(N, bs, W):
    w = _small(n_tokens=N, block_size=bs, window_tokens=W, topk=3)
    inp = make_inputs(w)
    p = oracle_problem_for(w)
    kmin, kmax, _ = oracle.build_meta(p, inp["k_pages"], inp["block_table"])
    ids, cnt = oracle.select(p, oracle.quest_scores(p, inp["q"], kmin, kmax))
    window = sorted({t // bs for t in range(max(0, N - W), N)})
    n_cand = w.num_blocks - len(window)
    for u in range(w.units):
        sel = list(ids[u, : cnt[u]])
        assert set(window) <= set(sel)
        assert cnt[u] == min(3, n_cand) + len(window)
        assert sel == sorted(set(sel))


# ----------------------------------------------------------------- decode --

def _dense(q, K, V, G, scale=None):
    """torch SDPA in fp64: q [B,Hq,D], K/V [B,Hkv,T,D]."""
    qt = torch.from_numpy(q).unsqueeze(2)
    kt = torch.from_numpy(K).repeat_interleave(G, dim=1)
    vt = torch.from_numpy(V).repeat_interleave(G, dim=1)
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)[:, :, 0].numpy()


@pytest.mark.parametrize("G,kv,N", [(1, torch.float32, 300), (4, torch.float32, 250),
                                    (4, torch.bfloat16, 256)])
def test_decode_all_blocks_equals_dense_attention(G, kv, N):
    w = _small(num_q_heads=2 * G, num_kv_heads=2, kv_dtype=kv, q_dtype=kv, n_tokens=N, topk=10 ** 6)
    inp = make_inputs(w)
    _poison_tail(w, inp)
    p = oracle_problem_for(w)
    kmin, kmax, _ = oracle.build_meta(p, inp["k_pages"], inp["block_table"])
    ids, cnt = oracle.select(p, oracle.quest_scores(p, inp["q"], kmin, kmax))
    assert np.all(cnt == w.num_blocks)
    out = oracle.decode(p, inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"], ids, cnt)
    K = _logical_kv(w, inp["k_pages"], inp["block_table"])
    V = _logical_kv(w, inp["v_pages"], inp["block_table"])
    ref = _dense(_q64(inp["q"]), K, V, G)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_decode_subset_equals_dense_over_gathered_subset():
    G = 2
    w = _small(num_q_heads=2 * G, num_kv_heads=2, n_tokens=290)
    inp = make_inputs(w)
    _poison_tail(w, inp)
    p = oracle_problem_for(w, softmax_scale=0.3)
    rng = np.random.default_rng(3)
    nb, bs = w.num_blocks, w.block_size
    stride = 7
    ids = np.full((w.units, stride), -1, np.int32)
    cnt = np.zeros(w.units, np.int32)
    for u in range(w.units):
        pick = np.sort(rng.choice(nb, size=int(rng.integers(1, stride + 1)), replace=False))
        if u == 0:
            pick[-1] = nb - 1                       # include the ragged last block
            pick = np.unique(pick)
        ids[u, : len(pick)] = pick
        cnt[u] = len(pick)
    out = oracle.decode(p, inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"], ids, cnt)
    K = _logical_kv(w, inp["k_pages"], inp["block_table"])
    V = _logical_kv(w, inp["v_pages"], inp["block_table"])
    q = _q64(inp["q"])
    for u in range(w.units):
        b, kvh = divmod(u, w.num_kv_heads)
        toks = [t for j in ids[u, : cnt[u]] for t in range(j * bs, min((j + 1) * bs, w.n_tokens))]
        ref = _dense(q[b:b + 1, kvh * G:(kvh + 1) * G], K[b:b + 1, kvh:kvh + 1, toks],
                     V[b:b + 1, kvh:kvh + 1, toks], G, scale=0.3)
        np.testing.assert_allclose(out[b, kvh * G:(kvh + 1) * G], ref[0], rtol=0, atol=1e-12)


def test_decode_single_token_and_zero_query():
    w = _small(block_size=1, n_tokens=50, num_q_heads=2, num_kv_heads=2)
    inp = make_inputs(w)
    p = oracle_problem_for(w)
    V = _logical_kv(w, inp["v_pages"], inp["block_table"])
    ids = np.array([[17], [3], [49], [0]], np.int32)
    cnt = np.ones(4, np.int32)
    out = oracle.decode(p, inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"], ids, cnt)
    for u in range(4):
        b, h = divmod(u, 2)
        assert np.array_equal(out[b, h], V[b, h, ids[u, 0]])
    # q == 0: uniform weights -> plain mean of the selected values
    w2 = _small(num_q_heads=2, num_kv_heads=2)
    inp2 = make_inputs(w2)
    inp2["q"].zero_()
    p2 = oracle_problem_for(w2)
    ids2 = np.array([[0, 4, 18]] * 4, np.int32)
    cnt2 = np.full(4, 3, np.int32)
    out2 = oracle.decode(p2, inp2["q"], inp2["k_pages"], inp2["v_pages"], inp2["block_table"],
                         ids2, cnt2)
    V2 = _logical_kv(w2, inp2["v_pages"], inp2["block_table"])
    toks = [t for j in (0, 4, 18) for t in range(j * 16, min((j + 1) * 16, w2.n_tokens))]
    for u in range(4):
        b, h = divmod(u, 2)
        np.testing.assert_allclose(out2[b, h], V2[b, h, toks].mean(axis=0), rtol=0, atol=1e-13)


# -------------------------------------------------------------- two-level --

def _two_level_case(**kw):
    base = dict(name="pin2", batch=2, num_q_heads=4, num_kv_heads=2, head_dim=16,
                n_tokens=1000, block_size=16, window_tokens=48, topk=6, two_level=True,
                coarse_block=64, topk_coarse=4, kv_dtype=torch.float32, q_dtype=torch.float32)
    base.update(kw)
    w = Workload(**base)
    inp = make_inputs(w)
    p = oracle_problem_for(w)
    kmin, kmax, kmean = oracle.build_meta(p, inp["k_pages"], inp["block_table"], with_mean=True)
    return w, inp, p, kmin, kmax, kmean


def test_two_level_with_every_coarse_block_is_single_level():
    w, inp, p, kmin, kmax, kmean = _two_level_case(topk_coarse=100)
    r = oracle.select_two_level(p, inp["q"], kmin, kmax, kmean)
    p1 = oracle_problem_for(w, two_level=False)
    ids, cnt = oracle.select(p1, oracle.quest_scores(p1, inp["q"], kmin, kmax))
    assert np.array_equal(r["sel_count"], cnt)
    for u in range(w.units):
        assert np.array_equal(r["sel_ids"][u, : cnt[u]], ids[u, : cnt[u]])


def test_two_level_coarse_equal_to_slice_keeps_the_survivors():
    w, inp, p, kmin, kmax, kmean = _two_level_case(coarse_block=16, topk_coarse=5, topk=9)
    r = oracle.select_two_level(p, inp["q"], kmin, kmax, kmean)
    wf = p.first_window_block()
    for u in range(w.units):
        surv = r["survivors"][u, : r["n_survivors"][u]]
        want = sorted(set(int(c) for c in surv if c < wf) | set(range(wf, w.num_blocks)))
        assert list(r["sel_ids"][u, : r["sel_count"][u]]) == want


def test_two_level_survivors_are_bruteforce_top_mean():
    w, inp, p, kmin, kmax, kmean = _two_level_case()
    r = oracle.select_two_level(p, inp["q"], kmin, kmax, kmean)
    K = _logical_kv(w, inp["k_pages"], inp["block_table"])
    qsum = _q64(inp["q"]).reshape(w.batch, w.num_kv_heads, 2, w.head_dim).sum(axis=2)
    rows = math.ceil(w.n_tokens / 64)
    for u in range(w.units):
        b, kvh = divmod(u, w.num_kv_heads)
        sc = np.array([qsum[b, kvh] @ K[b, kvh, c * 64:(c + 1) * 64].mean(axis=0) for c in range(rows)])
        np.testing.assert_allclose(r["coarse_scores"][u], sc, rtol=1e-11, atol=1e-11)
        order = sorted(range(rows), key=lambda c: (-sc[c], c))[:4]
        assert list(r["survivors"][u, :4]) == sorted(order)
        # level-2 candidates: exactly the non-window slices of the survivors
        cand = {c * 4 + s for c in order for s in range(4)}
        cand = {j for j in cand if j < p.first_window_block() and j < w.num_blocks}
        assert set(np.flatnonzero(~np.isnan(r["slice_scores"][u]))) == cand
