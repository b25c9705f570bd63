"""The oracle against values fixed outside it: arithmetic printed on the pages and a
hand-worked example with closed-form answers (fixtures under tests/golden/)."""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _closed_form(expr: str) -> float:
    return float(eval(expr, {"__builtins__": {}}, {"exp": math.exp}))


def _case_problem(c, **kw):
    args = dict(batch=1, num_q_heads=1, num_kv_heads=1, head_dim=2,
                n_tokens=c["n_tokens"], block_size=c.get("block_size", 64), num_pages=0,
                window_tokens=c.get("window_tokens", 0), topk=c.get("topk", 0),
                two_level="coarse_block" in c and "block_size" in c,
                coarse_block=c.get("coarse_block", 1024), topk_coarse=c.get("topk_coarse", 0),
                kv_bf16=False, q_bf16=False)
    args.update(kw)
    p = oracle.problem(**args)
    p.num_pages = p.num_blocks
    return p


def _random_pages(p, seed=0):
    rng = np.random.default_rng(seed)
    pages = rng.standard_normal((p.num_pages, 1, p.block_size, p.head_dim)).astype(np.float32)
    table = rng.permutation(p.num_pages).astype(np.int32).reshape(1, -1)
    q = rng.standard_normal((1, 1, p.head_dim)).astype(np.float32)
    return pages, table, q


@pytest.mark.parametrize("idx", range(4))
def test_page_arithmetic(idx):
    c = _load("page_arithmetic.json")["cases"][idx]
    if "expect_coarse_blocks" in c:
        p = _case_problem(c, two_level=True, block_size=64)
        assert p.num_mean_rows() == c["expect_coarse_blocks"]
    if "expect_blocks" in c:
        p = _case_problem(c)
        assert p.num_blocks == c["expect_blocks"]
    if "expect_level2_candidates" in c:
        p = _case_problem(c, two_level=True)
        pages, table, q = _random_pages(p)
        kmin, kmax, kmean = oracle.build_meta(p, pages, table, with_mean=True)
        r = oracle.select_two_level(p, q, kmin, kmax, kmean)
        assert r["n_survivors"][0] == c["topk_coarse"]
        assert np.count_nonzero(~np.isnan(r["slice_scores"][0])) == c["expect_level2_candidates"]
    if "expect_selected_tokens" in c:
        p = _case_problem(c)
        pages, table, q = _random_pages(p)
        kmin, kmax, _ = oracle.build_meta(p, pages, table)
        ids, cnt = oracle.select(p, oracle.quest_scores(p, q, kmin, kmax))
        assert cnt[0] * p.block_size == c["expect_selected_tokens"]


def test_hand_worked_example():
    g = _load("hand_worked_example.json")
    k = np.array(g["pages_k"], np.float32).reshape(2, 1, 2, 2)
    v = np.array(g["pages_v"], np.float32).reshape(2, 1, 2, 2)
    table = np.array([g["block_table"]], np.int32)
    q = np.array(g["q"], np.float32).reshape(1, 1, 2)
    for case in g["cases"]:
        p = oracle.problem(1, 1, 1, 2, 4, 2, 2, case["window_tokens"], case["topk"],
                           kv_bf16=False, q_bf16=False, softmax_scale=1.0)
        kmin, kmax, _ = oracle.build_meta(p, k, table)
        s = oracle.quest_scores(p, q, kmin, kmax)
        assert list(s[0]) == [_closed_form(e) for e in g["expect_scores"]]
        ids, cnt = oracle.select(p, s)
        assert list(ids[0, : cnt[0]]) == case["expect_sel"]
        out = oracle.decode(p, q, k, v, table, ids, cnt)
        want = [_closed_form(e) for e in case["expect_out"]]
        np.testing.assert_allclose(out[0, 0], want, rtol=0, atol=1e-15)
