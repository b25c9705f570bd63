"""The fused step (sparse_attn_step: selection and attention in one cooperative launch,
SGLang page §1.2 select-then-compute) against the fp64 oracle, and against the two
separate calls bit for bit (same selection, same output bits: both phases run the same
arithmetic in the same order)."""
import dataclasses

import numpy as np
import pytest
import torch

from query_guided_block_gb300 import binding as B
from query_guided_block_gb300.build import build
from query_guided_block_gb300.decoder import SparseDecoder
from query_guided_block_gb300.workloads import WORKLOADS, Workload, make_inputs
from tests.parity import as_np
from tests.test_gpu_parity import compare_all, compare_every_unit

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build()
    B.lib()


def _w(**kw):
    base = dict(name="step_small", batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128,
                n_tokens=5000, block_size=64, window_tokens=300, topk=9)
    base.update(kw)
    return Workload(**base)


def _q(inp):
    return inp["q"] if inp["q"].dim() == 3 else inp["q"][0]


def _pair(w, inp):
    """Two decoders on the same inputs: a = select + decode, b = fused step."""
    p = B.params_for(w)
    a, b = SparseDecoder(p), SparseDecoder(p)
    for d in (a, b):
        d.build_meta(inp["k_pages"], inp["block_table"])
    return a, b


def _run_both(w, inp, a, b, q):
    res = inp.get("reserve_ids")
    a.step(q, inp["k_pages"], inp["v_pages"], inp["block_table"], res)
    b.out.fill_(float("nan"))
    b.step_fused(q, inp["k_pages"], inp["v_pages"], inp["block_table"], res)
    assert a.device_error() == 0
    flags = b.device_error()
    assert flags == 0, f"device error flags 0x{flags:x}"


def _assert_same(a, b):
    cnt = as_np(a.sel_count).reshape(-1)
    assert np.array_equal(cnt, as_np(b.sel_count).reshape(-1))
    ia, ib = as_np(a.sel_ids).reshape(cnt.size, -1), as_np(b.sel_ids).reshape(cnt.size, -1)
    for u in range(cnt.size):
        assert np.array_equal(ia[u, : cnt[u]], ib[u, : cnt[u]]), f"unit {u}"
    assert torch.equal(a.out, b.out), "fused output differs from the two-launch output"


CASES = {
    "quest_g4": dict(),
    "quest_bs32": dict(block_size=32, planted_per_unit=5, n_tokens=20000, topk=12),
    "d64_g8": dict(head_dim=64, num_q_heads=16, block_size=16),
    "g1_bs128": dict(num_q_heads=2, block_size=128, n_tokens=9000, topk=4),
    "mean": dict(score="mean"),
    "q_fp32": dict(q_dtype=torch.float32),
    "q_fp32_d64": dict(head_dim=64, num_q_heads=16, q_dtype=torch.float32, block_size=128, n_tokens=20000),
    "reserve": dict(n_tokens=20000, block_size=32, topk=10, num_reserve=7, planted_per_unit=4),
    "k_zero": dict(topk=0),
    "window_only_all": dict(window_tokens=10 ** 6, topk=3),
    "no_window": dict(window_tokens=0, topk=4),
    "short": dict(n_tokens=37, block_size=16, window_tokens=20, topk=1),
    "many_units": dict(batch=40, num_q_heads=32, num_kv_heads=8, n_tokens=3000, topk=5),
}


@pytest.mark.parametrize("case", list(CASES), ids=list(CASES))
def test_step_matches_oracle_and_two_launches(case):
    w = _w(**CASES[case])
    inp = make_inputs(w, "cuda")
    a, b = _pair(w, inp)
    _run_both(w, inp, a, b, _q(inp))
    _assert_same(a, b)
    compare_all(w, inp, b)


def test_repeated_steps_reset_the_ready_flags():
    """Consecutive fused steps (new queries each time, two-launch calls in between)
    each wait for their own selection: every step equals the two-launch result."""
    w = _w(batch=4, num_q_heads=16, num_kv_heads=4, n_tokens=12000, block_size=32, topk=8)
    inp = make_inputs(w, "cuda")
    a, b = _pair(w, inp)
    g = torch.Generator(device="cuda").manual_seed(5)
    for i in range(6):
        q = torch.randn(_q(inp).shape, generator=g, device="cuda").to(w.q_dtype)
        if i % 2:
            b.select(q)   # a two-launch step on the fused decoder's workspace in between
            b.decode(q, inp["k_pages"], inp["v_pages"], inp["block_table"])
        _run_both(w, inp, a, b, q)
        _assert_same(a, b)
    _run_both(w, inp, a, b, _q(inp))   # the oracle sees the inputs' own query
    _assert_same(a, b)
    compare_all(w, inp, b)


def test_many_small_units():
    """9600 units of a few blocks each: more than one CTA per SM's decode ranges can
    cover, so the step runs as the select kernel followed by the decode kernel waiting
    per unit on the published selections; equal to the two calls."""
    w = _w(batch=1200, num_q_heads=8, num_kv_heads=8, n_tokens=200, block_size=16, window_tokens=40,
           topk=3, planted_per_unit=0)
    assert B.sparse_attn_step_launches(B.params_for(w)) == 2
    inp = make_inputs(w, "cuda")
    a, b = _pair(w, inp)
    for _ in range(2):   # consecutive steps: each waits for its own selections
        _run_both(w, inp, a, b, _q(inp))
        _assert_same(a, b)
    compare_every_unit(w, inp, b)


@pytest.mark.parametrize("case", ["two_level", "fp32_kv", "multi_query"])
def test_unsupported_problems_are_refused(case):
    kw = {"two_level": dict(two_level=True, n_tokens=40000, coarse_block=1024, topk_coarse=4),
          "fp32_kv": dict(kv_dtype=torch.float32, q_dtype=torch.float32),
          "multi_query": dict(num_queries=4)}[case]
    w = _w(**kw)
    inp = make_inputs(w, "cuda")
    d = SparseDecoder(B.params_for(w))
    d.build_meta(inp["k_pages"], inp["block_table"])
    q = _q(inp) if case != "multi_query" else inp["q"]
    with pytest.raises(B.SparseAttnError) as e:
        d.step_fused(q, inp["k_pages"], inp["v_pages"], inp["block_table"])
    assert e.value.status == B.UNSUPPORTED


def test_empty_inputs():
    w = _w(n_tokens=0)
    d = SparseDecoder(B.params_for(w))
    q = torch.randn(w.batch, w.num_q_heads, w.head_dim, device="cuda").to(w.q_dtype)
    dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(1, dtype=torch.int32, device="cuda")
    d.out.fill_(7.0)
    d.step_fused(q, dummy, dummy, bt)
    assert d.device_error() == 0
    assert np.all(as_np(d.sel_count) == 0) and np.all(as_np(d.out) == 0)
    d0 = SparseDecoder(B.params_for(dataclasses.replace(w, batch=0, n_tokens=100)))
    d0.step_fused(q, dummy, dummy, bt)
    assert d0.device_error() == 0


@pytest.mark.parametrize("name", ["gqa_128k", "reserve_128k", "mha_32k"])
def test_full_size(name):
    """The benchmark's workloads: fused equals two launches bit for bit on every unit,
    and every unit matches the oracle."""
    w = WORKLOADS[name]
    inp = make_inputs(w, "cuda")
    a, b = _pair(w, inp)
    _run_both(w, inp, a, b, _q(inp))
    _assert_same(a, b)
    compare_every_unit(w, inp, b)
    del inp, a, b
    torch.cuda.empty_cache()


def _random_cases(n, seed=11):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        D = int(rng.choice([64, 128]))
        Hkv = int(rng.choice([1, 2, 4]))
        G = int(rng.choice([1, 2, 4, 8]))
        bs = int(rng.choice([16, 32, 64, 128]))
        N = int(rng.integers(1, 40000))
        kw = dict(name=f"rand{i}", batch=int(rng.integers(1, 5)), num_kv_heads=Hkv, num_q_heads=Hkv * G,
                  head_dim=D, block_size=bs, n_tokens=N, window_tokens=int(rng.choice([0, 64, 300, 2000])),
                  topk=int(rng.integers(0, 80)), q_dtype=torch.bfloat16 if rng.random() < 0.7 else torch.float32,
                  score="mean" if rng.random() < 0.25 else "quest",
                  num_reserve=int(rng.choice([0, 0, 3, 17])), planted_per_unit=int(rng.integers(0, 6)))
        cases.append(kw)
    return cases


RANDOM = _random_cases(20)


@pytest.mark.parametrize("i", range(len(RANDOM)))
def test_random_problems_match_two_launches(i):
    """Seeded random small problems (group size, head dim, block size, context length,
    k, window, reserve set, scoring, query dtype): the fused step equals the two calls
    bit for bit; every fourth is also checked against the oracle."""
    w = Workload(**RANDOM[i])
    inp = make_inputs(w, "cuda")
    a, b = _pair(w, inp)
    _run_both(w, inp, a, b, _q(inp))
    _assert_same(a, b)
    if i % 4 == 0:
        compare_all(w, inp, b)


def test_wide_candidate_set():
    """6240 candidate blocks per unit (a 200K-token context of 32-token blocks): the
    ranking's keys span 28 per thread; the step equals the two calls and the oracle."""
    w = _w(batch=1, n_tokens=200000, block_size=32, window_tokens=300, topk=20, planted_per_unit=6)
    inp = make_inputs(w, "cuda")
    a, b = _pair(w, inp)
    _run_both(w, inp, a, b, _q(inp))
    _assert_same(a, b)
    compare_all(w, inp, b)


@pytest.mark.parametrize("levels", [1, 3], ids=["one_value", "three_values"])
@pytest.mark.parametrize("score", ["quest", "mean"])
def test_tied_scores_break_by_block_id(levels, score):
    """Keys quantised to one or three values: many blocks share one bound or mean, and
    the top-k takes the lowest block ids among equal scores (the ranking's tie and
    gather paths), as the oracle does."""
    w = _w(n_tokens=20000, block_size=32, topk=40, planted_per_unit=0, score=score)
    inp = make_inputs(w, "cuda")
    k = inp["k_pages"].float()
    k = torch.full_like(k, 0.5) if levels == 1 else torch.clamp(torch.round(k), -1.0, 1.0)
    inp["k_pages"] = k.to(inp["k_pages"].dtype)
    a, b = _pair(w, inp)
    _run_both(w, inp, a, b, _q(inp))
    _assert_same(a, b)
    compare_all(w, inp, b)
