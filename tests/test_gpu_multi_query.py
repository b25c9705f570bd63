"""Multi-query variant through the C ABI: Q query vectors per sequence share one
selection per KV head, scored by the Quest bound summed over all Q x G query heads
(the bound is linear in q, so the oracle sums its per-query scores), and each query
gets exact softmax attention over the selected tokens ("从HiSparse到QSA的移植实战"
§1.1, §4.3, the many-query setting).  Same tolerances as the one-query decode."""
import numpy as np
import pytest
import torch

import oracle
from query_guided_block_gb300 import binding as B
from query_guided_block_gb300.build import build
from query_guided_block_gb300.decoder import SparseDecoder
from query_guided_block_gb300.workloads import WORKLOADS, Workload, make_inputs
from tests.parity import ATOL, as_np, check_selection, oracle_meta, sub_problem, sub_workload
from tests.test_gpu_parity import compare_every_unit

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build()
    B.lib()


def _w(**kw):
    base = dict(name="mq_case", batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128,
                n_tokens=9000, block_size=32, window_tokens=256, topk=12, planted_per_unit=4,
                num_queries=4)
    base.update(kw)
    return Workload(**base)


def run_and_compare(w, every_unit_threads=False):
    inp = make_inputs(w, "cuda")
    dec = SparseDecoder(B.params_for(w))
    dec.build_meta(inp["k_pages"], inp["block_table"])
    dec.select(inp["q"])
    dec.decode(inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"])
    assert dec.device_error() == 0
    assert tuple(dec.out.shape) == (w.batch, w.num_queries, w.num_q_heads, w.head_dim)
    if every_unit_threads:
        compare_every_unit(w, inp, dec, check=check_sequences)
    else:
        check_sequences(w, inp, dec)
    return dec


def check_sequences(w, inp, dec, seqs=None):
    """Selection and every query's attention output of sequences `seqs` (all by
    default) against the oracle.  Returns the worst attention error."""
    seqs = list(range(w.batch)) if seqs is None else list(seqs)
    host = sub_problem(w, inp, seqs)
    ws = sub_workload(w, len(seqs))
    p, (kmin, kmax, kmean) = oracle_meta(ws, host)
    rows = [s * w.num_kv_heads + h for s in seqs for h in range(w.num_kv_heads)]
    hq = host["q"]                                       # [S, Q, Hq, D]
    scores = sum(oracle.quest_scores(p, hq[:, t].contiguous(), kmin, kmax) for t in range(w.num_queries))
    oid, ocnt = oracle.select(p, scores)
    gids = as_np(dec.sel_ids).reshape(w.units, -1)[rows]
    gcnt = as_np(dec.sel_count).reshape(-1)[rows]
    check_selection(gids, gcnt, oid, ocnt, scores, w.topk, p.first_window_block())
    got = as_np(dec.out[seqs]).astype(np.float64)       # [S, Q, Hq, D]
    worst = 0.0
    for t in range(w.num_queries):
        ref = oracle.decode(p, hq[:, t].contiguous(), host["k_pages"], host["v_pages"],
                            host["block_table"], gids, gcnt)
        worst = max(worst, float(np.abs(got[:, t] - ref).max()))
    assert worst <= ATOL[w.kv_dtype], f"max abs error {worst}"
    return worst


@pytest.mark.parametrize("cfg", [
    dict(),                                                         # 16 rows: one partial tile
    dict(num_queries=16),                                           # 64 rows: one full tile
    dict(num_queries=20, block_size=64, n_tokens=20001),            # 80 rows: two tiles
    dict(num_queries=3, q_dtype=torch.float32, block_size=16),      # fp32 query (hi + lo)
    dict(num_queries=8, head_dim=64, num_q_heads=16, num_kv_heads=2, block_size=128, n_tokens=7000),
    dict(num_queries=5, n_tokens=700, topk=3, window_tokens=64),    # one tile: one split
    dict(num_queries=16, batch=1, num_kv_heads=1, num_q_heads=4, n_tokens=60000, topk=100),  # many splits
    dict(num_queries=16, n_tokens=20000, block_size=16, topk=200, window_tokens=100),       # bs 16 boxes
    dict(num_queries=12, n_tokens=30000, block_size=128, topk=20),                          # bs 128 boxes
], ids=["q4", "q16", "q20", "fp32q", "d64", "short", "splits", "bs16", "bs128"])
def test_multi_query_small(cfg):
    run_and_compare(_w(**cfg))


def test_multi_query_full_size_every_unit():
    """mq_128k (B16, 131072 tokens, 16 queries x 4 heads per KV head) in the launch
    configuration the benchmark times; every sequence checked in full."""
    w = WORKLOADS["mq_128k"]
    run_and_compare(w, every_unit_threads=True)
    torch.cuda.empty_cache()
