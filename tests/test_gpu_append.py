"""Incremental metadata (SGLang page §2.2 / §3.1.1: keep the block representation
current as the context grows instead of rebuilding it): after each append, the rows of
sparse_attn_append_meta equal a fresh sparse_attn_build_meta bit for bit and the oracle
(exact box; means within the fp32 summation bound of tests.parity.check_means); select / decode read the capacity-strided metadata correctly."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from query_guided_block_gb300 import binding as B
from query_guided_block_gb300.build import build
from query_guided_block_gb300.decoder import SparseDecoder
from query_guided_block_gb300.workloads import Workload, make_inputs
from tests.parity import (ATOL, as_np, bf16_bits_to_f64, check_means, check_selection, oracle_meta, sub_problem,
                          sub_workload)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build()
    B.lib()


def _w(**kw):
    base = dict(name="append_case", batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128,
                n_tokens=20000, block_size=32, window_tokens=300, topk=10, planted_per_unit=5)
    base.update(kw)
    return Workload(**base)


def _meta(p, dev):
    rb, rm = B.meta_rows(p)
    kv = torch.bfloat16 if p.kv_dtype == B.BF16 else torch.float32
    kmin = torch.zeros(p.batch, p.num_kv_heads, rb, p.head_dim, dtype=kv, device=dev)
    kmax = torch.zeros_like(kmin)
    need_mean = bool(p.two_level) or p.score_kind == B.SCORE_MEAN
    kmean = torch.zeros(p.batch, p.num_kv_heads, rm, p.head_dim, dtype=torch.float32, device=dev) if need_mean else None
    return kmin, kmax, kmean


@pytest.mark.parametrize("cfg", [
    dict(),
    dict(score="mean", block_size=64, n_tokens=15000),
    dict(two_level=True, block_size=64, n_tokens=40000, coarse_block=1024, topk_coarse=5, topk=8),
], ids=["quest", "mean", "two_level"])
def test_append_matches_rebuild_and_oracle(cfg):
    w = _w(**cfg)
    dev = "cuda"
    base = make_inputs(w, dev)                        # pages for the whole final context
    inp = base
    cap = w.n_tokens + 3000                           # rows strided by a capacity > nb
    lengths = [w.n_tokens // 3 + 7, w.n_tokens // 3 + 8, w.n_tokens // 3 + 40,
               w.n_tokens // 2 + 1111, w.n_tokens - 1, w.n_tokens]
    p_of = lambda n: B.params_for(w, n_tokens=n, capacity_tokens=cap)
    # the page table is allocated for the capacity too: [B, ceil(capacity / block_size)]
    nb_cap, _ = B.meta_rows(p_of(w.n_tokens))
    bt = torch.zeros(w.batch, nb_cap, dtype=torch.int32, device=dev)
    bt[:, : inp["block_table"].shape[1]] = inp["block_table"]
    inp = dict(inp, block_table=bt)
    ws = torch.empty(B.sparse_attn_workspace_size(p_of(w.n_tokens)), dtype=torch.uint8, device=dev)
    B.sparse_attn_workspace_init(ws)
    kmin, kmax, kmean = _meta(p_of(w.n_tokens), dev)
    B.sparse_attn_build_meta(p_of(lengths[0]), inp["k_pages"], inp["block_table"], kmin, kmax, kmean, ws)
    prev = lengths[0]
    for n in lengths[1:]:
        try:
            B.sparse_attn_append_meta(p_of(n), prev, inp["k_pages"], inp["block_table"], kmin, kmax, kmean, ws)
        except B.SparseAttnError as e:
            raise AssertionError(f"append {prev} -> {n}: {e}")
        prev = n
        rmin, rmax, rmean = _meta(p_of(n), dev)
        B.sparse_attn_build_meta(p_of(n), inp["k_pages"], inp["block_table"], rmin, rmax, rmean, ws)
        torch.cuda.synchronize()
        assert B.sparse_attn_get_device_error(ws) == 0
        nb = -(-n // w.block_size)
        assert torch.equal(kmin[:, :, :nb], rmin[:, :, :nb]) and torch.equal(kmax[:, :, :nb], rmax[:, :, :nb])
        if kmean is not None:
            mb = w.coarse_block if w.two_level else w.block_size
            nm = -(-n // mb)
            assert torch.equal(kmean[:, :, :nm], rmean[:, :, :nm])
        # the oracle at this length (first sequence)
        wn = dataclasses.replace(w, n_tokens=n)
        host = sub_problem(wn, base, [0])
        po, (omin, omax, omean) = oracle_meta(sub_workload(wn, 1), host)
        assert np.array_equal(bf16_bits_to_f64(kmin[[0], :, :nb]), omin)
        assert np.array_equal(bf16_bits_to_f64(kmax[[0], :, :nb]), omax)
        if omean is not None:
            check_means(as_np(kmean[[0]]), omean, host, sub_workload(wn, 1), mb)

    # select + decode at the final length through the capacity-strided metadata
    dec = SparseDecoder(p_of(w.n_tokens))
    dec.kmin.copy_(kmin)
    dec.kmax.copy_(kmax)
    if kmean is not None:
        dec.kmean.copy_(kmean)
    dec.select(inp["q"])
    dec.decode(inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"])
    assert dec.device_error() == 0
    host = sub_problem(w, base, [0, 1])
    ws2 = sub_workload(w, 2)
    po, (omin, omax, omean) = oracle_meta(ws2, host)
    gids = as_np(dec.sel_ids).reshape(w.units, -1)
    gcnt = as_np(dec.sel_count).reshape(-1)
    if w.two_level:
        from tests.parity import check_two_level
        check_two_level(ws2, po, host["q"], omin, omax, omean, gids, gcnt, units=range(ws2.units))
    else:
        scores = (oracle.mean_scores(po, host["q"], omean) if w.score == "mean"
                  else oracle.quest_scores(po, host["q"], omin, omax))
        oid, ocnt = oracle.select(po, scores)
        check_selection(gids, gcnt, oid, ocnt, scores, w.topk, po.first_window_block())
    ref = oracle.decode(po, host["q"], host["k_pages"], host["v_pages"], host["block_table"], gids, gcnt)
    assert np.abs(as_np(dec.out).astype(np.float64) - ref).max() <= ATOL[w.kv_dtype]
