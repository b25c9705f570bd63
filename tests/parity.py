"""Helpers for comparing the CUDA path with the fp64 oracle (test code only)."""
from __future__ import annotations

import itertools

import numpy as np
import torch

import oracle
from query_guided_block_gb300.workloads import gather_sequences
from tests.conftest import oracle_problem_for

NEAR_TIE_REL = 1e-5      # selection swaps allowed within this relative band of the k-th score
ATOL = {torch.bfloat16: 2e-3, torch.float32: 1e-5}


def sub_problem(w, inp, seqs):
    """Host copies of the sequences `seqs` with their pages in a private pool."""
    return gather_sequences(inp, seqs, "cpu")


def sub_workload(w, n_seqs):
    import dataclasses
    return dataclasses.replace(w, batch=n_seqs)


def oracle_meta(w, host):
    p = oracle_problem_for(w, num_pages=host["k_pages"].shape[0])
    need_mean = w.two_level or w.score == "mean"
    return p, oracle.build_meta(p, host["k_pages"], host["block_table"], with_mean=need_mean)


def check_selection(gpu_ids, gpu_cnt, ora_ids, ora_cnt, scores, k, win_first, units=None,
                    rel=NEAR_TIE_REL):
    """GPU and oracle selections agree up to swaps among candidates whose oracle scores lie
    within `rel` of the k-th selected candidate score.  Returns the number of waived units."""
    gpu_ids = np.asarray(gpu_ids)
    gpu_cnt = np.asarray(gpu_cnt).reshape(-1)
    waived = 0
    for u in (range(len(ora_cnt)) if units is None else units):
        g = set(int(x) for x in gpu_ids[u, : gpu_cnt[u]])
        o = set(int(x) for x in ora_ids[u, : ora_cnt[u]])
        assert gpu_cnt[u] == ora_cnt[u], f"unit {u}: count {gpu_cnt[u]} != {ora_cnt[u]}"
        assert list(gpu_ids[u, : gpu_cnt[u]]) == sorted(g), f"unit {u}: ids not ascending"
        if g == o:
            continue
        chosen = [j for j in o if j < win_first]
        kth = min(scores[u, j] for j in chosen)
        for j in g ^ o:
            assert j < win_first, f"unit {u}: window block {j} differs"
            assert abs(scores[u, j] - kth) <= rel * abs(kth), \
                f"unit {u}: block {j} score {scores[u, j]} vs k-th {kth} is not a near tie"
        waived += 1
    return waived


def check_two_level(w, p, host_q, kmin, kmax, kmean, gpu_ids, gpu_cnt, units, rel=NEAR_TIE_REL,
                    reserve=None):
    """Two-level selection: level-1 survivors are unique unless coarse scores tie within
    `rel` of the K1-th; every admissible survivor set is tried, and level 2 is compared
    with the near-tie waiver."""
    r = oracle.select_two_level(p, host_q, kmin, kmax, kmean)
    cs = r["coarse_scores"]
    K1 = p.topk_coarse
    for u in units:
        sc = cs[u]
        order = sorted(range(len(sc)), key=lambda c: (-sc[c], c))
        k1 = min(K1, len(sc))
        base_sets = [sorted(order[:k1])]
        if 0 < k1 < len(sc):
            kth = sc[order[k1 - 1]]
            band = [c for c in range(len(sc)) if abs(sc[c] - kth) <= rel * abs(kth)]
            sure = [c for c in order[:k1] if c not in band]
            need = k1 - len(sure)
            if len(band) > 1:
                base_sets = [sorted(sure + list(comb)) for comb in itertools.combinations(band, need)]
        ok, last_err = False, None
        for surv in base_sets:
            sv = np.full((p.units, max(1, K1)), -1, np.int32)
            ns = np.zeros(p.units, np.int32)
            sv[u, : len(surv)] = surv
            ns[u] = len(surv)
            r2 = oracle.select_level2(p, host_q, kmin, kmax, sv, ns, units=(u, u + 1))
            if reserve is not None:   # the reserve set joins the level-2 result
                r2["sel_ids"], r2["sel_count"] = oracle.union_reserve(
                    p, r2["sel_ids"], r2["sel_count"], reserve, units=(u, u + 1))
            try:
                check_selection(gpu_ids, gpu_cnt, r2["sel_ids"], r2["sel_count"],
                                np.nan_to_num(r2["slice_scores"], nan=-np.inf), p.topk,
                                p.first_window_block(), units=[u], rel=rel)
                ok = True
                break
            except AssertionError as e:
                last_err = e
        assert ok, f"unit {u}: {last_err}"


U32 = 2.0 ** -24          # unit roundoff of IEEE binary32 (round to nearest)


def _gamma(m):
    """gamma_m = m u / (1 - m u): the classical bound on the relative error of m
    chained fp32 roundings (Higham, Accuracy and Stability of Numerical Algorithms,
    ch. 3)."""
    m = np.asarray(m, np.float64)
    return m * U32 / (1.0 - m * U32)


def abs_row_sums(host, w, mean_block):
    """Per (sequence, KV head, mean row, channel): the number of tokens n_r of the row
    and sum_t |k_t,d| over them, from the host keys of a gathered instance (pages in
    logical order).  Returned as float64 arrays [S, Hkv, rows, D] and [rows]."""
    bt = host["block_table"]
    S, nb = bt.shape
    Hkv, bs, D, N = w.num_kv_heads, w.block_size, w.head_dim, w.n_tokens
    rows = -(-N // mean_block)
    out = np.empty((S, Hkv, rows, D), np.float64)
    for s in range(S):   # one sequence at a time keeps the temporaries small
        k = host["k_pages"][s * nb:(s + 1) * nb].float().abs()          # [nb, Hkv, bs, D]
        k = k.permute(1, 0, 2, 3).reshape(Hkv, nb * bs, D)[:, :N]
        pad = rows * mean_block - N
        if pad:
            k = torch.cat([k, k.new_zeros(Hkv, pad, D)], 1)
        out[s] = k.view(Hkv, rows, mean_block, D).double().sum(2).numpy()
    n = np.minimum(mean_block, N - np.arange(rows) * mean_block).astype(np.float64)
    return out, n


def check_means(gpu_mean, ora_mean, host, w, mean_block):
    """Block means from fp32 accumulation against the fp64 oracle, within the bound
    that fp32 arithmetic guarantees.  The kernel forms s = fl(sum_t k_t) over the n
    tokens of a row in some order of n - 1 additions, then fl(s * fl(1/n)).  Whatever
    the summation tree, each key passes through at most n - 1 roundings, so
    |s - S| <= gamma_{n-1} sum_t |k_t| (Higham, ch. 4), and the
    reciprocal and the product add one rounding each, so
        |mean_gpu - S/n| <= (1+u)^2 gamma_{n-1} sum|k| / n + (2u + u^2) |S/n|.
    The bound is taken from the actual keys of each row and channel (x 1.001 for the
    fp64 evaluation of the bound itself).  For N(0,1) keys and n = 1024 it is about
    5e-5 per element, against the 1e-4 that a fixed tolerance allowed."""
    sabs, n = abs_row_sums(host, w, mean_block)
    ora = np.asarray(ora_mean, np.float64)
    gpu = np.asarray(gpu_mean, np.float64)[:, :, : ora.shape[2]]
    tol = ((1 + U32) ** 2 * _gamma(n - 1)[None, None, :, None] * sabs / n[None, None, :, None]
           + (2 * U32 + U32 * U32) * np.abs(ora)) * 1.001
    err = np.abs(gpu - ora)
    bad = err > tol
    assert not bad.any(), (f"{int(bad.sum())} block means outside the fp32 bound; worst excess "
                           f"{float((err - tol).max()):.3e} at {np.unravel_index(np.argmax(err - tol), err.shape)}")
    return float(err.max())


def as_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def bf16_bits_to_f64(t: torch.Tensor) -> np.ndarray:
    x = t.detach().cpu()
    if x.dtype == torch.bfloat16:
        x = x.float()
    return x.double().numpy()
