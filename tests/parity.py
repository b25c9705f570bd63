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


def as_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def bf16_bits_to_f64(t: torch.Tensor) -> np.ndarray:
    x = t.detach().cpu()
    if x.dtype == torch.bfloat16:
        x = x.float()
    return x.double().numpy()
