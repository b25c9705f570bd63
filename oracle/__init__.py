"""ctypes front end of the plain fp64 CPU oracle (``sparse_attn_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The CUDA library never imports, links or
calls anything here, and this package imports nothing from the CUDA side.

Arrays go in as numpy arrays or CPU torch tensors; bfloat16 tensors are passed as
their raw 16-bit patterns and widened exactly inside the C code.  Results come
back as numpy float64 / int32 arrays.  Every routine accepts ``units=(begin, end)``
to restrict the work to a range of (sequence, KV head) units, so that a caller
may spread independent units over threads (ctypes releases the GIL during a call).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sparse_attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, strict IEEE: no fast-math)."""
    stale = (not os.path.exists(_LIB_PATH)) or \
        os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC),
                                          os.path.getmtime(os.path.join(_HERE, "sparse_attn_oracle.h")))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Problem(C.Structure):
    _fields_ = [(n, C.c_int) for n in (
        "batch", "num_q_heads", "num_kv_heads", "head_dim", "n_tokens", "block_size",
        "num_pages", "window_tokens", "topk", "two_level", "coarse_block", "topk_coarse",
        "score_kind", "kv_bf16", "q_bf16")] + [("softmax_scale", C.c_double)]

    @property
    def num_blocks(self) -> int:
        return -(-self.n_tokens // self.block_size)

    @property
    def units(self) -> int:
        return self.batch * self.num_kv_heads

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def first_window_block(self) -> int:
        return lib().oracle_first_window_block(C.byref(self))

    def num_mean_rows(self) -> int:
        return lib().oracle_num_mean_rows(C.byref(self))

    def sel_stride(self) -> int:
        """Room per unit for the selected ids (top-k plus the window blocks)."""
        nb, wf = self.num_blocks, self.first_window_block()
        return max(1, min(self.topk, nb) + (nb - wf))


def problem(batch, num_q_heads, num_kv_heads, head_dim, n_tokens, block_size, num_pages,
            window_tokens, topk, two_level=False, coarse_block=1024, topk_coarse=48,
            score_kind="quest", kv_bf16=True, q_bf16=True, softmax_scale=0.0) -> Problem:
    kind = {"quest": 0, "mean": 1}[score_kind] if isinstance(score_kind, str) else int(score_kind)
    return Problem(batch, num_q_heads, num_kv_heads, head_dim, n_tokens, block_size, num_pages,
                   window_tokens, topk, int(bool(two_level)), coarse_block, topk_coarse, kind,
                   int(bool(kv_bf16)), int(bool(q_bf16)), float(softmax_scale))


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_LIB_PATH)
        P = C.POINTER(Problem)
        vp, ip, dp, i = C.c_void_p, C.c_void_p, C.c_void_p, C.c_int
        sig = {
            "oracle_num_blocks": [P], "oracle_first_window_block": [P],
            "oracle_mean_block": [P], "oracle_num_mean_rows": [P],
            "oracle_build_meta": [P, vp, ip, dp, dp, dp],
            "oracle_quest_scores": [P, i, i, vp, dp, dp, dp],
            "oracle_mean_scores": [P, i, i, vp, dp, i, dp],
            "oracle_select": [P, i, i, dp, ip, ip, i],
            "oracle_select_two_level": [P, i, i, vp, dp, dp, dp, dp, dp, ip, ip, ip, ip, i],
            "oracle_select_level2": [P, i, i, vp, dp, dp, ip, ip, i, dp, ip, ip, i],
            "oracle_decode": [P, i, i, vp, vp, vp, ip, ip, ip, i, dp],
            "oracle_lru_step": [i, i, i, ip, ip, i, ip, ip, i, ip, ip, ip, ip, ip, ip, ip, ip,
                                ip, i, ip],
            "oracle_union_reserve": [P, i, i, ip, ip, i, ip, i, ip, ip, i],
            "oracle_topk_for_length": [i, i],
        }
        for name, args in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = C.c_int
        _lib = L
    return _lib


# ----------------------------------------------------------------- helpers --

def host_array(x, kind: str = "auto") -> np.ndarray:
    """Contiguous numpy view of a CPU tensor / array.  bfloat16 -> its uint16 bits."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16)
            return x.numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x)


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _f32_or_bf16(a: np.ndarray, is_bf16: bool) -> np.ndarray:
    want = np.uint16 if is_bf16 else np.float32
    if a.dtype != want:
        raise TypeError(f"expected {want} storage, got {a.dtype}")
    return np.ascontiguousarray(a)


def _units(p: Problem, units: Optional[Tuple[int, int]]):
    return (0, p.units) if units is None else (int(units[0]), int(units[1]))


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (status {rc})")


# --------------------------------------------------------------- routines --

def build_meta(p: Problem, k_pages, block_table, with_mean: bool = False):
    k = _f32_or_bf16(host_array(k_pages), p.kv_bf16)
    bt = np.ascontiguousarray(host_array(block_table), dtype=np.int32)
    nb, D = p.num_blocks, p.head_dim
    kmin = np.empty((p.batch, p.num_kv_heads, nb, D), np.float64)
    kmax = np.empty_like(kmin)
    kmean = None
    if with_mean:
        kmean = np.empty((p.batch, p.num_kv_heads, p.num_mean_rows(), D), np.float64)
    _check(lib().oracle_build_meta(C.byref(p), _ptr(k), _ptr(bt), _ptr(kmin), _ptr(kmax),
                                   _ptr(kmean)), "build_meta")
    return kmin, kmax, kmean


def quest_scores(p: Problem, q, kmin, kmax, units=None) -> np.ndarray:
    qa = _f32_or_bf16(host_array(q), p.q_bf16)
    u0, u1 = _units(p, units)
    out = np.full((p.units, p.num_blocks), np.nan)
    _check(lib().oracle_quest_scores(C.byref(p), u0, u1, _ptr(qa),
                                     _ptr(np.ascontiguousarray(kmin, np.float64)),
                                     _ptr(np.ascontiguousarray(kmax, np.float64)), _ptr(out)),
           "quest_scores")
    return out


def mean_scores(p: Problem, q, kmean, units=None) -> np.ndarray:
    qa = _f32_or_bf16(host_array(q), p.q_bf16)
    u0, u1 = _units(p, units)
    rows = kmean.shape[2]
    out = np.full((p.units, rows), np.nan)
    _check(lib().oracle_mean_scores(C.byref(p), u0, u1, _ptr(qa),
                                    _ptr(np.ascontiguousarray(kmean, np.float64)), rows,
                                    _ptr(out)), "mean_scores")
    return out


def select(p: Problem, scores, units=None):
    """Single-level: top-k of ``scores`` [units, nb] over non-window blocks, plus the window."""
    u0, u1 = _units(p, units)
    stride = p.sel_stride()
    ids = np.full((p.units, stride), -1, np.int32)
    cnt = np.zeros(p.units, np.int32)
    _check(lib().oracle_select(C.byref(p), u0, u1,
                               _ptr(np.ascontiguousarray(scores, np.float64)),
                               _ptr(ids), _ptr(cnt), stride), "select")
    return ids, cnt


def select_two_level(p: Problem, q, kmin, kmax, kmean, units=None) -> dict:
    qa = _f32_or_bf16(host_array(q), p.q_bf16)
    u0, u1 = _units(p, units)
    rows, nb, stride = p.num_mean_rows(), p.num_blocks, p.sel_stride()
    r = {
        "coarse_scores": np.full((p.units, rows), np.nan),
        "slice_scores": np.full((p.units, nb), np.nan),
        "survivors": np.full((p.units, max(1, p.topk_coarse)), -1, np.int32),
        "n_survivors": np.zeros(p.units, np.int32),
        "sel_ids": np.full((p.units, stride), -1, np.int32),
        "sel_count": np.zeros(p.units, np.int32),
    }
    _check(lib().oracle_select_two_level(
        C.byref(p), u0, u1, _ptr(qa), _ptr(np.ascontiguousarray(kmin, np.float64)),
        _ptr(np.ascontiguousarray(kmax, np.float64)), _ptr(np.ascontiguousarray(kmean, np.float64)),
        _ptr(r["coarse_scores"]), _ptr(r["slice_scores"]), _ptr(r["survivors"]),
        _ptr(r["n_survivors"]), _ptr(r["sel_ids"]), _ptr(r["sel_count"]), stride),
        "select_two_level")
    return r


def select_level2(p: Problem, q, kmin, kmax, survivors, n_survivors, units=None) -> dict:
    qa = _f32_or_bf16(host_array(q), p.q_bf16)
    u0, u1 = _units(p, units)
    nb, stride = p.num_blocks, p.sel_stride()
    surv = np.ascontiguousarray(survivors, np.int32)
    r = {"slice_scores": np.full((p.units, nb), np.nan),
         "sel_ids": np.full((p.units, stride), -1, np.int32),
         "sel_count": np.zeros(p.units, np.int32)}
    _check(lib().oracle_select_level2(
        C.byref(p), u0, u1, _ptr(qa), _ptr(np.ascontiguousarray(kmin, np.float64)),
        _ptr(np.ascontiguousarray(kmax, np.float64)), _ptr(surv),
        _ptr(np.ascontiguousarray(n_survivors, np.int32)), surv.shape[1],
        _ptr(r["slice_scores"]), _ptr(r["sel_ids"]), _ptr(r["sel_count"]), stride),
        "select_level2")
    return r


def decode(p: Problem, q, k_pages, v_pages, block_table, sel_ids, sel_count, units=None,
           out: Optional[np.ndarray] = None) -> np.ndarray:
    qa = _f32_or_bf16(host_array(q), p.q_bf16)
    k = _f32_or_bf16(host_array(k_pages), p.kv_bf16)
    v = _f32_or_bf16(host_array(v_pages), p.kv_bf16)
    bt = np.ascontiguousarray(host_array(block_table), dtype=np.int32)
    ids = np.ascontiguousarray(host_array(sel_ids), dtype=np.int32)
    cnt = np.ascontiguousarray(host_array(sel_count), dtype=np.int32)
    u0, u1 = _units(p, units)
    if out is None:
        out = np.full((p.batch, p.num_q_heads, p.head_dim), np.nan)
    _check(lib().oracle_decode(C.byref(p), u0, u1, _ptr(qa), _ptr(k), _ptr(v), _ptr(bt),
                               _ptr(ids), _ptr(cnt), ids.shape[-1], _ptr(out)), "decode")
    return out


def union_reserve(p: Problem, sel_ids, sel_count, reserve, units=None):
    """Each unit's selection united with its reserve block ids [units, n_reserve]
    (SparDA page §3.4), ascending without repeats.  Returns (ids, count) with room for
    sel_stride + n_reserve ids per unit."""
    u0, u1 = _units(p, units)
    sel = np.ascontiguousarray(sel_ids, np.int32)
    res = np.ascontiguousarray(reserve, np.int32).reshape(p.units, -1)
    stride = sel.shape[1] + res.shape[1]
    ids = np.full((p.units, max(1, stride)), -1, np.int32)
    cnt = np.zeros(p.units, np.int32)
    _check(lib().oracle_union_reserve(C.byref(p), u0, u1, _ptr(sel),
                                      _ptr(np.ascontiguousarray(sel_count, np.int32)), sel.shape[1],
                                      _ptr(res), res.shape[1], _ptr(ids), _ptr(cnt), ids.shape[1]),
           "union_reserve")
    return ids, cnt


def topk_for_length(n_tokens: int, block_size: int) -> int:
    """k from the context length (SparDA page §3.2)."""
    k = lib().oracle_topk_for_length(int(n_tokens), int(block_size))
    if k < 0:
        raise ValueError("oracle_topk_for_length: bad argument")
    return k


def lru_step(step: int, cache_slots: int, cur_ids, cur_count, prev_ids, prev_count,
             slot_block: np.ndarray, slot_last_use: np.ndarray) -> dict:
    """One diff + LRU step; ``slot_block`` / ``slot_last_use`` [units, slots] update in place."""
    cur = np.ascontiguousarray(host_array(cur_ids), np.int32)
    cc = np.ascontiguousarray(host_array(cur_count), np.int32)
    prev = np.ascontiguousarray(host_array(prev_ids), np.int32)
    pc = np.ascontiguousarray(host_array(prev_count), np.int32)
    n_units = cur.shape[0]
    assert slot_block.dtype == np.int32 and slot_block.flags.c_contiguous
    assert slot_last_use.dtype == np.int32 and slot_last_use.flags.c_contiguous
    w = max(cur.shape[1], prev.shape[1])
    r = {k: np.full((n_units, w), -1, np.int32) for k in
         ("hit_ids", "miss_ids", "miss_slot", "evict_ids", "evict_slot", "new_ids", "dropped_ids")}
    r["counts"] = np.zeros((n_units, 5), np.int32)
    _check(lib().oracle_lru_step(
        n_units, step, cache_slots, _ptr(cur), _ptr(cc), cur.shape[1], _ptr(prev), _ptr(pc),
        prev.shape[1], _ptr(slot_block), _ptr(slot_last_use), _ptr(r["hit_ids"]),
        _ptr(r["miss_ids"]), _ptr(r["miss_slot"]), _ptr(r["evict_ids"]), _ptr(r["evict_slot"]),
        _ptr(r["new_ids"]), _ptr(r["dropped_ids"]), w, _ptr(r["counts"])), "lru_step")
    return r
