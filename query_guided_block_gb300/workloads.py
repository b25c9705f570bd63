"""Seeded synthetic workloads for query-guided block-sparse decode attention.

This module only draws random inputs; it holds none of the method's arithmetic
(no scoring, selection, softmax or cache logic).  Both the CUDA path's tests and
the CPU oracle's tests take their inputs from here, so the two sides always read
the same bytes.

Workload shapes follow the decode settings the pages describe:

* paged KV in 64-token blocks with a page table -- SparDA page
  (www.2kiu.com/news/4656707), §2.3 and §3.3;
* a 512-token local window and 1024-token coarse blocks with 64-token slices --
  "从HiSparse到QSA的移植实战" (xxmr.cn/news/247609), §2.2 and §3.1;
* 32-token Quest blocks -- "SGLang分层稀疏注意力技术解析与优化实践", §3.1.2;
* adjacent decode steps whose top-k sets overlap heavily -- same SGLang page, §3.2.

"Planted" blocks stand in for the relevant context a real query would find: every
key of a planted block is ``0.5 * u * sqrt(D) + N(0, 1)`` where ``u`` is the unit
direction of the query (of the sum of the group's queries under GQA).  No public
dataset is reproduced; these inputs replace the pages' long-context suites.

Random streams: each tensor gets its own ``torch.Generator`` seeded from
``(seed, workload name, tensor name)``, so adding a tensor never shifts another.
The stream depends on the device the tensors are drawn on (CPU and CUDA Philox
differ); a test draws once and hands the same bytes to both sides.
"""
from __future__ import annotations

import dataclasses
import math
import zlib
from typing import Dict, Optional

import torch

__all__ = ["Workload", "WORKLOADS", "make_inputs", "derive_seed", "scaled", "gather_sequences"]


@dataclasses.dataclass(frozen=True)
class Workload:
    """One decode-attention problem.  Token counts are per sequence."""

    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    n_tokens: int
    block_size: int
    window_tokens: int
    topk: int
    kv_dtype: torch.dtype = torch.bfloat16
    q_dtype: torch.dtype = torch.bfloat16
    score: str = "quest"             # "quest" (min/max bound) or "mean"
    two_level: bool = False
    coarse_block: int = 1024
    topk_coarse: int = 48
    planted_per_unit: int = 0        # planted blocks per (sequence, KV head)
    planted_scale: float = 0.5       # planted key = scale * u * sqrt(D) + N(0,1)
    steps: int = 1                   # consecutive decode steps (query drift)
    q_drift: float = 0.15            # q_t = normalise(q_{t-1} + drift*N(0,I)) * |q_0|
    cache_slots: int = 0             # LRU slots per (sequence, KV head); 0 = no diff
    num_reserve: int = 0             # random reserve blocks per (sequence, KV head)
    num_queries: int = 1             # query vectors per sequence sharing one selection
    seed: int = 0
    description: str = ""

    # ---- derived sizes -------------------------------------------------
    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def num_blocks(self) -> int:
        return -(-self.n_tokens // self.block_size)

    @property
    def num_pages(self) -> int:
        return self.batch * self.num_blocks

    @property
    def units(self) -> int:
        return self.batch * self.num_kv_heads


def _w(**kw) -> Workload:
    return Workload(**kw)


#: The five workloads: a tiny CPU-checkable case and four GB300-sized ones.
WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        _w(name="tiny_fp32_4k", batch=1, num_q_heads=4, num_kv_heads=4, head_dim=64,
           n_tokens=4096, block_size=64, window_tokens=128, topk=8,
           kv_dtype=torch.float32, q_dtype=torch.float32,
           description="B1 H4/4 D64 N4096 bs64 fp32, Quest, k=8 + last 2 blocks"),
        _w(name="mha_32k", batch=8, num_q_heads=32, num_kv_heads=32, head_dim=128,
           n_tokens=32768, block_size=64, window_tokens=512, topk=32,
           planted_per_unit=16,
           description="B8 H32/32 D128 N32768 bs64 bf16, Quest, k=32 + 512 window, 16 planted"),
        _w(name="gqa_128k", batch=16, num_q_heads=32, num_kv_heads=8, head_dim=128,
           n_tokens=131072, block_size=32, window_tokens=512, topk=64,
           planted_per_unit=41,
           description="B16 H32/8 D128 N131072 bs32 bf16, group-summed Quest, k=64 + 512 window, 1% planted"),
        _w(name="two_level_256k", batch=8, num_q_heads=32, num_kv_heads=8, head_dim=128,
           n_tokens=262144, block_size=64, window_tokens=512, topk=48,
           two_level=True, coarse_block=1024, topk_coarse=48, planted_per_unit=82,
           description="B8 H32/8 D128 N262144 bs64 bf16, L1 mean top-48 of 256x1024, "
                       "L2 Quest top-48 slices + 512 window, 2% planted"),
        _w(name="reserve_128k", batch=16, num_q_heads=32, num_kv_heads=8, head_dim=128,
           n_tokens=131072, block_size=32, window_tokens=512, topk=64,
           planted_per_unit=41, num_reserve=41,
           description="gqa_128k plus a 1% random reserve set (41 blocks) per KV head"),
        _w(name="mq_128k", batch=16, num_q_heads=32, num_kv_heads=8, head_dim=128,
           n_tokens=131072, block_size=32, window_tokens=512, topk=64,
           planted_per_unit=41, num_queries=16,
           description="gqa_128k with 16 queries per sequence sharing each KV head's selection"),
        _w(name="lru_64k", batch=32, num_q_heads=32, num_kv_heads=8, head_dim=128,
           n_tokens=65536, block_size=64, window_tokens=512, topk=32,
           steps=64, q_drift=0.15, cache_slots=128,
           description="B32 H32/8 D128 N65536 bs64 bf16, k=32 + 512 window, 64 drifting "
                       "steps, 128-slot LRU per KV head"),
    ]
}


def scaled(w: Workload, **overrides) -> Workload:
    """A copy of ``w`` with some fields replaced (smaller test variants)."""
    if "name" not in overrides:
        overrides["name"] = w.name + "_scaled"
    return dataclasses.replace(w, **overrides)


def derive_seed(seed: int, workload: str, tensor: str) -> int:
    return zlib.crc32(f"{seed}/{workload}/{tensor}".encode()) & 0x7FFFFFFF


def _gen(w: Workload, tensor: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(derive_seed(w.seed, w.name, tensor))
    return g


def _randn_into(dst: torch.Tensor, g: torch.Generator, chunk: int = 1 << 26) -> None:
    """Fill ``dst`` with N(0,1) drawn in fp32 and rounded to dst's dtype, in chunks."""
    flat = dst.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        flat[s:e].copy_(torch.randn(e - s, generator=g, device=dst.device, dtype=torch.float32))


def make_inputs(w: Workload, device="cpu", planted_blocks: Optional[torch.Tensor] = None) -> dict:
    """Draw one problem instance.

    Returns a dict of tensors on ``device``:

    * ``q``            [B, Hq, D] (``steps == 1``), [steps, B, Hq, D], or [B, Q, Hq, D] when
                       ``num_queries`` Q > 1 (then ``queries_per_seq`` = Q); dtype ``q_dtype``
    * ``k_pages``, ``v_pages``  [num_pages, Hkv, block_size, D]; dtype ``kv_dtype``
    * ``block_table``  [B, num_blocks] int32, a seeded permutation of the page pool
    * ``planted``      [B, Hkv, P] int64 logical block ids of planted blocks (P may be 0)
    * ``reserve_ids``  [B, Hkv, num_reserve] int32 random blocks (only when num_reserve > 0):
                       the first num_reserve of a seeded permutation of all nb blocks
    """
    device = torch.device(device)
    B, Hq, Hkv, D = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
    nb, bs = w.num_blocks, w.block_size

    # --- queries first (planted keys point along them) -------------------
    gq = _gen(w, "q", device)
    Qn = max(1, w.num_queries)
    q0 = torch.randn(B, Hq, D, generator=gq, device=device, dtype=torch.float32)
    if Qn > 1:
        if w.steps > 1:
            raise ValueError("num_queries > 1 with several steps is not a workload here")
        # queries 1.. of a sequence lie near query 0 (nearby positions of one chunk)
        rest = q0.unsqueeze(1) + 0.3 * torch.randn(B, Qn - 1, Hq, D, generator=gq, device=device,
                                                   dtype=torch.float32)
        q_f32 = torch.cat([q0.unsqueeze(1), rest], 1)          # [B, Q, Hq, D]
    elif w.steps > 1:
        qs = [q0]
        norm0 = q0.norm(dim=-1, keepdim=True)
        for _ in range(1, w.steps):
            prev = qs[-1]
            nxt = prev + w.q_drift * torch.randn(B, Hq, D, generator=gq, device=device,
                                                 dtype=torch.float32)
            qs.append(nxt / nxt.norm(dim=-1, keepdim=True) * norm0)
        q_f32 = torch.stack(qs, 0)
    else:
        q_f32 = q0
    q = q_f32.to(w.q_dtype)

    # --- page table: logical block (b, j) -> physical page ----------------
    gt = _gen(w, "block_table", device)
    perm = torch.randperm(w.num_pages, generator=gt, device=device)
    block_table = perm.view(B, nb).to(torch.int32)

    # --- K / V page pools ----------------------------------------------
    k_pages = torch.empty(w.num_pages, Hkv, bs, D, dtype=w.kv_dtype, device=device)
    v_pages = torch.empty_like(k_pages)
    _randn_into(k_pages, _gen(w, "k", device))
    _randn_into(v_pages, _gen(w, "v", device))

    # --- planted relevant blocks ----------------------------------------
    P = w.planted_per_unit
    if planted_blocks is not None:
        planted = planted_blocks.to(device=device, dtype=torch.int64)
        P = planted.shape[-1]
    elif P > 0:
        # distinct positions outside the local window
        first_window_block = (max(0, w.n_tokens - w.window_tokens) // bs
                              if w.window_tokens > 0 else nb)
        n_cand = first_window_block
        if P > n_cand:
            raise ValueError(f"{P} planted blocks do not fit in {n_cand} non-window blocks")
        gp = _gen(w, "planted", device)
        keys = torch.rand(B * Hkv, n_cand, generator=gp, device=device)
        planted = keys.argsort(dim=1)[:, :P].sort(dim=1).values.view(B, Hkv, P)
    else:
        planted = torch.zeros(B, Hkv, 0, dtype=torch.int64, device=device)

    if P > 0:
        q_first = q_f32[0] if w.steps > 1 else (q_f32[:, 0] if Qn > 1 else q_f32)   # [B, Hq, D]
        direction = q_first.view(B, Hkv, w.group, D).sum(dim=2)
        direction = direction / direction.norm(dim=-1, keepdim=True)   # [B, Hkv, D]
        shift = (w.planted_scale * math.sqrt(D)) * direction
        gn = _gen(w, "planted_noise", device)
        b_idx = torch.arange(B, device=device).view(B, 1, 1).expand(B, Hkv, P)
        h_idx = torch.arange(Hkv, device=device).view(1, Hkv, 1).expand(B, Hkv, P)
        pages = block_table.to(torch.int64)[b_idx, planted]            # [B, Hkv, P]
        noise = torch.randn(B, Hkv, P, bs, D, generator=gn, device=device, dtype=torch.float32)
        vals = noise + shift.view(B, Hkv, 1, 1, D)
        k_pages[pages.reshape(-1), h_idx.reshape(-1)] = vals.reshape(-1, bs, D).to(w.kv_dtype)

    out = {"q": q, "k_pages": k_pages, "v_pages": v_pages,
           "block_table": block_table, "planted": planted}
    if Qn > 1:
        out["queries_per_seq"] = Qn
    if w.num_reserve > 0:
        gr = _gen(w, "reserve", device)
        keys = torch.rand(B * Hkv, nb, generator=gr, device=device)
        out["reserve_ids"] = keys.argsort(dim=1)[:, :w.num_reserve].to(torch.int32).view(B, Hkv, -1)
    return out


def gather_sequences(inp: dict, seqs, device="cpu") -> dict:
    """The sequences ``seqs`` of a drawn instance with their pages copied into a private
    pool in logical order (page table = identity), on ``device``.  Pure data movement:
    used to hand a sample of a large instance to a host-side checker."""
    seqs = list(seqs)
    bt = inp["block_table"][seqs].long()
    pages = bt.reshape(-1)
    q = inp["q"]
    q = q[seqs] if inp.get("queries_per_seq", 1) > 1 or q.dim() == 3 else q[:, seqs]
    extra = {}
    if "queries_per_seq" in inp:
        extra["queries_per_seq"] = inp["queries_per_seq"]
    if "reserve_ids" in inp:
        extra["reserve_ids"] = inp["reserve_ids"][seqs].to(device)
    return {**extra, "k_pages": inp["k_pages"][pages].to(device),
            "v_pages": inp["v_pages"][pages].to(device),
            "block_table": torch.arange(pages.numel(), dtype=torch.int32,
                                        device=device).view(len(seqs), -1),
            "q": q.to(device)}
