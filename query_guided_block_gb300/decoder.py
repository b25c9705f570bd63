"""Device-buffer plumbing around the C ABI: allocates, with torch, the tensors one
decode problem needs and calls the entry points in order.  No arithmetic of the method
happens here."""
from __future__ import annotations

from typing import Optional

import torch

from . import binding as B


class SparseDecoder:
    """Owns metadata, selection, output and workspace buffers for one problem.

    The KV page pools, block table and queries belong to the caller.
    """

    def __init__(self, params: B.sparse_attn_params, device="cuda"):
        self.p = params
        self.device = torch.device(device)
        p = params
        self.nb = B.sparse_attn_num_blocks(p)
        self.sel_stride = B.sparse_attn_sel_stride(p)
        self.units = p.batch * p.num_kv_heads
        kv = torch.bfloat16 if p.kv_dtype == B.BF16 else torch.float32
        self.kv_dtype = kv
        dev = self.device
        rows_blk, rows_mean = B.meta_rows(p)             # capacity, >= the context's rows
        self.kmin = torch.empty(p.batch, p.num_kv_heads, rows_blk, p.head_dim, dtype=kv, device=dev)
        self.kmax = torch.empty_like(self.kmin)
        self.needs_mean = bool(p.two_level) or p.score_kind == B.SCORE_MEAN
        self.kmean = None
        if self.needs_mean:
            self.kmean = torch.empty(p.batch, p.num_kv_heads, rows_mean, p.head_dim, dtype=torch.float32,
                                     device=dev)
        self.ws_bytes = B.sparse_attn_workspace_size(p)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        B.sparse_attn_workspace_init(self.ws)
        self.sel_ids = torch.empty(p.batch, p.num_kv_heads, self.sel_stride, dtype=torch.int32,
                                   device=dev)
        self.sel_count = torch.empty(p.batch, p.num_kv_heads, dtype=torch.int32, device=dev)
        self.Q = max(1, p.num_queries)
        out_shape = ((p.batch, self.Q, p.num_q_heads, p.head_dim) if self.Q > 1
                     else (p.batch, p.num_q_heads, p.head_dim))
        self.out = torch.empty(out_shape, dtype=torch.float32, device=dev)

    def metadata_bytes(self) -> int:
        n = self.kmin.numel() * self.kmin.element_size() * 2
        if self.kmean is not None:
            n += self.kmean.numel() * 4
        return n

    def build_meta(self, k_pages, block_table, stream=None):
        B.sparse_attn_build_meta(self.p, k_pages, block_table, self.kmin, self.kmax, self.kmean,
                                 self.ws, stream)

    def append_meta(self, n_old, k_pages, block_table, stream=None):
        """Metadata after tokens [n_old, p.n_tokens) were appended to the pages."""
        B.sparse_attn_append_meta(self.p, n_old, k_pages, block_table, self.kmin, self.kmax,
                                  self.kmean, self.ws, stream)

    def select(self, q, reserve_ids=None, stream=None):
        """Selection; with ``reserve_ids`` [B, Hkv, num_reserve] int32 (drawn by the caller)
        the reserve set is united with every unit's top-k."""
        if self.p.num_reserve > 0:
            if reserve_ids is None:
                raise ValueError("this problem has num_reserve > 0: pass reserve_ids")
            B.sparse_attn_select_reserved(self.p, q, self.kmin, self.kmax, self.kmean, reserve_ids,
                                          self.sel_ids, self.sel_count, self.ws, stream)
            return
        B.sparse_attn_select(self.p, q, self.kmin, self.kmax, self.kmean, self.sel_ids,
                             self.sel_count, self.ws, stream)

    def decode(self, q, k_pages, v_pages, block_table, sel_ids=None, sel_count=None, out=None,
               stream=None):
        B.sparse_attn_decode(self.p, q, k_pages, v_pages, block_table,
                             self.sel_ids if sel_ids is None else sel_ids,
                             self.sel_count if sel_count is None else sel_count,
                             self.out if out is None else out, self.ws, stream)

    def step(self, q, k_pages, v_pages, block_table, reserve_ids=None, stream=None):
        """select + decode for one query batch (two launches); returns the output tensor."""
        self.select(q, reserve_ids, stream)
        self.decode(q, k_pages, v_pages, block_table, stream=stream)
        return self.out

    def step_fused(self, q, k_pages, v_pages, block_table, reserve_ids=None, stream=None):
        """select + decode for one query batch in one launch (sparse_attn_step); the same
        results as ``step``.  Raises SparseAttnError (unsupported) for two-level
        selection, fp32 K/V or several queries per sequence."""
        if self.p.num_reserve > 0 and reserve_ids is None:
            raise ValueError("this problem has num_reserve > 0: pass reserve_ids")
        B.sparse_attn_step(self.p, q, self.kmin, self.kmax, self.kmean, reserve_ids, k_pages, v_pages,
                           block_table, self.sel_ids, self.sel_count, self.out, self.ws, stream)
        return self.out

    def device_error(self, stream=None) -> int:
        return B.sparse_attn_get_device_error(self.ws, stream)

    def set_wait_limit(self, cycles: int, stream=None):
        """Bounded-wait limit of this decoder's kernels (SM clocks; 0 = the default)."""
        B.sparse_attn_workspace_set_wait_limit(self.ws, cycles, stream)


class SlotCache:
    """LRU slot-cache state and per-step diff outputs for ``sparse_attn_diff``."""

    def __init__(self, decoder: SparseDecoder, cache_slots: int):
        d = decoder
        dev = d.device
        u, w = d.units, d.sel_stride
        self.decoder = d
        self.cache_slots = cache_slots
        self.slot_block = torch.full((u, cache_slots), -1, dtype=torch.int32, device=dev)
        self.slot_last_use = torch.full((u, cache_slots), -1, dtype=torch.int32, device=dev)
        self.prev_ids = torch.full((u, w), -1, dtype=torch.int32, device=dev)
        self.prev_count = torch.zeros(u, dtype=torch.int32, device=dev)
        names = ("hit_ids", "miss_ids", "miss_slot", "evict_ids", "evict_slot", "new_ids",
                 "dropped_ids")
        self.lists = {n: torch.full((u, w), -1, dtype=torch.int32, device=dev) for n in names}
        self.counts = torch.zeros(u, 5, dtype=torch.int32, device=dev)

    def diff(self, step: int, sel_ids: Optional[torch.Tensor] = None,
             sel_count: Optional[torch.Tensor] = None, stream=None, sel_slot: Optional[torch.Tensor] = None):
        """The step's diff; with `sel_slot` also its slot map, in the same launch."""
        d = self.decoder
        ids = d.sel_ids if sel_ids is None else sel_ids
        cnt = d.sel_count if sel_count is None else sel_count
        L = self.lists
        args = (d.p, step, ids, cnt, self.prev_ids, self.prev_count, self.cache_slots,
                self.slot_block, self.slot_last_use, L["hit_ids"], L["miss_ids"],
                L["miss_slot"], L["evict_ids"], L["evict_slot"], L["new_ids"],
                L["dropped_ids"], self.counts)
        if sel_slot is None:
            B.sparse_attn_diff(*args, d.ws, stream)
        else:
            B.sparse_attn_diff_slots(*args, sel_slot, d.ws, stream)

    def advance(self, sel_ids: Optional[torch.Tensor] = None,
                sel_count: Optional[torch.Tensor] = None):
        """Remember this step's request set as the next step's previous set."""
        d = self.decoder
        self.prev_ids.copy_((d.sel_ids if sel_ids is None else sel_ids).view(self.prev_ids.shape))
        self.prev_count.copy_((d.sel_count if sel_count is None else sel_count).view(-1))


class SlotPool:
    """Per-unit slot pool of K/V page tiles fed from a host-resident page-first store:
    after the diff of a step, ``load_misses`` brings the misses in (one launch),
    ``slot_map`` finds each selected block's slot and ``decode`` attends through it;
    ``decode_io`` does the miss loads and the attention in one pass (after
    ``slot_map``), so that the transfer overlaps the attention over resident blocks."""

    def __init__(self, cache: SlotCache):
        d = cache.decoder
        p = d.p
        self.cache = cache
        shape = (d.units, cache.cache_slots, p.block_size, p.head_dim)
        self.pool_k = torch.zeros(shape, dtype=d.kv_dtype, device=d.device)
        self.pool_v = torch.zeros_like(self.pool_k)
        self.sel_slot = torch.full((d.units, d.sel_stride), -1, dtype=torch.int32, device=d.device)

    def tile_bytes(self) -> int:
        p = self.cache.decoder.p
        return p.block_size * p.head_dim * self.pool_k.element_size()

    def load_misses(self, host_k_pages, host_v_pages, block_table, stream=None):
        c, d = self.cache, self.cache.decoder
        B.sparse_attn_load_misses(d.p, host_k_pages, host_v_pages, block_table, c.lists["miss_ids"],
                                  c.lists["miss_slot"], c.counts, c.cache_slots, self.pool_k,
                                  self.pool_v, d.ws, stream)

    def slot_map(self, stream=None):
        c, d = self.cache, self.cache.decoder
        B.sparse_attn_slot_map(d.p, d.sel_ids, d.sel_count, c.slot_block, c.cache_slots,
                               self.sel_slot, d.ws, stream)

    def decode(self, q, out=None, stream=None):
        c, d = self.cache, self.cache.decoder
        B.sparse_attn_decode_slots(d.p, q, self.pool_k, self.pool_v, c.cache_slots, d.sel_ids,
                                   self.sel_slot, d.sel_count, d.out if out is None else out, d.ws,
                                   stream)

    def decode_io(self, q, host_k_pages, host_v_pages, block_table, out=None, stream=None):
        c, d = self.cache, self.cache.decoder
        B.sparse_attn_decode_slots_io(d.p, q, self.pool_k, self.pool_v, c.cache_slots, d.sel_ids,
                                      self.sel_slot, d.sel_count, host_k_pages, host_v_pages, block_table,
                                      c.lists["miss_ids"], c.lists["miss_slot"], c.counts,
                                      d.out if out is None else out, d.ws, stream)
