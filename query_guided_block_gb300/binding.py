"""Python binding of libsparse_attn (ctypes): argument marshalling only.

Every function here has the name of the C entry point it calls, takes torch CUDA
tensors (or raw integers for sizes) and passes their device pointers and the current
CUDA stream.  All computation happens in the library's kernels; there is no fallback
of any kind -- if the shared library is missing, every call raises.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsparse_attn.so")

OK, INVALID_ARG, UNSUPPORTED, CUDA_ERROR, DEVICE_BOUNDS = range(5)
F32, BF16 = 0, 1
SCORE_QUEST, SCORE_MEAN = 0, 1
ERR_PAGE, ERR_SEL_ID, ERR_SEL_COUNT, ERR_TIMEOUT, ERR_SLOT, ERR_CAPACITY = 1, 2, 4, 8, 16, 32


class SparseAttnError(RuntimeError):
    def __init__(self, fn: str, status: int, flags: int = 0):
        self.status = status
        self.flags = flags
        msg = f"{fn}: {_status_string(status)} (status {status})"
        if flags:
            msg += f", device error flags 0x{flags:x}"
        super().__init__(msg)


class sparse_attn_params(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "batch", "num_q_heads", "num_kv_heads", "head_dim", "n_tokens", "block_size",
        "num_pages", "window_tokens", "topk", "two_level", "coarse_block", "topk_coarse",
        "score_kind", "kv_dtype", "q_dtype")] + [("softmax_scale", C.c_float), ("num_reserve", C.c_int32),
                                                 ("num_queries", C.c_int32), ("capacity_tokens", C.c_int32)]


def make_params(batch, num_q_heads, num_kv_heads, head_dim, n_tokens, block_size, num_pages,
                window_tokens, topk, two_level=False, coarse_block=1024, topk_coarse=48,
                score_kind=SCORE_QUEST, kv_dtype=torch.bfloat16, q_dtype=torch.bfloat16,
                softmax_scale=0.0, num_reserve=0, num_queries=1, capacity_tokens=0) -> sparse_attn_params:
    def code(dt):
        if dt in (torch.bfloat16, BF16):
            return BF16
        if dt in (torch.float32, F32):
            return F32
        raise ValueError(f"unsupported dtype {dt}")
    if isinstance(score_kind, str):
        score_kind = {"quest": SCORE_QUEST, "mean": SCORE_MEAN}[score_kind]
    return sparse_attn_params(batch, num_q_heads, num_kv_heads, head_dim, n_tokens, block_size,
                              num_pages, window_tokens, topk, int(bool(two_level)), coarse_block,
                              topk_coarse, int(score_kind), code(kv_dtype), code(q_dtype),
                              float(softmax_scale), int(num_reserve), int(num_queries), int(capacity_tokens))


def params_for(w, **over) -> sparse_attn_params:
    """Parameters of a workload (query_guided_block_gb300.workloads.Workload)."""
    kw = dict(batch=w.batch, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
              head_dim=w.head_dim, n_tokens=w.n_tokens, block_size=w.block_size,
              num_pages=w.num_pages, window_tokens=w.window_tokens, topk=w.topk,
              two_level=w.two_level, coarse_block=w.coarse_block, topk_coarse=w.topk_coarse,
              score_kind=w.score, kv_dtype=w.kv_dtype, q_dtype=w.q_dtype,
              num_reserve=w.num_reserve, num_queries=w.num_queries)
    kw.update(over)
    return make_params(**kw)


_lib = None


def lib():
    """The loaded shared library.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build the CUDA library first "
                               "(query_guided_block_gb300.build.build())")
        L = C.CDLL(LIB_PATH)
        P = C.POINTER(sparse_attn_params)
        vp, sz, i32, u32p = C.c_void_p, C.c_size_t, C.c_int32, C.POINTER(C.c_uint32)
        sigs = {
            "sparse_attn_status_string": ([C.c_int], C.c_char_p),
            "sparse_attn_num_blocks": ([P], C.c_int32),
            "sparse_attn_sel_stride": ([P], C.c_int32),
            "sparse_attn_workspace_size": ([P, C.POINTER(C.c_size_t)], C.c_int),
            "sparse_attn_workspace_init": ([vp, sz, vp], C.c_int),
            "sparse_attn_workspace_set_wait_limit": ([vp, sz, C.c_uint64, vp], C.c_int),
            "sparse_attn_build_meta": ([P, vp, vp, vp, vp, vp, vp, sz, vp], C.c_int),
            "sparse_attn_append_meta": ([P, i32, vp, vp, vp, vp, vp, vp, sz, vp], C.c_int),
            "sparse_attn_select": ([P, vp, vp, vp, vp, vp, vp, vp, sz, vp], C.c_int),
            "sparse_attn_decode": ([P, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], C.c_int),
            "sparse_attn_step": ([P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], C.c_int),
            "sparse_attn_step_launches": ([P], C.c_int32),
            "sparse_attn_diff": ([P, i32, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                  vp, vp, vp, sz, vp], C.c_int),
            "sparse_attn_diff_slots": ([P, i32, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                        vp, vp, vp, vp, sz, vp], C.c_int),
            "sparse_attn_get_device_error": ([vp, sz, vp, u32p], C.c_int),
            "sparse_attn_select_noalloc": ([P, vp, vp, vp, vp, vp, vp, vp], C.c_int),
            "sparse_attn_select_noalloc_device_error": ([vp, u32p], C.c_int),
            "sparse_attn_select_reserved": ([P, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], C.c_int),
            "sparse_attn_topk_for_length": ([i32, i32], C.c_int32),
            "sparse_attn_slot_map": ([P, vp, vp, vp, i32, vp, vp, sz, vp], C.c_int),
            "sparse_attn_load_misses": ([P, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, sz, vp], C.c_int),
            "sparse_attn_decode_slots": ([P, vp, vp, vp, i32, vp, vp, vp, vp, vp, sz, vp], C.c_int),
            "sparse_attn_decode_slots_io": ([P, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz,
                                             vp], C.c_int),
        }
        for name, (args, res) in sigs.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def exported_symbols():
    return ["sparse_attn_status_string", "sparse_attn_num_blocks", "sparse_attn_sel_stride",
            "sparse_attn_workspace_size", "sparse_attn_workspace_init", "sparse_attn_build_meta",
            "sparse_attn_select", "sparse_attn_decode", "sparse_attn_diff",
            "sparse_attn_get_device_error", "sparse_attn_select_noalloc",
            "sparse_attn_select_reserved", "sparse_attn_topk_for_length",
            "sparse_attn_slot_map", "sparse_attn_load_misses", "sparse_attn_decode_slots",
            "sparse_attn_append_meta", "sparse_attn_step", "sparse_attn_step_launches",
            "sparse_attn_select_noalloc_device_error", "sparse_attn_workspace_set_wait_limit",
            "sparse_attn_decode_slots_io", "sparse_attn_diff_slots"]


def _status_string(status: int) -> str:
    try:
        return lib().sparse_attn_status_string(status).decode()
    except Exception:  # library not loadable: still report the number
        return "status"


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor (the library takes device pointers)")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return C.c_void_p(t.data_ptr())


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    return C.c_void_p(int(stream))


def _check(fn: str, status: int):
    if status != OK:
        raise SparseAttnError(fn, status)


# ----------------------------------------------------------- entry points --

def sparse_attn_num_blocks(p: sparse_attn_params) -> int:
    n = lib().sparse_attn_num_blocks(C.byref(p))
    if n < 0:
        raise SparseAttnError("sparse_attn_num_blocks", INVALID_ARG)
    return n


def sparse_attn_sel_stride(p: sparse_attn_params) -> int:
    n = lib().sparse_attn_sel_stride(C.byref(p))
    if n < 0:
        raise SparseAttnError("sparse_attn_sel_stride", INVALID_ARG)
    return n


def sparse_attn_workspace_size(p: sparse_attn_params) -> int:
    n = C.c_size_t(0)
    _check("sparse_attn_workspace_size", lib().sparse_attn_workspace_size(C.byref(p), C.byref(n)))
    return int(n.value)


def sparse_attn_workspace_init(ws: torch.Tensor, stream=None) -> None:
    _check("sparse_attn_workspace_init",
           lib().sparse_attn_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def sparse_attn_workspace_set_wait_limit(ws: torch.Tensor, cycles: int, stream=None) -> None:
    """Limit (SM clock cycles) of the bounded waits of kernels run on `ws`; 0 = default."""
    _check("sparse_attn_workspace_set_wait_limit",
           lib().sparse_attn_workspace_set_wait_limit(_ptr(ws), ws.numel() * ws.element_size(), int(cycles),
                                                      _stream(stream)))


def sparse_attn_build_meta(p, k_pages, block_table, kmin, kmax, kmean, ws, stream=None) -> None:
    _check("sparse_attn_build_meta", lib().sparse_attn_build_meta(
        C.byref(p), _ptr(k_pages), _ptr(block_table), _ptr(kmin), _ptr(kmax), _ptr(kmean),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def sparse_attn_append_meta(p, n_old, k_pages, block_table, kmin, kmax, kmean, ws, stream=None) -> None:
    _check("sparse_attn_append_meta", lib().sparse_attn_append_meta(
        C.byref(p), int(n_old), _ptr(k_pages), _ptr(block_table), _ptr(kmin), _ptr(kmax), _ptr(kmean),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def meta_rows(p) -> tuple:
    """(block rows, mean rows) allocated per unit in kmin / kmax and kmean: the capacity
    (capacity_tokens, or n_tokens when it is 0) in blocks and in mean rows."""
    cap = p.capacity_tokens if p.capacity_tokens > 0 else p.n_tokens
    mean_block = p.coarse_block if p.two_level else p.block_size
    return -(-cap // p.block_size), -(-cap // mean_block)


def sparse_attn_select(p, q, kmin, kmax, kmean, sel_ids, sel_count, ws, stream=None) -> None:
    _check("sparse_attn_select", lib().sparse_attn_select(
        C.byref(p), _ptr(q), _ptr(kmin), _ptr(kmax), _ptr(kmean), _ptr(sel_ids), _ptr(sel_count),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def sparse_attn_select_reserved(p, q, kmin, kmax, kmean, reserve_ids, sel_ids, sel_count, ws,
                                stream=None) -> None:
    _check("sparse_attn_select_reserved", lib().sparse_attn_select_reserved(
        C.byref(p), _ptr(q), _ptr(kmin), _ptr(kmax), _ptr(kmean), _ptr(reserve_ids), _ptr(sel_ids),
        _ptr(sel_count), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def sparse_attn_topk_for_length(n_tokens: int, block_size: int) -> int:
    k = lib().sparse_attn_topk_for_length(int(n_tokens), int(block_size))
    if k < 0:
        raise SparseAttnError("sparse_attn_topk_for_length", INVALID_ARG)
    return int(k)


def sparse_attn_decode(p, q, k_pages, v_pages, block_table, sel_ids, sel_count, out, ws,
                       stream=None) -> None:
    _check("sparse_attn_decode", lib().sparse_attn_decode(
        C.byref(p), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(sel_ids),
        _ptr(sel_count), _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def sparse_attn_step(p, q, kmin, kmax, kmean, reserve_ids, k_pages, v_pages, block_table, sel_ids,
                     sel_count, out, ws, stream=None) -> None:
    _check("sparse_attn_step", lib().sparse_attn_step(
        C.byref(p), _ptr(q), _ptr(kmin), _ptr(kmax), _ptr(kmean), _ptr(reserve_ids), _ptr(k_pages),
        _ptr(v_pages), _ptr(block_table), _ptr(sel_ids), _ptr(sel_count), _ptr(out), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def sparse_attn_step_launches(p) -> int:
    """Kernels a sparse_attn_step call launches (1 or 2), 0 for an empty batch, -1 when
    the problem is not supported by sparse_attn_step."""
    return int(lib().sparse_attn_step_launches(C.byref(p)))


def sparse_attn_diff(p, step, sel_ids, sel_count, prev_ids, prev_count, cache_slots, slot_block,
                     slot_last_use, hit_ids, miss_ids, miss_slot, evict_ids, evict_slot, new_ids,
                     dropped_ids, counts, ws, stream=None) -> None:
    _check("sparse_attn_diff", lib().sparse_attn_diff(
        C.byref(p), int(step), _ptr(sel_ids), _ptr(sel_count), _ptr(prev_ids), _ptr(prev_count),
        int(cache_slots), _ptr(slot_block), _ptr(slot_last_use), _ptr(hit_ids), _ptr(miss_ids),
        _ptr(miss_slot), _ptr(evict_ids), _ptr(evict_slot), _ptr(new_ids), _ptr(dropped_ids),
        _ptr(counts), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def sparse_attn_diff_slots(p, step, sel_ids, sel_count, prev_ids, prev_count, cache_slots, slot_block,
                           slot_last_use, hit_ids, miss_ids, miss_slot, evict_ids, evict_slot, new_ids,
                           dropped_ids, counts, sel_slot, ws, stream=None) -> None:
    _check("sparse_attn_diff_slots", lib().sparse_attn_diff_slots(
        C.byref(p), int(step), _ptr(sel_ids), _ptr(sel_count), _ptr(prev_ids), _ptr(prev_count),
        int(cache_slots), _ptr(slot_block), _ptr(slot_last_use), _ptr(hit_ids), _ptr(miss_ids),
        _ptr(miss_slot), _ptr(evict_ids), _ptr(evict_slot), _ptr(new_ids), _ptr(dropped_ids),
        _ptr(counts), _ptr(sel_slot), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def sparse_attn_select_noalloc(p, q, kmin, kmax, kmean, sel_ids, sel_count, stream=None) -> None:
    """sparse_attn_select with the library's fixed scratch instead of a workspace, for
    callers that cannot allocate device memory (see the C header)."""
    _check("sparse_attn_select_noalloc", lib().sparse_attn_select_noalloc(
        C.byref(p), _ptr(q), _ptr(kmin), _ptr(kmax), _ptr(kmean), _ptr(sel_ids), _ptr(sel_count),
        _stream(stream)))


def sparse_attn_select_noalloc_device_error(stream=None) -> int:
    """Error bits left in the noalloc scratch of the current device (synchronises the
    stream, clears them); 0 = clean."""
    flags = C.c_uint32(0)
    st = lib().sparse_attn_select_noalloc_device_error(_stream(stream), C.byref(flags))
    if st not in (OK, DEVICE_BOUNDS):
        raise SparseAttnError("sparse_attn_select_noalloc_device_error", st)
    return int(flags.value)


def _host_or_cuda_ptr(t: torch.Tensor):
    """Pointer of a contiguous tensor that may live in pinned host memory (the library
    reads pinned / registered host memory in place) or on the device."""
    if not isinstance(t, torch.Tensor) or not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    if not t.is_cuda and not t.is_pinned():
        raise ValueError("host K/V store must be in pinned memory")
    return C.c_void_p(t.data_ptr())


def sparse_attn_slot_map(p, sel_ids, sel_count, slot_block, cache_slots, sel_slot, ws,
                         stream=None) -> None:
    _check("sparse_attn_slot_map", lib().sparse_attn_slot_map(
        C.byref(p), _ptr(sel_ids), _ptr(sel_count), _ptr(slot_block), int(cache_slots),
        _ptr(sel_slot), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def sparse_attn_load_misses(p, host_k_pages, host_v_pages, block_table, miss_ids, miss_slot,
                            counts, cache_slots, pool_k, pool_v, ws, stream=None) -> None:
    _check("sparse_attn_load_misses", lib().sparse_attn_load_misses(
        C.byref(p), _host_or_cuda_ptr(host_k_pages), _host_or_cuda_ptr(host_v_pages),
        _ptr(block_table), _ptr(miss_ids), _ptr(miss_slot), _ptr(counts), int(cache_slots),
        _ptr(pool_k), _ptr(pool_v), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def sparse_attn_decode_slots(p, q, pool_k, pool_v, cache_slots, sel_ids, sel_slot, sel_count,
                             out, ws, stream=None) -> None:
    _check("sparse_attn_decode_slots", lib().sparse_attn_decode_slots(
        C.byref(p), _ptr(q), _ptr(pool_k), _ptr(pool_v), int(cache_slots), _ptr(sel_ids),
        _ptr(sel_slot), _ptr(sel_count), _ptr(out), _ptr(ws), ws.numel() * ws.element_size(),
        _stream(stream)))


def sparse_attn_decode_slots_io(p, q, pool_k, pool_v, cache_slots, sel_ids, sel_slot, sel_count,
                                host_k_pages, host_v_pages, block_table, miss_ids, miss_slot, counts, out,
                                ws, stream=None) -> None:
    _check("sparse_attn_decode_slots_io", lib().sparse_attn_decode_slots_io(
        C.byref(p), _ptr(q), _ptr(pool_k), _ptr(pool_v), int(cache_slots), _ptr(sel_ids),
        _ptr(sel_slot), _ptr(sel_count), _host_or_cuda_ptr(host_k_pages), _host_or_cuda_ptr(host_v_pages),
        _ptr(block_table), _ptr(miss_ids), _ptr(miss_slot), _ptr(counts), _ptr(out), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def sparse_attn_get_device_error(ws, stream=None) -> int:
    """Synchronises the stream; returns the error bits (0 = clean) and clears them."""
    flags = C.c_uint32(0)
    st = lib().sparse_attn_get_device_error(_ptr(ws), ws.numel() * ws.element_size(),
                                            _stream(stream), C.byref(flags))
    if st not in (OK, DEVICE_BOUNDS):
        raise SparseAttnError("sparse_attn_get_device_error", st)
    return int(flags.value)
