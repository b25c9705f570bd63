"""GB300 (sm_103a) query-guided block-sparse decode attention.

The compute lives in libsparse_attn.so (C ABI in include/sparse_attn.h); this package
holds its ctypes binding, device-buffer plumbing, the in-tree build step and the seeded
synthetic workloads.
"""
from . import binding, workloads  # noqa: F401
from .binding import (SparseAttnError, make_params, params_for,  # noqa: F401
                      sparse_attn_append_meta, sparse_attn_build_meta, sparse_attn_decode,
                      sparse_attn_decode_slots, sparse_attn_diff, sparse_attn_get_device_error,
                      sparse_attn_load_misses, sparse_attn_num_blocks, sparse_attn_select,
                      sparse_attn_select_noalloc, sparse_attn_select_noalloc_device_error,
                      sparse_attn_select_reserved, sparse_attn_sel_stride,
                      sparse_attn_slot_map, sparse_attn_step, sparse_attn_step_launches,
                      sparse_attn_topk_for_length, sparse_attn_workspace_init, sparse_attn_workspace_set_wait_limit,
                      sparse_attn_workspace_size)
from .decoder import SlotCache, SparseDecoder  # noqa: F401
