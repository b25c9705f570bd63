"""Host-side checks of the C ABI (no GPU needed): the library builds for sm_103a, loads,
exports every entry point the header declares, and rejects bad arguments on the host
before any CUDA call."""
import ctypes as C

import torch
import os
import re

import pytest

from query_guided_block_gb300 import binding as B
from query_guided_block_gb300.build import build
from query_guided_block_gb300.workloads import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build()
    return B.lib()


def declared_entry_points():
    text = open(os.path.join(ROOT, "include", "sparse_attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sparse_attn_\w+)\s*\(", text)))


def test_header_and_binding_agree(L):
    declared = declared_entry_points()
    assert declared == sorted(B.exported_symbols())
    for name in declared:
        assert getattr(L, name) is not None


def test_sizes_for_the_five_workloads(L):
    expect_stride = {"tiny_fp32_4k": 8 + 2, "mha_32k": 32 + 8, "gqa_128k": 64 + 16,
                     "two_level_256k": 48 + 8, "lru_64k": 32 + 8, "reserve_128k": 64 + 41 + 16,
                    "mq_128k": 64 + 16}
    for name, w in WORKLOADS.items():
        p = B.params_for(w)
        assert B.sparse_attn_num_blocks(p) == w.num_blocks
        assert B.sparse_attn_sel_stride(p) == expect_stride[name]
        assert B.sparse_attn_workspace_size(p) > 0


def test_bad_parameters_are_rejected(L):
    w = WORKLOADS["gqa_128k"]
    n = C.c_size_t()
    for change, want in [(dict(num_q_heads=30), B.INVALID_ARG),      # not a multiple of Hkv
                         (dict(num_q_heads=48), B.UNSUPPORTED),      # group of 6
                         (dict(head_dim=96), B.UNSUPPORTED),
                         (dict(block_size=48), B.UNSUPPORTED),
                         (dict(n_tokens=-1), B.INVALID_ARG),
                         (dict(topk=-2), B.INVALID_ARG),
                         (dict(n_tokens=16384 * 32 + 1), B.UNSUPPORTED),   # > 16384 blocks
                         (dict(two_level=True, coarse_block=1000), B.INVALID_ARG),
                         (dict(softmax_scale=float("nan")), B.INVALID_ARG),
                         (dict(num_pages=0), B.INVALID_ARG),
                         (dict(num_reserve=-1), B.INVALID_ARG),
                         (dict(num_queries=-1), B.INVALID_ARG),
                         (dict(num_queries=4, kv_dtype=torch.float32), B.UNSUPPORTED),
                         (dict(num_queries=4, two_level=True), B.UNSUPPORTED),
                         (dict(capacity_tokens=1000), B.INVALID_ARG)]:         # below n_tokens
        p = B.params_for(w, **change)
        assert L.sparse_attn_workspace_size(C.byref(p), C.byref(n)) == want, change
    assert L.sparse_attn_workspace_size(None, C.byref(n)) == B.INVALID_ARG


def test_null_and_misaligned_pointers_are_rejected_before_launch(L):
    w = WORKLOADS["mha_32k"]
    p = B.params_for(w)
    nbytes = B.sparse_attn_workspace_size(p)
    fake = C.c_void_p(1 << 20)          # never dereferenced: checks fail first
    odd = C.c_void_p((1 << 20) + 4)
    null = None
    # workspace missing / too small / misaligned
    assert L.sparse_attn_select(C.byref(p), fake, fake, fake, null, fake, fake, null, nbytes, null) == B.INVALID_ARG
    assert L.sparse_attn_select(C.byref(p), fake, fake, fake, null, fake, fake, fake, nbytes - 1, null) == B.INVALID_ARG
    assert L.sparse_attn_select(C.byref(p), fake, fake, fake, null, fake, fake, odd, nbytes, null) == B.INVALID_ARG
    # null / misaligned tensors
    assert L.sparse_attn_select(C.byref(p), null, fake, fake, null, fake, fake, fake, nbytes, null) == B.INVALID_ARG
    assert L.sparse_attn_decode(C.byref(p), odd, fake, fake, fake, fake, fake, fake, fake, nbytes, null) == B.INVALID_ARG
    assert L.sparse_attn_decode(C.byref(p), fake, fake, null, fake, fake, fake, fake, fake, nbytes, null) == B.INVALID_ARG
    assert L.sparse_attn_build_meta(C.byref(p), fake, fake, odd, fake, null, fake, nbytes, null) == B.INVALID_ARG
    # mean metadata required by the two-level path
    p2 = B.params_for(WORKLOADS["two_level_256k"])
    n2 = B.sparse_attn_workspace_size(p2)
    assert L.sparse_attn_build_meta(C.byref(p2), fake, fake, fake, fake, null, fake, n2, null) == B.INVALID_ARG
    # diff: cache smaller than a request set
    args = [fake] * 13
    assert L.sparse_attn_diff(C.byref(p), 0, fake, fake, fake, fake, 8, *args[:10], fake, nbytes, null) == B.INVALID_ARG
    assert L.sparse_attn_get_device_error(null, 256, null, C.byref(C.c_uint32())) == B.INVALID_ARG


def test_status_strings(L):
    for s in range(5):
        assert L.sparse_attn_status_string(s)


def test_topk_for_length_matches_the_oracle(L):
    """The host-side k rule (SparDA page §3.2) agrees with the oracle's statement of it."""
    import oracle
    for bs in (8, 32, 64, 128):
        for n in list(range(0, 70000, 777)) + [8192, 8193, 16384, 16385, 32768, 32769, 131072, 262144]:
            assert B.sparse_attn_topk_for_length(n, bs) == oracle.topk_for_length(n, bs), (n, bs)
    assert L.sparse_attn_topk_for_length(-1, 64) == -1
    assert L.sparse_attn_topk_for_length(100, 0) == -1


def test_plain_select_refuses_a_reserve_count(L):
    """A problem with num_reserve > 0 must go through sparse_attn_select_reserved; the
    check is on the host, before any device pointer is touched."""
    p = B.params_for(WORKLOADS["reserve_128k"])
    rc = L.sparse_attn_select(C.byref(p), None, None, None, None, None, None, None, 0, None)
    assert rc == B.INVALID_ARG


def test_append_rejects_bad_lengths(L):
    """n_old outside [0, n_tokens] is refused on the host, before any launch."""
    p = B.params_for(WORKLOADS["gqa_128k"], capacity_tokens=200000)
    for n_old in (-1, p.n_tokens + 1):
        rc = L.sparse_attn_append_meta(C.byref(p), n_old, None, None, None, None, None, None, 0, None)
        assert rc == B.INVALID_ARG


@pytest.mark.parametrize("name", ["gqa_128k", "reserve_128k", "two_level_256k", "lru_64k"])
def test_capacity_workspace_covers_every_length(name):
    """A workspace sized with capacity_tokens serves select / decode at every length up
    to the capacity (the window's block count alternates as it slides over block
    boundaries, so the size at the capacity alone is not always enough)."""
    w = WORKLOADS[name]
    cap = w.n_tokens + 5 * w.block_size + 3
    big = B.sparse_attn_workspace_size(B.params_for(w, capacity_tokens=cap))
    for n in range(w.n_tokens - 3 * w.block_size, cap + 1):
        assert B.sparse_attn_workspace_size(B.params_for(w, n_tokens=n)) <= big, n


def test_step_launch_plan():
    """sparse_attn_step's plan, decided on the host: one cooperative launch while the
    units fit one CTA per SM, select + dependent decode beyond that, refused for
    problems it does not cover."""
    import dataclasses
    assert B.sparse_attn_step_launches(B.params_for(WORKLOADS["gqa_128k"])) == 1      # 128 units
    assert B.sparse_attn_step_launches(B.params_for(WORKLOADS["reserve_128k"])) == 1
    assert B.sparse_attn_step_launches(B.params_for(WORKLOADS["mha_32k"])) == 2       # 256 units
    assert B.sparse_attn_step_launches(B.params_for(WORKLOADS["two_level_256k"])) == -1
    assert B.sparse_attn_step_launches(B.params_for(WORKLOADS["tiny_fp32_4k"])) == -1  # fp32 K/V
    assert B.sparse_attn_step_launches(B.params_for(WORKLOADS["mq_128k"])) == -1       # Q > 1
    empty = dataclasses.replace(WORKLOADS["gqa_128k"], batch=0)
    assert B.sparse_attn_step_launches(B.params_for(empty)) == 0
