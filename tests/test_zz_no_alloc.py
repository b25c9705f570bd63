"""The allocation-free selection entry point against the regular one.

sparse_attn_select_noalloc serves callers that cannot allocate device memory (code
running inside another framework's allocator or memory pool, in a host callback, or in
a plugin whose host owns every device allocation): it keeps its scratch in a fixed
array inside the library instead of a caller workspace.  Its results must equal
sparse_attn_select's, on consecutive calls that share that array.  This file is named to
run last, so a failure here never hides the other tests.
"""
import ctypes as C

import pytest
import torch

from query_guided_block_gb300 import binding as B
from query_guided_block_gb300.build import build
from query_guided_block_gb300.decoder import SparseDecoder
from query_guided_block_gb300.workloads import WORKLOADS, make_inputs, scaled

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available()
    build()
    B.lib()


def _stream():
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def _noalloc(p, q, dec, ids, cnt):
    return B.lib().sparse_attn_select_noalloc(
        C.byref(p), C.c_void_p(q.data_ptr()), C.c_void_p(dec.kmin.data_ptr()),
        C.c_void_p(dec.kmax.data_ptr()), None, C.c_void_p(ids.data_ptr()),
        C.c_void_p(cnt.data_ptr()), _stream())


@pytest.mark.parametrize("name,batch", [("gqa_128k", 4), ("mha_32k", 2)])
def test_noalloc_select_matches_workspace_select_twice(name, batch):
    w = scaled(WORKLOADS[name], batch=batch)
    inp = make_inputs(w, "cuda")
    p = B.params_for(w)
    dec = SparseDecoder(p)
    dec.build_meta(inp["k_pages"], inp["block_table"])
    dec.select(inp["q"])
    assert dec.device_error() == 0
    for call in range(2):
        ids = torch.full_like(dec.sel_ids, -7)
        cnt = torch.full_like(dec.sel_count, -7)
        assert _noalloc(p, inp["q"], dec, ids, cnt) == B.OK
        torch.cuda.synchronize()
        # selections are bit-exact between the two entry points (same kernel, same inputs)
        assert torch.equal(cnt, dec.sel_count), f"call {call}: counts differ"
        for u in range(w.units):
            n = int(cnt.view(-1)[u])
            assert torch.equal(ids.view(w.units, -1)[u, :n], dec.sel_ids.view(w.units, -1)[u, :n])
        # the private scratch's error word: clean calls leave no bit set
        assert B.sparse_attn_select_noalloc_device_error() == 0


def test_noalloc_select_rejects_what_does_not_fit():
    big = B.params_for(WORKLOADS["gqa_128k"], batch=64)          # 512 units x 4080 scores > 4 MiB
    dummy = torch.zeros(64, dtype=torch.int32, device="cuda")
    ptr = C.c_void_p(dummy.data_ptr())
    assert B.lib().sparse_attn_select_noalloc(C.byref(big), ptr, ptr, ptr, None, ptr, ptr, _stream()) \
        == B.UNSUPPORTED
    two = B.params_for(WORKLOADS["two_level_256k"], batch=1)
    assert B.lib().sparse_attn_select_noalloc(C.byref(two), ptr, ptr, ptr, ptr, ptr, ptr, _stream()) \
        == B.UNSUPPORTED
