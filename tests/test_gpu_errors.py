"""Bad inputs that only the device can see are caught by the kernels' own bounds
checks: the access is skipped, a bit is set in the workspace error word, and the
context stays usable.  Every input here is one the kernels check before use; nothing
is expected to fault."""
import time

import numpy as np
import pytest
import torch

from query_guided_block_gb300 import binding as B
from query_guided_block_gb300.build import build
from query_guided_block_gb300.decoder import SlotCache, SparseDecoder
from query_guided_block_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available()
    build()
    B.lib()


def _case():
    w = Workload(name="err", batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128,
                 n_tokens=4096, block_size=64, window_tokens=256, topk=6)
    inp = make_inputs(w, "cuda")
    dec = SparseDecoder(B.params_for(w))
    dec.build_meta(inp["k_pages"], inp["block_table"])
    dec.select(inp["q"])
    assert dec.device_error() == 0
    return w, inp, dec


def test_out_of_range_page_in_block_table():
    w, inp, dec = _case()
    bt = inp["block_table"].clone()
    j = int(dec.sel_ids[0, 0, 0])
    bt[0, j] = w.num_pages + 5
    dec.decode(inp["q"], inp["k_pages"], inp["v_pages"], bt)
    assert dec.device_error() & B.ERR_PAGE
    bt[0, 3] = -7
    dec.build_meta(inp["k_pages"], bt)
    assert dec.device_error() & B.ERR_PAGE
    # the error word was cleared by the read; a clean call reports nothing
    dec.build_meta(inp["k_pages"], inp["block_table"])
    dec.decode(inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"])
    assert dec.device_error() == 0


def test_out_of_range_selection():
    w, inp, dec = _case()
    ids = dec.sel_ids.clone()
    ids[1, 1, 2] = w.num_blocks + 3
    dec.decode(inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"], sel_ids=ids)
    assert dec.device_error() & B.ERR_SEL_ID
    cnt = dec.sel_count.clone()
    cnt[0, 1] = dec.sel_stride + 9
    dec.decode(inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"], sel_count=cnt)
    assert dec.device_error() & B.ERR_SEL_COUNT
    cnt[0, 1] = -1
    dec.decode(inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"], sel_count=cnt)
    assert dec.device_error() & B.ERR_SEL_COUNT
    dec.decode(inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"])
    assert dec.device_error() == 0
    assert torch.isfinite(dec.out).all()


def test_diff_rejects_corrupt_state_and_leaves_it_untouched():
    w, inp, dec = _case()
    cache = SlotCache(dec, 32)
    cache.slot_block[1, 4] = w.num_blocks + 1
    before = cache.slot_block.clone()
    cache.diff(0)
    assert dec.device_error() & B.ERR_SLOT
    assert torch.equal(cache.slot_block[1], before[1])
    assert int(cache.counts[1].abs().sum()) == 0
    # non-ascending request set
    cache.slot_block.fill_(-1)
    ids = dec.sel_ids.clone()
    ids[0, 0, 0], ids[0, 0, 1] = ids[0, 0, 1].item(), ids[0, 0, 0].item()
    cache.diff(0, sel_ids=ids)
    assert dec.device_error() & B.ERR_SEL_ID
    cache.diff(0)
    assert dec.device_error() == 0


def test_fused_step_reports_bad_pages_and_stays_usable():
    """The fused step's decode phase checks the page table like the decode call."""
    w, inp, dec = _case()
    bt = inp["block_table"].clone()
    j = int(dec.sel_ids[1, 0, 0])
    bt[1, j] = w.num_pages + 1
    dec.step_fused(inp["q"], inp["k_pages"], inp["v_pages"], bt)
    assert dec.device_error() & B.ERR_PAGE
    dec.step_fused(inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"])
    assert dec.device_error() == 0
    assert torch.isfinite(dec.out).all()


def test_tensor_core_multi_query_decode_reports_bad_inputs():
    """The tcgen05 multi-query decode skips (and reports) a page outside the pool and a
    selection id outside the context; its tensor-map loads never see them."""
    w = Workload(name="err_mq", batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128,
                 n_tokens=6000, block_size=32, window_tokens=256, topk=10, num_queries=8)
    inp = make_inputs(w, "cuda")
    dec = SparseDecoder(B.params_for(w))
    dec.build_meta(inp["k_pages"], inp["block_table"])
    dec.select(inp["q"])
    assert dec.device_error() == 0
    bt = inp["block_table"].clone()
    bt[0, int(dec.sel_ids[0, 1, 2])] = -3
    dec.decode(inp["q"], inp["k_pages"], inp["v_pages"], bt)
    assert dec.device_error() & B.ERR_PAGE
    ids = dec.sel_ids.clone()
    ids[1, 0, 1] = w.num_blocks + 2
    dec.decode(inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"], sel_ids=ids)
    assert dec.device_error() & B.ERR_SEL_ID
    dec.decode(inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"])
    assert dec.device_error() == 0
    assert torch.isfinite(dec.out).all()


@pytest.mark.parametrize("batch,ctx", [(4, 65536), (16, 16384)])
def test_bounded_wait_runs_out_and_the_next_step_is_clean(batch, ctx):
    """The fused step's decode phase waits for selections other CTAs publish: per unit
    of its range (batch 4: 32 units, each split over 4 CTAs) or, when every CTA decodes
    whole units (batch 16: 128 units), for the next unit in publication order.  With a
    limit of 64 cycles the CTAs that rank nothing poll while the rankers are still at
    work, so the wait runs out: the call returns promptly and the error word holds
    SPARSE_ATTN_ERR_TIMEOUT (with per-unit waits the output is also finite: every
    range is decoded with the selection in place).  With the default limit restored,
    the next step on the same workspace (new queries) equals the two-call result bit
    for bit: a selection published late by the timed-out step is never taken for the
    next step's."""
    from tests.test_gpu_step import _assert_same
    w = Workload(name="timeout", batch=batch, num_q_heads=32, num_kv_heads=8, head_dim=128,
                 n_tokens=ctx, block_size=32, window_tokens=512, topk=64, planted_per_unit=8)
    inp = make_inputs(w, "cuda")
    p = B.params_for(w)
    assert B.sparse_attn_step_launches(p) == 1
    two, fused = SparseDecoder(p), SparseDecoder(p)
    for d in (two, fused):
        d.build_meta(inp["k_pages"], inp["block_table"])
    kv = (inp["k_pages"], inp["v_pages"], inp["block_table"])
    fused.step_fused(inp["q"], *kv)
    assert fused.device_error() == 0              # valid selections in place
    fused.set_wait_limit(64)
    g = torch.Generator(device="cuda").manual_seed(3)
    new_q = lambda: torch.randn(inp["q"].shape, generator=g, device="cuda").to(w.q_dtype)
    timed_out = False
    for _ in range(4):
        fused.out.fill_(float("nan"))
        t0 = time.time()
        fused.step_fused(new_q(), *kv)
        flags = fused.device_error()               # synchronises
        assert time.time() - t0 < 2.0
        assert flags & ~B.ERR_TIMEOUT == 0, f"flags 0x{flags:x}"
        if batch == 4:
            assert torch.isfinite(fused.out).all()
        if flags & B.ERR_TIMEOUT:
            timed_out = True
            break
    assert timed_out, "no wait ran out with a 64-cycle limit"
    fused.set_wait_limit(0)
    for _ in range(2):
        q = new_q()
        two.step(q, *kv)
        fused.step_fused(q, *kv)
        assert two.device_error() == 0 and fused.device_error() == 0
        _assert_same(two, fused)
