import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size parity case")


def oracle_problem_for(w, num_pages=None, **over):
    """Oracle problem description for a workload (test glue only)."""
    import torch
    import oracle
    kw = dict(batch=w.batch, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
              head_dim=w.head_dim, n_tokens=w.n_tokens, block_size=w.block_size,
              num_pages=w.num_pages if num_pages is None else num_pages,
              window_tokens=w.window_tokens, topk=w.topk, two_level=w.two_level,
              coarse_block=w.coarse_block, topk_coarse=w.topk_coarse, score_kind=w.score,
              kv_bf16=(w.kv_dtype == torch.bfloat16), q_bf16=(w.q_dtype == torch.bfloat16))
    kw.update(over)
    return oracle.problem(**kw)


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle
