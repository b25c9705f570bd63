"""The derived tolerance of the GPU parity tests checked on the CPU: block means
computed in fp32 (as the metadata kernel does, here by torch in its own summation
order) pass tests.parity.check_means against the fp64 oracle, and means with a wrong
divisor (n + 1 tokens for n) do not."""
import dataclasses

import numpy as np
import pytest
import torch

from query_guided_block_gb300.workloads import Workload, make_inputs
from tests.parity import check_means, oracle_meta, sub_problem


def _means_fp32(host, w, mean_block, divisor_shift=0):
    bt = host["block_table"]
    S, nb = bt.shape
    Hkv, bs, D, N = w.num_kv_heads, w.block_size, w.head_dim, w.n_tokens
    rows = -(-N // mean_block)
    out = np.empty((S, Hkv, rows, D), np.float32)
    for s in range(S):
        k = host["k_pages"][s * nb:(s + 1) * nb].float().permute(1, 0, 2, 3).reshape(Hkv, nb * bs, D)[:, :N]
        for r in range(rows):
            t0, t1 = r * mean_block, min(N, (r + 1) * mean_block)
            tot = k[:, t0:t1].sum(1)                                   # fp32, torch's order
            inv = torch.tensor(1.0, dtype=torch.float32) / float(t1 - t0 + divisor_shift)
            out[s, :, r] = (tot * inv).numpy()
    return out


@pytest.mark.parametrize("mean_block,two_level", [(64, False), (1024, True)])
def test_fp32_means_pass_and_a_wrong_divisor_fails(mean_block, two_level):
    w = Workload(name="bounds", batch=1, num_q_heads=4, num_kv_heads=2, head_dim=64,
                 n_tokens=8 * 1024 + 100, block_size=64, window_tokens=256, topk=4,
                 kv_dtype=torch.bfloat16, q_dtype=torch.bfloat16,
                 score="quest" if two_level else "mean", two_level=two_level, coarse_block=1024,
                 topk_coarse=2)
    inp = make_inputs(w, "cpu")
    host = sub_problem(w, inp, [0])
    _, (_, _, kmean) = oracle_meta(w, host)
    good = _means_fp32(host, w, mean_block)
    check_means(good, kmean, host, w, mean_block)
    bad = _means_fp32(host, w, mean_block, divisor_shift=1)
    with pytest.raises(AssertionError):
        check_means(bad, kmean, host, w, mean_block)
