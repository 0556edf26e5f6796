"""Host-side logic of bench.py on CPU: the algorithmic work that every roofline figure divides by.

The counts are checked against the oracle's exact pair counts (themselves pinned to closed forms
in test_oracle.py), so a wrong numerator cannot inflate a reported fraction of peak.
"""
import numpy as np
import pytest

import bench
import oracle


@pytest.mark.parametrize("L,k", [(256, 64), (4096, 2048), (131072, 2048), (1000, 4096)])
def test_prefill_work_counts(L, k):
    H_I, H = 64, 128
    w = bench.prefill_work(L, H_I, H, k)
    assert w["indexer_flop"] == 2.0 * H_I * 128 * oracle.causal_pairs(L)
    assert w["attn_flop"] == 2.0 * H * (576 + 512) * oracle.selected_pairs(L, k)
    # scores read once (4 B per causal pair) plus the selection written (4 B per slot)
    assert w["topk_bytes"] == 4.0 * oracle.causal_pairs(L) + 4.0 * k * L
    # Q and O stream once, the selection is read, every latent row at least once
    assert w["attn_bytes"] == L * H * 1152 * 1.0 + L * H * 1024 * 1.0 + 4.0 * k * L + 1152.0 * L


def test_decode_work_counts():
    lens = [8192, 100, 131072, 2048, 2049]
    k, H_I, H = 2048, 64, 128
    w = bench.decode_work(lens, H_I, H, k)
    sel = sum(min(k, n) for n in lens)
    assert w["attn_flop"] == 2.0 * H * (576 + 512) * sel
    assert w["attn_bytes"] == sel * 1152 + len(lens) * H * (576 + 512) * 2.0 + 4.0 * k * len(lens)
    n = sum(lens)
    assert w["indexer_bytes"] == n * (128 + 4) + 4.0 * n + len(lens) * H_I * (128 + 8)
    assert w["topk_bytes"] == 4.0 * n + 4.0 * k * len(lens)


def test_aggregate_throughput_is_whole_job():
    # 4 ranks of 131072 tokens each, 5 steps, slowest rank 1000 ms in total
    assert bench.aggregate_tokens_per_s(131072, 4, 5, 1000.0) == pytest.approx(131072 * 4 * 5)
    assert bench.rank_seed(3, 0) == 3 and bench.rank_seed(3, 2) != bench.rank_seed(3, 1)
