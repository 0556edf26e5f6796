"""Input generators (CPU): the tail-rows generator reproduces the same rows of the full workload, and
the generated tensors follow the stated recipe (page tables, lengths, per-token FP8 scales)."""
import numpy as np
import torch

import synth


def test_randn_rows_matches_full_draw():
    cfg = synth.config(4, L=10000)
    full = synth._randn(cfg, 1, (10000, 3), "cpu", 4096)
    for r0, r1 in [(0, 10000), (4095, 4097), (8192, 10000), (9999, 10000), (100, 200)]:
        assert torch.equal(synth._randn_rows(cfg, 1, (10000, 3), r0, r1, "cpu", 4096), full[r0:r1])


def test_prefill_tail_inputs_match_full_workload():
    cfg = synth.config(4, L=9000, H=2, H_I=4)
    full = synth.prefill_inputs(cfg, device="cpu")
    tail = synth.prefill_tail_inputs(cfg, 700, device="cpu")
    assert tail["row0"] == 8300
    for name in ("q8", "q_scale", "w", "q"):
        assert torch.equal(tail[name], full[name][8300:]), name
    for name in ("k8", "k_scale", "kv"):
        assert torch.equal(tail[name], full[name]), name


def test_decode_inputs_follow_the_recipe():
    # lengths in [ctx_lo, ctx_hi]; each sequence's pages are a slice of one shuffled permutation of
    # all pages (every page owned by exactly one sequence); tokens past a sequence's end are zero;
    # the query scale is one value per token, repeated over the indexer heads
    cfg = synth.config(5, B=6, H=4, H_I=64, k=64, page=16, ctx_lo=20, ctx_hi=300, planted=3, seed=11)
    d = synth.decode_inputs(cfg)
    lens = d["seq_lens"].long()
    assert int(lens.min()) >= 20 and int(lens.max()) <= 300
    n_pages = d["k8_cache"].shape[0]
    owned = []
    for b in range(cfg.B):
        n = (int(lens[b]) + 15) // 16
        row = d["block_table"][b]
        assert torch.all(row[n:] == -1) and torch.all(row[:n] >= 0)
        owned += row[:n].tolist()
    assert sorted(owned) == list(range(n_pages))
    used = torch.zeros(n_pages * 16, dtype=torch.bool)
    for b in range(cfg.B):
        pages = d["block_table"][b][: (int(lens[b]) + 15) // 16].long()
        used[(pages[:, None] * 16 + torch.arange(16)).reshape(-1)[: int(lens[b])]] = True
    assert torch.all(d["kv_cache"].reshape(-1, 576)[~used].float() == 0)
    assert torch.all(d["k8_cache"].reshape(-1, 128)[~used] == 0)
    assert torch.all(d["q_scale"] == d["q_scale"][:, :1])


def test_prefill_inputs_scales_and_fp8_range():
    # per-token FP8 encoding: the scale is the token's absmax / 448, so the largest code of every
    # token decodes to +-448 (e4m3 max) and no code is NaN
    import oracle
    cfg = synth.config(1, L=64, H_I=8, H=4, k=16, planted=4, seed=3)
    d = synth.prefill_inputs(cfg)
    k = oracle.e4m3_to_f64(d["k8"].numpy())
    assert not np.isnan(k).any()
    assert np.allclose(np.abs(k).max(axis=1), 448.0)
    q = oracle.e4m3_to_f64(d["q8"].numpy()).reshape(64, -1)
    assert np.allclose(np.abs(q).max(axis=1), 448.0)
    assert torch.all(d["q_scale"] == d["q_scale"][:, :1])
