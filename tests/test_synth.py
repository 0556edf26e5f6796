"""Input generators (CPU): the tail-rows generator reproduces the same rows of the full workload."""
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
