"""dsa_decode_noalloc: the decode forward for callers that may not allocate device memory
themselves (for example a plugin inside a serving engine that owns all device memory).
It takes its scratch from a fixed array inside the library instead of a workspace; its
output must match dsa_forward's, call after call, since every call shares that array.

This file is collected last on purpose (tests run in file order)."""
import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_attention_30_b300 as m
    return m


def test_noalloc_decode_matches_forward_on_consecutive_calls(dsa):
    cases = [synth.config(5), synth.config(3, B=16, ctx=20000, seed=7)]
    for n, cfg in enumerate(cases):
        d = synth.decode_inputs(cfg, device="cuda")
        max_len = int(d["seq_lens"].max())
        lse_ref = torch.empty((cfg.B, cfg.H), dtype=torch.float32, device="cuda")
        idx_ref = torch.empty((cfg.B, cfg.k), dtype=torch.int32, device="cuda")
        ref = dsa.Forward.decode(d, cfg.k, cfg.scale, max_len, lse=lse_ref, idx=idx_ref)
        ref()
        assert ref.status() == 0 and dsa.device_status() == 0
        # the selection either stays in the static scratch (idx NULL) or goes to a caller-owned buffer,
        # in which case the scratch holds only the scores
        for own_idx in (False, True):
            out = torch.full_like(ref.out, float("nan"))
            lse = torch.full_like(lse_ref, float("nan"))
            idx = torch.full_like(idx_ref, -7) if own_idx else None
            args = dsa.ForwardArgs.from_buffer_copy(ref.args)
            args.out, args.lse, args.idx = out.data_ptr(), lse.data_ptr(), idx.data_ptr() if own_idx else None
            stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
            assert dsa.lib.dsa_decode_noalloc(ctypes.byref(args), stream) == 0
            assert dsa.device_status() == 0
            where = f"call {n}, caller idx {own_idx}"
            d_out = (out.float() - ref.out.float()).abs()
            assert d_out.max().item() <= 2e-2 and d_out.mean().item() <= 2e-3, where
            assert (lse - lse_ref).abs().max().item() <= 2e-3, where
            assert not torch.isnan(out).any(), where
            if own_idx:   # the same selected sets as dsa_forward's (slot order is not fixed)
                assert torch.equal(torch.sort(idx, dim=1).values, torch.sort(idx_ref, dim=1).values), where


def test_noalloc_rejects_requests_beyond_its_scratch(dsa):
    cap = dsa.lib.dsa_decode_noalloc_capacity()
    assert cap == 20 << 20
    a = dsa.ForwardArgs(mode=dsa.MODE_DECODE, H_I=64, H=128, k=2048, scale=0.07, B=64, page_size=64,
                        n_pages=1, bt_stride=2048, max_seq_len=131072)
    # 64 x 131072 fp32 scores need 32 MiB: refused before anything runs
    assert dsa.lib.dsa_decode_noalloc(ctypes.byref(a), None) == 3
    a.mode = dsa.MODE_PREFILL
    assert dsa.lib.dsa_decode_noalloc(ctypes.byref(a), None) == 1
    assert np.isfinite(cap)
