"""GPU parity of the sparse-attention backward (dsa_sparse_attn_backward) against the float64 oracle.

Criterion, per element, derived from the arithmetic of the kernel: the tensor cores multiply exact
bf16 inputs and accumulate in fp32, so the error comes from
  * rounding P and dS to bf16 (relative u = 2^-9 each);
  * the fp32 sums of S = q . c (576 terms) and of the forward's lse, which move p by a relative
    |dz| <= g576 scale sum_d |q_d c_d| each (g_n = n 2^-24, the classic bound of an n-term fp32 sum);
  * the fp32 sums of dp = do . c[:512] and of D = do . o (512 terms each): g512 sum_d |do_d| (|c_d| + |o_d|);
  * D being taken with the GPU's bf16 output instead of the exact o: |dD_h| = sum_d |do_h,d| |o_gpu - o_ref|_h,d;
  * rounding dq to bf16 (u |dq|).
With p, dp and D from the oracle:
    |ds - ds_ref|[h,s] <= p (|dp - D| (2u + 2|dz|) + |dD_h| + g512 sum_d |do_h,d| (|c_s,d| + |o_h,d|)) =: e[h,s]
    |dq - dq_ref|[h,d] <= 2 (scale sum_s e[h,s] |c_s,d|) + u |dq_ref|          (factor 2: the fp32 sums of dq)
    |dkv - ref|[s,d]   <= 2 sum_t (scale sum_h e[h,s] |q_h,d| + (u + 2|dz|) sum_h p |do_h,d| [d < 512])
Rows with no valid slot must give dq = 0 exactly and leave dkv untouched.  The dkv bound adds
absolute values over every token that selected a key, so it grows like the number of such tokens
while the gradient itself (terms of mixed sign) grows like its square root; for keys many tokens
share it is loose.  So the relative RMS error of dq and of dkv must also stay below 1e-2 (a few u
is expected; a dropped or misplaced term gives errors of the order of the gradient itself).
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

U = 2.0 ** -9
G576, G512 = 576 * 2.0 ** -24, 512 * 2.0 ** -24


@pytest.fixture(scope="module")
def dsa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_attention_30_b300 as m
    return m


def _bounds(q, kv, idx, do, o_gpu, scale):
    """Oracle gradients plus the per-element error bounds stated in the module docstring."""
    qd = q.double().numpy()
    kvd = kv.double().numpy()
    dod = do.double().numpy()
    T, H, _ = qd.shape
    dq_ref, dkv_ref = oracle.sparse_attention_backward(q, kv, idx, do, scale)
    tol_dq = np.zeros_like(dq_ref)
    tol_dkv = np.zeros_like(dkv_ref)
    for t in range(T):
        sel = idx[t][idx[t] >= 0]
        if len(sel) == 0:
            continue
        c = kvd[sel]
        o_ref, _ = oracle.attention_row(q[t], kv[torch.as_tensor(sel)], scale)
        z = scale * qd[t] @ c.T
        p = np.exp(z - z.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        dp = dod[t] @ c[:, :512].T
        D = (dod[t] * o_ref).sum(1)
        dD = (np.abs(dod[t]) * np.abs(o_gpu[t] - o_ref)).sum(1)
        dz = G576 * scale * (np.abs(qd[t]) @ np.abs(c).T)                   # [H, n]
        acc = G512 * (np.abs(dod[t]) @ np.abs(c[:, :512]).T + (np.abs(dod[t]) * np.abs(o_ref)).sum(1)[:, None])
        e = p * (np.abs(dp - D[:, None]) * (2 * U + 2 * dz) + dD[:, None] + acc)   # [H, n]
        tol_dq[t] = 2 * scale * (e @ np.abs(c)) + U * np.abs(dq_ref[t])
        part = scale * (e.T @ np.abs(qd[t]))                                 # [n, 576]
        part[:, :512] += ((U + 2 * dz) * p).T @ np.abs(dod[t])
        np.add.at(tol_dkv, sel, 2 * part)
    return dq_ref, dkv_ref, tol_dq, tol_dkv


def _check(dq, dkv, dq_ref, dkv_ref, tol_dq, tol_dkv, where):
    e_dq = np.abs(dq - dq_ref)
    bad = e_dq > tol_dq + 1e-30
    rows = sorted(set(np.nonzero(bad)[0].tolist()))[:8]
    assert not bad.any(), (f"{where}: {bad.sum()} dq entries off (tokens {rows}), worst excess "
                           f"{(e_dq - tol_dq).max():.3g}, max err {e_dq.max():.3g}, max |dq| {np.abs(dq_ref).max():.3g}")
    e_kv = np.abs(dkv - dkv_ref)
    bad = e_kv > tol_dkv + 1e-30
    keys = sorted(set(np.nonzero(bad)[0].tolist()))[:8]
    assert not bad.any(), (f"{where}: {bad.sum()} dkv entries off (rows {keys}), worst excess "
                           f"{(e_kv - tol_dkv).max():.3g}, max err {e_kv.max():.3g}, max |dkv| {np.abs(dkv_ref).max():.3g}")
    for name, got, ref in (("dq", dq, dq_ref), ("dkv", dkv, dkv_ref)):
        rel = np.sqrt(((got - ref) ** 2).sum() / max((ref ** 2).sum(), 1e-300))
        assert rel <= 1e-2, f"{where}: relative RMS error of {name} {rel:.3g}"


def _run(dsa, q, kv, idx, do, scale, status=None):
    qc, kvc, idxc, doc = q.cuda(), kv.cuda(), idx.cuda(), do.cuda()
    out, lse = dsa.sparse_attn(qc, kvc, idxc, scale)
    dq, dkv = dsa.sparse_attn_backward(qc, kvc, idxc, scale, out, doc, lse, status=status)
    return out.float().cpu().numpy(), dq.float().cpu().numpy(), dkv.cpu().numpy()


@pytest.mark.parametrize("H", [128, 8, 100])
def test_backward_ragged_selections_against_oracle(dsa, H):
    """Ragged selections (counts that are not multiples of the 32-key tile, -1 pads, an empty row,
    positions shared between tokens) over several tiles."""
    g = torch.Generator().manual_seed(61 + H)
    S, k = 400, 160
    counts = [160, 1, 33, 0, 95, 128, 64, 31, 160, 7]
    T = len(counts)
    q = torch.randn(T, H, 576, generator=g).to(torch.bfloat16)
    kv = torch.randn(S, 576, generator=g).to(torch.bfloat16)
    do = torch.randn(T, H, 512, generator=g).to(torch.bfloat16)
    idx = torch.full((T, k), -1, dtype=torch.int32)
    for t, c in enumerate(counts):
        idx[t, :c] = torch.randperm(S, generator=g)[:c].to(torch.int32)
    w = dsa.status_word()
    o_gpu, dq, dkv = _run(dsa, q, kv, idx, do, 0.07, status=w)
    assert dsa.read_status(w) == 0
    dq_ref, dkv_ref, tol_dq, tol_dkv = _bounds(q, kv, idx.numpy(), do, o_gpu, 0.07)
    assert np.all(dq[3] == 0)                                  # the empty row
    _check(dq, dkv, dq_ref, dkv_ref, tol_dq, tol_dkv, f"ragged H={H}")


def test_backward_accumulates_into_dkv_and_reports_range(dsa):
    g = torch.Generator().manual_seed(70)
    T, H, S, k = 4, 16, 200, 64
    q = torch.randn(T, H, 576, generator=g).to(torch.bfloat16).cuda()
    kv = torch.randn(S, 576, generator=g).to(torch.bfloat16).cuda()
    do = torch.randn(T, H, 512, generator=g).to(torch.bfloat16).cuda()
    idx = torch.stack([torch.randperm(S, generator=g)[:k] for _ in range(T)]).to(torch.int32).cuda()
    out, lse = dsa.sparse_attn(q, kv, idx, 0.05)
    dq1, dkv = dsa.sparse_attn_backward(q, kv, idx, 0.05, out, do, lse)
    once = dkv.clone()
    dq2, dkv = dsa.sparse_attn_backward(q, kv, idx, 0.05, out, do, lse, dkv=dkv)    # added, not overwritten
    assert torch.equal(dq1, dq2)
    torch.testing.assert_close(dkv, 2 * once, rtol=1e-5, atol=1e-6)
    assert dsa.device_status() == 0
    # an index past the end is skipped (as in the forward) and reported in the call's own word
    bad = idx.clone()
    bad[1, 3] = S + 9
    w = dsa.status_word()
    dsa.sparse_attn_backward(q, kv, bad, 0.05, out, do, lse, status=w)
    assert dsa.read_status(w) == 6 and dsa.device_status() == 0


def test_backward_config1_prefill_all_rows(dsa):
    """The tiny prefill (L=256, H=8, k=64) through the fused forward, then the backward of every row."""
    cfg = synth.config(1)
    hinp = synth.prefill_inputs(cfg)
    d = {k: v.cuda() for k, v in hinp.items()}
    idx = torch.empty((cfg.L, cfg.k), dtype=torch.int32, device="cuda")
    lse = torch.empty((cfg.L, cfg.H), dtype=torch.float32, device="cuda")
    f = dsa.Forward.prefill(d, cfg.k, cfg.scale, lse=lse, idx=idx)
    f()
    assert f.status() == 0
    g = torch.Generator().manual_seed(71)
    do = torch.randn(cfg.L, cfg.H, 512, generator=g).to(torch.bfloat16)
    dq, dkv = dsa.sparse_attn_backward(d["q"], d["kv"], idx, cfg.scale, f.out, do.cuda(), lse)
    assert dsa.device_status() == 0
    dq_ref, dkv_ref, tol_dq, tol_dkv = _bounds(hinp["q"], hinp["kv"], idx.cpu().numpy(), do,
                                               f.out.float().cpu().numpy(), cfg.scale)
    _check(dq.float().cpu().numpy(), dkv.cpu().numpy(), dq_ref, dkv_ref, tol_dq, tol_dkv, "config 1")


def test_backward_prefill4k_sampled_rows(dsa):
    """Rows of the 4K prefill (H=128, k=2048 selected from up to 4096 keys) with their own selections:
    the backward of those rows alone, checked in full (dq of every row, dkv of every key)."""
    cfg = synth.config(2)
    hinp = synth.prefill_inputs(cfg)
    d = {k: v.cuda() for k, v in hinp.items()}
    idx = torch.empty((cfg.L, cfg.k), dtype=torch.int32, device="cuda")
    lse = torch.empty((cfg.L, cfg.H), dtype=torch.float32, device="cuda")
    f = dsa.Forward.prefill(d, cfg.k, cfg.scale, lse=lse, idx=idx)
    f()
    assert f.status() == 0
    rows = torch.tensor([0, 1, 31, 32, 100, 2046, 2047, 2048, 2049, 3000, 4094, 4095])
    g = torch.Generator().manual_seed(72)
    do = torch.randn(len(rows), cfg.H, 512, generator=g).to(torch.bfloat16)
    rc = rows.cuda()
    q_r, idx_r, out_r, lse_r = d["q"][rc].contiguous(), idx[rc].contiguous(), f.out[rc].contiguous(), lse[rc].contiguous()
    dq, dkv = dsa.sparse_attn_backward(q_r, d["kv"], idx_r, cfg.scale, out_r, do.cuda(), lse_r)
    assert dsa.device_status() == 0
    dq_ref, dkv_ref, tol_dq, tol_dkv = _bounds(hinp["q"][rows], hinp["kv"], idx_r.cpu().numpy(), do,
                                               out_r.float().cpu().numpy(), cfg.scale)
    _check(dq.float().cpu().numpy(), dkv.cpu().numpy(), dq_ref, dkv_ref, tol_dq, tol_dkv, "4K rows")
