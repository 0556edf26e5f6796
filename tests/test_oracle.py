"""Pins for the float64 oracle: each test checks it against something other than itself.

- FP8 / bf16 decoders: torch's own float8_e4m3fn / bfloat16 conversions (library routines).
- Indexer: the identities I(k) - I(-k) = sum_j w_j (q_j.k) and I(k) + I(-k) = sum_j w_j |q_j.k|
  (ReLU(x) - ReLU(-x) = x, ReLU(x) + ReLU(-x) = |x|), evaluated with torch matmul on
  torch-decoded values; homogeneity in the scales; the causal mask.
- Top-k: brute-force enumeration of every subset on tiny rows.
- Attention: torch scaled_dot_product_attention in float64 (dense causal when k >= L,
  and with a boolean mask built from any index set).
- Paging: a paged decode equals the same sequence laid out contiguously.
- Work counts: the closed form k(k+1)/2 + (L-k)k and L(L+1)/2.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- formats

def test_e4m3_decode_all_codes_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_to_f64(codes.numpy())
    nan_ref, nan_got = np.isnan(ref), np.isnan(got)
    assert np.array_equal(nan_ref, nan_got)
    assert np.array_equal(ref[~nan_ref], got[~nan_got])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x80] == 0.0


def test_bf16_decode_matches_torch():
    g = torch.Generator().manual_seed(5)
    x = (torch.randn(10000, generator=g) * 100).to(torch.bfloat16)
    x[:3] = torch.tensor([0.0, -1.5, 3.0e38]).to(torch.bfloat16)
    got = oracle.bf16_bits_to_f64(x.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(got, x.to(torch.float64).numpy())


# ---------------------------------------------------------------- indexer

def _small_indexer_inputs(seed=0, T=24, S=40, H_I=4):
    g = torch.Generator().manual_seed(seed)
    q8, sq = synth.encode_e4m3_per_token(torch.randn(T, H_I, 128, generator=g))
    k8, sk = synth.encode_e4m3_per_token(torch.randn(S, 128, generator=g) * 3)
    w = torch.randn(T, H_I, generator=g)
    sq = (sq[:, None] * torch.linspace(0.5, 2.0, H_I)[None, :]).contiguous()  # distinct per head
    return q8, sq, w, k8, sk


def _torch_linear_and_abs(q8, sq, w, k8, sk):
    """sum_j w sq sk (q_j.k) and sum_j w sq sk |q_j.k| via torch's decode + matmul."""
    q = q8.view(torch.float8_e4m3fn).to(torch.float64)
    k = k8.view(torch.float8_e4m3fn).to(torch.float64)
    dots = torch.einsum("tjd,sd->tjs", q, k) * sq.double()[:, :, None] * sk.double()[None, None, :]
    wd = w.double()[:, :, None]
    return (wd * dots).sum(1).numpy(), (wd * dots.abs()).sum(1).numpy()


def test_indexer_relu_identities_against_matmul():
    q8, sq, w, k8, sk = _small_indexer_inputs()
    T, S = q8.shape[0], k8.shape[0]
    rows = list(range(T))
    neg_k8 = k8 ^ 0x80                                   # flip the sign bit: exact negation
    I_pos = oracle.indexer_scores(q8, sq, w, k8, sk, rows, q_pos0=S)   # every row sees all S keys
    I_neg = oracle.indexer_scores(q8, sq, w, neg_k8, sk, rows, q_pos0=S)
    lin, ab = _torch_linear_and_abs(q8, sq, w, k8, sk)
    np.testing.assert_allclose(I_pos - I_neg, lin, rtol=1e-12, atol=1e-9)
    np.testing.assert_allclose(I_pos + I_neg, ab, rtol=1e-12, atol=1e-9)


def test_indexer_scale_homogeneity_and_causal_mask():
    q8, sq, w, k8, sk = _small_indexer_inputs(seed=1)
    T, S = q8.shape[0], k8.shape[0]
    rows = list(range(T))
    base = oracle.indexer_scores(q8, sq, w, k8, sk, rows)
    # causal: row t sees s <= t only
    for t in rows:
        assert np.all(np.isfinite(base[t, : t + 1])) and np.all(np.isneginf(base[t, t + 1:]))
    sk2 = sk.clone()
    sk2[3] *= 2.0
    b2 = oracle.indexer_scores(q8, sq, w, k8, sk2, rows)
    np.testing.assert_allclose(b2[3:, 3], 2 * base[3:, 3], rtol=1e-14)
    m = np.isfinite(base)
    m[:, 3] = False
    assert np.array_equal(b2[m], base[m])
    b3 = oracle.indexer_scores(q8, sq, 4 * w, k8, sk, rows)       # power of two: exact in fp32
    assert np.array_equal(b3[np.isfinite(base)], 4 * base[np.isfinite(base)])


def test_indexer_single_head_closed_form():
    # H_I = 1, w = 1: I = ReLU(sq * sk * q.k); with q = e_0 * 2, k = e_0 * (+-3): q.k = +-6
    q8, sq = synth.encode_e4m3_per_token(torch.zeros(1, 1, 128))
    qv = torch.zeros(1, 1, 128)
    qv[0, 0, 0] = 2.0
    q8 = qv.to(torch.float8_e4m3fn).view(torch.uint8)
    kv = torch.zeros(2, 128)
    kv[0, 0], kv[1, 0] = 3.0, -3.0
    k8 = kv.to(torch.float8_e4m3fn).view(torch.uint8)
    sc = oracle.indexer_row(q8[0], np.array([0.5]), np.array([1.0]), k8, np.array([2.0, 2.0]), 2)
    assert sc.tolist() == [6.0, 0.0]


def test_fp8_dot_products_are_exact_in_f64():
    # e4m3 values are integers times 2^-9 with |integer| < 2^18, so a 128-term sum of
    # products fits in 53 bits: the oracle's f64 dot equals the exact integer sum.
    q8, sq, w, k8, sk = _small_indexer_inputs(seed=2, T=4, S=8, H_I=2)
    qi = (oracle.e4m3_to_f64(q8.numpy()) * 512).astype(np.int64)
    ki = (oracle.e4m3_to_f64(k8.numpy()) * 512).astype(np.int64)
    exact = np.einsum("tjd,sd->tjs", qi, ki)  # int64 exact
    f64 = np.einsum("tjd,sd->tjs", oracle.e4m3_to_f64(q8.numpy()), oracle.e4m3_to_f64(k8.numpy())) * 2.0 ** 18
    assert np.array_equal(exact.astype(np.float64), f64)


# ---------------------------------------------------------------- top-k

def _brute_valid_sets(scores, k):
    n = len(scores)
    m = min(k, n)
    out = []
    for sub in itertools.combinations(range(n), m):
        rest = [s for s in range(n) if s not in sub]
        if not rest or min(scores[list(sub)]) >= max(scores[rest]):
            out.append(set(sub))
    return out


@pytest.mark.parametrize("seed", range(6))
def test_topk_brute_force_distinct_scores(seed):
    rng = np.random.default_rng(seed)
    for n in range(1, 11):
        for k in range(1, 5):
            sc = rng.standard_normal(n)
            valid = _brute_valid_sets(sc, k)
            assert len(valid) == 1
            assert set(oracle.topk_row(sc, k).tolist()) == valid[0]


@pytest.mark.parametrize("seed", range(4))
def test_topk_brute_force_ties_and_lower_index_rule(seed):
    rng = np.random.default_rng(100 + seed)
    for n in range(1, 11):
        for k in range(1, 5):
            sc = rng.integers(0, 3, n).astype(np.float64)
            got = set(oracle.topk_row(sc, k).tolist())
            valid = _brute_valid_sets(sc, k)
            assert got in valid
            # ties at the threshold go to the lower positions
            thr = min(sc[list(got)])
            tied = sorted(s for s in range(n) if sc[s] == thr)
            taken = sorted(s for s in got if sc[s] == thr)
            assert taken == tied[: len(taken)]


def test_topk_rows_padding():
    sc = np.array([[1.0, 5.0, -np.inf, -np.inf], [3.0, 2.0, 9.0, 1.0]])
    out = oracle.topk_rows(sc, [2, 4], 3)
    assert out[0].tolist() == [1, 0, -1]
    assert out[1].tolist() == [2, 0, 1]


# ---------------------------------------------------------------- attention

def _sdpa_f64(q_bf16, kv_bf16, mask=None, causal=False, scale=1 / math.sqrt(192)):
    q = q_bf16.double().permute(1, 0, 2)[None]            # [1, H, T, 576]
    k = kv_bf16.double()[None, None].expand(1, q.shape[1], -1, -1)
    v = kv_bf16.double()[None, None, :, :512].expand(1, q.shape[1], -1, -1)
    o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, is_causal=causal, scale=scale)
    return o[0].permute(1, 0, 2).numpy()                   # [T, H, 512]


def test_dense_limit_equals_causal_sdpa_config1():
    cfg = synth.config(1, k=256)                            # k >= L: DSA is dense causal attention
    inp = synth.prefill_inputs(cfg)
    ref = _sdpa_f64(inp["q"], inp["kv"], causal=True, scale=cfg.scale)
    for t in [0, 1, 7, 100, 255]:
        r = oracle.prefill_row(inp, t, cfg.k, cfg.scale)
        assert sorted(r["idx"].tolist()) == list(range(t + 1))
        np.testing.assert_allclose(r["o"], ref[t], rtol=1e-12, atol=1e-12)


def test_dense_causal_row_equals_causal_sdpa_with_offset():
    # rows of a chunk that starts at absolute position q_pos0 see keys 0 .. q_pos0 + i
    g = torch.Generator().manual_seed(11)
    H, S, q_pos0, T = 6, 300, 170, 130
    q = torch.randn(T, H, 576, generator=g).to(torch.bfloat16)
    kv = torch.randn(S, 576, generator=g).to(torch.bfloat16)
    mask = torch.arange(S)[None, :] <= (q_pos0 + torch.arange(T))[:, None]
    ref = _sdpa_f64(q, kv, mask=mask[None, None], scale=0.05)
    for i in [0, 1, 63, 64, 129]:
        o, lse = oracle.dense_causal_row(q[i], kv, q_pos0 + i, 0.05)
        np.testing.assert_allclose(o, ref[i], rtol=1e-12, atol=1e-12)
        logits = 0.05 * (q[i].double() @ kv[: q_pos0 + i + 1].double().T)
        np.testing.assert_allclose(lse, torch.logsumexp(logits, dim=1).numpy(), rtol=1e-13)


def test_sparse_attention_equals_masked_sdpa():
    cfg = synth.config(1)
    inp = synth.prefill_inputs(cfg)
    rows = [0, 30, 64, 65, 200, 255]
    mask = torch.zeros(len(rows), cfg.L, dtype=torch.bool)
    outs = []
    for i, t in enumerate(rows):
        r = oracle.prefill_row(inp, t, cfg.k, cfg.scale)
        assert len(r["idx"]) == min(cfg.k, t + 1)
        assert r["idx"].max() <= t                          # causality of the selection
        mask[i, torch.as_tensor(r["idx"])] = True
        outs.append(r["o"])
    ref = _sdpa_f64(inp["q"][rows], inp["kv"], mask=mask[None, None], scale=cfg.scale)
    np.testing.assert_allclose(np.stack(outs), ref, rtol=1e-12, atol=1e-12)


def test_attention_single_row_returns_value_and_lse():
    g = torch.Generator().manual_seed(3)
    q = torch.randn(4, 576, generator=g).to(torch.bfloat16)
    c = torch.randn(1, 576, generator=g).to(torch.bfloat16)
    o, lse = oracle.attention_row(q, c, 0.1)
    assert np.array_equal(o, np.repeat(c.double().numpy()[:, :512], 4, axis=0))
    np.testing.assert_allclose(lse, 0.1 * (q.double() @ c.double().T).numpy()[:, 0], rtol=1e-14)


def test_attention_is_order_invariant_and_lse_matches_logsumexp():
    g = torch.Generator().manual_seed(4)
    q = torch.randn(3, 576, generator=g).to(torch.bfloat16)
    c = torch.randn(50, 576, generator=g).to(torch.bfloat16)
    o1, l1 = oracle.attention_row(q, c, 0.07)
    perm = torch.randperm(50, generator=g)
    o2, l2 = oracle.attention_row(q, c[perm], 0.07)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)
    ref_lse = torch.logsumexp(0.07 * (q.double() @ c.double().T), dim=1).numpy()
    np.testing.assert_allclose(l1, ref_lse, rtol=1e-13)


# ---------------------------------------------------------------- indexer loss

def test_indexer_kl_matches_torch_softmax_and_scipy_rel_entr():
    from scipy.special import rel_entr, softmax
    g = torch.Generator().manual_seed(31)
    H, n, scale = 5, 40, 0.09
    q = torch.randn(H, 576, generator=g).to(torch.bfloat16)
    c = torch.randn(n, 576, generator=g).to(torch.bfloat16)
    I = torch.randn(n, generator=g, dtype=torch.float64) * 3
    p, kl = oracle.indexer_kl_row(q, c, I.numpy(), scale)
    # head average of each head's attention weights (each head's weights sum to one)
    p_ref = torch.softmax(scale * (q.double() @ c.double().T), dim=1).mean(dim=0).numpy()
    np.testing.assert_allclose(p, p_ref, rtol=1e-12, atol=1e-15)
    assert abs(p.sum() - 1.0) < 1e-12
    kl_ref = rel_entr(p_ref, softmax(I.numpy())).sum()
    assert abs(kl - kl_ref) <= 1e-12 * max(1.0, abs(kl_ref))


def test_indexer_kl_vanishes_when_the_indexer_reproduces_the_target():
    g = torch.Generator().manual_seed(32)
    q = torch.randn(3, 576, generator=g).to(torch.bfloat16)
    c = torch.randn(25, 576, generator=g).to(torch.bfloat16)
    p, _ = oracle.indexer_kl_row(q, c, np.zeros(25), 0.05)
    _, kl = oracle.indexer_kl_row(q, c, np.log(p) + 3.7, 0.05)   # softmax(ln p + const) = p
    assert abs(kl) < 1e-12


def test_indexer_kl_binary_closed_form():
    # one head, two keys: p = (sigmoid(a - b), ...), q = (sigmoid(x - y), ...)
    q = torch.zeros(1, 576)
    q[0, 0] = 2.0
    c = torch.zeros(2, 576)
    c[0, 0], c[1, 0] = 1.0, -0.5
    a, b = 0.25 * 2.0 * 1.0, 0.25 * 2.0 * -0.5
    x, y = 1.3, -0.4
    p1, q1 = 1 / (1 + math.exp(-(a - b))), 1 / (1 + math.exp(-(x - y)))
    want = p1 * math.log(p1 / q1) + (1 - p1) * math.log((1 - p1) / (1 - q1))
    p, kl = oracle.indexer_kl_row(q.to(torch.bfloat16), c.to(torch.bfloat16), [x, y], 0.25)
    np.testing.assert_allclose(p, [p1, 1 - p1], rtol=1e-14)
    assert abs(kl - want) < 1e-14


def test_indexer_loss_rows_dense_variant_and_nonnegativity():
    cfg = synth.config(1, k=16)
    inp = synth.prefill_inputs(cfg)
    for t in [0, 5, 15, 16, 100, 255]:
        d = oracle.indexer_loss_prefill_row(inp, t, cfg.k, cfg.scale, dense=True)
        assert d["keys"].tolist() == list(range(t + 1))
        full = oracle.indexer_loss_prefill_row(inp, t, cfg.k, cfg.scale, idx_override=np.arange(t + 1))
        np.testing.assert_array_equal(d["p"], full["p"])
        assert d["kl"] == full["kl"] and d["kl"] >= 0
        sp = oracle.indexer_loss_prefill_row(inp, t, cfg.k, cfg.scale)
        assert len(sp["keys"]) == min(t + 1, cfg.k) and sp["kl"] >= -1e-15
        assert abs(sp["p"].sum() - 1) < 1e-12


# ---------------------------------------------------------------- paging / decode

def test_decode_paged_equals_contiguous_prefill_row():
    cfg = synth.config(3, B=3, ctx=300, k=64, H=8, H_I=4)
    inp = synth.decode_inputs(cfg)
    page = cfg.page
    for b in range(cfg.B):
        n = int(inp["seq_lens"][b])
        r = oracle.decode_row(inp, b, cfg.k, cfg.scale)
        # lay the sequence out contiguously by hand and run it as the last prefill row
        bt = inp["block_table"][b].long()
        pos = torch.arange(n)
        phys = bt[pos // page] * page + pos % page
        pre = dict(q8=inp["q8"][b:b + 1].expand(n, -1, -1), q_scale=inp["q_scale"][b:b + 1].expand(n, -1),
                   w=inp["w"][b:b + 1].expand(n, -1),
                   k8=inp["k8_cache"].reshape(-1, 128)[phys], k_scale=inp["k_scale_cache"].reshape(-1)[phys],
                   q=inp["q"][b:b + 1].expand(n, -1, -1), kv=inp["kv_cache"].reshape(-1, 576)[phys])
        r2 = oracle.prefill_row(pre, n - 1, cfg.k, cfg.scale)
        assert np.array_equal(r["scores"], r2["scores"])
        assert np.array_equal(r["idx"], r2["idx"])
        assert np.array_equal(r["o"], r2["o"])


def test_decode_mixed_lengths_block_table_is_a_permutation():
    cfg = synth.config(5, B=4, ctx_lo=100, ctx_hi=700, k=64, H=8, H_I=4)
    inp = synth.decode_inputs(cfg)
    bt, lens = inp["block_table"], inp["seq_lens"]
    pages = []
    for b in range(cfg.B):
        n = (int(lens[b]) + cfg.page - 1) // cfg.page
        assert torch.all(bt[b, :n] >= 0) and torch.all(bt[b, n:] == -1)
        pages += bt[b, :n].tolist()
    assert sorted(pages) == list(range(inp["k8_cache"].shape[0]))
    for b in range(cfg.B):
        r = oracle.decode_row(inp, b, cfg.k, cfg.scale)
        assert len(r["idx"]) == min(cfg.k, int(lens[b])) and r["idx"].max() < int(lens[b])


# ---------------------------------------------------------------- work counts

@pytest.mark.parametrize("L,k", [(1, 1), (5, 2), (256, 64), (4096, 2048), (131072, 2048), (100, 1000)])
def test_work_counts_closed_form(L, k):
    m = min(L, k)
    closed = m * (m + 1) // 2 + (L - m) * k
    assert oracle.selected_pairs(L, k) == closed
    assert oracle.causal_pairs(L) == L * (L + 1) // 2


def test_work_counts_golden_128k():
    with open(os.path.join(GOLDEN, "work_counts_128k.json")) as f:
        gold = json.load(f)
    L, k = gold["L"], gold["k"]
    assert oracle.selected_pairs(L, k) == gold["selected_pairs_causal"]
    assert oracle.causal_pairs(L) == gold["causal_pairs"]
    assert L * k / (L * L) == gold["noncausal_ratio"]


def test_selected_count_matches_oracle_selection_config1():
    cfg = synth.config(1)
    inp = synth.prefill_inputs(cfg)
    tot = sum(len(oracle.prefill_row(inp, t, cfg.k, cfg.scale)["idx"]) for t in range(cfg.L))
    assert tot == oracle.selected_pairs(cfg.L, cfg.k)


# ---------------------------------------------------------------- comparison rule

def test_index_set_rule_accepts_only_near_ties():
    sc = np.array([10.0, 9.0, 8.0, 7.99999, 1.0, 0.0])
    o = oracle.topk_row(sc, 3)                              # {0,1,2}
    assert oracle.index_sets_match(sc, o, np.array([0, 1, 3]))[0]      # 7.99999 within 1e-4 of 8
    assert not oracle.index_sets_match(sc, o, np.array([0, 1, 4]))[0]
    assert not oracle.index_sets_match(sc, o, np.array([0, 1, 1]))[0]
    assert not oracle.index_sets_match(sc, o, np.array([0, 1]))[0]
    z = np.array([5.0, 0.0, 0.0, -1.0])
    oz = oracle.topk_row(z, 2)
    assert oracle.index_sets_match(z, oz, np.array([0, 2]))[0]         # exact zero tie
    assert not oracle.index_sets_match(z, oz, np.array([0, 3]))[0]


# ---------------------------------------------------------------- golden regression

def test_config1_golden_fixture():
    with open(os.path.join(GOLDEN, "config1_oracle.json")) as f:
        gold = json.load(f)
    cfg = synth.config(1)
    inp = synth.prefill_inputs(cfg)
    for row in gold["rows"]:
        r = oracle.prefill_row(inp, row["t"], cfg.k, cfg.scale)
        assert sorted(r["idx"].tolist()) == row["idx_sorted"]
        np.testing.assert_allclose(r["o"].sum(axis=1), row["o_rowsum"], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(r["lse"], row["lse"], rtol=1e-12)


# ---------------------------------------------------------------- the parity checker itself

def test_attention_error_known_values_mixed_signs_over_rows_and_heads():
    # Two tokens x three heads x four value dims.  The reference is far from zero and differs
    # per element, so a relative error, a signed difference or a mean over the wrong axis gives
    # a different pair of numbers than the one written out here.
    ref = np.arange(24, dtype=np.float64).reshape(2, 3, 4) * 0.5 + 3.0
    delta = np.zeros((2, 3, 4))
    delta[0, 0, 0] = +0.25
    delta[0, 2, 3] = -0.75    # the largest error is negative: a signed max would report +0.5
    delta[1, 1, 2] = +0.5
    delta[1, 2, 1] = -0.125
    other = ref + delta
    mx, mean = oracle.attention_error(ref, other)
    assert mx == 0.75
    assert mean == (0.25 + 0.75 + 0.5 + 0.125) / 24          # = 1.625 / 24 over all 24 entries
    # symmetric in its arguments, zero on identical inputs, and bf16 output taken at its value
    assert oracle.attention_error(other, ref) == (mx, mean)
    assert oracle.attention_error(ref, ref) == (0.0, 0.0)
    ob = torch.tensor(other).to(torch.bfloat16).double().numpy()
    mx_b, _ = oracle.attention_error(ref, ob)
    assert mx_b == np.abs(ref - ob).max()
    # planted mistakes the checker must not make: each gives a different pair
    assert (float(delta.max()), float(delta.mean())) != (mx, mean)                 # signed
    assert float((np.abs(delta) / np.abs(ref)).max()) != mx                         # relative
    assert float(np.abs(delta).mean(axis=-1).max()) != mean                         # wrong axis
    assert oracle.attention_error(np.zeros((0, 4)), np.zeros((0, 4))) == (0.0, 0.0)


def test_indexer_loss_sparse_path_scrambled_selection_against_torch_and_scipy():
    """The sparse stage over a selection that is neither a prefix nor in order and holds -1 pads:
    the target must come from the rows of those positions and the indexer distribution from the
    scores at the same positions, slot by slot."""
    from scipy.special import rel_entr, softmax
    cfg = synth.config(1, k=16)
    inp = synth.prefill_inputs(cfg)
    t = 200
    rng = np.random.default_rng(7)
    keys = rng.permutation(t + 1)[:16]                       # 16 scrambled positions <= t
    sel = np.full(24, -1, np.int64)
    sel[: len(keys)] = keys                                  # padded like a selection row
    got = oracle.indexer_loss_prefill_row(inp, t, cfg.k, cfg.scale, idx_override=sel)
    assert got["keys"].tolist() == keys.tolist()
    # target: torch's per-head softmax over the selected latent rows, averaged over heads
    q = inp["q"][t].double()
    c = inp["kv"][torch.as_tensor(keys)].double()
    p_ref = torch.softmax(cfg.scale * (q @ c.T), dim=1).mean(dim=0).numpy()
    np.testing.assert_allclose(got["p"], p_ref, rtol=1e-12, atol=1e-15)
    # indexer scores at the same positions from torch's FP8 decode and a matmul
    q8 = inp["q8"][t].view(torch.float8_e4m3fn).double()                       # [H_I, 128]
    k8 = inp["k8"][torch.as_tensor(keys)].view(torch.float8_e4m3fn).double()   # [16, 128]
    dots = (q8 @ k8.T) * inp["q_scale"][t].double()[:, None] * inp["k_scale"][torch.as_tensor(keys)].double()[None]
    I_ref = (inp["w"][t].double()[:, None] * torch.relu(dots)).sum(0).numpy()
    kl_ref = rel_entr(p_ref, softmax(I_ref)).sum()
    assert abs(got["kl"] - kl_ref) <= 1e-12 * max(1.0, abs(kl_ref))
    # a selection in another order gives the same KL with p permuted alongside
    perm = rng.permutation(len(keys))
    sel2 = np.concatenate([keys[perm], [-1] * 8])
    got2 = oracle.indexer_loss_prefill_row(inp, t, cfg.k, cfg.scale, idx_override=sel2)
    np.testing.assert_allclose(got2["p"], got["p"][perm], rtol=1e-13, atol=1e-16)
    assert abs(got2["kl"] - got["kl"]) <= 1e-12 * max(1.0, abs(kl_ref))
    # misaligned scores (the same positions' scores rolled by one slot) change the KL
    I_bad = np.roll(I_ref, 1)
    assert abs(rel_entr(p_ref, softmax(I_bad)).sum() - got["kl"]) > 1e-6


# ---------------------------------------------------------------- attention backward

def _sdpa_grads(q, kv, idx, do, scale):
    """dq and d(latent rows) from torch autograd in float64 through SDPA with a boolean mask built
    from the selection (MQA: one latent row per position, keys = all 576 dims, values = first 512)."""
    T, H, D = q.shape
    S = kv.shape[0]
    qq = q.double().clone().requires_grad_(True)
    kk = kv.double().clone().requires_grad_(True)
    mask = torch.zeros(T, S, dtype=torch.bool)
    for t in range(T):
        sel = idx[t][idx[t] >= 0]
        mask[t, sel] = True
    out = F.scaled_dot_product_attention(qq.transpose(0, 1)[None], kk[None, None].expand(1, H, S, D),
                                         kk[:, :512][None, None].expand(1, H, S, 512),
                                         attn_mask=mask[None, None], scale=scale)        # [1, H, T, 512]
    out[0].transpose(0, 1).backward(do.double())
    return qq.grad.numpy(), kk.grad.numpy()


def test_attention_backward_matches_torch_autograd_through_masked_sdpa():
    g = torch.Generator().manual_seed(51)
    T, H, S, k, scale = 6, 5, 40, 9, 0.06
    q = torch.randn(T, H, 576, generator=g).to(torch.bfloat16)
    kv = torch.randn(S, 576, generator=g).to(torch.bfloat16)
    do = torch.randn(T, H, 512, generator=g).to(torch.bfloat16)
    idx = torch.full((T, k + 3), -1, dtype=torch.int64)
    for t in range(T):
        n = [k, 3, k, 1, k, 7][t]
        idx[t, :n] = torch.randperm(S, generator=g)[:n]      # overlapping selections, scrambled order
    dq, dkv = oracle.sparse_attention_backward(q, kv, idx.numpy(), do, scale)
    dq_ref, dkv_ref = _sdpa_grads(q, kv, idx, do, scale)
    np.testing.assert_allclose(dq, dq_ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dkv, dkv_ref, rtol=1e-10, atol=1e-12)
    # rows never selected get no gradient; the value role only touches the first 512 dims
    unused = np.setdiff1d(np.arange(S), idx[idx >= 0].numpy())
    assert np.all(dkv[unused] == 0)


def test_attention_backward_matches_finite_differences():
    # float64 inputs (the oracle takes them as they are), central differences of L = <do, o>
    rng = np.random.default_rng(52)
    H, n, scale = 3, 7, 0.3
    q = rng.standard_normal((H, 576))
    c = rng.standard_normal((n, 576))
    do = rng.standard_normal((H, 512))
    dq, dc = oracle.attention_row_backward(q, c, do, scale)

    def loss(qx, cx):
        z = scale * (qx @ cx.T)
        p = np.exp(z - z.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        return float(np.sum(do * (p @ cx[:, :512])))

    eps = 1e-6
    for (h, d) in [(0, 0), (1, 300), (2, 575), (0, 511), (2, 512)]:
        e = np.zeros_like(q)
        e[h, d] = eps
        fd = (loss(q + e, c) - loss(q - e, c)) / (2 * eps)
        assert abs(fd - dq[h, d]) <= 1e-6 * max(1.0, abs(fd)), (h, d, fd, dq[h, d])
    for (s, d) in [(0, 0), (3, 100), (6, 511), (6, 512), (1, 575)]:
        e = np.zeros_like(c)
        e[s, d] = eps
        fd = (loss(q, c + e) - loss(q, c - e)) / (2 * eps)
        assert abs(fd - dc[s, d]) <= 1e-6 * max(1.0, abs(fd)), (s, d, fd, dc[s, d])


def test_attention_backward_special_cases():
    g = torch.Generator().manual_seed(53)
    q = torch.randn(4, 576, generator=g).to(torch.bfloat16)
    c = torch.randn(1, 576, generator=g).to(torch.bfloat16)
    do = torch.randn(4, 512, generator=g).to(torch.bfloat16)
    # one selected row: the softmax is constant (p = 1), so dq = 0 and dc = [sum_h do_h, 0]
    dq, dc = oracle.attention_row_backward(q, c, do, 0.1)
    assert np.all(dq == 0)
    np.testing.assert_allclose(dc[0, :512], do.double().sum(0).numpy(), rtol=1e-14)
    assert np.all(dc[0, 512:] == 0)
    # an empty selection: no gradient at all
    dq, dc = oracle.attention_row_backward(q, c[:0], do, 0.1)
    assert np.all(dq == 0) and dc.shape == (0, 576)
    # a zero output gradient gives zero gradients
    c2 = torch.randn(5, 576, generator=g).to(torch.bfloat16)
    dq, dc = oracle.attention_row_backward(q, c2, torch.zeros(4, 512), 0.1)
    assert np.all(dq == 0) and np.all(dc == 0)
