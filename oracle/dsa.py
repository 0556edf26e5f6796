"""Float64 reference implementation of the DSA forward (test infrastructure only).

Page names used in citations:
  [digest]  freezhihu.org/question/1978819912970555965 (V3.2 technical-report digest)
  [2048ai]  2048ai.net/692e6ad2791c233193d1cff9.html (DeepSeek v3.2 analysis)

Inputs are taken as raw bits (FP8 e4m3 bytes, bf16 as uint16 or torch bf16)
and decoded here from the formats' definitions, so nothing of the CUDA path or
of torch's conversions is reused.
"""
from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------
# Format decoders (definitions of the formats, not of the method)
# ----------------------------------------------------------------------------


def e4m3_to_f64(b) -> np.ndarray:
    """Decode FP8 e4m3 (the 'fn' variant: no infinities) bytes to float64.

    Bit layout: sign(1) exponent(4, bias 7) mantissa(3).  Exponent 0 holds the
    subnormals m/8 * 2^-6; exponent 15 with mantissa 7 is NaN; every other code
    is (1 + m/8) * 2^(e-7).
    """
    b = np.asarray(b, dtype=np.uint8)
    sign = (b >> 7).astype(np.int64)
    e = ((b >> 3) & 0xF).astype(np.int64)
    m = (b & 0x7).astype(np.float64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64)))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


def bf16_bits_to_f64(u) -> np.ndarray:
    """Decode bf16 values, given as their 16-bit patterns, to float64 (bf16 is the top half of fp32)."""
    u = np.asarray(u)
    if u.dtype != np.uint16:
        u = u.view(np.uint16)
    return (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _as_np(x):
    """torch tensor or array -> numpy array of the raw storage (bf16 -> uint16 bits)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16)
            if x.dtype == torch.uint8:
                return x.numpy()
            return x.numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x)


# ----------------------------------------------------------------------------
# Lightning indexer  ([digest] §2.1.1, indexer equation)
# ----------------------------------------------------------------------------


def indexer_row(q8_t, q_scale_t, w_t, k8, k_scale, n: int) -> np.ndarray:
    """Scores I[t, s] of one query token against keys s = 0 .. n-1.

    q8_t [H_I, d] e4m3 bytes, q_scale_t [H_I], w_t [H_I], k8 [>=n, d] bytes,
    k_scale [>=n].  Each head's logit is the dot product of the decoded FP8
    vectors times the two per-token scales; the score is the head-weighted sum
    of the ReLU of those logits:  I = sum_j w_j * max(0, sq_j * sk_s * q_j . k_s).
    """
    q = e4m3_to_f64(_as_np(q8_t))                        # [H_I, d]
    k = e4m3_to_f64(_as_np(k8)[:n])                      # [n, d]
    sq = np.asarray(_as_np(q_scale_t), np.float64)       # [H_I]
    sk = np.asarray(_as_np(k_scale), np.float64)[:n]     # [n]
    w = np.asarray(_as_np(w_t), np.float64)              # [H_I]
    logits = (q @ k.T) * sq[:, None] * sk[None, :]       # [H_I, n]; FP8 products are exact in f64
    return w @ np.maximum(logits, 0.0)                   # [n]


def indexer_scores(q8, q_scale, w, k8, k_scale, rows, q_pos0: int = 0, S: int | None = None) -> np.ndarray:
    """Dense score rows for prefill query rows `rows` (absolute position q_pos0 + t).

    Returns float64 [len(rows), S] with -inf at the positions a row may not see
    (s > its position), [digest] §2.1.1 "preceding tokens".
    """
    q8, q_scale, w, k8, k_scale = map(_as_np, (q8, q_scale, w, k8, k_scale))
    S = k8.shape[0] if S is None else S
    out = np.full((len(rows), S), -np.inf)
    for i, t in enumerate(rows):
        n = min(S, q_pos0 + int(t) + 1)
        out[i, :n] = indexer_row(q8[t], q_scale[t], w[t], k8, k_scale, n)
    return out


# ----------------------------------------------------------------------------
# Fine-grained top-k  ([digest] §2.1.2; k = 2048 in §2.3.2)
# ----------------------------------------------------------------------------


def topk_row(scores: np.ndarray, k: int) -> np.ndarray:
    """Positions of the min(k, n) largest scores of one row (n = len(scores)).

    Stable full sort on (-score, position): equal scores go to the lower position.
    """
    scores = np.asarray(scores, np.float64)
    n = scores.shape[0]
    order = np.lexsort((np.arange(n), -scores))
    return order[: min(k, n)].astype(np.int64)


def topk_rows(score_rows: np.ndarray, row_lens, k: int) -> np.ndarray:
    """Top-k over the first row_lens[i] entries of each row, -1 padded to k slots."""
    out = np.full((len(score_rows), k), -1, np.int64)
    for i, r in enumerate(score_rows):
        sel = topk_row(r[: int(row_lens[i])], k)
        out[i, : len(sel)] = sel
    return out


# ----------------------------------------------------------------------------
# Sparse MQA attention over the selected latent rows  ([digest] §2.1.2, §2.2)
# ----------------------------------------------------------------------------


def attention_row(q_t, latent_rows, scale: float, d_value: int = 512):
    """Softmax attention of one token's heads over the given latent rows.

    q_t [H, 576] bf16, latent_rows [n, 576] bf16 (every head sees the same rows:
    MQA mode).  logits = scale * q . c, softmax over the n rows, output
    o = sum p * c[:d_value].  Returns (o [H, d_value], lse [H]) in float64,
    lse = natural-log sum-exp of the scaled logits.  n == 0 gives zeros and -inf.
    """
    q = bf16_bits_to_f64(_as_np(q_t))
    c = bf16_bits_to_f64(_as_np(latent_rows))
    H = q.shape[0]
    if c.shape[0] == 0:
        return np.zeros((H, d_value)), np.full(H, -np.inf)
    logits = scale * (q @ c.T)                            # [H, n]
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    l = p.sum(axis=1, keepdims=True)
    o = (p @ c[:, :d_value]) / l
    return o, (m + np.log(l))[:, 0]


def dense_causal_row(q_t, kv, pos: int, scale: float, d_value: int = 512):
    """Dense causal attention of one token at absolute position `pos` over every latent row
    0..pos: the MQA-mode MLA computation that DSA replaces.

    vpshk.cn/20260227158.html (the dense V3.1 model's cost grows with the text, V3.2's stays
    nearly flat) and 10100.com/article/43188788 §1 ("actual effect": about half the long-context
    cost of the dense model) compare against it; it is DSA with every preceding row selected
    (k >= pos + 1).  Returns (o [H, d_value], lse [H]) like attention_row.
    """
    return attention_row(q_t, _as_np(kv)[: pos + 1], scale, d_value)


# ----------------------------------------------------------------------------
# Indexer training loss  ([digest] §2.3.1 dense warm-up, §2.3.2 sparse training)
# ----------------------------------------------------------------------------


def indexer_kl_row(q_t, latent_rows, scores_sel, scale: float):
    """Target distribution and KL term of one query token over a key set.

    [digest] §2.3.1: the main attention scores of all heads are summed and L1-normalised along the
    keys into the target p; the indexer is fitted by KL(p || Softmax(I)).  §2.3.2 applies the same
    loss over the selected set S_t only.  Reading: the "attention scores" are the per-head softmax
    probabilities over the set (so p is their head average).  latent_rows [n, 576] are the rows of
    the set, scores_sel [n] the indexer scores I[t, s] at the same keys.  Returns (p [n], kl);
    an empty set gives (empty, 0.0).  0 * ln 0 is taken as 0.
    """
    q = bf16_bits_to_f64(_as_np(q_t))
    c = bf16_bits_to_f64(_as_np(latent_rows))
    n = c.shape[0]
    if n == 0:
        return np.zeros(0), 0.0
    logits = scale * (q @ c.T)                                  # [H, n]
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    probs = e / e.sum(axis=1, keepdims=True)                    # softmax of each head over the set
    u = probs.sum(axis=0)                                       # summed over heads
    p = u / np.abs(u).sum()                                     # L1 normalisation along the keys
    I = np.asarray(scores_sel, dtype=np.float64)
    log_q = I - (I.max() + np.log(np.exp(I - I.max()).sum()))  # log Softmax(I) over the set
    nz = p > 0
    kl = float(np.sum(p[nz] * (np.log(p[nz]) - log_q[nz])))
    return p, kl


def indexer_loss_prefill_row(inp: dict, t: int, k: int, scale: float, q_pos0: int = 0, dense: bool = False,
                             idx_override=None):
    """Indexer-loss term of one prefill row at position q_pos0 + t.

    dense=False: the sparse training stage, over the row's top-k set S_t (the oracle's own selection,
    or idx_override).  dense=True: the dense warm-up stage, over every key s <= q_pos0 + t.
    Returns dict(p, kl, keys) with the target p over `keys` (positions, in set order).
    """
    S = inp["k8"].shape[0]
    n = min(S, q_pos0 + t + 1)
    sc = indexer_row(inp["q8"][t], inp["q_scale"][t], inp["w"][t], inp["k8"], inp["k_scale"], n)
    if dense:
        keys = np.arange(n)
    else:
        keys = topk_row(sc, k) if idx_override is None else np.asarray(idx_override)
        keys = keys[keys >= 0]
    kv = _as_np(inp["kv"])
    p, kl = indexer_kl_row(inp["q"][t], kv[keys], sc[keys], scale)
    return dict(p=p, kl=kl, keys=keys)


# ----------------------------------------------------------------------------
# Backward of the sparse attention over a fixed selection  ([digest] §2.3.2: in
# the sparse training stage the main model is optimised through DSA, i.e. the
# gradient flows through the attention over the selected rows S_t)
# ----------------------------------------------------------------------------


def _to_f64(x) -> np.ndarray:
    """bf16 values (torch bf16 or their uint16 bit patterns) decoded exactly; other floats as they are."""
    a = _as_np(x)
    if a.dtype == np.uint16:
        return bf16_bits_to_f64(a)
    return np.asarray(a, dtype=np.float64)


def attention_row_backward(q_t, latent_rows, do_t, scale: float, d_value: int = 512):
    """Gradients of one token's sparse attention with respect to its query and the selected rows.

    Forward (attention_row): z[h,s] = scale * q[h] . c[s], p = softmax_s(z), o[h] = sum_s p[h,s] c[s, :d_value].
    With the output gradient do [H, d_value], by the chain rule through the softmax:
        dp[h,s] = do[h] . c[s, :d_value]
        dz[h,s] = p[h,s] * (dp[h,s] - sum_s' p[h,s'] dp[h,s'])      (the sum equals do[h] . o[h])
        dq[h]   = scale * sum_s dz[h,s] c[s]
        dc[s]   = scale * sum_h dz[h,s] q[h]  +  [sum_h p[h,s] do[h], 0]   (key role + value role)
    q_t [H, 576], latent_rows [n, 576], do_t [H, d_value]: bf16 (decoded exactly) or float arrays.
    Returns (dq [H, 576], dc [n, 576]) in float64; n == 0 gives zeros and an empty dc.
    """
    q = _to_f64(q_t)
    c = _to_f64(latent_rows)
    do = _to_f64(do_t)
    H = q.shape[0]
    if c.shape[0] == 0:
        return np.zeros_like(q), np.zeros((0, q.shape[1]))
    z = scale * (q @ c.T)                                   # [H, n]
    e = np.exp(z - z.max(axis=1, keepdims=True))
    p = e / e.sum(axis=1, keepdims=True)
    v = c[:, :d_value]
    dp = do @ v.T                                           # [H, n]
    dz = p * (dp - (p * dp).sum(axis=1, keepdims=True))
    dq = scale * (dz @ c)                                   # [H, 576]
    dc = scale * (dz.T @ q)                                 # [n, 576]
    dc[:, :d_value] += p.T @ do
    assert dq.shape == (H, q.shape[1])
    return dq, dc


def sparse_attention_backward(q, kv, idx, do, scale: float, d_value: int = 512):
    """Gradients of the sparse attention of several tokens over their selections.

    q [T, H, 576], kv [S, 576], idx [T, k] (positions, -1 = empty slot; a position may appear in
    many rows), do [T, H, d_value].  Returns (dq [T, H, 576], dkv [S, 576]): dkv[s] sums the row
    gradient of every token whose selection holds s.
    """
    kv_np = _as_np(kv)
    idx = np.asarray(_as_np(idx), dtype=np.int64)
    T = idx.shape[0]
    dq = np.zeros((T,) + tuple(_as_np(q).shape[1:]))
    dkv = np.zeros((kv_np.shape[0], kv_np.shape[1]))
    for t in range(T):
        sel = idx[t][idx[t] >= 0]
        dq[t], dc = attention_row_backward(q[t], kv_np[sel], do[t], scale, d_value)
        np.add.at(dkv, sel, dc)
    return dq, dkv


# ----------------------------------------------------------------------------
# Whole forward, one query row at a time
# ----------------------------------------------------------------------------


def prefill_row(inp: dict, t: int, k: int, scale: float, q_pos0: int = 0, idx_override=None):
    """One prefill row: scores over s <= pos, top-k, attention over the chosen rows.

    `inp` holds the prefill tensors (see synth.prefill_inputs).  If
    idx_override is given (e.g. the GPU's index set), attention runs over it
    instead of the oracle's own selection.  Returns dict(scores, idx, o, lse).
    """
    S = inp["k8"].shape[0]
    n = min(S, q_pos0 + t + 1)
    sc = indexer_row(inp["q8"][t], inp["q_scale"][t], inp["w"][t], inp["k8"], inp["k_scale"], n)
    idx = topk_row(sc, k)
    use = idx if idx_override is None else np.asarray(idx_override)
    use = use[use >= 0]
    kv = _as_np(inp["kv"])
    o, lse = attention_row(inp["q"][t], kv[use], scale)
    return dict(scores=sc, idx=idx, o=o, lse=lse)


def prefill_rows(inp: dict, rows, k: int, scale: float, q_pos0: int = 0):
    return [prefill_row(inp, int(t), k, scale, q_pos0) for t in rows]


def decode_gather(cache, block_table_row, n: int, page: int):
    """Logical rows 0..n-1 of one sequence from a paged cache [pages, page, ...].

    Logical position p lives in physical page block_table_row[p // page], slot p % page.
    """
    cache = _as_np(cache)
    bt = np.asarray(_as_np(block_table_row), np.int64)
    p = np.arange(n)
    return cache[bt[p // page], p % page]


def decode_row(inp: dict, b: int, k: int, scale: float, idx_override=None):
    """Decode step of sequence b: the new token (position seq_lens[b]-1) scores
    its whole context (itself included), selects top-k, attends over them.
    Indices are logical positions."""
    n = int(_as_np(inp["seq_lens"])[b])
    page = inp["k8_cache"].shape[1]
    bt = _as_np(inp["block_table"])[b]
    k8 = decode_gather(inp["k8_cache"], bt, n, page)
    ks = decode_gather(inp["k_scale_cache"], bt, n, page)
    sc = indexer_row(inp["q8"][b], inp["q_scale"][b], inp["w"][b], k8, ks, n)
    idx = topk_row(sc, k)
    use = idx if idx_override is None else np.asarray(idx_override)
    use = use[use >= 0]
    kv = decode_gather(inp["kv_cache"], bt, n, page)
    o, lse = attention_row(inp["q"][b], kv[use], scale)
    return dict(scores=sc, idx=idx, o=o, lse=lse)


# ----------------------------------------------------------------------------
# Work counts  ([digest] §2.1.2 O(L^2) -> O(Lk); [2048ai] §1.2 128K example)
# ----------------------------------------------------------------------------


def selected_pairs(L: int, k: int) -> int:
    """Number of (t, s) pairs the sparse attention visits over a causal prefill: sum_t min(t+1, k)."""
    t = np.arange(L, dtype=np.int64)
    return int(np.minimum(t + 1, k).sum())


def causal_pairs(L: int) -> int:
    """Number of (t, s) pairs with s <= t: what dense causal attention visits."""
    return int(np.arange(1, L + 1, dtype=np.int64).sum())


# ----------------------------------------------------------------------------
# Comparison rules used by the parity tests
# ----------------------------------------------------------------------------


def index_sets_match(oracle_scores, oracle_idx, other_idx, rel_tol: float = 1e-4):
    """Compare another implementation's top-k set with the oracle's.

    Returns (ok, n_swapped, message).  Sets must have the same size and hold
    distinct, in-range positions.  A position in one set but not the other is
    accepted only at a genuine near-tie: its oracle score lies within rel_tol
    (relative) of the oracle's k-th score.  When the k-th score is exactly 0,
    only positions whose oracle score is exactly 0 are interchangeable.
    """
    sc = np.asarray(oracle_scores, np.float64)
    a = np.asarray(oracle_idx)
    a = a[a >= 0]
    b = np.asarray(other_idx)
    valid = b >= 0
    nb = int(valid.sum())
    if not np.all(valid[:nb]):
        return False, 0, "valid slots are not all first"
    b = b[valid]
    if nb != len(a):
        return False, 0, f"set size {nb} != {len(a)}"
    if len(np.unique(b)) != nb:
        return False, 0, "duplicate positions"
    if nb and (b.min() < 0 or b.max() >= len(sc)):
        return False, 0, "position out of range"
    if nb == 0:
        return True, 0, ""
    kth = sc[a].min()
    diff = np.setxor1d(a, b)
    if kth == 0.0:
        bad = diff[sc[diff] != 0.0]
    else:
        bad = diff[np.abs(sc[diff] - kth) > rel_tol * abs(kth)]
    if len(bad):
        return False, len(diff), f"{len(bad)} positions differ beyond the near-tie window (e.g. {bad[:4]})"
    return True, len(diff), ""


def attention_error(o_ref, o_other):
    """(max |err|, mean |err|) between a float64 reference and another output."""
    d = np.abs(np.asarray(o_ref, np.float64) - np.asarray(o_other, np.float64))
    return float(d.max()) if d.size else 0.0, float(d.mean()) if d.size else 0.0
