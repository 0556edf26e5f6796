"""Row-sharded prefill of one sequence over several GPUs (one process per GPU).

Each query row's indexer scores, selection and sparse attention depend only on that row and on the
keys at or before its position (freezhihu.org/question/1978819912970555965 §2.1.1: a query scores
its preceding tokens; §2.1.2: the top-k and the attention are per query).  A prefill therefore
splits by query rows: rank r takes the contiguous rows [r0, r1) and runs the fused forward on them
with q_pos0 = r0.  The only exchange is the keys: every rank holds the indexer keys, their scales
and the latent rows of its own positions (as a model produces them), and one all-gather gives each
rank all of them in its own HBM before any kernel reads them.  No kernel reads another GPU's memory.

The rows are balanced by time, not by count: a row at position t costs the indexer (t + 1) key
products, the top-k one read of its t + 1 scores, and the attention min(t + 1, k) selected rows, so
late rows cost more and rank 0 gets the most rows.  The cost model weighs each part by the rate its
kernel reaches on one B300 (argument `rates`).

This module is host logic and torch.distributed plumbing; the compute is dsa_forward's.
"""
from __future__ import annotations

import torch

# Throughputs of the three kernels on one B300 at 128K (indexer FP8 TFLOP/s, attention bf16 TFLOP/s,
# top-k GB/s of scores read): the weights of the row cost model.
DEFAULT_RATES = {"indexer_tflops": 1760.0, "attn_tflops": 560.0, "topk_gbs": 3400.0}


def _sum_prefix(n: int) -> int:
    """sum_{t=0}^{n-1} (t + 1)."""
    return n * (n + 1) // 2


def _sum_min(n: int, k: int) -> int:
    """sum_{t=0}^{n-1} min(t + 1, k)."""
    m = min(n, k)
    return m * (m + 1) // 2 + max(0, n - k) * k


def rows_cost(r0: int, r1: int, H_I: int, H: int, k: int, rates=None) -> float:
    """Modelled time (seconds) of the forward over query rows [r0, r1) of a prefill."""
    rates = rates or DEFAULT_RATES
    if r1 <= r0:
        return 0.0
    pairs = _sum_prefix(r1) - _sum_prefix(r0)              # causal (t, s) pairs of the rows
    sel = _sum_min(r1, k) - _sum_min(r0, k)                # selected pairs of the rows
    t_index = 2.0 * H_I * 128 * pairs / (rates["indexer_tflops"] * 1e12)
    t_topk = 4.0 * pairs / (rates["topk_gbs"] * 1e9)
    t_attn = 2.0 * H * (576 + 512) * sel / (rates["attn_tflops"] * 1e12)
    return t_index + t_topk + t_attn


def partition_rows(L: int, world: int, H_I: int, H: int, k: int, rates=None, align: int = 1):
    """Contiguous row ranges [(r0, r1), ...], one per rank, of (nearly) equal modelled cost.

    Boundaries are multiples of `align` (except the last, L); every row belongs to exactly one
    range, and ranges are in rank order.  A rank may get an empty range when L is tiny."""
    if L < 0 or world < 1 or align < 1:
        raise ValueError("L >= 0, world >= 1 and align >= 1 required")
    total = rows_cost(0, L, H_I, H, k, rates)
    bounds = [0]
    for r in range(1, world):
        target = total * r / world
        lo, hi = bounds[-1], L                              # smallest b with cost(0, b) >= target
        while lo < hi:
            mid = (lo + hi) // 2
            if rows_cost(0, mid, H_I, H, k, rates) < target:
                lo = mid + 1
            else:
                hi = mid
        b = lo
        # round to the alignment, towards the closer of the two candidates
        down = b // align * align
        up = min(L, down + align)
        b = down if abs(rows_cost(0, down, H_I, H, k, rates) - target) <= abs(
            rows_cost(0, up, H_I, H, k, rates) - target) else up
        bounds.append(max(b, bounds[-1]))
    bounds.append(L)
    return [(bounds[r], bounds[r + 1]) for r in range(world)]


def all_gather_rows(local: torch.Tensor, ranges, rank: int, out: torch.Tensor | None = None, group=None):
    """Every rank's rows, in position order: rank r contributes `local` = rows ranges[r] of a
    [L, ...] tensor; returns the whole [L, ...] tensor (into `out` if given) on every rank.

    The ranges may have different lengths: each rank's block is padded to the longest, one
    all-gather moves them, and each block is copied into its positions."""
    import torch.distributed as dist
    world = len(ranges)
    r0, r1 = ranges[rank]
    if local.shape[0] != r1 - r0:
        raise ValueError(f"rank {rank}: {local.shape[0]} local rows, range {ranges[rank]}")
    L = ranges[-1][1]
    longest = max(b - a for a, b in ranges)
    pad = torch.zeros((longest,) + tuple(local.shape[1:]), dtype=local.dtype, device=local.device)
    pad[: r1 - r0].copy_(local)
    blocks = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(blocks, pad, group=group)
    if out is None:
        out = torch.empty((L,) + tuple(local.shape[1:]), dtype=local.dtype, device=local.device)
    for r, (a, b) in enumerate(ranges):
        out[a:b].copy_(blocks[r][: b - a])
    return out
