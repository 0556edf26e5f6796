"""Seeded synthetic inputs for the DeepSeek Sparse Attention (DSA) hot path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no scores, no selection, no attention).  Both the CUDA
path (through tests and the bench) and the float64 oracle read what it makes.

Workloads (sizes, distributions and seeds of the five configurations the hot
path is measured on):

  1  tiny prefill    L=256,   H_I=4,  k=64,   H=8,   8 planted keys per query, seed 0
  2  prefill 4K      L=4096,  H_I=64, k=2048, H=128, 32 planted keys per query, seed 1
  3  decode          B=64 sequences x 32768 cached tokens, 64-token pages, seed 2
  4  prefill 128K    L=131072, H_I=64, k=2048, H=128, lognormal(0, 0.5) key norms, seed 3
  5  mixed decode    B=32, lengths ~ U[8192, 131072], 16 planted keys/sequence, seed 4

Recipe (shared by all configurations):
  * indexer queries q^I [T, H_I, 128] and keys k^I [S, 128] ~ N(0, 1) in fp32;
  * planted keys: for each query t (in increasing t), min(P, t) distinct earlier
    positions s < t get k^I_s = q^I_{t,0} + 0.1 * N(0, I); later plants
    overwrite earlier ones;
  * lognormal key norms: k^I_s = g_s * z_s with g_s ~ LogNormal(0, 0.5);
  * FP8 e4m3 encoding with one fp32 scale per token: scale = absmax / 448
    (1 when the token is all zero), value = RNE(x / scale) clamped to +-448;
    the query scale covers all H_I * 128 entries of the token and is stored
    per (token, head) as [T, H_I] (all heads of a token share it);
  * head weights w [T, H_I] ~ N(0, 1 / H_I);
  * attention queries Q [T, H, 576] and latent rows KV [S, 576] ~ N(0, 1),
    rounded to bf16; the value is the first 512 latent dims;
  * decode: every page of the cache holds 64 tokens; the block table of each
    sequence lists its pages in logical order, drawn as one random
    permutation of all pages of the batch (pages are never shared).

Small configurations (and any configuration requested on the CPU) are drawn
with torch's CPU generator, so they are bit-for-bit reproducible; large ones
are drawn on the GPU with torch's CUDA generator in row chunks, and the
oracle receives copies of whatever rows it checks.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch

FP8_MAX = 448.0
D_LATENT = 576
D_VALUE = 512
D_INDEX = 128


@dataclass(frozen=True)
class Config:
    cid: int
    name: str
    mode: str            # "prefill" or "decode"
    seed: int
    H_I: int = 64
    k: int = 2048
    H: int = 128
    planted: int = 0
    lognormal_keys: bool = False
    # prefill
    L: int = 0
    # decode
    B: int = 0
    ctx: int = 0          # fixed context length (config 3)
    ctx_lo: int = 0       # uniform context lengths (config 5)
    ctx_hi: int = 0
    page: int = 64

    @property
    def scale(self) -> float:
        """Softmax scale 1/sqrt(192) used for every configuration."""
        return 1.0 / math.sqrt(192.0)


CONFIGS = {
    1: Config(1, "tiny prefill L=256", "prefill", seed=0, H_I=4, k=64, H=8, planted=8, L=256),
    2: Config(2, "prefill L=4096", "prefill", seed=1, planted=32, L=4096),
    3: Config(3, "decode B=64 x 32768", "decode", seed=2, B=64, ctx=32768),
    4: Config(4, "prefill L=131072", "prefill", seed=3, lognormal_keys=True, L=131072),
    5: Config(5, "mixed decode B=32, ctx~U[8192,131072]", "decode", seed=4, planted=16,
              B=32, ctx_lo=8192, ctx_hi=131072),
}


def config(cid: int, **overrides) -> Config:
    """The named configuration, optionally with sizes overridden (for reduced test cases)."""
    return replace(CONFIGS[cid], **overrides)


def _gen(cfg: Config, tensor_id: int, device, chunk: int = 0) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((cfg.seed * 1_000_003 + tensor_id * 7919 + chunk * 104_729) & 0x7FFF_FFFF_FFFF)
    return g


def _randn(cfg, tid, shape, device, rows_per_chunk=None, dtype=torch.float32):
    """N(0,1) draws in row chunks, each chunk from its own seeded generator."""
    n = shape[0]
    if rows_per_chunk is None or n <= rows_per_chunk:
        return torch.randn(shape, generator=_gen(cfg, tid, device), device=device).to(dtype)
    out = torch.empty(shape, dtype=dtype, device=device)
    for c, r0 in enumerate(range(0, n, rows_per_chunk)):
        r1 = min(n, r0 + rows_per_chunk)
        out[r0:r1] = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=_gen(cfg, tid, device, c),
                                 device=device).to(dtype)
    return out


def encode_e4m3_per_token(x: torch.Tensor):
    """FP8 e4m3 bytes and one fp32 scale per leading index (token).

    x: [N, ...] fp32.  Returns (uint8 [N, ...], fp32 [N]).  The cast itself is
    torch's float8_e4m3fn conversion (round to nearest even); values are clamped
    to the finite range first.
    """
    flat = x.reshape(x.shape[0], -1)
    amax = flat.abs().amax(dim=1)
    scale = torch.where(amax > 0, amax / FP8_MAX, torch.ones_like(amax))
    y = (flat / scale[:, None]).clamp_(-FP8_MAX, FP8_MAX)
    q = y.to(torch.float8_e4m3fn).view(torch.uint8).reshape(x.shape)
    return q, scale.float()


def _plant(cfg, kI, qI_head0, positions_upto, device, tid):
    """Planted keys: for each query (in order) overwrite min(P, t) distinct earlier keys.

    kI: [S, 128] fp32 (modified in place, logical key order); qI_head0: [T, 128];
    positions_upto[t] = number of earlier positions available to query t.
    """
    P = cfg.planted
    if P <= 0:
        return
    g = _gen(cfg, tid, "cpu")
    for t in range(qI_head0.shape[0]):
        n_avail = int(positions_upto[t])
        n = min(P, n_avail)
        if n == 0:
            continue
        pos = torch.randperm(n_avail, generator=g)[:n]
        noise = torch.randn((n, D_INDEX), generator=g)
        kI[pos.to(kI.device)] = qI_head0[t][None, :] + 0.1 * noise.to(kI.device)


def prefill_inputs(cfg: Config, device="cpu") -> dict:
    """All inputs of one prefill sequence, on `device`.

    Returns a dict of tensors:
      q8 [L,H_I,128] u8, q_scale [L,H_I] f32, w [L,H_I] f32, k8 [L,128] u8,
      k_scale [L] f32, q [L,H,576] bf16, kv [L,576] bf16.
    """
    assert cfg.mode == "prefill"
    L, H_I, H = cfg.L, cfg.H_I, cfg.H
    big = L > 8192
    gdev = device if big else "cpu"
    rc = 4096 if big else None
    qI = _randn(cfg, 1, (L, H_I, D_INDEX), gdev, rc)
    kI = _randn(cfg, 2, (L, D_INDEX), gdev, rc)
    if cfg.lognormal_keys:
        g = torch.exp(0.5 * _randn(cfg, 3, (L,), gdev))
        kI *= g[:, None]
    _plant(cfg, kI, qI[:, 0, :], torch.arange(L), gdev, tid=4)
    w = _randn(cfg, 5, (L, H_I), gdev) / math.sqrt(H_I)
    q8, sq = encode_e4m3_per_token(qI)
    del qI
    k8, sk = encode_e4m3_per_token(kI)
    del kI
    q = _randn(cfg, 6, (L, H, D_LATENT), gdev, 2048 if big else None, torch.bfloat16)
    kv = _randn(cfg, 7, (L, D_LATENT), gdev, rc, torch.bfloat16)
    out = dict(q8=q8, q_scale=sq[:, None].expand(L, H_I).contiguous(), w=w.float(), k8=k8,
               k_scale=sk, q=q, kv=kv)
    return {n: t.to(device).contiguous() for n, t in out.items()}


def _randn_rows(cfg, tid, shape, r0, r1, device, rows_per_chunk, dtype=torch.float32):
    """Rows [r0, r1) of _randn(cfg, tid, shape, device, rows_per_chunk, dtype), drawing only the
    chunks that cover them (bit-identical to the same rows of the full draw)."""
    out = []
    for c in range(r0 // rows_per_chunk, (r1 - 1) // rows_per_chunk + 1):
        c0 = c * rows_per_chunk
        c1 = min(shape[0], c0 + rows_per_chunk)
        x = torch.randn((c1 - c0,) + tuple(shape[1:]), generator=_gen(cfg, tid, device, c), device=device).to(dtype)
        out.append(x[max(r0, c0) - c0:min(r1, c1) - c0])
    return torch.cat(out)


def prefill_tail_inputs(cfg: Config, n_rows: int, device="cuda") -> dict:
    """The last n_rows query rows of a large prefill workload (L > 8192) with its full key side.

    Keys (k8, k_scale, kv) are those of prefill_inputs; the query-side tensors (q8, q_scale, w,
    q) are the rows [L - n_rows, L) of prefill_inputs, drawn without the rest.  For workloads
    without planted keys only (planting couples keys to every query).  Adds row0 = L - n_rows.
    """
    assert cfg.mode == "prefill" and cfg.L > 8192 and cfg.planted == 0
    L, H_I, H = cfg.L, cfg.H_I, cfg.H
    r0 = L - n_rows
    qI = _randn_rows(cfg, 1, (L, H_I, D_INDEX), r0, L, device, 4096)
    kI = _randn(cfg, 2, (L, D_INDEX), device, 4096)
    if cfg.lognormal_keys:
        g = torch.exp(0.5 * _randn(cfg, 3, (L,), device))
        kI *= g[:, None]
    w = (_randn(cfg, 5, (L, H_I), device) / math.sqrt(H_I))[r0:]
    q8, sq = encode_e4m3_per_token(qI)
    k8, sk = encode_e4m3_per_token(kI)
    del qI, kI
    q = _randn_rows(cfg, 6, (L, H, D_LATENT), r0, L, device, 2048, torch.bfloat16)
    kv = _randn(cfg, 7, (L, D_LATENT), device, 4096, torch.bfloat16)
    out = dict(q8=q8, q_scale=sq[:, None].expand(n_rows, H_I).contiguous(), w=w.float(), k8=k8, k_scale=sk, q=q,
               kv=kv)
    out = {n: t.to(device).contiguous() for n, t in out.items()}
    out["row0"] = r0
    return out


def decode_inputs(cfg: Config, device="cpu") -> dict:
    """All inputs of one decode step over a paged cache, on `device`.

    Returns a dict of tensors:
      q8 [B,H_I,128] u8, q_scale [B,H_I] f32, w [B,H_I] f32,
      k8_cache [pages,page,128] u8, k_scale_cache [pages,page] f32,
      kv_cache [pages,page,576] bf16, block_table [B,max_pages] i32 (-1 padded),
      seq_lens [B] i32 (attendable tokens including the new one; the query
      sits at position seq_lens[b]-1), q [B,H,576] bf16.
    """
    assert cfg.mode == "decode"
    B, H_I, H, page = cfg.B, cfg.H_I, cfg.H, cfg.page
    gcpu = _gen(cfg, 10, "cpu")
    if cfg.ctx:
        lens = torch.full((B,), cfg.ctx, dtype=torch.int64)
    else:
        lens = torch.randint(cfg.ctx_lo, cfg.ctx_hi + 1, (B,), generator=gcpu)
    n_pages_seq = (lens + page - 1) // page
    n_pages = int(n_pages_seq.sum())
    perm = torch.randperm(n_pages, generator=gcpu)
    max_pages = int(n_pages_seq.max())
    bt = torch.full((B, max_pages), -1, dtype=torch.int32)
    off = 0
    for b in range(B):
        n = int(n_pages_seq[b])
        bt[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    big = n_pages * page > 65536
    gdev = device if big else "cpu"
    qI = _randn(cfg, 11, (B, H_I, D_INDEX), gdev)
    kI = _randn(cfg, 12, (n_pages * page, D_INDEX), gdev, 1 << 18 if big else None)
    if cfg.lognormal_keys:
        kI *= torch.exp(0.5 * _randn(cfg, 13, (n_pages * page,), gdev))[:, None]
    if cfg.planted:
        gp = _gen(cfg, 14, "cpu")
        for b in range(B):
            n_avail = int(lens[b]) - 1            # positions strictly before the query
            n = min(cfg.planted, n_avail)
            logical = torch.randperm(n_avail, generator=gp)[:n]
            phys = bt[b, (logical // page)].long() * page + logical % page
            noise = torch.randn((n, D_INDEX), generator=gp)
            kI[phys.to(kI.device)] = qI[b, 0][None, :] + 0.1 * noise.to(kI.device)
    # tokens past the end of each sequence's last page are never read; zero them
    used = torch.zeros(n_pages * page, dtype=torch.bool)
    for b in range(B):
        n = int(lens[b])
        p = bt[b, : int(n_pages_seq[b])].long()
        slots = (p[:, None] * page + torch.arange(page)[None, :]).reshape(-1)[:n]
        used[slots] = True
    used = used.to(kI.device)
    kI[~used] = 0.0
    w = _randn(cfg, 15, (B, H_I), gdev) / math.sqrt(H_I)
    q8, sq = encode_e4m3_per_token(qI)
    k8, sk = encode_e4m3_per_token(kI)
    del kI
    kv = _randn(cfg, 16, (n_pages * page, D_LATENT), gdev, 1 << 16 if big else None, torch.bfloat16)
    kv[~used.to(kv.device)] = 0
    q = _randn(cfg, 17, (B, H, D_LATENT), gdev, None, torch.bfloat16)
    out = dict(q8=q8, q_scale=sq[:, None].expand(B, H_I).contiguous(), w=w.float(),
               k8_cache=k8.reshape(n_pages, page, D_INDEX), k_scale_cache=sk.reshape(n_pages, page),
               kv_cache=kv.reshape(n_pages, page, D_LATENT), block_table=bt,
               seq_lens=lens.to(torch.int32), q=q)
    return {n: t.to(device).contiguous() for n, t in out.items()}


def inputs(cfg: Config, device="cpu") -> dict:
    return prefill_inputs(cfg, device) if cfg.mode == "prefill" else decode_inputs(cfg, device)
