#!/usr/bin/env python
"""Benchmark of the DSA hot path (indexer -> top-k -> sparse MLA attention) on B300.

Default run (N=1): one step = the whole forward of one 128K-token prefill sequence
(L=131072, H_I=64, d_I=128 FP8, k=2048, H=128, 576-d bf16 latent), inputs resident in HBM.
`value` is prefill tokens/s; the decode figure (query tokens/s, B=32 mixed contexts up to
128K) rides along under "decode".  Prints ONE JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--shard sequences|rows]

Under torchrun each rank runs its own 128K sequence (weak scaling, no collective on the
data path); the step time is the max over ranks.  With --shard rows the ranks instead split
one 128K sequence by query rows (strong scaling) and all-gather the keys every step.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "DSA prefill tokens/s & decode query-tok/s at 128K ctx; % of FP8/HBM roofline"
L2_BYTES = 126 * 1024 * 1024


# ------------------------------------------------------------------------------------ utils

def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=p["hbm_gbs"], bf16=p["bf16_tflops"], bf16_sus=p["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6400.0, bf16=1800.0, bf16_sus=1400.0, src="fallback")


def measure_fp8_peak(n=8192, sustain_s=2.0):
    """Dense FP8 e4m3 tensor throughput of this GPU, measured with torch._scaled_mm (cuBLASLt) on an
    n x n x n product with bf16 output: the best of 10 timed launches (burst, for kernels timed alone)
    and the mean over back-to-back launches for `sustain_s` seconds (sustained, for kernels timed
    inside a long step).  Returns dict(burst, sustained) in TFLOP/s, or None if FP8 GEMMs are not
    available."""
    try:
        g = torch.Generator(device="cuda").manual_seed(0)
        a = torch.randn((n, n), device="cuda", generator=g).to(torch.float8_e4m3fn)
        b = torch.randn((n, n), device="cuda", generator=g).to(torch.float8_e4m3fn).t()  # column-major
        one = torch.ones((), device="cuda")

        def mm():
            return torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)

        for _ in range(3):
            mm()
        torch.cuda.synchronize()
        flop = 2.0 * n ** 3
        best = float("inf")
        for _ in range(10):
            e0, e1 = _rec(), None
            mm()
            e1 = _rec()
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1))
        # sustained: as many launches as fill sustain_s at the burst rate, timed as one block
        reps = max(10, int(sustain_s * 1e3 / best))
        e0 = _rec()
        for _ in range(reps):
            mm()
        e1 = _rec()
        e1.synchronize()
        sus = e0.elapsed_time(e1) / reps
        del a, b
        return {"burst": flop / (best * 1e-3) / 1e12, "sustained": flop / (sus * 1e-3) / 1e12,
                "how": f"torch._scaled_mm e4m3 x e4m3 -> bf16, {n}^3, best of 10 / mean of {reps} back to back"}
    except (RuntimeError, AttributeError, TypeError) as e:  # pragma: no cover (no FP8 GEMM on this build)
        return {"error": str(e)[:200]}


# DRAM bytes (ncu dram__bytes_read.sum + dram__bytes_write.sum) of one kernel per unit of its work,
# from a capture of a given build of that kernel's source.  A figure is reported only while the
# source still hashes to the captured build; otherwise `traffic` is null.
TRAFFIC_CAPTURES = {
    # dram__bytes_read.sum + dram__bytes_write.sum of one launch over the last 1024 query rows of the 128K
    # prefill (each row against ~131K keys), per query row; the capture replays from a flushed L2, so
    # it overstates the steady state a little
    "sparse_attn": {"src": "3554cd61266f950e", "bytes_per_unit": (496.199e6 + 117.142e6) / 1024,
                    "capture": "ncu dram read + write, sparse_attn_kernel<0> over the 1024-row 128K tail, per row x rows"},
    "indexer": {"src": "1e33e0a7572a36a2", "bytes_per_unit": (63.660e6 + 477.555e6) / 1024,
                "capture": "ncu dram read + write, indexer_kernel<64> over the 1024-row 128K tail, per row x rows"},
    "topk": {"src": "dca55ab2c805bc87", "bytes_per_unit": (616.624e6 + 8.071e6) / 1024,
             "capture": "ncu dram read + write, topk_kernel over the 1024-row 128K tail, per row x rows"},
}


def _src_hash(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "sparse_attention_30_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {"sparse_attn": ["sparse_attn.cu", "attn_common.cuh", "dsa_ptx.cuh", "dsa_internal.h"],
                  "indexer": ["indexer.cu", "dsa_ptx.cuh", "dsa_internal.h"],
                  "topk": ["topk.cu", "dsa_ptx.cuh", "dsa_internal.h"]}


def traffic_for(kernel, units):
    """Captured DRAM bytes per unit x units, with the capture it comes from, or (None, reason)."""
    cap = TRAFFIC_CAPTURES.get(kernel)
    if cap is None:
        return None, "no capture of this kernel"
    if cap["src"] != _src_hash(KERNEL_SOURCES[kernel]):
        return None, "kernel source changed since the capture"
    return round(cap["bytes_per_unit"] * units), cap["capture"]


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "-i", str(index),
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        time.sleep(0.25)
        self.p.terminate()
        try:
            self.p.wait(5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.seek(0)
        rows = [r.split(", ") for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip() == "Active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "samples": len(sm),
                "reasons": sorted(reasons)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        rank, local = dist.get_rank(), int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        return dist, rank, ws, local
    return None, 0, 1, 0


def _max_over_ranks(dist, x: float) -> float:
    """Max of x over all ranks (the step time the job is charged), NCCL or gloo."""
    if dist is None:
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(base_seed: int, rank: int) -> int:
    """Each rank runs its own sequence of the same workload (weak scaling)."""
    return base_seed + 1000 * rank


def aggregate_tokens_per_s(tokens_per_rank: int, world_size: int, steps: int, max_ms: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * world_size * steps / (max_ms / 1e3)


def _barrier(dist):
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()


# ------------------------------------------------------------------------------------ work counts

def prefill_work(L, H_I, H, k):
    causal = L * (L + 1) // 2
    sel = sum(min(t + 1, k) for t in range(0, min(L, k))) + max(0, L - k) * k
    return dict(
        indexer_flop=2.0 * H_I * 128 * causal,
        topk_bytes=4.0 * causal + 4.0 * k * L,
        attn_flop=2.0 * H * (576 + 512) * sel,
        attn_bytes=L * H * 576 * 2.0 + L * H * 512 * 2.0 + 4.0 * k * L + 576 * 2.0 * L,
    )


def decode_work(lens, H_I, H, k):
    n = float(sum(lens))
    sel = float(sum(min(k, x) for x in lens))
    B = len(lens)
    return dict(
        indexer_bytes=n * (128 + 4) + 4.0 * n + B * H_I * (128 + 8),
        topk_bytes=4.0 * n + 4.0 * k * B,
        attn_bytes=sel * 1152 + B * H * 576 * 2.0 + B * H * 512 * 2.0 + 4.0 * k * B,
        attn_flop=2.0 * H * (576 + 512) * sel,
    )


# ------------------------------------------------------------------------------------ our arm

class PrefillRunner:
    """One 128K prefill step through the C ABI, stage by stage, with CUDA events per launch
    on the launching stream.  The launches are exactly those dsa_forward makes (same chunking)."""

    def __init__(self, dsa, d, cfg, chunk):
        self.dsa, self.d, self.cfg, self.chunk = dsa, d, cfg, chunk
        L = cfg.L
        ld = (L + 3) // 4 * 4
        self.scores = torch.empty((chunk, ld), dtype=torch.float32, device="cuda")
        self.idx = torch.empty((L, cfg.k), dtype=torch.int32, device="cuda")
        self.out = torch.empty((L, cfg.H, 512), dtype=torch.bfloat16, device="cuda")
        self.lse = torch.empty((L, cfg.H), dtype=torch.float32, device="cuda")
        self.n_chunks = (L + chunk - 1) // chunk
        self.launches = 2 * self.n_chunks + 1

    def step(self, events=None):
        dsa, d, cfg = self.dsa, self.d, self.cfg
        ev = events
        for c in range(self.n_chunks):
            r0 = c * self.chunk
            r1 = min(cfg.L, r0 + self.chunk)
            sc = self.scores[: r1 - r0]
            if ev is not None:
                ev["index"].append(_rec())
            dsa.index(d["q8"][r0:r1], d["q_scale"][r0:r1], d["w"][r0:r1], d["k8"], d["k_scale"], q_pos0=r0,
                      scores=sc)
            if ev is not None:
                ev["index"].append(_rec())
                ev["topk"].append(_rec())
            dsa.topk(sc, cfg.k, q_pos0=r0, n_cols=cfg.L, idx=self.idx[r0:r1])
            if ev is not None:
                ev["topk"].append(_rec())
        if ev is not None:
            ev["attn"].append(_rec())
        dsa.sparse_attn(d["q"], d["kv"], self.idx, cfg.scale, out=self.out, lse=self.lse)
        if ev is not None:
            ev["attn"].append(_rec())


def _rec():
    e = torch.cuda.Event(enable_timing=True)
    e.record()
    return e


def _pairs_ms(lst):
    return sum(a.elapsed_time(b) for a, b in zip(lst[0::2], lst[1::2]))


def run_ours(args, dist, rank, ws):
    import synth
    from sparse_attention_30_b300 import build
    build.build()
    import sparse_attention_30_b300 as dsa

    peaks = _peaks()
    if args.workload.startswith("decode"):
        # decode-only run (used for profiler captures of the decode kernels)
        res = bench_decode(dsa, synth, args, peaks, cid=5 if args.workload == "decode" else 3)
        return {"metric": "decode query-tok/s", "value": res["value"], "unit": "query-tok/s", "n_gpus": ws,
                "steps": max(10, args.steps), "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp8-e4m3 / bf16",
                "data": "synthetic", "config": {"workload": res["workload"]}, "decode": res}
    if args.workload == "prefill128k_tail":
        return bench_prefill_tail(dsa, synth, args, peaks)
    if args.workload == "dense_curve":
        return bench_dense_curve(dsa, synth, args, peaks)
    if args.workload == "indexer_loss":
        return bench_indexer_loss(dsa, synth, args, peaks)
    if args.workload.startswith("backward"):
        res = bench_backward(dsa, synth, args, peaks, L=131072 if args.workload == "backward128k" else 4096)
        return {"metric": "sparse attention backward tokens/s", "value": res["tokens_per_s"], "unit": "tokens/s",
                "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16 (fp32 accum, fp32 dkv atomics)", "data": "synthetic",
                "config": {"workload": res["workload"]}, "backward": res}
    if args.shard == "rows":
        return bench_prefill_rows(dsa, synth, args, peaks, dist, rank, ws)
    cid = {"prefill128k": 4, "prefill4k": 2}[args.workload]
    cfg = synth.config(cid)
    if rank:
        cfg = synth.config(cid, seed=rank_seed(cfg.seed, rank))
    d = synth.prefill_inputs(cfg, device="cuda")
    fp8 = measure_fp8_peak() if not args.no_fp8_peak else {"error": "not measured (--no-fp8-peak)"}
    # the step the job is charged: dsa_forward (the library's fused entry point) over the sequence
    idx = torch.empty((cfg.L, cfg.k), dtype=torch.int32, device="cuda")
    lse = torch.empty((cfg.L, cfg.H), dtype=torch.float32, device="cuda")
    fwd = dsa.Forward.prefill(d, cfg.k, cfg.scale, chunk_rows=args.chunk, lse=lse, idx=idx)
    n_chunks = (cfg.L + args.chunk - 1) // args.chunk

    for _ in range(args.warmup):
        fwd()
    st = fwd.status()
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")

    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    _barrier(dist)
    t0, t1 = _rec(), None
    for _ in range(args.steps):
        fwd()
    t1 = _rec()
    _barrier(dist)
    clk = clocks.stop() if clocks else None
    total_ms = _max_over_ranks(dist, t0.elapsed_time(t1))
    st = fwd.status()
    if st != 0:
        raise RuntimeError(f"device status {st} in the timed region")
    ms_step = total_ms / args.steps
    value = aggregate_tokens_per_s(cfg.L, ws, args.steps, total_ms)

    # per-kernel times: the same launches (same chunking, same stream), one binding call per launch
    # with CUDA events around each, for as many steps again
    runner = PrefillRunner(dsa, d, cfg, args.chunk)
    ev = {"index": [], "topk": [], "attn": []}
    runner.step()
    _barrier(dist)
    b0 = _rec()
    for _ in range(args.steps):
        runner.step(ev)
    b1 = _rec()
    _barrier(dist)
    st = dsa.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} in the breakdown pass")
    breakdown_ms = b0.elapsed_time(b1) / args.steps

    # per-kernel rooflines (algorithmic work / summed launch time)
    w = prefill_work(cfg.L, cfg.H_I, cfg.H, cfg.k)
    t_index = _pairs_ms(ev["index"]) / args.steps
    t_topk = _pairs_ms(ev["topk"]) / args.steps
    t_attn = _pairs_ms(ev["attn"]) / args.steps
    if "sustained" in fp8:
        fp8_peak, fp8_src = fp8["sustained"], "measured e4m3 _scaled_mm (sustained)"
    else:
        fp8_peak, fp8_src = 2.0 * peaks["bf16_sus"], f"2 x {peaks['src']} bf16 sustained (FP8 not measured)"
    bf16_peak = peaks["bf16_sus"]
    kern = {
        "indexer": dict(bound="tensor", achieved=w["indexer_flop"] / (t_index * 1e-3) / 1e12, peak=fp8_peak,
                        unit="TFLOP/s", ms=t_index, launches=n_chunks, peak_source=fp8_src,
                        frac_of_2x_bf16_sustained=None),
        "topk": dict(bound="hbm", achieved=w["topk_bytes"] / (t_topk * 1e-3) / 1e9, peak=peaks["hbm"],
                     unit="GB/s", ms=t_topk, launches=n_chunks, peak_source=f"{peaks['src']} copy bandwidth"),
        "sparse_attn": dict(bound="tensor", achieved=w["attn_flop"] / (t_attn * 1e-3) / 1e12, peak=bf16_peak,
                            unit="TFLOP/s", ms=t_attn, launches=1, peak_source=f"{peaks['src']} bf16 sustained"),
    }
    for v in kern.values():
        v["frac"] = v["achieved"] / v["peak"]
    kern["indexer"]["frac_of_2x_bf16_sustained"] = kern["indexer"]["achieved"] / (2.0 * peaks["bf16_sus"])
    dom_name = max(kern, key=lambda n: kern[n]["ms"])
    dom = kern[dom_name]
    # DRAM traffic per launch: the captured bytes per query row x the rows one launch covers
    traffic, traffic_src = traffic_for(dom_name, cfg.L / kern[dom_name]["launches"])
    roofline = {"kernel": dom_name, "bound": dom["bound"], "achieved": round(dom["achieved"], 2),
                "peak": round(dom["peak"], 1), "unit": dom["unit"], "frac": round(dom["frac"], 4),
                "traffic": traffic, "traffic_source": traffic_src, "peak_source": dom["peak_source"]}

    line = {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp8-e4m3 indexer / bf16 attention (fp32 accum)",
            "data": "synthetic (seeded; shapes and distributions of the 128K prefill workload)",
            "config": {"workload": f"prefill L={cfg.L}, H_I=64, d_I=128, k=2048, H=128, D=576/512",
                       "seq_len": cfg.L, "global_batch": ws, "chunk_rows": args.chunk,
                       "l2": "inputs larger than L2 (Q %.1f GB, O %.1f GB per step)"
                             % (cfg.L * cfg.H * 1152 / 1e9, cfg.L * cfg.H * 1024 / 1e9), "parallelism": f"dp{ws}"},
            "roofline": roofline,
            "kernels": {n: {kk: (round(vv, 4) if isinstance(vv, float) else vv) for kk, vv in v.items()}
                        for n, v in kern.items()},
            "kernel_times": f"a second pass of {args.steps} steps making the same launches one binding call at a "
                            f"time with CUDA events around each ({breakdown_ms:.3f} ms per step there)",
            "fp8_peak_tflops": {k: (round(v, 1) if isinstance(v, float) else v) for k, v in fp8.items()},
            "path": "dsa_forward (C ABI) via Forward.prefill, inputs resident in HBM",
            "gpu_launches": (2 * n_chunks + 1) * args.steps,
            "clocks": clk}

    if not args.no_decode:
        line["decode"] = bench_decode(dsa, synth, args, peaks, cid=5)
        line["decode_b64_32k"] = bench_decode(dsa, synth, args, peaks, cid=3)
    if not args.no_e2e:
        line["e2e"] = bench_e2e(dsa, d, cfg, args, dist, ws)
    del d, runner, fwd
    torch.cuda.empty_cache()
    if not args.no_backward:
        # the training-side companion: the attention backward over the same 128K selections
        line["backward_128k"] = bench_backward(dsa, synth, args, peaks, L=cfg.L)
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(cfg, budget_s=args.cpu_seconds)
    return line


def bench_prefill_rows(dsa, synth, args, peaks, dist, rank, ws):
    """One 128K prefill split by query rows over the ranks (strong scaling: the total work is one
    sequence whatever N is).  Rank r owns the contiguous rows partition_rows gives it (balanced by
    modelled time) and the keys of those positions; each step all-gathers every rank's indexer keys,
    key scales and latent rows into local HBM (NCCL), then runs dsa_forward on its own rows with
    q_pos0 at their first position.  The step time is the slowest rank's."""
    from sparse_attention_30_b300 import shard
    cfg = synth.config(4)
    ranges = shard.partition_rows(cfg.L, ws, cfg.H_I, cfg.H, cfg.k, align=128)
    r0, r1 = ranges[rank]
    d = synth.prefill_inputs(cfg, device="cuda")     # the same sequence on every rank (same seed)
    key_names = ("k8", "k_scale", "kv")
    local_keys = {n: d[n][r0:r1].clone() for n in key_names}        # what this rank produced
    keys = {n: torch.zeros_like(d[n]) for n in key_names}            # every position, filled each step
    inp = {n: d[n][r0:r1].clone() for n in ("q8", "q_scale", "w", "q")}
    inp.update(keys)
    del d
    torch.cuda.empty_cache()
    T = r1 - r0
    lse = torch.empty((T, cfg.H), dtype=torch.float32, device="cuda")
    idx = torch.empty((T, cfg.k), dtype=torch.int32, device="cuda")
    fwd = dsa.Forward.prefill(inp, cfg.k, cfg.scale, q_pos0=r0, chunk_rows=args.chunk, lse=lse, idx=idx)

    def step():
        for n in key_names:
            if dist is None:
                keys[n].copy_(local_keys[n])
            else:
                shard.all_gather_rows(local_keys[n], ranges, rank, out=keys[n])
        if T > 0:
            fwd()

    for _ in range(args.warmup):
        step()
    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    _barrier(dist)
    t0 = _rec()
    for _ in range(args.steps):
        step()
    t1 = _rec()
    _barrier(dist)
    clk = clocks.stop() if clocks else None
    my_ms = t0.elapsed_time(t1)
    total_ms = _max_over_ranks(dist, my_ms)
    st = fwd.status() if T > 0 else 0
    if _max_over_ranks(dist, float(st)) != 0:
        raise RuntimeError(f"device status {st} on rank {rank}")
    value = cfg.L * args.steps / (total_ms / 1e3)
    n_chunks = (T + args.chunk - 1) // args.chunk
    return {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 3), "higher_is_better": True,
            "scaling": "strong", "vs_baseline": None, "dtype": "fp8-e4m3 indexer / bf16 attention (fp32 accum)",
            "data": "synthetic (seeded; shapes and distributions of the 128K prefill workload)",
            "config": {"workload": f"one prefill L={cfg.L}, H_I=64, d_I=128, k=2048, H=128, D=576/512, query rows "
                                   f"split over {ws} ranks by modelled time, keys all-gathered every step",
                       "seq_len": cfg.L, "global_batch": 1, "chunk_rows": args.chunk, "row_ranges": ranges,
                       "l2": "inputs larger than L2", "parallelism": f"rows{ws}"},
            "rank0_ms_per_step": round(my_ms / args.steps, 3) if rank == 0 else None,
            "gpu_launches": (2 * n_chunks + 1) * args.steps if T > 0 else 0,
            "path": "all-gather of the keys (torch.distributed) + dsa_forward (C ABI) on each rank's rows",
            "clocks": clk}


def backward_work(L, H, k):
    """Algorithmic work of the sparse-attention backward over a causal prefill's selections."""
    sel = sum(min(t + 1, k) for t in range(min(L, k))) + max(0, L - k) * k
    # per (token, key): S and dq over 576 dims, dP and dv over 512, dk over 576 -> 2 H (576 + 512 + 576 + 576 + 512)
    return dict(flop=2.0 * H * 2752 * sel, selected=sel,
                atomic_bytes=4.0 * 576 * sel,                        # fp32 adds into dkv, per (token, key)
                stream_bytes=L * H * (576 + 512 + 512 + 576) * 2.0)  # q, o, do read and dq written


def bench_backward(dsa, synth, args, peaks, L=4096):
    """The backward of the sparse attention over one prefill's selections (k=2048, H=128): the forward
    runs once (dsa_forward: indexer, top-k, attention) to give the selection, O and lse; the timed
    step is dsa_sparse_attn_backward over every row, with a random output gradient."""
    cfg = synth.config(4, L=L)
    d = synth.prefill_inputs(cfg, device="cuda")
    idx = torch.empty((L, cfg.k), dtype=torch.int32, device="cuda")
    lse = torch.empty((L, cfg.H), dtype=torch.float32, device="cuda")
    f = dsa.Forward.prefill(d, cfg.k, cfg.scale, chunk_rows=min(args.chunk, L), lse=lse, idx=idx)
    f()
    if f.status() != 0:
        raise RuntimeError("forward status")
    g = torch.Generator(device="cuda").manual_seed(5)
    do = torch.randn((L, cfg.H, 512), generator=g, device="cuda").to(torch.bfloat16)
    dq = torch.empty((L, cfg.H, 576), dtype=torch.bfloat16, device="cuda")
    dkv = torch.zeros((L, 576), dtype=torch.float32, device="cuda")
    w = dsa.status_word()

    def step():
        dkv.zero_()
        dsa.sparse_attn_backward(d["q"], d["kv"], idx, cfg.scale, f.out, do, lse, dq=dq, dkv=dkv, status=w)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ev = []
    for _ in range(args.steps):
        dkv.zero_()
        ev.append(_rec())
        dsa.sparse_attn_backward(d["q"], d["kv"], idx, cfg.scale, f.out, do, lse, dq=dq, dkv=dkv, status=w)
        ev.append(_rec())
    torch.cuda.synchronize()
    st = dsa.read_status(w)
    if st != 0:
        raise RuntimeError(f"backward status {st}")
    ms = _pairs_ms(ev) / args.steps
    wk = backward_work(L, cfg.H, cfg.k)
    tf = wk["flop"] / (ms * 1e-3) / 1e12
    res = {"L": L, "ms": round(ms, 3), "tokens_per_s": round(L / (ms * 1e-3), 1),
           "workload": f"backward of the sparse attention over a prefill L={L}, k=2048, H=128 (dq bf16, dkv fp32)",
           "kernel": {"bound": "tensor", "achieved": round(tf, 1), "peak": peaks["bf16_sus"], "unit": "TFLOP/s",
                      "frac": round(tf / peaks["bf16_sus"], 4), "peak_source": f"{peaks['src']} bf16 sustained",
                      "work": "2 H (576 + 512 + 576 + 576 + 512) FLOP per selected (token, key) pair"},
           "atomic_GBps": round(wk["atomic_bytes"] / (ms * 1e-3) / 1e9, 1),
           "launches": 1}
    del d, f, do, dq, dkv
    torch.cuda.empty_cache()
    return res


def bench_prefill_tail(dsa, synth, args, peaks, n_rows=1024):
    """The last 1024 query rows of the 128K prefill (each against ~131K keys): the steady state of
    the 128K step at a size small enough for full profiler captures (under 1 GB on the device)."""
    cfg = synth.config(4)
    d = synth.prefill_tail_inputs(cfg, n_rows, device="cuda")
    r0 = d["row0"]
    ld = (cfg.L + 3) // 4 * 4
    scores = torch.empty((n_rows, ld), dtype=torch.float32, device="cuda")
    idx = torch.empty((n_rows, cfg.k), dtype=torch.int32, device="cuda")
    out = torch.empty((n_rows, cfg.H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((n_rows, cfg.H), dtype=torch.float32, device="cuda")
    torch.cuda.empty_cache()
    ev = {"index": [], "topk": [], "attn": []}

    def step(ev=None):
        for name, fn in (("index", lambda: dsa.index(d["q8"], d["q_scale"], d["w"], d["k8"], d["k_scale"], q_pos0=r0,
                                                      scores=scores)),
                         ("topk", lambda: dsa.topk(scores, cfg.k, q_pos0=r0, n_cols=cfg.L, idx=idx)),
                         ("attn", lambda: dsa.sparse_attn(d["q"], d["kv"], idx, cfg.scale, out=out, lse=lse))):
            if ev is not None:
                ev[name].append(_rec())
            fn()
            if ev is not None:
                ev[name].append(_rec())

    for _ in range(max(3, args.warmup)):
        step()
    for _ in range(args.steps):
        step(ev)
    torch.cuda.synchronize()
    st = dsa.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st}")
    kms = {k: round(_pairs_ms(v) / args.steps, 4) for k, v in ev.items()}
    ms = sum(kms.values())
    # the other kernels on the same rows (run after the step, timed apart): the indexer loss over the
    # selected sets, dense causal attention over every preceding key, and the dense warm-up loss
    dense_lse = torch.empty_like(lse)
    extras = {
        "loss": lambda: dsa.indexer_loss(d["q"], d["kv"], lse, scores, cfg.scale, idx=idx, want_p=False),
        "dense_attn": lambda: dsa.dense_causal_attn(d["q"], d["kv"], cfg.scale, q_pos0=r0, out=out, lse=dense_lse),
        "dense_loss": lambda: dsa.indexer_loss(d["q"], d["kv"], dense_lse, scores, cfg.scale, q_pos0=r0),
    }
    for name, fn in extras.items():
        for _ in range(max(3, args.warmup)):
            fn()
        e = []
        for _ in range(args.steps):
            e.append(_rec())
            fn()
            e.append(_rec())
        torch.cuda.synchronize()
        kms[name] = round(_pairs_ms(e) / args.steps, 4)
    st = dsa.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st}")
    return {"metric": "prefill tail tokens/s", "value": round(n_rows / (ms * 1e-3), 1), "unit": "tokens/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "dtype": "fp8-e4m3 / bf16", "data": "synthetic",
            "config": {"workload": f"prefill L={cfg.L}: query rows {r0}..{cfg.L - 1}, k=2048, H=128, H_I=64"},
            "kernels_ms": kms}


def bench_dense_curve(dsa, synth, args, peaks, lengths=(4096, 16384, 32768, 65536, 131072)):
    """Prefill time of one sequence against its length, DSA (indexer -> top-k -> sparse attention)
    beside dense causal MLA attention over the same Q / latent rows: the cost-versus-length
    comparison of the pages (dense cost grows with L^2, DSA's attention with k L)."""
    curve = []
    for L in lengths:
        cfg = synth.config(4, L=L)
        d = synth.prefill_inputs(cfg, device="cuda")
        runner = PrefillRunner(dsa, d, cfg, min(args.chunk, L))
        out = torch.empty((L, cfg.H, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((L, cfg.H), dtype=torch.float32, device="cuda")

        def dense():
            dsa.dense_causal_attn(d["q"], d["kv"], cfg.scale, out=out, lse=lse)

        res = {"L": L}
        for name, fn in (("dsa", runner.step), ("dense", dense)):
            for _ in range(args.warmup):
                fn()
            torch.cuda.synchronize()
            n = args.steps if L <= 32768 else max(2, min(args.steps, 3))
            a = _rec()
            for _ in range(n):
                fn()
            b = _rec()
            b.synchronize()
            res[f"{name}_ms"] = round(a.elapsed_time(b) / n, 3)
        st = dsa.device_status()
        if st != 0:
            raise RuntimeError(f"device status {st} at L={L}")
        dense_flop = 2.0 * cfg.H * (576 + 512) * L * (L + 1) / 2
        res["dense_tflops"] = round(dense_flop / (res["dense_ms"] * 1e-3) / 1e12, 1)
        res["dense_frac"] = round(res["dense_tflops"] / peaks["bf16_sus"], 4)
        res["dsa_tok_s"] = round(L / (res["dsa_ms"] * 1e-3), 1)
        res["dense_tok_s"] = round(L / (res["dense_ms"] * 1e-3), 1)
        res["dense_over_dsa"] = round(res["dense_ms"] / res["dsa_ms"], 3)
        curve.append(res)
        del d, runner, out, lse
        torch.cuda.empty_cache()
    last = curve[-1]
    return {"metric": "prefill tokens/s, DSA vs dense causal MLA attention, against sequence length",
            "value": last["dsa_tok_s"], "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": last["dsa_ms"], "higher_is_better": True,
            "dtype": "fp8-e4m3 indexer / bf16 attention (fp32 accum)", "data": "synthetic",
            "config": {"workload": "one prefill sequence per L (128K recipe), H=128, k=2048, H_I=64",
                       "dense": "dsa_dense_causal_attn over the same Q and latent rows (no indexer, no top-k)"},
            "curve": curve}


def bench_indexer_loss(dsa, synth, args, peaks, dense_L=32768):
    """Training-side forward of the 128K prefill through dsa_forward_loss (per 8192-row chunk: the
    indexer, top-k, sparse attention for lse and the indexer's KL loss over the selected sets); plus
    the dense warm-up stage (indexer, dense causal attention, KL over every preceding key) on a 32K
    sequence.  The loss kernel's own time comes from a second pass that makes the same launches one
    by one with CUDA events around the loss launches."""
    out = {}
    for stage, L in (("sparse", 131072), ("dense_warmup", dense_L)):
        cfg = synth.config(4, L=L)
        d = synth.prefill_inputs(cfg, device="cuda")
        chunk = min(args.chunk, L)
        sparse = stage == "sparse"
        idx = torch.empty((L, cfg.k), dtype=torch.int32, device="cuda") if sparse else None
        f = dsa.ForwardLoss(d, cfg.k, cfg.scale, stage=dsa.LOSS_SPARSE if sparse else dsa.LOSS_DENSE_WARMUP,
                            chunk_rows=chunk, idx=idx)
        for _ in range(args.warmup):
            f()
        torch.cuda.synchronize()
        n = max(2, min(args.steps, 3))
        a = _rec()
        for _ in range(n):
            f()
        b = _rec()
        b.synchronize()
        ms = a.elapsed_time(b) / n
        loss_value = float(f.loss.item())
        # breakdown: the same launches one by one, events around the loss launches
        ld = (L + 3) // 4 * 4
        scores = torch.empty((chunk, ld), dtype=torch.float32, device="cuda")
        loss = torch.zeros((1,), dtype=torch.float64, device="cuda")
        ev = []
        for c in range((L + chunk - 1) // chunk):
            r0, r1 = c * chunk, min(L, (c + 1) * chunk)
            sc = scores[: r1 - r0]
            dsa.index(d["q8"][r0:r1], d["q_scale"][r0:r1], d["w"][r0:r1], d["k8"], d["k_scale"], q_pos0=r0, scores=sc)
            if sparse:
                dsa.topk(sc, cfg.k, q_pos0=r0, n_cols=L, idx=idx[r0:r1])
                dsa.sparse_attn(d["q"][r0:r1], d["kv"], idx[r0:r1], cfg.scale, out=f.out[r0:r1], lse=f.lse[r0:r1])
            else:
                dsa.dense_causal_attn(d["q"][r0:r1], d["kv"], cfg.scale, q_pos0=r0, out=f.out[r0:r1], lse=f.lse[r0:r1])
            ev.append(_rec())
            dsa.indexer_loss(d["q"][r0:r1], d["kv"], f.lse[r0:r1], sc, cfg.scale, idx=idx[r0:r1] if sparse else None,
                             q_pos0=0 if sparse else r0, want_p=False, kl=f.kl[r0:r1], loss=loss)
            ev.append(_rec())
        torch.cuda.synchronize()
        st = f.status() or dsa.device_status()
        if st != 0:
            raise RuntimeError(f"device status {st} ({stage})")
        loss_ms = _pairs_ms(ev)
        pairs = (sum(min(t + 1, cfg.k) for t in range(min(L, cfg.k))) + max(0, L - cfg.k) * cfg.k
                 if sparse else L * (L + 1) // 2)
        flop = 2.0 * cfg.H * 576 * pairs
        tf = flop / (loss_ms * 1e-3) / 1e12
        out[stage] = {"L": L, "step_ms": round(ms, 3), "tokens_per_s": round(L / (ms * 1e-3), 1),
                      "path": "dsa_forward_loss (C ABI)",
                      "loss_kernel_ms": round(loss_ms, 3), "loss_launches": len(ev) // 2,
                      "loss_kernel": {"bound": "tensor", "achieved": round(tf, 1), "peak": peaks["bf16_sus"],
                                      "unit": "TFLOP/s", "frac": round(tf / peaks["bf16_sus"], 4),
                                      "work": "2 H 576 FLOP per (row, key) pair of the set (QK^T recomputed)"},
                      "loss_value": loss_value, "loss_value_breakdown_pass": float(loss.item())}
        del d, scores, f, idx
        torch.cuda.empty_cache()
    sp = out["sparse"]
    return {"metric": "training-side prefill tokens/s with the indexer KL loss (128K, sparse stage)",
            "value": sp["tokens_per_s"], "unit": "tokens/s", "n_gpus": 1, "steps": max(2, min(args.steps, 3)),
            "warmup": args.warmup, "ms_per_step": sp["step_ms"], "higher_is_better": True,
            "dtype": "fp8-e4m3 indexer / bf16 attention and loss (fp32 accum, fp64 row sums)", "data": "synthetic",
            "config": {"workload": "prefill L=131072 in 8192-row chunks: indexer, top-k, sparse attention, KL loss; "
                                   f"dense warm-up stage at L={dense_L}"},
            "stages": out}


def bench_decode(dsa, synth, args, peaks, cid=5):
    """Decode step through dsa_forward, replayed from a CUDA graph of that call (value; the eager
    call is timed too), and stage by stage with CUDA events (breakdown).  L2 is flushed between
    steps: a 252 MB write, then a read of another 252 MB buffer, so that the write's dirty lines
    are written back before the timed region instead of inside the first kernel of the step."""
    cfg = synth.config(cid)
    d = synth.decode_inputs(cfg, device="cuda")
    lens = d["seq_lens"].cpu().tolist()
    max_len = max(lens)
    f = dsa.Forward.decode(d, cfg.k, cfg.scale, max_len)
    flush_w = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    flush_r = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")

    def flush():
        flush_w.fill_(1.0)
        flush_r.sum()

    ld = (max_len + 3) // 4 * 4
    scores = torch.empty((cfg.B, ld), dtype=torch.float32, device="cuda")
    idx = torch.empty((cfg.B, cfg.k), dtype=torch.int32, device="cuda")
    out = torch.empty((cfg.B, cfg.H, 512), dtype=torch.bfloat16, device="cuda")
    n_split = dsa.decode_split(cfg.B)   # the key split dsa_forward's decode uses
    n_ws = dsa.lib.dsa_sparse_attn_split_workspace_size(cfg.B, cfg.H, n_split)
    split_ws = torch.empty(n_ws, dtype=torch.uint8, device="cuda") if n_ws else None

    def stages(ev):
        ev["index"].append(_rec())
        dsa.index_paged(d["q8"], d["q_scale"], d["w"], d["k8_cache"], d["k_scale_cache"], d["block_table"],
                        d["seq_lens"], max_len, scores=scores)
        ev["index"].append(_rec())
        ev["topk"].append(_rec())
        dsa.topk(scores, cfg.k, row_lens=d["seq_lens"], idx=idx)
        ev["topk"].append(_rec())
        ev["attn"].append(_rec())
        dsa.sparse_attn_split(d["q"], d["kv_cache"], idx, cfg.scale, n_split, block_table=d["block_table"], out=out,
                              ws=split_ws)
        ev["attn"].append(_rec())

    for _ in range(max(3, args.warmup)):
        f()
        stages({"index": [], "topk": [], "attn": []})
    # the step as a serving loop runs it: the dsa_forward call (four launches) captured once into a
    # CUDA graph and replayed, so that no launch gap sits between its kernels
    graph = f.capture()
    for _ in range(max(3, args.warmup)):
        graph.replay()
    n = max(10, args.steps)
    times, eager, ev = [], [], {"index": [], "topk": [], "attn": []}
    for _ in range(n):
        flush()
        a = _rec()
        graph.replay()
        b = _rec()
        b.synchronize()
        times.append(a.elapsed_time(b))
    for _ in range(n):
        flush()
        a = _rec()
        f()
        b = _rec()
        b.synchronize()
        eager.append(a.elapsed_time(b))
    for _ in range(n):
        flush()
        stages(ev)
    torch.cuda.synchronize()
    st = f.status() or dsa.device_status()
    if st != 0:
        raise RuntimeError(f"decode status {st}")
    ms = float(np.median(times))
    w = decode_work(lens, cfg.H_I, cfg.H, cfg.k)
    kms = {k: _pairs_ms(v) / n for k, v in ev.items()}
    kern = {
        "indexer": dict(bound="hbm", ms=kms["index"], achieved=w["indexer_bytes"] / (kms["index"] * 1e-3) / 1e9,
                        peak=peaks["hbm"], unit="GB/s"),
        "topk": dict(bound="hbm", ms=kms["topk"], achieved=w["topk_bytes"] / (kms["topk"] * 1e-3) / 1e9,
                     peak=peaks["hbm"], unit="GB/s"),
        "sparse_attn": dict(bound="hbm", ms=kms["attn"], achieved=w["attn_bytes"] / (kms["attn"] * 1e-3) / 1e9,
                            peak=peaks["hbm"], unit="GB/s"),
    }
    for v in kern.values():
        v["frac"] = round(v["achieved"] / v["peak"], 4)
        v["ms"] = round(v["ms"], 4)
        v["achieved"] = round(v["achieved"], 1)
    tot_bytes = w["indexer_bytes"] + w["topk_bytes"] + w["attn_bytes"]
    return {"metric": "decode query-tok/s", "value": round(cfg.B / (ms * 1e-3), 1), "unit": "query-tok/s",
            "ms_per_step": round(ms, 4), "eager_ms_per_step": round(float(np.median(eager)), 4),
            "path": "dsa_forward (C ABI) replayed from a CUDA graph of the call",
            "workload": cfg.name + ", k=2048, H=128, H_I=64",
            "algorithmic_bytes": tot_bytes, "hbm_frac_of_step": round(tot_bytes / (ms * 1e-3) / 1e9 / peaks["hbm"], 4),
            "kernels": kern,
            "l2": "flushed between steps (252 MB write, then a 252 MB read of another buffer so the write's "
                  "dirty lines leave L2 before the timed region)"}


def _min_over_ranks(dist, x: float) -> float:
    return -_max_over_ranks(dist, -x)


def bench_e2e(dsa, d, cfg, args, dist=None, ws=1):
    """The prefill step with inputs and output in pinned host memory, through dsa_prefill_host (the
    library's host-buffer entry point): every step copies every input in and the attention output
    back, chunk by chunk, overlapped with the kernels.  Under torchrun every rank pins its own
    buffers, so the host must hold all local ranks' at once; the ranks decide together."""
    names = ["q8", "q_scale", "w", "k8", "k_scale", "q", "kv"]
    need = sum(d[n].numel() * d[n].element_size() for n in names) + cfg.L * cfg.H * 512 * 2
    local_ws = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
    try:
        avail = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError):
        avail = 0
    fits = avail >= 1.5 * need * local_ws
    if _min_over_ranks(dist, 1.0 if fits else 0.0) < 0.5:
        return {"value": None, "unit": "tokens/s",
                "skipped": f"host memory {avail / 2**30:.0f} GiB < 1.5 x {local_ws} ranks x {need / 2**30:.0f} GiB"}
    host = {n: torch.empty_like(d[n], device="cpu").pin_memory() for n in names}
    for n in names:
        host[n].copy_(d[n])
    f = dsa.PrefillHost(host, cfg.k, cfg.scale, chunk_rows=args.e2e_chunk)
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = f.out.numel() * 2

    f()
    n_steps = args.steps
    _barrier(dist)
    a = _rec()
    for _ in range(n_steps):
        f()
    b = _rec()
    b.synchronize()
    ms = _max_over_ranks(dist, a.elapsed_time(b) / n_steps)
    st = f.status()
    if st != 0:
        raise RuntimeError(f"e2e status {st}")
    return {"value": round(aggregate_tokens_per_s(cfg.L, ws, 1, ms), 1), "unit": "tokens/s",
            "ms_per_step": round(ms, 2), "h2d_bytes_per_step": h2d * ws, "d2h_bytes_per_step": d2h * ws,
            "steps": n_steps,
            "path": f"dsa_prefill_host (C ABI), pinned host buffers, {args.e2e_chunk}-row chunks, all ranks"}


# ------------------------------------------------------------------------------------ oracle arm

def _oracle_rows_rate(cfg, d, rows):
    """Times the float64 oracle on the given prefill rows; returns (rows/s, seconds)."""
    import oracle
    keys = {n: d[n].cpu() for n in ("k8", "k_scale", "kv")}
    t_sum = 0.0
    for t in rows:
        row = dict(keys, **{n: {t: d[n][t].cpu()} for n in ("q8", "q_scale", "w", "q")})
        t0 = time.perf_counter()
        oracle.prefill_row(row, int(t), cfg.k, cfg.scale)
        t_sum += time.perf_counter() - t0
    return len(rows) / t_sum, t_sum


def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:  # pragma: no cover
        return os.cpu_count() or 1


def cpu_baseline(cfg, budget_s=12.0, d=None):
    """Oracle tokens/s on a stratified sample of rows of the same 128K workload."""
    import synth
    if d is None:
        d = synth.prefill_inputs(cfg, device="cuda")
    rng = np.random.default_rng(0)
    rows, spent, n = [], 0.0, 0
    strata = 64
    while spent < budget_s and n < 4096:
        s = n % strata
        rows_s = [int((s + rng.random()) * cfg.L / strata)]
        _, dt = _oracle_rows_rate(cfg, d, rows_s)
        spent += dt
        rows += rows_s
        n += 1
    rate = len(rows) / spent
    return {"value": round(rate, 3), "unit": "tokens/s", "cores": _blas_threads(), "kind": "oracle",
            "sample": f"{len(rows)} prefill rows of the 128K workload, stratified over positions "
                      f"(float64 NumPy oracle: scores, full sort, attention), {spent:.1f} s"}


def run_reference(args, dist, rank, ws):
    """The oracle as the reference arm: each step is a bounded sample of the 128K workload."""
    import synth
    if rank != 0:
        return None
    cfg = synth.config(4)
    d = synth.prefill_inputs(cfg, device="cuda" if torch.cuda.is_available() else "cpu")
    rng = np.random.default_rng(1)
    per_step = 4
    for _ in range(args.warmup):
        _oracle_rows_rate(cfg, d, [int(rng.integers(0, cfg.L))])
    total_rows, total_s = 0, 0.0
    for i in range(args.steps):
        rows = [int((j + rng.random()) * cfg.L / per_step) for j in range(per_step)]
        _, dt = _oracle_rows_rate(cfg, d, rows)
        total_rows += len(rows)
        total_s += dt
    value = total_rows / total_s
    cores = _blas_threads()
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total_s / args.steps, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; the 128K prefill workload)",
            "config": {"workload": "prefill L=131072 (128K), H_I=64, d_I=128, k=2048, H=128, D=576/512",
                       "seq_len": cfg.L, "global_batch": 1},
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{per_step} stratified rows per step, {total_rows} rows"},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--chunk", type=int, default=8192)
    p.add_argument("--workload", default="prefill128k", choices=["prefill128k", "prefill4k", "prefill128k_tail", "decode", "decode32k",
                                                       "dense_curve", "indexer_loss", "backward", "backward128k"],
                   help="the others run single pieces (used for profiler captures)")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--e2e-chunk", type=int, default=2048, help="query rows per chunk of the host-buffer pipeline")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-decode", action="store_true")
    p.add_argument("--no-fp8-peak", action="store_true", help="skip the e4m3 GEMM that measures the FP8 peak")
    p.add_argument("--no-backward", action="store_true", help="skip the 128K attention backward sub-line")
    p.add_argument("--shard", default="sequences", choices=["sequences", "rows"],
                   help="N > 1: one 128K sequence per rank (weak scaling), or one sequence split by query rows "
                        "over the ranks (strong scaling)")
    args = p.parse_args()
    args.warmup = max(3, args.warmup)
    dist, rank, ws, _ = _dist()
    line = run_reference(args, dist, rank, ws) if args.impl == "reference" else run_ours(args, dist, rank, ws)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
