"""Host-side logic of the N-GPU bench path on CPU: two gloo ranks (127.0.0.1), each with its own
sequence seed, agree on the max step time, on the whole-job throughput and on skipping a leg that
one rank cannot run."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = 100.0 + 50.0 * rank                     # rank 1 is the slower one
        mx = bench._max_over_ranks(dist, my_ms)
        value = bench.aggregate_tokens_per_s(131072, world, 5, mx * 5)
        # a leg that needs every rank (the end-to-end copies) runs only if all ranks can
        fits = bench._min_over_ranks(dist, 1.0 if rank == 0 else 0.0)
        q.put((rank, mx, value, bench.rank_seed(3, rank), fits))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [150.0, 150.0]           # both see the slowest rank
    assert res[0][2] == pytest.approx(131072 * 2 / 0.150)   # tokens of both ranks / max time
    assert res[0][3] != res[1][3]                           # distinct sequences per rank
    assert [r[4] for r in res] == [0.0, 0.0]                # one rank short of memory: both skip


# ----------------------------------------------------------------------------- row-sharded prefill

@pytest.mark.parametrize("L,world,align", [(131072, 2, 1), (131072, 8, 128), (4096, 2, 1), (4096, 4, 8),
                                           (300, 3, 1), (5, 4, 1), (0, 2, 1)])
def test_partition_covers_every_row_once_with_balanced_work(L, world, align):
    from sparse_attention_30_b300 import shard
    H_I, H, k = 64, 128, 2048
    ranges = shard.partition_rows(L, world, H_I, H, k, align=align)
    assert len(ranges) == world and ranges[0][0] == 0 and ranges[-1][1] == L
    rows = [t for a, b in ranges for t in range(a, b)]
    assert rows == list(range(L))                                   # each row exactly once, in order
    for a, b in ranges[:-1]:
        assert b % align == 0
    cost = [shard.rows_cost(a, b, H_I, H, k) for a, b in ranges]
    total = shard.rows_cost(0, L, H_I, H, k)
    assert abs(sum(cost) - total) <= 1e-9 * max(total, 1e-30)
    if L >= 4096:
        mean = total / world
        assert max(abs(c - mean) for c in cost) <= 0.02 * mean, cost  # within 2% of an equal share
        # causal rows cost more late in the sequence: the first rank takes the most rows
        assert ranges[0][1] - ranges[0][0] >= ranges[-1][1] - ranges[-1][0]


def test_rows_cost_closed_forms_against_loops():
    from sparse_attention_30_b300 import shard
    rates = {"indexer_tflops": 1.0, "attn_tflops": 2.0, "topk_gbs": 3.0}
    H_I, H, k = 4, 8, 5
    for r0, r1 in [(0, 1), (0, 12), (3, 9), (7, 7), (4, 30)]:
        pairs = sum(t + 1 for t in range(r0, r1))
        sel = sum(min(t + 1, k) for t in range(r0, r1))
        want = (2.0 * H_I * 128 * pairs / 1e12 + 4.0 * pairs / 3e9 + 2.0 * H * 1088 * sel / 2e12)
        assert shard.rows_cost(r0, r1, H_I, H, k, rates) == pytest.approx(want, rel=1e-12, abs=0)


def _gather_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch
    from sparse_attention_30_b300 import shard
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        L = 1000
        ranges = shard.partition_rows(L, world, 64, 128, 64)
        g = torch.Generator().manual_seed(3)
        full_kv = torch.randn(L, 576, generator=g).to(torch.bfloat16)       # latent rows
        full_k8 = torch.randint(0, 256, (L, 128), generator=g, dtype=torch.uint8)
        full_ks = torch.rand(L, generator=g)
        a, b = ranges[rank]
        got = [shard.all_gather_rows(t[a:b].clone(), ranges, rank) for t in (full_kv, full_k8, full_ks)]
        ok = all(torch.equal(x, y) for x, y in zip(got, (full_kv, full_k8, full_ks)))
        q.put((rank, ok, ranges))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_gather_every_key_row_in_position_order():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gather_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert all(r[1] for r in res)
    assert res[0][2] == res[1][2]                                   # both ranks computed the same partition
    (a0, b0), (a1, b1) = res[0][2]
    assert a0 == 0 and b0 == a1 and b1 == 1000 and b0 - a0 > b1 - a1   # uneven, contiguous, rank 0 larger
