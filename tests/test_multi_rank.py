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
