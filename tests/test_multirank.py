"""The bench's multi-rank logic on CPU with two gloo ranks: each rank serves
its own requests (distinct seeds, same shapes) and the job is timed by its
slowest rank."""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from host_latent_cache_gb300 import workloads as W
    cfg = bench.rank_workload(W.long_128k(), rank)
    mine = [10.0 + 5.0 * rank, 3.0 - rank]          # per-rank step and e2e milliseconds
    got = bench.max_over_ranks(mine, dist, device="cpu")
    dist.barrier()
    q.put((rank, cfg.seed, cfg.batch, cfg.T, got))
    dist.destroy_process_group()


def test_two_ranks_shard_requests_and_take_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, b0, t0, g0), (r1, s1, b1, t1, g1) = out
    assert s0 != s1 and (b0, t0) == (b1, t1)       # independent requests, same shapes
    assert g0 == g1 == [15.0, 3.0]                   # element-wise max over the ranks


def test_job_throughput_counts_every_rank():
    import bench
    assert bench.job_throughput(8, 4, 10, 100.0) == 8 * 4 * 10 / 0.1
