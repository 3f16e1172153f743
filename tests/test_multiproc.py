"""The N > 1 host logic of bench.py on CPU: two gloo ranks, token sharding
with no data exchange, max-over-ranks timing and the whole-job rate."""
import os
import socket

import numpy as np
import torch.multiprocessing as mp

import moe_inputs as mi


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    cfg = bench.rank_workload(mi.custom_config("t", T=8, d=64, E=8, inter=64), rank)
    x = mi.make_x(cfg)
    elapsed = [0.5, 0.8][rank]                     # rank 1 is the slow one
    m = bench.max_over_ranks(elapsed, world, "cpu")
    q.put((rank, cfg.seed, x.tobytes()[:64], m, bench.throughput(8, world, 10, m)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_tokens_and_take_the_max_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, x0, m0, v0), (r1, s1, x1, m1, v1) = res
    assert (s0, s1) == (0, 1) and x0 != x1          # each rank its own tokens
    assert m0 == m1 == 0.8                          # both see the slowest rank
    assert v0 == v1 == 2 * 8 * 10 / 0.8             # tokens of all ranks / max time


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.throughput(107520, 1, 50, 1.0) == 107520 * 50
