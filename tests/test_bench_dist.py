"""The benchmark's multi-rank host logic (weak scaling, max-over-ranks timing) on two gloo
ranks on the CPU."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, lr = bench.dist_info()
    assert (w, r, lr) == (world, rank, rank)
    bench.barrier(world)
    got = bench.reduce_max(1.5 + rank, world)
    q.put((rank, got))
    dist.destroy_process_group()


def test_two_rank_timing_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 2.5, 1: 2.5}


def test_bench_args_defaults():
    import bench
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.workload == "glm_decode_t1"


def test_spec_accounting_counts_the_accepted_prefix():
    """a forward yields its verified token plus the drafts accepted before the first rejection"""
    import numpy as np

    import bench
    acc = np.array([[True, True, False, True], [False, True, True, True], [True] * 4, [False] * 4])
    assert bench.emitted_tokens(acc).tolist() == [3, 1, 5, 1]
    assert bench.emitted_tokens(np.zeros((3, 0), bool)).tolist() == [1, 1, 1]
    # the simulated acceptance gives 1 + p + p^2 + p^3 tokens per forward with 3 drafts: 2.2..2.8
    rng = np.random.default_rng(0)
    m = bench.emitted_tokens(rng.random((200000, 3)) < bench.SPEC_ACCEPT).mean()
    p = bench.SPEC_ACCEPT
    assert abs(m - (1 + p + p * p + p ** 3)) < 0.01 and 2.2 <= m <= 2.8
