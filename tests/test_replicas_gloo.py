"""The multi-rank host logic with two gloo ranks on the CPU: per-rank seeds
differ, the step time is the maximum over ranks, and the throughput counts
every rank's work over that maximum."""

import os
import socket

import pytest
import torch.multiprocessing as mp

from exact_tiled_attention_28_gb300 import replicas


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [3.0, 5.0][rank]  # rank 1 is the slow one
        m = replicas.max_over_ranks(ms)
        tp = replicas.aggregate_throughput(1e12, world, m)
        dist.barrier()
        out.put((rank, replicas.replica_seed(1000, rank), m, tp))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, m0, t0), (r1, s1, m1, t1) = res
    assert s0 != s1
    assert m0 == m1 == 5.0
    assert t0 == t1 == pytest.approx(2 * 1e12 / 5e-3 / 1e12)


def test_single_process_is_identity():
    assert replicas.max_over_ranks(7.5) == 7.5
    with pytest.raises(ValueError):
        replicas.aggregate_throughput(1.0, 1, 0.0)
