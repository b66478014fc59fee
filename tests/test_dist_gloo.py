"""Multi-process host logic of bench.py with the gloo backend on CPU (world size 2).

Every (sequence, KV head) is independent, so N GPUs run N copies of the per-GPU
workload (weak scaling) with no data-path collective; the only exchange is the
max-over-ranks of the timed region.  These tests run that exchange and the
aggregate throughput formula on two CPU ranks.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        ms = [3.0, 5.5][rank]
        m = bench.max_over_ranks(ms)
        value = bench.aggregate_gbs(1_000_000_000, m, world)
        q.put((rank, m, value))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_with_gloo():
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
    for rank, m, value in res:
        assert m == 5.5  # slowest rank
        assert value == pytest.approx(2 * 1.0 / 5.5e-3)  # 2 ranks x 1 GB in 5.5 ms, in GB/s


def test_single_process_is_identity():
    import bench

    assert bench.max_over_ranks(7.25) == 7.25
    assert bench.aggregate_gbs(2_000_000_000, 1.0, 1) == pytest.approx(2000.0)
