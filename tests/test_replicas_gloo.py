"""The bench's multi-rank path on CPU: two gloo ranks (127.0.0.1) reduce their step times to the
slowest one and report whole-job throughput.  The path shards as independent replicas (rows and
heads are independent, and nothing is exchanged between them), so the only collective is this
timing reduction."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = [1.0 + rank, 10.0 - rank]  # per-rank (ms, e2e ms)
    red = bench.reduce_max_over_ranks(local, dist, device="cpu")
    value = bench.job_throughput(256, world, red[0])
    q.put((rank, red, value))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=90) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, red, value in got:
        assert red == [2.0, 10.0]
        assert value == pytest.approx(2 * 256 / 2e-3)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert bench.job_throughput(256, 1, 0.128) == pytest.approx(2e6)
