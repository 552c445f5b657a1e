"""bench.py's multi-rank aggregation on CPU: two gloo ranks, each an independent replica, with
no data-path collective; the timing is the maximum over ranks and the throughput counts every
rank's bytes."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [120.0, 150.0][rank]  # rank 1 is the slow one
    m = bench.max_over_ranks(local_ms)
    q.put((rank, m, bench.whole_job_gbs(1000, 10, world, m)))
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [150.0, 150.0]
    # 2 ranks x 1000 bytes x 10 steps in 150 ms
    assert res[0][2] == pytest.approx(2 * 1000 * 10 / 0.150 / 1e9)


def test_single_process_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_gbs(603996160, 1, 1, 0.1) == pytest.approx(6039.9616)
