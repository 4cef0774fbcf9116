"""bench.py's multi-rank timing on CPU: world size 2 over gloo (no GPU).

Each rank runs its own replica of the workload (the decode path shards by
sequence with no exchange); the reported step time is the slowest rank's and
the value counts the bytes of every rank.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [2.5, 4.0][rank]
    m = bench.max_over_ranks(local_ms)
    dist.barrier()
    out[rank] = (m, bench.job_throughput(1e9, m, world))
    dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == out[1]
    m, gbs = out[0]
    assert m == 4.0
    assert gbs == pytest.approx(2 * 1e9 / 4e-3 / 1e9)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.job_throughput(2e9, 1.0, 1) == pytest.approx(2000.0)
