"""Multi-rank logic of bench.py on CPU: two gloo ranks on 127.0.0.1 agree on
the max-over-ranks time and on the whole-job (weak scaling) throughput."""
import os
import socket

import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    import torch.distributed as dist
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    ms = bench.reduce_max(1.0 + rank, "cpu")            # rank 1 is the slower one
    val = bench.weak_scaling_value(2048, world, ms)
    q.put((rank, ms, val))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
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
    assert [r[1] for r in res] == [2.0, 2.0]
    assert res[0][2] == res[1][2] == pytest.approx(2 * 2048 / 2e-3)


def test_single_process_is_identity():
    import bench
    assert bench.reduce_max(3.5) == 3.5
    assert bench.weak_scaling_value(100, 1, 10.0) == pytest.approx(1e4)
