"""Multi-rank host logic of the benchmark (replicas: no collective in the data
path), run as two gloo ranks on the CPU: the step time is the maximum over ranks
and the whole-job value counts the tokens of every rank."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, port: int, q):
    dist.init_process_group("gloo", rank=rank, world_size=2, init_method=f"tcp://127.0.0.1:{port}")
    import bench
    ms = bench._max_over_ranks(dist, 1.0 + rank, torch.device("cpu"))
    bench._barrier(dist)
    q.put((rank, ms, bench._replica_tokens_per_s(dist.get_world_size(), 4, ms)))
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_all_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    old = os.environ.get("PYTHONPATH", "")
    os.environ["PYTHONPATH"] = root + (os.pathsep + old if old else "")
    try:
        procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
        for p in procs:
            p.start()
        res = sorted(q.get(timeout=120) for _ in procs)
        for p in procs:
            p.join(timeout=60)
            assert p.exitcode == 0
    finally:
        os.environ["PYTHONPATH"] = old
    assert [r for r, _, _ in res] == [0, 1]
    for _, ms, v in res:
        assert ms == pytest.approx(2.0)                 # the slower rank's 2 ms
        assert v == pytest.approx(2 * 4 / 2.0e-3)      # 8 tokens in 2 ms
