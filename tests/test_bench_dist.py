"""bench.py's multi-process host logic on CPU: two gloo ranks on 127.0.0.1.

Under torchrun every rank times its own replica of the workload (the path
shards into independent (b, h, q-block) items, so there is no exchange); the
reported time is the largest of the ranks' times and the rate counts the work
of all ranks.  No GPU is involved."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, queue) -> None:
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        step_ms = bench.max_over_ranks(local_ms, dist, device="cpu")
        rate = bench.whole_job_rate(3.0e12, step_ms, world)
        queue.put((rank, step_ms, rate))
    finally:
        dist.destroy_process_group()


def test_two_ranks_report_the_slowest_time_and_the_whole_job_rate():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
            p.join()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    results = sorted(queue.get(timeout=10) for _ in range(2))
    assert [r[0] for r in results] == [0, 1]
    for _, step_ms, rate in results:
        assert step_ms == pytest.approx(15.0)
        assert rate == pytest.approx(2 * 3.0e12 / 15.0e-3 / 1e12)


def test_single_process_is_its_own_maximum():
    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.whole_job_rate(4.432e12, 3.2, 1) == pytest.approx(1385.0)
