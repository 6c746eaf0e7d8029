"""The multi-GPU path of bench.py on CPU: two gloo ranks stand in for two
replicas.  Streams shard across replicas with no exchange, so the only
cross-rank steps are the barrier around the timed region and the max of the
ranks' times; the job rate is every rank's units over the slowest rank's
time.  Also: the reference arm does no work on ranks other than 0."""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        local_ms = 100.0 * (rank + 1)                      # rank 1 is the slow replica
        ms = bench.max_over_ranks(local_ms, world)
        rate = bench.job_throughput(1280.0, ms, world)
        bench.barrier(world)
        out.put((rank, ms, rate))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, rate in res:
        assert ms == 200.0                                 # every rank sees the max
        assert rate == pytest.approx(2 * 1280.0 / 0.2)     # both replicas' audio over the slowest time


def test_single_process_is_identity():
    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert bench.job_throughput(100.0, 500.0, 1) == pytest.approx(200.0)


def test_reference_arm_idle_on_other_ranks(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        decoder, steps, warmup = "tiny", 1, 0

    assert bench.run_reference(Args()) == 0


def test_playback_gaps():
    # 80 ms frames: a 1-frame chunk ready at 10 ms plays until 90 ms; the next
    # (ready at 10 + 100 = 110 ms) leaves a 20 ms gap; the third is ready at
    # 115 ms while the second plays until 110 + 2 x 80 = 270 ms: no gap
    assert bench.playback_gaps([10.0, 100.0, 5.0], [1, 2, 1], 80.0) == [20.0, 0.0]
    assert bench.playback_gaps([1.0], [25], 80.0) == []


def test_stream_timeline_reproduces_the_one_then_25_cliff():
    """A producer at 8 ms per 80 ms frame: the 25-frame chunk after a 1-frame
    first chunk is ready long after the first frame's audio ran out (the
    cliff the vllm-omni page describes); with all codes up front it is not."""
    import bench
    lat = [2.0, 3.0, 2.5]
    r = bench.stream_timeline(lat, [1, 25, 25], 80.0, 8.0)
    assert r["ttfa_ms"] == 8.0 + 2.0
    assert r["uninterrupted_playback_ms"] == 26 * 8.0 + 3.0 - 80.0
    assert r["playback_stall_ms_total"] == 26 * 8.0 + 3.0 - (10.0 + 80.0)
    u = bench.stream_timeline(lat, [1, 25, 25], 80.0, 0.0)
    assert u["ttfa_ms"] == 2.0 and u["playback_stall_ms_total"] == 0.0 and u["uninterrupted_playback_ms"] == 2.0
