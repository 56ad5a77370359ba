"""Multi-process (gloo, world size 2, CPU) checks of the replica path of
bench.py: the step time is the slowest rank's, the throughput counts every
rank's bytes, and the reference arm does no work on ranks other than 0."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = [0.002, 0.003][rank]          # seconds per step on this rank
    slowest, gbs = bench.replica_throughput(local, 1.5e9)
    q.put((rank, slowest, gbs, bench.max_over_ranks(rank + 10.0)))
    dist.barrier()
    dist.destroy_process_group()


def test_replica_throughput_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, gbs, mx in got:
        assert slowest == pytest.approx(0.003)
        assert gbs == pytest.approx(2 * 1.5e9 / 0.003 / 1e9)
        assert mx == pytest.approx(11.0)


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.replica_throughput(0.5, 1e9) == (0.5, pytest.approx(2.0))


def test_reference_arm_idle_on_other_ranks(monkeypatch):
    import argparse

    import bench
    import synth
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(gpus=2, steps=1, warmup=0, impl="reference")
    assert bench.run_reference(args, synth.v7b()) == 0
