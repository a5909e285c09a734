"""The N > 1 path of the benchmark: independent replicas, one process per GPU,
whose figures are combined on the host (the slowest rank's time, the bytes
of all ranks).  Run here as two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, b = bench.combine_ranks(dist, torch, world, 10.0 + 5.0 * rank, 1e9 * (rank + 1), torch.device("cpu"))
        q.put((rank, ms, b))
    finally:
        dist.destroy_process_group()


def test_two_replicas_combine_on_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, b in got:  # every rank sees the same whole-job figures
        assert ms == pytest.approx(15.0) and b == pytest.approx(3e9)


def test_reference_arm_other_ranks_do_nothing(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    assert bench.run_reference(bench.parse(["--impl", "reference"])) is None
    assert capsys.readouterr().out == ""
