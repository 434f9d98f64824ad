"""The multi-GPU path of bench.py on CPU: world size 2 over gloo.

Decode of independent sequences needs no exchange, so N GPUs run N replicas;
the only cross-rank steps are the barrier around the timed region and the
max-over-ranks of the elapsed time, from which rank 0 reports the whole-job
throughput.  These run here with the gloo backend and fake timings.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        local_ms = [120.0, 150.0][rank]          # the slower rank decides
        ms_max = bench.max_over_ranks(local_ms, world)
        value = bench.job_throughput(4, 10, world, ms_max / 1000.0)
        dist.barrier()
        q.put((rank, ms_max, value))
    finally:
        dist.destroy_process_group()


def test_two_ranks_report_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms_max, value in got:
        assert ms_max == 150.0
        # 4 sequences x 10 steps on each of 2 ranks over the slowest rank's 0.15 s
        assert value == pytest.approx(4 * 10 * 2 / 0.150)


def test_reference_arm_only_rank0_works(monkeypatch, capsys):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    bench.run_reference(bench.parse())     # returns at once on ranks other than 0
    assert capsys.readouterr().out == ""
