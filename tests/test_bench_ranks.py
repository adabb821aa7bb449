"""The multi-rank path of bench.py on the CPU: two gloo ranks, one replica of
the work each (weak scaling).  The whole-job rate counts every rank's units
over the slowest rank's time, as the GPU run does over NCCL."""
import os
import socket

import pytest


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, seconds, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()                      # the timed region starts together
        rate, t = bench.whole_job(100.0, seconds[rank], world,
                                  bench.dist_max(dist, torch.device("cpu")))
        dist.barrier()
        out.put((rank, rate, t))
    finally:
        dist.destroy_process_group()


def test_whole_job_rate_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    seconds = [1.0, 2.5]                    # rank 1 is the slower one
    procs = [ctx.Process(target=_rank, args=(r, 2, port, seconds, out)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(out.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [r for r, _, _ in got] == [0, 1]
    for _, rate, t in got:
        assert t == 2.5                     # every rank reports the slowest rank's time
        assert rate == pytest.approx(2 * 100.0 / 2.5)


def test_whole_job_single_rank_needs_no_group():
    import bench
    assert bench.whole_job(300.0, 1.5, 1) == (200.0, 1.5)
