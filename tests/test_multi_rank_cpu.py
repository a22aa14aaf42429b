"""The N > 1 path of bench.py (independent replicas, no data-path collective)
on CPU: two gloo ranks agree on the slowest rank's time and report the
weak-scaling job throughput from it."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = [2.0, 3.5][rank]
        ms = bench.max_over_ranks(my_ms)
        q.put((rank, ms, bench.job_throughput(1e9, world, ms)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, value in res:
        assert ms == 3.5
        assert value == pytest.approx(2 * 1e9 / 3.5e-3)


def test_single_process_is_identity():
    import bench

    assert bench.max_over_ranks(1.25) == 1.25
    assert bench.job_throughput(10.0, 1, 1000.0) == pytest.approx(10.0)


def test_gpus_flag_starts_one_rank_per_gpu():
    """`bench.py --gpus N` outside torchrun re-runs itself as N ranks of torch.distributed.run on 127.0.0.1."""
    import sys

    import bench

    cmd = bench.relaunch_cmd(8, ["--gpus", "8", "--steps", "5"], 29511)
    assert cmd[:3] == [sys.executable, "-m", "torch.distributed.run"]
    assert "--nproc-per-node=8" in cmd and "--nnodes=1" in cmd
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert cmd[cmd.index("--master-port") + 1] == "29511"
    assert cmd[-5].endswith("bench.py") and cmd[-4:] == ["--gpus", "8", "--steps", "5"]
    assert 0 < bench.free_port() < 65536
