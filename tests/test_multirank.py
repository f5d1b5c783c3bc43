"""The N > 1 host logic of bench.py on CPU: two gloo ranks, each with its own
time; the reported time is the slowest rank's (no data-path collective exists:
every rank runs a whole workload on its own GPU)."""
import os
import socket

import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, values, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world)})
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = bench.dist_info()
        assert (r, lr, w) == (rank, rank, world)
        out[rank] = bench.reduce_max(values[rank], world)
        cfg = bench.config_block(world)
        assert f"x{world}" in cfg["parallelism"]
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_reduction():
    world = 2
    values = [3.25, 7.5]
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), values, out), nprocs=world, join=True,
                       start_method="spawn")
    assert out[0] == out[1] == max(values)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(4.0, 1) == 4.0
    f, b = bench.step_flops()
    assert abs(f - 1.0995e12) / 1.0995e12 < 1e-3 and abs(b - 2.7488e12) / 2.7488e12 < 1e-3
