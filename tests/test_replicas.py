"""The multi-GPU path of bench.py on CPU: two gloo ranks on 127.0.0.1.

Each box has one GPU and the path has no data exchange (replicas only), so
what is tested is the host logic: every rank ends with the slowest rank's
times, and the whole-job throughput counts the work of all ranks over that
time.
"""
import os
import socket

import pytest


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_dir):
    import torch.distributed as dist

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        total_ms, s8_ms = bench.replica_times(dist, "cpu", *times[rank])
        tops = bench.job_tops(1e12, 5, world, s8_ms)
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(f"{total_ms} {s8_ms} {tops}\n")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_replica_times_take_the_slowest_rank(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    world = 2
    times = [(30.0, 4.0), (25.0, 5.0)]  # (step total ms, INT8 GEMM ms) per rank
    mp.start_processes(_rank_main, args=(world, _free_port(), times, str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    got = [tuple(float(v) for v in (tmp_path / f"r{r}.txt").read_text().split()) for r in range(world)]
    for total_ms, s8_ms, tops in got:
        assert total_ms == 30.0 and s8_ms == 5.0
        # 2 ranks x 5 steps x 1e12 ops over the slowest 5 ms
        assert tops == pytest.approx(2 * 5 * 1e12 / 5e-3 / 1e12)


def test_single_process_keeps_its_own_times():
    import bench
    assert bench.replica_times(None, "cpu", 12.5, 3.0) == (12.5, 3.0)
    assert bench.job_tops(2.0 * 8192 ** 3, 5, 1, 3.6) == pytest.approx(5 * 2.0 * 8192 ** 3 / 3.6e-3 / 1e12)
