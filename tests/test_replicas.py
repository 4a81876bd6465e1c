"""The multi-GPU path of bench.py is N independent replicas (one process per
GPU, no collective on the data path): the timed region is bracketed by
barriers on every rank, the reported time is the slowest rank's, and the rate
counts the tokens of all replicas.  These tests run that host logic with two
gloo ranks on the CPU, with a fake step whose duration differs by rank."""
import os
import socket
import time

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        calls = []

        def step():
            calls.append(1)
            time.sleep(0.004 * (rank + 1))   # rank 1 is the slow one

        def wall_clock():
            t = {}

            def start():
                t["0"] = time.perf_counter()
            return start, lambda: (time.perf_counter() - t["0"]) * 1e3

        ms = bench.timed_replicas(step, 5, 3, dist.barrier, bench.make_allmax(world, torch.device("cpu")), wall_clock)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{ms} {len(calls)}\n")
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_time_the_slowest_rank(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(world)]
    ms = [float(r[0]) for r in res]
    assert ms[0] == ms[1]                      # every rank reports the max over ranks
    assert ms[0] >= 8.0                        # at least the slow rank's 8 ms per step
    assert all(int(r[1]) == 8 for r in res)    # 3 warm-up + 5 timed steps on each rank


def test_replica_rate_counts_all_ranks():
    assert bench.replica_rate(1, 262144, 29.0) == pytest.approx(262144 / 29.0 / 1e3)
    assert bench.replica_rate(4, 262144, 29.0) == pytest.approx(4 * 262144 / 29.0 / 1e3)


def test_single_process_allmax_is_identity():
    assert bench.make_allmax(1, torch.device("cpu"))(3.5) == 3.5


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the reference arm (the CPU oracle) runs on rank 0 alone;
    the other ranks exit 0 without work and print nothing."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_cpulist_parsing_for_the_host_binding():
    """The end-to-end pass binds to the GPU's local cores from a sysfs cpulist."""
    assert bench.parse_cpulist("0-3,8,10-11\n") == {0, 1, 2, 3, 8, 10, 11}
    assert bench.parse_cpulist("5") == {5}
    assert bench.parse_cpulist("") == set()
