"""Multi-rank host logic on CPU (gloo, world_size 2).

The path shards by output rows with no exchange; `bench.py --gpus N` runs N
independent replicas.  What crosses ranks is only the barrier and the
max-over-ranks of the timings, checked here without a GPU, plus the
reference arm's rule that ranks other than 0 exit without work.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r is (r+1) times slower on the kernel timing, and rank 0 is
        # slower end to end, so each max comes from a different rank
        mine = [10.0 * (rank + 1), 30.0 - 5.0 * rank]
        got = bench.max_over_ranks(mine, world, "cpu")
        dist.barrier()
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump(got, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    for r in range(2):
        got = json.load(open(tmp_path / f"r{r}.json"))
        assert got == [20.0, 30.0]


def test_job_throughput_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.job_throughput(1, 581_861_376, 20, 6.0)
    assert one == pytest.approx(581_861_376 * 20 / 6e-3 / 1e9)
    assert bench.job_throughput(4, 581_861_376, 20, 6.0) == pytest.approx(4 * one)


def test_reference_arm_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
