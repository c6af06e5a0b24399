"""The benchmark's multi-process path on the CPU: two gloo ranks (world_size 2) agree on
the slowest rank's times, the whole-job rate counts every rank's work, and the
reference arm prints only on rank 0."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        vals = bench.reduce_max_over_ranks([1.0 + rank, 10.0 - rank, 0.25 * rank])
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump(vals, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest(tmp_path):
    port = _free_port()
    mp.spawn(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        assert json.load(open(tmp_path / f"r{r}.json")) == [2.0, 10.0, 0.25]


def test_whole_job_rate_counts_all_ranks():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_tflops(1e12, 1, 1.0)
    assert abs(one - 1000.0) < 1e-9
    assert abs(bench.whole_job_tflops(1e12, 4, 1.0) - 4 * one) < 1e-9


def test_reference_arm_is_silent_on_other_ranks():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
