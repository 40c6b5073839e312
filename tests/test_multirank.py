"""The multi-GPU host logic of bench.py on CPU: two gloo ranks.

The path shards by tokens with no data-path collective (weak-scaling
replicas); the only cross-rank steps are the max-over-ranks step time and the
whole-job value built from it, and the reference arm runs on rank 0 only.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

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
    ms = [2.5, 3.0][rank]                       # rank 1 is the slowest
    ms_max = bench.reduce_max(ms, dist, "cpu")
    value = bench.whole_job_tflops(1.0e12, ms_max, world)
    with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
        f.write(f"{ms_max} {value}")
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for r in range(2):
        ms_max, value = map(float, (tmp_path / f"r{r}.txt").read_text().split())
        assert ms_max == 3.0                    # both ranks see the slowest rank
        assert value == pytest.approx(2 * 1.0e12 / 3.0e-3 / 1e12)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
