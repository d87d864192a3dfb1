"""The multi-GPU path of bench.py on the host: world_size 2 over gloo on CPU.

The layer has no exchange step, so N GPUs run N independent replicas; what crosses ranks is
the timing only (the job takes as long as its slowest rank) and rank 0 alone reports.  These
tests run that host logic with two gloo ranks and no GPU."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 1.5 + rank  # this rank's timed seconds
        slowest = bench.reduce_max(dist, mine, "cpu")
        dist.barrier()
        res = {"rank": rank, "slowest": slowest, "seed": bench.rank_seed(rank),
               "value": bench.job_value(world, 16, 10, slowest)}
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump(res, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time(tmp_path):
    import torch.multiprocessing as mp
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    # both ranks see the slower rank's time, and report the whole job's tokens over it
    assert [r["slowest"] for r in res] == [2.5, 2.5]
    assert all(r["value"] == world * 16 * 10 / 2.5 for r in res)
    # independent replicas: every rank draws its own layers and inputs
    assert res[0]["seed"] != res[1]["seed"]


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(None, 3.25, "cpu") == 3.25
    assert bench.job_value(1, 16, 50, 0.005) == 16 * 50 / 0.005


def test_reference_arm_runs_on_rank_0_only():
    """Under torchrun the reference arm's other ranks exit 0 at once and print nothing."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, env=env, timeout=120, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.strip() == ""


if __name__ == "__main__":
    sys.exit(pytest.main([__file__, "-q"]))
