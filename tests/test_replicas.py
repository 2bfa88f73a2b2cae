"""The host side of bench.py on the CPU: the multi-process path (gloo, world
size 2) and the reference arm.

The hot path does not shard across GPUs here: under torch.distributed.run
every rank runs an independent replica, the job's time is the slowest
replica's, and the throughput counts every replica's bytes. These tests run
that host logic with two gloo ranks, and one step of the reference arm (the
CPU oracle); no GPU and no CUDA call is involved.
"""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, lr = bench.replica_env()
        elapsed = [0.25, 0.75][rank]          # seconds of this replica's timed region
        slowest = bench.max_over_ranks(elapsed, w)
        value = bench.job_throughput(w, 1.0e9, 4, slowest)
        dist.barrier()
    finally:
        dist.destroy_process_group()
    with open(os.path.join(out_dir, f"{rank}.json"), "w") as f:
        json.dump(dict(world=w, rank=r, local_rank=lr, slowest=slowest, value=value), f)


def test_two_gloo_ranks_time_the_slowest_replica(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    for rank in (0, 1):
        with open(tmp_path / f"{rank}.json") as f:
            d = json.load(f)
        assert (d["world"], d["rank"], d["local_rank"]) == (2, rank, rank)
        assert d["slowest"] == 0.75
        # two replicas, 1 GB each per step, 4 steps, in the slowest replica's 0.75 s
        assert abs(d["value"] - 2 * 4 / 0.75) < 1e-12


def test_one_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.5, 1) == 0.5
    assert abs(bench.job_throughput(1, 2.0e9, 3, 1.5) - 4.0) < 1e-12


def test_reference_arm_prints_only_on_rank_zero():
    """Under torch.distributed.run the reference arm runs on rank 0 alone: any
    other rank exits 0 without output (and without starting the oracle)."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_json_line():
    """One step of the reference arm (the CPU oracle) on a single process: the
    JSON line carries the bench's metric, a cpu_baseline describing the run
    and an e2e entry without host-device copies."""
    sys.path.insert(0, ROOT)
    import bench
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["steps"] == 1
    assert d["value"] > 0 and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
