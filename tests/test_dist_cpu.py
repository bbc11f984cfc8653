"""The multi-process path of bench.py without a GPU: two gloo ranks on CPU.

The verify call has no exchange step, so N GPUs run N independent replicas;
what the ranks share is the bench's host logic -- rendezvous, the barriers
around the timed region, the max over ranks of the elapsed time, and the
whole-job figure computed from it -- and the rule that only rank 0 prints.
"""
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


def _worker(rank, world, port, out_dir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.init_dist(world, "gloo")
    assert d is not None and d.get_world_size() == world and d.get_rank() == rank
    bench.barrier(d)
    elapsed = 100.0 + 7.0 * rank          # each rank's own timed region (ms)
    slowest = bench.max_over_ranks(d, elapsed)
    bench.barrier(d)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"slowest": slowest, "us_per_call": bench.job_us_per_call(slowest / 4, world)}, f)
    d.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    for r in res:
        assert r["slowest"] == 107.0                     # max over ranks, seen by every rank
        assert r["us_per_call"] == 107.0 / 4 * 1000 / 2  # 2 calls per step, 4 steps


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(None, 3.5) == 3.5
    assert bench.job_us_per_call(2.0, 1) == 2000.0


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1"],
                       capture_output=True, text=True, env=env, cwd=ROOT, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "", r.stdout + r.stderr


def test_gpus_flag_without_launcher_spawns_one_process_per_replica():
    # `bench.py --gpus 2` with no WORLD_SIZE relaunches itself as two local
    # processes; the reference arm needs no GPU, and only rank 0 prints
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--workload", "tiny", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, env=env, cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2


def test_gpus_flag_must_match_the_launcher():
    env = dict(os.environ, RANK="0", WORLD_SIZE="2", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "4",
                        "--steps", "1"], capture_output=True, text=True, env=env, cwd=ROOT, timeout=300)
    assert r.returncode != 0 and "disagrees" in (r.stdout + r.stderr)
