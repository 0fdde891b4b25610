"""The multi-rank (replica) harness of bench.py on CPU: two gloo ranks.

bench.py runs one independent replica of the step per GPU; ranks only meet in
a barrier and in the max over ranks of their timings.  Here two CPU ranks
check that reduction and the whole-job throughput, and that the reference arm
does its work on rank 0 only.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [1.0 + rank, 10.0 - rank, 0.5 * (rank + 1)]
        got = bench.max_over_ranks(mine, dist, "cpu")
        value = bench.replica_throughput(1_000_000, world, got[0])
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"max": got, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_throughput_two_gloo_ranks(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    results = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in results:
        assert r["max"] == [2.0, 10.0, 1.0]
        # 2 replicas x 1 MB in 2 ms (the slower rank) = 1 GB/s
        assert r["value"] == pytest.approx(1.0)


def test_reference_arm_rank1_does_no_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                          "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    assert res.stdout.strip() == ""


def test_single_process_refuses_multi_gpu_without_launcher():
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2"], env=env,
                         capture_output=True, text=True, timeout=300)
    assert res.returncode != 0 and "torch.distributed.run" in res.stderr


def test_reference_arm_prints_one_line_on_rank0():
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                          "--steps", "3", "--warmup", "3", "--cpu-seconds", "1"], env=env, capture_output=True,
                         text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    lines = [l for l in res.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
