"""Host-side logic of bench.py that needs no GPU: the whole-job aggregation,
the max-over-ranks timing on two gloo ranks, and the reference arm's rank
handling under a multi-rank launch."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_aggregate_is_all_ranks_bytes_over_the_slowest_time():
    # 2 replicas of 1 GB each in 0.5 s (the slower rank's time) = 4 GB/s
    assert bench.aggregate(10 ** 9, 0.5, 2) == pytest.approx(4.0)
    assert bench.aggregate(10 ** 9, 0.5, 1) == pytest.approx(2.0)


def test_single_rank_reduce_and_barrier_are_no_ops():
    assert bench.reduce_max(3.5, 1) == 3.5
    bench.barrier(1)


def _rank_main(rank, world, port, results):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        t = bench.reduce_max(1.0 + rank, world)       # rank 1 is the slower one
        results[rank] = (t, bench.aggregate(10 ** 9, t, world))
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(results)
    assert res[0][0] == res[1][0] == 2.0
    assert res[0][1] == pytest.approx(1.0)             # 2 x 1 GB / 2 s


def test_dist_env_reads_the_launcher_variables(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "4")
    monkeypatch.setenv("RANK", "3")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.dist_env() == (4, 3, 1)


def test_reference_arm_on_a_non_zero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_reference_arm_prints_one_json_line():
    import json
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "2", "--warmup", "3"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_kernel_hash_ignores_comments_but_not_code():
    src = "int a = 1;  // one\n/* block\n comment */\n\nint b = 2;\n"
    assert bench.code_of(src) == "int a = 1;\nint b = 2;"
    assert bench.code_of(src.replace("// one", "// changed")) == bench.code_of(src)
    assert bench.code_of(src.replace("= 2", "= 3")) != bench.code_of(src)
