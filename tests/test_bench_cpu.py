"""The benchmark's host logic without a GPU: the max over ranks and the
whole-job throughput with two gloo ranks, and the reference arm (the fp64
oracle on the host), which only rank 0 runs."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r took 10 + r ms for its GEMMs and 20 - r ms for its step
    got = bench.max_over_ranks([10.0 + rank, 20.0 - rank], dist)
    value = bench.whole_job_tflops(world, 2.0e12, got[0])
    q.put((rank, got, value))
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, value in res:
        assert got == [11.0, 20.0]                     # the slowest rank's times
        assert value == pytest.approx(2 * 2.0e12 / 11e-3 / 1e12)
    assert bench.max_over_ranks([3.5, 4.0]) == [3.5, 4.0]   # one process


def _run_reference(env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--steps", "3", "--warmup", "3"], capture_output=True, text=True,
                          env=env, timeout=600, cwd=ROOT)


def test_reference_arm_runs_on_rank_zero_only():
    r1 = _run_reference({"RANK": "1", "WORLD_SIZE": "2"})
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _run_reference({"RANK": "0", "WORLD_SIZE": "1"})
    assert r0.returncode == 0, r0.stderr[-2000:]
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 3 and line["warmup"] == 3
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_rejects_short_warmup():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "1"], capture_output=True, text=True,
                       timeout=300, cwd=ROOT)
    assert r.returncode != 0 and "warmup" in r.stderr


def test_bench_inputs_do_not_reuse_a_cache_stream():
    # paged_kv(seed) draws K and V from seeds seed + 1 and seed + 2; a query
    # drawn from one of them would equal cached keys row for row
    assert bench.seed_collisions() == []
    bad = dict(bench.SEEDS["step"], q=bench.SEEDS["step"]["kv"] + 1)
    saved = bench.SEEDS["step"]
    try:
        bench.SEEDS["step"] = bad
        assert ("step", "q") in bench.seed_collisions()
    finally:
        bench.SEEDS["step"] = saved
