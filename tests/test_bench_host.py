"""Host-side logic of bench.py that runs without a GPU: the max-over-ranks
reduction across two processes (gloo, world size 2), the whole-job
throughput formula, and the launch and kernel-name bookkeeping."""

import importlib.util
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench = load_bench()
        # rank r's (total, e2e) times: the slowest rank must win per element
        mine = [10.0 + rank, 30.0 - rank]
        q.put((rank, bench.reduce_max(mine, world)))
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_ranks():
    world, port = 2, free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0] == got[1] == [11.0, 30.0]


def test_reduce_max_single_rank_is_identity():
    bench = load_bench()
    assert bench.reduce_max([1.5, 2.5], 1) == [1.5, 2.5]


def test_job_throughput_is_weak_scaling_over_the_slowest_rank():
    bench = load_bench()
    # 1 TFLOP per step per rank, 10 steps, slowest rank 5 ms -> 2 PFLOP/s per rank
    one = bench.job_throughput(1e12, 1, 10, 5.0)
    assert one == pytest.approx(2000.0)
    assert bench.job_throughput(1e12, 4, 10, 5.0) == pytest.approx(4 * one)


def test_launch_and_kernel_bookkeeping():
    bench = load_bench()
    for d in (64, 128, 256):
        assert bench.bwd_launches(d) == 2        # dQ (with Delta) + dK/dV
    assert "fa_bwd_dq_kernel<128,true>" in bench.bwd_kernel_names(128, True)
    assert "fa_bwd256_dq_kernel<false> (with Delta)" in bench.bwd_kernel_names(256, False)
    # the benchmark's algorithmic count: 4 N^2 D per head forward, 2.5x backward
    assert bench.flops_fwd(128, 8, 1024, 128, False, 1024) == pytest.approx(4 * 1024 * 1024 ** 2 * 128)


def test_reference_arm_prints_its_line():
    # the reference arm is the fp64 CPU oracle on a bounded sample of the
    # workload; it needs no GPU
    import json
    import subprocess
    import sys
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [json.loads(x) for x in out.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["warmup"] >= 3
