"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

The forward does not shard: under torchrun every rank runs its own replica on
its own batch, and the only cross-rank steps are the barrier, the max of the
timed totals and the whole-job throughput. These run here on gloo ranks.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank, dist)
        value = bench.job_throughput(world, 2048, 20, slowest)
        q.put((rank, slowest, value))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_slowest_rank_time_and_job_throughput_on_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = {}
        for _ in range(2):
            rank, slowest, value = q.get(timeout=120)
            got[rank] = (slowest, value)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    # both ranks see the slower rank's 15 ms; the job processed 2 x 2048 x 20 samples
    for rank in (0, 1):
        slowest, value = got[rank]
        assert slowest == 15.0
        assert value == pytest.approx(2 * 2048 * 20 / 15e-3)


def test_single_process_keeps_its_own_time():
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.job_throughput(1, 64, 1, 1.0) == pytest.approx(64000.0)


def test_reference_arm_under_torchrun_prints_once_from_rank_0():
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny_b64_k3",
           "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
