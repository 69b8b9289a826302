"""The benchmark's multi-GPU path, exercised on CPU with gloo ranks.

The step has no exchange between GPUs (each rank is an independent replica),
so what N > 1 adds is host logic: every rank times its own step, the
slowest rank's time counts (max over ranks), and rank 0 reports the whole
job's rate, N times one replica's work over that time.  Two gloo processes
check the reduction and the aggregate; a torchrun launch of the reference arm
checks that only rank 0 prints, once.
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
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_q):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        # rank r's step and end-to-end times (ms)
        mine = [1.0 + rank, 10.0 - 3.0 * rank]
        got = bench.max_over_ranks(mine, "cpu")
        out_q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # every rank sees the slowest rank's step time and e2e time
    assert results[0] == results[1] == [2.0, 10.0]


def test_single_process_reduction_is_identity():
    assert bench.max_over_ranks([3.5, 1.25], "cpu") == [3.5, 1.25]


def test_aggregate_rate_is_whole_job_over_slowest_rank():
    # 2 replicas, 1e9 bytes each per step, slowest step 2 ms -> 1e12 B/s
    assert bench.aggregate_rate(2, 1e9, 2.0) == pytest.approx(1e12)
    assert bench.aggregate_rate(1, 64, 0.5) == pytest.approx(128000.0)


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                       timeout=300)
    assert r.returncode == 0, r.stderr.decode()[-2000:]
    lines = [ln for ln in r.stdout.decode().splitlines() if ln.startswith("{")]
    assert len(lines) == 1, lines
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["value"] > 0 and rec["n_gpus"] == 2
    # the reference arm's line carries the contract's keys, on the product's metric
    assert rec["metric"] == bench.METRIC and rec["unit"] == "GB/s"
    assert rec["higher_is_better"] is True and rec["scaling"] == "weak"
    cb = rec["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == rec["value"]
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["e2e"]["value"] == rec["value"]
