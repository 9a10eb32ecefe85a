"""The multi-rank path on CPU (gloo, world size 2): the path shards into independent replicas,
one per rank ("replicas only", weak scaling), so the only cross-rank steps are the barrier and
the reductions of the timed totals; the reference arm runs on rank 0 alone."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r timed 10 (r + 1) ms over 5 steps and processed 32 + r queries
        value, ms_per_step = bench.job_throughput(10.0 * (rank + 1), 32 + rank, 5, dist, "cpu")
        dist.barrier()
    finally:
        dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"value": value, "ms_per_step": ms_per_step}, f)


def test_job_throughput_over_two_gloo_ranks(tmp_path):
    """Every rank sees the slowest rank's time and the queries of all ranks."""
    mp.spawn(_worker, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    for rank in range(2):
        r = json.load(open(tmp_path / f"rank{rank}.json"))
        assert r["ms_per_step"] == pytest.approx(20.0 / 5)            # max(10, 20) ms / 5 steps
        assert r["value"] == pytest.approx((32 + 33) / (4.0 / 1000))  # 65 queries per 4 ms


def test_job_throughput_single_rank():
    import importlib
    sys.path.insert(0, ROOT)
    bench = importlib.import_module("bench")
    value, ms = bench.job_throughput(30.0, 32, 10)
    assert ms == pytest.approx(3.0) and value == pytest.approx(32 / 0.003)


def test_reference_arm_under_torchrun_two_ranks():
    """`bench.py --impl reference` launched under torchrun with 2 ranks: rank 0 alone runs the
    oracle and prints one JSON line; rank 1 exits 0 without work or output."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "--tee", "3",
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--workload", "decode_1x4096", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if '"impl": "reference"' in ln]
    assert len(lines) == 1, r.stdout[-2000:]
    rec = json.loads(lines[0][lines[0].index("{"):])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["e2e"]["unit"] == rec["unit"]
