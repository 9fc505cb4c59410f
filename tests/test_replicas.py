"""The multi-process path of bench.py on the CPU (gloo, world size 2): the
slowest rank times the replicas, the whole-job throughput counts every rank's
rows, and under torchrun the reference arm runs on rank 0 alone."""

import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    import bench

    # rank r took (r + 1) seconds for 10 steps of 4096 rows
    slowest = bench.max_over_ranks(float(rank + 1), torch.device("cpu"))
    q.put((rank, slowest, bench.replica_rows_per_s(4096, world, slowest / 10)))
    dist.destroy_process_group()


def test_slowest_rank_times_the_replicas():
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [2.0, 2.0]
    assert all(g[2] == pytest.approx(2 * 4096 / 0.2) for g in got)


def test_single_process_needs_no_process_group():
    import bench

    assert bench.max_over_ranks(1.5, torch.device("cpu")) == 1.5
    assert bench.replica_rows_per_s(8, 1, 0.5) == 16.0


def test_reference_arm_prints_once_under_torchrun():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3",
           "--workload", "tiny_8x10_f32", "--cpu-sample-s", "0.3"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["value"] > 0
