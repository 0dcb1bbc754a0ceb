"""The N > 1 path of bench.py on CPU: world-size-2 gloo ranks.

The decode does not shard across GPUs in this build (replicas only): each rank
runs the whole workload on its own GPU, with no collective on the data path.
What the ranks share is the timing.  The job took the slowest rank's time and
processed every rank's units, so the whole-job rate is ws * units / max_s.
This runs that aggregation over a real process group, and checks the
reference arm's rule that only rank 0 works and prints.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, ws: int, port: int, q) -> None:
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=ws)
    local_s = [0.5, 2.0][rank]  # rank 1 is the slow one
    rate, max_s = bench.replica_rate(local_s, 10, ws, "cpu")
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, rate, max_s))


def test_replica_rate_over_gloo():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(ws))
    for rank, rate, max_s in got:
        assert max_s == 2.0                   # every rank sees the slowest time
        assert rate == pytest.approx(ws * 10 / 2.0)


def test_single_rank_rate_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.replica_rate(0.25, 5, 1) == (20.0, 0.25)


def test_reference_arm_nonzero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_reference_arm_rank0_prints_one_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["n_gpus"] == 1


def test_routed_traffic_only_for_the_captured_kernel_source(tmp_path, monkeypatch):
    """roofline.traffic comes from a committed ncu record that carries the hash
    of the kernel source it was captured from; once the source changes the
    figure must be withheld (None), not reused."""
    sys.path.insert(0, ROOT)
    import bench
    src = tmp_path / "kernel.cu"
    src.write_text("// one version of the kernel\n")
    rec = tmp_path / "traffic.txt"
    rec.write_text("# comment\ndram_bytes_per_launch=1234\n"
                   f"source_sha256_16={bench.source_hash(str(src))}\n")
    monkeypatch.setattr(bench, "FFN_SOURCE", str(src))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(rec))
    got = bench.routed_traffic()
    assert got is not None and got["bytes_per_launch"] == 1234.0
    src.write_text("// another version of the kernel\n")
    assert bench.routed_traffic() is None
    rec.unlink()
    assert bench.routed_traffic() is None
