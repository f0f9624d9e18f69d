"""The multi-rank side of the benchmark on CPU (gloo, world size 2): the
whole-job aggregation of a weak-scaling run, and the reference arm under
torchrun, where rank 0 alone does work and prints one JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r: 10 steps taking 100 + 50 r ms in total, its own workload size
        ms, tflops, tok_s = bench.aggregate(100.0 + 50.0 * rank, 10, 1e12 * (1 + rank),
                                            1000 * (1 + rank), world)
        out.put((rank, ms, tflops, tok_s, bench.reduce_over_ranks(rank + 1.0, world, "sum")))
    finally:
        dist.destroy_process_group()


def test_aggregate_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    slow_ms = 150.0 / 10  # the slower rank sets the job's time
    for rank, ms, tflops, tok_s, s in res:
        assert ms == pytest.approx(slow_ms)
        assert tflops == pytest.approx(3e12 / (slow_ms * 1e-3) / 1e12)
        assert tok_s == pytest.approx(3000 / (slow_ms * 1e-3))
        assert s == 3.0


def test_aggregate_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    ms, tflops, tok_s = bench.aggregate(50.0, 5, 2e12, 4000, 1)
    assert ms == 10.0 and tflops == pytest.approx(200.0) and tok_s == pytest.approx(4e5)


@pytest.mark.slow
def test_reference_arm_under_torchrun():
    env = dict(os.environ, OMP_NUM_THREADS=str(max(1, (os.cpu_count() or 2) // 2)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "3", "--sample-seconds", "0.5",
           "--sample-max-tokens", "256"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_recorded_traffic_follows_the_sources(tmp_path, monkeypatch):
    # The DRAM bytes of a committed ncu record count only while the kernel's
    # sources hash to the value recorded with them.
    import hashlib
    sys.path.insert(0, ROOT)
    import bench
    (tmp_path / "profiles").mkdir()
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    rec = {"kernel": "k", "workload": "w", "bytes_per_launch": 123,
           "source_files": ["k.cu"],
           "source_sha256_16": hashlib.sha256(b"kernel v1\n").hexdigest()[:16]}
    (tmp_path / "profiles" / "k_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("k", "w") == 123
    assert bench.recorded_traffic("k", "another workload") is None
    assert bench.recorded_traffic("missing", "w") is None
    src.write_text("kernel v2\n")
    assert bench.recorded_traffic("k", "w") is None

