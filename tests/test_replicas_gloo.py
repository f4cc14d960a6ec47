"""The N>1 host path of bench.py on CPU: world size 2 over gloo.

Replicas only: every rank runs the whole workload on its own GPU, so the only
cross-rank step is the timing reduction (barrier + max over ranks) and rank 0's
single JSON line.  These tests run that logic with gloo ranks on the CPU."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier()
        t_max = bench.reduce_max(times[rank])
        v = bench.whole_job_value(1e12, world, t_max)
        q.put((rank, t_max, v))
    finally:
        dist.destroy_process_group()


def test_reduce_max_and_weak_scaling_value_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [0.5, 2.0]
    procs = [ctx.Process(target=_worker, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t_max, v in out:
        assert t_max == 2.0                      # the slowest rank decides
        assert v == pytest.approx(1e12 * 2 / 2.0 * 1e-12)  # N * units / t_max


def test_single_process_reduce_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(1.25) == 1.25
    assert bench.whole_job_value(2e12, 1, 2.0) == pytest.approx(1.0)


def test_reference_arm_under_torchrun_two_ranks():
    """bench.py --impl reference with 2 gloo ranks: rank 0 prints one JSON line,
    rank 1 exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.join(ROOT, "bench.py"),
           "--gpus", "2", "--impl", "reference", "--workload", "1", "--steps", "2",
           "--warmup", "0", "--ref-step-seconds", "0.2"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT,
                       env={**os.environ, "OMP_NUM_THREADS": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0
