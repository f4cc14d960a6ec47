"""AG_GEMM_LOG: the library's stderr log (0 off, 1 errors, 2 plans, 3 runs),
read once per process, so each case runs in a child process."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys
sys.path.insert(0, {root!r})
from all_gather_gemm_chunked_gb300 import binding as B
try:
    B.ag_gemm_validate(2, 64, 100, 64, 1, 0)   # int8 needs K % 16 == 0
except Exception as e:
    print("raised", type(e).__name__)
print("chunk", B.ag_gemm_choose_chunk_rows(4096))
"""


def _run(level):
    env = dict(os.environ)
    env.pop("AG_GEMM_LOG", None)
    if level is not None:
        env["AG_GEMM_LOG"] = str(level)
    r = subprocess.run([sys.executable, "-c", SCRIPT.format(root=ROOT)], env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "raised" in r.stdout and "chunk 64" in r.stdout
    return r.stderr


def test_log_off_by_default():
    assert "[ag_gemm]" not in _run(None)
    assert "[ag_gemm]" not in _run(0)


@pytest.mark.parametrize("level", [1, 3])
def test_log_reports_errors(level):
    err = _run(level)
    lines = [l for l in err.splitlines() if l.startswith("[ag_gemm]")]
    assert len(lines) == 1, err
    assert "error -1" in lines[0] and "K % 16 == 0" in lines[0]


GPU_SCRIPT = r"""
import sys
sys.path.insert(0, {root!r})
import torch
from all_gather_gemm_chunked_gb300.plan import Plan
dev = torch.device("cuda:0")
shards = [torch.randn(128, 256, device=dev).half() for _ in range(2)]
B = torch.randn(256, 128, device=dev).half()
with Plan(2, 256, 256, 128, "f16") as plan:
    plan.run(shards, B)
    assert plan.status() == 0
torch.cuda.synchronize()
print("ok")
"""


@pytest.mark.gpu
def test_log_plans_and_runs_gpu():
    env = dict(os.environ, AG_GEMM_LOG="3")
    r = subprocess.run([sys.executable, "-c", GPU_SCRIPT.format(root=ROOT)], env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "ok" in r.stdout, r.stderr
    lines = [l for l in r.stderr.splitlines() if l.startswith("[ag_gemm]")]
    assert any("fused path" in l and "S=2 M=256 K=256 N=128" in l for l in lines), r.stderr
    assert any("fused run enqueued" in l for l in lines), r.stderr
    assert any("destroyed" in l for l in lines), r.stderr
    assert not any("error" in l for l in lines), r.stderr
