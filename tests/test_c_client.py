"""A plain C program as a user of the C ABI (tests/c_client/ag_gemm_client.c).

It includes only include/ag_gemm.h and the CUDA runtime, and links
libaggemm.so, with no Python and no torch in the way.  On CPU: it compiles and
links with gcc.  On a GB300: it runs an fp16 problem, an int8 problem on the
skinny path (80 rows) and one on the fused int8 path (200 rows), and its
output files are compared with the oracle (fp16 within the tolerance of the
parity tests, int8 C_i32 bit-exact and D within 1 fp16 ulp).
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

from all_gather_gemm_chunked_gb300 import build as _build
from all_gather_gemm_chunked_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    lib = _build.build()
    libdir = os.path.dirname(lib)
    exe = str(tmp_path_factory.mktemp("c_client") / "ag_gemm_client")
    cmd = ["gcc", "-O2", "-std=c99", "-Wall", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           os.path.join(HERE, "c_client", "ag_gemm_client.c"), "-o", exe,
           "-L", libdir, "-laggemm", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           f"-Wl,-rpath,{libdir}:{os.path.join(CUDA, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_client_compiles_and_links(client):
    assert os.access(client, os.X_OK)


def _write_problem(d, S, R, K, N, dtype, x):
    code = {"f16": 0, "i8": 1}[dtype]
    with open(os.path.join(d, "meta.txt"), "w") as f:
        f.write(f"{S} {R} {K} {N} {code}\n")
    for s, a in enumerate(x["shards"]):
        np.ascontiguousarray(a).tofile(os.path.join(d, f"shard{s}.bin"))
    np.ascontiguousarray(x["B"]).tofile(os.path.join(d, "B.bin"))
    if dtype == "i8":
        np.ascontiguousarray(x["bias"], dtype=np.int32).tofile(os.path.join(d, "bias.bin"))
        np.ascontiguousarray(x["scale"], dtype=np.float32).tofile(os.path.join(d, "scale.bin"))


@pytest.mark.gpu
@pytest.mark.parametrize("S,R,K,N,dtype", [
    (2, 100, 264, 200, "f16"),
    (2, 40, 512, 96, "i8"),       # 80 rows: the skinny kernel
    (2, 100, 512, 96, "i8"),      # 200 rows: the fused int8 kernel
])
def test_c_client_matches_oracle(client, oracle, tmp_path, S, R, K, N, dtype):
    from gpu_util import check_f16, f16_ulp_distance
    x = synth.make_inputs(S, R, K, N, dtype, 6100 + S * R + K + N)
    _write_problem(str(tmp_path), S, R, K, N, dtype, x)
    r = subprocess.run([client, str(tmp_path)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    M = S * R
    if dtype == "f16":
        C = np.fromfile(tmp_path / "C.bin", dtype=np.float32).reshape(M, N)
        check_f16(C, oracle.ag_gemm_f16(x["shards"], x["B"]), K, "C client fp16")
    else:
        Ci = np.fromfile(tmp_path / "Ci.bin", dtype=np.int32).reshape(M, N)
        D = np.fromfile(tmp_path / "D.bin", dtype=np.float16).reshape(M, N)
        Cref, Dref = oracle.ag_gemm_dequant(x["shards"], x["B"], x["bias"], x["scale"])
        assert np.array_equal(Ci, Cref)
        assert f16_ulp_distance(D, Dref).max() <= 1
