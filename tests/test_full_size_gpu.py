"""Full-size parity of the workloads that extend the method, in the launch
configuration bench.py times, on sampled outputs the oracle computes one by one.

Workload 7: one rank of the N-sharded collective matmul: B and C are the rank's
column blocks of K x 8192 / M x 8192 matrices (row pitches), the plan's local
rank sets the ring order.  Workloads 8 and 9: workloads 4 and 3 with the remote
rows staged through a bounded window of 16 slots of 256 rows.  Every (shard,
m-tile, n-tile) contributes its four corners and random points; int8 C_i32 is
bit-exact and D within 1 fp16 ulp, fp16 within the fp16 tolerance.  Row and
column checksums over the whole fp16 output hold at any size.
"""
import numpy as np
import pytest

from gpu_util import check_f16, f16_ulp_distance, tile_samples

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from all_gather_gemm_chunked_gb300 import synth  # noqa: E402
from all_gather_gemm_chunked_gb300.plan import Plan  # noqa: E402

DEV = torch.device("cuda:0")


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def test_full_size_nsharded_rank(oracle):
    w = synth.WORKLOADS[7]
    x = synth.workload_inputs(w)
    shards = [_dev(s) for s in x["shards"]]
    cols = slice(w.rank * w.N, (w.rank + 1) * w.N)
    B_full = _dev(x["B"])                                    # K x (n_blocks * N)
    C_full = torch.full((w.M, w.N * w.n_blocks), float("nan"), dtype=torch.float32, device=DEV)
    with Plan(w.S, w.M, w.K, w.N, w.dtype, w.chunk_rows) as plan:
        plan.set_local_rank(w.rank)
        plan.run(shards, B_full[:, cols], C_full[:, cols])
        torch.cuda.synchronize()
        assert plan.status() == 0
    C = C_full[:, cols].cpu().numpy()
    others = C_full.cpu().numpy()
    others = np.delete(others, np.arange(cols.start, cols.stop), axis=1)
    assert np.isnan(others).all(), "columns outside the rank's block were written"
    rng = np.random.default_rng(7)
    rows, cc = tile_samples(rng, w.M, w.N, w.R)
    Bb = np.ascontiguousarray(x["B_rank"])
    check_f16(C[rows, cc], oracle.ag_gemm_f16_at(x["shards"], Bb, rows, cc), w.K,
              "workload 7 samples")
    A = np.concatenate(x["shards"]).astype(np.float64)
    Bf = Bb.astype(np.float64)
    Cd = C.astype(np.float64)
    assert np.abs(Cd.sum(axis=1) - A @ Bf.sum(axis=1)).max() <= 1e-3 * np.sqrt(w.K * w.N)
    assert np.abs(Cd.sum(axis=0) - A.sum(axis=0) @ Bf).max() <= 1e-3 * np.sqrt(w.K * w.M)


def test_full_size_window_int8(oracle):
    w = synth.WORKLOADS[8]
    x = synth.workload_inputs(w)
    with Plan(w.S, w.M, w.K, w.N, w.dtype, w.chunk_rows, staging_slots=w.staging_slots) as plan:
        assert plan.geometry["staging_slots"] == w.staging_slots
        Ci, D = plan.dequant_run([_dev(s) for s in x["shards"]], _dev(x["B"]), _dev(x["bias"]),
                                 _dev(x["scale"]))
        torch.cuda.synchronize()
        assert plan.status() == 0
    Ci, D = Ci.cpu().numpy(), D.cpu().numpy()
    rng = np.random.default_rng(8)
    rows, cc = tile_samples(rng, w.M, w.N, w.R)
    Cref, Dref = oracle.ag_gemm_dequant_at(x["shards"], x["B"], x["bias"], x["scale"], rows, cc)
    assert np.array_equal(Ci[rows, cc], Cref)
    assert f16_ulp_distance(D[rows, cc], Dref).max() <= 1


def test_full_size_window_f16(oracle):
    w = synth.WORKLOADS[9]
    x = synth.workload_inputs(w)
    with Plan(w.S, w.M, w.K, w.N, w.dtype, w.chunk_rows, staging_slots=w.staging_slots) as plan:
        assert plan.geometry["staging_slots"] == w.staging_slots
        C = plan.run([_dev(s) for s in x["shards"]], _dev(x["B"]))
        torch.cuda.synchronize()
        assert plan.status() == 0
    C = C.cpu().numpy()
    rng = np.random.default_rng(9)
    rows, cc = tile_samples(rng, w.M, w.N, w.R)
    check_f16(C[rows, cc], oracle.ag_gemm_f16_at(x["shards"], x["B"], rows, cc), w.K,
              "workload 9 samples")
    A = np.concatenate(x["shards"]).astype(np.float64)
    Bf = x["B"].astype(np.float64)
    Cd = C.astype(np.float64)
    assert np.abs(Cd.sum(axis=1) - A @ Bf.sum(axis=1)).max() <= 1e-3 * np.sqrt(w.K * w.N)
    assert np.abs(Cd.sum(axis=0) - A.sum(axis=0) @ Bf).max() <= 1e-3 * np.sqrt(w.K * w.M)
