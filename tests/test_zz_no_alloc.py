"""The no-allocation fp16 entry point against the plan-based one.

ag_gemm_run_noalloc is for callers that must not call cudaMalloc, for example
an application whose own allocator already holds the device's memory, or a
latency-critical path where cudaMalloc/cudaFree (which may synchronise the
device) are not allowed.  Its staging workspace, counters and status word live
in a fixed array inside the library, shared by every call.  These tests call it
through the C ABI and require its C to match ag_gemm_run's within the fp16
tolerance used by the other GPU tests, on two calls in a row with different
inputs (the second call starts from the first call's leftovers in the array), and
compare the small cases with the CPU oracle as well.  A further test checks that
a call allocates nothing: the device's free memory is the same before and after
a second call on buffers that already exist.
"""
import numpy as np
import pytest

from gpu_util import check_f16

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from all_gather_gemm_chunked_gb300 import binding as B_  # noqa: E402
from all_gather_gemm_chunked_gb300 import synth  # noqa: E402
from all_gather_gemm_chunked_gb300.plan import Plan  # noqa: E402

DEV = torch.device("cuda:0")


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _plan_result(x, S, R, K, N, c):
    with Plan(S, S * R, K, N, "f16", c) as plan:
        C = plan.run([_dev(s) for s in x["shards"]], _dev(x["B"]))
        torch.cuda.synchronize()
        assert plan.status() == 0
    return C.cpu().numpy()


def _noalloc_result(x, S, R, K, N, c):
    shards = [_dev(s) for s in x["shards"]]
    Bd = _dev(x["B"])
    C = torch.full((S * R, N), float("nan"), dtype=torch.float32, device=DEV)
    status = torch.full((2,), -1, dtype=torch.int32, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    B_.ag_gemm_run_noalloc(S, S * R, K, N, c, [s.data_ptr() for s in shards], Bd.data_ptr(),
                           C.data_ptr(), status.data_ptr(), stream)
    torch.cuda.synchronize()
    assert status.cpu().tolist() == [0, 0], "device status of the no-allocation run"
    return C.cpu().numpy()


@pytest.mark.parametrize("S,R,K,N,c", [
    (2, 128, 256, 128, 16),   # the small fp16 workload
    (3, 200, 328, 392, 0),    # ragged tiles, K and N tails
    (2, 2048, 4096, 4096, 0), # the 2 x 2048-row, K = N = 4096 workload (16 MiB of staging)
])
def test_noalloc_matches_plan_on_two_calls_in_a_row(S, R, K, N, c, oracle):
    x1 = synth.make_inputs(S, R, K, N, "f16", 4100 + S + K)
    x2 = synth.make_inputs(S, R, K, N, "f16", 4200 + S + K)
    ref1 = _plan_result(x1, S, R, K, N, c)
    ref2 = _plan_result(x2, S, R, K, N, c)
    got1 = _noalloc_result(x1, S, R, K, N, c)
    got2 = _noalloc_result(x2, S, R, K, N, c)
    check_f16(got1, ref1, K, "first no-allocation call vs ag_gemm_run")
    check_f16(got2, ref2, K, "second no-allocation call vs ag_gemm_run")
    if S * R * K * N <= 64 * 1024 * 1024:
        # small enough for the fp64 CPU oracle: the same tolerance against it
        check_f16(got1, oracle.ag_gemm_f16(x1["shards"], x1["B"]), K,
                  "first no-allocation call vs the oracle")
        check_f16(got2, oracle.ag_gemm_f16(x2["shards"], x2["B"]), K,
                  "second no-allocation call vs the oracle")


def test_noalloc_call_allocates_no_device_memory():
    S, R, K, N = 2, 512, 1024, 512
    x = synth.make_inputs(S, R, K, N, "f16", 4300)
    shards = [_dev(s) for s in x["shards"]]
    Bd = _dev(x["B"])
    C = torch.empty((S * R, N), dtype=torch.float32, device=DEV)
    status = torch.zeros((2,), dtype=torch.int32, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    ptrs = [s.data_ptr() for s in shards]

    def call():
        B_.ag_gemm_run_noalloc(S, S * R, K, N, 0, ptrs, Bd.data_ptr(), C.data_ptr(),
                               status.data_ptr(), stream)
        torch.cuda.synchronize()

    call()  # the first call on the device looks up the array (and may load the module)
    free_before, _ = torch.cuda.mem_get_info(DEV)
    call()
    free_after, _ = torch.cuda.mem_get_info(DEV)
    assert status.cpu().tolist() == [0, 0]
    assert free_after == free_before, (
        f"device free memory changed across a no-allocation call: {free_before} -> {free_after}")


def test_noalloc_rejects_problems_beyond_its_scratch():
    S, R, K, N = 8, 4096, 4096, 256   # 7 x 4096 x 4096 x 2 B of staging > 64 MiB
    a = torch.zeros((R, K), dtype=torch.float16, device=DEV)
    Bd = torch.zeros((K, N), dtype=torch.float16, device=DEV)
    C = torch.zeros((S * R, N), dtype=torch.float32, device=DEV)
    with pytest.raises(B_.AgGemmError) as e:
        B_.ag_gemm_run_noalloc(S, S * R, K, N, 0, [a.data_ptr()] * S, Bd.data_ptr(),
                               C.data_ptr(), 0, 0)
    assert e.value.code == B_.ERR_UNSUPPORTED
    assert "scratch" in e.value.message
