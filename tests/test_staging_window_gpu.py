"""Bounded staging window on the GPU: a plan whose remote rows pass through W
slots of 256 rows, refilled under back-pressure, must give exactly the C of the
plain plan (same tiles, same fp32 sums) and of the oracle -- with slots reused
within a run, across repeated runs (monotonic credit counters), under injected
producer delays, after copy-only runs and after a timeout and reset.
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


def _dev(a, dt):
    t = torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    return t.view(torch.bfloat16) if dt == "bf16" else t


def _run(plan, x, dt, mode=None, check_status=True):
    if mode is not None:
        plan.set_mode(mode)
    shards = [_dev(s, dt) for s in x["shards"]]
    Bd = _dev(x["B"], dt)
    M, N = plan.M, plan.N
    if dt == "i8":
        Ci = torch.full((M, N), -7, dtype=torch.int32, device=DEV)
        D = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
        plan.dequant_run(shards, Bd, _dev(x["bias"], dt), _dev(x["scale"], dt), Ci, D)
        out = (Ci, D)
    else:
        C = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
        plan.run(shards, Bd, C)
        out = (C,)
    torch.cuda.synchronize()
    if check_status:
        assert plan.status() == 0, f"status word {plan.status_word():#x}"
    return [o.cpu().numpy() for o in out]


def _same(a, b):
    return all(np.array_equal(x.view(np.uint8), y.view(np.uint8)) for x, y in zip(a, b))


def _inputs(dt, S, R, K, N, seed):
    return synth.make_inputs(S, R, K, N, dt, seed)


CASES = [
    # dt, S, R, K, N, W: every case has more remote row blocks than slots
    ("f16", 4, 600, 256, 384, 8),    # 9 blocks, a ragged last block per shard (88 rows)
    ("f16", 8, 512, 320, 136, 8),    # 14 blocks, N not a multiple of 64
    ("bf16", 5, 1024, 128, 256, 8),  # 16 blocks, two uses of every slot
    ("i8", 5, 520, 1056, 208, 9),    # 12 blocks: slots 0-2 used twice, 3-8 once; 2 K segments
]


@pytest.mark.parametrize("dt,S,R,K,N,W", CASES)
def test_window_matches_plain_plan_and_oracle(oracle, dt, S, R, K, N, W):
    x = _inputs(dt, S, R, K, N, 6000 + S * 13 + K)
    with Plan(S, S * R, K, N, dt, staging_slots=W) as bp:
        g = bp.geometry
        assert g["staging_slots"] == W and g["staging_bytes"] == W * 256 * K * 2
        assert 256 % g["chunk_rows"] == 0
        got = _run(bp, x, dt)
        chunk = g["chunk_rows"]
    with Plan(S, S * R, K, N, dt, chunk) as pp:
        assert pp.geometry["staging_slots"] == 0
        plain = _run(pp, x, dt)
    assert _same(got, plain)
    if dt == "i8":
        Cref, Dref = oracle.ag_gemm_dequant(x["shards"], x["B"], x["bias"], x["scale"])
        assert np.array_equal(got[0], Cref)
    else:
        ref = (oracle.ag_gemm_f16 if dt == "f16" else oracle.ag_gemm_bf16)(x["shards"], x["B"])
        check_f16(got[0], ref, K, f"window {dt} S={S} R={R}")


def test_window_repeats_delays_modes_and_local_rank():
    dt, S, R, K, N, W = "f16", 4, 600, 256, 384, 8
    x = _inputs(dt, S, R, K, N, 61)
    with Plan(S, S * R, K, N, dt, staging_slots=W) as bp:
        ref = _run(bp, x, dt)
        for _ in range(3):                      # credit epochs 2..4
            assert _same(_run(bp, x, dt), ref)
        _run(bp, x, dt, B_.MODE_COPY_ONLY)      # no readers: credits untouched
        _run(bp, x, dt, B_.MODE_COMPUTE_ONLY)   # reads the window as it stands (timing only)
        assert _same(_run(bp, x, dt, B_.MODE_PIPELINED), ref)
        # a slow producer: every copy item sleeps, the readers must wait for it
        bp.set_debug(B_.DEBUG_DELAY_NS, 20000)
        assert _same(_run(bp, x, dt), ref)
        bp.set_debug(0, 0)
        for local in range(1, S):
            bp.set_local_rank(local)
            assert _same(_run(bp, x, dt), ref)
        bp.set_local_rank(0)
        with pytest.raises(B_.AgGemmError) as e:
            _run(bp, x, dt, B_.MODE_SEQUENTIAL)
        assert e.value.code == B_.ERR_UNSUPPORTED
        bp.reset()
        assert _same(_run(bp, x, dt, B_.MODE_PIPELINED), ref)


def test_window_timeout_then_reset():
    dt, S, R, K, N, W = "f16", 5, 1024, 128, 256, 8
    x = _inputs(dt, S, R, K, N, 62)
    with Plan(S, S * R, K, N, dt, staging_slots=W) as bp:
        ref = _run(bp, x, dt)
        bp.set_timeout_ns(20_000_000)
        bp.set_debug(B_.DEBUG_SKIP_ITEM, 3)     # a chunk of the first remote block never lands
        _run(bp, x, dt, check_status=False)
        assert bp.status() == B_.ERR_TIMEOUT
        bp.set_debug(0, 0)
        bp.reset()
        assert _same(_run(bp, x, dt), ref)


def test_window_plan_checks():
    with Plan(8, 8 * 1024, 256, 256, "f16", staging_slots=0) as p:  # default: two groups
        assert p.geometry["staging_slots"] == 16
    with Plan(2, 2 * 1024, 256, 256, "f16", staging_slots=8) as p:  # 4 blocks: plain layout
        assert p.geometry["staging_slots"] == 0
    with Plan(2, 64, 1024, 256, "i8", staging_slots=8) as p:        # skinny: plain layout
        assert p.geometry["staging_slots"] == 0 and p.path == B_.PATH_SKINNY_I8
    for slots, chunk in ((7, 0), (-1, 0), (8, 24)):
        with pytest.raises(B_.AgGemmError) as e:
            Plan(4, 4 * 3072, 256, 256, "f16", chunk, staging_slots=slots)
        assert e.value.code == B_.ERR_INVALID


GRID_CASES = [
    # dt, S, R, K, N, W (None = plain staging)
    ("f16", 4, 600, 256, 384, 8),
    ("i8", 5, 520, 1056, 208, 9),
    ("f16", 3, 1000, 512, 520, None),
    ("f16", 2, 1536, 8192, 512, None),    # 24 tiles split in two along K (both parts add into C)
    ("bf16", 2, 1536, 2048, 520, None),   # 24 tiles of 32 k-blocks split in two
    ("f16", 2, 2560, 2048, 1024, None),   # 76 whole tiles, then 4 split ones: on a small grid
                                          # a pair reaches its parts long before the others'
                                          # pairs start, and zeroes the tail blocks itself
    ("i8", 3, 512, 8192, 768, None),      # 18 tiles split in two (int32 partial sums)
]


@pytest.mark.parametrize("dt,S,R,K,N,W", GRID_CASES)
def test_any_grid_gives_the_same_result(dt, S, R, K, N, W):
    """Pair tiles are handed out at run time in schedule order, so the grid does
    not change C: one pair, a few pairs, and four times the pairs the GPU holds
    at once (the extra pairs start only as earlier ones finish -- the partial
    residency of a shared GPU -- and must never be waited for)."""
    x = _inputs(dt, S, R, K, N, 6500 + S * 7 + K)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    with Plan(S, S * R, K, N, dt, staging_slots=W) as plan:
        ref = _run(plan, x, dt)
        for ctas in (2, 6, 4 * sms - (4 * sms) % 2, 0):
            plan.set_grid(ctas)
            assert plan.grid == (ctas or plan.grid)
            assert _same(_run(plan, x, dt), ref), f"grid {ctas}"
        with pytest.raises(B_.AgGemmError):
            plan.set_grid(3)
