"""GPU parity: the CUDA path against the CPU oracle, through the C ABI.

fp16 path: relative Frobenius error <= 1e-4 and max abs error <= 1e-3 sqrt(K)
against the fp64 oracle.  int8 path: C_i32 bit-exact; D within 1 fp16 ulp (the
oracle follows the same fp32 dequant definition, so D is expected bit-exact).
Small and ragged cases are compared element by element; the full-size
workloads are compared at sampled points (every tile's corners plus random
points) and through row/column checksums that hold at any size.  The streaming
machinery is checked by invariants: every run mode, chunk size and local rank
gives bit-identical C, poisoned staging never leaks, injected delays change
nothing, and a chunk that never lands ends in a TIMEOUT status, not a hang.
"""
import numpy as np
import pytest

from gpu_util import check_f16, f16_ulp_distance, tile_samples

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from all_gather_gemm_chunked_gb300 import binding as B_  # noqa: E402
from all_gather_gemm_chunked_gb300 import synth  # noqa: E402
from all_gather_gemm_chunked_gb300.plan import Plan  # noqa: E402

DEV = torch.device("cuda:0")


def _to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def run_f16(x, S, R, K, N, chunk_rows=0, mode=None, local=None, debug=None, plan=None):
    own = plan is None
    if own:
        plan = Plan(S, S * R, K, N, "f16", chunk_rows)
    try:
        if mode is not None:
            plan.set_mode(mode)
        if local is not None:
            plan.set_local_rank(local)
        if debug is not None:
            plan.set_debug(*debug)
        shards = [_to_dev(s) for s in x["shards"]]
        Bd = _to_dev(x["B"])
        C = torch.full((S * R, N), float("nan"), dtype=torch.float32, device=DEV)
        plan.run(shards, Bd, C)
        torch.cuda.synchronize()
        assert plan.status() == 0, f"status word {plan.status_word():#x}"
        return C.cpu().numpy()
    finally:
        if own:
            plan.close()


def run_i8(x, S, R, K, N, chunk_rows=0, mode=None, local=None, plan=None):
    own = plan is None
    if own:
        plan = Plan(S, S * R, K, N, "i8", chunk_rows)
    try:
        if mode is not None:
            plan.set_mode(mode)
        if local is not None:
            plan.set_local_rank(local)
        shards = [_to_dev(s) for s in x["shards"]]
        Ci = torch.full((S * R, N), -7, dtype=torch.int32, device=DEV)
        D = torch.full((S * R, N), float("nan"), dtype=torch.float16, device=DEV)
        plan.dequant_run(shards, _to_dev(x["B"]), _to_dev(x["bias"]), _to_dev(x["scale"]), Ci, D)
        torch.cuda.synchronize()
        assert plan.status() == 0, f"status word {plan.status_word():#x}"
        return Ci.cpu().numpy(), D.cpu().numpy()
    finally:
        if own:
            plan.close()


# ---------------------------------------------------------------------------
# fp16, element by element
# ---------------------------------------------------------------------------

def test_f16_workload1_full(oracle):
    w = synth.WORKLOADS[1]
    x = synth.workload_inputs(w)
    C = run_f16(x, w.S, w.R, w.K, w.N, w.chunk_rows)
    check_f16(C, oracle.ag_gemm_f16(x["shards"], x["B"]), w.K, "workload 1")


@pytest.mark.parametrize("S,R,K,N,c", [
    (3, 200, 328, 392, 0),    # ragged M tiles, K tail (328 = 5*64 + 8), N tail
    (2, 130, 72, 136, 0),     # N < 256 after the first tile
    (1, 257, 136, 264, 0),    # single shard = plain GEMM
    (4, 37, 64, 8, 1),        # N = 8, one-row chunks
    (2, 300, 8, 520, 0),      # K = 8
    (5, 256, 1024, 512, 64),  # several full tiles per shard
])
def test_f16_ragged_full(oracle, S, R, K, N, c):
    x = synth.make_inputs(S, R, K, N, "f16", 1000 + S * 7 + K)
    C = run_f16(x, S, R, K, N, c)
    check_f16(C, oracle.ag_gemm_f16(x["shards"], x["B"]), K, f"S={S} R={R} K={K} N={N}")


def test_f16_gather_placement(oracle):
    """Shard s holds s+1 in column 0 and B = e_0 e_0^T: C rows of shard s equal s+1."""
    S, R, K, N = 4, 160, 64, 256
    shards = [np.zeros((R, K), np.float16) for _ in range(S)]
    for s in range(S):
        shards[s][:, 0] = s + 1
    Bm = np.zeros((K, N), np.float16)
    Bm[0, 0] = 1
    for local in range(S):
        C = run_f16({"shards": shards, "B": Bm}, S, R, K, N, 0, local=local)
        want = np.zeros((S * R, N))
        want[:, 0] = np.repeat(np.arange(1, S + 1), R)
        assert np.array_equal(C, want)


# ---------------------------------------------------------------------------
# streaming machinery (invariants)
# ---------------------------------------------------------------------------

def test_f16_modes_bit_identical():
    S, R, K, N = 3, 256, 512, 512
    x = synth.make_inputs(S, R, K, N, "f16", 77)
    with Plan(S, S * R, K, N, "f16") as plan:
        pipelined = run_f16(x, S, R, K, N, plan=plan, mode=B_.MODE_PIPELINED)
        compute = run_f16(x, S, R, K, N, plan=plan, mode=B_.MODE_COMPUTE_ONLY)
        sequential = run_f16(x, S, R, K, N, plan=plan, mode=B_.MODE_SEQUENTIAL)
        plan.set_mode(B_.MODE_COPY_ONLY)
        plan.run([_to_dev(s) for s in x["shards"]], _to_dev(x["B"]))
        torch.cuda.synchronize()
        assert plan.status() == 0
        compute2 = run_f16(x, S, R, K, N, plan=plan, mode=B_.MODE_COMPUTE_ONLY)
    assert np.array_equal(pipelined, compute)
    assert np.array_equal(pipelined, sequential)
    assert np.array_equal(pipelined, compute2)


def test_f16_invariant_to_chunk_rows_and_local_rank():
    S, R, K, N = 4, 256, 256, 384
    x = synth.make_inputs(S, R, K, N, "f16", 78)
    ref = run_f16(x, S, R, K, N, 0)
    for c in (256, 128, 64, 16, 1):
        assert np.array_equal(run_f16(x, S, R, K, N, c), ref), f"chunk_rows={c}"
    for local in range(S):
        assert np.array_equal(run_f16(x, S, R, K, N, 0, local=local), ref), f"local={local}"


def test_f16_poisoned_staging_and_delays():
    S, R, K, N = 3, 384, 512, 512
    x = synth.make_inputs(S, R, K, N, "f16", 79)
    ref = run_f16(x, S, R, K, N, 0)
    poisoned = run_f16(x, S, R, K, N, 0, debug=(B_.DEBUG_POISON_STAGING, 0))
    assert np.array_equal(poisoned, ref)
    delayed = run_f16(x, S, R, K, N, 0, debug=(B_.DEBUG_POISON_STAGING | B_.DEBUG_DELAY_NS, 20000))
    assert np.array_equal(delayed, ref)


def test_f16_repeated_runs_epochs():
    """Counters are monotonic across runs (epoch * pieces): many runs stay right."""
    S, R, K, N = 2, 256, 128, 256
    x = synth.make_inputs(S, R, K, N, "f16", 80)
    with Plan(S, S * R, K, N, "f16") as plan:
        ref = run_f16(x, S, R, K, N, plan=plan)
        shards = [_to_dev(s) for s in x["shards"]]
        Bd = _to_dev(x["B"])
        C = torch.empty((S * R, N), dtype=torch.float32, device=DEV)
        for _ in range(50):
            plan.run(shards, Bd, C)
        torch.cuda.synchronize()
        assert plan.status() == 0
        assert np.array_equal(C.cpu().numpy(), ref)


def test_f16_timeout_then_reset():
    """A chunk whose copy is skipped never becomes ready: the consumer's bounded
    wait ends with TIMEOUT (no hang, context stays usable); after a reset the
    plan runs correctly again."""
    S, R, K, N = 2, 256, 128, 256
    x = synth.make_inputs(S, R, K, N, "f16", 81)
    with Plan(S, S * R, K, N, "f16") as plan:
        ref = run_f16(x, S, R, K, N, plan=plan)
        plan.set_timeout_ns(20_000_000)
        plan.set_debug(B_.DEBUG_SKIP_ITEM, 3)
        shards = [_to_dev(s) for s in x["shards"]]
        Bd = _to_dev(x["B"])
        plan.run(shards, Bd)
        torch.cuda.synchronize()
        assert plan.status() == B_.ERR_TIMEOUT
        assert plan.status_word() & 0xFF == 1
        plan.set_debug(0, 0)
        plan.reset()
        again = run_f16(x, S, R, K, N, plan=plan)
        assert np.array_equal(again, ref)


def test_f16_abi_errors_on_gpu():
    S, R, K, N = 2, 128, 64, 64
    with Plan(S, S * R, K, N, "f16") as plan:
        a = torch.zeros((R, K), dtype=torch.float16, device=DEV)
        Bd = torch.zeros((K, N), dtype=torch.float16, device=DEV)
        C = torch.zeros((S * R, N), dtype=torch.float32, device=DEV)
        h = plan.handle
        with pytest.raises(B_.AgGemmError) as e:
            B_.ag_gemm_run(h, [a.data_ptr(), 0], Bd.data_ptr(), C.data_ptr(), 0)
        assert e.value.code == B_.ERR_INVALID
        with pytest.raises(B_.AgGemmError) as e:
            B_.ag_gemm_run(h, [a.data_ptr(), a.data_ptr() + 2], Bd.data_ptr(), C.data_ptr(), 0)
        assert e.value.code == B_.ERR_INVALID
        with pytest.raises(B_.AgGemmError) as e:
            B_.ag_gemm_dequant_run(h, [a.data_ptr()] * 2, Bd.data_ptr(), C.data_ptr(),
                                   C.data_ptr(), C.data_ptr(), C.data_ptr(), 0)
        assert e.value.code == B_.ERR_INVALID
        with pytest.raises(B_.AgGemmError):
            plan.set_local_rank(2)
        with pytest.raises(B_.AgGemmError):
            plan.set_mode(9)


# ---------------------------------------------------------------------------
# fp16 full-size workloads (the bench's launch configuration)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("wid", [2, 3])
def test_f16_full_size_workload(oracle, wid):
    w = synth.WORKLOADS[wid]
    x = synth.workload_inputs(w)
    C = run_f16(x, w.S, w.R, w.K, w.N, w.chunk_rows)
    assert np.all(np.isfinite(C))
    rng = np.random.default_rng(wid)
    rows, cols = tile_samples(rng, w.M, w.N, w.R)
    ref = oracle.ag_gemm_f16_at(x["shards"], x["B"], rows, cols)
    check_f16(C[rows, cols], ref, w.K, f"workload {wid} samples")
    A = np.concatenate(x["shards"]).astype(np.float64)
    Bf = x["B"].astype(np.float64)
    row_ref = A @ Bf.sum(axis=1)
    col_ref = A.sum(axis=0) @ Bf
    Cd = C.astype(np.float64)
    assert np.abs(Cd.sum(axis=1) - row_ref).max() <= 1e-3 * np.sqrt(w.K * w.N)
    assert np.abs(Cd.sum(axis=0) - col_ref).max() <= 1e-3 * np.sqrt(w.K * w.M)


# ---------------------------------------------------------------------------
# bf16 operands (same kernel, kind::f16 with the bf16 operand format)
# ---------------------------------------------------------------------------

def _bf16_to_dev(bits):
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).to(DEV)


def run_bf16(x, S, R, K, N, chunk_rows=0, mode=None, local=None, plan=None):
    own = plan is None
    if own:
        plan = Plan(S, S * R, K, N, "bf16", chunk_rows)
    try:
        if mode is not None:
            plan.set_mode(mode)
        if local is not None:
            plan.set_local_rank(local)
        shards = [_bf16_to_dev(s) for s in x["shards"]]
        C = torch.full((S * R, N), float("nan"), dtype=torch.float32, device=DEV)
        plan.run(shards, _bf16_to_dev(x["B"]), C)
        torch.cuda.synchronize()
        assert plan.status() == 0, f"status word {plan.status_word():#x}"
        return C.cpu().numpy()
    finally:
        if own:
            plan.close()


@pytest.mark.parametrize("S,R,K,N,c", [
    (3, 200, 328, 392, 0),    # ragged M tiles, K tail, N tail
    (2, 130, 72, 136, 0),
    (1, 257, 136, 264, 0),
    (4, 37, 64, 8, 1),
    (5, 256, 1024, 512, 64),
])
def test_bf16_ragged_full(oracle, S, R, K, N, c):
    x = synth.make_inputs(S, R, K, N, "bf16", 1500 + S * 7 + K)
    C = run_bf16(x, S, R, K, N, c)
    check_f16(C, oracle.ag_gemm_bf16(x["shards"], x["B"]), K, f"bf16 S={S} R={R} K={K} N={N}")


def test_bf16_full_size_workload(oracle):
    """The 4096^3 case with bfloat16 operands: sampled points against the oracle,
    every element against an fp64 BLAS product of the oracle-decoded operands."""
    w = synth.WORKLOADS[6]
    x = synth.workload_inputs(w)
    C = run_bf16(x, w.S, w.R, w.K, w.N, w.chunk_rows)
    rng = np.random.default_rng(6)
    rows, cols = tile_samples(rng, w.M, w.N, w.R)
    check_f16(C[rows, cols], oracle.ag_gemm_bf16_at(x["shards"], x["B"], rows, cols), w.K,
              "bf16 workload samples")
    A = oracle.bf16_bits_to_f64(np.concatenate(x["shards"]))
    check_f16(C, A @ oracle.bf16_bits_to_f64(x["B"]), w.K, "bf16 workload full")


def test_bf16_modes_chunks_and_local_rank_bit_identical():
    S, R, K, N = 3, 256, 512, 384
    x = synth.make_inputs(S, R, K, N, "bf16", 79)
    ref = run_bf16(x, S, R, K, N)
    with Plan(S, S * R, K, N, "bf16") as plan:
        for mode in (B_.MODE_SEQUENTIAL, B_.MODE_COMPUTE_ONLY, B_.MODE_PIPELINED):
            assert np.array_equal(run_bf16(x, S, R, K, N, plan=plan, mode=mode), ref)
    for c in (128, 16, 1):
        assert np.array_equal(run_bf16(x, S, R, K, N, c), ref), f"chunk_rows={c}"
    for local in range(S):
        assert np.array_equal(run_bf16(x, S, R, K, N, local=local), ref), f"local={local}"


def test_bf16_plan_checks_operand_dtype():
    with Plan(2, 256, 64, 128, "bf16") as plan:
        f16 = [torch.zeros((128, 64), dtype=torch.float16, device=DEV) for _ in range(2)]
        with pytest.raises(TypeError):
            plan.run(f16, torch.zeros((64, 128), dtype=torch.float16, device=DEV))


# ---------------------------------------------------------------------------
# int8 dequant
# ---------------------------------------------------------------------------

def _check_i8(Ci, D, Cref, Dref, what=""):
    assert np.array_equal(Ci, Cref), f"{what}: C_i32 differs in {np.count_nonzero(Ci != Cref)} places"
    ulp = f16_ulp_distance(D, Dref)
    assert ulp.max() <= 1, f"{what}: D off by {ulp.max()} ulp"


@pytest.mark.parametrize("S,R,K,N,c", [
    (2, 200, 1056, 208, 0),    # two K segments (1024 + 32), ragged tiles
    (3, 64, 2064, 96, 0),
    (1, 130, 16, 16, 0),
    (4, 33, 3072, 272, 3),
])
def test_i8_ragged_full(oracle, S, R, K, N, c):
    x = synth.make_inputs(S, R, K, N, "i8", 2000 + S * 11 + K)
    Ci, D = run_i8(x, S, R, K, N, c)
    Cref, Dref = oracle.ag_gemm_dequant(x["shards"], x["B"], x["bias"], x["scale"])
    _check_i8(Ci, D, Cref, Dref, f"S={S} R={R} K={K} N={N}")


def test_i8_worst_case_magnitudes_exact(oracle):
    """All entries +-127 and K = 27392: every fp32 segment partial reaches
    1024 * 127^2 and the int32 sum reaches 27392 * 127^2 - the exactness limit
    of the fp16-emulated int8 MMA is exercised."""
    S, R, K, N = 2, 64, 27392, 256
    rng = np.random.default_rng(5)
    shards = [np.full((R, K), 127, np.int8) for _ in range(S)]
    shards[1][::2] = -127
    Bm = np.full((K, N), 127, np.int8)
    Bm[:, 1::3] = -127
    signs = rng.choice(np.array([-127, 127], np.int8), size=(K, 8))
    Bm[:, -8:] = signs
    x = {"shards": shards, "B": Bm, "bias": rng.integers(-1000, 1001, N, dtype=np.int32),
         "scale": rng.uniform(1e-5, 1e-4, N).astype(np.float32)}
    Ci, D = run_i8(x, S, R, K, N)
    Cref, Dref = oracle.ag_gemm_dequant(x["shards"], x["B"], x["bias"], x["scale"])
    _check_i8(Ci, D, Cref, Dref, "worst case")


def test_i8_modes_and_local_rank_bit_identical():
    S, R, K, N = 3, 128, 1024, 256
    x = synth.make_inputs(S, R, K, N, "i8", 90)
    ref = run_i8(x, S, R, K, N)
    with Plan(S, S * R, K, N, "i8") as plan:
        for mode in (B_.MODE_SEQUENTIAL, B_.MODE_PIPELINED, B_.MODE_COMPUTE_ONLY):
            got = run_i8(x, S, R, K, N, plan=plan, mode=mode)
            assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
    for local in range(S):
        got = run_i8(x, S, R, K, N, local=local)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


@pytest.mark.parametrize("wid", [4, 5])
def test_i8_full_size_workload(oracle, wid):
    w = synth.WORKLOADS[wid]
    x = synth.workload_inputs(w)
    Ci, D = run_i8(x, w.S, w.R, w.K, w.N, w.chunk_rows)
    rng = np.random.default_rng(wid)
    rows, cols = tile_samples(rng, w.M, w.N, w.R, per_tile=2)
    Cs, Ds = oracle.ag_gemm_dequant_at(x["shards"], x["B"], x["bias"], x["scale"], rows, cols)
    _check_i8(Ci[rows, cols], D[rows, cols], Cs, Ds, f"workload {wid} samples")
    # exact checksums over every element
    bsum = x["B"].astype(np.int64).sum(axis=1).astype(np.float64)
    row_ref = np.concatenate([s.astype(np.float64) @ bsum for s in x["shards"]])
    row_ref = row_ref.astype(np.int64) + int(x["bias"].astype(np.int64).sum())
    assert np.array_equal(Ci.astype(np.int64).sum(axis=1), row_ref)
    asum = sum(s.astype(np.int64).sum(axis=0) for s in x["shards"]).astype(np.float64)
    col_ref = (asum @ x["B"].astype(np.float64)).astype(np.int64) + w.M * x["bias"].astype(np.int64)
    assert np.array_equal(Ci.astype(np.int64).sum(axis=0), col_ref)
    # every D element is the fp32 dequant of its (checked) C_i32
    with np.errstate(over="ignore"):
        want = (Ci.astype(np.float32) * x["scale"][None, :]).astype(np.float16)
    assert f16_ulp_distance(D, want).max() <= 1


# ---------------------------------------------------------------------------
# int8 with few gathered rows (the B-streaming skinny kernel: M <= 128)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("S,R,K,N,c", [
    (2, 32, 1056, 208, 0),     # two K segments + a K tail, a ragged 256-column n-tile
    (2, 24, 768, 400, 0),      # two n-tiles, the second ragged inside its second B box
    (4, 8, 64, 16, 0),         # one k-block, one tiny n-tile
    (2, 64, 2048, 384, 16),    # 128 rows (every TMEM lane)
    (1, 40, 512, 128, 0),      # a single shard
    (3, 16, 4096, 256, 2),
    (3, 13, 1040, 144, 0),     # rows of a shard not a multiple of 8, 3 lane quadrants
    (2, 20, 112, 48, 0),       # K below one 128-row B box, two k-blocks; the second box of
                               # the n-tile lies past N (zero fill)
    (1, 128, 320, 128, 0),     # 128 rows of one shard, a 1-k-block last unit
])
def test_i8_skinny_full(oracle, S, R, K, N, c):
    x = synth.make_inputs(S, R, K, N, "i8", 3000 + S * 13 + K)
    Ci, D = run_i8(x, S, R, K, N, c)
    Cref, Dref = oracle.ag_gemm_dequant(x["shards"], x["B"], x["bias"], x["scale"])
    _check_i8(Ci, D, Cref, Dref, f"skinny S={S} R={R} K={K} N={N}")


def test_plan_path_and_grid():
    """The plan picks its kernels by dtype and M; the skinny path runs one CTA per SM."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    with Plan(2, 64, 1024, 256, "i8") as p:
        assert p.path == B_.PATH_SKINNY_I8 and p.grid == sms
    with Plan(2, 512, 256, 256, "i8") as p:
        assert p.path == B_.PATH_FUSED_I8
    with Plan(2, 256, 256, 128, "f16") as p:
        assert p.path == B_.PATH_FUSED_F16 and p.grid % 2 == 0 and 0 < p.grid <= sms


def test_skinny_plan_geometry():
    """A skinny plan reports its own kernel's tiling (rows x 256-column n-tiles) and
    what it allocates (split-K slots, no fp16 copy of B)."""
    with Plan(2, 64, 16384, 7168, "i8") as p:
        g = p.geometry
        assert (g["block_m"], g["block_n"], g["m_tiles"]) == (64, 256, 1)
        assert g["n_tiles"] == g["tiles"] == 28
        assert g["workspace_bytes"] < 64 * 1024 * 1024    # fp16 B alone would be 235 MB
    with Plan(2, 128, 1024, 400, "i8") as p:
        g = p.geometry
        assert (g["block_m"], g["block_n"], g["n_tiles"]) == (128, 256, 2)


def test_i8_skinny_worst_case_magnitudes_exact(oracle):
    S, R, K, N = 2, 32, 16384, 256
    rng = np.random.default_rng(6)
    shards = [np.full((R, K), 127, np.int8), np.full((R, K), -127, np.int8)]
    Bm = np.full((K, N), 127, np.int8)
    Bm[:, ::5] = -127
    x = {"shards": shards, "B": Bm, "bias": rng.integers(-1000, 1001, N, dtype=np.int32),
         "scale": rng.uniform(1e-5, 1e-4, N).astype(np.float32)}
    Ci, D = run_i8(x, S, R, K, N)
    Cref, Dref = oracle.ag_gemm_dequant(x["shards"], x["B"], x["bias"], x["scale"])
    _check_i8(Ci, D, Cref, Dref, "skinny worst case")


def test_i8_skinny_modes_local_rank_and_repeats():
    S, R, K, N = 2, 32, 2048, 640
    x = synth.make_inputs(S, R, K, N, "i8", 91)
    ref = run_i8(x, S, R, K, N)
    with Plan(S, S * R, K, N, "i8") as plan:
        for mode in (B_.MODE_SEQUENTIAL, B_.MODE_PIPELINED, B_.MODE_COMPUTE_ONLY,
                     B_.MODE_PIPELINED, B_.MODE_PIPELINED):
            got = run_i8(x, S, R, K, N, plan=plan, mode=mode)
            assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
    for local in range(S):
        got = run_i8(x, S, R, K, N, local=local)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


@pytest.mark.parametrize("S,R,K,N", [
    (2, 16, 16384, 128),       # one n-tile of 128 units: 128 CTAs share it, the others hold none
    (1, 8, 4096, 2048),        # 8 n-tiles of 32 units over 152 CTAs
])
def test_i8_skinny_shared_tiles_and_repeats(oracle, S, R, K, N):
    """Split-K sums of one n-tile spread over many CTAs (some CTAs own no unit),
    reduced by the CTA that stores the tile's last piece.  The per-tile counters
    are monotonic across runs of one plan; a copy-only run leaves them alone."""
    x = synth.make_inputs(S, R, K, N, "i8", 4000 + K + N)
    Cref, Dref = oracle.ag_gemm_dequant(x["shards"], x["B"], x["bias"], x["scale"])
    with Plan(S, S * R, K, N, "i8") as plan:
        for i, mode in enumerate((B_.MODE_PIPELINED, B_.MODE_COPY_ONLY, B_.MODE_PIPELINED,
                                  B_.MODE_COMPUTE_ONLY, B_.MODE_SEQUENTIAL, B_.MODE_PIPELINED)):
            got = run_i8(x, S, R, K, N, plan=plan, mode=mode)
            if mode != B_.MODE_COPY_ONLY:
                _check_i8(got[0], got[1], Cref, Dref, f"run {i} mode {mode}")
        plan.reset()
        got = run_i8(x, S, R, K, N, plan=plan, mode=B_.MODE_PIPELINED)
        _check_i8(got[0], got[1], Cref, Dref, "after reset")


def test_i8_skinny_timeout_then_reset():
    S, R, K, N = 2, 32, 1024, 256
    x = synth.make_inputs(S, R, K, N, "i8", 92)
    ref = run_i8(x, S, R, K, N)
    with Plan(S, S * R, K, N, "i8") as plan:
        plan.set_timeout_ns(20_000_000)
        plan.set_debug(B_.DEBUG_SKIP_ITEM, 5)
        shards = [_to_dev(s) for s in x["shards"]]
        plan.dequant_run(shards, _to_dev(x["B"]), _to_dev(x["bias"]), _to_dev(x["scale"]))
        torch.cuda.synchronize()
        assert plan.status() == B_.ERR_TIMEOUT
        plan.set_debug(0, 0)
        plan.reset()
        got = run_i8(x, S, R, K, N, plan=plan)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


# ---------------------------------------------------------------------------
# N-sharded layout ("Collective matrix multiplication", Ring All-Gather): rank d
# computes C[:, block d] = AllGather(A) x B[:, block d], its row slices taken
# in ring order from d (the plan's local rank); B and C are column blocks of
# the full matrices, passed with their row pitches (ag_gemm_run_ld).
# ---------------------------------------------------------------------------

def _nshard_inputs(dt, D, R, K, ns, seed):
    x = synth.make_inputs(D, R, K, D * ns, dt, seed)
    conv = _bf16_to_dev if dt == "bf16" else _to_dev
    return x, [conv(s) for s in x["shards"]], conv(x["B"])


@pytest.mark.parametrize("dt,D,R,K,ns", [
    ("f16", 2, 256, 512, 256),
    ("f16", 4, 96, 320, 72),     # n_shard not a multiple of 64: the 2-D B map
    ("bf16", 3, 130, 256, 136),  # ragged rows per shard
    ("f16", 2, 256, 2048, 256),  # 2 tiles per rank, split in two along K: zeroed and reduced
                                 # C blocks inside a wider C (row pitch 2 x 256)
])
def test_nshard_ranks_assemble_the_product(oracle, dt, D, R, K, ns):
    x, shards, Bfull = _nshard_inputs(dt, D, R, K, ns, 5000 + D * 7 + K)
    N = D * ns
    C = torch.full((D * R, N), float("nan"), dtype=torch.float32, device=DEV)
    with Plan(D, D * R, K, ns, dt) as plan:
        for d in range(D):
            plan.set_local_rank(d)
            plan.run(shards, Bfull[:, d * ns:(d + 1) * ns], C[:, d * ns:(d + 1) * ns])
            torch.cuda.synchronize()
            assert plan.status() == 0, f"rank {d}: status word {plan.status_word():#x}"
            if d + 1 < D:  # columns of later ranks untouched
                assert torch.isnan(C[:, (d + 1) * ns:]).all()
    got = C.cpu().numpy()
    ref_fn = oracle.ag_gemm_f16 if dt == "f16" else oracle.ag_gemm_bf16
    check_f16(got, ref_fn(x["shards"], x["B"]), K, f"{dt} N-sharded D={D}")
    # each rank's block against the ring-order oracle of that rank
    for d in range(D):
        ring = oracle.collective_matmul_ring(x["shards"], x["B"][:, d * ns:(d + 1) * ns], d, dt)
        check_f16(got[:, d * ns:(d + 1) * ns], ring, K, f"{dt} rank {d}")
    # the same fp32 sums as one run over all columns with contiguous operands
    with Plan(D, D * R, K, N, dt) as plan:
        whole = plan.run(shards, Bfull)
        torch.cuda.synchronize()
    assert torch.equal(C, whole)


def test_nshard_modes_bit_identical():
    D, R, K, ns = 2, 128, 256, 128
    _, shards, Bfull = _nshard_inputs("f16", D, R, K, ns, 77)
    outs = []
    with Plan(D, D * R, K, ns, "f16") as plan:
        plan.set_local_rank(1)
        for mode in (B_.MODE_PIPELINED, B_.MODE_SEQUENTIAL, B_.MODE_PIPELINED):
            plan.set_mode(mode)
            C = torch.full((D * R, D * ns), float("nan"), dtype=torch.float32, device=DEV)
            plan.run(shards, Bfull[:, ns:], C[:, ns:])
            torch.cuda.synchronize()
            assert plan.status() == 0
            outs.append(C)
    assert all(torch.equal(outs[0][:, ns:], o[:, ns:]) for o in outs[1:])
    assert not torch.isnan(outs[0][:, ns:]).any()
    assert all(torch.isnan(o[:, :ns]).all() for o in outs)


def test_nshard_pitch_checks():
    D, R, K, ns = 2, 64, 128, 64
    _, shards, Bfull = _nshard_inputs("f16", D, R, K, ns, 78)
    C = torch.empty((D * R, D * ns), dtype=torch.float32, device=DEV)
    ptrs = [s.data_ptr() for s in shards]
    with Plan(D, D * R, K, ns, "f16") as plan:
        for ldb, ldc in ((ns - 8, D * ns), (D * ns, ns - 4), (D * ns + 4, D * ns),
                         (D * ns, D * ns + 2)):
            with pytest.raises(B_.AgGemmError) as e:
                B_.ag_gemm_run_ld(plan.handle, ptrs, Bfull.data_ptr(), ldb, C.data_ptr(), ldc)
            assert e.value.code == B_.ERR_INVALID
    with Plan(D, D * R, K, ns, "i8") as plan:
        with pytest.raises(B_.AgGemmError) as e:
            B_.ag_gemm_run_ld(plan.handle, ptrs, Bfull.data_ptr(), D * ns, C.data_ptr(), D * ns)
        assert e.value.code == B_.ERR_INVALID


# ---------------------------------------------------------------------------
# the last round's tiles split along K over otherwise idle CTA pairs: int8
# parts store partial sums and the last part adds them in part order; fp16 /
# bf16 parts both add into C blocks zeroed at the start of the run
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dt,S,R,K,N", [
    ("f16", 2, 384, 8192, 512),    # 8 tiles, 2 parts of 64 k-blocks each
    ("bf16", 3, 300, 8192, 264),   # 12 tiles (ragged rows and columns), 2 parts each
    ("f16", 2, 384, 2048, 512),    # 8 tiles, 2 parts of 16 k-blocks
    ("f16", 3, 200, 2112, 264),    # 6 tiles of 200 rows, 2 parts of 16 and 17 k-blocks
    ("bf16", 2, 640, 4096, 520),   # 18 tiles (ragged last m-tile and n-tile), 2 parts of 32
    ("i8", 2, 384, 8256, 512),     # 4 tiles, 2 parts of 64 and 65 k-blocks (int32 partials)
])
def test_split_tail_parity_modes_and_repeats(oracle, dt, S, R, K, N):
    x = synth.make_inputs(S, R, K, N, dt, 7000 + S * 17 + K)
    run = {"f16": run_f16, "bf16": run_bf16, "i8": run_i8}[dt]
    with Plan(S, S * R, K, N, dt) as plan:
        g = plan.geometry
        assert g["split_parts"] > 1 and g["split_tiles"] > 0, g
        first = run(x, S, R, K, N, plan=plan)
        if dt == "i8":
            Cref, Dref = oracle.ag_gemm_dequant(x["shards"], x["B"], x["bias"], x["scale"])
            _check_i8(first[0], first[1], Cref, Dref, "split tail")
        else:
            ref = (oracle.ag_gemm_f16 if dt == "f16" else oracle.ag_gemm_bf16)(x["shards"], x["B"])
            check_f16(first, ref, K, f"split tail {dt}")
        # the part flags and zero-task counters are monotonic across runs and
        # modes; a reset restarts them
        for mode in (B_.MODE_PIPELINED, B_.MODE_COMPUTE_ONLY, B_.MODE_SEQUENTIAL,
                     B_.MODE_PIPELINED):
            again = run(x, S, R, K, N, plan=plan, mode=mode)
            same = (np.array_equal(again[0], first[0]) and np.array_equal(again[1], first[1])
                    if dt == "i8" else np.array_equal(again, first))
            assert same, f"mode {mode}"
        plan.reset()
        again = run(x, S, R, K, N, plan=plan, mode=B_.MODE_PIPELINED)
        assert (np.array_equal(again[0], first[0]) if dt == "i8" else np.array_equal(again, first))


def test_split_tail_plan_geometry():
    """The split is chosen for the device's full grid: when the last round's
    tiles fill at most half of the CTA pairs and a tile has at least 32
    k-blocks (fp16 / bf16) or 128 (int8), each is split in two along K."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    pairs = sms // 2
    with Plan(2, 4096, 8192, 4096, "f16") as p:      # 256 pair tiles, 128 k-blocks
        g = p.geometry
        assert g["split_tiles"] == 256 % pairs and g["split_parts"] == 2
    with Plan(2, 4096, 4096, 4096, "f16") as p:      # 64 k-blocks: fp16 parts add into C
        g = p.geometry
        assert g["split_tiles"] == 256 % pairs and g["split_parts"] == 2
    with Plan(2, 4096, 4096, 4096, "i8") as p:       # int8 at 64 k-blocks: the hand-off would not pay
        assert p.geometry["split_parts"] == 1
    with Plan(2, 4096, 1024, 4096, "f16") as p:      # 16 k-blocks: too short
        assert p.geometry["split_parts"] == 1
    with Plan(8, 8192, 4096, 4096, "f16") as p:      # 512 tiles: the last round is too full
        assert p.geometry["split_parts"] == 1
    with Plan(2, 512, 256, 512, "f16") as p:         # 4 k-blocks: too short to split
        assert p.geometry["split_parts"] == 1 and p.geometry["split_tiles"] == 0
    with Plan(4, 4096, 2048, 2048, "f16", staging_slots=8) as p:   # a staging window
        assert p.geometry["split_parts"] == 1
