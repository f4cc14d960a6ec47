"""GPU parity on a seeded sweep of random shapes, against the CPU oracle.

The fixed cases of test_parity_gpu.py pick the edges by hand; these draw shard
counts, rows per shard, K, N and the chunk size at random (seeded, so every run
checks the same shapes) within the library's validation rules.  Every case
covers the skinny int8 kernel (M <= 128 rows: M = 64 or 128 MMA rows, ragged
256-column n-tiles, K tails shorter than a 2-k-block unit), the fused int8
kernel (register-resident int32 sums, BN = 128 or 256), or the fused
fp16 / bf16 kernel (ragged M tiles, K and N tails).  Tolerances as in
test_parity_gpu.py: int8 C_i32 bit-exact and D within 1 fp16 ulp; fp16 / bf16
relative Frobenius error <= 1e-4 and max abs error <= 1e-3 sqrt(K).
"""
import numpy as np
import pytest

from gpu_util import check_f16

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from all_gather_gemm_chunked_gb300 import synth  # noqa: E402
from test_parity_gpu import _check_i8, run_bf16, run_f16, run_i8  # noqa: E402


def _divisor_chunk(rng, R):
    """0 (the library's rule) half of the time, else a random divisor of R."""
    if rng.random() < 0.5:
        return 0
    divs = [c for c in range(1, R + 1) if R % c == 0]
    return int(rng.choice(divs))


def _cases():
    rng = np.random.default_rng(0x5EED)
    skinny, fused_i8, f16, bf16 = [], [], [], []
    while len(skinny) < 12:
        S = int(rng.integers(1, 5))
        R = int(rng.integers(1, 128 // S + 1))
        K = 16 * int(rng.integers(1, 300))
        N = 16 * int(rng.integers(1, 70))
        skinny.append((S, R, K, N, _divisor_chunk(rng, R)))
    while len(fused_i8) < 6:
        S = int(rng.integers(1, 5))
        R = int(rng.integers(129 // S + 1, 300))
        K = 16 * int(rng.integers(1, 130))
        N = 16 * int(rng.integers(1, 30))
        fused_i8.append((S, R, K, N, _divisor_chunk(rng, R)))
    while len(f16) < 6:
        S = int(rng.integers(1, 7))
        R = int(rng.integers(1, 300))
        K = 8 * int(rng.integers(1, 200))
        N = 8 * int(rng.integers(1, 90))
        f16.append((S, R, K, N, _divisor_chunk(rng, R)))
    while len(bf16) < 4:
        S = int(rng.integers(1, 5))
        R = int(rng.integers(1, 300))
        K = 8 * int(rng.integers(1, 200))
        N = 8 * int(rng.integers(1, 90))
        bf16.append((S, R, K, N, _divisor_chunk(rng, R)))
    return skinny, fused_i8, f16, bf16


SKINNY, FUSED_I8, F16, BF16 = _cases()


def _id(c):
    return "S{}R{}K{}N{}c{}".format(*c)


@pytest.mark.parametrize("S,R,K,N,c", SKINNY, ids=[_id(c) for c in SKINNY])
def test_sweep_i8_skinny(oracle, S, R, K, N, c):
    assert S * R <= 128
    x = synth.make_inputs(S, R, K, N, "i8", 7000 + S * 131 + R * 17 + K + N)
    Ci, D = run_i8(x, S, R, K, N, c)
    Cref, Dref = oracle.ag_gemm_dequant(x["shards"], x["B"], x["bias"], x["scale"])
    _check_i8(Ci, D, Cref, Dref, f"skinny S={S} R={R} K={K} N={N} c={c}")


@pytest.mark.parametrize("S,R,K,N,c", FUSED_I8, ids=[_id(c) for c in FUSED_I8])
def test_sweep_i8_fused(oracle, S, R, K, N, c):
    assert S * R > 128
    x = synth.make_inputs(S, R, K, N, "i8", 8000 + S * 131 + R * 17 + K + N)
    Ci, D = run_i8(x, S, R, K, N, c)
    Cref, Dref = oracle.ag_gemm_dequant(x["shards"], x["B"], x["bias"], x["scale"])
    _check_i8(Ci, D, Cref, Dref, f"fused int8 S={S} R={R} K={K} N={N} c={c}")


@pytest.mark.parametrize("S,R,K,N,c", F16, ids=[_id(c) for c in F16])
def test_sweep_f16(oracle, S, R, K, N, c):
    x = synth.make_inputs(S, R, K, N, "f16", 9000 + S * 131 + R * 17 + K + N)
    C = run_f16(x, S, R, K, N, c)
    check_f16(C, oracle.ag_gemm_f16(x["shards"], x["B"]), K, f"f16 S={S} R={R} K={K} N={N} c={c}")


@pytest.mark.parametrize("S,R,K,N,c", BF16, ids=[_id(c) for c in BF16])
def test_sweep_bf16(oracle, S, R, K, N, c):
    x = synth.make_inputs(S, R, K, N, "bf16", 9500 + S * 131 + R * 17 + K + N)
    C = run_bf16(x, S, R, K, N, c)
    check_f16(C, oracle.ag_gemm_bf16(x["shards"], x["B"]), K, f"bf16 S={S} R={R} K={K} N={N} c={c}")


# Many shards, down to one row per shard (chunk = row), on every path.
MANY = [
    (8, 1, 1040, 272, "i8"),      # 8 rows: skinny, M = 64 MMA rows, one row per shard
    (7, 18, 2064, 528, "i8"),     # 126 rows: skinny, M = 128 MMA rows
    (6, 30, 1024, 160, "i8"),     # 180 rows: fused int8
    (8, 1, 200, 72, "f16"),       # one row per shard
    (8, 3, 520, 136, "f16"),
    (5, 61, 64, 264, "bf16"),
]


@pytest.mark.parametrize("S,R,K,N,dtype", MANY,
                         ids=["S{}R{}K{}N{}{}".format(*c) for c in MANY])
def test_sweep_many_shards(oracle, S, R, K, N, dtype):
    x = synth.make_inputs(S, R, K, N, dtype, 9900 + S * 131 + R * 17 + K + N)
    if dtype == "i8":
        Ci, D = run_i8(x, S, R, K, N)
        Cref, Dref = oracle.ag_gemm_dequant(x["shards"], x["B"], x["bias"], x["scale"])
        _check_i8(Ci, D, Cref, Dref, f"int8 S={S} R={R} K={K} N={N}")
    elif dtype == "f16":
        check_f16(run_f16(x, S, R, K, N), oracle.ag_gemm_f16(x["shards"], x["B"]), K,
                  f"f16 S={S} R={R} K={K} N={N}")
    else:
        check_f16(run_bf16(x, S, R, K, N), oracle.ag_gemm_bf16(x["shards"], x["B"]), K,
                  f"bf16 S={S} R={R} K={K} N={N}")
