"""Pins for the CPU oracle: checks against facts the oracle does not compute.

Every check here compares the oracle with something independent of it:
numpy's IEEE conversions (library routines), exact big-integer arithmetic,
closed forms, torch float64 matmul on the CPU, and the all-ones debug mode of
"AllGather矩阵乘法反量化算子设计文档" 8.6.  The ``PINS`` table at the bottom
also runs every GEMM pin against deliberately wrong implementations (a
transposed operand, a dropped k term, swapped shards, a bias indexed by row, a
truncating fp16 cast) and requires each of them to be caught.
"""
from fractions import Fraction

import numpy as np
import pytest

# ---------------------------------------------------------------------------
# IEEE binary16 / binary32
# ---------------------------------------------------------------------------


def test_f16_decode_all_bit_patterns(oracle):
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.f16_bits_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # sign of zero survives
    assert np.signbit(got[0x8000]) and not np.signbit(got[0])


def _random_doubles(rng, n):
    parts = [
        rng.standard_normal(n) * 10.0 ** rng.integers(-9, 5, n),
        rng.uniform(-65600, 65600, n // 4),
        rng.uniform(-2.0 ** -14, 2.0 ** -14, n // 4),       # subnormal range
        rng.uniform(-2.0 ** -23, 2.0 ** -23, n // 8),       # underflow to 0
    ]
    return np.concatenate(parts)


def test_f16_encode_random_vs_numpy(oracle):
    x = _random_doubles(np.random.default_rng(1), 1_000_000)
    got = oracle.f64_to_f16_bits(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_f16_encode_exact_ties_vs_numpy(oracle):
    # every midpoint between consecutive finite binary16 values (ties)
    h = np.arange(0, 0x7BFF, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    mid = (lo + hi) / 2
    for x in (mid, -mid, np.nextafter(mid, 0), np.nextafter(mid, np.inf)):
        assert np.array_equal(oracle.f64_to_f16_bits(x),
                              x.astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("x,bits", [
    (0.0, 0x0000), (-0.0, 0x8000), (1.0, 0x3C00), (-2.0, 0xC000),
    (1.0 + 2.0 ** -11, 0x3C00),            # tie -> even (down)
    (1.0 + 3 * 2.0 ** -11, 0x3C02),        # tie -> even (up)
    (65504.0, 0x7BFF), (65519.999, 0x7BFF),
    (65520.0, 0x7C00), (-65520.0, 0xFC00),  # tie at the top -> inf
    (1e300, 0x7C00), (float("inf"), 0x7C00),
    (2.0 ** -24, 0x0001), (2.0 ** -25, 0x0000),  # tie -> even (zero)
    (3 * 2.0 ** -25, 0x0002),              # 1.5 ulp -> 2 ulp (even)
    (2.0 ** -14, 0x0400), (2.0 ** -14 - 2.0 ** -25, 0x0400),  # round up to min normal
])
def test_f16_encode_boundaries(oracle, x, bits):
    assert int(oracle.f64_to_f16_bits(np.array([x]))[0]) == bits


def test_f16_encode_nan(oracle):
    b = int(oracle.f64_to_f16_bits(np.array([np.nan]))[0])
    assert (b & 0x7C00) == 0x7C00 and (b & 0x3FF) != 0


def test_f32_encode_random_vs_numpy(oracle):
    rng = np.random.default_rng(2)
    x = np.concatenate([
        rng.standard_normal(500_000) * 10.0 ** rng.integers(-40, 39, 500_000),
        rng.integers(-2 ** 31, 2 ** 31, 200_000).astype(np.float64),
        rng.uniform(-1e-38, 1e-38, 100_000),
    ])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float32).view(np.uint32)
    assert np.array_equal(oracle.f64_to_f32(x).view(np.uint32), ref)


# ---------------------------------------------------------------------------
# fp16 AllGather + GEMM
# ---------------------------------------------------------------------------

def _shards(rng, S, R, K, scale=1.0):
    return [(rng.standard_normal((R, K)) * scale).astype(np.float16) for _ in range(S)]


def pin_one_hot_permutation(impl):
    """B[k][n] = [k == pi(n)]  =>  C[:, n] = A[:, pi(n)] exactly."""
    rng = np.random.default_rng(10)
    S, R, K, N = 3, 5, 11, 7
    shards = _shards(rng, S, R, K)
    pi = rng.permutation(K)[:N]
    B = np.zeros((K, N), np.float16)
    B[pi, np.arange(N)] = 1
    A = np.concatenate(shards).astype(np.float64)
    return np.array_equal(impl(shards, B), A[:, pi])


def pin_single_entry(impl):
    """B = v * e_k0 e_n0^T  =>  exactly one non-zero column, = v * A[:, k0]."""
    rng = np.random.default_rng(11)
    S, R, K, N = 2, 4, 9, 6
    shards = _shards(rng, S, R, K)
    B = np.zeros((K, N), np.float16)
    B[7, 2] = -0.75
    A = np.concatenate(shards).astype(np.float64)
    want = np.zeros((S * R, N))
    want[:, 2] = -0.75 * A[:, 7]
    return np.array_equal(impl(shards, B), want)


def pin_rank_one(impl):
    """A[m][k] = a_m, B[k][n] = b_n (small integers)  =>  C = K a_m b_n."""
    S, R, K, N = 2, 3, 37, 5
    a = np.arange(1, S * R + 1) - 3.0
    b = np.array([2.0, -1.0, 3.0, 0.5, -4.0])
    shards = [np.repeat(a[s * R:(s + 1) * R, None], K, 1).astype(np.float16)
              for s in range(S)]
    B = np.repeat(b[None, :], K, 0).astype(np.float16)
    return np.array_equal(impl(shards, B), K * np.outer(a, b))


def pin_gather_order(impl):
    """Shard s carries the value s+1 in column 0; B = e_0 e_0^T: row block s of C is s+1."""
    S, R, K, N = 4, 3, 4, 2
    shards = [np.zeros((R, K), np.float16) for _ in range(S)]
    for s in range(S):
        shards[s][:, 0] = s + 1
    B = np.zeros((K, N), np.float16)
    B[0, 0] = 1
    want = np.zeros((S * R, N))
    want[:, 0] = np.repeat(np.arange(1, S + 1), R)
    return np.array_equal(impl(shards, B), want)


def _exact_dot(a16, b16):
    """Exact value of sum_k a[k] b[k] for fp16 vectors, as a Fraction."""
    ai = [int(v) for v in (a16.astype(np.float64) * 2.0 ** 24)]
    bi = [int(v) for v in (b16.astype(np.float64) * 2.0 ** 24)]
    return Fraction(sum(x * y for x, y in zip(ai, bi)), 2 ** 48)


def pin_brute_force(impl):
    """Tiny random shapes: fp64 result within the k-ordered summation bound of the exact sum."""
    rng = np.random.default_rng(12)
    for S, R, K, N in [(1, 3, 5, 4), (2, 2, 16, 3), (4, 1, 7, 9), (2, 5, 13, 2)]:
        shards = _shards(rng, S, R, K, scale=3.0)
        B = (rng.standard_normal((K, N)) * 3.0).astype(np.float16)
        C = impl(shards, B)
        A = np.concatenate(shards)
        if C.shape != (S * R, N):
            return False
        for m in range(S * R):
            for n in range(N):
                exact = _exact_dot(A[m], B[:, n])
                absdot = float(np.abs(A[m].astype(np.float64)) @ np.abs(B[:, n].astype(np.float64)))
                bound = K * 2.0 ** -53 * absdot * 1.01
                if abs(Fraction(C[m, n]) - exact) > Fraction(bound):
                    return False
    return True


def pin_brute_force_exact(impl):
    """Dyadic inputs with small exponents: every partial sum is exact in fp64."""
    rng = np.random.default_rng(13)
    S, R, K, N = 3, 2, 16, 5
    shards = [(rng.integers(-8, 9, (R, K)) / 4.0).astype(np.float16) for _ in range(S)]
    B = (rng.integers(-8, 9, (K, N)) / 8.0).astype(np.float16)
    A = np.concatenate(shards)
    want = np.array([[float(_exact_dot(A[m], B[:, n])) for n in range(N)]
                     for m in range(S * R)])
    return np.array_equal(impl(shards, B), want)


def pin_torch_f64(impl):
    """Mid-size random case against torch.matmul in float64 on the CPU."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(14)
    S, R, K, N = 3, 37, 129, 65
    shards = _shards(rng, S, R, K)
    B = rng.standard_normal((K, N)).astype(np.float16)
    A = torch.from_numpy(np.concatenate(shards).astype(np.float64))
    ref = (A @ torch.from_numpy(B.astype(np.float64))).numpy()
    C = impl(shards, B)
    return C.shape == ref.shape and np.allclose(C, ref, rtol=1e-12, atol=1e-12)


F16_PINS = [pin_one_hot_permutation, pin_single_entry, pin_rank_one,
            pin_gather_order, pin_brute_force, pin_brute_force_exact,
            pin_torch_f64]


@pytest.mark.parametrize("pin", F16_PINS, ids=lambda p: p.__name__)
def test_oracle_f16_pins(oracle, pin):
    assert pin(oracle.ag_gemm_f16)


# Plausible mistakes; each must fail at least one pin.
def _mut_transposed_b(shards, B):
    A = np.concatenate(shards).astype(np.float64)
    Bt = B.astype(np.float64)
    K, N = Bt.shape
    Bsq = np.zeros((K, N))
    Bsq[:min(K, N), :min(K, N)] = Bt[:min(K, N), :min(K, N)].T
    return A @ Bsq


def _mut_drop_last_k(shards, B):
    A = np.concatenate(shards).astype(np.float64)
    return A[:, :-1] @ B.astype(np.float64)[:-1]


def _mut_reversed_shards(shards, B):
    return np.concatenate(shards[::-1]).astype(np.float64) @ B.astype(np.float64)


def _mut_sign(shards, B):
    A = np.concatenate(shards).astype(np.float64)
    C = A @ B.astype(np.float64)
    C[-1, -1] = -C[-1, -1]
    return C


def _mut_fp32_accumulate(shards, B):
    A = np.concatenate(shards).astype(np.float32)
    return (A @ B.astype(np.float32)).astype(np.float64)


def _mut_one_shard_repeated(shards, B):
    return np.concatenate([shards[0]] * len(shards)).astype(np.float64) @ B.astype(np.float64)


@pytest.mark.parametrize("mutant", [_mut_transposed_b, _mut_drop_last_k,
                                    _mut_reversed_shards, _mut_sign,
                                    _mut_fp32_accumulate, _mut_one_shard_repeated],
                         ids=lambda f: f.__name__)
def test_f16_pins_catch_mutant(mutant):
    assert not all(pin(mutant) for pin in F16_PINS)


def test_oracle_f16_at_matches_full(oracle):
    rng = np.random.default_rng(15)
    S, R, K, N = 3, 9, 33, 17
    shards = _shards(rng, S, R, K)
    B = rng.standard_normal((K, N)).astype(np.float16)
    full = oracle.ag_gemm_f16(shards, B)
    rows = rng.integers(0, S * R, 200)
    cols = rng.integers(0, N, 200)
    assert np.array_equal(oracle.ag_gemm_f16_at(shards, B, rows, cols), full[rows, cols])


def test_oracle_single_shard_is_plain_gemm(oracle):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(16)
    A = rng.standard_normal((23, 40)).astype(np.float16)
    B = rng.standard_normal((40, 31)).astype(np.float16)
    ref = (torch.from_numpy(A.astype(np.float64)) @ torch.from_numpy(B.astype(np.float64))).numpy()
    assert np.allclose(oracle.ag_gemm_f16([A], B), ref, rtol=1e-13, atol=1e-13)


def test_oracle_allgather_concatenates_in_rank_order(oracle):
    rng = np.random.default_rng(17)
    shards = [rng.integers(-127, 128, (4, 6), dtype=np.int8) for _ in range(3)]
    assert np.array_equal(oracle.allgather(shards), np.concatenate(shards))


# ---------------------------------------------------------------------------
# int8 AllGatherMatmulDequant
# ---------------------------------------------------------------------------

def _i8_case(rng, S, R, K, N):
    shards = [rng.integers(-127, 128, (R, K), dtype=np.int8) for _ in range(S)]
    B = rng.integers(-127, 128, (K, N), dtype=np.int8)
    bias = rng.integers(-1000, 1001, N, dtype=np.int32)
    scale = rng.uniform(1e-5, 1e-4, N).astype(np.float32)
    return shards, B, bias, scale


def pin_i8_bigint(impl):
    """Exact Python-integer brute force of A x B + bias."""
    rng = np.random.default_rng(20)
    for S, R, K, N in [(1, 2, 5, 3), (2, 3, 17, 4), (4, 1, 9, 6)]:
        shards, B, bias, scale = _i8_case(rng, S, R, K, N)
        C, _ = impl(shards, B, bias, scale)
        A = np.concatenate(shards)
        for m in range(S * R):
            for n in range(N):
                want = sum(int(A[m, k]) * int(B[k, n]) for k in range(K)) + int(bias[n])
                if int(C[m, n]) != want:
                    return False
    return True


def pin_i8_all_127(impl):
    """Worst case of the pages' range: all +127 gives acc = K * 127^2; -127 in B flips it."""
    S, R, K, N = 2, 2, 300, 3
    shards = [np.full((R, K), 127, np.int8) for _ in range(S)]
    B = np.full((K, N), 127, np.int8)
    B[:, 1] = -127
    bias = np.array([5, -7, 0], np.int32)
    scale = np.full(N, 1e-5, np.float32)
    C, _ = impl(shards, B, bias, scale)
    want = np.array([K * 16129 + 5, -K * 16129 - 7, K * 16129], np.int64)
    return np.array_equal(C.astype(np.int64), np.broadcast_to(want, C.shape))


def pin_i8_debug_mode(impl):
    """All-ones A and B with a bias and scale per channel (debug mode of the
    dequant design doc, 8.6): C = K + bias[n], D = fp16(fp32(K + bias[n]) * scale[n])."""
    S, R, K, N = 2, 3, 64, 5
    shards = [np.ones((R, K), np.int8) for _ in range(S)]
    B = np.ones((K, N), np.int8)
    bias = np.array([0, 1, -64, 1000, 7], np.int32)
    scale = np.array([1e-5, 0.5, 3.0, 2.0 ** -20, 1.0 / 3.0], np.float32)
    C, D = impl(shards, B, bias, scale)
    wantC = (K + bias).astype(np.int32)
    wantD = (wantC.astype(np.float32) * scale).astype(np.float16)   # numpy IEEE fp32 multiply
    return (np.array_equal(C, np.broadcast_to(wantC, C.shape))
            and np.array_equal(D.view(np.uint16), np.broadcast_to(wantD.view(np.uint16), D.shape)))


def pin_i8_dequant_numpy(impl):
    """Random case: D equals numpy's fp16(fp32(C) * scale) of the (pinned) C."""
    rng = np.random.default_rng(21)
    shards, B, bias, scale = _i8_case(rng, 3, 4, 96, 11)
    C, D = impl(shards, B, bias, scale)
    wantD = (C.astype(np.float32) * scale[None, :]).astype(np.float16)
    return np.array_equal(D.view(np.uint16), wantD.view(np.uint16))


def pin_i8_gather_order(impl):
    S, R, K, N = 3, 2, 16, 2
    shards = [np.zeros((R, K), np.int8) for _ in range(S)]
    for s in range(S):
        shards[s][:, 0] = s + 1
    B = np.zeros((K, N), np.int8)
    B[0, 0] = 1
    bias = np.zeros(N, np.int32)
    scale = np.ones(N, np.float32)
    C, _ = impl(shards, B, bias, scale)
    want = np.zeros((S * R, N), np.int32)
    want[:, 0] = np.repeat(np.arange(1, S + 1), R)
    return np.array_equal(C, want)


I8_PINS = [pin_i8_bigint, pin_i8_all_127, pin_i8_debug_mode,
           pin_i8_dequant_numpy, pin_i8_gather_order]


@pytest.mark.parametrize("pin", I8_PINS, ids=lambda p: p.__name__)
def test_oracle_i8_pins(oracle, pin):
    assert pin(oracle.ag_gemm_dequant)


def _i8_numpy(shards, B, bias, scale, bias_by_row=False, trunc=False, order=None):
    A = np.concatenate(shards if order is None else [shards[i] for i in order]).astype(np.int64)
    C = A @ B.astype(np.int64)
    C = C + (bias[: C.shape[0], None] if bias_by_row and C.shape[0] <= bias.size
             else bias[None, :].astype(np.int64))
    f = C.astype(np.float32) * scale[None, :]
    if trunc:
        D = np.trunc(f.astype(np.float64) * 1024) / 1024
        D = D.astype(np.float32).astype(np.float16)
        D = np.where(np.abs(f) > 1, (np.sign(f) * np.floor(np.abs(f))).astype(np.float16), D)
    else:
        D = f.astype(np.float16)
    return C.astype(np.int32), D


@pytest.mark.parametrize("mutant", [
    lambda *a: _i8_numpy(*a, bias_by_row=True),
    lambda *a: _i8_numpy(*a, trunc=True),
    lambda sh, B, b, s: _i8_numpy(sh[::-1], B, b, s),
    lambda sh, B, b, s: (lambda C, D: (C - 1, D))(*_i8_numpy(sh, B, b, s)),
], ids=["bias_by_row", "truncating_cast", "reversed_shards", "off_by_one"])
def test_i8_pins_catch_mutant(mutant):
    assert not all(pin(mutant) for pin in I8_PINS)


def test_i8_reference_numpy_passes_pins():
    """The numpy restatement used for the mutants is itself right when unmutated."""
    assert all(pin(_i8_numpy) for pin in I8_PINS)


def test_oracle_i8_at_matches_full(oracle):
    rng = np.random.default_rng(22)
    shards, B, bias, scale = _i8_case(rng, 3, 7, 48, 13)
    C, D = oracle.ag_gemm_dequant(shards, B, bias, scale)
    rows = rng.integers(0, 21, 150)
    cols = rng.integers(0, 13, 150)
    Cs, Ds = oracle.ag_gemm_dequant_at(shards, B, bias, scale, rows, cols)
    assert np.array_equal(Cs, C[rows, cols])
    assert np.array_equal(Ds.view(np.uint16), D.view(np.uint16)[rows, cols])


def test_oracle_i8_rejects_int32_overflow(oracle):
    shards = [np.full((1, 4), 127, np.int8)]
    B = np.full((4, 1), 127, np.int8)
    bias = np.array([2 ** 31 - 1], np.int32)
    with pytest.raises(oracle.OracleError):
        oracle.ag_gemm_dequant(shards, B, bias, np.ones(1, np.float32))


def test_oracle_dequant_vs_numpy(oracle):
    rng = np.random.default_rng(23)
    c = rng.integers(-2 ** 31, 2 ** 31, 200_000, dtype=np.int64).astype(np.int32)
    s = rng.uniform(1e-6, 1e-3, c.size).astype(np.float32)
    with np.errstate(over="ignore"):
        want = (c.astype(np.float32) * s).astype(np.float16)
    assert np.array_equal(oracle.dequant(c, s).view(np.uint16), want.view(np.uint16))


# ---------------------------------------------------------------------------
# bfloat16 (the Pallas:MGPU page's default operand type)
# ---------------------------------------------------------------------------
# numpy has no bfloat16; values are uint16 bit patterns.  A bfloat16 is the
# upper half of a binary32, so numpy's float32 decoding of (bits << 16) and an
# integer round-half-even on float32 bit patterns are independent references.

def _bf16_ref_decode(bits):
    with np.errstate(invalid="ignore"):
        return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bf16_ref_round_f32(x32):
    """Round-to-nearest-even of float32 values to bfloat16, on the bit patterns."""
    u = x32.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def test_bf16_decode_all_bit_patterns(oracle):
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.bf16_bits_to_f64(bits)
    ref = _bf16_ref_decode(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.signbit(got[0x8000]) and not np.signbit(got[0])


def test_bf16_encode_random_float32_vs_bit_rounding(oracle):
    rng = np.random.default_rng(30)
    x = np.concatenate([
        rng.standard_normal(300_000) * 10.0 ** rng.integers(-40, 39, 300_000),
        rng.uniform(-1e-38, 1e-38, 100_000),
        rng.integers(-2 ** 24, 2 ** 24, 100_000).astype(np.float64),
    ])
    with np.errstate(over="ignore"):
        x32 = x.astype(np.float32)
    x32 = x32[np.isfinite(x32)]
    got = oracle.f64_to_bf16_bits(x32.astype(np.float64))
    assert np.array_equal(got, _bf16_ref_round_f32(x32))


@pytest.mark.parametrize("x,bits", [
    (1.0, 0x3F80), (-2.0, 0xC000), (1 + 2 ** -8, 0x3F80),      # tie -> even (1.0)
    (1 + 3 * 2 ** -8, 0x3F82),                                  # tie -> even (1 + 2^-6)
    (1 + 2 ** -8 + 2 ** -30, 0x3F81),                           # just above the tie
    ((2 - 2 ** -7) * 2.0 ** 127, 0x7F7F),                       # largest finite
    ((2 - 2 ** -8) * 2.0 ** 127, 0x7F80),                       # tie above it -> inf
    (2.0 ** -133, 0x0001), (2.0 ** -134, 0x0000),               # smallest subnormal, its half
    (1.5 * 2.0 ** -133, 0x0002), (2.0 ** -126, 0x0080),         # subnormal tie, smallest normal
    (-0.0, 0x8000), (float("inf"), 0x7F80), (-float("inf"), 0xFF80),
])
def test_bf16_encode_boundaries(oracle, x, bits):
    assert int(oracle.f64_to_bf16_bits(np.array([x]))[0]) == bits


def _bf16_bits(rng, shape, scale=1.0):
    return _bf16_ref_round_f32((rng.standard_normal(shape) * scale).astype(np.float32))


def _bf16_of(values):
    """Bit patterns of float values that bfloat16 represents exactly."""
    x32 = np.asarray(values, np.float32)
    bits = (x32.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(_bf16_ref_decode(bits), x32.astype(np.float64))
    return bits


def bpin_one_hot_permutation(impl):
    """B[k][n] = [k == pi(n)]  =>  C[:, n] = A[:, pi(n)] exactly."""
    rng = np.random.default_rng(31)
    S, R, K, N = 3, 5, 11, 7
    shards = [_bf16_bits(rng, (R, K)) for _ in range(S)]
    pi = rng.permutation(K)[:N]
    B = np.zeros((K, N), np.float32)
    B[pi, np.arange(N)] = 1
    A = _bf16_ref_decode(np.concatenate(shards))
    return np.array_equal(impl(shards, _bf16_of(B)), A[:, pi])


def bpin_rank_one(impl):
    """A[m][k] = a_m, B[k][n] = b_n (small integers)  =>  C = K a_m b_n."""
    S, R, K, N = 2, 3, 37, 5
    a = np.arange(1, S * R + 1) - 3.0
    b = np.array([2.0, -1.0, 3.0, 0.5, -4.0])
    shards = [_bf16_of(np.repeat(a[s * R:(s + 1) * R, None], K, 1)) for s in range(S)]
    B = _bf16_of(np.repeat(b[None, :], K, 0))
    return np.array_equal(impl(shards, B), K * np.outer(a, b))


def bpin_gather_order(impl):
    """Shard s carries s + 1 in column 0, B = e_0 e_0^T: row block s of C is s + 1."""
    S, R, K, N = 4, 3, 4, 2
    vals = [np.zeros((R, K)) for _ in range(S)]
    for s in range(S):
        vals[s][:, 0] = s + 1
    B = np.zeros((K, N))
    B[0, 0] = 1
    want = np.zeros((S * R, N))
    want[:, 0] = np.repeat(np.arange(1, S + 1), R)
    return np.array_equal(impl([_bf16_of(v) for v in vals], _bf16_of(B)), want)


def bpin_brute_force_exact(impl):
    """Dyadic inputs with small exponents: every partial sum is exact in fp64."""
    rng = np.random.default_rng(32)
    S, R, K, N = 3, 2, 16, 5
    vals = [rng.integers(-8, 9, (R, K)) / 4.0 for _ in range(S)]
    Bv = rng.integers(-8, 9, (K, N)) / 8.0
    A = np.concatenate(vals)
    want = np.array([[float(sum(Fraction(A[m, k]) * Fraction(Bv[k, n]) for k in range(K)))
                      for n in range(N)] for m in range(S * R)])
    return np.array_equal(impl([_bf16_of(v) for v in vals], _bf16_of(Bv)), want)


def bpin_torch_f64(impl):
    """Mid-size random case against torch's bfloat16 -> float64 matmul on the CPU."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(33)
    S, R, K, N = 3, 37, 129, 65
    shards = [_bf16_bits(rng, (R, K)) for _ in range(S)]
    B = _bf16_bits(rng, (K, N))
    to_t = lambda b: torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).double()  # noqa: E731
    ref = (to_t(np.concatenate(shards)) @ to_t(B)).numpy()
    C = impl(shards, B)
    return C.shape == ref.shape and np.allclose(C, ref, rtol=1e-12, atol=1e-12)


BF16_PINS = [bpin_one_hot_permutation, bpin_rank_one, bpin_gather_order,
             bpin_brute_force_exact, bpin_torch_f64]


@pytest.mark.parametrize("pin", BF16_PINS, ids=lambda p: p.__name__)
def test_oracle_bf16_pins(oracle, pin):
    assert pin(oracle.ag_gemm_bf16)


def _bmut_decoded_as_f16(shards, B):
    A = np.concatenate(shards).view(np.float16).astype(np.float64)
    return A @ B.view(np.float16).astype(np.float64)


def _bmut_transposed_b(shards, B):
    A = _bf16_ref_decode(np.concatenate(shards))
    Bd = _bf16_ref_decode(B)
    return A @ (Bd.T if Bd.shape[0] == Bd.shape[1] else Bd[::-1])


def _bmut_reversed_shards(shards, B):
    return _bf16_ref_decode(np.concatenate(shards[::-1])) @ _bf16_ref_decode(B)


def _bmut_truncated_mantissa(shards, B):
    # a decode that drops the lowest fraction bit
    A = _bf16_ref_decode(np.concatenate(shards) & 0xFFFE)
    return A @ _bf16_ref_decode(B & 0xFFFE)


@pytest.mark.parametrize("mutant", [_bmut_decoded_as_f16, _bmut_transposed_b,
                                    _bmut_reversed_shards, _bmut_truncated_mantissa],
                         ids=lambda f: f.__name__)
def test_bf16_pins_catch_mutant(mutant):
    assert not all(pin(mutant) for pin in BF16_PINS)


def test_oracle_bf16_at_matches_full(oracle):
    rng = np.random.default_rng(34)
    shards = [_bf16_bits(rng, (6, 40)) for _ in range(3)]
    B = _bf16_bits(rng, (40, 9))
    C = oracle.ag_gemm_bf16(shards, B)
    rows = rng.integers(0, 18, 50)
    cols = rng.integers(0, 9, 50)
    assert np.array_equal(oracle.ag_gemm_bf16_at(shards, B, rows, cols), C[rows, cols])


# ---------------------------------------------------------------------------
# N-sharded collective matmul: ring order ("Collective matrix multiplication",
# 算法概述：Ring All-Gather)
# ---------------------------------------------------------------------------

def _ring_placement_pin(ring, D, d):
    """Shards whose column 0 holds their rank index and B_d with a single row of
    ones: row block s of rank d's output must be all s -- a closed form that
    does not depend on the oracle's GEMM."""
    R, K, ns = 3, 5, 4
    shards = [np.zeros((R, K), np.float16) for _ in range(D)]
    for s in range(D):
        shards[s][:, 0] = s
    B_d = np.zeros((K, ns), np.float16)
    B_d[0, :] = 1
    out = ring(shards, B_d, d)
    want = np.repeat(np.arange(D, dtype=np.float64), R)[:, None] * np.ones((1, ns))
    return out.shape == want.shape and np.array_equal(out, want)


@pytest.mark.parametrize("D", [1, 2, 3, 4])
def test_ring_places_each_step_in_its_row_slice(oracle, D):
    for d in range(D):
        assert _ring_placement_pin(oracle.collective_matmul_ring, D, d)


@pytest.mark.parametrize("D,R,K,ns", [(2, 5, 7, 3), (3, 4, 16, 8), (4, 2, 9, 5)])
def test_ring_column_shards_assemble_the_product(oracle, D, R, K, ns):
    """Ranks 0..D-1, each with its column shard B_d, together give
    AllGather(A) x B: checked against torch float64 matmul on the CPU."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(100 + D * 10 + K)
    shards = [rng.standard_normal((R, K)).astype(np.float16) for _ in range(D)]
    B = rng.standard_normal((K, D * ns)).astype(np.float16)
    full = np.concatenate([oracle.collective_matmul_ring(shards, B[:, d * ns:(d + 1) * ns], d)
                           for d in range(D)], axis=1)
    A = np.concatenate(shards).astype(np.float64)
    ref = (torch.from_numpy(A) @ torch.from_numpy(B.astype(np.float64))).numpy()
    assert np.allclose(full, ref, rtol=1e-13, atol=1e-13)
    # the same sums as the one-shot definition, element by element
    assert np.array_equal(full, oracle.ag_gemm_f16(shards, B))


def test_ring_bf16_matches_definition(oracle):
    rng = np.random.default_rng(7)
    D, R, K, ns = 3, 4, 24, 8
    shards = [oracle.f64_to_bf16_bits(rng.standard_normal((R, K))) for _ in range(D)]
    B = oracle.f64_to_bf16_bits(rng.standard_normal((K, D * ns)))
    full = np.concatenate([oracle.collective_matmul_ring(shards, B[:, d * ns:(d + 1) * ns], d,
                                                         dtype="bf16") for d in range(D)], axis=1)
    assert np.array_equal(full, oracle.ag_gemm_bf16(shards, B))


def test_ring_pin_catches_misplaced_steps(oracle):
    """Planted mistakes in the ring's bookkeeping: step i written to slice i,
    the ring walked backwards with the forward slice index, one step repeated."""
    def to_step_index(shards, B_d, d):
        D, R = len(shards), shards[0].shape[0]
        out = np.empty((D * R, B_d.shape[1]))
        for i in range(D):
            out[i * R:(i + 1) * R] = oracle.ag_gemm_f16([shards[(d + i) % D]], B_d)
        return out

    def backwards(shards, B_d, d):
        D, R = len(shards), shards[0].shape[0]
        out = np.empty((D * R, B_d.shape[1]))
        for i in range(D):
            out[((d + i) % D) * R:((d + i) % D + 1) * R] = \
                oracle.ag_gemm_f16([shards[(d - i) % D]], B_d)
        return out

    def repeated(shards, B_d, d):
        D, R = len(shards), shards[0].shape[0]
        out = np.empty((D * R, B_d.shape[1]))
        for i in range(D):
            src = (d + min(i, 1)) % D
            out[((d + i) % D) * R:((d + i) % D + 1) * R] = oracle.ag_gemm_f16([shards[src]], B_d)
        return out

    for bad in (to_step_index, backwards, repeated):
        assert not all(_ring_placement_pin(bad, 3, d) for d in range(3)), bad.__name__
