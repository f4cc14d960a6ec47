"""Helpers for the GPU parity tests: tolerances, fp16 ulp distance, sampling."""
import numpy as np

# fp16 path (fp32 accumulation): relative Frobenius error and max abs error.
F16_REL_FRO = 1e-4


def f16_max_abs(K):
    return 1e-3 * np.sqrt(K)


def f16_ulp_distance(got, ref):
    """Distance in fp16 ulps between bit patterns (+0 and -0 are equal)."""
    g = np.asarray(got).view(np.uint16).astype(np.int64)
    r = np.asarray(ref).view(np.uint16).astype(np.int64)

    def key(b):
        return np.where(b & 0x8000, -(b & 0x7FFF), b)

    return np.abs(key(g) - key(r))


def check_f16(got, ref, K, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite outputs"
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    mx = np.abs(got - ref).max() if got.size else 0.0
    assert rel <= F16_REL_FRO, f"{what}: relative Frobenius error {rel:.3e}"
    assert mx <= f16_max_abs(K), f"{what}: max abs error {mx:.3e} > {f16_max_abs(K):.3e}"
    return rel, mx


def tile_samples(rng, M, N, R, bm=128, bn=256, per_tile=4):
    """Sample points so that every (shard, m-tile, n-tile) gets corners and random points."""
    rows, cols = [], []
    S = M // R
    for s in range(S):
        for m0 in range(0, R, bm):
            m1 = min(m0 + bm, R)
            for n0 in range(0, N, bn):
                n1 = min(n0 + bn, N)
                rr = [m0, m1 - 1, m0, m1 - 1] + list(rng.integers(m0, m1, per_tile))
                cc = [n0, n0, n1 - 1, n1 - 1] + list(rng.integers(n0, n1, per_tile))
                rows += [s * R + r for r in rr]
                cols += cc
    return np.array(rows, np.int64), np.array(cols, np.int64)
