"""C-ABI boundary and host logic, without a GPU: the library loads, exports
every function include/ag_gemm.h declares, validates arguments, sizes chunks
as the chunk-size rule says, and its tile schedule and copy items cover the
problem exactly once in consumption order."""
import subprocess

import pytest

from all_gather_gemm_chunked_gb300 import build as _build


@pytest.fixture(scope="module")
def B():
    _build.build()
    from all_gather_gemm_chunked_gb300 import binding
    return binding


def test_library_exports_every_header_function(B):
    names = B.header_functions()
    assert len(names) >= 20
    lib = B.library_handle()
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(names) <= exported


@pytest.mark.parametrize("R,c", [(128, 2), (2048, 32), (1024, 16), (4096, 64), (32, 1),
                                 (63, 1), (64, 1), (100, 1), (200, 2), (1000, 10),
                                 (917, 7), (65536, 1024)])
def test_chunk_rule(B, R, c):
    assert B.ag_gemm_choose_chunk_rows(R) == c
    q = R // c
    assert R % c == 0
    if R >= 64:
        assert q >= 64


def test_chunk_rule_keeps_64_to_128_chunks_when_possible(B):
    for R in range(64, 5000):
        c = B.ag_gemm_choose_chunk_rows(R)
        q = R // c
        assert R % c == 0 and q >= 64
        if any(R % d == 0 for d in range(64, 129)):
            assert 64 <= q <= 128


@pytest.mark.parametrize("args,code", [
    ((2, 256, 256, 128, 7, 0), -1),         # dtype
    ((2, 256, 12, 128, 2, 0), -1),          # bf16: K % 8
    ((0, 256, 256, 128, 0, 0), -1),         # n_shards
    ((65, 65 * 4, 256, 128, 0, 0), -1),
    ((3, 256, 256, 128, 0, 0), -1),         # M % S
    ((2, 256, 252, 128, 0, 0), -1),         # fp16 K % 8
    ((2, 256, 256, 124, 0, 0), -1),         # fp16 N % 8
    ((2, 256, 264, 128, 1, 0), -1),         # int8 K % 16
    ((2, 256, 256, 136, 1, 0), -1),         # int8 N % 16
    ((2, 256, 256, 128, 0, 3), -1),         # chunk_rows does not divide R
    ((2, 256, 256, 128, 0, -1), -1),
    ((2, 0, 256, 128, 0, 0), -1),
    ((2, 256, 133008, 128, 1, 0), -2),      # int8 K too large for exact int32
    ((2, 1 << 31, 256, 1 << 26, 0, 0), -2),  # 2^31 x 2^26 output: more than 2^30 pair tiles
])
def test_validate_rejects(B, args, code):
    with pytest.raises(B.AgGemmError) as e:
        B.ag_gemm_validate(*args)
    assert e.value.code == code
    assert B.ag_gemm_last_error() == code
    assert B.ag_gemm_last_error_message()


_DT = {"f16": 0, "i8": 1, "bf16": 2}


def test_validate_accepts_workloads(B):
    from all_gather_gemm_chunked_gb300.synth import WORKLOADS
    for w in WORKLOADS.values():
        assert B.ag_gemm_validate(w.S, w.M, w.K, w.N, _DT[w.dtype], w.chunk_rows) == 0


def test_geometry_of_workloads(B):
    from all_gather_gemm_chunked_gb300.synth import WORKLOADS
    want = {1: (16, 8), 2: (32, 64), 3: (16, 64), 4: (64, 64), 5: (1, 32), 6: (32, 64),
            7: (16, 64), 8: (64, 64), 9: (16, 64)}
    for wid, w in WORKLOADS.items():
        g = B.ag_gemm_geometry_of(w.S, w.M, w.K, w.N, _DT[w.dtype], w.chunk_rows)
        assert (g.chunk_rows, g.chunks_per_source) == want[wid]
        assert g.tiles == w.S * g.m_tiles * g.n_tiles
        assert g.producer_items == (w.S - 1) * g.chunks_per_source * g.pieces_per_chunk
        esz = 1 if w.dtype == "i8" else 2
        assert g.chunk_rows * w.K * esz // g.pieces_per_chunk <= 32 * 1024 + 16


def _geo(B, S, M, K, N, dtype=0, c=0):
    return B.ag_gemm_geometry_of(S, M, K, N, dtype, c)


@pytest.mark.parametrize("S,M,K,N,c", [(2, 256, 256, 128, 16), (3, 600, 328, 392, 0),
                                       (8, 8192, 64, 4096, 0), (1, 300, 64, 72, 0),
                                       (4, 4 * 37, 128, 520, 1)])
def test_tile_schedule_covers_each_tile_once_local_first(B, S, M, K, N, c):
    g = _geo(B, S, M, K, N, 0, c)
    for local in range(S):
        seen = []
        for t in range(g.tiles):
            seen.append(B.ag_gemm_tile_at(g, local, t))
        assert len(set(seen)) == g.tiles
        assert set(seen) == {(s, m, n) for s in range(S) for m in range(g.m_tiles)
                             for n in range(g.n_tiles)}
        # consumption order: local shard first, then (local+1) % S, ... (ring order)
        order = []
        for s, _, _ in seen:
            if not order or order[-1] != s:
                order.append(s)
        assert order == [(local + p) % S for p in range(S)]


@pytest.mark.parametrize("S,M,K,N,dt,c", [(2, 256, 256, 128, 0, 16), (3, 600, 328, 392, 0, 0),
                                          (4, 4 * 64, 27392 // 8, 64, 1, 0), (2, 64, 1024, 64, 1, 0)])
def test_copy_items_cover_remote_shards_in_consumption_order(B, S, M, K, N, dt, c):
    g = _geo(B, S, M, K, N, dt, c)
    esz = 2 if dt == 0 else 1
    shard_bytes = g.R * K * esz
    for local in range(S):
        cover = {s: [] for s in range(S)}
        last_pos = 0
        for i in range(g.producer_items):
            s, q, b0, b1 = B.ag_gemm_item_at(g, local, i)
            pos = (s - local) % S
            assert pos >= 1, "the local shard is never copied"
            assert pos >= last_pos, "items are numbered in consumption order"
            last_pos = pos
            chunk_bytes = g.chunk_rows * K * esz
            assert q * chunk_bytes <= b0 < b1 <= (q + 1) * chunk_bytes
            assert b0 % 16 == 0 and b1 % 16 == 0
            cover[s].append((b0, b1))
        for s in range(S):
            if s == local:
                assert cover[s] == []
                continue
            iv = sorted(cover[s])
            assert iv[0][0] == 0 and iv[-1][1] == shard_bytes
            assert all(a[1] == b[0] for a, b in zip(iv, iv[1:]))


def test_out_of_range_schedule_queries(B):
    g = _geo(B, 2, 256, 256, 128)
    with pytest.raises(B.AgGemmError):
        B.ag_gemm_tile_at(g, 0, g.tiles)
    with pytest.raises(B.AgGemmError):
        B.ag_gemm_tile_at(g, 2, 0)
    with pytest.raises(B.AgGemmError):
        B.ag_gemm_item_at(g, 0, g.producer_items)


def test_null_plan_is_rejected(B):
    lib = B.library_handle()
    assert lib.ag_gemm_run(None, None, None, None, None) == B.ERR_INVALID
    assert lib.ag_gemm_run_ld(None, None, None, 0, None, 0, None) == B.ERR_INVALID
    assert lib.ag_gemm_plan_set_mode(None, 0) == B.ERR_INVALID
    assert lib.ag_gemm_plan_status(None) == B.ERR_INVALID
    assert lib.ag_gemm_plan_path(None) == B.ERR_INVALID
    assert lib.ag_gemm_plan_grid(None) == B.ERR_INVALID
    lib.ag_gemm_plan_destroy(None)  # no-op


def test_plan_create_without_gpu_reports_cuda_error(B):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(B.AgGemmError) as e:
        B.ag_gemm_plan_create(2, 256, 256, 128, 0, 16)
    assert e.value.code in (B.ERR_CUDA, B.ERR_UNSUPPORTED)
