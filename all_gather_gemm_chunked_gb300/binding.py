"""ctypes binding of libaggemm.so (include/ag_gemm.h).

Argument marshalling only: every step of the path runs in the CUDA library.
The functions keep the C names; pointers are passed as Python ints (device
addresses), ``shard_ptrs`` as a sequence of ints, ``stream`` as a
cudaStream_t handle (int, 0 = legacy default stream).  Failures raise
:class:`AgGemmError` with the library's code and message.

Importing this module loads the library and fails loudly if it is missing:
there is no CPU or framework fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

from . import build as _build

F16, I8, BF16 = 0, 1, 2
MODE_PIPELINED, MODE_COMPUTE_ONLY, MODE_SEQUENTIAL, MODE_COPY_ONLY = 0, 1, 2, 3
DEBUG_POISON_STAGING, DEBUG_SKIP_ITEM, DEBUG_DELAY_NS = 1, 2, 4
PATH_FUSED_F16, PATH_FUSED_I8, PATH_SKINNY_I8 = 0, 1, 2
(TRACE_CTA_START, TRACE_CTA_END, TRACE_LANDED, TRACE_WAIT_START, TRACE_WAIT_END, TRACE_TILE_DONE,
 TRACE_UNIT_ISSUED, TRACE_UNIT_LANDED, TRACE_KB_WIDENED, TRACE_KB_MMA,
 TRACE_PIECE_DONE, TRACE_COPY_START, TRACE_ACC_READY, TRACE_PARTS_READY) = range(1, 15)
OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_CUDA, ERR_OOM, ERR_TIMEOUT, ERR_STATE = 0, -1, -2, -3, -4, -5, -6
ERROR_NAMES = {ERR_INVALID: "INVALID", ERR_UNSUPPORTED: "UNSUPPORTED", ERR_CUDA: "CUDA",
               ERR_OOM: "OOM", ERR_TIMEOUT: "TIMEOUT", ERR_STATE: "STATE"}

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "ag_gemm.h")


class AgGemmError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"ag_gemm error {code} ({ERROR_NAMES.get(code, '?')}): {message}")
        self.code = code
        self.message = message


class Geometry(ctypes.Structure):
    _fields_ = [
        ("n_shards", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("M", ctypes.c_int64), ("K", ctypes.c_int64), ("N", ctypes.c_int64), ("R", ctypes.c_int64),
        ("chunk_rows", ctypes.c_int64), ("chunks_per_source", ctypes.c_int64),
        ("pieces_per_chunk", ctypes.c_int32),
        ("block_m", ctypes.c_int32), ("block_n", ctypes.c_int32), ("block_k", ctypes.c_int32),
        ("group_m", ctypes.c_int32), ("kseg_blocks", ctypes.c_int32),
        ("m_tiles", ctypes.c_int64), ("n_tiles", ctypes.c_int64), ("tiles", ctypes.c_int64),
        ("producer_items", ctypes.c_int64), ("staging_bytes", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_int64), ("staging_slots", ctypes.c_int64),
        ("split_tiles", ctypes.c_int64), ("split_parts", ctypes.c_int64),
    ]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class TraceEvent(ctypes.Structure):
    """ag_gemm_trace_event."""
    _fields_ = [("t_ns", ctypes.c_uint64), ("kind", ctypes.c_uint32), ("cta", ctypes.c_uint32),
                ("warp", ctypes.c_uint32), ("id", ctypes.c_uint32), ("aux", ctypes.c_uint64)]


def _load():
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"libaggemm.so is not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    i32, i64, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
    geo_p = ctypes.POINTER(Geometry)
    i64_arr = ctypes.POINTER(ctypes.c_int64)
    sig = {
        "ag_gemm_choose_chunk_rows": (i64, [i64]),
        "ag_gemm_validate": (i32, [i32, i64, i64, i64, i32, i64]),
        "ag_gemm_geometry_of": (i32, [i32, i64, i64, i64, i32, i64, geo_p]),
        "ag_gemm_tile_at": (i32, [geo_p, i32, i64, i64_arr]),
        "ag_gemm_item_at": (i32, [geo_p, i32, i64, i64_arr]),
        "ag_gemm_plan_create": (vp, [i32, i64, i64, i64, i32, i64]),
        "ag_gemm_plan_create_bounded": (vp, [i32, i64, i64, i64, i32, i64, i32]),
        "ag_gemm_choose_chunk_rows_bounded": (i64, [i64]),
        "ag_gemm_plan_destroy": (None, [vp]),
        "ag_gemm_plan_geometry": (i32, [vp, geo_p]),
        "ag_gemm_plan_chunk_rows": (i64, [vp]),
        "ag_gemm_run": (i32, [vp, ctypes.POINTER(vp), vp, vp, vp]),
        "ag_gemm_run_ld": (i32, [vp, ctypes.POINTER(vp), vp, i64, vp, i64, vp]),
        "ag_gemm_dequant_run": (i32, [vp, ctypes.POINTER(vp), vp, vp, vp, vp, vp, vp]),
        "ag_gemm_plan_status": (i32, [vp]),
        "ag_gemm_plan_status_word": (i64, [vp]),
        "ag_gemm_plan_reset": (i32, [vp, vp]),
        "ag_gemm_plan_set_mode": (i32, [vp, i32]),
        "ag_gemm_plan_set_local_rank": (i32, [vp, i32]),
        "ag_gemm_plan_set_timeout_ns": (i32, [vp, i64]),
        "ag_gemm_plan_set_debug": (i32, [vp, i32, i64]),
        "ag_gemm_plan_grid": (i32, [vp]),
        "ag_gemm_plan_path": (i32, [vp]),
        "ag_gemm_run_noalloc": (i32, [i32, i64, i64, i64, i64, ctypes.POINTER(vp), vp, vp, vp, vp]),
        "ag_gemm_plan_set_trace": (i32, [vp, i64]),
        "ag_gemm_plan_set_grid": (i32, [vp, i32]),
        "ag_gemm_plan_trace": (i64, [vp, ctypes.POINTER(TraceEvent), i64]),
        "ag_gemm_last_error": (i32, []),
        "ag_gemm_last_error_message": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def header_functions(path: str = HEADER):
    """Names of the functions include/ag_gemm.h declares."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ag_gemm_\w+)\s*\(", text)))


def library_handle():
    return _lib


def _err():
    return AgGemmError(_lib.ag_gemm_last_error(), (_lib.ag_gemm_last_error_message() or b"").decode())


def _check(rc):
    if rc < 0:
        raise _err()
    return rc


def _ptrs(seq):
    arr = (ctypes.c_void_p * len(seq))(*[int(x) for x in seq])
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)), arr


# -- thin wrappers, same names as the C ABI ---------------------------------

def ag_gemm_choose_chunk_rows(R: int) -> int:
    return _check(_lib.ag_gemm_choose_chunk_rows(R))


def ag_gemm_choose_chunk_rows_bounded(R: int) -> int:
    return _check(_lib.ag_gemm_choose_chunk_rows_bounded(R))


def ag_gemm_validate(n_shards, M, K, N, dtype, chunk_rows) -> int:
    return _check(_lib.ag_gemm_validate(n_shards, M, K, N, dtype, chunk_rows))


def ag_gemm_geometry_of(n_shards, M, K, N, dtype, chunk_rows) -> Geometry:
    g = Geometry()
    _check(_lib.ag_gemm_geometry_of(n_shards, M, K, N, dtype, chunk_rows, ctypes.byref(g)))
    return g


def ag_gemm_tile_at(geometry: Geometry, local_rank: int, t: int):
    out = (ctypes.c_int64 * 3)()
    _check(_lib.ag_gemm_tile_at(ctypes.byref(geometry), local_rank, t, out))
    return tuple(out)


def ag_gemm_item_at(geometry: Geometry, local_rank: int, i: int):
    out = (ctypes.c_int64 * 4)()
    _check(_lib.ag_gemm_item_at(ctypes.byref(geometry), local_rank, i, out))
    return tuple(out)


def ag_gemm_plan_create(n_shards, M, K, N, dtype, chunk_rows=0) -> int:
    h = _lib.ag_gemm_plan_create(n_shards, M, K, N, dtype, chunk_rows)
    if not h:
        raise _err()
    return h


def ag_gemm_plan_create_bounded(n_shards, M, K, N, dtype, chunk_rows=0, staging_slots=0) -> int:
    h = _lib.ag_gemm_plan_create_bounded(n_shards, M, K, N, dtype, chunk_rows, staging_slots)
    if not h:
        raise _err()
    return h


def ag_gemm_plan_destroy(plan: int) -> None:
    _lib.ag_gemm_plan_destroy(plan)


def ag_gemm_plan_geometry(plan: int) -> Geometry:
    g = Geometry()
    _check(_lib.ag_gemm_plan_geometry(plan, ctypes.byref(g)))
    return g


def ag_gemm_plan_chunk_rows(plan: int) -> int:
    return _check(_lib.ag_gemm_plan_chunk_rows(plan))


def ag_gemm_run(plan: int, shard_ptrs, B: int, C: int, stream: int = 0) -> int:
    p, _keep = _ptrs(shard_ptrs)
    return _check(_lib.ag_gemm_run(plan, p, B, C, stream))


def ag_gemm_run_ld(plan: int, shard_ptrs, B: int, ldb: int, C: int, ldc: int,
                   stream: int = 0) -> int:
    p, _keep = _ptrs(shard_ptrs)
    return _check(_lib.ag_gemm_run_ld(plan, p, B, ldb, C, ldc, stream))


def ag_gemm_dequant_run(plan: int, shard_ptrs, B: int, bias: int, scale: int, C_i32: int,
                        D_f16: int, stream: int = 0) -> int:
    p, _keep = _ptrs(shard_ptrs)
    return _check(_lib.ag_gemm_dequant_run(plan, p, B, bias, scale, C_i32, D_f16, stream))


def ag_gemm_plan_status(plan: int) -> int:
    """AG_GEMM_OK or a negative code (not raised: a timeout is an expected outcome)."""
    return _lib.ag_gemm_plan_status(plan)


def ag_gemm_plan_status_word(plan: int) -> int:
    return _check(_lib.ag_gemm_plan_status_word(plan))


def ag_gemm_plan_reset(plan: int, stream: int = 0) -> int:
    return _check(_lib.ag_gemm_plan_reset(plan, stream))


def ag_gemm_plan_set_mode(plan: int, mode: int) -> int:
    return _check(_lib.ag_gemm_plan_set_mode(plan, mode))


def ag_gemm_plan_set_local_rank(plan: int, local_rank: int) -> int:
    return _check(_lib.ag_gemm_plan_set_local_rank(plan, local_rank))


def ag_gemm_plan_set_timeout_ns(plan: int, ns: int) -> int:
    return _check(_lib.ag_gemm_plan_set_timeout_ns(plan, ns))


def ag_gemm_plan_set_debug(plan: int, flags: int, arg: int = 0) -> int:
    return _check(_lib.ag_gemm_plan_set_debug(plan, flags, arg))


def ag_gemm_plan_set_grid(plan: int, ctas: int) -> int:
    return _check(_lib.ag_gemm_plan_set_grid(plan, ctas))


def ag_gemm_plan_grid(plan: int) -> int:
    return _check(_lib.ag_gemm_plan_grid(plan))


def ag_gemm_plan_path(plan: int) -> int:
    return _check(_lib.ag_gemm_plan_path(plan))


def ag_gemm_run_noalloc(n_shards, M, K, N, chunk_rows, shard_ptrs, B: int, C: int,
                        status_out: int = 0, stream: int = 0) -> int:
    """fp16 run that allocates nothing: scratch comes from the library's fixed array."""
    p, _keep = _ptrs(shard_ptrs)
    return _check(_lib.ag_gemm_run_noalloc(n_shards, M, K, N, chunk_rows, p, B, C,
                                           status_out or None, stream))


def ag_gemm_plan_set_trace(plan: int, capacity: int) -> int:
    return _check(_lib.ag_gemm_plan_set_trace(plan, capacity))


def ag_gemm_plan_trace(plan: int, max_events: int):
    """(events recorded by the last run, numpy structured array of the kept ones)."""
    import numpy as np
    buf = (TraceEvent * max(max_events, 1))()
    n = _check(_lib.ag_gemm_plan_trace(plan, buf, max_events))
    kept = min(n, max_events)
    dt = np.dtype([("t_ns", "<u8"), ("kind", "<u4"), ("cta", "<u4"), ("warp", "<u4"),
                   ("id", "<u4"), ("aux", "<u8")])
    arr = np.frombuffer(bytes(buf), dtype=dt, count=kept).copy()
    return n, arr


def ag_gemm_last_error() -> int:
    return _lib.ag_gemm_last_error()


def ag_gemm_last_error_message() -> str:
    return (_lib.ag_gemm_last_error_message() or b"").decode()
