"""CPU oracle for the streamed AllGather+GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library never loads it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, single-threaded, fp64 for the
fp16 GEMM, exact int64 for the int8 GEMM, IEEE round-to-nearest-even written
out for binary16/binary32).  This module compiles it with gcc on first use
and marshals numpy arrays to it; it adds no arithmetic of its own.

Functions and what they state (page titles and sections):

* ``ag_gemm_f16`` -- "AllGather + GEMM 通算融合算子示例", 计算功能:
  C = AllGather(A) x B, fp16 in, fp32 (here fp64) out.
* ``ag_gemm_dequant`` -- "AllGather矩阵乘法反量化算子设计文档", 1.2 / 2.2:
  C_i32 = A x B + bias, D = fp16(fp32(C_i32) * scale).
* ``*_at`` -- the same definitions evaluated at chosen output points.
* ``collective_matmul_ring`` -- "Collective matrix multiplication",
  算法概述：Ring All-Gather: rank d's column shard of C, built in the ring's
  step order from the one-shard definition (index bookkeeping only).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
ERR_ARGS = -1
ERR_INT32_RANGE = -2


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, -O2, no SIMD intrinsics)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, u16p = ctypes.c_int64, ctypes.POINTER(ctypes.c_uint16)
        vpp = ctypes.POINTER(ctypes.c_void_p)
        dp, fp = ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_float)
        i32p, i64p = ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)
        i8p = ctypes.POINTER(ctypes.c_int8)
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f64.restype = ctypes.c_double
        lib.oracle_f64_to_f16_rn.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_f16_rn.restype = ctypes.c_uint16
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_f64_to_bf16_rn.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_bf16_rn.restype = ctypes.c_uint16
        lib.oracle_f64_to_f32_rn.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_f32_rn.restype = ctypes.c_float
        lib.oracle_allgather.argtypes = [ctypes.c_int, i64, i64, ctypes.c_size_t,
                                         vpp, ctypes.c_void_p]
        lib.oracle_ag_gemm_f16.argtypes = [ctypes.c_int, i64, i64, i64, vpp,
                                           u16p, dp]
        lib.oracle_ag_gemm_f16_at.argtypes = [ctypes.c_int, i64, i64, i64, vpp,
                                              u16p, i64, i64p, i64p, dp]
        lib.oracle_ag_gemm_bf16.argtypes = [ctypes.c_int, i64, i64, i64, vpp,
                                            u16p, dp]
        lib.oracle_ag_gemm_bf16_at.argtypes = [ctypes.c_int, i64, i64, i64, vpp,
                                               u16p, i64, i64p, i64p, dp]
        lib.oracle_ag_gemm_dequant.argtypes = [ctypes.c_int, i64, i64, i64, vpp,
                                               i8p, i32p, fp, i32p, u16p]
        lib.oracle_ag_gemm_dequant_at.argtypes = [ctypes.c_int, i64, i64, i64,
                                                  vpp, i8p, i32p, fp, i64,
                                                  i64p, i64p, i32p, u16p]
        lib.oracle_dequant.argtypes = [i64, i32p, fp, u16p]
        lib.oracle_f64_to_f16_rn_array.argtypes = [i64, dp, u16p]
        lib.oracle_f16_to_f64_array.argtypes = [i64, u16p, dp]
        lib.oracle_f64_to_f32_rn_array.argtypes = [i64, dp, fp]
        lib.oracle_f64_to_bf16_rn_array.argtypes = [i64, dp, u16p]
        lib.oracle_bf16_to_f64_array.argtypes = [i64, u16p, dp]
        for name in ("oracle_allgather", "oracle_ag_gemm_f16",
                     "oracle_ag_gemm_f16_at", "oracle_ag_gemm_dequant",
                     "oracle_ag_gemm_dequant_at", "oracle_dequant",
                     "oracle_ag_gemm_bf16", "oracle_ag_gemm_bf16_at"):
            getattr(lib, name).restype = ctypes.c_int
        for name in ("oracle_f64_to_f16_rn_array", "oracle_f16_to_f64_array",
                     "oracle_f64_to_f32_rn_array", "oracle_f64_to_bf16_rn_array",
                     "oracle_bf16_to_f64_array"):
            getattr(lib, name).restype = None
        _lib = lib
        return lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _shard_array(shards, dtype):
    arrs = [np.ascontiguousarray(s, dtype=dtype) for s in shards]
    if not arrs:
        raise OracleError("need at least one shard")
    R, K = arrs[0].shape
    for a in arrs:
        if a.shape != (R, K):
            raise OracleError("all shards must have the same shape")
    ptrs = (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
    return arrs, ptrs, R, K


def _check(rc, what):
    if rc == ERR_INT32_RANGE:
        raise OracleError(f"{what}: an output left the int32 range")
    if rc != OK:
        raise OracleError(f"{what}: error {rc}")


# -- IEEE conversions -------------------------------------------------------

def f64_to_f16_bits(x) -> np.ndarray:
    """binary16 round-to-nearest-even of float64 values -> uint16 bit patterns."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    lib.oracle_f64_to_f16_rn_array(x.size, _ptr(x, ctypes.c_double),
                                   _ptr(out, ctypes.c_uint16))
    return out


def f16_bits_to_f64(h) -> np.ndarray:
    lib = _load()
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float64)
    lib.oracle_f16_to_f64_array(h.size, _ptr(h, ctypes.c_uint16),
                                _ptr(out, ctypes.c_double))
    return out


def f64_to_bf16_bits(x) -> np.ndarray:
    """bfloat16 round-to-nearest-even of float64 values -> uint16 bit patterns."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    lib.oracle_f64_to_bf16_rn_array(x.size, _ptr(x, ctypes.c_double),
                                    _ptr(out, ctypes.c_uint16))
    return out


def bf16_bits_to_f64(h) -> np.ndarray:
    lib = _load()
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float64)
    lib.oracle_bf16_to_f64_array(h.size, _ptr(h, ctypes.c_uint16),
                                 _ptr(out, ctypes.c_double))
    return out


def f64_to_f32(x) -> np.ndarray:
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.float32)
    lib.oracle_f64_to_f32_rn_array(x.size, _ptr(x, ctypes.c_double),
                                   _ptr(out, ctypes.c_float))
    return out


# -- AllGather + GEMM ---------------------------------------------------------

def allgather(shards) -> np.ndarray:
    """Rows of the shards concatenated in rank order (as the pages' golden)."""
    lib = _load()
    first = np.asarray(shards[0])
    arrs, ptrs, R, K = _shard_array(shards, first.dtype)
    out = np.empty((len(arrs) * R, K), dtype=first.dtype)
    _check(lib.oracle_allgather(len(arrs), R, K, first.dtype.itemsize, ptrs,
                                out.ctypes.data), "allgather")
    return out


def ag_gemm_f16(shards, B) -> np.ndarray:
    """fp64 C = AllGather(shards) x B.  shards: list of R x K float16 arrays."""
    lib = _load()
    arrs, ptrs, R, K = _shard_array([np.asarray(s, np.float16).view(np.uint16)
                                     for s in shards], np.uint16)
    Bh = np.ascontiguousarray(np.asarray(B, np.float16).view(np.uint16))
    if Bh.shape[0] != K:
        raise OracleError("B must be K x N")
    N = Bh.shape[1]
    C = np.empty((len(arrs) * R, N), dtype=np.float64)
    _check(lib.oracle_ag_gemm_f16(len(arrs), R, K, N, ptrs,
                                  _ptr(Bh, ctypes.c_uint16),
                                  _ptr(C, ctypes.c_double)), "ag_gemm_f16")
    return C


def ag_gemm_f16_at(shards, B, rows, cols) -> np.ndarray:
    """fp64 C[rows[i], cols[i]] of AllGather(shards) x B."""
    lib = _load()
    arrs, ptrs, R, K = _shard_array([np.asarray(s, np.float16).view(np.uint16)
                                     for s in shards], np.uint16)
    Bh = np.ascontiguousarray(np.asarray(B, np.float16).view(np.uint16))
    N = Bh.shape[1]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    out = np.empty(rows.shape, dtype=np.float64)
    _check(lib.oracle_ag_gemm_f16_at(len(arrs), R, K, N, ptrs,
                                     _ptr(Bh, ctypes.c_uint16), rows.size,
                                     _ptr(rows, ctypes.c_int64),
                                     _ptr(cols, ctypes.c_int64),
                                     _ptr(out, ctypes.c_double)),
           "ag_gemm_f16_at")
    return out


def ag_gemm_dequant(shards, B, bias, scale):
    """(C_i32, D_f16) of the int8 AllGatherMatmulDequant definition."""
    lib = _load()
    arrs, ptrs, R, K = _shard_array(shards, np.int8)
    B8 = np.ascontiguousarray(B, dtype=np.int8)
    N = B8.shape[1]
    bias = np.ascontiguousarray(bias, dtype=np.int32)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    C = np.empty((len(arrs) * R, N), dtype=np.int32)
    D = np.empty((len(arrs) * R, N), dtype=np.uint16)
    _check(lib.oracle_ag_gemm_dequant(len(arrs), R, K, N, ptrs,
                                      _ptr(B8, ctypes.c_int8),
                                      _ptr(bias, ctypes.c_int32),
                                      _ptr(scale, ctypes.c_float),
                                      _ptr(C, ctypes.c_int32),
                                      _ptr(D, ctypes.c_uint16)),
           "ag_gemm_dequant")
    return C, D.view(np.float16)


def ag_gemm_dequant_at(shards, B, bias, scale, rows, cols):
    lib = _load()
    arrs, ptrs, R, K = _shard_array(shards, np.int8)
    B8 = np.ascontiguousarray(B, dtype=np.int8)
    N = B8.shape[1]
    bias = np.ascontiguousarray(bias, dtype=np.int32)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    C = np.empty(rows.shape, dtype=np.int32)
    D = np.empty(rows.shape, dtype=np.uint16)
    _check(lib.oracle_ag_gemm_dequant_at(len(arrs), R, K, N, ptrs,
                                         _ptr(B8, ctypes.c_int8),
                                         _ptr(bias, ctypes.c_int32),
                                         _ptr(scale, ctypes.c_float),
                                         rows.size, _ptr(rows, ctypes.c_int64),
                                         _ptr(cols, ctypes.c_int64),
                                         _ptr(C, ctypes.c_int32),
                                         _ptr(D, ctypes.c_uint16)),
           "ag_gemm_dequant_at")
    return C, D.view(np.float16)


def dequant(c, scale) -> np.ndarray:
    """Element-wise fp16(fp32(c) * scale) for int32 c and fp32 scale."""
    lib = _load()
    c = np.ascontiguousarray(c, dtype=np.int32)
    scale = np.ascontiguousarray(np.broadcast_to(scale, c.shape), dtype=np.float32)
    out = np.empty(c.shape, dtype=np.uint16)
    _check(lib.oracle_dequant(c.size, _ptr(c, ctypes.c_int32),
                              _ptr(scale, ctypes.c_float),
                              _ptr(out, ctypes.c_uint16)), "dequant")
    return out.view(np.float16)


# -- bf16 AllGather + GEMM ------------------------------------------------------
# numpy has no bfloat16: shards and B are uint16 arrays of bfloat16 bit patterns.

def ag_gemm_bf16(shards, B) -> np.ndarray:
    """fp64 C = AllGather(shards) x B for bfloat16 bit patterns (uint16 arrays)."""
    lib = _load()
    arrs, ptrs, R, K = _shard_array(shards, np.uint16)
    Bh = np.ascontiguousarray(B, dtype=np.uint16)
    if Bh.shape[0] != K:
        raise OracleError("B must be K x N")
    N = Bh.shape[1]
    C = np.empty((len(arrs) * R, N), dtype=np.float64)
    _check(lib.oracle_ag_gemm_bf16(len(arrs), R, K, N, ptrs,
                                   _ptr(Bh, ctypes.c_uint16),
                                   _ptr(C, ctypes.c_double)), "ag_gemm_bf16")
    return C


def ag_gemm_bf16_at(shards, B, rows, cols) -> np.ndarray:
    """fp64 C[rows[i], cols[i]] of AllGather(shards) x B, bfloat16 bit patterns."""
    lib = _load()
    arrs, ptrs, R, K = _shard_array(shards, np.uint16)
    Bh = np.ascontiguousarray(B, dtype=np.uint16)
    N = Bh.shape[1]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    out = np.empty(rows.shape, dtype=np.float64)
    _check(lib.oracle_ag_gemm_bf16_at(len(arrs), R, K, N, ptrs,
                                      _ptr(Bh, ctypes.c_uint16), rows.size,
                                      _ptr(rows, ctypes.c_int64),
                                      _ptr(cols, ctypes.c_int64),
                                      _ptr(out, ctypes.c_double)),
           "ag_gemm_bf16_at")
    return out


# -- N-sharded collective matmul (ring order) -----------------------------------

def collective_matmul_ring(shards, B_d, d, dtype="f16") -> np.ndarray:
    """Rank d's output of the ring collective matmul: AllGather(shards) x B_d.

    "Collective matrix multiplication", 算法概述：Ring All-Gather: with D ranks,
    at step i (0 <= i < D) rank d holds shard A_{(d + i) % D}, multiplies it by
    its own column shard B_d and writes the product into the output's row
    slice (d + i) % D.  Each step is the one-shard definition (ag_gemm_f16 or
    ag_gemm_bf16 with a single shard); this function only places the slices.
    """
    D = len(shards)
    R = np.asarray(shards[0]).shape[0]
    one = ag_gemm_f16 if dtype == "f16" else ag_gemm_bf16
    out = None
    for i in range(D):
        src = (d + i) % D
        part = one([shards[src]], B_d)
        if out is None:
            out = np.empty((D * R, part.shape[1]), dtype=np.float64)
        out[src * R:(src + 1) * R] = part
    return out
