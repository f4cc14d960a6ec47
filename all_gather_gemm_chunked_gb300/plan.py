"""Torch-tensor front end of the C ABI: checks tensors and passes their device
pointers and the current CUDA stream to libaggemm.so.  No arithmetic here."""
from __future__ import annotations

import torch

from . import binding as B_

_DTYPES = {"f16": B_.F16, "i8": B_.I8, "bf16": B_.BF16}
_TORCH_2B = {"f16": torch.float16, "bf16": torch.bfloat16}


def _stream_handle(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _check(t: torch.Tensor, name: str, dtype, shape, pitched: bool = False) -> int:
    """Validate a device matrix; returns its row pitch in elements.  With
    `pitched`, a column block of a wider row-major matrix (unit column stride)
    is accepted as well as a contiguous matrix."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.is_contiguous():
        return int(shape[-1]) if len(shape) > 1 else 1
    if pitched and t.dim() == 2 and t.stride(1) == 1 and t.stride(0) >= t.shape[1]:
        return int(t.stride(0))
    raise ValueError(f"{name} must be contiguous" +
                     (" or a column block of a row-major matrix" if pitched else ""))


class Plan:
    """One AllGather+GEMM problem: owns the library plan (staging, counters)."""

    def __init__(self, n_shards: int, M: int, K: int, N: int, dtype: str = "f16",
                 chunk_rows: int = 0, staging_slots=None):
        """staging_slots: None = every remote row staged (ag_gemm_plan_create);
        an int = a bounded staging window of that many 256-row slots, 0 = the
        default window (ag_gemm_plan_create_bounded)."""
        if dtype not in _DTYPES:
            raise ValueError("dtype must be 'f16', 'bf16' or 'i8'")
        self.n_shards, self.M, self.K, self.N, self.dtype = n_shards, M, K, N, dtype
        self.R = M // n_shards if n_shards else 0
        if staging_slots is None:
            self.handle = B_.ag_gemm_plan_create(n_shards, M, K, N, _DTYPES[dtype], chunk_rows)
        else:
            self.handle = B_.ag_gemm_plan_create_bounded(n_shards, M, K, N, _DTYPES[dtype],
                                                         chunk_rows, int(staging_slots))

    # -- lifecycle
    def close(self):
        if getattr(self, "handle", None):
            B_.ag_gemm_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # -- knobs
    @property
    def geometry(self) -> dict:
        return B_.ag_gemm_plan_geometry(self.handle).as_dict()

    @property
    def chunk_rows(self) -> int:
        return B_.ag_gemm_plan_chunk_rows(self.handle)

    @property
    def grid(self) -> int:
        return B_.ag_gemm_plan_grid(self.handle)

    @property
    def path(self) -> int:
        """binding.PATH_FUSED_F16, PATH_FUSED_I8 or PATH_SKINNY_I8."""
        return B_.ag_gemm_plan_path(self.handle)

    def set_mode(self, mode: int):
        B_.ag_gemm_plan_set_mode(self.handle, mode)

    def set_local_rank(self, r: int):
        B_.ag_gemm_plan_set_local_rank(self.handle, r)

    def set_timeout_ns(self, ns: int):
        B_.ag_gemm_plan_set_timeout_ns(self.handle, ns)

    def set_grid(self, ctas: int):
        """CTAs of the fused kernel (0 = one per SM, the default; even otherwise)."""
        B_.ag_gemm_plan_set_grid(self.handle, ctas)

    def set_debug(self, flags: int, arg: int = 0):
        B_.ag_gemm_plan_set_debug(self.handle, flags, arg)

    def set_trace(self, capacity: int):
        """Record an event trace of every later run (capacity events; 0 = off)."""
        self.trace_capacity = int(capacity)
        B_.ag_gemm_plan_set_trace(self.handle, self.trace_capacity)

    def trace(self):
        """(events the last run recorded, numpy structured array of the kept events)."""
        return B_.ag_gemm_plan_trace(self.handle, getattr(self, "trace_capacity", 0))

    def status(self) -> int:
        return B_.ag_gemm_plan_status(self.handle)

    def status_word(self) -> int:
        return B_.ag_gemm_plan_status_word(self.handle)

    def reset(self, stream=None):
        B_.ag_gemm_plan_reset(self.handle, _stream_handle(stream))

    # -- runs
    def run(self, shards, B, C=None, stream=None) -> torch.Tensor:
        """C (M x N fp32) = AllGather(shards) x B for fp16 (bf16 plans: bfloat16)
        shards (R x K) and B (K x N).  B and C may be column blocks of wider
        row-major matrices (the N-sharded layout: rank d passes B[:, block d]
        and C[:, block d]); they then go through ag_gemm_run_ld."""
        if self.dtype not in _TORCH_2B:
            raise ValueError("run() needs an f16 or bf16 plan")
        if len(shards) != self.n_shards:
            raise ValueError(f"expected {self.n_shards} shards")
        tdt = _TORCH_2B[self.dtype]
        for i, s in enumerate(shards):
            _check(s, f"shards[{i}]", tdt, (self.R, self.K))
        ldb = _check(B, "B", tdt, (self.K, self.N), pitched=True)
        if C is None:
            C = torch.empty((self.M, self.N), dtype=torch.float32, device=B.device)
        ldc = _check(C, "C", torch.float32, (self.M, self.N), pitched=True)
        ptrs = [s.data_ptr() for s in shards]
        if ldb == self.N and ldc == self.N:
            B_.ag_gemm_run(self.handle, ptrs, B.data_ptr(), C.data_ptr(), _stream_handle(stream))
        else:
            B_.ag_gemm_run_ld(self.handle, ptrs, B.data_ptr(), ldb, C.data_ptr(), ldc,
                              _stream_handle(stream))
        return C

    def dequant_run(self, shards, B, bias, scale, C_i32=None, D=None, stream=None):
        """(C_i32, D) of the int8 AllGatherMatmulDequant for int8 shards and B."""
        if self.dtype != "i8":
            raise ValueError("dequant_run() needs an i8 plan")
        if len(shards) != self.n_shards:
            raise ValueError(f"expected {self.n_shards} shards")
        for i, s in enumerate(shards):
            _check(s, f"shards[{i}]", torch.int8, (self.R, self.K))
        _check(B, "B", torch.int8, (self.K, self.N))
        _check(bias, "bias", torch.int32, (self.N,))
        _check(scale, "scale", torch.float32, (self.N,))
        if C_i32 is None:
            C_i32 = torch.empty((self.M, self.N), dtype=torch.int32, device=B.device)
        if D is None:
            D = torch.empty((self.M, self.N), dtype=torch.float16, device=B.device)
        _check(C_i32, "C_i32", torch.int32, (self.M, self.N))
        _check(D, "D", torch.float16, (self.M, self.N))
        B_.ag_gemm_dequant_run(self.handle, [s.data_ptr() for s in shards], B.data_ptr(),
                               bias.data_ptr(), scale.data_ptr(), C_i32.data_ptr(), D.data_ptr(),
                               _stream_handle(stream))
        return C_i32, D
