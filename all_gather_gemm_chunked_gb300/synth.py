"""Seeded synthetic inputs for the streamed AllGather+GEMM workloads.

This module only draws random numbers; it holds none of the method's
arithmetic, and both the CUDA path and the CPU oracle consume what it makes.

Distributions follow the workloads the pages describe:

* fp16 path: A and B ~ N(0, 1) rounded to fp16 (the Pallas collective-matmul
  page draws ``jax.random.normal`` operands; the Triton-distributed tutorial
  draws ``torch.randn`` fp16 operands).
* bf16 path: the same N(0, 1) operands rounded to bfloat16 (the Pallas
  collective-matmul page's default dtype), as uint16 bit patterns (numpy has
  no bfloat16 type).
* int8 path ("AllGather矩阵乘法反量化算子设计文档", 1.3 and 8.3): A, B uniform
  int8 on [-127, 127] (symmetric quantisation), bias uniform int32 on
  [-1000, 1000], per-channel scale uniform fp32 on [1e-5, 1e-4].

Each shard is an independent array, so shards behave like separate ranks'
buffers.  Seeds: ``0xA66E0000 + workload id``, then a fixed offset per tensor.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np

SEED_BASE = 0xA66E0000
OFF_B, OFF_BIAS, OFF_SCALE = 100, 200, 300


@dataclass(frozen=True)
class Workload:
    """One AllGather+GEMM problem: S shards of R rows, K, N, dtype, chunking."""
    wid: int
    name: str
    S: int
    M: int
    K: int
    N: int
    dtype: str           # "f16", "bf16" or "i8"
    chunk_rows: int      # 0 = chosen by the library (64..128 chunks per source)
    n_blocks: int = 1    # N-sharded layout: B and C have n_blocks * N columns and the
                         # problem is rank `rank`'s column block (ring order from `rank`)
    rank: int = 0
    staging_slots: Optional[int] = None  # bounded staging window (256-row slots), None = plain

    @property
    def R(self) -> int:
        return self.M // self.S

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


# The five workloads: a small parity case, two compute-bound fp16 cases, a
# compute-bound int8 dequant case and a memory-bound skinny int8 case; 6 is the
# 4096^3 fp16 case with bfloat16 operands; 7 is one rank of the N-sharded
# collective matmul with the per-device shape of "Collective matrix
# multiplication" (2 devices, 1024 rows per shard, K = 4096, 4096 columns of B
# per device): rank 0's column block of B (K x 8192) and C.  8 and 9 are
# workloads 4 and 3 with the remote rows staged through a bounded window of 16
# slots of 256 rows (two swizzle groups) instead of one place per remote row.
WORKLOADS = {
    1: Workload(1, "f16 2x128 rows, K=256, N=128, chunk 16", 2, 256, 256, 128, "f16", 16),
    2: Workload(2, "f16 2x2048 rows, K=4096, N=4096", 2, 4096, 4096, 4096, "f16", 0),
    3: Workload(3, "f16 8x1024 rows, K=4096, N=4096", 8, 8192, 4096, 4096, "f16", 0),
    4: Workload(4, "i8 dequant 4x4096 rows, K=27392, N=4096", 4, 16384, 27392, 4096, "i8", 0),
    5: Workload(5, "i8 dequant skinny 2x32 rows, K=16384, N=7168", 2, 64, 16384, 7168, "i8", 0),
    6: Workload(6, "bf16 2x2048 rows, K=4096, N=4096", 2, 4096, 4096, 4096, "bf16", 0),
    7: Workload(7, "f16 N-sharded rank 0 of 2: 2x1024 rows, K=4096, 4096 of 8192 columns",
                2, 2048, 4096, 4096, "f16", 0, n_blocks=2, rank=0),
    8: Workload(8, "i8 dequant 4x4096 rows, K=27392, N=4096, staging window 16 x 256 rows",
                4, 16384, 27392, 4096, "i8", 0, staging_slots=16),
    9: Workload(9, "f16 8x1024 rows, K=4096, N=4096, staging window 16 x 256 rows",
                8, 8192, 4096, 4096, "f16", 0, staging_slots=16),
}


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def normal_f16(seed: int, shape) -> np.ndarray:
    """N(0,1) samples rounded to float16 (numpy's round-to-nearest cast)."""
    return _rng(seed).standard_normal(shape, dtype=np.float64).astype(np.float16)


def normal_bf16_bits(seed: int, shape) -> np.ndarray:
    """N(0,1) samples rounded to bfloat16 (nearest, ties to even), as bit patterns:
    cast to float32, then round the upper 16 bits of the float32 pattern."""
    x = _rng(seed).standard_normal(shape, dtype=np.float64).astype(np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def uniform_i8(seed: int, shape, lo: int = -127, hi: int = 127) -> np.ndarray:
    return _rng(seed).integers(lo, hi + 1, size=shape, dtype=np.int8)


def uniform_i32(seed: int, shape, lo: int = -1000, hi: int = 1000) -> np.ndarray:
    return _rng(seed).integers(lo, hi + 1, size=shape, dtype=np.int32)


def uniform_f32(seed: int, shape, lo: float = 1e-5, hi: float = 1e-4) -> np.ndarray:
    return _rng(seed).uniform(lo, hi, size=shape).astype(np.float32)


def make_inputs(S: int, R: int, K: int, N: int, dtype: str, seed: int):
    """Return dict(shards=[S arrays R x K], B=K x N, bias, scale) on the host."""
    if dtype == "f16":
        shards = [normal_f16(seed + s, (R, K)) for s in range(S)]
        B = normal_f16(seed + OFF_B, (K, N))
        return {"shards": shards, "B": B, "bias": None, "scale": None}
    if dtype == "bf16":
        shards = [normal_bf16_bits(seed + s, (R, K)) for s in range(S)]
        B = normal_bf16_bits(seed + OFF_B, (K, N))
        return {"shards": shards, "B": B, "bias": None, "scale": None}
    if dtype == "i8":
        shards = [uniform_i8(seed + s, (R, K)) for s in range(S)]
        B = uniform_i8(seed + OFF_B, (K, N))
        bias = uniform_i32(seed + OFF_BIAS, (N,))
        scale = uniform_f32(seed + OFF_SCALE, (N,))
        return {"shards": shards, "B": B, "bias": bias, "scale": scale}
    raise ValueError(f"unknown dtype {dtype!r}")


def workload_inputs(w: Workload):
    """Inputs of a workload; for an N-sharded one, B is the full K x (n_blocks * N)
    matrix and ``B_rank`` the rank's column block (a view)."""
    x = make_inputs(w.S, w.R, w.K, w.N * w.n_blocks, w.dtype, SEED_BASE + w.wid)
    x["B_rank"] = x["B"][:, w.rank * w.N:(w.rank + 1) * w.N]
    return x
