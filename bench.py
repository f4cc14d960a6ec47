"""Benchmark of the streamed AllGather+GEMM on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 4]
                    [--extra-workloads 2,3,5] [--impl ours|reference]

Metric: streamed gather+GEMM throughput 2*M*N*K / t in TFLOP/s (TOP/s for the
int8 workloads), where t is the device time of one run (PIPELINED mode: chunk
copies and GEMM concurrently in one persistent launch) on inputs already
resident in HBM.  The headline workload is the largest one: int8
AllGatherMatmulDequant, 4 shards of 4096 rows, K = 27392, N = 4096 (the first
test shape of "AllGather矩阵乘法反量化算子设计文档", 8.3).  The fp16 workloads
2 and 3 and the HBM-bound skinny int8 workload 5 are measured in the same call
and reported under "workloads", each with its own roofline.

L2 is flushed before every timed step, outside the timed events: a 512 MiB
buffer is written, then a second 512 MiB buffer is read, so that the written
lines are back in HBM and L2 holds no data of the run and no dirty lines whose
write-back would land in the timed step.  Each batch of timed steps is
enqueued behind a GPU spin, so the host has queued every event and launch of
the batch before the GPU reaches the first one (host latency never falls
inside a timed event).  One JSON line is printed by rank 0.

N > 1 (torchrun): every rank runs its own full replica of the workload on its
own GPU (the shards are simulated ranks inside one GPU, so nothing is
exchanged between GPUs); the step time is the max over ranks and `value` is
the whole-job throughput N * flops / t_max ("scaling": "weak").  The extra
workloads are measured at N = 1 only.

--impl reference times the CPU oracle (plain single-threaded C loops) on a
bounded sample of the same workload: a step is one sample of whole rows of C.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "streamed gather+GEMM TFLOPS/TOPS (2MNK/t), % of GB300 dense tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PROFILE_DIR = os.path.join(ROOT, "profiles")
_COMMON_SOURCES = ["all_gather_gemm_chunked_gb300/csrc/sm103.cuh",
                   "all_gather_gemm_chunked_gb300/csrc/fused_kernel.cuh",
                   "all_gather_gemm_chunked_gb300/csrc/schedule.h"]
# sources of the dominant kernel of each plan path (fused fp16, fused int8, skinny int8)
KERNEL_SOURCES = {
    0: ["all_gather_gemm_chunked_gb300/csrc/fused_kernel.cu"] + _COMMON_SOURCES,
    1: ["all_gather_gemm_chunked_gb300/csrc/fused_kernel.cu"] + _COMMON_SOURCES,
    2: ["all_gather_gemm_chunked_gb300/csrc/skinny_kernel.cu"] + _COMMON_SOURCES,
}


# ---------------------------------------------------------------------------
# distributed plumbing (also exercised on CPU with gloo by the tests)
# ---------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), ws, int(os.environ.get("LOCAL_RANK", "0"))


def reduce_max(value: float, device=None) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


def whole_job_value(units_per_rank: float, n_ranks: int, t_max_s: float, scale=1e-12) -> float:
    """Weak scaling: every rank does units_per_rank; the job takes the slowest rank's time."""
    return units_per_rank * n_ranks / t_max_s * scale


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_hash(path_id: int = 0) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[path_id]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload_id: int, path_id: int):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary,
    if it was taken on the current kernel sources (else None)."""
    path = os.path.join(PROFILE_DIR, f"traffic_workload{workload_id}.txt")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_sources_sha256_16\s*=\s*(\w+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch\s*=\s*([0-9.eE+]+)", text)
    if not (m_hash and m_bytes) or m_hash.group(1) != kernel_hash(path_id):
        return None
    return float(m_bytes.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def wait_ready(self, timeout_s: float = 5.0):
        """Return once nvidia-smi has written its first sample (its start-up can
        stall CUDA calls of this process for up to a second), or after timeout_s."""
        t0 = time.time()
        while self.proc is not None and time.time() - t0 < timeout_s:
            try:
                if os.path.getsize(self.path) > 0:
                    return
            except OSError:
                return
            time.sleep(0.05)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = max(smax, float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        finally:
            os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_model() -> str:
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part", "hardware")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------

def time_oracle(w, x, budget_s: float, row_block: int = 2):
    """Run the oracle on whole rows of C (all N columns) until `budget_s` passes."""
    import oracle
    oracle.build()
    rows_done, t0 = 0, time.perf_counter()
    cols = np.arange(w.N, dtype=np.int64)
    while True:
        rows = np.arange(rows_done, rows_done + row_block) % w.M
        rr = np.repeat(rows, w.N)
        cc = np.tile(cols, row_block)
        if w.dtype == "f16":
            oracle.ag_gemm_f16_at(x["shards"], x["B_rank"], rr, cc)
        elif w.dtype == "bf16":
            oracle.ag_gemm_bf16_at(x["shards"], x["B_rank"], rr, cc)
        else:
            oracle.ag_gemm_dequant_at(x["shards"], x["B_rank"], x["bias"], x["scale"], rr, cc)
        rows_done += row_block
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    ops = 2.0 * rows_done * w.N * w.K
    return ops / el * 1e-12, rows_done, el


_START_BARRIER = None


def _oracle_worker_init(barrier):
    global _START_BARRIER
    _START_BARRIER = barrier


def _oracle_rows_worker(task):
    """One process of the all-cores CPU figure (started with spawn): time the
    oracle on whole rows of C for `budget_s`, from row `row0` of one shard.
    Only that shard and B (plus bias and scale) are generated here, from the
    same seeded streams as the workload; the rows' arithmetic is the same as
    in the full problem (the oracle over the one-shard list)."""
    wid, row0, budget_s = task
    import oracle
    from all_gather_gemm_chunked_gb300 import synth
    w = synth.WORKLOADS[wid]
    seed = synth.SEED_BASE + w.wid
    s = (row0 // w.R) % w.S
    gen = {"f16": synth.normal_f16, "bf16": synth.normal_bf16_bits, "i8": synth.uniform_i8}[w.dtype]
    shard = gen(seed + s, (w.R, w.K))
    B = gen(seed + synth.OFF_B, (w.K, w.N * w.n_blocks))[:, w.rank * w.N:(w.rank + 1) * w.N]
    B = np.ascontiguousarray(B)
    if w.dtype == "i8":
        bias = synth.uniform_i32(seed + synth.OFF_BIAS, (w.N * w.n_blocks,))[:w.N]
        scale = synth.uniform_f32(seed + synth.OFF_SCALE, (w.N * w.n_blocks,))[:w.N]
    oracle.build()
    cols = np.arange(w.N, dtype=np.int64)
    r, rows_done = row0 % w.R, 0
    if _START_BARRIER is not None:
        try:  # every process starts its timed rows together
            _START_BARRIER.wait(timeout=300)
        except Exception:
            pass
    t0 = time.time()
    while True:
        rows = np.arange(r, r + 2) % w.R
        rr, cc = np.repeat(rows, w.N), np.tile(cols, 2)
        if w.dtype == "f16":
            oracle.ag_gemm_f16_at([shard], B, rr, cc)
        elif w.dtype == "bf16":
            oracle.ag_gemm_bf16_at([shard], B, rr, cc)
        else:
            oracle.ag_gemm_dequant_at([shard], B, bias, scale, rr, cc)
        rows_done += 2
        r += 2
        if time.time() - t0 >= budget_s:
            break
    return rows_done, t0, time.time()


def time_oracle_all_cores(w, budget_s: float):
    """The same oracle on every host core as separate processes (spawn), each on
    its own rows for `budget_s`: (value, rows, cores, wall seconds), or None."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    cores = max(1, int(cores or 1))
    tasks = [(w.wid, (i * w.M) // cores, budget_s) for i in range(cores)]
    ctx = mp.get_context("spawn")
    pool = ctx.Pool(cores, initializer=_oracle_worker_init, initargs=(ctx.Barrier(cores),))
    try:
        res = pool.map_async(_oracle_rows_worker, tasks).get(timeout=budget_s * 4 + 300)
        pool.close()
    except Exception:  # a failed or stuck worker costs the figure, never the bench line
        pool.terminate()
        return None
    finally:
        pool.join()
    rows = sum(r for r, _, _ in res)
    wall = max(t1 for _, _, t1 in res) - min(t0 for _, t0, _ in res)
    return 2.0 * rows * w.N * w.K / wall * 1e-12, rows, cores, wall


def run_reference(args, w, rank):
    if rank != 0:
        return 0
    from all_gather_gemm_chunked_gb300 import synth
    x = synth.workload_inputs(w)
    per_step_s, per_row_s = [], []
    rows_total = 0
    # one untimed warm-up sample, then K bounded samples; a step is one sample
    for i in range(args.warmup + args.steps):
        v, rows, el = time_oracle(w, x, budget_s=args.ref_step_seconds)
        if i >= args.warmup:
            per_step_s.append(el)
            per_row_s.append(el / rows)
            rows_total += rows
    s_per_row = float(np.mean(per_row_s))
    value = 2.0 * w.N * w.K / s_per_row * 1e-12
    unit = "TOP/s" if w.dtype == "i8" else "TFLOP/s"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": float(np.mean(per_step_s)) * 1e3,
        "ms_per_step_median": float(np.median(per_step_s)) * 1e3,
        "full_workload_ms_extrapolated": s_per_row * w.M * 1e3,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int64" if w.dtype == "i8" else "f64",
        "data": "synthetic", "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle",
                         "sample": f"{rows_total} whole rows of C over {args.steps} steps "
                                   f"(~{args.ref_step_seconds:.0f} s each); a step is one such "
                                   f"sample, full_workload_ms_extrapolated scales it to all "
                                   f"{w.M} rows",
                         "cpu": cpu_model()},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w, flush=True):
    cfg = {"workload": w.name, "n_shards": w.S, "M": w.M, "K": w.K, "N": w.N,
           "dtype": w.dtype, "chunk_rows": w.chunk_rows or "auto",
           "l2": ("flushed before each timed step (512 MiB written, then 512 MiB read)" if flush
                  else "NOT flushed (analysis run; inputs may be L2-resident)")}
    if w.staging_slots is not None:
        cfg["staging"] = (f"bounded window of {w.staging_slots} slots x 256 rows, producer "
                          f"back-pressure by per-slot credits")
    if w.n_blocks > 1:
        cfg["layout"] = (f"N-sharded: rank {w.rank} of {w.n_blocks} computes its column block of "
                         f"C (B and C column blocks, ldb = ldc = {w.n_blocks * w.N}), row slices "
                         f"in ring order from its own shard")
    return cfg


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def timed_events(torch, stream, dev, n, body, before=None, batch=64, gate_ms=20.0):
    """Device times (ms) of n calls of body(), each bracketed by CUDA events on
    `stream` and preceded, outside the events, by before().

    Every batch of up to `batch` steps is enqueued behind a GPU spin of
    `gate_ms`, so that the host has enqueued all events and launches of the
    batch before the GPU reaches the first of them: host latency (Python,
    ctypes, the clock sampler starting) cannot leave the GPU idle inside a
    timed event.  If the spin had already ended when the host finished
    enqueueing, the batch is timed again behind a longer spin."""
    times, late_batches, redone = [], 0, 0
    while len(times) < n:
        b = min(batch, n - len(times))
        for attempt in range(4):
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(b)]
            gate = torch.cuda.Event()
            torch.cuda._sleep(int(gate_ms * 2.1e6))  # ~gate_ms at <= 2.1 GHz SM clock
            gate.record(stream)
            t0 = time.perf_counter()
            for a, e in evs:
                if before is not None:
                    before()
                a.record(stream)
                body()
                e.record(stream)
            host_ms = (time.perf_counter() - t0) * 1e3
            late = gate.query()
            torch.cuda.synchronize(dev)
            if not late:
                break
            redone += 1
            gate_ms = max(2.0 * gate_ms, 2.0 * host_ms)
        else:
            late_batches += 1
        times += [a.elapsed_time(e) for a, e in evs]
    return times, {"batches_redone": redone, "batches_host_bound": late_batches,
                   "gate_ms": gate_ms}


class Runner:
    """One workload on one GPU: inputs resident in HBM, a plan, the run and
    (optionally) the end-to-end run from pinned host buffers."""

    def __init__(self, torch, w, dev, args, host=False):
        from all_gather_gemm_chunked_gb300 import synth
        from all_gather_gemm_chunked_gb300.plan import Plan
        self.torch, self.w, self.dev, self.args = torch, w, dev, args
        x = synth.workload_inputs(w)
        self.x = x
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
        h_shards = [pin(s) for s in x["shards"]]
        h_B = pin(x["B_rank"])  # this rank's B (its column block, for the N-sharded layout)
        if w.dtype == "bf16":  # bit patterns (numpy has no bfloat16) -> bfloat16 tensors
            h_shards = [t.view(torch.int16).view(torch.bfloat16) for t in h_shards]
            h_B = h_B.view(torch.int16).view(torch.bfloat16)
        self.shards = [t.to(dev) for t in h_shards]
        # B (and C below) at full width; the run takes the rank's column block
        cols = slice(w.rank * w.N, (w.rank + 1) * w.N)
        B_full = torch.empty((w.K, w.N * w.n_blocks), dtype=h_B.dtype, device=dev)
        self.Bd = B_full[:, cols]
        self.Bd.copy_(h_B)
        self.cols = cols
        self.int8 = w.dtype == "i8"
        if self.int8:
            h_bias, h_scale = pin(x["bias"]), pin(x["scale"])
            self.bias, self.scale = h_bias.to(dev), h_scale.to(dev)
            self.Ci = torch.empty((w.M, w.N), dtype=torch.int32, device=dev)
            self.D = torch.empty((w.M, w.N), dtype=torch.float16, device=dev)
        else:
            C_full = torch.empty((w.M, w.N * w.n_blocks), dtype=torch.float32, device=dev)
            self.C = C_full[:, cols]
        self.plan = Plan(w.S, w.M, w.K, w.N, w.dtype, w.chunk_rows, staging_slots=w.staging_slots)
        self.geometry = self.plan.geometry  # the plan's own sizes (staging window included)
        self.path = self.plan.path
        if w.rank:
            self.plan.set_local_rank(w.rank)
        self.stream = torch.cuda.current_stream(dev)
        self.host = host
        if host:
            self.h_shards, self.h_B = h_shards, h_B
            if self.int8:
                self.h_bias, self.h_scale = h_bias, h_scale
                self.h_Ci = torch.empty((w.M, w.N), dtype=torch.int32).pin_memory()
                self.h_D = torch.empty((w.M, w.N), dtype=torch.float16).pin_memory()
            else:
                self.h_C = torch.empty((w.M, w.N), dtype=torch.float32).pin_memory()

    def step(self):
        if self.int8:
            self.plan.dequant_run(self.shards, self.Bd, self.bias, self.scale, self.Ci, self.D)
        else:
            self.plan.run(self.shards, self.Bd, self.C)

    def e2e_step(self):
        for hs, ds in zip(self.h_shards, self.shards):
            ds.copy_(hs, non_blocking=True)
        self.Bd.copy_(self.h_B, non_blocking=True)
        if self.int8:
            self.bias.copy_(self.h_bias, non_blocking=True)
            self.scale.copy_(self.h_scale, non_blocking=True)
        self.step()
        if self.int8:
            self.h_Ci.copy_(self.Ci, non_blocking=True)
            self.h_D.copy_(self.D, non_blocking=True)
        else:
            self.h_C.copy_(self.C, non_blocking=True)

    # -- end to end, pipelined over steps ------------------------------------
    def _outputs(self):
        return [self.Ci, self.D] if self.int8 else [self.C]

    def _set_of(self, shards, Bd, outputs, extra=()):
        # extra: the int8 path's bias and scale (copied in every step as well)
        return {"shards": shards, "Bd": Bd, "out": outputs, "extra": list(extra)}

    def _second_set(self):
        """Device buffers for a second step in flight: the layout of the first
        (B and C as column blocks of full-width matrices for the N-sharded layout)."""
        torch, w, dev = self.torch, self.w, self.dev
        shards = [torch.empty_like(t) for t in self.shards]
        Bd = torch.empty((w.K, w.N * w.n_blocks), dtype=self.Bd.dtype, device=dev)[:, self.cols]
        extra = ()
        if self.int8:
            out = [torch.empty_like(self.Ci), torch.empty_like(self.D)]
            extra = (torch.empty_like(self.bias), torch.empty_like(self.scale))
        else:
            out = [torch.empty((w.M, w.N * w.n_blocks), dtype=torch.float32,
                               device=dev)[:, self.cols]]
        return self._set_of(shards, Bd, out, extra)

    def _run_set(self, st):
        if self.int8:
            self.plan.dequant_run(st["shards"], st["Bd"], *st["extra"], *st["out"])
        else:
            self.plan.run(st["shards"], st["Bd"], st["out"][0])

    def e2e_pipelined(self, n, gate_ms=20.0):
        """Milliseconds per step of n end-to-end steps with two steps' buffers:
        step i's host->device copies (on one stream) and step i-1's
        device->host copies (on another) run beside step i-1's or step i's
        run.  Every step still copies all of its inputs in and its outputs
        out inside the timed region; only the order of the engines overlaps.
        The runs stay on one stream, one at a time, as the plan requires."""
        torch, dev, main = self.torch, self.dev, self.stream
        if not hasattr(self, "_e2e"):
            extra = (self.bias, self.scale) if self.int8 else ()
            sets = [self._set_of(self.shards, self.Bd, self._outputs(), extra), self._second_set()]
            hosts = [[self.h_Ci, self.h_D] if self.int8 else [self.h_C],
                     [torch.empty_like(t).pin_memory() for t in
                      ([self.h_Ci, self.h_D] if self.int8 else [self.h_C])]]
            self._e2e = (sets, hosts, torch.cuda.Stream(dev), torch.cuda.Stream(dev))
        sets, hosts, s_in, s_out = self._e2e
        ev = lambda: torch.cuda.Event()  # noqa: E731
        ev_in, ev_run, ev_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for attempt in range(4):
            torch.cuda._sleep(int(gate_ms * 2.1e6))
            gate = torch.cuda.Event()
            gate.record(main)
            start.record(main)
            s_in.wait_event(start)
            s_out.wait_event(start)
            t0 = time.perf_counter()
            for i in range(n):
                b, st = i % 2, sets[i % 2]
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(ev_run[b])  # step i - 2 has read these inputs
                    for hs, ds in zip(self.h_shards, st["shards"]):
                        ds.copy_(hs, non_blocking=True)
                    st["Bd"].copy_(self.h_B, non_blocking=True)
                    if self.int8:
                        st["extra"][0].copy_(self.h_bias, non_blocking=True)
                        st["extra"][1].copy_(self.h_scale, non_blocking=True)
                    ev_in[b].record(s_in)
                main.wait_event(ev_in[b])
                if i >= 2:
                    main.wait_event(ev_out[b])  # step i - 2's outputs have been read back
                self._run_set(st)
                ev_run[b].record(main)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_run[b])
                    for ht, dt in zip(hosts[b], st["out"]):
                        ht.copy_(dt, non_blocking=True)
                    ev_out[b].record(s_out)
            for b in range(min(n, 2)):
                main.wait_event(ev_out[b])
            end.record(main)
            host_ms = (time.perf_counter() - t0) * 1e3
            late = gate.query()
            torch.cuda.synchronize(dev)
            if not late:
                break
            gate_ms = max(2.0 * gate_ms, 2.0 * host_ms)
        # every step computed the same inputs: the last step's host copy must
        # equal the other buffer set's device outputs bit for bit
        last = hosts[(n - 1) % 2]
        other = sets[n % 2]["out"]
        self.e2e_outputs_match = all(torch.equal(h, d.cpu()) for h, d in zip(last, other))
        return start.elapsed_time(end) / n

    def copies_only(self, n):
        """Milliseconds per step of one step's copies alone: its host->device
        copies and its device->host copies on their two streams at once, no
        run.  With the runs overlapped, this is the floor of the pipelined
        end-to-end step when the copies take longer than the run."""
        torch, dev, main = self.torch, self.dev, self.stream
        if not hasattr(self, "_e2e"):
            self.e2e_pipelined(1)
        sets, hosts, s_in, s_out = self._e2e
        st, ho = sets[0], hosts[0]
        ts = []
        for _ in range(n + 1):
            start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            start.record(main)
            s_in.wait_event(start)
            s_out.wait_event(start)
            with torch.cuda.stream(s_in):
                for hs, ds in zip(self.h_shards, st["shards"]):
                    ds.copy_(hs, non_blocking=True)
                st["Bd"].copy_(self.h_B, non_blocking=True)
                if self.int8:
                    st["extra"][0].copy_(self.h_bias, non_blocking=True)
                    st["extra"][1].copy_(self.h_scale, non_blocking=True)
            with torch.cuda.stream(s_out):
                for ht, dt in zip(ho, st["out"]):
                    ht.copy_(dt, non_blocking=True)
            main.wait_stream(s_in)
            main.wait_stream(s_out)
            end.record(main)
            torch.cuda.synchronize(dev)
            ts.append(start.elapsed_time(end))
        return float(np.median(ts[1:]))

    def e2e_bytes(self):
        h2d = (sum(t.numel() * t.element_size() for t in self.h_shards)
               + self.h_B.numel() * self.h_B.element_size())
        if self.int8:
            return h2d + self.h_bias.numel() * 4 + self.h_scale.numel() * 4, \
                self.h_Ci.numel() * 4 + self.h_D.numel() * 2
        return h2d, self.h_C.numel() * 4

    def timed(self, n, mode, flush, fn=None):
        from all_gather_gemm_chunked_gb300 import binding as B_
        self.plan.set_mode(mode)
        try:
            return timed_events(self.torch, self.stream, self.dev, n, fn or self.step, flush)
        finally:
            self.plan.set_mode(B_.MODE_PIPELINED)

    def warm(self, n):
        for _ in range(n):
            self.step()
        self.torch.cuda.synchronize(self.dev)
        if self.plan.status() != 0:
            raise RuntimeError(f"{self.w.name}: warm-up run failed: status "
                               f"{self.plan.status_word():#x}")

    def read_floor(self, n, flush):
        """Median device time (ms) of one library kernel that only reads B once
        (a PyTorch int64 sum over its bytes), each after the same L2 flush: what
        a single launch needs just to stream B from HBM, start-up included.  For
        the skinny int8 path, which is bound by reading B, it is the practical
        floor beside the copy-bandwidth roofline.  None if B is not contiguous."""
        torch = self.torch
        if not self.Bd.is_contiguous():
            return None
        flat = self.Bd.reshape(-1)
        src = flat.view(torch.int64) if flat.numel() % 8 == 0 else flat
        out = torch.empty((), dtype=torch.int64, device=self.dev)

        def body():
            torch.sum(src, dim=0, dtype=torch.int64, out=out)

        body()
        torch.cuda.synchronize(self.dev)
        return float(np.median(timed_events(torch, self.stream, self.dev, n, body, flush)[0]))

    def check_status(self, what):
        if self.plan.status() != 0:
            raise RuntimeError(f"{self.w.name}: {what} failed: status {self.plan.status_word():#x}")

    def modes(self, n, flush, t_pipe):
        from all_gather_gemm_chunked_gb300 import binding as B_
        t_compute = float(np.median(self.timed(n, B_.MODE_COMPUTE_ONLY, flush)[0]))
        t_copy = float(np.median(self.timed(n, B_.MODE_COPY_ONLY, flush)[0]))
        # a staging window cannot hold the whole gather: no SEQUENTIAL run
        t_seq = (float(np.median(self.timed(n, B_.MODE_SEQUENTIAL, flush)[0]))
                 if self.w.staging_slots is None else None)
        self.check_status("mode runs")
        overlap = (t_copy + t_compute - t_pipe) / max(min(t_copy, t_compute), 1e-9)
        return {"pipelined_ms": t_pipe, "compute_only_ms": t_compute, "copy_only_ms": t_copy,
                "sequential_ms": t_seq, "overlap_efficiency": overlap,
                "speedup_vs_sequential": t_seq / t_pipe if t_seq is not None else None}

    def close(self):
        self.plan.close()


def roofline_of(w, path_id, kernel_ms, clk, peaks, peak_src):
    """Roofline of one run's device time against the measured peak of its bound."""
    from all_gather_gemm_chunked_gb300 import binding as B_
    traffic = profiled_traffic(w.wid, path_id)
    if path_id == B_.PATH_SKINNY_I8:
        # bound by HBM: algorithmic bytes of one run = B once, the gathered rows
        # once, the remote shards copied (read + write), bias, scale, C_i32, D
        algo = (w.K * w.N + w.M * w.K + 2 * (w.S - 1) * w.R * w.K + 8 * w.N
                + 6 * w.M * w.N)
        peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        achieved = algo / (kernel_ms * 1e-3) * 1e-9
        return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic, "algorithmic_bytes": algo,
                "peak_source": f"{peak_src} HBM copy bandwidth",
                "kernel": "ag_skinny_kernel + ag_skinny_finish_kernel (one run)"}
    # a dense fp16 contraction: its peak is the measured dense bf16 figure
    # (fp16 and bf16 share the same nominal dense rate): the burst figure, or
    # the sustained one (cuBLAS back to back under the power cap) when the
    # clock samples of this timed region saw sw_power_cap
    capped = bool(clk) and "sw_power_cap" in (clk.get("reasons") or [])
    key = "bf16_tflops_sustained" if capped else "bf16_tflops"
    peak = float(peaks.get(key, FALLBACK_PEAKS[key]))
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    achieved = w.flops / (kernel_ms * 1e-3) * 1e-12
    int8 = w.dtype == "i8"
    r = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
         "frac": achieved / peak, "traffic": traffic,
         "peak_source": f"{peak_src} bf16 dense "
                        + ("sustained (the timed region ran under sw_power_cap)" if capped
                           else "burst")
                        + " (fp16 dense = bf16 dense nominal; int8 runs exactly on the fp16 "
                          "tensor path)",
         "kernel": "ag_fused_kernel" + ("<int8> + widen_kernel (one run)" if int8 else "<fp16>")}
    if capped:
        r["frac_of_burst"] = achieved / burst
    return r


def add_read_floor(roof, w, floor_ms, run_ms):
    """Record beside an HBM roofline the measured time of a bare read of B."""
    if floor_ms is None:
        return
    roof["read_floor_ms"] = floor_ms
    roof["read_floor_gbs"] = w.K * w.N / (floor_ms * 1e-3) * 1e-9
    roof["frac_of_read_floor"] = floor_ms / run_ms
    roof["read_floor_kernel"] = "torch.sum over B's bytes (one launch reading B once)"


def measure_extra(torch, w, dev, args, flush_fn, peaks, peak_src):
    """A compact record of one more workload, timed like the headline one."""
    r = Runner(torch, w, dev, args)
    try:
        r.warm(max(args.warmup, 3))
        from all_gather_gemm_chunked_gb300 import binding as B_
        steps = args.steps if args.steps is not None else 20
        times, gate = r.timed(steps, B_.MODE_PIPELINED, flush_fn)
        r.check_status("timed runs")
        mean_ms, med_ms = float(np.mean(times)), float(np.median(times))
        unit = "TOP/s" if w.dtype == "i8" else "TFLOP/s"
        roof = roofline_of(w, r.path, mean_ms, None, peaks, peak_src)
        if r.path == B_.PATH_SKINNY_I8:
            add_read_floor(roof, w, r.read_floor(steps, flush_fn), mean_ms)
        rec = {"workload": w.name, "value": w.flops / (mean_ms * 1e-3) * 1e-12, "unit": unit,
               "steps": steps, "ms_per_step": mean_ms, "ms_per_step_median": med_ms,
               "roofline": roof,
               "config": workload_config(w, flush_fn is not None), "enqueue": gate}
        if not args.no_modes:
            rec["modes"] = r.modes(max(3, min(steps, 10)), flush_fn, med_ms)
        return rec
    finally:
        r.close()


def run_ours(args, w, rank, world, local_rank):
    import torch

    from all_gather_gemm_chunked_gb300 import binding as B_
    from all_gather_gemm_chunked_gb300 import synth

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    r = Runner(torch, w, dev, args, host=True)
    flush_buf = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    flush_rd = torch.ones(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    flush_sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush():
        flush_buf.fill_(1.0)
        torch.sum(flush_rd, dim=0, out=flush_sink)

    flush_fn = None if args.no_flush else flush

    r.warm(max(args.warmup, 3))
    if args.steps is None:
        # size the timed region so that the clock sampler sees it for ~2 s
        est = float(np.median(r.timed(5, B_.MODE_PIPELINED, flush_fn)[0])) * 1e-3 + 1e-4
        args.steps = int(min(20000, max(20, np.ceil(2.0 / est))))
        args.steps = int(reduce_max(args.steps, dev))

    clocks = ClockSampler(local_rank)
    barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    clocks.wait_ready()
    times_ms, gate = r.timed(args.steps, B_.MODE_PIPELINED, flush_fn)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    barrier()
    r.check_status("timed runs")
    t_local = float(np.sum(times_ms)) / 1e3
    t_max = reduce_max(t_local, dev)
    ms_per_step = t_max / args.steps * 1e3          # the mean step (max over ranks)
    ms_median = reduce_max(float(np.median(times_ms)), dev)  # the median step (max over ranks)
    value = whole_job_value(w.flops * args.steps, world, t_max)

    # the other run modes (context: overlap of copy and GEMM)
    modes = {}
    if not args.no_modes:
        modes = r.modes(max(3, min(args.steps, 10)), flush_fn, float(np.median(times_ms)))

    # end to end through the C ABI with host buffers: every step copies its
    # inputs from pinned host memory and reads its outputs back
    ne = max(3, min(args.steps, 10))
    for _ in range(2):  # warm-up: the first DMA from or to a pinned buffer is slower
        r.e2e_step()
    torch.cuda.synchronize(dev)
    e2e_ms, _ = r.timed(ne, B_.MODE_PIPELINED, None, fn=r.e2e_step)
    r.check_status("end-to-end runs")
    e2e_serial_t = reduce_max(float(np.sum(e2e_ms)) / 1e3, dev)
    r.e2e_pipelined(2)  # warm-up: the second buffer set and the copy streams
    e2e_t = reduce_max(r.e2e_pipelined(ne) * ne / 1e3, dev)
    r.check_status("pipelined end-to-end runs")
    h2d, d2h = r.e2e_bytes()
    unit = "TOP/s" if r.int8 else "TFLOP/s"
    e2e = {"value": whole_job_value(w.flops * ne, world, e2e_t), "unit": unit,
           "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
           "steps": ne,
           "overlap": "two steps' buffers: step i's host->device copies and step i-1's "
                      "device->host copies run on their own streams beside the runs",
           "serial": {"value": whole_job_value(w.flops * ne, world, e2e_serial_t),
                      "unit": unit, "ms_per_step": e2e_serial_t * 1e3 / ne},
           "ms_per_step": e2e_t * 1e3 / ne,
           "copies_only_ms_per_step": r.copies_only(ne),
           "outputs_match": bool(r.e2e_outputs_match)}

    peaks, peak_src = load_peaks()
    path_id = r.path
    tensor_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    # kernels launched by one PIPELINED run: the fused kernel (fp16); the widening
    # kernel and the fused kernel (int8); the skinny and the finish kernel (skinny)
    launches_per_run = 1 if path_id == B_.PATH_FUSED_F16 else 2
    roofline = roofline_of(w, path_id, float(np.mean(times_ms)), clk, peaks, peak_src)
    if path_id == B_.PATH_SKINNY_I8:
        add_read_floor(roofline, w, r.read_floor(args.steps, flush_fn), float(np.mean(times_ms)))

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, rows, el = time_oracle(w, r.x, budget_s=args.cpu_seconds)
        cpu = {"value": v, "unit": unit, "cores": 1, "kind": "oracle",
               "sample": f"{rows} whole rows of C ({rows * w.N} outputs), {el:.1f} s",
               "cpu": cpu_model()}
        par = time_oracle_all_cores(w, args.cpu_seconds)
        if par is not None:
            pv, prow, pcores, pwall = par
            cpu["all_cores"] = {"value": pv, "unit": unit, "cores": pcores,
                                "sample": f"{prow} whole rows of C over {pcores} processes "
                                          f"(one per core, spawn), {pwall:.1f} s wall"}
    geometry = r.geometry
    r.close()
    del r

    # the other workloads of the suite, measured in the same call (rank 0 reports)
    extras = {}
    for wid in (args.extra_workloads if world == 1 else []):
        if wid == w.wid:
            continue
        extras[str(wid)] = measure_extra(torch, synth.WORKLOADS[wid], dev, args, flush_fn,
                                         peaks, peak_src)

    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step,
        "ms_per_step_median": ms_median,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "config": workload_config(w, not args.no_flush),
        "pct_of_peak": 100.0 * value / world / tensor_peak,
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
        "gpu_launches": launches_per_run * args.steps, "modes": modes,
        "enqueue": gate, "grid": geometry, "workloads": extras,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: enough for ~2 s of timed GPU work, >= 20)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=4, choices=list(range(1, 10)))
    ap.add_argument("--extra-workloads", default="2,3,5",
                    help="comma-separated workloads measured after the headline one in the same "
                         "call and reported under 'workloads' ('' for none)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-step-seconds", type=float, default=4.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-modes", action="store_true")
    ap.add_argument("--no-flush", action="store_true",
                    help="analysis only: keep inputs L2-resident between timed steps")
    args = ap.parse_args(argv)
    args.extra_workloads = [int(s) for s in args.extra_workloads.split(",") if s.strip()]
    for wid in args.extra_workloads:
        if wid not in range(1, 10):
            ap.error(f"unknown workload {wid} in --extra-workloads")

    from all_gather_gemm_chunked_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            if args.steps is None:
                args.steps = 10
            return run_reference(args, w, rank)
        return run_ours(args, w, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            if dist.is_initialized():
                dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
