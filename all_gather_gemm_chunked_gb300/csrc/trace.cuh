// trace.cuh -- opt-in per-run event trace of the streamed kernels: when a
// chunk (or chunk part) landed, when a tile (or unit) started and stopped
// waiting for its remote rows, and a few pipeline milestones, each stamped
// with the GPU's global nanosecond timer.  It exists to show the overlap of
// communication and compute that the method is about, the counterpart of the
// overlap analysis the PTO example ships ("AllGather + GEMM 通算融合算子示例",
// 目录结构: prof_analysis).
//
// The kernels take a trace only in their trace-enabled instantiation (a
// template flag), so the untraced kernels carry no trace code at all.
#pragma once

#include <stdint.h>

#include "sm103.cuh"

namespace agg {

// One event; the layout of ag_gemm_trace_event in include/ag_gemm.h.
struct TraceEvent {
  uint64_t t_ns;   // %globaltimer when the event happened
  uint32_t kind;   // ag_gemm_trace_kind
  uint32_t cta;    // blockIdx.x
  uint32_t warp;   // warp index within the CTA
  uint32_t id;     // meaning per kind (tile, unit, counter index, ...)
  uint64_t aux;    // meaning per kind (item or task index, chunk range, part, ...)
};
static_assert(sizeof(TraceEvent) == 32, "trace event layout");

enum : uint32_t {
  kTrCtaStart = 1,
  kTrCtaEnd = 2,
  kTrLanded = 3,     // a copy item / task is in the staging (recorded before its release)
  kTrWaitStart = 4,  // the TMA warp starts waiting for remote rows
  kTrWaitEnd = 5,    // ... and has acquired them
  kTrTileDone = 6,   // fused: an epilogue warp issued its last store of a tile
  kTrUnitIssued = 7, // skinny: the TMA warp issued a unit's loads
  kTrUnitLanded = 8, // skinny: a unit's raw stage is complete (seen by the B-widening warps)
  kTrKbWidened = 9,  // skinny: one k-block of B widened into an fp16 stage
  kTrKbMma = 10,     // skinny: the MMAs of one k-block issued and committed
  kTrPieceDone = 11, // skinny: a piece's int32 sums stored to its workspace slot
  kTrCopyStart = 12, // a copy warp starts a copy item / task (before its loads)
  kTrAccReady = 13,  // fused: the accumulator of a work item's last segment is ready
  kTrPartsReady = 14,// fused split tile: int8, its last part saw every earlier part stored;
                     // fp16 / bf16, a part saw the run's zeroing done
};

// The buffer is cut into one region per (CTA, warp slot): 32 slots per CTA,
// slot = the emitting warp, or kTrCtaSlot for the CTA-wide events of thread 0.
// Each emitter keeps its own event count, so an event is one plain 32-byte
// store: no atomics that would stall the pipeline being observed.  The host
// clears the buffer before a traced run and keeps the slots whose time is
// non-zero; an emitter whose region is full counts the event as dropped.
constexpr uint32_t kTrSlots = 32;
constexpr uint32_t kTrCtaSlot = 31;

struct TraceBuf {
  TraceEvent* ev;                 // nullptr: tracing off
  unsigned long long* dropped;    // events that did not fit their region
  uint32_t per_slot;              // events per (CTA, slot) region
};

__device__ __forceinline__ void trace_emit(const TraceBuf& tb, uint32_t& n, uint32_t slot,
                                           uint32_t kind, uint32_t id, uint64_t aux) {
  if (n < tb.per_slot) {
    TraceEvent e;
    e.t_ns = globaltimer_ns();
    e.kind = kind;
    e.cta = blockIdx.x;
    e.warp = threadIdx.x >> 5;
    e.id = id;
    e.aux = aux;
    tb.ev[(static_cast<uint64_t>(blockIdx.x) * kTrSlots + slot) * tb.per_slot + n] = e;
  } else {
    atomicAdd(tb.dropped, 1ull);
  }
  ++n;
}

}  // namespace agg
