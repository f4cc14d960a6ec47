// skinny_kernel.cu -- int8 AllGatherMatmulDequant when the gathered A has at
// most 128 rows (decode-like shapes such as 2 x 32 rows, K = 16384, N = 7168).
//
// Such a problem is bound by reading B from HBM once ("AllGather矩阵乘法反量化
// 算子设计文档", 8.3 lists the 64 x 16384 x 7168 shape): every k-block of B is
// shared by all rows, so the kernel streams B exactly once as int8, widens it
// in shared memory and runs the tensor core on it.  sm_103a has no tcgen05
// kind::i8, so the product is computed exactly on kind::f16: every int8 is an
// exact fp16, and an fp32 accumulation never spans more than 16 k-blocks
// (1024 k), which keeps every fp32 partial an integer below 2^24; segments are
// folded into an int32 sum in TMEM.
//
// The MMA computes the tile as it stands: the gathered rows are the M operand
// (M = 64 for up to 64 rows, else 128; K-major), 256 columns of the widened B
// are the N operand (MN-major).  On GB300 one tcgen05.mma of K = 16 occupies
// the tensor pipe for ~200 cycles at any shape up to 128 x 256, so the count
// of instructions, not their size, sets the rate: 64 x 256 per instruction is
// twice the work of the transposed 128-column x 64-row tile.  The fp32
// accumulator (256 TMEM columns) and the int32 running sums (256 more) fill
// TMEM, so the accumulator is single-buffered: at the end of each segment the
// MMA waits until the epilogue has folded it into the sums.
//
// A raw stage holds one k-block of one 256-column n-tile: 16 KB of B (two
// 128-column x 64-k-row halves, 128-byte swizzled), loaded with ONE TMA
// instruction through a 3D view of B (128 columns, K, N / 128) when N is a
// multiple of 128 -- a TMA instruction carries a fixed cost of several
// hundred cycles -- else as two 2D boxes; then the k-block's gathered rows
// (M x 64 int8, two more boxes: the local shard and all staged shards), so A
// arrives with B.  Five such stages let a stage be refilled as soon as its one
// k-block is widened.  The rows land in consumption order (local shard
// first), which the epilogue maps back to global rows.
//
// Work: the (256-column n-tile, 2-k-block unit) pairs, n-tile major, are cut
// into one contiguous range per CTA (stream-K), so a CTA holds at most a few
// pieces of n-tiles.  At the end of a piece its exact int32 sums (M rows x 256
// columns) go to a workspace slot of their own (plain stores, no atomics);
// ag_skinny_finish_kernel then adds the slots of each n-tile in a fixed order,
// adds the bias and writes C_i32 and the fp16 dequant D.  The workspace needs
// no clearing: every slot the finish kernel reads is written by the same run.
//
// Roles (20 warps).  The scheduler of warp w is w % 4; the MMA issue thread
// shares scheduler 0 only with warps that mostly sleep, and the widening work
// is spread over schedulers 1-3.  TMEM lane quadrant q is reachable only from
// warps w with w % 4 == q, hence the epilogue warps 16, 1, 2, 3.
//   warp 0                 MMA: one thread issues tcgen05.mma (M = 64 or 128,
//                          N = 256, K = 16).
//   warp 4                 TMA: streams the CTA's units into a raw ring, one
//                          k-block (B, then the row boxes) per stage; B and
//                          the local rows go out at once, the staged rows once
//                          the unit's k-part of every remote chunk has landed.
//   warps 8, 12            copy: remote chunks, one k-part at a time, into the
//                          int8 staging workspace; one ready counter per
//                          (k-part, chunk).
//   warps 16, 1, 2, 3      epilogue: fold fp32 segments into the int32 sums in
//                          TMEM; store each finished piece to its workspace slot.
//   warps 5-7, 9-11, 13,14 B widening: raw int8 B -> fp16 in the MN-major
//                          128-byte swizzled layout the MMA reads.
//   warps 15, 17, 18, 19   A widening: raw int8 rows -> fp16, K-major 128-byte
//                          swizzled, one k-block per fp16 stage.
// The raw ring's stages are released by both widening roles.

#include <cuda_fp16.h>

#include "fused_kernel.cuh"
#include "sm103.cuh"

namespace agg {

namespace {

constexpr int kSkWarps = 20;
constexpr int kSkThreads = kSkWarps * 32;
constexpr int kSkN = 256;              // n-tile (the MMA's N)
constexpr int kSkHalf = 128;           // columns of one B box
constexpr int kSkUnitBlocks = 2;       // k-blocks per unit (128 k-rows)
constexpr int kSkRawMax = 5;           // raw stages (one k-block of B + rows each), at most
constexpr int kSkFpMax = 3;            // fp16 stages (B + A, one k-block each), at most
constexpr int kSkBwThreads = 256;      // 8 B-widening warps
constexpr int kSkAwThreads = 128;      // 4 A-widening warps
constexpr int kSkBoxB = kSkHalf * kBlockK;     // 8 KB: 128 columns x 64 k-rows of int8 B
constexpr int kSkRawB = 2 * kSkBoxB;           // 16 KB int8 B per raw stage (one k-block)
constexpr int kSkARow = kBlockK;               // 64 bytes of a row per raw stage
constexpr int kSkFpB = kSkN * kBlockK * 2;                   // 32 KB: one fp16 k-block of B
// M <= 64: raw 5 x 21 KB, fp16 3 x (32 + 8) KB = 225 KB;
// M <= 128: raw 5 x 25 KB, fp16 2 x (32 + 16) KB = 221 KB.  (A raw stage is
// 16 KB of B, the rows and up to 128 bytes of padding, rounded up to 1 KB so
// that every stage's swizzled B boxes start 1024-byte aligned.)
constexpr int kSkDataBytes = 225 * 1024;
constexpr int kSkSmem = kSkDataBytes + 1024 /*alignment*/ + 256 /*barriers*/;
constexpr uint32_t kSkDcol = 0;        // TMEM columns [0, 256): the fp32 accumulator
constexpr uint32_t kSkScol = 256;      // [256, 512): int32 running sums

enum SkRole { kRoleMma, kRoleTma, kRoleCopy, kRoleEpi, kRoleBw, kRoleAw };

// role and rank within the role of warp w
__device__ __forceinline__ void sk_role(int w, int& role, int& rank) {
  rank = 0;
  if (w == 0) { role = kRoleMma; return; }
  if (w == 4) { role = kRoleTma; return; }
  if (w == 8 || w == 12) { role = kRoleCopy; rank = w == 8 ? 0 : 1; return; }
  if (w == 16 || w == 1 || w == 2 || w == 3) { role = kRoleEpi; return; }
  if (w == 15 || w >= 17) { role = kRoleAw; rank = w == 15 ? 0 : w - 16; return; }
  role = kRoleBw;  // 5, 6, 7, 9, 10, 11, 13, 14
  rank = w < 8 ? w - 5 : (w < 12 ? w - 6 : w - 7);
}

// A ring stage index and phase, advanced without divisions.
struct Ring {
  int s;
  uint32_t ph;
  int n;
  __device__ __forceinline__ explicit Ring(int n_) : s(0), ph(0), n(n_) {}
  __device__ __forceinline__ void next() {
    if (++s == n) {
      s = 0;
      ph ^= 1u;
    }
  }
};

// Shared-memory plan, from the row count: the MMA's M, the A stage, the depth
// of both rings.
struct SkLayout {
  int mm;         // rows of the MMA (64 or 128)
  int a_stage;    // bytes of one fp16 A stage (mm rows x 128 bytes)
  int n_raw, n_fp;
  int raw_stage;  // one k-block: two 8 KB B boxes, then the rows (sk_row_offset)
  __device__ __forceinline__ explicit SkLayout(int64_t M) {
    mm = M <= 64 ? 64 : 128;
    a_stage = mm * 128;
    n_raw = kSkRawMax;
    n_fp = mm == 64 ? 3 : 2;
    raw_stage = (kSkRawB + mm * kSkARow + 128 + 1023) & ~1023;
  }
};

// Byte offset of gathered row j (consumption order) in a raw stage's rows:
// the local shard's R rows of 64 bytes, then the staged rows, which start at
// the next 128-byte boundary (a TMA destination must be 128-byte aligned).
__device__ __forceinline__ int sk_staged_offset(int R) { return (R * kSkARow + 127) & ~127; }
__device__ __forceinline__ int sk_row_offset(int j, int R) {
  return j < R ? j * kSkARow : sk_staged_offset(R) + (j - R) * kSkARow;
}

__device__ __forceinline__ void sk_set_status(uint32_t* status, uint32_t kind, uint32_t detail) {
  if (atomicCAS(status, 0u, kind) == 0u) atomicExch(status + 1, detail);
}

__device__ __forceinline__ void widen16x(const uint4 v, uint4& a, uint4& b) {
  i8x4_to_f16x4(v.x, a.x, a.y);
  i8x4_to_f16x4(v.y, a.z, a.w);
  i8x4_to_f16x4(v.z, b.x, b.y);
  i8x4_to_f16x4(v.w, b.z, b.w);
}

// k-blocks [kb0, kb1) of unit u.
// (32-bit: a skinny plan has fewer than 2^31 units)
__device__ __forceinline__ void unit_blocks(const Geometry& g, int64_t KQ, int64_t u, int64_t& kb0,
                                            int64_t& kb1) {
  kb0 = static_cast<int64_t>(static_cast<uint32_t>(u) % static_cast<uint32_t>(KQ)) * kSkUnitBlocks;
  kb1 = kb0 + kSkUnitBlocks < g.KB ? kb0 + kSkUnitBlocks : g.KB;
}

// The piece that starts at unit u: n-tile nt, units [u, ue), k-blocks [kb0, kb1).
__device__ __forceinline__ void piece_at(const Geometry& g, int64_t KQ, int64_t u, int64_t u1,
                                         int64_t& nt, int64_t& ue, int64_t& kb0, int64_t& kb1) {
  const uint32_t u32 = static_cast<uint32_t>(u), kq = static_cast<uint32_t>(KQ);
  nt = u32 / kq;
  ue = (nt + 1) * KQ < u1 ? (nt + 1) * KQ : u1;
  kb0 = static_cast<int64_t>(u32 - static_cast<uint32_t>(nt) * kq) * kSkUnitBlocks;
  const int64_t end = (ue - nt * KQ) * kSkUnitBlocks;
  kb1 = end < g.KB ? end : g.KB;
}

// ------------------------------------------------------------------ copy warps
// Copy task t = (k-part j, position pos, chunk q): the chunk's c rows over the
// part's k-range, from the source shard into the int8 staging, then one
// release of the task's own counter.  Tasks are numbered in part-major order
// and handed out by a grid-wide ticket counter (ticket i is task i), so the
// resident warps always take the lowest tasks left; each warp draws its first
// ticket before the CTA's set-up, so the first parts are in flight at once.
template <bool kTrace>
__device__ void sk_copy_warp(const SkinnyParams& p, int lane, unsigned long long first_ticket) {
  const Geometry& g = p.g;
  [[maybe_unused]] uint32_t tn = 0;  // trace events of this warp
  const int64_t tasks = (int64_t)(g.S - 1) * g.Q * p.np;
  for (bool first = true;; first = false) {
    // (the first ticket was drawn by lane 0 while the CTA was being set up)
    unsigned long long ticket = first_ticket;
    if (lane == 0 && !first) ticket = atomicAdd(p.item_counter, 1ull);
    ticket = __shfl_sync(0xffffffffu, ticket, 0);
    const int64_t t = static_cast<int64_t>(ticket - p.item_base);
    if (t >= tasks) break;  // exactly one failing ticket per copy warp and run
    if (t < 0) {
      // tickets behind this run's base: the counters were not reset after a
      // failed run; copy nothing (the readers time out and report it)
      if (lane == 0) sk_set_status(p.status, kStatusChunkTimeout, 0xFFFFFFu);
      break;
    }
    int j, pos;
    int64_t q, k0, k1;
    skinny_task(g, p.kq, p.np, t, j, pos, q, k0, k1);
    if (t == p.debug_skip_item) continue;  // failure injection: this part never lands
    if (p.debug_delay_ns) __nanosleep(p.debug_delay_ns);
    if constexpr (kTrace)
      if (lane == 0)
        trace_emit(p.trace, tn, threadIdx.x >> 5, kTrCopyStart,
                   static_cast<uint32_t>(skinny_counter(g, j, pos, q)), t);
    const int64_t n = (k1 - k0) / 16;  // 16-byte vectors of one row
    for (int64_t r = q * g.c; r < (q + 1) * g.c; ++r) {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.src[pos]) +
                                                        r * g.K + k0);
      uint4* dst = reinterpret_cast<uint4*>(p.staging + ((int64_t)(pos - 1) * g.R + r) * g.K + k0);
      // 8 independent 16-byte loads in flight per lane
      int64_t v = lane;
      for (; v + 7 * 32 < n; v += 8 * 32) {
        uint4 x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = ld_nc_v4(src + v + u * 32);
#pragma unroll
        for (int u = 0; u < 8; ++u) dst[v + u * 32] = x[u];
      }
      for (; v < n; v += 32) dst[v] = ld_nc_v4(src + v);
    }
    // the warp barrier orders every lane's stores before lane 0's release
    // (release is cumulative), which publishes them at GPU scope
    __syncwarp();
    if (lane == 0) {
      const int64_t ci = skinny_counter(g, j, pos, q);
      if constexpr (kTrace) trace_emit(p.trace, tn, threadIdx.x >> 5, kTrLanded, static_cast<uint32_t>(ci), t);
      red_release_gpu_add(p.counters + ci, 1u);
    }
  }
}

// Parts (bit j) whose counters have all reached this epoch's target, read
// once without waiting: each lane acquires its share of all np parts' counters.
// (Relaxed loads, 8 in flight per lane, then one acquire fence per lane.)
__device__ uint32_t sk_parts_landed(const SkinnyParams& p, int lane) {
  const Geometry& g = p.g;
  const int64_t per_part = (int64_t)(g.S - 1) * g.Q, total = per_part * p.np;
  uint32_t missing = 0;
  for (int64_t i0 = lane; i0 < total; i0 += 8 * 32) {
    uint32_t v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t i = i0 + u * 32;
      v[u] = i < total ? ld_relaxed_gpu(p.counters + i) : p.epoch;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t i = i0 + u * 32;
      if (v[u] < p.epoch)
        missing |= 1u << (static_cast<uint32_t>(i) / static_cast<uint32_t>(per_part));
    }
  }
  fence_acq_rel_gpu();
  missing = __reduce_or_sync(0xffffffffu, missing);
  const uint32_t all = p.np >= 32 ? 0xffffffffu : ((1u << p.np) - 1u);
  return all & ~missing;
}

// All lanes acquire the counters of part j (every remote chunk's slice of the
// part's k-range); true once all have landed in this epoch (false on timeout
// or abort, with the status set).
__device__ bool sk_wait_part(const SkinnyParams& p, int j, int lane, volatile int* abort) {
  const Geometry& g = p.g;
  const int64_t per_part = (int64_t)(g.S - 1) * g.Q;
  const uint32_t* cnt = p.counters + (int64_t)j * per_part;
  const uint32_t target = p.epoch;
  bool ok = true;
  for (int64_t q = lane; q < per_part && ok; q += 32) {
    if (ld_relaxed_gpu(cnt + q) >= target) continue;
    const uint64_t deadline = globaltimer_ns() + p.timeout_ns;
    uint32_t spins = 0;
    while (ld_relaxed_gpu(cnt + q) < target) {
      __nanosleep(64);
      if (++spins == 16) {
        spins = 0;
        if (*abort || *reinterpret_cast<volatile uint32_t*>(p.status) != 0u ||
            globaltimer_ns() > deadline) {
          ok = false;
          break;
        }
      }
    }
  }
  fence_acq_rel_gpu();  // with the relaxed reads above: an acquire of every counter seen
  ok = __all_sync(0xffffffffu, ok);
  if (!ok && lane == 0) {
    sk_set_status(p.status, kStatusChunkTimeout, 0x10000u | static_cast<uint32_t>(j));
    *abort = 1;
  }
  __syncwarp();
  return ok;
}

// ------------------------------------------------------------------ TMA warp
// k-block kb of n-tile nt into the raw stage at `st`: B (both halves), then
// the rows (the local shard, then every staged shard: consumption order).
__device__ __forceinline__ void sk_issue_b(const SkinnyParams& p, uint8_t* st, uint64_t* bar,
                                           int64_t nt, int64_t kb) {
  const int32_t y = static_cast<int32_t>(kb * kBlockK);
  if (p.b3d) {
    // both 128-column halves of the n-tile: blocks 2 nt and 2 nt + 1 of the 3D view
    tma_load_3d(st, &p.tm_b8, bar, 0, y, static_cast<int32_t>(2 * nt));
  } else {
    tma_load_2d(st, &p.tm_b8, bar, static_cast<int32_t>(nt * kSkN), y);
    tma_load_2d(st + kSkBoxB, &p.tm_b8, bar, static_cast<int32_t>(nt * kSkN + kSkHalf), y);
  }
}

// The streamed gather: for each k-block of a unit, B and the local shard's
// rows go out at once (no wait: the local row group comes first, "AllGather + GEMM 通算融合
// 算子示例", 流式流水线); the staged rows of the other shards go out as soon as
// the k-part the unit reads has landed for every remote chunk, which the
// warp's 32 lanes check together on the part's ready counters.  A part that
// has been checked once stays checked for the rest of the run.
template <bool kTrace>
__device__ void sk_tma_warp(const SkinnyParams& p, uint8_t* sRaw, const SkLayout& L,
                            uint64_t* raw_full, uint64_t* raw_empty, int lane,
                            volatile int* abort) {
  const Geometry& g = p.g;
  [[maybe_unused]] uint32_t tn = 0;  // trace events of this warp
  const volatile uint32_t* gstatus = p.status;
  const int64_t KQ = p.kq;
  int64_t u0, u1;
  skinny_cta_range(p.n_tiles * KQ, blockIdx.x, gridDim.x, u0, u1);
  const uint32_t tx = static_cast<uint32_t>(kSkRawB + g.M * kSkARow);
  const bool remote = g.S > 1;
  const bool wait = remote && (p.flags & kFlagWait) != 0;
  if (lane == 0) {
    tma_prefetch_desc(&p.tm_b8);
    tma_prefetch_desc(&p.tm_a8_local);
    if (remote) tma_prefetch_desc(&p.tm_a8_stage);
  }
  uint32_t ready = 0;                       // bit j: part j checked in this run
  uint32_t issued = 0, issued_phase = 0;    // bit s: stage s used / parity of its last use
  bool ok = true, wait_failed = false;
  Ring r(L.n_raw);
  int64_t i = 0;  // raw stages issued
  for (int64_t u = u0; u < u1 && ok; ++u) {
    const int64_t nt = static_cast<uint32_t>(u) / static_cast<uint32_t>(KQ), q = u - nt * KQ;
    int64_t kb0, kb1;
    unit_blocks(g, KQ, u, kb0, kb1);
    for (int64_t kb = kb0; kb < kb1; ++kb, ++i, r.next()) {
      uint8_t* st = sRaw + r.s * L.raw_stage;
      const int32_t x = static_cast<int32_t>(kb * kBlockK);
      if (lane == 0) {
        if (i >= L.n_raw &&
            !mbar_wait(&raw_empty[r.s], r.ph ^ 1u, p.pipe_timeout_ns, abort, gstatus))
          ok = false;
        if (ok) {
          mbar_arrive_expect_tx(&raw_full[r.s], tx);
          sk_issue_b(p, st, &raw_full[r.s], nt, kb);
          tma_load_2d(st + kSkRawB, &p.tm_a8_local, &raw_full[r.s], x, 0);
          issued |= 1u << r.s;
          issued_phase = (issued_phase & ~(1u << r.s)) | (r.ph << r.s);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      if (remote) {
        const int j = skinny_part_of(q, KQ, p.np);
        if (wait && !((ready >> j) & 1u)) {
          if constexpr (kTrace)
            if (lane == 0) trace_emit(p.trace, tn, threadIdx.x >> 5, kTrWaitStart, static_cast<uint32_t>(u), j);
          if (!sk_wait_part(p, j, lane, abort)) {
            ok = false;
            wait_failed = true;
            break;
          }
          if constexpr (kTrace)
            if (lane == 0) trace_emit(p.trace, tn, threadIdx.x >> 5, kTrWaitEnd, static_cast<uint32_t>(u), j);
          // the other parts have usually landed by now as well: one sweep over
          // their counters spares the later units the wait
          ready |= (1u << j) | sk_parts_landed(p, lane);
          if (lane == 0) {
            // the staged rows were written by other SMs' generic stores; TMA reads them
            fence_acq_rel_gpu();
            fence_proxy_async_global();
          }
        }
        if (lane == 0)
          tma_load_3d(st + kSkRawB + sk_staged_offset(static_cast<int>(g.R)), &p.tm_a8_stage,
                      &raw_full[r.s], x, 0, 0);
      }
    }
    if constexpr (kTrace)
      if (ok && lane == 0) trace_emit(p.trace, tn, threadIdx.x >> 5, kTrUnitIssued, static_cast<uint32_t>(u), 0);
  }
  if (!ok && lane == 0) {
    if (!wait_failed) sk_set_status(p.status, kStatusPipelineTimeout, 0x1100u);
    *abort = 1;
    // Loads already issued must land before the CTA exits.  A stage whose
    // staged rows were never issued cannot complete; its B boxes and local
    // rows land well within the bounded waits below.
    volatile int never = 0;
    for (int s = 0; s < L.n_raw; ++s)
      if (issued & (1u << s))
        mbar_wait(&raw_full[s], (issued_phase >> s) & 1u, 20000000ull, &never);
  }
  __syncwarp();
}

// ------------------------------------------------------------------ B widening (8 warps)
// Per k-block and box half h (columns 128h .. 128h + 127), thread t widens 32
// bytes of one k-row: columns qt * 32 .. +31 of the half (half of one
// 64-column swizzle group of the MN-major fp16 tile) of k-row krow.  The 8
// lanes of a shared-memory phase take 8 consecutive k-rows of one quarter qt,
// so both the swizzled raw reads and the swizzled fp16 writes hit 8 distinct
// 16-byte bank groups.
template <bool kTrace>
__device__ void sk_bwiden(const SkinnyParams& p, const uint8_t* sRaw, const SkLayout& L,
                          uint8_t* sFp, uint64_t* raw_full, uint64_t* raw_empty,
                          uint64_t* fp_full, uint64_t* fp_empty, int t, volatile int* abort) {
  const Geometry& g = p.g;
  [[maybe_unused]] uint32_t tn = 0;  // trace events of this warp
  const volatile uint32_t* gstatus = p.status;
  const int lane = t & 31, krow = 8 * (t >> 5) + (t & 7), qt = (t >> 3) & 3;
  const int cb = (qt & 1) * 4;  // first 16-byte chunk within the 64-column group
  const int64_t KQ = p.kq;
  int64_t u0, u1;
  skinny_cta_range(p.n_tiles * KQ, blockIdx.x, gridDim.x, u0, u1);
  Ring rr(L.n_raw), fr(L.n_fp);
  for (int64_t u = u0; u < u1; ++u) {
    int64_t kb0, kb1;
    unit_blocks(g, KQ, u, kb0, kb1);
    for (int b = 0; b < static_cast<int>(kb1 - kb0); ++b, fr.next(), rr.next()) {
      if (!mbar_wait(&raw_full[rr.s], rr.ph, p.pipe_timeout_ns, abort, gstatus)) {
        if (lane == 0) {
          sk_set_status(p.status, kStatusPipelineTimeout, 0x1200u);
          *abort = 1;
        }
        return;
      }
      if constexpr (kTrace)
        if (t == 0 && b == 0)
          trace_emit(p.trace, tn, threadIdx.x >> 5, kTrUnitLanded, static_cast<uint32_t>(u), 0);
      const uint8_t* raw = sRaw + rr.s * L.raw_stage;
      if (!mbar_wait(&fp_empty[fr.s], fr.ph ^ 1u, p.pipe_timeout_ns, abort, gstatus)) {
        if (lane == 0) {
          sk_set_status(p.status, kStatusPipelineTimeout, 0x1201u);
          *abort = 1;
        }
        return;
      }
      // raw B arrives 128-byte swizzled: 16-byte chunk c of box row r sits at c ^ (r % 8)
      const int r = krow;
      uint4 v[4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint8_t* src = raw + h * kSkBoxB + r * kSkHalf;
        v[2 * h] = *reinterpret_cast<const uint4*>(src + (((2 * qt) ^ (r & 7)) * 16));
        v[2 * h + 1] = *reinterpret_cast<const uint4*>(src + (((2 * qt + 1) ^ (r & 7)) * 16));
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        // 64-column group 2h + qt / 2 of the fp16 k-block
        uint8_t* dst = sFp + fr.s * kSkFpB + (2 * h + (qt >> 1)) * (64 * kBlockK * 2) + krow * 128;
        uint4 a, c;
        widen16x(v[2 * h], a, c);
        *reinterpret_cast<uint4*>(dst + (((cb + 0) ^ (krow & 7)) * 16)) = a;
        *reinterpret_cast<uint4*>(dst + (((cb + 1) ^ (krow & 7)) * 16)) = c;
        widen16x(v[2 * h + 1], a, c);
        *reinterpret_cast<uint4*>(dst + (((cb + 2) ^ (krow & 7)) * 16)) = a;
        *reinterpret_cast<uint4*>(dst + (((cb + 3) ^ (krow & 7)) * 16)) = c;
      }
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&fp_full[fr.s]);
        mbar_arrive(&raw_empty[rr.s]);  // this k-block's raw stage is read
      }
      if constexpr (kTrace)
        if (t == 0) trace_emit(p.trace, tn, threadIdx.x >> 5, kTrKbWidened, static_cast<uint32_t>(kb0 + b), u);
    }
  }
}

// ------------------------------------------------------------------ A widening (4 warps)
// Thread t widens the 16 k at k-offset (t % 4) * 16 of rows t / 4 + 32 e,
// e < NE (NE = 2 for M <= 64, 4 for M <= 128), from the raw stage's rows
// (64 bytes each, consumption order) into fp16 A stages: K-major, 128-byte
// rows, 16-byte chunk c of row j at c ^ (j % 8).  Rows M .. mm - 1 are left
// as they are: they only reach rows of the accumulator nobody reads.
template <int NE>
__device__ void sk_awiden(const SkinnyParams& p, const uint8_t* sRaw, const SkLayout& L,
                          uint8_t* sA, uint64_t* raw_full, uint64_t* raw_empty,
                          uint64_t* a_full, uint64_t* a_empty, int t, volatile int* abort) {
  const Geometry& g = p.g;
  const volatile uint32_t* gstatus = p.status;
  const int lane = t & 31, j0 = t >> 2, h = t & 3;
  const int R = static_cast<int>(g.R);
  const int64_t KQ = p.kq;
  int64_t u0, u1;
  skinny_cta_range(p.n_tiles * KQ, blockIdx.x, gridDim.x, u0, u1);
  Ring rr(L.n_raw), ar(L.n_fp);
  for (int64_t u = u0; u < u1; ++u) {
    int64_t kb0, kb1;
    unit_blocks(g, KQ, u, kb0, kb1);
    for (int b = 0; b < static_cast<int>(kb1 - kb0); ++b, ar.next(), rr.next()) {
      if (!mbar_wait(&raw_full[rr.s], rr.ph, p.pipe_timeout_ns, abort, gstatus)) {
        if (lane == 0) {
          sk_set_status(p.status, kStatusPipelineTimeout, 0x1300u);
          *abort = 1;
        }
        return;
      }
      const uint8_t* raw = sRaw + rr.s * L.raw_stage + kSkRawB;
      if (!mbar_wait(&a_empty[ar.s], ar.ph ^ 1u, p.pipe_timeout_ns, abort, gstatus)) {
        if (lane == 0) {
          sk_set_status(p.status, kStatusPipelineTimeout, 0x1301u);
          *abort = 1;
        }
        return;
      }
#pragma unroll
      for (int e = 0; e < NE; ++e) {
        const int j = j0 + 32 * e;
        if (j < g.M) {
          const uint4 v =
              *reinterpret_cast<const uint4*>(raw + sk_row_offset(j, R) + h * 16);
          uint4 lo, hi;
          widen16x(v, lo, hi);
          uint8_t* dst = sA + ar.s * L.a_stage + j * 128;
          *reinterpret_cast<uint4*>(dst + (((2 * h) ^ (j & 7)) * 16)) = lo;
          *reinterpret_cast<uint4*>(dst + (((2 * h + 1) ^ (j & 7)) * 16)) = hi;
        }
      }
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&a_full[ar.s]);
        mbar_arrive(&raw_empty[rr.s]);  // this k-block's raw stage is read
      }
    }
  }
}

// ------------------------------------------------------------------ MMA warp
// Pieces: maximal runs of this CTA's units inside one n-tile; segments: at most
// kSegBlocks k-blocks of a piece, accumulated into the fp32 accumulator, which
// the epilogue folds into the int32 sums before the next segment starts.
template <bool kTrace>
__device__ void sk_mma(const SkinnyParams& p, const uint8_t* sFp, const uint8_t* sA,
                       const SkLayout& L, uint64_t* st_full, uint64_t* st_empty,
                       uint64_t* dfull, uint64_t* dempty, uint32_t tmem, volatile int* abort) {
  const Geometry& g = p.g;
  [[maybe_unused]] uint32_t tn = 0;  // trace events of this warp
  const volatile uint32_t* gstatus = p.status;
  // D fp32 (mm rows x 256 columns); A operand = gathered rows (K-major),
  // B operand = the widened B tile (MN-major)
  const uint32_t idesc = idesc_f16_f32(L.mm, kSkN, /*a_mn=*/false, /*b_mn=*/true);
  // Descriptors of stage 0, k-step 0; the start address sits in the low bits
  // (16-byte units), so other stages and k-steps are plain additions.
  // Rows: 8-row groups 1 KB apart.  B: 64-column groups 8 KB apart (LBO),
  // 8-k-row groups 1 KB apart (SBO).
  const uint64_t ad0 = smem_desc_sw128(smem_u32(sA), 16, 1024);
  const uint64_t bd0 = smem_desc_sw128(smem_u32(sFp), 64 * kBlockK * 2, 1024);
  const int64_t KQ = p.kq;
  int64_t u0, u1;
  skinny_cta_range(p.n_tiles * KQ, blockIdx.x, gridDim.x, u0, u1);
  Ring kr(L.n_fp);
  uint32_t seg = 0;  // segment sequence index
  bool ok = true;
  for (int64_t u = u0; u < u1 && ok;) {
    int64_t nt, ue, kb0, kb1;
    piece_at(g, KQ, u, u1, nt, ue, kb0, kb1);
    for (int64_t s0 = kb0; s0 < kb1 && ok; s0 += kSegBlocks, ++seg) {
      const int n = static_cast<int>((s0 + kSegBlocks < kb1 ? s0 + kSegBlocks : kb1) - s0);
      // the epilogue has read the previous segment's accumulator
      if (!mbar_wait(dempty, (seg & 1u) ^ 1u, p.pipe_timeout_ns, abort, gstatus)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem + kSkDcol;
      for (int b = 0; b < n; ++b, kr.next()) {
        if (!mbar_wait(&st_full[kr.s], kr.ph, p.pipe_timeout_ns, abort, gstatus)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ad = ad0 + static_cast<uint64_t>((kr.s * L.a_stage) >> 4);
        const uint64_t bd = bd0 + static_cast<uint64_t>((kr.s * kSkFpB) >> 4);
#pragma unroll
        for (int k = 0; k < kBlockK / kUmmaK; ++k)
          // rows: +16 k = 32 bytes; B: +16 k-rows = two 8-row groups (2048 bytes)
          mma_f16(d, ad + static_cast<uint64_t>((k * kUmmaK * 2) >> 4),
                  bd + static_cast<uint64_t>((k * kUmmaK * 128) >> 4), idesc,
                  (b > 0 || k > 0) ? 1u : 0u);
        mma_commit(&st_empty[kr.s]);
        if constexpr (kTrace)
          trace_emit(p.trace, tn, threadIdx.x >> 5, kTrKbMma, static_cast<uint32_t>(s0 + b), static_cast<uint64_t>(nt));
      }
      if (!ok) break;
      mma_commit(dfull);
    }
    u = ue;
  }
  if (!ok) {
    sk_set_status(p.status, kStatusPipelineTimeout, 0x1400u);
    *abort = 1;
  }
}

// ------------------------------------------------------------------ epilogue (4 warps)
// TMEM lane = row of the tile, TMEM column = column of the n-tile.  With
// mm = 128, gathered row j sits on lane j; with mm = 64, rows 16q .. 16q + 15
// sit on lanes 32q .. 32q + 15 of quadrant q (lanes 32q + 16 .. 32q + 31 are
// not written by the MMA and their values are never stored).  The kernel runs
// this one for mm = 128 and sk_epilogue64 below for mm = 64.
template <bool kTrace>
__device__ void sk_epilogue(const SkinnyParams& p, const SkLayout& L, uint64_t* dfull,
                            uint64_t* dempty, uint32_t tmem, int quad, int lane,
                            volatile int* abort) {
  const Geometry& g = p.g;
  [[maybe_unused]] uint32_t tn = 0;  // trace events of this warp
  const volatile uint32_t* gstatus = p.status;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
  // gathered row of this thread (consumption order), -1 for none
  const int jr = L.mm == 128 ? quad * 32 + lane : (lane < 16 ? quad * 16 + lane : -1);
  const bool row_ok = jr >= 0 && jr < g.M;
  // its C row: row r of the shard at position jr / R, s = (local + position) % S
  int64_t crow = 0;
  if (row_ok) {
    const int R = static_cast<int>(g.R), pos = jr / R;
    crow = static_cast<int64_t>((p.local + pos) % g.S) * R + (jr - pos * R);
  }
  const int64_t KQ = p.kq, U = p.n_tiles * KQ;
  int64_t u0, u1;
  skinny_cta_range(U, blockIdx.x, gridDim.x, u0, u1);
  uint32_t seg = 0;
  for (int64_t u = u0; u < u1;) {
    int64_t nt, ue, kb0, kb1;
    piece_at(g, KQ, u, u1, nt, ue, kb0, kb1);
    const int64_t slot = nt * p.cmax + (blockIdx.x - skinny_owner(nt * KQ, U, gridDim.x));
    int4* out = reinterpret_cast<int4*>(p.ws + (slot * g.M + crow) * kSkN);
    for (int64_t s0 = kb0; s0 < kb1; s0 += kSegBlocks, ++seg) {
      const bool first = s0 == kb0, last = s0 + kSegBlocks >= kb1;
      const bool mine = mbar_wait(dfull, seg & 1u, p.pipe_timeout_ns, abort, gstatus);
      // the four epilogue warps decide together
      uint32_t all_ok;
      asm volatile(
          "{\n\t.reg .pred q, r;\n\tsetp.ne.u32 q, %1, 0;\n\t"
          "bar.red.and.pred r, 1, 128, q;\n\tselp.u32 %0, 1, 0, r;\n\t}"
          : "=r"(all_ok)
          : "r"(mine ? 1u : 0u)
          : "memory");
      if (!all_ok) {
        if (lane == 0) {
          sk_set_status(p.status, kStatusPipelineTimeout, 0x1500u);
          *abort = 1;
        }
        return;
      }
      tc_fence_after();
      for (int j = 0; j < kSkN / 32; ++j) {
        uint32_t f[32], s[32];
        tmem_ld32(lane_base + kSkDcol + j * 32, f);
        if (!first) tmem_ld32(lane_base + kSkScol + j * 32, s);
        tmem_ld_wait();
        if (j == kSkN / 32 - 1) {
          // the accumulator has been read: the MMA may start the next segment
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(dempty);
        }
        uint32_t acc[32];
#pragma unroll
        for (int e = 0; e < 32; ++e)
          acc[e] = (first ? 0u : s[e]) +
                   static_cast<uint32_t>(__float2int_rn(__uint_as_float(f[e])));
        if (!last) {
          tmem_st32(lane_base + kSkScol + j * 32, acc);
          continue;
        }
        // columns 32j .. 32j + 31 of the thread's row: 128 contiguous bytes
        if (row_ok) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            out[j * 8 + e] = make_int4(static_cast<int32_t>(acc[4 * e]),
                                       static_cast<int32_t>(acc[4 * e + 1]),
                                       static_cast<int32_t>(acc[4 * e + 2]),
                                       static_cast<int32_t>(acc[4 * e + 3]));
        }
      }
      if (!last) tmem_st_wait();
    }
    if constexpr (kTrace)
      if (quad == 0 && lane == 0) trace_emit(p.trace, tn, threadIdx.x >> 5, kTrPieceDone, static_cast<uint32_t>(nt), u);
    u = ue;
  }
}

// The epilogue for mm = 64: the accumulator fills lanes 32q .. 32q + 15 of
// each quadrant, which the 16x256b shape reads without the 16 idle lanes:
// thread t holds rows 16q + t / 4 and 16q + t / 4 + 8, columns 8i + 2(t % 4)
// and +1 of each 8-column block i of a 64-column chunk.
template <bool kTrace>
__device__ void sk_epilogue64(const SkinnyParams& p, uint64_t* dfull, uint64_t* dempty,
                              uint32_t tmem, int quad, int lane, volatile int* abort) {
  const Geometry& g = p.g;
  [[maybe_unused]] uint32_t tn = 0;  // trace events of this warp
  const volatile uint32_t* gstatus = p.status;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
  const int R = static_cast<int>(g.R);
  // C row of gathered row j (consumption order): row j % R of the shard at
  // position j / R, i.e. shard (local + position) % S
  auto c_row = [&](int j) -> int64_t {
    const int pos = j / R;
    return static_cast<int64_t>((p.local + pos) % g.S) * R + (j - pos * R);
  };
  const int ja = quad * 16 + (lane >> 2), jb = ja + 8;
  const bool oka = ja < g.M, okb = jb < g.M;
  const int64_t cra = oka ? c_row(ja) : 0, crb = okb ? c_row(jb) : 0;
  const int cp = 2 * (lane & 3);
  const int64_t KQ = p.kq, U = p.n_tiles * KQ;
  int64_t u0, u1;
  skinny_cta_range(U, blockIdx.x, gridDim.x, u0, u1);
  uint32_t seg = 0;
  for (int64_t u = u0; u < u1;) {
    int64_t nt, ue, kb0, kb1;
    piece_at(g, KQ, u, u1, nt, ue, kb0, kb1);
    const int64_t slot = nt * p.cmax + (blockIdx.x - skinny_owner(nt * KQ, U, gridDim.x));
    int32_t* out_a = p.ws + (slot * g.M + cra) * kSkN + cp;
    int32_t* out_b = p.ws + (slot * g.M + crb) * kSkN + cp;
    for (int64_t s0 = kb0; s0 < kb1; s0 += kSegBlocks, ++seg) {
      const bool first = s0 == kb0, last = s0 + kSegBlocks >= kb1;
      const bool mine = mbar_wait(dfull, seg & 1u, p.pipe_timeout_ns, abort, gstatus);
      uint32_t all_ok;
      asm volatile(
          "{\n\t.reg .pred q, r;\n\tsetp.ne.u32 q, %1, 0;\n\t"
          "bar.red.and.pred r, 1, 128, q;\n\tselp.u32 %0, 1, 0, r;\n\t}"
          : "=r"(all_ok)
          : "r"(mine ? 1u : 0u)
          : "memory");
      if (!all_ok) {
        if (lane == 0) {
          sk_set_status(p.status, kStatusPipelineTimeout, 0x1500u);
          *abort = 1;
        }
        return;
      }
      tc_fence_after();
      for (int j = 0; j < kSkN / 64; ++j) {
        uint32_t f[32], s[32];
        tmem_ld16x64(lane_base + kSkDcol + j * 64, f);
        if (!first) tmem_ld16x64(lane_base + kSkScol + j * 64, s);
        tmem_ld_wait();
        if (j == kSkN / 64 - 1) {
          // the accumulator has been read: the MMA may start the next segment
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(dempty);
        }
#pragma unroll
        for (int e = 0; e < 32; ++e)
          s[e] = (first ? 0u : s[e]) +
                 static_cast<uint32_t>(__float2int_rn(__uint_as_float(f[e])));
        if (!last) {
          tmem_st16x64(lane_base + kSkScol + j * 64, s);
          continue;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (oka)
            *reinterpret_cast<int2*>(out_a + j * 64 + 8 * i) =
                make_int2(static_cast<int32_t>(s[4 * i]), static_cast<int32_t>(s[4 * i + 1]));
          if (okb)
            *reinterpret_cast<int2*>(out_b + j * 64 + 8 * i) =
                make_int2(static_cast<int32_t>(s[4 * i + 2]), static_cast<int32_t>(s[4 * i + 3]));
        }
      }
      if (!last) tmem_st_wait();
    }
    if constexpr (kTrace)
      if (quad == 0 && lane == 0) trace_emit(p.trace, tn, threadIdx.x >> 5, kTrPieceDone, static_cast<uint32_t>(nt), u);
    u = ue;
  }
}

template <bool kTrace>
__global__ void __launch_bounds__(kSkThreads, 1) ag_skinny_kernel(const __grid_constant__ SkinnyParams p) {
  [[maybe_unused]] uint32_t tc = 0;  // trace events of the CTA slot
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const SkLayout L(p.g.M);
  uint8_t* sFp = smem;                          // 1024-aligned swizzled fp16 B stages
  uint8_t* sA = sFp + L.n_fp * kSkFpB;          // swizzled fp16 A stages
  uint8_t* sRaw = sA + L.n_fp * L.a_stage;      // raw ring: per k-block, B, then the rows
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kSkDataBytes);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = raw_full + kSkRawMax;
  // One full/empty pair per fp16 stage: the B and the A half of stage s are
  // written by the two widening roles (12 arrivals) and released by one commit.
  uint64_t* st_full = raw_empty + kSkRawMax;
  uint64_t* st_empty = st_full + kSkFpMax;
  uint64_t* dfull = st_empty + kSkFpMax;
  uint64_t* dempty = dfull + 1;
  uint64_t* drain = dempty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool gemm = (p.flags & kFlagGemm) != 0;
  int role, rank;
  sk_role(warp, role, rank);
  // A copy warp draws its first ticket before the set-up below, so the
  // atomic's latency overlaps it (tickets keep the copies live whichever CTAs
  // are resident).
  const bool copier = role == kRoleCopy && (p.flags & kFlagCopy) != 0;
  unsigned long long first_ticket = 0;
  if (copier && lane == 0) first_ticket = atomicAdd(p.item_counter, 1ull);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSkRawMax; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], (kSkBwThreads + kSkAwThreads) / 32);  // both widening roles
    }
    for (int s = 0; s < kSkFpMax; ++s) {
      mbar_init(&st_full[s], (kSkBwThreads + kSkAwThreads) / 32);
      mbar_init(&st_empty[s], 1);
    }
    mbar_init(dfull, 1);
    mbar_init(dempty, 4);
    mbar_init(drain, 1);
    *tmem_slot = 0;
    *abort = 0;
    fence_mbar_init();
  }
  if (gemm && warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if constexpr (kTrace)
    if (threadIdx.x == 0) trace_emit(p.trace, tc, kTrCtaSlot, kTrCtaStart, 0, 0);
  if (role == kRoleCopy) {
    if (copier) sk_copy_warp<kTrace>(p, lane, first_ticket);
  } else if (gemm) {
    switch (role) {
      case kRoleMma:
        if (lane == 0)
          sk_mma<kTrace>(p, sFp, sA, L, st_full, st_empty, dfull, dempty, tmem, abort);
        break;
      case kRoleTma:
        sk_tma_warp<kTrace>(p, sRaw, L, raw_full, raw_empty, lane, abort);
        break;
      case kRoleEpi:
        if (L.mm == 64)
          sk_epilogue64<kTrace>(p, dfull, dempty, tmem, warp & 3, lane, abort);
        else
          sk_epilogue<kTrace>(p, L, dfull, dempty, tmem, warp & 3, lane, abort);
        break;
      case kRoleBw:
        sk_bwiden<kTrace>(p, sRaw, L, sFp, raw_full, raw_empty, st_full, st_empty,
                          rank * 32 + lane, abort);
        break;
      default:
        if (L.mm == 64)
          sk_awiden<2>(p, sRaw, L, sA, raw_full, raw_empty, st_full, st_empty, rank * 32 + lane,
                       abort);
        else
          sk_awiden<4>(p, sRaw, L, sA, raw_full, raw_empty, st_full, st_empty, rank * 32 + lane,
                       abort);
        break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (gemm && warp == 0) {
    if (lane == 0) {
      mma_commit(drain);
      volatile int never = 0;
      mbar_wait(drain, 0, p.pipe_timeout_ns, &never);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if constexpr (kTrace)
    if (threadIdx.x == 0) trace_emit(p.trace, tc, kTrCtaSlot, kTrCtaEnd, 0, 0);
}

// C_i32 = (sum of the n-tile's workspace slots) + bias,
// D = fp16(fp32(C_i32) * scale): one thread per 8 consecutive outputs of a row
// (N % 16 == 0, so they never straddle a row or an n-tile).
__global__ void __launch_bounds__(256) ag_skinny_finish_kernel(
    const int32_t* __restrict__ ws, const int32_t* __restrict__ bias,
    const float* __restrict__ scale, int32_t* __restrict__ C_i32, uint16_t* __restrict__ D,
    int64_t M, int64_t N, int64_t n_tiles, int64_t KQ, int64_t cmax, int grid) {
  // launched as a programmatic dependent of the skinny kernel: wait for it to
  // complete (all of its workspace stores visible)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t groups = M * N / 8, U = n_tiles * KQ;
  // the CTA ranges U b / G in 32-bit arithmetic when U and G allow it
  const bool narrow =
      static_cast<uint64_t>(U + 1) * static_cast<uint64_t>(grid) + static_cast<uint64_t>(U) <
      (1ull << 32);
  const uint32_t U32 = static_cast<uint32_t>(U), G32 = static_cast<uint32_t>(grid);
  auto owner = [&](int64_t x) -> int64_t {
    if (narrow)
      return static_cast<int64_t>((static_cast<uint32_t>(x + 1) * G32 + U32 - 1) / U32) - 1;
    return skinny_owner(x, U, grid);
  };
  auto has_units = [&](int64_t b) -> bool {
    if (narrow)
      return U32 * static_cast<uint32_t>(b) / G32 < U32 * static_cast<uint32_t>(b + 1) / G32;
    int64_t lo, hi;
    skinny_cta_range(U, b, grid, lo, hi);
    return lo < hi;
  };
  for (int64_t gi = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; gi < groups;
       gi += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t off = gi * 8, m = off / N, n = off - m * N;
    const int64_t nt = n / kSkN, nl = n - nt * kSkN;
    const int64_t b_lo = owner(nt * KQ);
    const int64_t b_hi = owner((nt + 1) * KQ - 1);
    int32_t c[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    // four slots per step: their eight 16-byte loads are issued before any is
    // used (a CTA without units wrote no slot: its loads are skipped)
    for (int64_t b0 = b_lo; b0 <= b_hi; b0 += 4) {
      int4 x[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t b = b0 + i;
        x[2 * i] = x[2 * i + 1] = make_int4(0, 0, 0, 0);
        if (b <= b_hi && has_units(b)) {
          const int4* sp = reinterpret_cast<const int4*>(
              ws + ((nt * cmax + (b - b_lo)) * M + m) * kSkN + nl);
          x[2 * i] = __ldcg(sp);
          x[2 * i + 1] = __ldcg(sp + 1);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int4 x0 = x[2 * i], x1 = x[2 * i + 1];
        c[0] += x0.x; c[1] += x0.y; c[2] += x0.z; c[3] += x0.w;
        c[4] += x1.x; c[5] += x1.y; c[6] += x1.z; c[7] += x1.w;
      }
    }
    const int4 b0 = __ldg(reinterpret_cast<const int4*>(bias + n));
    const int4 b1 = __ldg(reinterpret_cast<const int4*>(bias + n + 4));
    const float4 s0 = __ldg(reinterpret_cast<const float4*>(scale + n));
    const float4 s1 = __ldg(reinterpret_cast<const float4*>(scale + n + 4));
    const int32_t bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    uint32_t h[4];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      c[e] = static_cast<int32_t>(static_cast<uint32_t>(c[e]) + static_cast<uint32_t>(bb[e]));
      const uint32_t hb =
          __half_as_ushort(__float2half_rn(__fmul_rn(__int2float_rn(c[e]), ss[e])));
      if (e & 1)
        h[e >> 1] |= hb << 16;
      else
        h[e >> 1] = hb;
    }
    *reinterpret_cast<int4*>(C_i32 + off) = make_int4(c[0], c[1], c[2], c[3]);
    *reinterpret_cast<int4*>(C_i32 + off + 4) = make_int4(c[4], c[5], c[6], c[7]);
    *reinterpret_cast<uint4*>(D + off) = make_uint4(h[0], h[1], h[2], h[3]);
  }
}

}  // namespace

cudaError_t skinny_prepare() {
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&ag_skinny_kernel<false>),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSkSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(reinterpret_cast<const void*>(&ag_skinny_kernel<true>),
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kSkSmem);
}

cudaError_t launch_skinny(const SkinnyParams& p, int grid, cudaStream_t stream) {
  if (p.trace.ev)
    ag_skinny_kernel<true><<<grid, kSkThreads, kSkSmem, stream>>>(p);
  else
    ag_skinny_kernel<false><<<grid, kSkThreads, kSkSmem, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !(p.flags & kFlagGemm)) return e;
  // Programmatic dependent launch: the finish grid's launch is processed while
  // the skinny kernel runs, and its griddepcontrol.wait holds it until the
  // skinny grid has completed.  The skinny kernel triggers nothing early: a
  // trigger at its start let the finish grid in sooner and measured slower
  // (59.4 us against 55.3 us on 2 x 32 rows, K = 16384, N = 7168).
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid * 2);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, ag_skinny_finish_kernel, static_cast<const int32_t*>(p.ws),
                            p.bias, p.scale, p.C_i32, p.D_f16, p.g.M, p.g.N, p.n_tiles, p.kq,
                            p.cmax, grid);
}

}  // namespace agg
