// fused_kernel.cu -- the streamed AllGather+GEMM as ONE persistent,
// warp-specialised kernel of CTA pairs for sm_103a.
//
// The method ("AllGather + GEMM 通算融合算子示例", sections 整体架构 and
// 优化说明): a communication engine sends A chunk by chunk and bumps a
// per-source counter after each chunk; the compute engine first multiplies the
// local row group with no wait, then each remote row group after waiting on
// its counter, with continuous K accumulation and multi-buffered operand
// staging.  On one GB300 the "ranks" are shards in this GPU's memory, and both
// engines live in the same launch.
//
// Tiles are 256 x BN (BN = 256, or 128 for narrow N) and belong to a cluster
// of two CTAs on neighbouring SMs that run one tcgen05 MMA with cta_group::2:
// each CTA stages its own 128 rows of A and its own BN/2 columns of B, the
// even CTA issues the MMA, and each CTA's TMEM receives its 128 rows of the
// 256 x BN accumulator.  Per SM that is 32 KB of operands per 64-deep k-block
// instead of 48 KB for a single-SM 128 x 256 tile, and six stages fit.
//
//   warp 0      TMA warp (both CTAs): for remote tiles all 32 lanes poll the
//               ready counters of the chunks this CTA's 128 rows read, then
//               lane 0 streams A and B k-blocks into a 6-stage ring; the bytes
//               of both CTAs are counted on the even CTA's "full" barrier.
//   warp 1      MMA warp (even CTA): one thread issues tcgen05.mma; commits
//               free both CTAs' ring stages and signal both epilogues.
//               Owns the pair's TMEM allocation (512 columns per CTA).
//   warps 2-3   copy warps ("comm blocks"): take copy items in consumption
//               order from a grid-wide counter, copy (or, for int8, widen) them
//               into the staging workspace and release the chunk's counter.
//   warps 4-11  epilogue: TMEM -> registers -> global (fp32 C, or for int8
//               the exact int32 fold, bias, int32 C and fp16 D); warp w reads
//               TMEM lane quadrant w % 4 and half of the tile's columns.
//
// No CTA ever waits for a copy item that only a specific other CTA could
// perform: items are taken dynamically, so any resident CTA's copy warps make
// progress and the waits need no co-residency guarantee.  Every wait is
// bounded; on timeout the kernel records a status word, stops issuing work,
// drains what it has in flight, frees TMEM and returns.
//
// int8: sm_103a has no tcgen05 kind::i8, so int8 x int8 is computed exactly on
// the fp16 tensor path: int8 values are exact in fp16, products of two int8
// values are exact in fp32, and K is cut into segments of 1024 so every fp32
// partial sum is an integer below 2^24 (exact).  After each segment the
// epilogue converts the fp32 accumulator to int32 and adds it to the int32
// running sums it keeps in registers (one row x 128 columns per thread), so
// the two TMEM accumulators alternate as on the fp16 path and the MMA never
// waits for a fold.

#include <cuda_fp16.h>

#include "fused_kernel.cuh"
#include "sm103.cuh"

namespace agg {

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t kind, uint32_t detail) {
  if (atomicCAS(status, 0u, kind) == 0u) atomicExch(status + 1, detail);
}

// ------------------------------------------------------------------ copy warps
__device__ __forceinline__ void warp_copy16(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                            int64_t n, int lane) {
  constexpr int U = 8;
  int64_t i = lane;
  for (; i + (U - 1) * 32 < n; i += U * 32) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) v[u] = ld_nc_v4(src + i + u * 32);
#pragma unroll
    for (int u = 0; u < U; ++u) dst[i + u * 32] = v[u];
  }
  for (; i < n; i += 32) dst[i] = ld_nc_v4(src + i);
}

__device__ __forceinline__ void widen16(const uint4 v, uint4& a, uint4& b) {
  i8x4_to_f16x4(v.x, a.x, a.y);
  i8x4_to_f16x4(v.y, a.z, a.w);
  i8x4_to_f16x4(v.z, b.x, b.y);
  i8x4_to_f16x4(v.w, b.z, b.w);
}

// n source vectors of 16 int8 -> 2n destination vectors of 8 fp16.
__device__ __forceinline__ void warp_widen16(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                             int64_t n, int lane) {
  constexpr int U = 4;
  int64_t i = lane;
  for (; i + (U - 1) * 32 < n; i += U * 32) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) v[u] = ld_nc_v4(src + i + u * 32);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      uint4 a, b;
      widen16(v[u], a, b);
      dst[2 * (i + u * 32)] = a;
      dst[2 * (i + u * 32) + 1] = b;
    }
  }
  for (; i < n; i += 32) {
    uint4 a, b;
    widen16(ld_nc_v4(src + i), a, b);
    dst[2 * i] = a;
    dst[2 * i + 1] = b;
  }
}

// Bounded staging: lane 0 waits until slot `slot` may take its next block
// (the credits of the previous block's readers reached `target`).  Bounded by
// the plan's timeout; false once another wait has failed or the time is up.
__device__ bool wait_slot(const FusedParams& p, int64_t slot, uint32_t target, int lane) {
  bool ok = true;
  if (lane == 0 && ld_acquire_gpu(p.credits + slot) < target) {
    const uint64_t deadline = globaltimer_ns() + p.timeout_ns;
    uint32_t spins = 0;
    while (ld_acquire_gpu(p.credits + slot) < target) {
      __nanosleep(128);
      if (++spins == 16) {
        spins = 0;
        if (*reinterpret_cast<volatile uint32_t*>(p.status) != 0u ||
            globaltimer_ns() > deadline) {
          ok = false;
          break;
        }
      }
    }
    if (!ok) set_status(p.status, kStatusCreditTimeout, static_cast<uint32_t>(slot));
  }
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

template <bool kI8, bool kTrace>
__device__ void copy_warp(const FusedParams& p, int lane, unsigned long long first_ticket) {
  const Geometry& g = p.g;
  [[maybe_unused]] uint32_t tn = 0;  // trace events of this warp
  // With bounded staging and the GEMM in the same launch, a block may only
  // overwrite its slot after the slot's previous block has been read.  (A
  // copy-only launch has no readers and writes freely.)
  const bool credit = p.window > 0 && (p.flags & kFlagGemm) != 0;
  int64_t ready_block = -1;  // the last block whose slot this warp saw released
  for (bool first = true;; first = false) {
    // (the first ticket was drawn by lane 0 while the CTA was being set up)
    unsigned long long ticket = first_ticket;
    if (lane == 0 && !first) ticket = atomicAdd(p.item_counter, 1ull);
    ticket = __shfl_sync(0xffffffffu, ticket, 0);
    const int64_t i = static_cast<int64_t>(ticket - p.item_base);
    if (i >= g.items) break;  // exactly one failing ticket per copy warp and run
    if (i < 0) {
      // tickets behind this run's base: the counters were not reset after a
      // failed run; copy nothing (the readers time out and report it)
      if (lane == 0) set_status(p.status, kStatusChunkTimeout, 0xFFFFFFu);
      break;
    }
    int pos, piece;
    int64_t q, v0, v1;
    item_coords(g, i, pos, q, piece, v0, v1);
    if (i == p.debug_skip_item) continue;  // failure injection: this chunk never completes
    if (p.debug_delay_ns) __nanosleep(p.debug_delay_ns);
    if constexpr (kTrace)
      if (lane == 0)
        trace_emit(p.trace, tn, threadIdx.x >> 5, kTrCopyStart,
                   static_cast<uint32_t>((int64_t)(pos - 1) * g.Q + q), i);
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.src[pos]) +
                                                      q * g.c * g.K * g.src_esize);
    int64_t drow = (int64_t)(pos - 1) * g.R + q * g.c;  // staging row of the chunk's first row
    if (p.window > 0) {
      // chunks never straddle a 256-row block (the plan requires 256 % c == 0)
      const int64_t r = q * g.c, b = (int64_t)(pos - 1) * g.MT + r / kPairM;
      const int64_t slot = b % p.window;
      if (credit && b >= p.window && b != ready_block) {
        // On a timeout the item is skipped (its chunk never becomes ready and
        // its readers report the failure); the warp keeps drawing tickets so
        // that it still draws exactly one failing ticket.
        if (!wait_slot(p, slot, window_target(g, p.window, b, p.credit_epoch), lane)) continue;
        ready_block = b;
      }
      drow = slot * kPairM + r % kPairM;
    }
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.staging) + drow * g.K * 2);
    if (kI8)
      warp_widen16(src + v0, dst + 2 * v0, v1 - v0, lane);
    else
      warp_copy16(src + v0, dst + v0, v1 - v0, lane);
    // the warp barrier orders every lane's stores before lane 0's release
    // (release is cumulative), which publishes them at GPU scope
    __syncwarp();
    if (lane == 0) {
      const int64_t ci = (int64_t)(pos - 1) * g.Q + q;
      if constexpr (kTrace) trace_emit(p.trace, tn, threadIdx.x >> 5, kTrLanded, static_cast<uint32_t>(ci), i);
      red_release_gpu_add(p.counters + ci, 1u);
    }
  }
}

// ------------------------------------------------------------------ work items
// A pair's items: first the items dealt round-robin -- pair k takes items
// k, k + pairs, ... below static_items -- then items handed out at run time.
// The dealt items wait on no other pair (whole tiles of plain staging, the
// local shard's tiles of a plan with a staging window, and the fp16 / bf16
// split parts, which add into C blocks that ticketed tasks zero), so they
// need no coordination; the rest -- the int8 split parts of the last round's
// tiles, and the remote tiles when a staging window's credits tie tiles to
// one another -- are drawn from a grid-wide ticket counter in schedule
// order.  Whichever pairs are resident therefore always take the lowest items
// left: no item waits on a pair that has not started (the window's credits
// and an int8 split tile's partial sums come only from items drawn earlier),
// even when fewer pairs are resident than were launched.
//
// The even CTA's TMA warp (lane 1) draws the tickets and publishes the drawn
// items, two ahead of use, in a kTq-deep ring in the shared memory of both
// CTAs of the pair.  The TMA warps and the MMA thread read the ring; the 16
// epilogue warps read it after the MMA has finished the item's first segment
// and are the ones that free a slot: by then both TMA warps and the MMA
// thread have read the item (their reads precede the loads and MMAs the
// epilogue waited for).
//
// An entry is one 64-bit word, ((n + 1) << 32) | item for entry n, stored
// with a relaxed store (into the peer's ring with st.shared::cluster) and
// polled until its tag reads n + 1: the word is its own payload, so no
// acquire is needed.  (Publishing with an mbarrier arrival at cluster scope
// instead slowed the odd CTA's next gpu-scope acquire loads -- its chunk-
// counter probes -- from ~0.55 us to ~2 us.)
struct TileRing {
  uint64_t* tag;       // this CTA's ring of tagged items
  uint64_t* empty;     // the even CTA's "read" barriers (kTqReaders arrivals)
  uint32_t empty0;     // shared::cluster address of the even CTA's empty[0]
};

struct PairItems {
  int64_t pair, pairs, n_static;  // this pair, all pairs, this pair's dealt items
  bool drawn;                     // does the plan have drawn items at all?
  __device__ __forceinline__ explicit PairItems(const FusedParams& p) {
    pair = blockIdx.x / 2;
    pairs = gridDim.x / 2;
    n_static = pair < p.static_items ? (p.static_items - pair + pairs - 1) / pairs : 0;
    drawn = p.work_items > p.static_items;
  }
  __device__ __forceinline__ bool dealt(uint32_t seq) const { return seq < n_static; }
  // Every item dealt: the pair is done after its own, with no ring traffic.
  __device__ __forceinline__ bool done(uint32_t seq) const { return !drawn && seq >= n_static; }
  __device__ __forceinline__ int64_t dealt_item(uint32_t seq) const { return pair + seq * pairs; }
  __device__ __forceinline__ uint32_t ring_index(uint32_t seq) const {
    return seq - static_cast<uint32_t>(n_static);
  }
};

// Ring entry n (the caller's single thread); `release` frees the slot.
// false on timeout/abort.
__device__ __forceinline__ bool ring_read(const TileRing& r, uint32_t n, int64_t& t,
                                          uint64_t timeout_ns, volatile int* abort,
                                          const volatile uint32_t* gstatus, bool release) {
  const uint32_t slot = n % kTq;
  const volatile uint64_t* w = r.tag + slot;
  uint64_t v = *w;
  if ((v >> 32) != n + 1u) {
    const uint64_t start = globaltimer_ns();
    for (;;) {
      __nanosleep(32);
      v = *w;
      if ((v >> 32) == n + 1u) break;
      if (*abort) return false;
      const uint64_t waited = globaltimer_ns() - start;
      if (waited > timeout_ns) return false;
      if (waited > kSlowWaitNs && gstatus && *gstatus) return false;
    }
  }
  t = static_cast<int32_t>(static_cast<uint32_t>(v));
  if (release) mbar_arrive_cluster(r.empty0 + slot * 8);
  return true;
}

// The producer's side (even CTA, lane 1 of the TMA warp).  Ticket i is item
// static_items + i; exactly one failing ticket per pair and run (a negative
// one means the counters were not reset after a failed run: take nothing).
__device__ __forceinline__ int64_t ring_item(const FusedParams& p, unsigned long long ticket) {
  const int64_t i = static_cast<int64_t>(ticket - p.tile_base);
  return (i >= 0 && p.static_items + i < p.work_items) ? p.static_items + i : -1;
}

// Publish item t as ring entry n in both CTAs' rings once the slot is free.
__device__ __forceinline__ bool ring_put(const FusedParams& p, const TileRing& r, uint32_t n,
                                         int64_t t, volatile int* abort,
                                         const volatile uint32_t* gstatus) {
  const uint32_t slot = n % kTq, ph = (n / kTq) & 1u;
  if (!mbar_wait_cluster(&r.empty[slot], ph ^ 1u, p.pipe_timeout_ns, abort, gstatus))
    return false;
  const uint64_t v = (static_cast<uint64_t>(n + 1u) << 32) |
                     static_cast<uint32_t>(static_cast<int32_t>(t));
  *reinterpret_cast<volatile uint64_t*>(r.tag + slot) = v;
  st_relaxed_cluster_u64(mapa_shared(smem_u32(r.tag + slot), 1), v);
  return true;
}

// ------------------------------------------------------------------ TMA warp
// All 32 lanes poll the counters of the chunks that the 128 rows starting at
// row0 of position `pos` read; false (and the abort flag raised) on timeout.
__device__ bool wait_chunks(const FusedParams& p, int pos, int64_t row0, int lane,
                            volatile int* abort) {
  const Geometry& g = p.g;
  int64_t q0, q1;
  if (!rows_chunks(g, row0, q0, q1)) return true;  // rows past the shard: nothing to wait for
  const uint32_t target = p.epoch * static_cast<uint32_t>(g.P);
  const uint32_t* cnt = p.counters + (int64_t)(pos - 1) * g.Q;
  bool ok = true;
  for (int64_t q = q0 + lane; q <= q1 && ok; q += 32) {
    if (ld_acquire_gpu(cnt + q) >= target) continue;
    const uint64_t deadline = globaltimer_ns() + p.timeout_ns;
    uint32_t spins = 0;
    while (ld_acquire_gpu(cnt + q) < target) {
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
  ok = __all_sync(0xffffffffu, ok);
  if (!ok && lane == 0) {
    set_status(p.status, kStatusChunkTimeout,
               (static_cast<uint32_t>(pos) << 24) | static_cast<uint32_t>(q0 & 0xFFFFFF));
    *abort = 1;
  }
  __syncwarp();
  return ok;
}

// A work item's operand sources: A rows from the local shard at row0, or the
// staging: [S-1][R][K] at (row0, pos - 1), or the window's [W][256][K] at
// (this CTA's half, slot); B's columns from xb.
struct ItemSource {
  int pos;
  int32_t y, z, xb;
};
__device__ __forceinline__ ItemSource item_source(const FusedParams& p, uint32_t rank, int pos,
                                                  int64_t mt, int64_t nt, int64_t row0,
                                                  int half) {
  const Geometry& g = p.g;
  const bool win = pos > 0 && p.window > 0;
  ItemSource s;
  s.pos = pos;
  s.y = win ? static_cast<int32_t>(rank * kBlockM) : static_cast<int32_t>(row0);
  s.z = win ? static_cast<int32_t>(static_cast<uint32_t>((pos - 1) * g.MT + mt) %
                                   static_cast<uint32_t>(p.window))
            : pos - 1;
  s.xb = static_cast<int32_t>(nt * g.BN + rank * half);
  return s;
}

// A remote item's wait for the chunks its 128 rows read (all lanes), with the
// trace's wait events; true when the rows may be loaded.
template <bool kTrace>
__device__ __forceinline__ bool wait_item_rows(const FusedParams& p, int pos, int64_t row0,
                                               int64_t tile, bool wait, int lane,
                                               volatile int* abort, uint32_t& tn) {
  if constexpr (kTrace) {
    int64_t q0 = 0, q1 = -1;
    const bool rows = pos > 0 && wait && rows_chunks(p.g, row0, q0, q1);
    const uint64_t aux = (static_cast<uint64_t>(pos) << 48) |
                         (static_cast<uint64_t>(q0 & 0xFFFFFF) << 24) |
                         static_cast<uint64_t>(q1 & 0xFFFFFF);
    if (rows && lane == 0) trace_emit(p.trace, tn, threadIdx.x >> 5, kTrWaitStart, static_cast<uint32_t>(tile), aux);
    if (pos > 0 && wait && !wait_chunks(p, pos, row0, lane, abort)) return false;
    if (rows && lane == 0) trace_emit(p.trace, tn, threadIdx.x >> 5, kTrWaitEnd, static_cast<uint32_t>(tile), aux);
    return true;
  } else {
    return !(pos > 0 && wait && !wait_chunks(p, pos, row0, lane, abort));
  }
}

// Lane 0: stream k-blocks [kbs, kbe) of an item into the ring from (stage,
// phase) on; the pair's bytes are counted on the even CTA's full barrier.
// false on timeout / abort.
struct RingPos {
  int stage;
  uint32_t phase, issued, issued_phase;  // issued bit s: stage s used; its last parity
};
__device__ __forceinline__ bool issue_kblocks(const FusedParams& p, uint32_t rank, uint8_t* sA,
                                              uint8_t* sB, uint64_t* full, uint64_t* empty,
                                              const ItemSource& src, int64_t kbs, int64_t kbe,
                                              RingPos& r, volatile int* abort) {
  const int half = p.g.BN / 2;
  const uint32_t pair_tx = static_cast<uint32_t>(2 * (kABytes + half * kBlockK * 2));
  const uint32_t full0 = mapa_shared(smem_u32(full), 0);  // the even CTA's barriers
  for (int64_t kb = kbs; kb < kbe; ++kb) {
    if (!mbar_wait(&empty[r.stage], r.phase ^ 1u, p.pipe_timeout_ns, abort, p.status)) return false;
    const uint32_t bar = full0 + r.stage * 8;
    if (rank == 0) mbar_arrive_expect_tx(&full[r.stage], pair_tx);
    const int32_t x = static_cast<int32_t>(kb * kBlockK);
    uint8_t* a_dst = sA + r.stage * kABytes;
    if (src.pos == 0)
      tma_load_2d_pair(a_dst, &p.tm_a_local, bar, x, src.y);
    else
      tma_load_3d_pair(a_dst, &p.tm_a_stage, bar, x, src.y, src.z);
    uint8_t* b_dst = sB + r.stage * kBBytes;
    // One TMA instruction per operand and k-block where possible: the TMA
    // unit's per-instruction cost, not bandwidth, limits the ring on GB300.
    if (p.b3d)
      tma_load_3d_pair(b_dst, &p.tm_b, bar, 0, x, src.xb / 64);
    else
      for (int i = 0; i < half / 64; ++i)
        tma_load_2d_pair(b_dst + i * (64 * kBlockK * 2), &p.tm_b, bar, src.xb + i * 64, x);
    r.issued |= 1u << r.stage;
    r.issued_phase = (r.issued_phase & ~(1u << r.stage)) | (r.phase << r.stage);
    if (++r.stage == kStages) {
      r.stage = 0;
      r.phase ^= 1u;
    }
  }
  return true;
}

template <bool kI8, bool kTrace>
__device__ void tma_warp(const FusedParams& p, uint32_t rank, uint8_t* sA, uint8_t* sB,
                         uint64_t* full, uint64_t* empty, const TileRing& ring, int lane,
                         volatile int* abort) {
  const Geometry& g = p.g;
  [[maybe_unused]] uint32_t tn = 0;  // trace events of this warp
  const volatile uint32_t* gstatus = p.status;
  const bool wait = (p.flags & kFlagWait) != 0;
  const int half = g.BN / 2;                                   // B columns this CTA stages
  RingPos r{0, 0u, 0u, 0u};
  if (lane == 0) {
    tma_prefetch_desc(&p.tm_a_local);
    tma_prefetch_desc(&p.tm_a_stage);
    tma_prefetch_desc(&p.tm_b);
  }
  bool ok = true;
  const PairItems items(p);
  // Even CTA, lane 1: ring entries published so far, and whether the end
  // marker (-1) is among them.  Entries go out two ahead of use: while item
  // seq runs, entries up to seq + 2 - n_static are drawn.
  int64_t published = 0;
  bool drawn_all = false;
  if (rank == 0 && lane == 1 && items.drawn && items.n_static == 0) {
    // a pair with no dealt item publishes its first item before any load
    // (one ticket: every pair takes exactly one failing ticket per run, the
    // count the host advances the ticket base by); the loop below keeps two
    // entries ahead from the first item on
    const int64_t t = ring_item(p, atomicAdd(p.tile_counter, 1ull));
    ok = ring_put(p, ring, 0u, t, abort, gstatus);
    published = 1;
    drawn_all = t < 0;
  }
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 1) != 0;
  for (uint32_t seq = 0; ok && !items.done(seq); ++seq) {
    int64_t t = -1;
    bool got = true;
    if (items.dealt(seq)) {
      t = items.dealt_item(seq);
    } else if (lane == 0) {
      got = ring_read(ring, items.ring_index(seq), t, p.pipe_timeout_ns, abort, gstatus, false);
    }
    got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
    t = __shfl_sync(0xffffffffu, t, 0);
    // lane 1 of the even CTA draws one more ticket during this item?
    const bool draw = rank == 0 && items.drawn &&
                      __shfl_sync(0xffffffffu,
                                  (!drawn_all && published < static_cast<int64_t>(seq) + 3 -
                                                                 items.n_static) ? 1 : 0,
                                  1) != 0;
    if (!got) {
      ok = false;
      break;
    }
    if (t < 0) break;
    // work item t: tile `tile`, k-blocks [kbs, kbe) (the whole K unless the tile is split)
    int64_t tile, kbs, kbe;
    int part, parts;
    work_item(g, p.full_tiles, p.split, t, tile, part, parts, kbs, kbe);
    int pos;
    int64_t mt, nt;
    tile_coords(g, tile, pos, mt, nt);
    const int64_t row0 = mt * kPairM + rank * kBlockM;
    if (!wait_item_rows<kTrace>(p, pos, row0, tile, wait, lane, abort, tn)) break;
    unsigned long long ticket = 0;
    if (lane == 1 && draw) ticket = atomicAdd(p.tile_counter, 1ull);
    if (lane == 0) {
      if (pos > 0) {
        fence_acq_rel_gpu();
        fence_proxy_async_global();
      }
      ok = issue_kblocks(p, rank, sA, sB, full, empty, item_source(p, rank, pos, mt, nt, row0, half),
                         kbs, kbe, r, abort);
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (lane == 1 && ok && draw) {
      const int64_t ahead = ring_item(p, ticket);
      ok = ring_put(p, ring, static_cast<uint32_t>(published), ahead, abort, gstatus);
      ++published;
      drawn_all = ahead < 0;
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 1) != 0;
  }
  if (lane == 0) {
    if (!ok) {
      set_status(p.status, kStatusPipelineTimeout, 0x100u | rank);
      *abort = 1;
    }
    if (rank == 0) {
      // Drain: every load counted on this CTA's barriers must have landed
      // (the peer's bytes are counted here too) before the pair exits.
      volatile int never = 0;
      const uint64_t limit = ok ? p.pipe_timeout_ns : 20000000ull;
      for (int s = 0; s < kStages; ++s)
        if (r.issued & (1u << s)) mbar_wait(&full[s], (r.issued_phase >> s) & 1u, limit, &never);
    }
  }
  __syncwarp();
}

// Two producers for a plan whose tiles are all dealt (fp16 / bf16 kernel):
// producer 0 (warp 0) streams the pair's items 0, 2, 4, ..., producer 1 (the
// extra warp) items 1, 3, 5, ...  Each decodes its next item and waits for
// its chunks while the other streams, so a tile boundary no longer stalls the
// ring for the decode, the chunk wait and the fences.  A producer issues an
// item's first k-block only after the other has issued all of the previous
// item (a hand-off barrier per producer), so every stage's uses stay in
// order and each empty-barrier parity wait sees at most one pending use.
// Item seq's k-blocks occupy the ring from the global block that follows
// every earlier item's: KB per whole tile, a tail part's K share after them
// (the pair's whole tiles come first among its dealt items).
template <bool kI8, bool kTrace>
__device__ void tma_warp_dealt(const FusedParams& p, uint32_t rank, uint8_t* sA, uint8_t* sB,
                               uint64_t* full, uint64_t* empty, uint64_t* hand, int producer,
                               int lane, volatile int* abort) {
  const Geometry& g = p.g;
  [[maybe_unused]] uint32_t tn = 0;  // trace events of this warp
  const volatile uint32_t* gstatus = p.status;
  const bool wait = (p.flags & kFlagWait) != 0;
  const int half = g.BN / 2;
  if (lane == 0) {
    tma_prefetch_desc(&p.tm_a_local);
    tma_prefetch_desc(&p.tm_a_stage);
    tma_prefetch_desc(&p.tm_b);
  }
  const PairItems items(p);
  const uint64_t KB = static_cast<uint64_t>(g.KB);
  // this pair's whole tiles: items pair, pair + pairs, ... below full_tiles
  // (32-bit: a plan has fewer than 2^30 tiles)
  const uint32_t pairs32 = static_cast<uint32_t>(items.pairs);
  const uint32_t pair32 = static_cast<uint32_t>(items.pair);
  const uint32_t full32 = static_cast<uint32_t>(p.full_tiles);
  const uint32_t n_whole = pair32 < full32 ? (full32 - pair32 + pairs32 - 1) / pairs32 : 0u;
  bool ok = true;
  uint32_t handoffs = 0;  // items of the other producer waited for
  RingPos r{0, 0u, 0u, 0u};
  for (uint32_t seq = static_cast<uint32_t>(producer); ok && items.dealt(seq); seq += 2) {
    const int64_t t = items.dealt_item(seq);
    int64_t tile, kbs, kbe;
    int part, parts;
    work_item(g, p.full_tiles, p.split, t, tile, part, parts, kbs, kbe);
    int pos;
    int64_t mt, nt;
    tile_coords(g, tile, pos, mt, nt);
    const int64_t row0 = mt * kPairM + rank * kBlockM;
    if (!wait_item_rows<kTrace>(p, pos, row0, tile, wait, lane, abort, tn)) {
      ok = false;
      break;
    }
    if (lane == 0) {
      if (pos > 0) {
        fence_acq_rel_gpu();
        fence_proxy_async_global();
      }
      // the other producer has issued every k-block of item seq - 1
      if (seq > 0) {
        ok = mbar_wait(&hand[producer ^ 1], handoffs & 1u, p.pipe_timeout_ns, abort, gstatus);
        ++handoffs;
      }
      // item seq's k-blocks start at global ring block g0
      uint64_t g0 = static_cast<uint64_t>(seq < n_whole ? seq : n_whole) * KB;
      for (uint32_t j = n_whole; j < seq; ++j) {
        int64_t tj, kj0, kj1;
        int pj, nj;
        work_item(g, p.full_tiles, p.split, items.dealt_item(j), tj, pj, nj, kj0, kj1);
        g0 += static_cast<uint64_t>(kj1 - kj0);
      }
      r.stage = static_cast<int>(g0 % kStages);
      r.phase = static_cast<uint32_t>((g0 / kStages) & 1u);
      if (ok)
        ok = issue_kblocks(p, rank, sA, sB, full, empty,
                           item_source(p, rank, pos, mt, nt, row0, half), kbs, kbe, r, abort);
      if (ok) mbar_arrive(&hand[producer]);  // item seq is issued
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  }
  if (lane == 0 && !ok) {
    set_status(p.status, kStatusPipelineTimeout, 0x600u | (static_cast<uint32_t>(producer) << 4) | rank);
    *abort = 1;
    if (rank == 0) {
      // Loads counted on this CTA's barriers must land before the pair
      // exits (bounded: a stage reused by the other producer may be a phase on).
      volatile int never = 0;
      for (int s = 0; s < kStages; ++s)
        if (r.issued & (1u << s)) mbar_wait(&full[s], (r.issued_phase >> s) & 1u, 20000000ull, &never);
    }
  }
  __syncwarp();
}

// ------------------------------------------------------------------ MMA warp (even CTA)
template <bool kI8>
__device__ void mma_warp(const FusedParams& p, const uint8_t* sA, const uint8_t* sB,
                         uint64_t* full, uint64_t* empty, uint64_t* tfull, uint64_t* tempty,
                         const TileRing& ring, uint32_t tmem, volatile int* abort) {
  const Geometry& g = p.g;
  const volatile uint32_t* gstatus = p.status;
  const uint32_t idesc = idesc_f16_f32(kPairM, g.BN, /*a_mn=*/false, /*b_mn=*/true) |
                         (p.bf16 ? kIdescAbBf16 : 0u);
  const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
  // bounded staging, pipelined launch: credit the slot a remote tile read
  const bool credit = p.window > 0 && (p.flags & kFlagWait) != 0;
  int stage = 0;
  uint32_t phase = 0, unit = 0;
  bool ok = true;
  const PairItems items(p);
  for (uint32_t seq = 0; ok && !items.done(seq); ++seq) {
    int64_t t = -1;
    if (items.dealt(seq)) {
      t = items.dealt_item(seq);
    } else if (!ring_read(ring, items.ring_index(seq), t, p.pipe_timeout_ns, abort, gstatus,
                          false)) {
      ok = false;
      break;
    }
    if (t < 0) {
      // no more items: complete one more accumulator phase without MMAs, so
      // that the epilogue, which reads the ring only after an accumulator is
      // ready, can read the end marker
      const uint32_t buf = unit & 1u, use = unit >> 1;
      if (!mbar_wait(&tempty[buf], (use & 1u) ^ 1u, p.pipe_timeout_ns, abort, gstatus)) {
        ok = false;
        break;
      }
      tc_fence_after();
      mma_commit_pair_both(&tfull[buf]);
      break;
    }
    int64_t tile, kbs, kbe;
    int part, parts;
    work_item(g, p.full_tiles, p.split, t, tile, part, parts, kbs, kbe);
    // fp32 accumulation spans the whole item (fp16), or segments of kSegBlocks (int8)
    const int64_t seg_len = kI8 ? kSegBlocks : kbe - kbs;
    // (no 64-bit division at the item boundary: kSegBlocks is a power of two)
    const int64_t nseg = kI8 ? (kbe - kbs + kSegBlocks - 1) / kSegBlocks : 1;
    int64_t slot = -1;  // the window slot this remote tile reads (bounded staging)
    if (credit) {
      int pos;
      int64_t mt, nt;
      tile_coords(g, tile, pos, mt, nt);
      if (pos > 0)
        slot = static_cast<uint32_t>((pos - 1) * g.MT + mt) % static_cast<uint32_t>(p.window);
    }
    for (int64_t seg = 0; seg < nseg && ok; ++seg) {
      const uint32_t buf = unit & 1u, use = unit >> 1;
      if (!mbar_wait(&tempty[buf], (use & 1u) ^ 1u, p.pipe_timeout_ns, abort, gstatus)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem + buf * 256u;
      const int64_t kb0 = kbs + seg * seg_len;
      const int64_t kb1 = kb0 + seg_len < kbe ? kb0 + seg_len : kbe;
      for (int64_t kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&full[stage], phase, p.pipe_timeout_ns, abort, gstatus)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t as = a0 + stage * kABytes, bs = b0 + stage * kBBytes;
#pragma unroll
        for (int k = 0; k < kBlockK / kUmmaK; ++k) {
          // A: K-major, 128B swizzle: 8-row groups 1024 B apart; a 16-element
          // K slice is 32 B further along the swizzled row.  Rows 0..127 come
          // from this CTA, rows 128..255 from the peer (same offset).
          const uint64_t ad = smem_desc_sw128(as + k * (kUmmaK * 2), 16, 1024);
          // B: MN-major, 128B swizzle: 64-column groups 8 KB apart (LBO),
          // 8-k-row groups 1024 B apart (SBO); a 16-row K slice is 2 KB on.
          // Columns 0..BN/2-1 come from this CTA, the rest from the peer.
          const uint64_t bd = smem_desc_sw128(bs + k * (kUmmaK * 128), 64 * kBlockK * 2, 1024);
          mma_f16_pair(d, ad, bd, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
        }
        mma_commit_pair_both(&empty[stage]);  // frees this stage in both CTAs
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (slot >= 0 && seg == nseg - 1) {
        // The tile's last k-block of both CTAs' rows has landed (the pair's
        // bytes are counted on the full barrier): the staged rows are no
        // longer read.  (Kept out of the k-block loop: code there, even when
        // not taken, slows the MMA issue.)
        fence_proxy_async_global();
        red_release_gpu_add(p.credits + slot, 1u);
      }
      mma_commit_pair_both(&tfull[buf]);  // accumulator ready for both epilogues
      ++unit;
    }
  }
  if (!ok) {
    set_status(p.status, kStatusPipelineTimeout, 0x200u);
    *abort = 1;
  }
}

// ------------------------------------------------------------------ epilogue
__device__ __forceinline__ void st_v4(void* ptr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// An int8 split tile's last part: lane 0 waits (bounded) until every warp of
// the earlier parts has stored its partial sums; then every lane acquires the
// flag, which orders its reads of the partials after those stores.
__device__ bool wait_parts(const FusedParams& p, int64_t tail, uint32_t rank, int lane,
                           volatile int* abort) {
  const uint32_t* flag = p.part_flags + tail;
  bool ok = true;
  if (lane == 0 && ld_acquire_gpu(flag) < p.part_target) {
    const uint64_t deadline = globaltimer_ns() + p.pipe_timeout_ns;
    uint32_t spins = 0;
    while (ld_acquire_gpu(flag) < p.part_target) {
      __nanosleep(128);
      if (++spins == 16) {
        spins = 0;
        if (*abort || *reinterpret_cast<volatile uint32_t*>(p.status) != 0u ||
            globaltimer_ns() > deadline) {
          ok = false;
          break;
        }
      }
    }
    if (!ok) {
      set_status(p.status, kStatusPipelineTimeout, 0x500u | rank);
      *abort = 1;
    }
  }
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  if (ok) (void)ld_acquire_gpu(flag);
  return ok;
}

// An earlier part has stored this warp's share of its partial sums: the warp
// barrier orders every lane's stores before lane 0's (cumulative) release.
__device__ __forceinline__ void signal_part(const FusedParams& p, int64_t tail, int lane) {
  __syncwarp();
  if (lane == 0) red_release_gpu_add(p.part_flags + tail, 1u);
}

// fp16 split plan: zero the C blocks of the tail tiles, into which both
// K-parts of each tile add with TMA reductions (two fp32 additions onto +0
// give the same sum in either order).  A task is 32 rows of a tail tile over
// all its columns, stored from this warp's staging box filled with zeros.
// Tasks are drawn by ticket; this run's tickets start at zero_base (the
// counter is first raised to it).  A warp draws one ticket, or -- before it
// waits for the zeros itself -- every ticket left (it draws at most twice a
// run, so at most two of its tickets fail), so the resident CTAs zero them
// all whichever CTAs run.  The warp counts the tasks it did once their
// stores are performed.
__device__ void zero_tail_tiles(const FusedParams& p, uint8_t* box, int lane, bool all) {
  const Geometry& g = p.g;
  uint4* row = reinterpret_cast<uint4*>(box + lane * 128);
#pragma unroll
  for (int c = 0; c < 8; ++c) row[c] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_shared();
  __syncwarp();
  constexpr uint32_t kGroups = kPairM / 32;  // 32-row groups of a pair tile
  uint32_t done = 0;
  if (lane == 0) atomicMax(p.zero_ticket, p.zero_base);
  for (;;) {
    unsigned long long ticket = 0;
    if (lane == 0) ticket = atomicAdd(p.zero_ticket, 1ull) - p.zero_base;
    ticket = __shfl_sync(0xffffffffu, ticket, 0);
    if (ticket >= static_cast<unsigned long long>(p.zero_tasks)) break;
    if (lane == 0) {
      const uint32_t tk = static_cast<uint32_t>(ticket);
      const int64_t tile = p.full_tiles + tk / kGroups;
      int pos;
      int64_t mt, nt;
      tile_coords(g, tile, pos, mt, nt);
      const int src = source_of(g, p.local, pos);
      const int64_t r0 = mt * kPairM + (tk % kGroups) * 32;
      if (r0 < g.R)
        for (int b = 0; b < g.BN / 32; ++b) {
          const int64_t n0 = nt * g.BN + b * 32;
          if (n0 >= g.N) break;
          tma_store_3d(&p.tm_c, box, static_cast<int32_t>(n0), static_cast<int32_t>(r0), src);
        }
      bulk_commit_group();
    }
    ++done;
    if (!all) break;
  }
  if (lane == 0 && done > 0) {
    bulk_wait_group_all();       // the zeros are written
    fence_proxy_async_global();  // (async-proxy writes, ordered before the release)
    red_release_gpu_add(p.zero_done, done);
  }
  __syncwarp();
}

// A split tile's first reduction waits (bounded) until this run's zero tasks
// are all done; lane 0 then orders its TMA reductions after the zeros.
__device__ bool wait_zeroed(const FusedParams& p, uint32_t rank, int lane, volatile int* abort) {
  bool ok = true;
  if (lane == 0) {
    if (ld_acquire_gpu(p.zero_done) < p.zero_target) {
      const uint64_t deadline = globaltimer_ns() + p.pipe_timeout_ns;
      uint32_t spins = 0;
      while (ld_acquire_gpu(p.zero_done) < p.zero_target) {
        __nanosleep(128);
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
    if (ok) {
      fence_proxy_async_global();
    } else {
      set_status(p.status, kStatusPipelineTimeout, 0x700u | rank);
      *abort = 1;
    }
  }
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

template <bool kI8, bool kTrace, bool kSplit>
__device__ void epilogue_warp(const FusedParams& p, uint32_t rank, int quad, int half, int lane,
                              uint64_t* tfull, uint64_t* tempty, const TileRing& ring,
                              uint32_t tmem, uint8_t* sEpi, volatile int* abort) {
  const Geometry& g = p.g;
  [[maybe_unused]] uint32_t tn = 0;  // trace events of this warp
  const volatile uint32_t* gstatus = p.status;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
  const uint32_t tempty0 = mapa_shared(smem_u32(tempty), 0);  // the even CTA's barriers
  const int nchunks = g.BN / 64;                      // 32-column chunks in this warp's half
  const int chunk0 = half * nchunks;
  uint8_t* box = sEpi + (half * 4 + quad) * kEpiBoxBytes;  // this warp's staging box
  // int8: the running int32 sums of this thread's row over the warp's columns
  // (at most 4 chunks of 32), kept in registers across the tile's segments
  uint32_t sums[kI8 ? 128 : 1];
  uint32_t unit = 0;
  // fp16 split plan: the warp draws one zero task after its last whole tile
  // (while its pair computes a tail part, or as the pair finishes; at the end
  // if it had no item), and every task left before its first reduction, so
  // that it never waits for a task no running warp holds (fewer pairs may be
  // resident than were launched).  All pairs thus zero the tail tiles, about
  // one task per warp, while the parts are computed, and no zeroing competes
  // with the full rounds' loads (measured: zeroing after the first item
  // slowed the next two rounds by ~2 us; only the pairs without a part,
  // zeroing after their last item, took ~7 us); `zeroed`: this run's zero
  // tasks seen done
  bool drew = true, zeroed = true;
  if constexpr (kSplit && !kI8) {
    drew = p.zero_tasks <= 0;
    zeroed = drew;
  }
  const PairItems items(p);
  for (uint32_t seq = 0; !items.done(seq); ++seq) {
    int64_t t = -1;
    bool got = true;
    if (items.dealt(seq)) {
      t = items.dealt_item(seq);
    } else {
      // a drawn item: read it (and free its slot) once its first accumulator
      // is ready -- or the MMA's closing phase, if there is no item left
      const uint32_t buf = unit & 1u, use = unit >> 1;
      got = mbar_wait(&tfull[buf], use & 1u, p.pipe_timeout_ns, abort, gstatus);
      if (lane == 0 && got)
        got = ring_read(ring, items.ring_index(seq), t, p.pipe_timeout_ns, abort, gstatus, true);
      got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
      t = __shfl_sync(0xffffffffu, t, 0);
    }
    if (!got) {
      if (lane == 0) {
        set_status(p.status, kStatusPipelineTimeout, 0x400u | rank);
        *abort = 1;
        bulk_wait_group_all();
      }
      return;
    }
    if (t < 0) break;
    int64_t tile, kbs, kbe;
    int part, parts;
    work_item(g, p.full_tiles, p.split, t, tile, part, parts, kbs, kbe);
    // (no 64-bit division at the item boundary: kSegBlocks is a power of two)
    const int64_t nseg = kI8 ? (kbe - kbs + kSegBlocks - 1) / kSegBlocks : 1;
    // a split tile (compiled only into the kernel a splitting plan launches:
    // the split paths would raise the register count of every tile's
    // epilogue): int8 -- earlier parts store partial sums, the last part adds
    // them; fp16 -- every part adds its sums into the zeroed C block
    const bool store_part = kI8 && kSplit && parts > 1 && part < parts - 1;
    const bool add_parts = kI8 && kSplit && parts > 1 && part == parts - 1;
    const bool reduce = !kI8 && kSplit && parts > 1;
    const int64_t tail = tile - p.full_tiles;
    // int8: partial sums of part j of this tail tile, laid out for this warp: 16-byte
    // vector c of every lane of the warp is contiguous (512 bytes), so each
    // store and load of the warp moves whole lines.  Vector c (c < BN / 8) of
    // a lane holds its row's columns 4c .. 4c + 3 of the warp's half of the
    // tile; a (tile, part) takes 2 CTAs x 8 warps x BN / 8 x 32 lanes x 16 B
    // = 2 x 128 rows x BN x 4 bytes, the size the plan allocates per part.
    // (part j's vector c of this lane: base + j * part_stride + c * 32)
    const int64_t vecs = g.BN / 8;
    const int64_t part_stride = 2 * kEpiWarps * vecs * 32;
    uint4* const part_base =
        kI8 && parts > 1 ? static_cast<uint4*>(p.partials) +
                        ((((tail * (p.split - 1)) * 2 + rank) * kEpiWarps + half * 4 + quad) * vecs *
                             32 + lane)
                  : nullptr;
    auto part_vec = [&](int j, int c) -> uint4* { return part_base + j * part_stride + c * 32; };
    int pos;
    int64_t mt, nt;
    tile_coords(g, tile, pos, mt, nt);
    const int src = source_of(g, p.local, pos);
    const int64_t r = mt * kPairM + rank * kBlockM + quad * 32 + lane;
    const bool row_ok = r < g.R;
    const int64_t grow = static_cast<int64_t>(src) * g.R + r;
    for (int64_t seg = 0; seg < nseg; ++seg) {
      const uint32_t buf = unit & 1u, use = unit >> 1;
      if (!mbar_wait(&tfull[buf], use & 1u, p.pipe_timeout_ns, abort, gstatus)) {
        if (lane == 0) {
          set_status(p.status, kStatusPipelineTimeout, 0x300u | rank);
          *abort = 1;
          bulk_wait_group_all();
        }
        return;
      }
      tc_fence_after();
      if constexpr (kTrace)
        if (quad == 0 && half == 0 && lane == 0 && seg == nseg - 1)
          trace_emit(p.trace, tn, threadIdx.x >> 5, kTrAccReady, static_cast<uint32_t>(tile),
                     static_cast<uint64_t>(part) | (static_cast<uint64_t>(parts) << 8));
      // Called once this warp has read its last accumulator column of the
      // unit: the pair leader's MMA may then overwrite the buffer while this
      // warp finishes converting and storing.
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0)
            mbar_arrive(&tempty[buf]);
          else
            mbar_arrive_cluster(tempty0 + buf * 8);
        }
      };
      if constexpr (!kI8) {
        // 32 rows (one per lane) x 32 columns at a time: registers -> swizzled
        // shared box -> one TMA store of 32 full 128-byte row segments.  Rows
        // past the shard and columns past N are clipped by the descriptor.
        const int64_t r0 = mt * kPairM + rank * kBlockM + quad * 32;
        if (reduce && !zeroed) {
          // every task left, unless they are all done already (as they are
          // when every pair runs: 1000 warps drawing at once cost ~2 us)
          uint32_t all_done = 0;
          if (lane == 0) all_done = ld_acquire_gpu(p.zero_done) >= p.zero_target ? 1u : 0u;
          if (__shfl_sync(0xffffffffu, all_done, 0) == 0u) {
            if (lane == 0) bulk_wait_group_read<0>();  // the box is no longer read
            __syncwarp();
            zero_tail_tiles(p, box, lane, true);
          }
          drew = true;
          if (!wait_zeroed(p, rank, lane, abort)) {
            if (lane == 0) bulk_wait_group_all();
            return;
          }
          zeroed = true;
          if constexpr (kTrace)
            if (quad == 0 && half == 0 && lane == 0)
              trace_emit(p.trace, tn, threadIdx.x >> 5, kTrPartsReady, static_cast<uint32_t>(tile), 0);
        }
        for (int jj = 0; jj < nchunks; ++jj) {
          const int j = chunk0 + jj;
          uint32_t v[32];
          tmem_ld32(lane_base + buf * 256u + j * 32, v);
          tmem_ld_wait();
          if (jj == nchunks - 1) release();
          const int64_t n0 = nt * g.BN + j * 32;
          if (r0 >= g.R || n0 >= g.N) continue;  // warp-uniform: nothing of this box exists
          if (lane == 0) bulk_wait_group_read<0>();  // the previous store has read the box
          __syncwarp();
          uint8_t* row = box + lane * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t off = static_cast<uint32_t>((c ^ (lane & 7)) * 16);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(row + off)),
                         "r"(v[4 * c]), "r"(v[4 * c + 1]), "r"(v[4 * c + 2]), "r"(v[4 * c + 3])
                         : "memory");
          }
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) {
            if (reduce)
              tma_reduce_add_3d(&p.tm_c, box, static_cast<int32_t>(n0), static_cast<int32_t>(r0), src);
            else
              tma_store_3d(&p.tm_c, box, static_cast<int32_t>(n0), static_cast<int32_t>(r0), src);
            bulk_commit_group();
          }
        }
      } else {
        const bool first = seg == 0, last = seg == nseg - 1;
        // fp32 partials (exact integers) -> int32, added to the running sums;
        // 16 columns per TMEM load keep the sums in registers
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          if (jj < nchunks) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t f[16];
              tmem_ld16(lane_base + buf * 256u + (chunk0 + jj) * 32 + hh * 16, f);
              tmem_ld_wait();
              if (jj == nchunks - 1 && hh == 1) release();
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const uint32_t v = static_cast<uint32_t>(__float2int_rn(__uint_as_float(f[e])));
                sums[jj * 32 + hh * 16 + e] = first ? v : sums[jj * 32 + hh * 16 + e] + v;
              }
            }
          }
        }
        if (last && store_part) {
          // this part's exact int32 sums of the thread's row
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (c < nchunks * 8)
              *part_vec(part, c) =
                  make_uint4(sums[4 * c], sums[4 * c + 1], sums[4 * c + 2], sums[4 * c + 3]);
          signal_part(p, tail, lane);
        }
        if (last && add_parts) {
          if (!wait_parts(p, tail, rank, lane, abort)) {
            if (lane == 0) bulk_wait_group_all();
            return;
          }
          if constexpr (kTrace)
            if (quad == 0 && half == 0 && lane == 0)
              trace_emit(p.trace, tn, threadIdx.x >> 5, kTrPartsReady, static_cast<uint32_t>(tile), 0);
          // integer sums: exact in any order; 8 vectors in flight at a time
          for (int pj = 0; pj < parts - 1; ++pj) {
#pragma unroll
            for (int c0 = 0; c0 < 32; c0 += 8) {
              if (c0 >= nchunks * 8) break;
              uint4 x[8];
#pragma unroll
              for (int c = 0; c < 8; ++c) x[c] = __ldcg(part_vec(pj, c0 + c));
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                sums[4 * (c0 + c)] += x[c].x;
                sums[4 * (c0 + c) + 1] += x[c].y;
                sums[4 * (c0 + c) + 2] += x[c].z;
                sums[4 * (c0 + c) + 3] += x[c].w;
              }
            }
          }
        }
        if (last && row_ok && !store_part) {
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            if (jj >= nchunks) continue;
            const int64_t n0 = nt * g.BN + (chunk0 + jj) * 32;
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              if (n0 + e >= g.N) continue;
              const int4 b0 = __ldg(reinterpret_cast<const int4*>(p.bias + n0 + e));
              const int4 b1 = __ldg(reinterpret_cast<const int4*>(p.bias + n0 + e + 4));
              const float4 s0 = __ldg(reinterpret_cast<const float4*>(p.scale + n0 + e));
              const float4 s1 = __ldg(reinterpret_cast<const float4*>(p.scale + n0 + e + 4));
              const int32_t bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
              const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
              uint32_t c[8];
              uint32_t h[4];
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const int32_t cv =
                    static_cast<int32_t>(sums[jj * 32 + e + u] + static_cast<uint32_t>(bb[u]));
                c[u] = static_cast<uint32_t>(cv);
                const float dv = __fmul_rn(__int2float_rn(cv), ss[u]);
                const uint32_t hb = __half_as_ushort(__float2half_rn(dv));
                if (u & 1)
                  h[u >> 1] |= hb << 16;
                else
                  h[u >> 1] = hb;
              }
              int32_t* cdst = p.C_i32 + grow * g.N + n0 + e;
              st_v4(cdst, c[0], c[1], c[2], c[3]);
              st_v4(cdst + 4, c[4], c[5], c[6], c[7]);
              st_v4(p.D_f16 + grow * g.N + n0 + e, h[0], h[1], h[2], h[3]);
            }
          }
        }
      }
      ++unit;
    }
    if constexpr (kTrace)
      if (quad == 0 && half == 0 && lane == 0)
        trace_emit(p.trace, tn, threadIdx.x >> 5, kTrTileDone, static_cast<uint32_t>(tile),
                   static_cast<uint64_t>(part) | (static_cast<uint64_t>(parts) << 8));
    // (every item of an fp16 split plan is dealt: the next is a tail part, or
    // there is none, once its index reaches full_tiles)
    if (!drew && items.dealt_item(seq + 1) >= p.full_tiles) {
      if (lane == 0) bulk_wait_group_read<0>();  // the box is no longer read
      __syncwarp();
      zero_tail_tiles(p, box, lane, false);
      drew = true;
    }
  }
  if (!drew) {
    if (lane == 0) bulk_wait_group_read<0>();  // the box is no longer read
    __syncwarp();
    zero_tail_tiles(p, box, lane, false);
  }
  if (lane == 0) bulk_wait_group_all();  // every C store performed before the CTA exits
  __syncwarp();
}

// ------------------------------------------------------------------ kernel
template <bool kI8, bool kTrace, bool kSplit>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(fused_threads(kI8), 1)
    ag_fused_kernel(const __grid_constant__ FusedParams p) {
  [[maybe_unused]] uint32_t tc = 0;  // trace events of the CTA slot
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint8_t* sEpi = sB + kStages * kBBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + kEpiBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* tq_tag = drain + 1;
  uint64_t* tq_empty = tq_tag + kTq;
  uint64_t* hand = tq_empty + kTq;  // the two TMA producers' "item issued" barriers
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(hand + 2);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool gemm = (p.flags & kFlagGemm) != 0;
  // A copy warp draws its first ticket before the set-up below, so the
  // atomic's latency overlaps it (tickets keep the copies live whichever CTAs
  // are resident).
  const bool copier = warp >= 2 && warp < 2 + kCopyWarpsPerCta && (p.flags & kFlagCopy) != 0;
  unsigned long long first_ticket = 0;
  if (copier && lane == 0) first_ticket = atomicAdd(p.item_counter, 1ull);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 2 * kEpiWarps);  // the epilogue warps of both CTAs of the pair
    }
    mbar_init(drain, 1);
    mbar_init(&hand[0], 1);
    mbar_init(&hand[1], 1);
    for (int i = 0; i < kTq; ++i) {
      tq_tag[i] = 0;  // no entry yet (entry n carries the tag n + 1)
      mbar_init(&tq_empty[i], kTqReaders);
    }
    *tmem_slot = 0;
    *abort = 0;
    fence_mbar_init();
  }
  if (gemm && warp == 1) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const TileRing ring{tq_tag, tq_empty, mapa_shared(smem_u32(tq_empty), 0)};

  if constexpr (kTrace)
    if (threadIdx.x == 0) trace_emit(p.trace, tc, kTrCtaSlot, kTrCtaStart, 0, 0);
  // two TMA producers when every tile of the plan is dealt (fp16 / bf16 kernel)
  const bool two_producers = !kI8 && p.work_items == p.static_items;
  if (warp == 0) {
    if (gemm) {
      if (two_producers)
        tma_warp_dealt<kI8, kTrace>(p, rank, sA, sB, full, empty, hand, 0, lane, abort);
      else
        tma_warp<kI8, kTrace>(p, rank, sA, sB, full, empty, ring, lane, abort);
    }
  } else if (!kI8 && warp == kExtraTmaWarp) {
    if (gemm && two_producers)
      tma_warp_dealt<kI8, kTrace>(p, rank, sA, sB, full, empty, hand, 1, lane, abort);
  } else if (warp == 1) {
    if (gemm && rank == 0 && lane == 0)
      mma_warp<kI8>(p, sA, sB, full, empty, tfull, tempty, ring, tmem, abort);
  } else if (warp < 2 + kCopyWarpsPerCta) {
    if (copier) copy_warp<kI8, kTrace>(p, lane, first_ticket);
  } else {
    if (gemm)
      epilogue_warp<kI8, kTrace, kSplit>(p, rank, warp & 3, (warp - 4) >> 2, lane, tfull, tempty,
                                         ring,
                                 tmem, sEpi, abort);
  }

  tc_fence_before();
  __syncthreads();
  if (gemm && rank == 0 && warp == 1 && lane == 0) {
    // Every MMA of the pair must be complete before either CTA releases TMEM
    // or shared memory.
    mma_commit_pair_local(drain);
    volatile int never = 0;
    mbar_wait(drain, 0, p.pipe_timeout_ns, &never);
  }
  if (*abort || *reinterpret_cast<volatile uint32_t*>(p.status) != 0u) {
    // After a timeout the peer may still have TMA loads landing in this CTA's
    // shared memory that no barrier of ours counts; give them time to land.
    if (threadIdx.x == 0) __nanosleep(100000);
  }
  __syncthreads();
  tc_fence_before();
  cluster_sync();
  if (gemm && warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
  if constexpr (kTrace)
    if (threadIdx.x == 0) trace_emit(p.trace, tc, kTrCtaSlot, kTrCtaEnd, 0, 0);
}

// ------------------------------------------------------------------ int8 widening
// fp16 copies of B and of the local shard for the int8 path (exact).  Each
// thread keeps four 16-byte loads in flight before widening and storing them:
// the copy is bound by memory latency otherwise.
__global__ void __launch_bounds__(256) widen_kernel(const uint4* __restrict__ s0,
                                                    uint4* __restrict__ d0, int64_t n0,
                                                    const uint4* __restrict__ s1,
                                                    uint4* __restrict__ d1, int64_t n1) {
  constexpr int U = 4;
  const int64_t total = n0 + n1;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i0 < total;
       i0 += U * stride) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < total) v[u] = ld_nc_v4(i < n0 ? s0 + i : s1 + (i - n0));
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + u * stride;
      if (i >= total) break;
      uint4 a, b;
      widen16(v[u], a, b);
      uint4* d = i < n0 ? d0 + 2 * i : d1 + 2 * (i - n0);
      d[0] = a;
      d[1] = b;
    }
  }
}

// ------------------------------------------------------------------ launchers
template <bool kI8, bool kTrace, bool kSplit>
static const void* fused_fn_t() {
  return reinterpret_cast<const void*>(&ag_fused_kernel<kI8, kTrace, kSplit>);
}
static const void* fused_fn(int dtype, bool trace, bool split) {
  const bool i8 = dtype == 1;
  if (i8) {
    if (trace) return split ? fused_fn_t<true, true, true>() : fused_fn_t<true, true, false>();
    return split ? fused_fn_t<true, false, true>() : fused_fn_t<true, false, false>();
  }
  if (trace) return split ? fused_fn_t<false, true, true>() : fused_fn_t<false, true, false>();
  return split ? fused_fn_t<false, false, true>() : fused_fn_t<false, false, false>();
}

cudaError_t fused_max_clusters(int dtype, int grid, int* clusters) {
  for (int v = 0; v < 4; ++v) {
    cudaError_t e = cudaFuncSetAttribute(fused_fn(dtype, (v & 1) != 0, (v & 2) != 0),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
  }
  const void* fn = fused_fn(dtype, false, false);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(fused_threads(dtype == 1));
  cfg.dynamicSmemBytes = kSmemBytes;
  return cudaOccupancyMaxActiveClusters(clusters, fn, &cfg);
}

cudaError_t launch_fused(const FusedParams& p, int grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(fused_threads(p.g.dtype == 1));
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  const void* fn = fused_fn(p.g.dtype, p.trace.ev != nullptr, p.split > 1);
  void* args[] = {const_cast<FusedParams*>(&p)};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t launch_widen(const int8_t* src0, uint16_t* dst0, int64_t n0, const int8_t* src1,
                         uint16_t* dst1, int64_t n1, int grid, cudaStream_t stream) {
  widen_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const uint4*>(src0),
                                         reinterpret_cast<uint4*>(dst0), n0 / 16,
                                         reinterpret_cast<const uint4*>(src1),
                                         reinterpret_cast<uint4*>(dst1), n1 / 16);
  return cudaGetLastError();
}

}  // namespace agg
