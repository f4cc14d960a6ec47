// skinny_kernel.cu -- int8 AllGatherMatmulDequant when the gathered A has at
// most 128 rows (decode-like shapes such as 2 x 32 rows, K = 16384, N = 7168).
//
// Such a problem is bound by reading B from HBM once ("AllGather矩阵乘法反量化
// 算子设计文档", 8.3 lists the 64 x 16384 x 7168 shape): every k-block of B is
// shared by all rows, so the kernel streams B exactly once as int8, widens it
// in shared memory and runs the tensor core on it with the (tiny) A held in
// tensor memory.  sm_103a has no tcgen05 kind::i8, so the product is computed
// exactly on kind::f16: every int8 is an exact fp16, and an fp32 accumulation
// never spans more than 16 k-blocks (1024 k), which keeps every fp32 partial an
// integer below 2^24; segments are folded into an int32 sum in TMEM.
//
// B moves in 32 KB TMA boxes (128 columns x 256 k-rows, four k-blocks): a TMA
// box carries a fixed cost of several hundred cycles, and on GB300 machines of
// 8 KB cap a one-box-per-k-block stream near 2.6 TB/s while 32 KB boxes run at
// the read bandwidth of HBM.  A (at most 128 x K int8, resident in L2) is read
// straight from global memory by the A-widening warps, so it costs the TMA
// unit nothing.
//
// Work: the (128-column n-tile, 4-k-block unit) pairs, n-tile major, are cut
// into one contiguous range per CTA (stream-K), so a CTA holds at most a few
// pieces of n-tiles.  At the end of a piece its exact int32 sums (all rows x
// 128 columns) are added with coalesced red.add.s32 into an L2-resident int32
// accumulator (integer addition is exact in any order).  A small stream-ordered
// kernel (ag_skinny_finish_kernel) then adds the bias, writes C_i32 and the
// fp16 dequant D, and zeroes the accumulator for the next run.
//
// Roles (20 warps):
//   warp 6        TMA warp: streams the int8 B boxes of the CTA's range into a
//                 raw ring; B does not depend on the gathered rows, so the
//                 stream starts at once.
//   warps 0-3     B widening: raw int8 B -> fp16 in the MN-major 128-byte
//                 swizzled layout the MMA reads, one k-block per fp16 stage.
//   warps 8-11,   A widening: wait once for every remote chunk (the rows of the
//   16-19         other shards, copied by the copy warp), then per k-block load
//                 the int8 rows from the local shard or the staging workspace,
//                 widen to fp16 and tcgen05.st them into TMEM (one row per
//                 lane; the MMA's A operand comes from TMEM).  Warps w and
//                 w + 8 serve lane quadrant w % 4 and take alternate k-blocks.
//   warp 4        MMA: one thread issues tcgen05.mma (M = 128, N = 128, K = 16).
//   warp 5        copy warp: copies remote chunks into the int8 staging
//                 workspace and releases their ready counters.
//   warps 12-15   epilogue: fold fp32 segments into the int32 sums in TMEM;
//                 flush each finished piece through shared memory with red.add.

#include <cuda_fp16.h>

#include "fused_kernel.cuh"
#include "sm103.cuh"

namespace agg {

namespace {

constexpr int kSkWarps = 20;
constexpr int kSkThreads = kSkWarps * 32;
constexpr int kSkN = 128;              // n-tile
constexpr int kSkUnitBlocks = 4;       // k-blocks per B box (256 k-rows)
constexpr int kSkRaw = 4;              // raw int8 B ring stages
constexpr int kSkFp = 4;               // fp16 B stages (one k-block each)
constexpr int kSkA = 4;                // A stages in TMEM (32 columns each)
constexpr int kSkRawStage = kSkN * kBlockK * kSkUnitBlocks;  // 32 KB int8
constexpr int kSkFpStage = kSkN * kBlockK * 2;               // 16 KB fp16
constexpr int kSkTrans = 4 * 32 * 33 * 4;                    // epilogue transposes
constexpr int kSkSmem = kSkRaw * kSkRawStage + kSkFp * kSkFpStage + kSkTrans + 1024 + 1024;
constexpr uint32_t kSkAcol = 0;        // TMEM columns [0, 128): A stages
constexpr uint32_t kSkDcol = 128;      // [128, 384): two fp32 accumulators
constexpr uint32_t kSkScol = 384;      // [384, 512): int32 running sums

__device__ __forceinline__ void sk_set_status(uint32_t* status, uint32_t kind, uint32_t detail) {
  if (atomicCAS(status, 0u, kind) == 0u) atomicExch(status + 1, detail);
}

__device__ __forceinline__ void widen16x(const uint4 v, uint4& a, uint4& b) {
  i8x4_to_f16x4(v.x, a.x, a.y);
  i8x4_to_f16x4(v.y, a.z, a.w);
  i8x4_to_f16x4(v.z, b.x, b.y);
  i8x4_to_f16x4(v.w, b.z, b.w);
}

// Units: (n-tile, q) with q the 4-k-block group; KQ groups per n-tile.
__device__ __forceinline__ int64_t units_per_tile(const Geometry& g) {
  return (g.KB + kSkUnitBlocks - 1) / kSkUnitBlocks;
}

// This CTA's unit range [u0, u1) of the n-major unit space.
__device__ __forceinline__ void cta_range(const SkinnyParams& p, int64_t& u0, int64_t& u1) {
  const int64_t U = p.n_tiles * units_per_tile(p.g);
  u0 = U * blockIdx.x / gridDim.x;
  u1 = U * (blockIdx.x + 1) / gridDim.x;
}

// k-blocks [kb0, kb1) of unit u.
__device__ __forceinline__ void unit_blocks(const Geometry& g, int64_t KQ, int64_t u, int64_t& kb0,
                                            int64_t& kb1) {
  kb0 = (u % KQ) * kSkUnitBlocks;
  kb1 = kb0 + kSkUnitBlocks < g.KB ? kb0 + kSkUnitBlocks : g.KB;
}

// The piece that starts at unit u: n-tile nt, units [u, ue), k-blocks [kb0, kb1).
__device__ __forceinline__ void piece_at(const Geometry& g, int64_t KQ, int64_t u, int64_t u1,
                                         int64_t& nt, int64_t& ue, int64_t& kb0, int64_t& kb1) {
  nt = u / KQ;
  ue = (nt + 1) * KQ < u1 ? (nt + 1) * KQ : u1;
  kb0 = (u % KQ) * kSkUnitBlocks;
  const int64_t end = (ue - nt * KQ) * kSkUnitBlocks;
  kb1 = end < g.KB ? end : g.KB;
}

// Walks this CTA's k-block sequence (the k-blocks of its units in order).
struct KbWalk {
  int64_t u, u1, kb, kb1, KQ;
  __device__ __forceinline__ void start(const Geometry& g, int64_t u0_, int64_t u1_) {
    KQ = units_per_tile(g);
    u = u0_;
    u1 = u1_;
    if (u < u1) unit_blocks(g, KQ, u, kb, kb1);
  }
  __device__ __forceinline__ bool valid() const { return u < u1; }
  __device__ __forceinline__ void next(const Geometry& g) {
    if (++kb == kb1 && ++u < u1) unit_blocks(g, KQ, u, kb, kb1);
  }
};

// ------------------------------------------------------------------ copy warp
__device__ void sk_copy_warp(const SkinnyParams& p, int lane) {
  const Geometry& g = p.g;
  for (;;) {
    unsigned long long ticket = 0;
    if (lane == 0) ticket = atomicAdd(p.item_counter, 1ull);
    ticket = __shfl_sync(0xffffffffu, ticket, 0);
    const int64_t i = static_cast<int64_t>(ticket - p.item_base);
    if (i >= g.items) break;
    int pos, piece;
    int64_t q, v0, v1;
    item_coords(g, i, pos, q, piece, v0, v1);
    if (i == p.debug_skip_item) continue;
    if (p.debug_delay_ns) __nanosleep(p.debug_delay_ns);
    const uint4* src =
        reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.src[pos]) + q * g.c * g.K);
    uint4* dst = reinterpret_cast<uint4*>(p.staging + ((int64_t)(pos - 1) * g.R + q * g.c) * g.K);
    // 8 independent 16-byte loads in flight per lane
    int64_t v = v0 + lane;
    for (; v + 7 * 32 < v1; v += 8 * 32) {
      uint4 t[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) t[u] = ld_nc_v4(src + v + u * 32);
#pragma unroll
      for (int u = 0; u < 8; ++u) dst[v + u * 32] = t[u];
    }
    for (; v < v1; v += 32) dst[v] = ld_nc_v4(src + v);
    __threadfence();
    __syncwarp();
    if (lane == 0) red_release_gpu_add(p.counters + (int64_t)(pos - 1) * g.Q + q, 1u);
  }
}

// Every lane acquires a share of the ready counters; true once all chunks of
// this epoch have landed (false on timeout / abort, with the status set).
__device__ bool sk_wait_all_chunks(const SkinnyParams& p, int lane, volatile int* abort) {
  const Geometry& g = p.g;
  const int64_t total = (int64_t)(g.S - 1) * g.Q;
  const uint32_t target = p.epoch * static_cast<uint32_t>(g.P);
  bool ok = true;
  for (int64_t q = lane; q < total && ok; q += 32) {
    if (ld_acquire_gpu(p.counters + q) >= target) continue;
    const uint64_t deadline = globaltimer_ns() + p.timeout_ns;
    uint32_t spins = 0;
    while (ld_acquire_gpu(p.counters + q) < target) {
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
    sk_set_status(p.status, kStatusChunkTimeout, 0x10000u);
    *abort = 1;
  }
  __syncwarp();
  return ok;
}

// ------------------------------------------------------------------ TMA warp
__device__ void sk_tma_warp(const SkinnyParams& p, uint8_t* sRaw, uint64_t* raw_full,
                            uint64_t* raw_empty, int lane, volatile int* abort) {
  if (lane != 0) return;
  const Geometry& g = p.g;
  const volatile uint32_t* gstatus = p.status;
  const int64_t KQ = units_per_tile(g);
  int64_t u0, u1;
  cta_range(p, u0, u1);
  tma_prefetch_desc(&p.tm_b8);
  uint32_t issued = 0, issued_phase = 0;
  bool ok = true;
  for (int64_t i = 0; i < u1 - u0; ++i) {
    const int stage = static_cast<int>(i % kSkRaw);
    const uint32_t phase = static_cast<uint32_t>((i / kSkRaw) & 1);
    if (!mbar_wait(&raw_empty[stage], phase ^ 1u, p.pipe_timeout_ns, abort, gstatus)) {
      ok = false;
      break;
    }
    const int64_t u = u0 + i, nt = u / KQ, q = u % KQ;
    mbar_arrive_expect_tx(&raw_full[stage], kSkRawStage);
    tma_load_2d(sRaw + stage * kSkRawStage, &p.tm_b8, &raw_full[stage],
                static_cast<int32_t>(nt * kSkN), static_cast<int32_t>(q * kSkUnitBlocks * kBlockK));
    issued |= 1u << stage;
    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
  }
  if (!ok) {
    sk_set_status(p.status, kStatusPipelineTimeout, 0x1100u);
    *abort = 1;
    // loads already issued must land before the CTA exits
    volatile int never = 0;
    for (int s = 0; s < kSkRaw; ++s)
      if (issued & (1u << s))
        mbar_wait(&raw_full[s], (issued_phase >> s) & 1u, 20000000ull, &never);
  }
}

// ------------------------------------------------------------------ B widening (warps 0-3)
// Thread t widens 64 bytes of one k-row: k-row t / 2 of the k-block, columns
// (t % 2) * 64 .. +63 (= one 64-column swizzle group of the MN-major fp16 tile).
__device__ void sk_bwiden(const SkinnyParams& p, const uint8_t* sRaw, uint8_t* sFp,
                          uint64_t* raw_full, uint64_t* raw_empty, uint64_t* fp_full,
                          uint64_t* fp_empty, int t, volatile int* abort) {
  const Geometry& g = p.g;
  const volatile uint32_t* gstatus = p.status;
  const int krow = t >> 1, grp = t & 1, lane = t & 31;
  const int64_t KQ = units_per_tile(g);
  int64_t u0, u1;
  cta_range(p, u0, u1);
  int64_t i = 0;  // k-block sequence index
  for (int64_t j = 0; j < u1 - u0; ++j) {
    const int rs = static_cast<int>(j % kSkRaw);
    const uint32_t rph = static_cast<uint32_t>((j / kSkRaw) & 1);
    if (!mbar_wait(&raw_full[rs], rph, p.pipe_timeout_ns, abort, gstatus)) {
      if (lane == 0) {
        sk_set_status(p.status, kStatusPipelineTimeout, 0x1200u);
        *abort = 1;
      }
      return;
    }
    int64_t kb0, kb1;
    unit_blocks(g, KQ, u0 + j, kb0, kb1);
    for (int64_t b = 0; b < kb1 - kb0; ++b, ++i) {
      const int fs = static_cast<int>(i % kSkFp);
      const uint32_t fph = static_cast<uint32_t>((i / kSkFp) & 1);
      if (!mbar_wait(&fp_empty[fs], fph ^ 1u, p.pipe_timeout_ns, abort, gstatus)) {
        if (lane == 0) {
          sk_set_status(p.status, kStatusPipelineTimeout, 0x1201u);
          *abort = 1;
        }
        return;
      }
      // raw B arrives 128-byte swizzled: 16-byte chunk c of box row r sits at c ^ (r % 8)
      const int r = static_cast<int>(b) * kBlockK + krow;
      const uint8_t* src = sRaw + rs * kSkRawStage + r * kSkN;
      uint4 v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        v[k] = *reinterpret_cast<const uint4*>(src + (((grp * 4 + k) ^ (r & 7)) * 16));
      uint8_t* dst = sFp + fs * kSkFpStage + grp * (64 * kBlockK * 2) + krow * 128;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint4 a, c;
        widen16x(v[k], a, c);
        const int c0 = 2 * k, c1 = 2 * k + 1;  // 16-byte chunks of 8 fp16 within the row
        *reinterpret_cast<uint4*>(dst + ((c0 ^ (krow & 7)) * 16)) = a;
        *reinterpret_cast<uint4*>(dst + ((c1 ^ (krow & 7)) * 16)) = c;
      }
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive(&fp_full[fs]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&raw_empty[rs]);
  }
}

// ------------------------------------------------------------------ A widening
// Lane l of a warp serving quadrant q holds row m = 32 q + l: 64 int8 of the
// k-block -> 64 fp16 = 32 TMEM columns (k = 2c in the low half of column c).
__device__ __forceinline__ void sk_load_a(const uint8_t* row, int64_t K, int64_t kb, uint4 (&v)[4]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int64_t k0 = kb * kBlockK + c * 16;
    // __ldcg: the staging rows were written during this launch by other SMs
    v[c] = (row != nullptr && k0 < K) ? __ldcg(reinterpret_cast<const uint4*>(row + k0))
                                      : make_uint4(0u, 0u, 0u, 0u);
  }
}

// Widens one k-block of this lane's row (in `v`) into A stage `as` of TMEM.
__device__ __forceinline__ bool sk_store_a(const SkinnyParams& p, const uint4 (&v)[4], int64_t i,
                                           uint64_t* a_full, uint64_t* a_empty,
                                           uint32_t lane_base, int lane, volatile int* abort) {
  const int as = static_cast<int>(i % kSkA);
  const uint32_t aph = static_cast<uint32_t>((i / kSkA) & 1);
  if (!mbar_wait(&a_empty[as], aph ^ 1u, p.pipe_timeout_ns, abort, p.status)) {
    if (lane == 0) {
      sk_set_status(p.status, kStatusPipelineTimeout, 0x1300u);
      *abort = 1;
    }
    return false;
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t r[16];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      uint4 a, b;
      widen16x(v[2 * h + k], a, b);
      r[8 * k + 0] = a.x; r[8 * k + 1] = a.y; r[8 * k + 2] = a.z; r[8 * k + 3] = a.w;
      r[8 * k + 4] = b.x; r[8 * k + 5] = b.y; r[8 * k + 6] = b.z; r[8 * k + 7] = b.w;
    }
    tmem_st16(lane_base + kSkAcol + as * 32 + h * 16, r);
  }
  tmem_st_wait();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(&a_full[as]);
  return true;
}

// A warp serves the TMEM lane quadrant of its warp id (a warp reaches only the
// 32 lanes of quadrant warp % 4); the two warps of a quadrant take alternate
// k-blocks (parity `par`), which keeps every use of an A stage with one warp.
// Each warp keeps the loads of its next two k-blocks in flight, in three
// register buffers used in rotation (so no pending load is ever copied).
__device__ void sk_awiden(const SkinnyParams& p, uint64_t* a_full, uint64_t* a_empty,
                          uint32_t tmem, int quad, int par, int lane, volatile int* abort) {
  const Geometry& g = p.g;
  constexpr int kPer = 2;  // warps per quadrant
  static_assert(kSkA % kPer == 0, "A stages per warp");
  if (quad * 32 >= g.M) return;  // no rows in this quadrant (warp-uniform)
  const int m = quad * 32 + lane;
  if ((p.flags & kFlagWait) && g.S > 1 && !sk_wait_all_chunks(p, lane, abort)) return;
  const uint8_t* row = nullptr;
  if (m < g.M) {
    const int s = static_cast<int>(m / g.R);
    const int64_t r = m - static_cast<int64_t>(s) * g.R;
    const int pos = (s - p.local + g.S) % g.S;
    row = pos == 0 ? static_cast<const uint8_t*>(p.src[0]) + r * g.K
                   : reinterpret_cast<const uint8_t*>(p.staging) + ((int64_t)(pos - 1) * g.R + r) * g.K;
  }
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
  int64_t u0, u1;
  cta_range(p, u0, u1);
  const int64_t KQ = units_per_tile(g);
  int64_t nkb = 0;  // k-blocks of this CTA
  for (int64_t u = u0; u < u1; ++u) {
    int64_t kb0, kb1;
    unit_blocks(g, KQ, u, kb0, kb1);
    nkb += kb1 - kb0;
  }
  const int64_t mine = nkb > par ? (nkb - par + kPer - 1) / kPer : 0;
  KbWalk ld;  // the next k-block to load
  ld.start(g, u0, u1);
  for (int s = 0; s < par && ld.valid(); ++s) ld.next(g);
  auto advance = [&]() {
    for (int s = 0; s < kPer && ld.valid(); ++s) ld.next(g);
  };
  uint4 X[4], Y[4], Z[4];
  if (mine > 0) { sk_load_a(row, g.K, ld.kb, X); advance(); }
  if (mine > 1) { sk_load_a(row, g.K, ld.kb, Y); advance(); }
  for (int64_t t = 0; t < mine; t += 3) {
    if (t + 2 < mine) { sk_load_a(row, g.K, ld.kb, Z); advance(); }
    if (!sk_store_a(p, X, par + t * kPer, a_full, a_empty, lane_base, lane, abort)) return;
    if (t + 1 >= mine) break;
    if (t + 3 < mine) { sk_load_a(row, g.K, ld.kb, X); advance(); }
    if (!sk_store_a(p, Y, par + (t + 1) * kPer, a_full, a_empty, lane_base, lane, abort)) return;
    if (t + 2 >= mine) break;
    if (t + 4 < mine) { sk_load_a(row, g.K, ld.kb, Y); advance(); }
    if (!sk_store_a(p, Z, par + (t + 2) * kPer, a_full, a_empty, lane_base, lane, abort)) return;
  }
}

// ------------------------------------------------------------------ MMA warp
// Pieces: maximal runs of this CTA's units inside one n-tile; segments: at most
// kSegBlocks k-blocks of a piece, each accumulated into one fp32 buffer.
__device__ void sk_mma(const SkinnyParams& p, const uint8_t* sFp, uint64_t* fp_full,
                       uint64_t* fp_empty, uint64_t* a_full, uint64_t* a_empty, uint64_t* dfull,
                       uint64_t* dempty, uint32_t tmem, volatile int* abort) {
  const Geometry& g = p.g;
  const volatile uint32_t* gstatus = p.status;
  // D fp32, A fp16 from TMEM (K-major), B fp16 MN-major, M = 128, N = 128
  const uint32_t idesc = idesc_f16_f32(128, kSkN, /*a_mn=*/false, /*b_mn=*/true);
  const uint32_t b0 = smem_u32(sFp);
  const int64_t KQ = units_per_tile(g);
  int64_t u0, u1;
  cta_range(p, u0, u1);
  int64_t i = 0;     // k-block sequence index of this CTA
  uint32_t seg = 0;  // segment sequence index (accumulator buffer = seg & 1)
  bool ok = true;
  for (int64_t u = u0; u < u1 && ok;) {
    int64_t nt, ue, kb0, kb1;
    piece_at(g, KQ, u, u1, nt, ue, kb0, kb1);
    for (int64_t s0 = kb0; s0 < kb1 && ok; s0 += kSegBlocks, ++seg) {
      const int64_t s1 = s0 + kSegBlocks < kb1 ? s0 + kSegBlocks : kb1;
      const uint32_t buf = seg & 1u, use = seg >> 1;
      if (!mbar_wait(&dempty[buf], (use & 1u) ^ 1u, p.pipe_timeout_ns, abort, gstatus)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem + kSkDcol + buf * kSkN;
      for (int64_t kb = s0; kb < s1; ++kb, ++i) {
        const int fs = static_cast<int>(i % kSkFp), as = static_cast<int>(i % kSkA);
        const uint32_t fph = static_cast<uint32_t>((i / kSkFp) & 1);
        const uint32_t aph = static_cast<uint32_t>((i / kSkA) & 1);
        if (!mbar_wait(&fp_full[fs], fph, p.pipe_timeout_ns, abort, gstatus) ||
            !mbar_wait(&a_full[as], aph, p.pipe_timeout_ns, abort, gstatus)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t bs = b0 + fs * kSkFpStage;
#pragma unroll
        for (int k = 0; k < kBlockK / kUmmaK; ++k) {
          const uint32_t a_tmem = tmem + kSkAcol + as * 32 + k * 8;
          const uint64_t bd = smem_desc_sw128(bs + k * (kUmmaK * 128), 64 * kBlockK * 2, 1024);
          asm volatile(
              "{\n\t.reg .pred p;\n\t"
              "setp.ne.b32 p, %4, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
              "r"(a_tmem), "l"(bd), "r"(idesc), "r"((kb > s0 || k > 0) ? 1u : 0u)
              : "memory");
        }
        mma_commit(&fp_empty[fs]);
        mma_commit(&a_empty[as]);
      }
      if (!ok) break;
      mma_commit(&dfull[buf]);
    }
    u = ue;
  }
  if (!ok) {
    sk_set_status(p.status, kStatusPipelineTimeout, 0x1400u);
    *abort = 1;
  }
}

// ------------------------------------------------------------------ epilogue (warps 12-15)
__device__ void sk_epilogue(const SkinnyParams& p, uint64_t* dfull, uint64_t* dempty,
                            uint32_t tmem, float* sTrans, int quad, int lane,
                            volatile int* abort) {
  const Geometry& g = p.g;
  const volatile uint32_t* gstatus = p.status;
  const int row0 = quad * 32;
  const bool has_rows = row0 < g.M;  // warp-uniform
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(row0) << 16);
  int32_t* tr = reinterpret_cast<int32_t*>(sTrans) + quad * (32 * 33);
  const int64_t KQ = units_per_tile(g);
  int64_t u0, u1;
  cta_range(p, u0, u1);
  uint32_t seg = 0;
  for (int64_t u = u0; u < u1;) {
    int64_t nt, ue, kb0, kb1;
    piece_at(g, KQ, u, u1, nt, ue, kb0, kb1);
    for (int64_t s0 = kb0; s0 < kb1; s0 += kSegBlocks, ++seg) {
      const bool first = s0 == kb0, last = s0 + kSegBlocks >= kb1;
      const uint32_t buf = seg & 1u, use = seg >> 1;
      const bool mine = mbar_wait(&dfull[buf], use & 1u, p.pipe_timeout_ns, abort, gstatus);
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
      if (has_rows) {
        for (int j = 0; j < kSkN / 32; ++j) {
          uint32_t f[32], s[32];
          tmem_ld32(lane_base + kSkDcol + buf * kSkN + j * 32, f);
          if (!first) tmem_ld32(lane_base + kSkScol + j * 32, s);
          tmem_ld_wait();
          if (j == kSkN / 32 - 1) {
            // the fp32 buffer has been read: the MMA may reuse it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&dempty[buf]);
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
          // flush: transpose so that a warp instruction adds 32 consecutive
          // columns of one row
#pragma unroll
          for (int e = 0; e < 32; ++e) tr[lane * 33 + e] = static_cast<int32_t>(acc[e]);
          __syncwarp();
          const int64_t n = nt * kSkN + j * 32 + lane;
          if (n < g.N) {
            int32_t* col = p.acc + n;
            for (int rr = 0; rr < 32 && row0 + rr < g.M; ++rr) {
              const int32_t val = tr[rr * 33 + lane];
              if (val != 0) atomicAdd(col + (int64_t)(row0 + rr) * g.N, val);
            }
          }
          __syncwarp();
        }
        if (!last) tmem_st_wait();
      } else {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&dempty[buf]);
      }
    }
    u = ue;
  }
}

__global__ void __launch_bounds__(kSkThreads, 1) ag_skinny_kernel(const __grid_constant__ SkinnyParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sFp = smem;                                   // 1024-aligned swizzled fp16 B stages
  uint8_t* sRaw = sFp + kSkFp * kSkFpStage;              // raw int8 B ring (1024-aligned)
  float* sTrans = reinterpret_cast<float*>(sRaw + kSkRaw * kSkRawStage);
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sTrans) + kSkTrans);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = raw_full + kSkRaw;
  uint64_t* fp_full = raw_empty + kSkRaw;
  uint64_t* fp_empty = fp_full + kSkFp;
  uint64_t* a_full = fp_empty + kSkFp;
  uint64_t* a_empty = a_full + kSkA;
  uint64_t* dfull = a_empty + kSkA;
  uint64_t* dempty = dfull + 2;
  uint64_t* drain = dempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool gemm = (p.flags & kFlagGemm) != 0;
  const int a_quads = static_cast<int>((p.g.M + 31) / 32);  // lane quadrants holding rows
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSkRaw; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], 4);  // the B-widening warps
    }
    for (int s = 0; s < kSkFp; ++s) {
      mbar_init(&fp_full[s], 4);
      mbar_init(&fp_empty[s], 1);
    }
    for (int s = 0; s < kSkA; ++s) {
      mbar_init(&a_full[s], a_quads);  // one A warp per quadrant holding rows
      mbar_init(&a_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&dfull[b], 1);
      mbar_init(&dempty[b], 4);
    }
    mbar_init(drain, 1);
    *tmem_slot = 0;
    *abort = 0;
    fence_mbar_init();
  }
  if (gemm && warp == 4) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    if (gemm) sk_bwiden(p, sRaw, sFp, raw_full, raw_empty, fp_full, fp_empty, threadIdx.x, abort);
  } else if (warp == 4) {
    if (gemm && lane == 0)
      sk_mma(p, sFp, fp_full, fp_empty, a_full, a_empty, dfull, dempty, tmem, abort);
  } else if (warp == 5) {
    if (p.flags & kFlagCopy) sk_copy_warp(p, lane);
  } else if (warp == 6) {
    if (gemm) sk_tma_warp(p, sRaw, raw_full, raw_empty, lane, abort);
  } else if ((warp >= 8 && warp < 12) || warp >= 16) {
    if (gemm) sk_awiden(p, a_full, a_empty, tmem, warp & 3, warp >= 16 ? 1 : 0, lane, abort);
  } else if (warp >= 12 && warp < 16) {
    if (gemm) sk_epilogue(p, dfull, dempty, tmem, sTrans, warp & 3, lane, abort);
  }

  tc_fence_before();
  __syncthreads();
  if (gemm && warp == 4) {
    if (lane == 0) {
      mma_commit(drain);
      volatile int never = 0;
      mbar_wait(drain, 0, p.pipe_timeout_ns, &never);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// C_i32 = acc + bias, D = fp16(fp32(C_i32) * scale), acc = 0: one thread per 8
// consecutive outputs (N % 16 == 0, so a row holds a whole number of them).
__global__ void __launch_bounds__(256) ag_skinny_finish_kernel(int32_t* __restrict__ acc,
                                                               const int32_t* __restrict__ bias,
                                                               const float* __restrict__ scale,
                                                               int32_t* __restrict__ C_i32,
                                                               uint16_t* __restrict__ D,
                                                               int64_t M, int64_t N) {
  const int64_t groups = M * N / 8;
  for (int64_t gi = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; gi < groups;
       gi += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t off = gi * 8, n = off % N;
    int4* ap = reinterpret_cast<int4*>(acc + off);
    const int4 a0 = __ldcg(ap), a1 = __ldcg(ap + 1);
    const int4 b0 = __ldg(reinterpret_cast<const int4*>(bias + n));
    const int4 b1 = __ldg(reinterpret_cast<const int4*>(bias + n + 4));
    const float4 s0 = __ldg(reinterpret_cast<const float4*>(scale + n));
    const float4 s1 = __ldg(reinterpret_cast<const float4*>(scale + n + 4));
    const int32_t av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const int32_t bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    int32_t c[8];
    uint32_t h[4];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      c[e] = static_cast<int32_t>(static_cast<uint32_t>(av[e]) + static_cast<uint32_t>(bb[e]));
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
    ap[0] = make_int4(0, 0, 0, 0);  // the accumulator starts every run at zero
    ap[1] = make_int4(0, 0, 0, 0);
  }
}

}  // namespace

cudaError_t skinny_prepare() {
  return cudaFuncSetAttribute(reinterpret_cast<const void*>(&ag_skinny_kernel),
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kSkSmem);
}

cudaError_t launch_skinny(const SkinnyParams& p, int grid, cudaStream_t stream) {
  ag_skinny_kernel<<<grid, kSkThreads, kSkSmem, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !(p.flags & kFlagGemm)) return e;
  ag_skinny_finish_kernel<<<grid * 2, 256, 0, stream>>>(p.acc, p.bias, p.scale, p.C_i32, p.D_f16,
                                                        p.g.M, p.g.N);
  return cudaGetLastError();
}

}  // namespace agg
