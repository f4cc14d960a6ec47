// skinny_kernel.cu -- int8 AllGatherMatmulDequant when the gathered A has at
// most 128 rows (decode-like shapes such as 2 x 32 rows, K = 16384, N = 7168).
//
// Such a problem is bound by reading B from HBM once ("AllGather矩阵乘法反量化
// 算子设计文档", 8.3 lists the 64 x 16384 x 7168 shape): every k-block of B is
// shared by all rows, so the kernel streams B exactly once as int8, widens it
// in shared memory and runs the tensor core on it with the (tiny) A held in
// tensor memory.  sm_103a has no tcgen05 kind::i8, so the product is computed
// exactly on kind::f16: every int8 is an exact fp16, and a unit never spans
// more than 16 k-blocks (1024 k), which keeps every fp32 partial an integer
// below 2^24.
//
// Work unit = (128-column n-tile, segment of <= 16 k-blocks); CTA b takes
// units b, b + grid, ...  A unit's exact int32 partial is added with
// coalesced red.add.s32 to an L2-resident int32 accumulator (integer addition
// is exact in any order); the last unit of an n-tile to finish (a monotonic
// per-n-tile counter reaching epoch * segments) adds the bias, writes C_i32
// and the fp16 dequant D, and zeroes the accumulator for the next run.
//
// Roles (16 warps):
//   warp 6      TMA warp: waits once for every remote chunk (the rows of the
//               other shards, copied by the copy warps), then streams int8
//               k-blocks of B (64 x 128) and of A (all rows x 64) into a raw
//               shared-memory ring.
//   warps 0-3   B widening: raw int8 B -> fp16 in the MN-major 128-byte
//               swizzled layout the MMA reads.
//   warps 8-11  A widening: raw int8 A rows -> fp16 -> tcgen05.st into TMEM
//               (one row per TMEM lane; the MMA's A operand comes from TMEM).
//   warp 4      MMA: one thread issues tcgen05.mma (M = 128, N = 128, K = 16).
//   warp 5      copy warp: copies remote chunks into the int8 staging
//               workspace and releases their ready counters.
//   warps 12-15 epilogue: fp32 accumulator -> int32 -> transpose through
//               shared memory -> red.add.s32; the n-tile's last unit finishes
//               the dequant.

#include <cuda_fp16.h>

#include "fused_kernel.cuh"
#include "sm103.cuh"

namespace agg {

namespace {

constexpr int kSkThreads = 512;
constexpr int kSkN = 128;              // n-tile
constexpr int kSkRaw = 8;              // raw int8 ring stages
constexpr int kSkFp = 4;               // fp16 B stages = A TMEM stages
constexpr int kSkRawB = kSkN * kBlockK;              // 8 KB int8
constexpr int kSkRawA = kSkMaxRows * kBlockK;        // 8 KB int8 (<= 128 rows)
constexpr int kSkRawStage = kSkRawB + kSkRawA;
constexpr int kSkFpStage = kSkN * kBlockK * 2;       // 16 KB fp16
constexpr int kSkTrans = 4 * 32 * 33 * 4;            // epilogue transposes
constexpr int kSkSmem = kSkRaw * kSkRawStage + kSkFp * kSkFpStage + kSkTrans + 1024 + 1024;
constexpr uint32_t kSkAcol = 0;        // TMEM columns [0, 128): A stages (32 each)
constexpr uint32_t kSkDcol = 128;      // TMEM columns [128, 384): two 128-column accumulators

__device__ __forceinline__ void sk_set_status(uint32_t* status, uint32_t kind, uint32_t detail) {
  if (atomicCAS(status, 0u, kind) == 0u) atomicExch(status + 1, detail);
}

__device__ __forceinline__ void widen16x(const uint4 v, uint4& a, uint4& b) {
  i8x4_to_f16x4(v.x, a.x, a.y);
  i8x4_to_f16x4(v.y, a.z, a.w);
  i8x4_to_f16x4(v.z, b.x, b.y);
  i8x4_to_f16x4(v.w, b.z, b.w);
}

__device__ __forceinline__ void unit_coords(const SkinnyParams& p, int64_t u, int64_t& nt,
                                            int64_t& kb0, int64_t& kb1) {
  nt = u % p.n_tiles;
  const int64_t seg = u / p.n_tiles;
  kb0 = seg * kSegBlocks;
  kb1 = kb0 + kSegBlocks < p.g.KB ? kb0 + kSegBlocks : p.g.KB;
}

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

// ------------------------------------------------------------------ TMA warp
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

__device__ void sk_tma_warp(const SkinnyParams& p, uint8_t* sRaw, uint64_t* raw_full,
                            uint64_t* raw_empty, int lane, volatile int* abort) {
  const Geometry& g = p.g;
  const volatile uint32_t* gstatus = p.status;
  const uint32_t tx = static_cast<uint32_t>(kSkRawB + g.M * kBlockK);
  if ((p.flags & kFlagWait) && g.S > 1 && !sk_wait_all_chunks(p, lane, abort)) return;
  if (lane != 0) return;
  fence_acq_rel_gpu();
  fence_proxy_async_global();
  tma_prefetch_desc(&p.tm_b8);
  int stage = 0;
  uint32_t phase = 0, issued = 0, issued_phase = 0;
  bool ok = true;
  for (int64_t u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
    int64_t nt, kb0, kb1;
    unit_coords(p, u, nt, kb0, kb1);
    for (int64_t kb = kb0; kb < kb1; ++kb) {
      if (!mbar_wait(&raw_empty[stage], phase ^ 1u, p.pipe_timeout_ns, abort, gstatus)) {
        ok = false;
        break;
      }
      mbar_arrive_expect_tx(&raw_full[stage], tx);
      uint8_t* st = sRaw + stage * kSkRawStage;
      const int32_t x = static_cast<int32_t>(kb * kBlockK);
      tma_load_2d(st, &p.tm_b8, &raw_full[stage], static_cast<int32_t>(nt * kSkN), x);
      // A rows in global order: shard s fills rows [s*R, (s+1)*R)
      for (int s = 0; s < g.S; ++s) {
        uint8_t* a_dst = st + kSkRawB + s * g.R * kBlockK;
        const int pos = (s - p.local + g.S) % g.S;
        if (pos == 0)
          tma_load_2d(a_dst, &p.tm_a8_local, &raw_full[stage], x, 0);
        else
          tma_load_3d(a_dst, &p.tm_a8_stage, &raw_full[stage], x, 0, pos - 1);
      }
      issued |= 1u << stage;
      issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
      if (++stage == kSkRaw) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (!ok) {
    sk_set_status(p.status, kStatusPipelineTimeout, 0x1100u);
    *abort = 1;
  }
  volatile int never = 0;
  const uint64_t limit = ok ? p.pipe_timeout_ns : 20000000ull;
  for (int s = 0; s < kSkRaw; ++s)
    if (issued & (1u << s)) mbar_wait(&raw_full[s], (issued_phase >> s) & 1u, limit, &never);
}

// ------------------------------------------------------------------ B widening (warps 0-3)
// Thread t widens 64 bytes of one k-row: k-row t / 2, columns (t % 2) * 64 .. +63
// (= one 64-column swizzle group of the MN-major fp16 tile).
__device__ void sk_bwiden(const SkinnyParams& p, const uint8_t* sRaw, uint8_t* sFp,
                          uint64_t* raw_full, uint64_t* raw_empty, uint64_t* fp_full,
                          uint64_t* fp_empty, int t, volatile int* abort) {
  const volatile uint32_t* gstatus = p.status;
  const int krow = t >> 1, grp = t & 1, lane = t & 31;
  int rs = 0, fs = 0;
  uint32_t rphase = 0, fphase = 0;
  for (int64_t u = blockIdx.x; u < p.units; u += gridDim.x) {
    int64_t nt, kb0, kb1;
    unit_coords(p, u, nt, kb0, kb1);
    for (int64_t kb = kb0; kb < kb1; ++kb) {
      if (!mbar_wait(&raw_full[rs], rphase, p.pipe_timeout_ns, abort, gstatus) ||
          !mbar_wait(&fp_empty[fs], fphase ^ 1u, p.pipe_timeout_ns, abort, gstatus)) {
        if (lane == 0) {
          sk_set_status(p.status, kStatusPipelineTimeout, 0x1200u);
          *abort = 1;
        }
        return;
      }
      // raw B arrives 128-byte swizzled: 16-byte chunk j of k-row r sits at j ^ (r % 8)
      const uint8_t* src = sRaw + rs * kSkRawStage + krow * kSkN;
      uint4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        v[i] = *reinterpret_cast<const uint4*>(src + (((grp * 4 + i) ^ (krow & 7)) * 16));
      uint8_t* dst = sFp + fs * kSkFpStage + grp * (64 * kBlockK * 2) + krow * 128;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint4 a, b;
        widen16x(v[i], a, b);
        const int c0 = 2 * i, c1 = 2 * i + 1;  // 16-byte chunks of 8 fp16 within the row
        *reinterpret_cast<uint4*>(dst + ((c0 ^ (krow & 7)) * 16)) = a;
        *reinterpret_cast<uint4*>(dst + ((c1 ^ (krow & 7)) * 16)) = b;
      }
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&fp_full[fs]);
        mbar_arrive(&raw_empty[rs]);
      }
      if (++rs == kSkRaw) {
        rs = 0;
        rphase ^= 1u;
      }
      if (++fs == kSkFp) {
        fs = 0;
        fphase ^= 1u;
      }
    }
  }
}

// ------------------------------------------------------------------ A widening (warps 8-11)
// Lane l of warp w holds row m = 32 * (w % 4) + l: 64 int8 of the k-block ->
// 64 fp16 = 32 TMEM columns (k = 2c in the low half of column c).
__device__ void sk_awiden(const SkinnyParams& p, const uint8_t* sRaw, uint64_t* raw_full,
                          uint64_t* raw_empty, uint64_t* a_full, uint64_t* fp_empty,
                          uint32_t tmem, int quad, int lane, volatile int* abort) {
  const volatile uint32_t* gstatus = p.status;
  const int m = quad * 32 + lane;
  const bool has_rows = quad * 32 < p.g.M;  // warp-uniform
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
  int rs = 0, fs = 0;
  uint32_t rphase = 0, fphase = 0;
  for (int64_t u = blockIdx.x; u < p.units; u += gridDim.x) {
    int64_t nt, kb0, kb1;
    unit_coords(p, u, nt, kb0, kb1);
    for (int64_t kb = kb0; kb < kb1; ++kb) {
      if (!mbar_wait(&raw_full[rs], rphase, p.pipe_timeout_ns, abort, gstatus) ||
          !mbar_wait(&fp_empty[fs], fphase ^ 1u, p.pipe_timeout_ns, abort, gstatus)) {
        if (lane == 0) {
          sk_set_status(p.status, kStatusPipelineTimeout, 0x1300u);
          *abort = 1;
        }
        return;
      }
      if (has_rows) {
        uint32_t r[32];
        if (m < p.g.M) {
          // raw A arrives 64-byte swizzled: chunk j of row m sits at j ^ ((m / 2) % 4)
          const uint8_t* src = sRaw + rs * kSkRawStage + kSkRawB + m * kBlockK;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 a, b;
            widen16x(*reinterpret_cast<const uint4*>(src + ((i ^ ((m >> 1) & 3)) * 16)), a, b);
            r[8 * i + 0] = a.x; r[8 * i + 1] = a.y; r[8 * i + 2] = a.z; r[8 * i + 3] = a.w;
            r[8 * i + 4] = b.x; r[8 * i + 5] = b.y; r[8 * i + 6] = b.z; r[8 * i + 7] = b.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
        tmem_st32(lane_base + kSkAcol + fs * 32, r);
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&a_full[fs]);
        mbar_arrive(&raw_empty[rs]);
      }
      if (++rs == kSkRaw) {
        rs = 0;
        rphase ^= 1u;
      }
      if (++fs == kSkFp) {
        fs = 0;
        fphase ^= 1u;
      }
    }
  }
}

// ------------------------------------------------------------------ MMA warp
__device__ void sk_mma(const SkinnyParams& p, const uint8_t* sFp, uint64_t* fp_full,
                       uint64_t* a_full, uint64_t* fp_empty, uint64_t* dfull, uint64_t* dempty,
                       uint32_t tmem, volatile int* abort) {
  const volatile uint32_t* gstatus = p.status;
  // D fp32, A fp16 from TMEM (K-major), B fp16 MN-major, M = 128, N = 128
  const uint32_t idesc = idesc_f16_f32(128, kSkN, /*a_mn=*/false, /*b_mn=*/true);
  const uint32_t b0 = smem_u32(sFp);
  int fs = 0;
  uint32_t fphase = 0, unit = 0;
  bool ok = true;
  for (int64_t u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
    int64_t nt, kb0, kb1;
    unit_coords(p, u, nt, kb0, kb1);
    const uint32_t buf = unit & 1u, use = unit >> 1;
    if (!mbar_wait(&dempty[buf], (use & 1u) ^ 1u, p.pipe_timeout_ns, abort, gstatus)) {
      ok = false;
      break;
    }
    tc_fence_after();
    const uint32_t d = tmem + kSkDcol + buf * kSkN;
    for (int64_t kb = kb0; kb < kb1; ++kb) {
      if (!mbar_wait(&fp_full[fs], fphase, p.pipe_timeout_ns, abort, gstatus) ||
          !mbar_wait(&a_full[fs], fphase, p.pipe_timeout_ns, abort, gstatus)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t bs = b0 + fs * kSkFpStage;
#pragma unroll
      for (int k = 0; k < kBlockK / kUmmaK; ++k) {
        const uint32_t a_tmem = tmem + kSkAcol + fs * 32 + k * 8;
        const uint64_t bd = smem_desc_sw128(bs + k * (kUmmaK * 128), 64 * kBlockK * 2, 1024);
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
            "r"(a_tmem), "l"(bd), "r"(idesc), "r"((kb > kb0 || k > 0) ? 1u : 0u)
            : "memory");
      }
      mma_commit(&fp_empty[fs]);
      if (++fs == kSkFp) {
        fs = 0;
        fphase ^= 1u;
      }
    }
    if (!ok) break;
    mma_commit(&dfull[buf]);
    ++unit;
  }
  if (!ok) {
    sk_set_status(p.status, kStatusPipelineTimeout, 0x1400u);
    *abort = 1;
  }
}

// ------------------------------------------------------------------ epilogue (warps 12-15)
__device__ void sk_epilogue(const SkinnyParams& p, uint64_t* dfull, uint64_t* dempty,
                            uint32_t tmem, float* sTrans, volatile uint32_t* sLast, int quad,
                            int lane, volatile int* abort) {
  const Geometry& g = p.g;
  const volatile uint32_t* gstatus = p.status;
  const int row0 = quad * 32;
  const bool has_rows = row0 < g.M;  // warp-uniform
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(row0) << 16);
  float* tr = sTrans + quad * (32 * 33);
  const uint32_t target = p.tile_epoch * static_cast<uint32_t>(p.k_segs);
  uint32_t unit = 0;
  for (int64_t u = blockIdx.x; u < p.units; u += gridDim.x) {
    int64_t nt, kb0, kb1;
    unit_coords(p, u, nt, kb0, kb1);
    const uint32_t buf = unit & 1u, use = unit >> 1;
    const bool mine = mbar_wait(&dfull[buf], use & 1u, p.pipe_timeout_ns, abort, gstatus);
    // all four epilogue warps take the same decision (they meet at named barriers)
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
        uint32_t v[32];
        tmem_ld32(lane_base + kSkDcol + buf * kSkN + j * 32, v);
        tmem_ld_wait();
        // row (row0 + lane), columns 32j..32j+31 -> transpose so that a warp
        // instruction adds 32 consecutive columns of one row
#pragma unroll
        for (int e = 0; e < 32; ++e) tr[lane * 33 + e] = __uint_as_float(v[e]);
        __syncwarp();
        const int64_t n = nt * kSkN + j * 32 + lane;
        if (n < g.N) {
          for (int rr = 0; rr < 32 && row0 + rr < g.M; ++rr) {
            const int32_t val = __float2int_rn(tr[rr * 33 + lane]);
            if (val != 0) atomicAdd(p.acc + (int64_t)(row0 + rr) * g.N + n, val);
          }
        }
        __syncwarp();
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&dempty[buf]);
    ++unit;
    // the n-tile's last unit finishes the dequant
    __threadfence();
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (quad == 0 && lane == 0) {
      const uint32_t old = atomicAdd(p.tile_cnt + nt, 1u);
      *sLast = (old + 1u == target) ? 1u : 0u;
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (*sLast && has_rows) {
      __threadfence();
      const int m = row0 + lane;
      if (m < g.M) {
        const int64_t n0 = nt * kSkN;
        for (int64_t n = n0; n < n0 + kSkN && n < g.N; n += 8) {
          int32_t* ap = p.acc + (int64_t)m * g.N + n;
          const int4 a0 = __ldcg(reinterpret_cast<const int4*>(ap));
          const int4 a1 = __ldcg(reinterpret_cast<const int4*>(ap + 4));
          const int4 b0 = __ldg(reinterpret_cast<const int4*>(p.bias + n));
          const int4 b1 = __ldg(reinterpret_cast<const int4*>(p.bias + n + 4));
          const float4 s0 = __ldg(reinterpret_cast<const float4*>(p.scale + n));
          const float4 s1 = __ldg(reinterpret_cast<const float4*>(p.scale + n + 4));
          const int32_t av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
          const int32_t bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
          const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
          int32_t c[8];
          uint32_t h[4];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            c[e] = static_cast<int32_t>(static_cast<uint32_t>(av[e]) + static_cast<uint32_t>(bb[e]));
            const uint32_t hb = __half_as_ushort(__float2half_rn(__fmul_rn(__int2float_rn(c[e]), ss[e])));
            if (e & 1) h[e >> 1] |= hb << 16; else h[e >> 1] = hb;
          }
          *reinterpret_cast<int4*>(p.C_i32 + (int64_t)m * g.N + n) = make_int4(c[0], c[1], c[2], c[3]);
          *reinterpret_cast<int4*>(p.C_i32 + (int64_t)m * g.N + n + 4) = make_int4(c[4], c[5], c[6], c[7]);
          *reinterpret_cast<uint4*>(p.D_f16 + (int64_t)m * g.N + n) = make_uint4(h[0], h[1], h[2], h[3]);
          // the accumulator starts every run at zero
          *reinterpret_cast<int4*>(ap) = make_int4(0, 0, 0, 0);
          *reinterpret_cast<int4*>(ap + 4) = make_int4(0, 0, 0, 0);
        }
      }
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
  }
}

__global__ void __launch_bounds__(kSkThreads, 1) ag_skinny_kernel(const __grid_constant__ SkinnyParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sFp = smem;                                   // 1024-aligned swizzled fp16 B stages
  uint8_t* sRaw = sFp + kSkFp * kSkFpStage;              // raw int8 ring
  float* sTrans = reinterpret_cast<float*>(sRaw + kSkRaw * kSkRawStage);
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sTrans) + kSkTrans);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = raw_full + kSkRaw;
  uint64_t* fp_full = raw_empty + kSkRaw;
  uint64_t* a_full = fp_full + kSkFp;
  uint64_t* fp_empty = a_full + kSkFp;
  uint64_t* dfull = fp_empty + kSkFp;
  uint64_t* dempty = dfull + 2;
  uint64_t* drain = dempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile uint32_t* sLast = tmem_slot + 1;
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool gemm = (p.flags & kFlagGemm) != 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSkRaw; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], 8);  // 4 B-widening warps + 4 A-widening warps
    }
    for (int s = 0; s < kSkFp; ++s) {
      mbar_init(&fp_full[s], 4);
      mbar_init(&a_full[s], 4);
      mbar_init(&fp_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&dfull[b], 1);
      mbar_init(&dempty[b], 4);
    }
    mbar_init(drain, 1);
    *tmem_slot = 0;
    *sLast = 0;
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
    if (gemm && lane == 0) sk_mma(p, sFp, fp_full, a_full, fp_empty, dfull, dempty, tmem, abort);
  } else if (warp == 5) {
    if (p.flags & kFlagCopy) sk_copy_warp(p, lane);
  } else if (warp == 6) {
    if (gemm) sk_tma_warp(p, sRaw, raw_full, raw_empty, lane, abort);
  } else if (warp >= 8 && warp < 12) {
    if (gemm) sk_awiden(p, sRaw, raw_full, raw_empty, a_full, fp_empty, tmem, warp & 3, lane, abort);
  } else if (warp >= 12) {
    if (gemm) sk_epilogue(p, dfull, dempty, tmem, sTrans, sLast, warp & 3, lane, abort);
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

}  // namespace

cudaError_t skinny_prepare() {
  return cudaFuncSetAttribute(reinterpret_cast<const void*>(&ag_skinny_kernel),
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kSkSmem);
}

cudaError_t launch_skinny(const SkinnyParams& p, int grid, cudaStream_t stream) {
  ag_skinny_kernel<<<grid, kSkThreads, kSkSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace agg
