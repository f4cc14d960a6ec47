// fused_kernel.cuh -- parameters shared by the host plan and the fused
// streamed AllGather+GEMM kernel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "schedule.h"
#include "trace.cuh"

namespace agg {

// Status word values (low byte = kind, upper bits = detail).
enum : uint32_t {
  kStatusOk = 0,
  kStatusChunkTimeout = 1,     // a ready counter did not reach its target in time
  kStatusPipelineTimeout = 2,  // an mbarrier of the TMA/MMA/epilogue pipeline ran out
  kStatusCreditTimeout = 3,    // bounded staging: a slot was not released by its readers in time
};

enum : int {
  kFlagCopy = 1,   // producer warps copy remote chunks and release counters
  kFlagGemm = 2,   // TMA / MMA / epilogue warps compute C
  kFlagWait = 4,   // the TMA warp waits on the ready counters of remote chunks
};

struct FusedParams {
  CUtensorMap tm_a_local;   // fp16 [R][K] local shard (2D: K, R)
  CUtensorMap tm_a_stage;   // fp16 staging (3D: K, rows, slot): [S-1][R][K], or [window][256][K]
  CUtensorMap tm_b;         // fp16 [K][N], loaded MN-major: 3D (64, K, N/64) when b3d, else 2D (N, K)
  CUtensorMap tm_c;         // fp16 path: fp32 C as [S][R][N] (3D: N, R, S), stored in 32x32 boxes
  Geometry g;
  const void* src[kMaxShards];  // shard pointers by consumption position
  void* staging;                // fp16 [(S-1)][R][K], or bounded: [window][256][K]
  uint32_t* counters;           // [(S-1)][Q] ready counters, monotonic
  unsigned long long* item_counter;  // copy items handed out so far (monotonic)
  unsigned long long item_base;      // item_counter value at the start of this run
  unsigned long long* tile_counter;  // work items handed out so far (monotonic)
  unsigned long long tile_base;      // tile_counter value at the start of this run
  // Work items: tiles [0, full_tiles) whole, the others in `split` K-parts.
  // int8: every part but the last stores its partial sums (int32) to
  // `partials` and counts its 16 epilogue warps on the tile's flag; the last
  // part waits for the flag to reach part_target, adds the partials in part
  // order and writes the outputs.  fp16 / bf16 (two parts): both parts add
  // their fp32 sums into C with TMA reductions, into tiles that the epilogue
  // warps zeroed at the start of the run (zero tasks, drawn by ticket).
  int64_t full_tiles;
  int64_t work_items;
  int64_t static_items;      // items below this are dealt round-robin: pair k takes k, k + pairs, ...
  int split;
  void* partials;            // [tail tiles][split - 1][2 CTAs][128 rows][BN] 4-byte sums
  uint32_t* part_flags;      // [tail tiles], monotonic
  uint32_t part_target;      // flag value once every earlier part of this run has stored
  int64_t zero_tasks;        // fp16 split: 32-row groups of the tail tiles to zero (0: none)
  unsigned long long* zero_ticket;  // zero tasks handed out so far (monotonic)
  unsigned long long zero_base;     // this run's first ticket (the counter is raised to it)
  uint32_t* zero_done;       // zero tasks completed, monotonic
  uint32_t zero_target;      // zero_done once this run's tasks are all done
  uint32_t* status;             // [2]: status word, detail
  float* C;                     // f16 path output, M x N fp32
  int32_t* C_i32;               // i8 path outputs
  uint16_t* D_f16;
  const int32_t* bias;
  const float* scale;
  int local;                    // local rank
  int flags;                    // kFlag*
  int b3d;                      // B half of a CTA in one 3D box (N % 64 == 0) instead of 64-wide 2D boxes
  int bf16;                     // fp16-path operands are bfloat16 (same layout, kind::f16 bf16 format)
  uint32_t epoch;               // run number since the last reset (>= 1)
  uint64_t timeout_ns;          // limit of a wait on a ready counter
  uint64_t pipe_timeout_ns;     // limit of a wait on a pipeline mbarrier (longer)
  int64_t debug_skip_item;      // -1 = none
  uint32_t debug_delay_ns;
  // Bounded staging (window > 0): remote row block b (256 rows: m-tile mt of
  // position pos, b = (pos - 1) * MT + mt) lives in slot b % window.  Each
  // remote tile that has loaded its rows adds one credit to the slot; block b
  // may overwrite the slot once block b - window's NT tiles have all done so.
  int window;                   // slots of 256 rows; 0 = every remote row has its own place
  uint32_t* credits;            // [window] tiles done reading the slot, monotonic
  uint32_t credit_epoch;        // pipelined runs of this plan since the last reset (>= 1)
  TraceBuf trace;               // event trace (count == nullptr: off)
};

constexpr int kThreads = 384;                         // 12 warps (int8 kernel)
// The fp16 / bf16 kernel adds a second TMA producer warp (warp 12), used when
// every tile of the plan is dealt; the int8 kernel's 168 registers per thread
// leave no room for a thirteenth warp.
constexpr int kExtraTmaWarp = 12;
constexpr int kThreadsF16 = 416;
__host__ __device__ constexpr int fused_threads(bool i8) { return i8 ? kThreads : kThreadsF16; }
constexpr int kEpiWarps = 8;                          // 4 lane quadrants x 2 column halves
constexpr int kABytes = kBlockM * kBlockK * 2;        // 16 KB: this CTA's 128 rows of A
constexpr int kBBytes = kMaxBlockN / 2 * kBlockK * 2; // 16 KB: this CTA's half of B's columns
// fp16 epilogue: each of the 8 epilogue warps stages 32 rows x 32 fp32 columns
// (4 KB, 128-byte swizzled) in its own buffer and writes it with a TMA store.
constexpr int kEpiBoxBytes = 32 * 32 * 4;
constexpr int kEpiBytes = kEpiWarps * kEpiBoxBytes;  // 32 KB
constexpr int kSmemBytes =
    kStages * (kABytes + kBBytes) + kEpiBytes + 1024 /*barriers*/ + 1024 /*align*/;
constexpr int kCopyWarpsPerCta = 2;
// The pair's ring of drawn work items: published by the even CTA's TMA warp
// (lane 1), read by both TMA warps and the MMA thread, and freed by the 16
// epilogue warps of the pair, which read each entry last.
constexpr int kTq = 8;
constexpr int kTqReaders = 2 * kEpiWarps;

// ---------------------------------------------------------------- skinny int8 path
constexpr int kSkMaxRows = 128;   // the gathered rows are the MMA's N operand (N <= 128 here)

struct SkinnyParams {
  CUtensorMap tm_b8;        // int8 B, 128-byte swizzle: 3D (128, K, N / 128), box 128 x 64 x 2
                            // when b3d, else 2D (N, K), box 128 x 64
  CUtensorMap tm_a8_local;  // int8 local shard (2D: K, R), box 64 x R, unswizzled
  CUtensorMap tm_a8_stage;  // int8 staging (3D: K, R, S - 1), box 64 x R x (S - 1)
  Geometry g;
  const void* src[kMaxShards];  // shard pointers by consumption position
  int8_t* staging;              // int8 [S-1][R][K]
  uint32_t* counters;           // [np][S-1][Q] ready counters, one release per task, monotonic
  unsigned long long* item_counter;
  unsigned long long item_base;
  int32_t* ws;                  // [n_tiles][cmax][M][256] int32 piece sums
  uint32_t* status;
  const int32_t* bias;
  const float* scale;
  int32_t* C_i32;
  uint16_t* D_f16;
  int local;
  int flags;
  uint32_t epoch;               // ready-counter epoch (as the fused kernel)
  uint64_t timeout_ns;
  uint64_t pipe_timeout_ns;
  int64_t debug_skip_item;
  uint32_t debug_delay_ns;
  int64_t n_tiles;              // ceil(N / 256)
  int64_t kq;                   // 2-k-block units per n-tile: ceil(KB / 2)
  int64_t cmax;                 // workspace slots per n-tile
  int np;                       // k-parts of the remote rows (copy tasks and counters per chunk)
  int b3d;                      // tm_b8 is the 3D view (N % 128 == 0)
  TraceBuf trace;               // event trace (count == nullptr: off)
};
constexpr int kSkCopyWarpsPerCta = 2;

// Launchers (fused_kernel.cu, skinny_kernel.cu).
cudaError_t launch_fused(const FusedParams& p, int grid, cudaStream_t stream);
cudaError_t fused_max_clusters(int dtype, int grid, int* clusters);
cudaError_t skinny_prepare();
cudaError_t launch_skinny(const SkinnyParams& p, int grid, cudaStream_t stream);
cudaError_t launch_widen(const int8_t* src0, uint16_t* dst0, int64_t n0, const int8_t* src1,
                         uint16_t* dst1, int64_t n1, int grid, cudaStream_t stream);


}  // namespace agg
