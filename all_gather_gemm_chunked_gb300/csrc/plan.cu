// plan.cu -- host side of libaggemm.so: argument validation, chunk sizing,
// workspace ownership, TMA descriptors and the launch sequence of each run
// mode.  Implements include/ag_gemm.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "ag_gemm.h"
#include "fused_kernel.cuh"
#include "schedule.h"

using agg::Geometry;

// ------------------------------------------------------------------ errors, log
namespace {
thread_local int g_last_error = AG_GEMM_OK;
thread_local char g_last_msg[512] = "";

// AG_GEMM_LOG=0..3 in the environment (read once): 1 errors, 2 plans, 3 runs.
int log_level() {
  static const int level = [] {
    const char* v = std::getenv("AG_GEMM_LOG");
    if (!v || !*v) return 0;
    const int l = std::atoi(v);
    return l < 0 ? 0 : (l > 3 ? 3 : l);
  }();
  return level;
}

void log_msg(int level, const char* fmt, ...) {
  if (log_level() < level) return;
  char buf[640];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  std::fprintf(stderr, "[ag_gemm] %s\n", buf);
}

int fail(int code, const char* fmt, ...) {
  g_last_error = code;
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_msg, sizeof(g_last_msg), fmt, ap);
  va_end(ap);
  log_msg(1, "error %d: %s", code, g_last_msg);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(e == cudaErrorMemoryAllocation ? AG_GEMM_ERR_OOM : AG_GEMM_ERR_CUDA, "%s: %s",
              what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------------ TMA descriptors
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// Tensor, innermost dimension first; 128-byte swizzle, zero fill out of bounds.
int encode_tiled(CUtensorMap* map, CUtensorMapDataType type, const void* base, int rank,
                 const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box,
                 CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(AG_GEMM_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = fn(map, type, static_cast<cuuint32_t>(rank),
                  const_cast<void*>(base), dims, strides_bytes, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(AG_GEMM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return AG_GEMM_OK;
}

// 2-byte operands.  bf16 plans use the same descriptors: TMA copies bytes, the
// element type only fixes the element size, and the zero fill is +0 in both.
int encode_f16(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
               const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, base, rank, dims, strides_bytes, box);
}

// int8 B (K x N row-major) of the skinny path, one k-block (64 k-rows) of a
// 256-column n-tile per load, 128-byte swizzle.  With N % 128 == 0 a 3D view
// (128 columns, K, N / 128 column blocks) takes both 128-column halves in one
// box of 128 x 64 x 2 (one TMA instruction); otherwise 2D (N, K) boxes of
// 128 x 64, two per k-block.  Rows past K, columns past N and blocks past
// N / 128 read as zero.
bool b8_is_3d(int64_t N) { return N % 128 == 0; }
int encode_b8(CUtensorMap* map, const void* base, int64_t K, int64_t N) {
  if (b8_is_3d(N)) {
    cuuint64_t dims[3] = {128, (cuuint64_t)K, (cuuint64_t)(N / 128)};
    cuuint64_t strides[2] = {(cuuint64_t)N, 128};
    cuuint32_t box[3] = {128, agg::kBlockK, 2};
    return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, 3, dims, strides, box);
  }
  cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)K};
  cuuint64_t strides[1] = {(cuuint64_t)N};
  cuuint32_t box[2] = {128, agg::kBlockK};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, 2, dims, strides, box);
}
// int8 gathered rows of the skinny path, one k-block (64 k) at a time,
// unswizzled: a shard (K, R) in 64 x R boxes, the staging (K, R, S - 1) in
// 64 x R x (S - 1) boxes.
int encode_a8(CUtensorMap* map, const void* base, int64_t R, int64_t K) {
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)R};
  cuuint64_t strides[1] = {(cuuint64_t)K};
  cuuint32_t box[2] = {agg::kBlockK, (cuuint32_t)R};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, 2, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
}
int encode_stage8(CUtensorMap* map, const void* base, int64_t slots, int64_t R, int64_t K) {
  cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)R, (cuuint64_t)slots};
  cuuint64_t strides[2] = {(cuuint64_t)K, (cuuint64_t)R * K};
  cuuint32_t box[3] = {agg::kBlockK, (cuuint32_t)R, (cuuint32_t)slots};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, 3, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
}

// fp32 C viewed as [S][R][N] so that a box never crosses into the next shard's
// rows: box 32 columns x 32 rows (128-byte rows, swizzled like the staging box).
// Row m of C starts ldc floats after row m - 1 (ldc = N, or the row pitch of a
// wider matrix whose column block C is).
int encode_c(CUtensorMap* map, const void* base, int64_t S, int64_t R, int64_t N, int64_t ldc) {
  cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)R, (cuuint64_t)S};
  cuuint64_t strides[2] = {(cuuint64_t)ldc * 4, (cuuint64_t)R * ldc * 4};
  cuuint32_t box[3] = {32, 32, 1};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, 3, dims, strides, box);
}

// A operand rows x K (K contiguous), box 64 x 128.
int encode_a(CUtensorMap* map, const void* base, int64_t rows, int64_t K) {
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {agg::kBlockK, agg::kBlockM};
  return encode_f16(map, base, 2, dims, strides, box);
}

// Staging: slots x R x K, box 64 x 128 x 1 (rows past R of a slot read as zero).
int encode_stage(CUtensorMap* map, const void* base, int64_t slots, int64_t R, int64_t K) {
  cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)R, (cuuint64_t)slots};
  cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)R * K * 2};
  cuuint32_t box[3] = {agg::kBlockK, agg::kBlockM, 1};
  return encode_f16(map, base, 3, dims, strides, box);
}

// B: K x N (N contiguous), loaded MN-major in 64-column swizzle groups.  When
// N % 64 == 0 it is described as 3D (64 columns, K, N / 64 groups) so that one
// box brings a CTA's whole half of the tile (BN / 128 groups); otherwise as 2D
// (N, K) with one 64 x 64 box per group.
bool b_is_3d(int64_t N) { return N % 64 == 0; }
// Row k of B starts ldb elements after row k - 1 (ldb = N, or the row pitch of a
// wider matrix whose column block B is).
int encode_b(CUtensorMap* map, const void* base, int64_t K, int64_t N, int64_t ldb, int BN) {
  if (b_is_3d(N)) {
    cuuint64_t dims[3] = {64, (cuuint64_t)K, (cuuint64_t)N / 64};
    cuuint64_t strides[2] = {(cuuint64_t)ldb * 2, 128};
    cuuint32_t box[3] = {64, agg::kBlockK, (cuuint32_t)(BN / 128)};
    return encode_f16(map, base, 3, dims, strides, box);
  }
  cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)K};
  cuuint64_t strides[1] = {(cuuint64_t)ldb * 2};
  cuuint32_t box[2] = {64, agg::kBlockK};
  return encode_f16(map, base, 2, dims, strides, box);
}

int check_problem(int S, int64_t M, int64_t K, int64_t N, int dtype, int64_t chunk_rows) {
  if (dtype != AG_GEMM_F16 && dtype != AG_GEMM_I8 && dtype != AG_GEMM_BF16)
    return fail(AG_GEMM_ERR_INVALID,
                "dtype must be AG_GEMM_F16, AG_GEMM_I8 or AG_GEMM_BF16 (got %d)", dtype);
  if (S < 1 || S > agg::kMaxShards)
    return fail(AG_GEMM_ERR_INVALID, "n_shards must be in [1, %d] (got %d)", agg::kMaxShards, S);
  if (M <= 0 || K <= 0 || N <= 0)
    return fail(AG_GEMM_ERR_INVALID, "M, K, N must be positive (got %lld, %lld, %lld)",
                (long long)M, (long long)K, (long long)N);
  if (M % S != 0)
    return fail(AG_GEMM_ERR_INVALID, "M (%lld) must be a multiple of n_shards (%d)", (long long)M, S);
  const int64_t R = M / S;
  if (chunk_rows < 0 || (chunk_rows > 0 && R % chunk_rows != 0))
    return fail(AG_GEMM_ERR_INVALID, "chunk_rows (%lld) must be 0 or divide the %lld rows of a shard",
                (long long)chunk_rows, (long long)R);
  if (dtype != AG_GEMM_I8 && (K % 8 != 0 || N % 8 != 0))
    return fail(AG_GEMM_ERR_INVALID, "fp16 and bf16 need K %% 8 == 0 and N %% 8 == 0 (16-byte rows)");
  if (dtype == AG_GEMM_I8 && (K % 16 != 0 || N % 16 != 0))
    return fail(AG_GEMM_ERR_INVALID, "int8 needs K %% 16 == 0 and N %% 16 == 0 (16-byte rows)");
  if (dtype == AG_GEMM_I8 && K > agg::kMaxKI8)
    return fail(AG_GEMM_ERR_UNSUPPORTED, "int8 needs K <= %lld so that K*127^2 fits in int32",
                (long long)agg::kMaxKI8);
  // TMA coordinates are 32-bit.
  if (K > (1LL << 31) || N > (1LL << 31) || R > (1LL << 31))
    return fail(AG_GEMM_ERR_UNSUPPORTED, "dimension too large for 32-bit TMA coordinates");
  // The kernels decode tiles and work items in 32-bit arithmetic.
  const int64_t tiles = static_cast<int64_t>(S) * ((R + agg::kPairM - 1) / agg::kPairM) *
                        ((N + 127) / 128);  // an upper bound of the pair tiles
  if (tiles >= (1LL << 30))
    return fail(AG_GEMM_ERR_UNSUPPORTED, "more than 2^30 pair tiles");
  return AG_GEMM_OK;
}

void to_public(const Geometry& g, ag_gemm_geometry* out) {
  std::memset(out, 0, sizeof(*out));
  out->n_shards = g.S;
  out->dtype = g.dtype;
  out->M = g.M;
  out->K = g.K;
  out->N = g.N;
  out->R = g.R;
  out->chunk_rows = g.c;
  out->chunks_per_source = g.Q;
  out->pieces_per_chunk = g.P;
  out->block_m = agg::kBlockM;
  out->block_n = g.BN;
  out->block_k = agg::kBlockK;
  out->group_m = agg::kGroupM;
  out->kseg_blocks = g.dtype == AG_GEMM_I8 ? agg::kSegBlocks : 0;
  out->m_tiles = g.MT;
  out->n_tiles = g.NT;
  out->tiles = g.tiles;
  out->producer_items = g.items;
  const int64_t slots = g.S > 1 ? g.S - 1 : 1;
  out->staging_bytes = slots * g.R * g.K * 2;
  int64_t ws = out->staging_bytes + slots * g.Q * 4 + 64;
  if (g.dtype == AG_GEMM_I8) ws += (g.K * g.N + g.R * g.K) * 2;
  out->workspace_bytes = ws;
  out->staging_slots = 0;
  out->split_tiles = 0;
  out->split_parts = 1;
}

bool from_public(const ag_gemm_geometry* in, Geometry& g) {
  if (!in || check_problem(in->n_shards, in->M, in->K, in->N, in->dtype, in->chunk_rows) != AG_GEMM_OK)
    return false;
  agg::make_geometry(g, in->n_shards, in->M, in->K, in->N, in->dtype, in->chunk_rows);
  return true;
}

// Restores the caller's current device on scope exit.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

}  // namespace

// ------------------------------------------------------------------ plan
struct ag_gemm_plan {
  Geometry g{};
  int device = 0;
  int sm_count = 0;
  int grid = 0;
  int grid_override = 0;  // ag_gemm_plan_set_grid (fused kernel), 0 = grid
  int mode = AG_GEMM_MODE_PIPELINED;
  int local = 0;
  uint64_t timeout_ns = 1000000000ull;
  int debug_flags = 0;
  int64_t debug_arg = 0;
  void* staging = nullptr;
  int64_t staging_bytes = 0;
  uint32_t* counters = nullptr;
  int64_t counter_count = 0;
  unsigned long long* item_counter = nullptr;  // copy items handed out (monotonic)
  unsigned long long item_base = 0;
  unsigned long long* tile_counter = nullptr;  // fused kernel: pair tiles handed out (monotonic)
  unsigned long long tile_base = 0;
  uint32_t* status = nullptr;
  uint16_t* b16 = nullptr;  // int8 path: fp16 copy of B
  uint16_t* a16 = nullptr;  // int8 path: fp16 copy of the local shard
  uint32_t epoch = 0;
  cudaEvent_t done = nullptr;
  cudaStream_t last_stream = nullptr;
  bool has_run = false;
  CUtensorMap tm_stage{};
  CUtensorMap tm_a16{}, tm_b16{};
  const void* cached_a = nullptr;
  CUtensorMap tm_a_cached{};
  const void* cached_b = nullptr;
  CUtensorMap tm_b_cached{};
  const void* cached_c = nullptr;
  int64_t cached_ldb = 0, cached_ldc = 0;  // row pitches the cached B / C maps were made for
  CUtensorMap tm_c_cached{};
  // int8 with at most 128 gathered rows: the skinny kernel
  bool skinny = false;
  int sk_grid = 0;
  int32_t* sk_ws = nullptr;      // piece sums, [n-tiles][sk_cmax][M][256] int32
  // bounded staging of the fused path (window > 0): 256-row slots
  int window = 0;
  uint32_t* credits = nullptr;   // [window] tiles done reading each slot, monotonic
  uint32_t credit_epoch = 0;     // pipelined runs since the last reset
  int64_t sk_tiles = 0;          // 256-column n-tiles
  int64_t sk_kq = 0;             // 2-k-block units per n-tile
  int64_t sk_cmax = 0;           // CTAs sharing an n-tile, at most
  int sk_np = 1;                 // k-parts of the remote rows (copy tasks per chunk)
  // fused kernel: the last round's tiles split into K-parts (split > 1)
  int split = 1;
  int64_t full_tiles = 0;        // tiles computed whole
  int64_t work_items = 0;        // full_tiles + split tiles x split
  void* partials = nullptr;      // partial sums of the earlier parts
  int64_t partials_bytes = 0;
  uint32_t* part_flags = nullptr;
  uint32_t part_epoch = 0;       // runs of the GEMM since the last reset
  // fp16 / bf16 split: both parts add into C blocks zeroed at the start of a run
  int64_t zero_tasks = 0;        // 32-row groups of the tail tiles
  unsigned long long* zero_ticket = nullptr;  // zero tasks handed out (monotonic)
  unsigned long long zero_base = 0;
  uint32_t* zero_done = nullptr;  // zero tasks done (monotonic)
  uint32_t zero_epoch = 0;       // runs of the GEMM since the last reset
  // event trace (ag_gemm_plan_set_trace): [0] count, then the events
  unsigned long long* trace_buf = nullptr;
  int64_t trace_cap = 0;
  const void* cached_b8 = nullptr;
  CUtensorMap tm_b8_cached{};
  const void* cached_a8 = nullptr;
  CUtensorMap tm_a8_cached{};
  CUtensorMap tm_stage8{};
};

namespace {

void free_plan(ag_gemm_plan* p) {
  if (!p) return;
  if (p->done) cudaEventSynchronize(p->done);
  cudaFree(p->staging);
  cudaFree(p->counters);
  cudaFree(p->item_counter);
  cudaFree(p->tile_counter);
  cudaFree(p->status);
  cudaFree(p->b16);
  cudaFree(p->a16);
  cudaFree(p->sk_ws);
  cudaFree(p->credits);
  cudaFree(p->trace_buf);
  cudaFree(p->partials);
  cudaFree(p->part_flags);
  cudaFree(p->zero_ticket);
  cudaFree(p->zero_done);
  if (p->done) cudaEventDestroy(p->done);
  delete p;
}

int launch_skinny(ag_gemm_plan* p, agg::SkinnyParams& sp, int flags, cudaStream_t stream) {
  sp.flags = flags;
  sp.item_base = p->item_base;
  cudaError_t e = agg::launch_skinny(sp, p->sk_grid, stream);
  if (e != cudaSuccess) return cuda_fail(e, "skinny kernel launch");
  // Every task is drawn by a ticket, and every copy warp draws one failing ticket.
  if (flags & agg::kFlagCopy) {
    const int64_t tasks = (p->g.S - 1) * p->g.Q * p->sk_np;
    const int64_t W = static_cast<int64_t>(p->sk_grid) * agg::kSkCopyWarpsPerCta;
    p->item_base += static_cast<unsigned long long>(tasks + W);
  }
  return AG_GEMM_OK;
}

int launch_fused(ag_gemm_plan* p, agg::FusedParams& fp, int flags, cudaStream_t stream) {
  fp.flags = flags;
  fp.item_base = p->item_base;
  fp.tile_counter = p->tile_counter;
  fp.tile_base = p->tile_base;
  fp.full_tiles = p->full_tiles;
  fp.work_items = p->work_items;
  fp.split = p->split;
  fp.partials = p->partials;
  fp.part_flags = p->part_flags;
  if ((flags & agg::kFlagGemm) && p->split > 1 && p->part_flags) {
    // every earlier part's 16 epilogue warps count once on the tile's flag per
    // run: restart the flags before they would overflow
    const uint64_t per_run = static_cast<uint64_t>(p->split - 1) * 2 * agg::kEpiWarps;
    if ((static_cast<uint64_t>(p->part_epoch) + 1) * per_run >= (1ull << 31)) {
      cudaError_t e = cudaMemsetAsync(p->part_flags, 0,
                                      sizeof(uint32_t) * (p->g.tiles - p->full_tiles), stream);
      if (e != cudaSuccess) return cuda_fail(e, "split-tile flag reset");
      p->part_epoch = 0;
    }
    ++p->part_epoch;
    fp.part_target = static_cast<uint32_t>(p->part_epoch * per_run);
  }
  fp.zero_tasks = (flags & agg::kFlagGemm) ? p->zero_tasks : 0;
  fp.zero_ticket = p->zero_ticket;
  fp.zero_base = p->zero_base;
  fp.zero_done = p->zero_done;
  fp.zero_target = 0;
  if (fp.zero_tasks > 0) {
    // restart the count of zero tasks done before it would overflow
    if ((static_cast<uint64_t>(p->zero_epoch) + 1) * static_cast<uint64_t>(p->zero_tasks) >=
        (1ull << 31)) {
      cudaError_t e = cudaMemsetAsync(p->zero_done, 0, sizeof(uint32_t), stream);
      if (e != cudaSuccess) return cuda_fail(e, "zero-task count reset");
      p->zero_epoch = 0;
    }
    ++p->zero_epoch;
    fp.zero_target = static_cast<uint32_t>(p->zero_epoch * p->zero_tasks);
  }
  const int grid = p->grid_override > 0 ? p->grid_override : p->grid;
  // Whole tiles are dealt round-robin (they wait on no other pair), and so
  // are the fp16 / bf16 split parts, which add into zeroed C blocks and wait
  // on no other part.  With a staging window the remote tiles' credits tie
  // them together, so only the local shard's tiles (consumption position 0:
  // the first MT x NT in schedule order, which neither wait for rows nor add
  // credits) are dealt and every remote tile is drawn; int8 split parts are
  // drawn, the last part of a tile after all the others it adds.
  const int64_t stat = p->window > 0 ? p->g.MT * p->g.NT
                                     : (p->zero_tasks > 0 ? p->work_items : p->full_tiles);
  fp.static_items = stat;
  cudaError_t e = agg::launch_fused(fp, grid, stream);
  if (e != cudaSuccess) return cuda_fail(e, "fused kernel launch");
  // Each copy warp draws every item's ticket plus one failing ticket; when
  // the plan has drawn work items, each pair draws every drawn item it
  // computes plus one failing ticket (with every item dealt, none at all).
  if (flags & agg::kFlagCopy)
    p->item_base += static_cast<unsigned long long>(p->g.items) +
                    static_cast<unsigned long long>(grid) * agg::kCopyWarpsPerCta;
  if ((flags & agg::kFlagGemm) && p->work_items > stat)
    p->tile_base += static_cast<unsigned long long>(p->work_items - stat) +
                    static_cast<unsigned long long>(grid / 2);
  // A run draws each zero task's ticket once, plus at most two failing
  // tickets per epilogue warp; the next run's tickets start past all of them.
  if (fp.zero_tasks > 0)
    p->zero_base += static_cast<unsigned long long>(p->zero_tasks) +
                    2ull * static_cast<unsigned long long>(grid) * agg::kEpiWarps;
  return AG_GEMM_OK;
}

// One run: the launch sequence of the plan's mode on `stream`.
int run_impl(ag_gemm_plan* p, const void* const* shard_ptrs, const void* B, int64_t ldb, float* C,
             int64_t ldc, int32_t* C_i32, void* D, const int32_t* bias, const float* scale,
             void* stream_v) {
  const Geometry& g = p->g;
  const bool int8 = g.dtype == AG_GEMM_I8;
  if (ldb < g.N || ldc < g.N)
    return fail(AG_GEMM_ERR_INVALID, "ldb (%lld) and ldc (%lld) must be at least N (%lld)",
                (long long)ldb, (long long)ldc, (long long)g.N);
  if (ldb % 8 != 0 || ldc % 4 != 0)
    return fail(AG_GEMM_ERR_INVALID,
                "row pitches must be multiples of 16 bytes: ldb %% 8 == 0, ldc %% 4 == 0");
  if (!shard_ptrs) return fail(AG_GEMM_ERR_INVALID, "shard_ptrs is NULL");
  for (int s = 0; s < g.S; ++s) {
    if (!shard_ptrs[s]) return fail(AG_GEMM_ERR_INVALID, "shard_ptrs[%d] is NULL", s);
    if (!aligned16(shard_ptrs[s])) return fail(AG_GEMM_ERR_INVALID, "shard_ptrs[%d] is not 16-byte aligned", s);
  }
  const void* outs[4] = {B, int8 ? static_cast<const void*>(C_i32) : static_cast<const void*>(C),
                         int8 ? D : B, int8 ? static_cast<const void*>(bias) : B};
  const char* names[4] = {"B", int8 ? "C_i32" : "C", "D_f16", "bias"};
  for (int i = 0; i < 4; ++i) {
    if (!outs[i]) return fail(AG_GEMM_ERR_INVALID, "%s is NULL", names[i]);
    if (!aligned16(outs[i])) return fail(AG_GEMM_ERR_INVALID, "%s is not 16-byte aligned", names[i]);
  }
  if (int8 && (!scale || !aligned16(scale)))
    return fail(AG_GEMM_ERR_INVALID, "scale is NULL or not 16-byte aligned");

  DeviceGuard dg(p->device);
  if (!dg.ok) return fail(AG_GEMM_ERR_CUDA, "cannot select the plan's device %d", p->device);
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  cudaError_t e;
  // Runs on one plan share its staging and counters: order them.
  if (p->has_run && p->last_stream != stream) {
    e = cudaStreamWaitEvent(stream, p->done, 0);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent");
  }
  // Counters are monotonic: after run e each holds e * P (e on the skinny path,
  // whose counters take one release per copy task).  Restart before overflow.
  const uint64_t releases = p->skinny ? 1u : static_cast<uint64_t>(g.P);
  if (static_cast<uint64_t>(p->epoch + 1) * releases >= (1ull << 31)) {
    e = cudaMemsetAsync(p->counters, 0, sizeof(uint32_t) * p->counter_count, stream);
    if (e != cudaSuccess) return cuda_fail(e, "counter reset");
    p->epoch = 0;
  }

  agg::FusedParams fp;
  std::memset(&fp, 0, sizeof(fp));
  fp.g = g;
  for (int pos = 0; pos < g.S; ++pos) fp.src[pos] = shard_ptrs[agg::source_of(g, p->local, pos)];
  const void* local_ptr = fp.src[0];
  int rc;
  if (int8) {
    fp.tm_a_local = p->tm_a16;
    fp.tm_b = p->tm_b16;
  } else {
    if (p->cached_a != local_ptr) {
      p->cached_a = nullptr;
      if ((rc = encode_a(&p->tm_a_cached, local_ptr, g.R, g.K)) != AG_GEMM_OK) return rc;
      p->cached_a = local_ptr;
    }
    if (p->cached_b != B || p->cached_ldb != ldb) {
      p->cached_b = nullptr;
      if ((rc = encode_b(&p->tm_b_cached, B, g.K, g.N, ldb, g.BN)) != AG_GEMM_OK) return rc;
      p->cached_b = B;
      p->cached_ldb = ldb;
    }
    if (p->cached_c != C || p->cached_ldc != ldc) {
      p->cached_c = nullptr;
      if ((rc = encode_c(&p->tm_c_cached, C, g.S, g.R, g.N, ldc)) != AG_GEMM_OK) return rc;
      p->cached_c = C;
      p->cached_ldc = ldc;
    }
    fp.tm_a_local = p->tm_a_cached;
    fp.tm_b = p->tm_b_cached;
    fp.tm_c = p->tm_c_cached;
  }
  fp.tm_a_stage = p->tm_stage;
  fp.staging = p->staging;
  fp.counters = p->counters;
  fp.item_counter = p->item_counter;
  fp.status = p->status;
  fp.C = C;
  fp.C_i32 = C_i32;
  fp.D_f16 = static_cast<uint16_t*>(D);
  fp.bias = bias;
  fp.scale = scale;
  fp.local = p->local;
  fp.b3d = b_is_3d(g.N) ? 1 : 0;
  fp.bf16 = g.dtype == AG_GEMM_BF16 ? 1 : 0;
  fp.epoch = p->epoch + 1;
  fp.timeout_ns = p->timeout_ns;
  // Pipeline stages only wait on each other; give them more room than the
  // counter waits so that a missing chunk is reported as such.
  fp.pipe_timeout_ns = p->timeout_ns * 4 > 2000000000ull ? p->timeout_ns * 4 : 2000000000ull;
  fp.debug_skip_item = (p->debug_flags & AG_GEMM_DEBUG_SKIP_ITEM) ? p->debug_arg : -1;
  fp.debug_delay_ns = (p->debug_flags & AG_GEMM_DEBUG_DELAY_NS)
                          ? static_cast<uint32_t>(p->debug_arg > 1000000 ? 1000000 : p->debug_arg)
                          : 0u;
  if (p->trace_buf) {
    // the run's events replace the previous run's: a cleared buffer cut into
    // one region per (CTA, warp slot) of the launch
    e = cudaMemsetAsync(p->trace_buf, 0, 32 + static_cast<size_t>(p->trace_cap) * 32, stream);
    if (e != cudaSuccess) return cuda_fail(e, "trace reset");
    const int64_t ctas = p->skinny ? p->sk_grid
                                   : (p->grid_override > 0 ? p->grid_override : p->grid);
    fp.trace.ev = reinterpret_cast<agg::TraceEvent*>(p->trace_buf + 4);
    fp.trace.dropped = p->trace_buf;
    fp.trace.per_slot = static_cast<uint32_t>(p->trace_cap / (ctas * agg::kTrSlots));
  }

  const int mode = p->mode;
  const bool runs_gemm = mode != AG_GEMM_MODE_COPY_ONLY;
  const bool runs_copy = mode != AG_GEMM_MODE_COMPUTE_ONLY && g.S > 1;
  if (p->window > 0) {
    // a copy that runs ahead of the GEMM would need every remote row at once
    if (mode == AG_GEMM_MODE_SEQUENTIAL)
      return fail(AG_GEMM_ERR_UNSUPPORTED,
                  "SEQUENTIAL mode needs the whole gather staged: use a plan without a staging "
                  "window");
    fp.window = p->window;
    fp.credits = p->credits;
    if (mode == AG_GEMM_MODE_PIPELINED) {
      // after pipelined run e slot s holds e * uses(s) * NT credits: restart before overflow
      const uint64_t per_run = static_cast<uint64_t>(agg::window_uses(g, p->window, 0)) * g.NT;
      if ((static_cast<uint64_t>(p->credit_epoch) + 1) * per_run >= (1ull << 31)) {
        e = cudaMemsetAsync(p->credits, 0, sizeof(uint32_t) * p->window, stream);
        if (e != cudaSuccess) return cuda_fail(e, "credit counter reset");
        p->credit_epoch = 0;
      }
      fp.credit_epoch = ++p->credit_epoch;
    }
  }
  if (runs_copy && (p->debug_flags & AG_GEMM_DEBUG_POISON_STAGING)) {
    // fp16 0x7E7E is a NaN: a tile read before its chunk landed turns C into NaN.
    e = cudaMemsetAsync(p->staging, 0x7E, static_cast<size_t>(p->staging_bytes), stream);
    if (e != cudaSuccess) return cuda_fail(e, "poison staging");
  }
  if (p->skinny) {
    agg::SkinnyParams sp;
    std::memset(&sp, 0, sizeof(sp));
    sp.g = g;
    for (int pos = 0; pos < g.S; ++pos) sp.src[pos] = fp.src[pos];
    if (p->cached_b8 != B) {
      p->cached_b8 = nullptr;
      if ((rc = encode_b8(&p->tm_b8_cached, B, g.K, g.N)) != AG_GEMM_OK) return rc;
      p->cached_b8 = B;
    }
    if (p->cached_a8 != local_ptr) {
      p->cached_a8 = nullptr;
      if ((rc = encode_a8(&p->tm_a8_cached, local_ptr, g.R, g.K)) != AG_GEMM_OK) return rc;
      p->cached_a8 = local_ptr;
    }
    sp.tm_b8 = p->tm_b8_cached;
    sp.b3d = b8_is_3d(g.N) ? 1 : 0;
    sp.tm_a8_local = p->tm_a8_cached;
    sp.tm_a8_stage = p->tm_stage8;
    sp.staging = static_cast<int8_t*>(p->staging);
    sp.counters = p->counters;
    sp.item_counter = p->item_counter;
    sp.ws = p->sk_ws;
    sp.status = p->status;
    sp.bias = bias;
    sp.scale = scale;
    sp.C_i32 = C_i32;
    sp.D_f16 = static_cast<uint16_t*>(D);
    sp.local = p->local;
    sp.epoch = fp.epoch;
    sp.timeout_ns = fp.timeout_ns;
    sp.pipe_timeout_ns = fp.pipe_timeout_ns;
    sp.debug_skip_item = fp.debug_skip_item;
    sp.debug_delay_ns = fp.debug_delay_ns;
    sp.n_tiles = p->sk_tiles;
    sp.kq = p->sk_kq;
    sp.cmax = p->sk_cmax;
    sp.np = p->sk_np;
    sp.trace = fp.trace;
    using namespace agg;
    switch (mode) {
      case AG_GEMM_MODE_PIPELINED:
        rc = launch_skinny(p, sp, kFlagGemm | kFlagWait | (runs_copy ? kFlagCopy : 0), stream);
        break;
      case AG_GEMM_MODE_COMPUTE_ONLY:
        rc = launch_skinny(p, sp, kFlagGemm, stream);
        break;
      case AG_GEMM_MODE_SEQUENTIAL:
        rc = runs_copy ? launch_skinny(p, sp, kFlagCopy, stream) : AG_GEMM_OK;
        if (rc == AG_GEMM_OK) rc = launch_skinny(p, sp, kFlagGemm | kFlagWait, stream);
        break;
      case AG_GEMM_MODE_COPY_ONLY:
        rc = runs_copy ? launch_skinny(p, sp, kFlagCopy, stream) : AG_GEMM_OK;
        break;
      default:
        rc = fail(AG_GEMM_ERR_STATE, "unknown mode %d", mode);
    }
    if (rc != AG_GEMM_OK) return rc;
    if (runs_copy) p->epoch += 1;
    e = cudaEventRecord(p->done, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    p->last_stream = stream;
    p->has_run = true;
    log_msg(3, "plan %p: skinny run enqueued, mode %d, epoch %u", static_cast<void*>(p), mode,
            p->epoch);
    return AG_GEMM_OK;
  }
  if (int8 && runs_gemm) {
    e = agg::launch_widen(static_cast<const int8_t*>(B), p->b16, g.K * g.N,
                          static_cast<const int8_t*>(local_ptr), p->a16, g.R * g.K,
                          p->sm_count * 4, stream);
    if (e != cudaSuccess) return cuda_fail(e, "int8 widen launch");
  }
  using namespace agg;
  switch (mode) {
    case AG_GEMM_MODE_PIPELINED:
      rc = launch_fused(p, fp, kFlagGemm | kFlagWait | (runs_copy ? kFlagCopy : 0), stream);
      break;
    case AG_GEMM_MODE_COMPUTE_ONLY:
      rc = launch_fused(p, fp, kFlagGemm, stream);
      break;
    case AG_GEMM_MODE_SEQUENTIAL:
      rc = runs_copy ? launch_fused(p, fp, kFlagCopy, stream) : AG_GEMM_OK;
      if (rc == AG_GEMM_OK) rc = launch_fused(p, fp, kFlagGemm | kFlagWait, stream);
      break;
    case AG_GEMM_MODE_COPY_ONLY:
      rc = runs_copy ? launch_fused(p, fp, kFlagCopy, stream) : AG_GEMM_OK;
      break;
    default:
      rc = fail(AG_GEMM_ERR_STATE, "unknown mode %d", mode);
  }
  if (rc != AG_GEMM_OK) return rc;
  // The counters advanced only if copies ran; compute-only runs leave them as they are.
  if (runs_copy) p->epoch += 1;
  e = cudaEventRecord(p->done, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  p->last_stream = stream;
  p->has_run = true;
  log_msg(3, "plan %p: fused run enqueued, mode %d, epoch %u, grid %d", static_cast<void*>(p),
          mode, p->epoch, p->grid_override > 0 ? p->grid_override : p->grid);
  return AG_GEMM_OK;
}

}  // namespace

extern "C" {

int64_t ag_gemm_choose_chunk_rows(int64_t R) {
  if (R < 1) return fail(AG_GEMM_ERR_INVALID, "R must be positive");
  return agg::choose_chunk_rows(R);
}

int ag_gemm_validate(int n_shards, int64_t M, int64_t K, int64_t N, int dtype,
                     int64_t chunk_rows) {
  return check_problem(n_shards, M, K, N, dtype, chunk_rows);
}

int ag_gemm_geometry_of(int n_shards, int64_t M, int64_t K, int64_t N, int dtype,
                        int64_t chunk_rows, ag_gemm_geometry* out) {
  if (!out) return fail(AG_GEMM_ERR_INVALID, "out is NULL");
  int rc = check_problem(n_shards, M, K, N, dtype, chunk_rows);
  if (rc != AG_GEMM_OK) return rc;
  Geometry g;
  agg::make_geometry(g, n_shards, M, K, N, dtype, chunk_rows);
  to_public(g, out);
  return AG_GEMM_OK;
}

int ag_gemm_tile_at(const ag_gemm_geometry* geo, int local_rank, int64_t t, int64_t out[3]) {
  Geometry g;
  if (!out || !from_public(geo, g)) return fail(AG_GEMM_ERR_INVALID, "bad geometry");
  if (local_rank < 0 || local_rank >= g.S || t < 0 || t >= g.tiles)
    return fail(AG_GEMM_ERR_INVALID, "tile or local rank out of range");
  int pos;
  int64_t mt, nt;
  agg::tile_coords(g, t, pos, mt, nt);
  out[0] = agg::source_of(g, local_rank, pos);
  out[1] = mt;
  out[2] = nt;
  return AG_GEMM_OK;
}

int ag_gemm_item_at(const ag_gemm_geometry* geo, int local_rank, int64_t i, int64_t out[4]) {
  Geometry g;
  if (!out || !from_public(geo, g)) return fail(AG_GEMM_ERR_INVALID, "bad geometry");
  if (local_rank < 0 || local_rank >= g.S || i < 0 || i >= g.items)
    return fail(AG_GEMM_ERR_INVALID, "item or local rank out of range");
  int pos, piece;
  int64_t q, v0, v1;
  agg::item_coords(g, i, pos, q, piece, v0, v1);
  const int64_t chunk0 = q * g.c * g.K * g.src_esize;
  out[0] = agg::source_of(g, local_rank, pos);
  out[1] = q;
  out[2] = chunk0 + v0 * 16;
  out[3] = chunk0 + v1 * 16;
  return AG_GEMM_OK;
}

}  // extern "C"

extern "C" {

}  // extern "C"

namespace {

// staging_slots < 0: every remote row has its own place in the staging;
// otherwise a bounded window of 256-row slots (0 = 2 swizzle groups).
ag_gemm_plan* create_plan(int n_shards, int64_t M, int64_t K, int64_t N, int dtype,
                          int64_t chunk_rows, int staging_slots) {
  if (check_problem(n_shards, M, K, N, dtype, chunk_rows) != AG_GEMM_OK) return nullptr;
  const bool skinny = dtype == AG_GEMM_I8 && M <= agg::kSkMaxRows;
  // the skinny path stages at most 127 x K bytes: it keeps the plain layout
  const bool bounded = staging_slots >= 0 && !skinny && n_shards > 1;
  if (staging_slots > 0 && staging_slots < agg::kGroupM) {
    fail(AG_GEMM_ERR_INVALID,
         "staging_slots must be 0 (default) or at least %d: the tiles of one swizzle group "
         "read %d row blocks at once", agg::kGroupM, agg::kGroupM);
    return nullptr;
  }
  if (bounded && chunk_rows > 0 && agg::kPairM % chunk_rows != 0) {
    fail(AG_GEMM_ERR_INVALID, "bounded staging needs chunk_rows dividing %d (got %lld)",
         agg::kPairM, (long long)chunk_rows);
    return nullptr;
  }
  if (bounded && chunk_rows == 0) chunk_rows = agg::choose_chunk_rows_bounded(M / n_shards);
  ag_gemm_plan* p = new (std::nothrow) ag_gemm_plan();
  if (!p) {
    fail(AG_GEMM_ERR_OOM, "host allocation failed");
    return nullptr;
  }
  agg::make_geometry(p->g, n_shards, M, K, N, dtype, chunk_rows);
  const Geometry& g = p->g;
  cudaError_t e;
  int major = 0, minor = 0;
  if ((e = cudaGetDevice(&p->device)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, p->device)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, p->device)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&p->sm_count, cudaDevAttrMultiProcessorCount, p->device)) != cudaSuccess) {
    cuda_fail(e, "device query");
    delete p;
    return nullptr;
  }
  if (major != 10 || minor != 3) {
    fail(AG_GEMM_ERR_UNSUPPORTED, "needs an sm_103 (GB300) device, found sm_%d%d", major, minor);
    delete p;
    return nullptr;
  }
  // One CTA per SM, in clusters of two (a CTA pair shares each MMA tile).
  int clusters = 0;
  const int want = (p->sm_count / 2) * 2;
  if ((e = agg::fused_max_clusters(dtype, want, &clusters)) != cudaSuccess || clusters < 1) {
    if (e == cudaSuccess) fail(AG_GEMM_ERR_UNSUPPORTED, "fused kernel clusters do not fit");
    else cuda_fail(e, "fused kernel occupancy");
    delete p;
    return nullptr;
  }
  p->grid = clusters * 2 < want ? clusters * 2 : want;
  const int64_t slots = g.S > 1 ? g.S - 1 : 1;
  if (bounded) {
    const int64_t blocks = static_cast<int64_t>(g.S - 1) * g.MT;
    const int64_t w = staging_slots == 0 ? 2 * agg::kGroupM : staging_slots;
    // a window as large as all remote row blocks is the plain layout
    p->window = w < blocks ? static_cast<int>(w) : 0;
  }
  // The last round's tiles of the fused kernel, split along K over the pairs
  // that would otherwise idle (not with a staging window, whose slot credits
  // count whole tiles).  Chosen for the full grid, so a smaller or larger grid
  // (ag_gemm_plan_set_grid) computes the same sums.
  p->split = (skinny || p->window > 0) ? 1 : agg::choose_split(g, p->grid / 2);
  const int64_t tail = p->split > 1 ? g.tiles % (p->grid / 2) : 0;
  p->full_tiles = g.tiles - tail;
  p->work_items = p->full_tiles + tail * p->split;
  const bool i8 = g.dtype == AG_GEMM_I8;
  // int8 parts hand partial sums to the last part; fp16 / bf16 parts add
  // into C blocks zeroed by 32-row tasks
  p->partials_bytes = i8 ? tail * (p->split - 1) * 2 * agg::kBlockM * g.BN * 4 : 0;
  p->zero_tasks = i8 ? 0 : tail * (agg::kPairM / 32);
  p->staging_bytes = p->window > 0 ? static_cast<int64_t>(p->window) * agg::kPairM * g.K * 2
                                   : slots * g.R * g.K * 2;
  p->skinny = skinny;
  if (skinny) {
    p->sk_tiles = (g.N + 255) / 256;
    p->sk_kq = (g.KB + 1) / 2;
    p->sk_np = agg::skinny_parts(g, p->sk_kq);
  }
  // one counter per chunk; on the skinny path one per (k-part, chunk)
  p->counter_count = slots * g.Q * (skinny ? p->sk_np : 1);
  if ((e = cudaMalloc(&p->staging, p->staging_bytes)) != cudaSuccess ||
      (e = cudaMalloc(&p->counters, sizeof(uint32_t) * p->counter_count)) != cudaSuccess ||
      (e = cudaMalloc(&p->item_counter, sizeof(unsigned long long))) != cudaSuccess ||
      (e = cudaMemset(p->item_counter, 0, sizeof(unsigned long long))) != cudaSuccess ||
      (e = cudaMalloc(&p->tile_counter, sizeof(unsigned long long))) != cudaSuccess ||
      (e = cudaMemset(p->tile_counter, 0, sizeof(unsigned long long))) != cudaSuccess ||
      (e = cudaMalloc(&p->status, 2 * sizeof(uint32_t))) != cudaSuccess ||
      (e = cudaMemset(p->counters, 0, sizeof(uint32_t) * p->counter_count)) != cudaSuccess ||
      (e = cudaMemset(p->status, 0, 2 * sizeof(uint32_t))) != cudaSuccess ||
      (e = cudaEventCreateWithFlags(&p->done, cudaEventDisableTiming)) != cudaSuccess ||
      (p->window > 0 &&
       ((e = cudaMalloc(&p->credits, sizeof(uint32_t) * p->window)) != cudaSuccess ||
        (e = cudaMemset(p->credits, 0, sizeof(uint32_t) * p->window)) != cudaSuccess)) ||
      (p->partials_bytes > 0 &&
       ((e = cudaMalloc(&p->partials, static_cast<size_t>(p->partials_bytes))) != cudaSuccess ||
        (e = cudaMalloc(&p->part_flags, sizeof(uint32_t) * tail)) != cudaSuccess ||
        (e = cudaMemset(p->part_flags, 0, sizeof(uint32_t) * tail)) != cudaSuccess)) ||
      (p->zero_tasks > 0 &&
       ((e = cudaMalloc(&p->zero_ticket, sizeof(unsigned long long))) != cudaSuccess ||
        (e = cudaMemset(p->zero_ticket, 0, sizeof(unsigned long long))) != cudaSuccess ||
        (e = cudaMalloc(&p->zero_done, sizeof(uint32_t))) != cudaSuccess ||
        (e = cudaMemset(p->zero_done, 0, sizeof(uint32_t))) != cudaSuccess))) {
    cuda_fail(e, "plan allocation");
    free_plan(p);
    return nullptr;
  }
  if (p->skinny) {
    p->sk_grid = p->sm_count;
    p->sk_cmax = agg::skinny_max_sharers(p->sk_tiles, p->sk_kq, p->sk_grid);
    if ((e = agg::skinny_prepare()) != cudaSuccess ||
        (e = cudaMalloc(&p->sk_ws, static_cast<size_t>(p->sk_tiles * p->sk_cmax * g.M * 256 * 4))) !=
            cudaSuccess) {
      cuda_fail(e, "plan allocation (skinny int8 path)");
      free_plan(p);
      return nullptr;
    }
    if (g.S > 1 && encode_stage8(&p->tm_stage8, p->staging, g.S - 1, g.R, g.K) != AG_GEMM_OK) {
      free_plan(p);
      return nullptr;
    }
  } else if (dtype == AG_GEMM_I8) {
    if ((e = cudaMalloc(&p->b16, static_cast<size_t>(g.K * g.N * 2))) != cudaSuccess ||
        (e = cudaMalloc(&p->a16, static_cast<size_t>(g.R * g.K * 2))) != cudaSuccess) {
      cuda_fail(e, "plan allocation (int8 widening buffers)");
      free_plan(p);
      return nullptr;
    }
    if (encode_a(&p->tm_a16, p->a16, g.R, g.K) != AG_GEMM_OK ||
        encode_b(&p->tm_b16, p->b16, g.K, g.N, g.N, g.BN) != AG_GEMM_OK) {
      free_plan(p);
      return nullptr;
    }
  }
  // staging map: [S-1][R][K], or the window's [W][256][K]
  if ((p->window > 0 ? encode_stage(&p->tm_stage, p->staging, p->window, agg::kPairM, g.K)
                     : encode_stage(&p->tm_stage, p->staging, slots, g.R, g.K)) != AG_GEMM_OK) {
    free_plan(p);
    return nullptr;
  }
  log_msg(2,
          "plan %p: %s path, S=%d M=%lld K=%lld N=%lld dtype=%d, chunk_rows=%lld (%lld chunks per "
          "source), %lld pair tiles, grid %d, split %d (%lld tail tiles), staging %lld B%s",
          static_cast<void*>(p), p->skinny ? "skinny" : "fused", g.S, (long long)g.M,
          (long long)g.K, (long long)g.N, g.dtype, (long long)g.c, (long long)g.Q,
          (long long)g.tiles, p->skinny ? p->sk_grid : p->grid, p->split,
          (long long)(g.tiles - p->full_tiles), (long long)p->staging_bytes,
          p->window > 0 ? " (staging window)" : "");
  return p;
}

}  // namespace

extern "C" {

ag_gemm_plan* ag_gemm_plan_create(int n_shards, int64_t M, int64_t K, int64_t N, int dtype,
                                  int64_t chunk_rows) {
  return create_plan(n_shards, M, K, N, dtype, chunk_rows, -1);
}

ag_gemm_plan* ag_gemm_plan_create_bounded(int n_shards, int64_t M, int64_t K, int64_t N,
                                          int dtype, int64_t chunk_rows, int staging_slots) {
  if (staging_slots < 0) {
    fail(AG_GEMM_ERR_INVALID, "staging_slots must be >= 0 (got %d)", staging_slots);
    return nullptr;
  }
  return create_plan(n_shards, M, K, N, dtype, chunk_rows, staging_slots);
}

int64_t ag_gemm_choose_chunk_rows_bounded(int64_t R) {
  if (R < 1) return fail(AG_GEMM_ERR_INVALID, "R must be positive");
  return agg::choose_chunk_rows_bounded(R);
}

void ag_gemm_plan_destroy(ag_gemm_plan* plan) {
  if (!plan) return;
  log_msg(2, "plan %p destroyed", static_cast<void*>(plan));
  DeviceGuard dg(plan->device);
  free_plan(plan);
}

int ag_gemm_plan_geometry(const ag_gemm_plan* plan, ag_gemm_geometry* out) {
  if (!plan || !out) return fail(AG_GEMM_ERR_INVALID, "plan or out is NULL");
  to_public(plan->g, out);
  if (plan->skinny) {
    // the skinny kernel's own tiling and allocations
    out->block_m = plan->g.M <= 64 ? 64 : 128;
    out->block_n = 256;
    out->m_tiles = 1;
    out->n_tiles = plan->sk_tiles;
    out->tiles = plan->sk_tiles;
    out->workspace_bytes = plan->staging_bytes +
                           static_cast<int64_t>(sizeof(uint32_t)) * plan->counter_count + 64 +
                           plan->sk_tiles * plan->sk_cmax * plan->g.M * 256 * 4;
  }
  if (!plan->skinny) {
    out->split_tiles = plan->g.tiles - plan->full_tiles;
    out->split_parts = plan->split;
    out->workspace_bytes += plan->partials_bytes + (plan->part_flags ? 4 * out->split_tiles : 0) +
                            (plan->zero_ticket ? 12 : 0);
  }
  if (plan->window > 0) {
    out->workspace_bytes += plan->staging_bytes - out->staging_bytes + 4 * plan->window;
    out->staging_bytes = plan->staging_bytes;
    out->staging_slots = plan->window;
  }
  return AG_GEMM_OK;
}

int64_t ag_gemm_plan_chunk_rows(const ag_gemm_plan* plan) {
  if (!plan) return fail(AG_GEMM_ERR_INVALID, "plan is NULL");
  return plan->g.c;
}

int ag_gemm_plan_grid(const ag_gemm_plan* plan) {
  if (!plan) return fail(AG_GEMM_ERR_INVALID, "plan is NULL");
  if (plan->skinny) return plan->sk_grid;
  return plan->grid_override > 0 ? plan->grid_override : plan->grid;
}

int ag_gemm_plan_path(const ag_gemm_plan* plan) {
  if (!plan) return fail(AG_GEMM_ERR_INVALID, "plan is NULL");
  if (plan->skinny) return AG_GEMM_PATH_SKINNY_I8;
  return plan->g.dtype == AG_GEMM_I8 ? AG_GEMM_PATH_FUSED_I8 : AG_GEMM_PATH_FUSED_F16;
}

int ag_gemm_run(ag_gemm_plan* plan, const void* const* shard_ptrs, const void* B, float* C,
                void* stream) {
  if (!plan) return fail(AG_GEMM_ERR_INVALID, "plan is NULL");
  if (plan->g.dtype == AG_GEMM_I8)
    return fail(AG_GEMM_ERR_INVALID,
                "ag_gemm_run needs an fp16 or bf16 plan (use ag_gemm_dequant_run)");
  return run_impl(plan, shard_ptrs, B, plan->g.N, C, plan->g.N, nullptr, nullptr, nullptr,
                  nullptr, stream);
}

int ag_gemm_run_ld(ag_gemm_plan* plan, const void* const* shard_ptrs, const void* B, int64_t ldb,
                   float* C, int64_t ldc, void* stream) {
  if (!plan) return fail(AG_GEMM_ERR_INVALID, "plan is NULL");
  if (plan->g.dtype == AG_GEMM_I8)
    return fail(AG_GEMM_ERR_INVALID, "ag_gemm_run_ld needs an fp16 or bf16 plan");
  return run_impl(plan, shard_ptrs, B, ldb, C, ldc, nullptr, nullptr, nullptr, nullptr, stream);
}

int ag_gemm_dequant_run(ag_gemm_plan* plan, const void* const* shard_ptrs, const void* B,
                        const int32_t* bias, const float* scale, int32_t* C_i32, void* D_f16,
                        void* stream) {
  if (!plan) return fail(AG_GEMM_ERR_INVALID, "plan is NULL");
  if (plan->g.dtype != AG_GEMM_I8)
    return fail(AG_GEMM_ERR_INVALID, "ag_gemm_dequant_run needs an int8 plan");
  return run_impl(plan, shard_ptrs, B, plan->g.N, nullptr, plan->g.N, C_i32, D_f16, bias, scale,
                  stream);
}

int64_t ag_gemm_plan_status_word(ag_gemm_plan* plan) {
  if (!plan) return fail(AG_GEMM_ERR_INVALID, "plan is NULL");
  DeviceGuard dg(plan->device);
  cudaError_t e;
  if (plan->has_run && (e = cudaEventSynchronize(plan->done)) != cudaSuccess)
    return cuda_fail(e, "cudaEventSynchronize");
  uint32_t w[2] = {0, 0};
  if ((e = cudaMemcpy(w, plan->status, sizeof(w), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "status read");
  return static_cast<int64_t>(w[0]) | (static_cast<int64_t>(w[1]) << 32);
}

int ag_gemm_plan_status(ag_gemm_plan* plan) {
  int64_t w = ag_gemm_plan_status_word(plan);
  if (w < 0) return static_cast<int>(w);
  const uint32_t kind = static_cast<uint32_t>(w & 0xFF);
  if (kind == agg::kStatusOk) return AG_GEMM_OK;
  return fail(AG_GEMM_ERR_TIMEOUT, "device wait timed out (status 0x%llx)", (unsigned long long)w);
}

int ag_gemm_plan_reset(ag_gemm_plan* plan, void* stream_v) {
  if (!plan) return fail(AG_GEMM_ERR_INVALID, "plan is NULL");
  DeviceGuard dg(plan->device);
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  cudaError_t e;
  if (plan->has_run && plan->last_stream != stream &&
      (e = cudaStreamWaitEvent(stream, plan->done, 0)) != cudaSuccess)
    return cuda_fail(e, "cudaStreamWaitEvent");
  if ((e = cudaMemsetAsync(plan->counters, 0, sizeof(uint32_t) * plan->counter_count, stream)) != cudaSuccess ||
      (e = cudaMemsetAsync(plan->item_counter, 0, sizeof(unsigned long long), stream)) != cudaSuccess ||
      (e = cudaMemsetAsync(plan->tile_counter, 0, sizeof(unsigned long long), stream)) != cudaSuccess ||
      (e = cudaMemsetAsync(plan->status, 0, 2 * sizeof(uint32_t), stream)) != cudaSuccess ||
      (plan->window > 0 && (e = cudaMemsetAsync(plan->credits, 0, sizeof(uint32_t) * plan->window,
                                                stream)) != cudaSuccess) ||
      (plan->part_flags &&
       (e = cudaMemsetAsync(plan->part_flags, 0,
                            sizeof(uint32_t) * (plan->g.tiles - plan->full_tiles), stream)) != cudaSuccess) ||
      (plan->zero_ticket &&
       ((e = cudaMemsetAsync(plan->zero_ticket, 0, sizeof(unsigned long long), stream)) != cudaSuccess ||
        (e = cudaMemsetAsync(plan->zero_done, 0, sizeof(uint32_t), stream)) != cudaSuccess)) ||
      (e = cudaEventRecord(plan->done, stream)) != cudaSuccess)
    return cuda_fail(e, "plan reset");
  plan->credit_epoch = 0;
  plan->part_epoch = 0;
  plan->zero_epoch = 0;
  plan->zero_base = 0;
  plan->epoch = 0;
  plan->item_base = 0;
  plan->tile_base = 0;
  plan->last_stream = stream;
  plan->has_run = true;
  return AG_GEMM_OK;
}

int ag_gemm_plan_set_mode(ag_gemm_plan* plan, int mode) {
  if (!plan) return fail(AG_GEMM_ERR_INVALID, "plan is NULL");
  if (mode < AG_GEMM_MODE_PIPELINED || mode > AG_GEMM_MODE_COPY_ONLY)
    return fail(AG_GEMM_ERR_INVALID, "unknown mode %d", mode);
  plan->mode = mode;
  return AG_GEMM_OK;
}

int ag_gemm_plan_set_local_rank(ag_gemm_plan* plan, int local_rank) {
  if (!plan) return fail(AG_GEMM_ERR_INVALID, "plan is NULL");
  if (local_rank < 0 || local_rank >= plan->g.S)
    return fail(AG_GEMM_ERR_INVALID, "local_rank %d out of [0, %d)", local_rank, plan->g.S);
  plan->local = local_rank;
  return AG_GEMM_OK;
}

int ag_gemm_plan_set_timeout_ns(ag_gemm_plan* plan, int64_t ns) {
  if (!plan) return fail(AG_GEMM_ERR_INVALID, "plan is NULL");
  if (ns <= 0) return fail(AG_GEMM_ERR_INVALID, "timeout must be positive");
  plan->timeout_ns = static_cast<uint64_t>(ns);
  return AG_GEMM_OK;
}

int ag_gemm_plan_set_grid(ag_gemm_plan* plan, int ctas) {
  if (!plan) return fail(AG_GEMM_ERR_INVALID, "plan is NULL");
  if (plan->skinny)
    return fail(AG_GEMM_ERR_UNSUPPORTED,
                "the skinny int8 path keeps one CTA per SM (its split-K slots are sized for it)");
  if (ctas != 0 && (ctas < 2 || ctas % 2 != 0 || ctas > 4 * plan->sm_count))
    return fail(AG_GEMM_ERR_INVALID, "ctas must be 0 or an even number in [2, %d] (got %d)",
                4 * plan->sm_count, ctas);
  plan->grid_override = ctas;
  return AG_GEMM_OK;
}

int ag_gemm_plan_set_debug(ag_gemm_plan* plan, int flags, int64_t arg) {
  if (!plan) return fail(AG_GEMM_ERR_INVALID, "plan is NULL");
  if (flags & ~(AG_GEMM_DEBUG_POISON_STAGING | AG_GEMM_DEBUG_SKIP_ITEM | AG_GEMM_DEBUG_DELAY_NS))
    return fail(AG_GEMM_ERR_INVALID, "unknown debug flags 0x%x", flags);
  if ((flags & AG_GEMM_DEBUG_SKIP_ITEM) && (flags & AG_GEMM_DEBUG_DELAY_NS))
    return fail(AG_GEMM_ERR_INVALID, "SKIP_ITEM and DELAY_NS share `arg`; set one at a time");
  if (arg < 0) return fail(AG_GEMM_ERR_INVALID, "arg must be >= 0");
  plan->debug_flags = flags;
  plan->debug_arg = arg;
  return AG_GEMM_OK;
}

int ag_gemm_plan_set_trace(ag_gemm_plan* plan, int64_t capacity) {
  if (!plan) return fail(AG_GEMM_ERR_INVALID, "plan is NULL");
  if (capacity < 0 || capacity > (int64_t{1} << 26))
    return fail(AG_GEMM_ERR_INVALID, "trace capacity must be in [0, 2^26] events (got %lld)",
                (long long)capacity);
  DeviceGuard dg(plan->device);
  cudaError_t e;
  // the buffer may still be written by the last run
  if (plan->has_run && (e = cudaEventSynchronize(plan->done)) != cudaSuccess)
    return cuda_fail(e, "cudaEventSynchronize");
  if ((e = cudaFree(plan->trace_buf)) != cudaSuccess) return cuda_fail(e, "cudaFree (trace)");
  plan->trace_buf = nullptr;
  plan->trace_cap = 0;
  if (capacity == 0) return AG_GEMM_OK;
  static_assert(sizeof(agg::TraceEvent) == sizeof(ag_gemm_trace_event), "trace event layout");
  void* buf = nullptr;
  const size_t bytes = 32 + static_cast<size_t>(capacity) * sizeof(agg::TraceEvent);
  if ((e = cudaMalloc(&buf, bytes)) != cudaSuccess) return cuda_fail(e, "trace allocation");
  if ((e = cudaMemset(buf, 0, 32)) != cudaSuccess) {
    cudaFree(buf);
    return cuda_fail(e, "trace allocation");
  }
  plan->trace_buf = static_cast<unsigned long long*>(buf);
  plan->trace_cap = capacity;
  return AG_GEMM_OK;
}

int64_t ag_gemm_plan_trace(ag_gemm_plan* plan, ag_gemm_trace_event* out, int64_t max_events) {
  if (!plan) return fail(AG_GEMM_ERR_INVALID, "plan is NULL");
  if (!plan->trace_buf) return fail(AG_GEMM_ERR_STATE, "tracing is off (ag_gemm_plan_set_trace)");
  if (max_events < 0 || (max_events > 0 && !out))
    return fail(AG_GEMM_ERR_INVALID, "out is NULL or max_events < 0");
  DeviceGuard dg(plan->device);
  cudaError_t e;
  if (plan->has_run && (e = cudaEventSynchronize(plan->done)) != cudaSuccess)
    return cuda_fail(e, "cudaEventSynchronize");
  // the dropped count, then every region; recorded events have a non-zero time
  std::vector<agg::TraceEvent> all;
  unsigned long long dropped = 0;
  try {
    all.resize(static_cast<size_t>(plan->trace_cap));
  } catch (...) {
    return fail(AG_GEMM_ERR_OOM, "host allocation for the trace failed");
  }
  if ((e = cudaMemcpy(&dropped, plan->trace_buf, sizeof(dropped), cudaMemcpyDeviceToHost)) != cudaSuccess ||
      (e = cudaMemcpy(all.data(), plan->trace_buf + 4, all.size() * sizeof(agg::TraceEvent),
                      cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "trace read");
  size_t kept = 0;
  for (size_t i = 0; i < all.size(); ++i)
    if (all[i].t_ns != 0) all[kept++] = all[i];
  all.resize(kept);
  std::stable_sort(all.begin(), all.end(), [](const agg::TraceEvent& a, const agg::TraceEvent& b) {
    return a.t_ns < b.t_ns;
  });
  const size_t n = kept < static_cast<size_t>(max_events) ? kept : static_cast<size_t>(max_events);
  if (n > 0) std::memcpy(out, all.data(), n * sizeof(agg::TraceEvent));
  return static_cast<int64_t>(kept + dropped);
}

int ag_gemm_last_error(void) { return g_last_error; }

const char* ag_gemm_last_error_message(void) { return g_last_msg; }

}  // extern "C"

// ------------------------------------------------------------------ no-allocation entry point
// The fp16 run above needs a plan, and a plan allocates its staging workspace,
// ready counters and status word with cudaMalloc.  This entry point runs the
// same fused kernel with all of that scratch taken from a fixed array that is
// part of the library's device image, so a call allocates nothing.
namespace {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;  // 64 MiB, held on every device that loads the library
constexpr size_t kNoAllocCtrlBytes = 512;              // status, item and tile counters (8 B each), padded
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocDevice {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int grid = 0;
};
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];
std::mutex g_noalloc_mu;

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Once per device, with that device current: find the array's device address
// (the host-side symbol is only a stand-in) and prepare the kernel.
int noalloc_setup(int dev, NoAllocDevice** out) {
  if (dev < 0 || dev >= kNoAllocMaxDevices)
    return fail(AG_GEMM_ERR_UNSUPPORTED, "device ordinal %d beyond %d", dev, kNoAllocMaxDevices);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocDevice& d = g_noalloc_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "device query");
    if (major != 10 || minor != 3)
      return fail(AG_GEMM_ERR_UNSUPPORTED, "needs an sm_103 (GB300) device, found sm_%d%d", major, minor);
    void* ptr = nullptr;
    if ((e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch)) != cudaSuccess)
      return cuda_fail(e, "cudaGetSymbolAddress of the no-allocation scratch array");
    int clusters = 0;
    const int want = (sms / 2) * 2;
    if ((e = agg::fused_max_clusters(AG_GEMM_F16, want, &clusters)) != cudaSuccess)
      return cuda_fail(e, "fused kernel occupancy");
    if (clusters < 1) return fail(AG_GEMM_ERR_UNSUPPORTED, "fused kernel clusters do not fit");
    d.scratch = static_cast<unsigned char*>(ptr);
    d.grid = clusters * 2 < want ? clusters * 2 : want;
    d.ready = true;
  }
  *out = &d;
  return AG_GEMM_OK;
}

}  // namespace

extern "C" int ag_gemm_run_noalloc(int n_shards, int64_t M, int64_t K, int64_t N,
                                   int64_t chunk_rows, const void* const* shard_ptrs,
                                   const void* B, float* C, uint32_t* status_out,
                                   void* stream_v) {
  int rc = check_problem(n_shards, M, K, N, AG_GEMM_F16, chunk_rows);
  if (rc != AG_GEMM_OK) return rc;
  Geometry g;
  agg::make_geometry(g, n_shards, M, K, N, AG_GEMM_F16, chunk_rows);
  const int64_t slots = g.S > 1 ? g.S - 1 : 1;
  const size_t counter_bytes = round256(sizeof(uint32_t) * static_cast<size_t>(slots * g.Q));
  const size_t staging_bytes = static_cast<size_t>(slots * g.R * g.K * 2);
  const size_t need = kNoAllocCtrlBytes + counter_bytes + staging_bytes;
  if (need > kNoAllocScratchBytes)
    return fail(AG_GEMM_ERR_UNSUPPORTED,
                "ag_gemm_run_noalloc: this problem needs %zu bytes of scratch, more than the "
                "library's fixed %zu-byte array (use a plan instead)",
                need, kNoAllocScratchBytes);
  if (!shard_ptrs) return fail(AG_GEMM_ERR_INVALID, "shard_ptrs is NULL");
  for (int s = 0; s < g.S; ++s)
    if (!shard_ptrs[s] || !aligned16(shard_ptrs[s]))
      return fail(AG_GEMM_ERR_INVALID, "shard_ptrs[%d] is NULL or not 16-byte aligned", s);
  if (!B || !aligned16(B)) return fail(AG_GEMM_ERR_INVALID, "B is NULL or not 16-byte aligned");
  if (!C || !aligned16(C)) return fail(AG_GEMM_ERR_INVALID, "C is NULL or not 16-byte aligned");
  if (status_out && (reinterpret_cast<uintptr_t>(status_out) & 7u))
    return fail(AG_GEMM_ERR_INVALID, "status_out is not 8-byte aligned");

  int dev = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  NoAllocDevice* d = nullptr;
  if ((rc = noalloc_setup(dev, &d)) != AG_GEMM_OK) return rc;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);

  unsigned char* ctrl = d->scratch;
  uint32_t* status = reinterpret_cast<uint32_t*>(ctrl);
  unsigned long long* item_counter = reinterpret_cast<unsigned long long*>(ctrl + 256);
  unsigned long long* tile_counter = reinterpret_cast<unsigned long long*>(ctrl + 384);
  uint32_t* counters = reinterpret_cast<uint32_t*>(ctrl + kNoAllocCtrlBytes);
  unsigned char* staging = ctrl + kNoAllocCtrlBytes + counter_bytes;

  agg::FusedParams fp;
  std::memset(&fp, 0, sizeof(fp));
  fp.g = g;
  for (int pos = 0; pos < g.S; ++pos) fp.src[pos] = shard_ptrs[agg::source_of(g, 0, pos)];
  if ((rc = encode_a(&fp.tm_a_local, fp.src[0], g.R, g.K)) != AG_GEMM_OK ||
      (rc = encode_b(&fp.tm_b, B, g.K, g.N, g.N, g.BN)) != AG_GEMM_OK ||
      (rc = encode_stage(&fp.tm_a_stage, staging, slots, g.R, g.K)) != AG_GEMM_OK ||
      (rc = encode_c(&fp.tm_c, C, g.S, g.R, g.N, g.N)) != AG_GEMM_OK)
    return rc;
  fp.staging = staging;
  fp.counters = counters;
  fp.item_counter = item_counter;
  fp.item_base = 0;
  fp.tile_counter = tile_counter;
  fp.tile_base = 0;
  fp.full_tiles = g.tiles;  // whole tiles only: no partial-sum workspace
  fp.work_items = g.tiles;
  fp.split = 1;
  fp.static_items = g.tiles;  // every tile dealt round-robin
  fp.zero_tasks = 0;
  fp.zero_ticket = nullptr;
  fp.zero_base = 0;
  fp.zero_done = nullptr;
  fp.zero_target = 0;
  fp.status = status;
  fp.C = C;
  fp.local = 0;
  fp.b3d = b_is_3d(g.N) ? 1 : 0;
  fp.epoch = 1;
  fp.timeout_ns = 1000000000ull;
  fp.pipe_timeout_ns = 4000000000ull;
  fp.debug_skip_item = -1;
  fp.flags = agg::kFlagGemm | agg::kFlagWait | (g.S > 1 ? agg::kFlagCopy : 0);
  // Every call shares the array and finds the previous call's values in it:
  // the status word, the item and tile counters and the ready counters must start at zero.
  if ((e = cudaMemsetAsync(ctrl, 0, kNoAllocCtrlBytes + counter_bytes, stream)) != cudaSuccess)
    return cuda_fail(e, "clearing the no-allocation scratch");
  if ((e = agg::launch_fused(fp, d->grid, stream)) != cudaSuccess)
    return cuda_fail(e, "fused kernel launch");
  if (status_out &&
      (e = cudaMemcpyAsync(status_out, status, 2 * sizeof(uint32_t), cudaMemcpyDeviceToDevice,
                           stream)) != cudaSuccess)
    return cuda_fail(e, "status copy");
  return AG_GEMM_OK;
}
