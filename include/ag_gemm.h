/*
 * ag_gemm.h -- C ABI of the GB300 (sm_103a) streamed AllGather+GEMM library
 * (libaggemm.so).
 *
 * What it computes
 *   C = AllGather(A) x B.  A (M x K) arrives as n_shards row shards of
 *   R = M / n_shards rows each; shard s owns global rows [s*R, (s+1)*R).
 *   B (K x N) is replicated.  Each shard is cut into chunks of chunk_rows rows
 *   and the GEMM consumes a chunk as soon as it has landed, instead of after
 *   the whole gather ("AllGather + GEMM 通算融合算子示例", sections 计算功能
 *   and 流式流水线).  One GPU holds every shard ("simulated ranks"): the local
 *   shard is read in place, every other shard is copied chunk by chunk into a
 *   plan-owned staging workspace, and a per-chunk ready counter is released
 *   after each copy.
 *
 *   fp16 path (ag_gemm_run): fp16 A and B, fp32 accumulation, fp32 C.
 *   int8 path (ag_gemm_dequant_run), "AllGather矩阵乘法反量化算子设计文档"
 *   sections 1.2 and 2.2:
 *       C_i32[m][n] = sum_k A[m][k] * B[k][n] + bias[n]          (exact int32)
 *       D[m][n]     = fp16_rn( fp32_rn( fp32_rn(C_i32[m][n]) * scale[n] ) )
 *
 * Conventions (every entry point)
 *   - Matrices are dense and row-major: shard s is R x K, B is K x N, C, C_i32
 *     and D are M x N.  Row m of C belongs to shard m / R.
 *   - All matrix, vector and workspace pointers are DEVICE pointers of the
 *     current CUDA device; shard_ptrs itself is a HOST array of n_shards
 *     device pointers.  The caller owns every pointer it passes; the library
 *     never frees them and keeps none of them after the call returns
 *     (except as keys of a cache of TMA descriptors).
 *   - Every device pointer must be 16-byte aligned.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Runs
 *     are asynchronous: on return the work is enqueued on `stream`, and any
 *     later work on `stream` observes C (and C_i32 / D) complete.  Runs on one
 *     plan are serialised by the library: a run on a different stream first
 *     waits for the plan's previous run.
 *   - Errors are returned as negative ag_gemm_status codes (or NULL from
 *     ag_gemm_plan_create); the thread-local ag_gemm_last_error() and
 *     ag_gemm_last_error_message() describe the last failure.  Nothing aborts
 *     and no C++ exception crosses this boundary.
 *   - Logging: the environment variable AG_GEMM_LOG (read once per process)
 *     makes the library write lines starting "[ag_gemm] " to stderr: 1 every
 *     error as it is raised, 2 also each plan's geometry, path, grid and split
 *     at creation and its destruction, 3 also every run enqueued.  Unset or 0:
 *     silent.
 */
#ifndef AG_GEMM_H
#define AG_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ag_gemm_plan ag_gemm_plan;

typedef enum {
    AG_GEMM_F16 = 0,  /* fp16 x fp16 -> fp32 */
    AG_GEMM_I8 = 1,   /* int8 x int8 -> int32 (+bias) -> fp16 dequant */
    AG_GEMM_BF16 = 2  /* bf16 x bf16 -> fp32 (the operand type of "Collective matrix
                         multiplication", section 使用 Pallas 实现; the fp16 path otherwise) */
} ag_gemm_dtype;

typedef enum {
    AG_GEMM_OK = 0,
    AG_GEMM_ERR_INVALID = -1,     /* bad shape, pointer, alignment or argument */
    AG_GEMM_ERR_UNSUPPORTED = -2, /* not an sm_103 device, or a size limit */
    AG_GEMM_ERR_CUDA = -3,        /* a CUDA runtime/driver call failed */
    AG_GEMM_ERR_OOM = -4,         /* device allocation failed */
    AG_GEMM_ERR_TIMEOUT = -5,     /* a device-side wait ran out (see status) */
    AG_GEMM_ERR_STATE = -6        /* the call does not fit the plan's state */
} ag_gemm_status;

/*
 * Run modes (the three benchmark modes of "AllGather + GEMM 通算融合算子示例",
 * section Benchmark 与输出说明, plus a copy-only mode):
 *   PIPELINED    -- chunk copies and GEMM run concurrently; the GEMM waits on
 *                   each remote chunk's ready counter (the method itself).
 *   COMPUTE_ONLY -- GEMM only; every chunk is treated as ready and the staging
 *                   workspace is read as it stands (it must hold the current
 *                   shards from an earlier run for C to be right).
 *   SEQUENTIAL   -- all chunk copies complete, then the GEMM runs.
 *   COPY_ONLY    -- chunk copies only; C is not written.
 * A plan with a staging window (ag_gemm_plan_create_bounded) cannot run
 * SEQUENTIAL (AG_GEMM_ERR_UNSUPPORTED): the copy would have to run ahead of
 * the GEMM by the whole gather.  Its COMPUTE_ONLY runs read the window as it
 * stands (timing only: earlier row blocks have been overwritten).
 */
typedef enum {
    AG_GEMM_MODE_PIPELINED = 0,
    AG_GEMM_MODE_COMPUTE_ONLY = 1,
    AG_GEMM_MODE_SEQUENTIAL = 2,
    AG_GEMM_MODE_COPY_ONLY = 3
} ag_gemm_mode;

/* Debug knobs for race and failure testing (ag_gemm_plan_set_debug). */
typedef enum {
    AG_GEMM_DEBUG_NONE = 0,
    AG_GEMM_DEBUG_POISON_STAGING = 1, /* fill staging with NaN / 0x7E before each run */
    AG_GEMM_DEBUG_SKIP_ITEM = 2,      /* producer skips copy item `arg` (its chunk never becomes
                                         ready); on the skinny path copy task `arg`, one k-part
                                         of one chunk (see AG_GEMM_TRACE_LANDED) */
    AG_GEMM_DEBUG_DELAY_NS = 4        /* producer sleeps `arg` ns before each copy item */
} ag_gemm_debug_flag;

/* Which kernels a plan runs (ag_gemm_plan_path). */
typedef enum {
    AG_GEMM_PATH_FUSED_F16 = 0,  /* fp16 / bf16: the fused copy + tcgen05 GEMM kernel (CTA pairs) */
    AG_GEMM_PATH_FUSED_I8 = 1,   /* int8, M > 128: B and the local shard widened to fp16,
                                    then the fused kernel with the exact int8 epilogue */
    AG_GEMM_PATH_SKINNY_I8 = 2   /* int8, M <= 128: the B-streaming skinny kernel and its
                                    finish kernel (bias, dequant) */
} ag_gemm_path;

/* Sizes the library derives from a problem (no GPU needed to compute them). */
typedef struct {
    int32_t n_shards;
    int32_t dtype;
    int64_t M, K, N, R;
    int64_t chunk_rows;        /* c: rows per chunk */
    int64_t chunks_per_source; /* Q = R / c */
    int32_t pieces_per_chunk;  /* P: copy items per chunk (counter target = epoch * P) */
    int32_t block_m, block_n, block_k;
    int32_t group_m;           /* m-tiles per swizzle group */
    int32_t kseg_blocks;       /* int8 path: k-blocks accumulated in fp32 before an int32 fold */
    int64_t m_tiles;           /* per source */
    int64_t n_tiles;
    int64_t tiles;             /* n_shards * m_tiles * n_tiles */
    int64_t producer_items;    /* (n_shards - 1) * Q * P */
    int64_t staging_bytes;     /* plan-owned staging workspace */
    int64_t workspace_bytes;   /* everything the plan allocates on the device */
    int64_t staging_slots;     /* staging window in 256-row slots; 0 = one place per remote row */
    int64_t split_tiles;       /* fused kernel: tiles computed in K-parts by several CTA pairs
                                  (the last round's tiles; ag_gemm_plan_geometry only) */
    int64_t split_parts;       /* parts per split tile (1 = no split) */
} ag_gemm_geometry;

/*
 * Chunk size rule (ComputeOptimalChunkSize of "AllGather + GEMM 通算融合算子示例",
 * section 优化说明: keep 64-128 chunks per source).  For R rows per source:
 * Q = the smallest divisor of R in [64, 128], c = R / Q; if R has no such
 * divisor, c = the largest divisor of R with R / c >= 64; if R < 64, c = 1.
 * Returns c, or AG_GEMM_ERR_INVALID for R < 1.  Pure host function.
 */
int64_t ag_gemm_choose_chunk_rows(int64_t R);

/*
 * Check a problem without touching the GPU: n_shards in [1, 64], M, K, N > 0,
 * M % n_shards == 0, chunk_rows == 0 (auto) or a divisor of R;
 * fp16 and bf16: K % 8 == 0 and N % 8 == 0; int8: K % 16 == 0, N % 16 == 0 and
 * K <= 133000 (so that K * 127^2 plus a bias stays inside int32).
 * Returns AG_GEMM_OK or the error code (and sets the last error).
 */
int ag_gemm_validate(int n_shards, int64_t M, int64_t K, int64_t N, int dtype,
                     int64_t chunk_rows);

/* Fill *out with the derived sizes of a valid problem.  Pure host function. */
int ag_gemm_geometry_of(int n_shards, int64_t M, int64_t K, int64_t N,
                        int dtype, int64_t chunk_rows, ag_gemm_geometry *out);

/*
 * Persistent tile schedule, as the kernel walks it.  Tile t in
 * [0, geometry.tiles) maps to out[0] = source shard (global rank), out[1] =
 * m-tile within that shard, out[2] = n-tile.  Tiles are ordered by
 * consumption position p = 0..n_shards-1, where position p holds shard
 * (local_rank + p) % n_shards: the local shard first with no wait, then the
 * remote shards in ring order ("Collective matrix multiplication", section
 * Ring All-Gather: at step i device d computes A_{(d+i) % D}).  Within a
 * shard, tiles are swizzled in groups of group_m m-tiles.
 */
int ag_gemm_tile_at(const ag_gemm_geometry *g, int local_rank, int64_t t,
                    int64_t out[3]);

/*
 * Producer copy item i in [0, geometry.producer_items): out[0] = source
 * shard, out[1] = chunk index q within it, out[2] / out[3] = first / one-past-
 * last byte of the shard covered by the item.  Items are numbered in
 * consumption order (the send order equals the consumption order,
 * "AllGather + GEMM 通算融合算子示例" section 优化说明) and handed to the
 * producer warps round-robin.
 */
int ag_gemm_item_at(const ag_gemm_geometry *g, int local_rank, int64_t i,
                    int64_t out[4]);

/*
 * Create a plan on the current CUDA device: validates the problem (as
 * ag_gemm_validate), requires an sm_103 device, and allocates the staging
 * workspace ((n_shards-1) x R x K 2-byte elements), the per-chunk ready counters and a
 * status word (plus, for int8, fp16 copies of B and of the local shard).
 * chunk_rows = 0 picks c with ag_gemm_choose_chunk_rows.
 * Returns NULL on failure (see ag_gemm_last_error()).
 */
ag_gemm_plan *ag_gemm_plan_create(int n_shards, int64_t M, int64_t K,
                                  int64_t N, int dtype, int64_t chunk_rows);

/*
 * Create a plan whose remote rows pass through a bounded staging window with
 * back-pressure (the double-buffered workspace of "AllGather + GEMM 通算融合算子
 * 示例" section 优化说明 and of "AllGather矩阵乘法反量化算子设计文档" 6.1: two
 * workspace stages that the producer refills once the consumer is done).
 *
 * The remote rows, in consumption order, form row blocks of 256 rows (one
 * m-tile of a shard; the last block of a shard may be shorter): block
 * b = (p - 1) * m_tiles + mt for consumption position p >= 1.  Block b is
 * staged in slot b % W of a [W][256][K] workspace.  Every tile that has read
 * its rows adds one credit to the slot's counter; the producer writes block b
 * only after the n_tiles tiles of block b - W have done so.  The tiles of a
 * swizzle group (group_m = 8 m-tiles) read their blocks together, so W must
 * be at least 8; staging_slots = 0 picks W = 16, two groups: one being read
 * while the producer fills the other.  A window that covers every remote
 * block is the plain layout (geometry.staging_slots = 0).  The staging then
 * takes W * 256 * K * 2 bytes instead of (n_shards - 1) * R * K * 2.
 *
 * A chunk must not straddle a slot: chunk_rows must divide 256 (and R);
 * chunk_rows = 0 picks ag_gemm_choose_chunk_rows_bounded(R).  int8 plans with
 * M <= 128 (the skinny path, whose staging is at most 127 x K bytes) keep the
 * plain layout.  Producer waits on a slot are bounded by the plan's timeout
 * and end in the status kind 3 (credit timeout).
 */
ag_gemm_plan *ag_gemm_plan_create_bounded(int n_shards, int64_t M, int64_t K,
                                          int64_t N, int dtype, int64_t chunk_rows,
                                          int staging_slots);

/*
 * Chunk rule of a plan with a staging window: ag_gemm_choose_chunk_rows(R)
 * when it divides 256; else the largest power of two dividing R and 256 with
 * R / c >= 64; else 1.  Pure host function.
 */
int64_t ag_gemm_choose_chunk_rows_bounded(int64_t R);

/* Wait for the plan's last run, then free everything the plan owns. NULL is a no-op. */
void ag_gemm_plan_destroy(ag_gemm_plan *plan);

/*
 * The derived sizes of a plan.  For a plan on the skinny int8 path
 * (AG_GEMM_PATH_SKINNY_I8) the tile fields describe that kernel: block_m = 64
 * or 128 (the MMA's rows: M rounded up), block_n = 256, m_tiles = 1,
 * n_tiles = tiles = ceil(N / 256), and workspace_bytes counts its split-K
 * slots instead of fp16 copies of B and the local shard.
 */
int ag_gemm_plan_geometry(const ag_gemm_plan *plan, ag_gemm_geometry *out);

/* c actually used by the plan, or a negative status. */
int64_t ag_gemm_plan_chunk_rows(const ag_gemm_plan *plan);

/*
 * fp16 (or bf16, for an AG_GEMM_BF16 plan) AllGather+GEMM.  shard_ptrs: host
 * array of n_shards device pointers, each to an R x K fp16 (bf16) matrix;
 * B: K x N fp16 (bf16); C: M x N fp32 (written, every element), accumulated in
 * fp32.  Enqueues the work on `stream` (see the run modes).
 */
int ag_gemm_run(ag_gemm_plan *plan, const void *const *shard_ptrs,
                const void *B, float *C, void *stream);

/*
 * ag_gemm_run with row pitches: B element (k, n) at B[k * ldb + n] and C
 * element (m, n) at C[m * ldc + n] (ldb, ldc >= N; ldb % 8 == 0 and
 * ldc % 4 == 0, i.e. 16-byte row pitches; the base pointers 16-byte aligned).
 * Columns of a row past N are neither read nor written.
 *
 * This is the N-sharded layout of "Collective matrix multiplication"
 * (sections 算法概述：Ring All-Gather and 将 kernel 与 JAX 集成): A is
 * sharded by rows, B by columns, and rank d computes AllGather(A) x B_d, the
 * column block d of C, taking the row slices of its output in ring order
 * d, d+1, ..., d+D-1 (mod D) -- on this library, a plan with
 * ag_gemm_plan_set_local_rank(plan, d).  With one GPU holding every rank,
 * rank d passes B_d = B + d * n_shard and C_d = C + d * n_shard with
 * ldb = ldc = D * n_shard (so n_shard % 8 == 0 for alignment).
 * fp16 and bf16 plans only (AG_GEMM_ERR_INVALID otherwise).
 */
int ag_gemm_run_ld(ag_gemm_plan *plan, const void *const *shard_ptrs,
                   const void *B, int64_t ldb, float *C, int64_t ldc, void *stream);

/*
 * int8 AllGatherMatmulDequant.  shard_ptrs: n_shards device pointers to
 * R x K int8; B: K x N int8; bias: N int32; scale: N fp32; C_i32: M x N int32
 * and D_f16: M x N fp16, both written.  If |A x B + bias| reaches 2^31 the
 * int32 result wraps (two's complement) -- keep |bias| < 2^31 - K * 127^2.
 */
int ag_gemm_dequant_run(ag_gemm_plan *plan, const void *const *shard_ptrs,
                        const void *B, const int32_t *bias, const float *scale,
                        int32_t *C_i32, void *D_f16, void *stream);

/*
 * Wait for the plan's last run and read its device status word: AG_GEMM_OK,
 * or AG_GEMM_ERR_TIMEOUT if a wait on a ready counter or a pipeline barrier
 * ran out (C is then undefined).  A timed-out plan keeps failing until
 * ag_gemm_plan_reset.
 */
int ag_gemm_plan_status(ag_gemm_plan *plan);

/* Raw status word of the last run (0 = ok; low byte = kind: 1 a ready counter,
 * 2 a pipeline barrier, 3 a staging-window slot ran out of time). */
int64_t ag_gemm_plan_status_word(ag_gemm_plan *plan);

/* Zero the ready counters and the status word on `stream`; the epoch restarts. */
int ag_gemm_plan_reset(ag_gemm_plan *plan, void *stream);

/* Select an ag_gemm_mode for later runs (default PIPELINED). */
int ag_gemm_plan_set_mode(ag_gemm_plan *plan, int mode);

/*
 * Which shard is local (default 0).  It only changes the consumption order
 * (local first, then (local+1) % n, ...); C does not depend on it.
 */
int ag_gemm_plan_set_local_rank(ag_gemm_plan *plan, int local_rank);

/* Limit of every device-side wait, in ns (default 1e9; must be > 0). */
int ag_gemm_plan_set_timeout_ns(ag_gemm_plan *plan, int64_t ns);

/* OR of ag_gemm_debug_flag values; `arg` is the item index or the delay. */
int ag_gemm_plan_set_debug(ag_gemm_plan *plan, int flags, int64_t arg);

/*
 * Per-run event trace (opt-in): when each chunk landed in the staging, when
 * each consumer started and stopped waiting for remote rows, and a few
 * pipeline milestones, stamped with the GPU's global nanosecond timer.  It
 * shows the overlap of the copy and the GEMM, the measurement the PTO example
 * ships as its overlap analysis ("AllGather + GEMM 通算融合算子示例", section
 * 目录结构, prof_analysis).  A plan with tracing on runs the trace-enabled
 * instantiation of its kernels (slower: every event is a global atomic); with
 * tracing off the kernels contain no trace code.
 *
 * Event kinds and the meaning of id / aux:
 *   CTA_START, CTA_END    thread 0 of a CTA (id = aux = 0)
 *   LANDED                a copy warp finished a copy item and is about to
 *                         release its ready counter: id = counter index,
 *                         aux = item index.  Fused paths: counter
 *                         (p - 1) * Q + q of chunk q at consumption position
 *                         p, item as ag_gemm_item_at.  Skinny path: a copy
 *                         task (k-part j, position p, chunk q) with counter
 *                         (j * (n_shards - 1) + p - 1) * Q + q.
 *   WAIT_START, WAIT_END  the TMA warp before / after acquiring remote rows.
 *                         Fused: id = tile, aux = p << 48 | q0 << 24 | q1
 *                         (chunks q0..q1 of position p; one pair per CTA of a
 *                         pair tile).  Skinny: id = unit, aux = k-part j.
 *   TILE_DONE             fused: an epilogue warp issued its last store of a work item
 *                         (id = tile, aux = part | parts << 8; parts = 1 for a whole tile)
 *   ACC_READY             fused: the accumulator of a work item's last segment is ready
 *                         for the epilogue (id, aux as for TILE_DONE)
 *   PARTS_READY           fused, split tile: int8 -- its last part saw every earlier
 *                         part's partial sums stored; fp16 / bf16 -- a part saw the run's
 *                         zeroing of the tail tiles done, before its first reduction into
 *                         C (id = tile)
 *   UNIT_ISSUED           skinny: a unit's loads issued (id = unit)
 *   UNIT_LANDED           skinny: a unit's operands in shared memory (id = unit)
 *   KB_WIDENED            skinny: a k-block of B widened to fp16 (id = k-block of the n-tile, aux = unit)
 *   KB_MMA                skinny: a k-block's MMAs issued (id = k-block of the n-tile, aux = n-tile)
 *   PIECE_DONE            skinny: a CTA's split-K sums of one n-tile stored (id = n-tile, aux = next unit)
 *   COPY_START            a copy warp starts a copy item (id, aux as for LANDED)
 */
typedef enum {
    AG_GEMM_TRACE_CTA_START = 1,
    AG_GEMM_TRACE_CTA_END = 2,
    AG_GEMM_TRACE_LANDED = 3,
    AG_GEMM_TRACE_WAIT_START = 4,
    AG_GEMM_TRACE_WAIT_END = 5,
    AG_GEMM_TRACE_TILE_DONE = 6,
    AG_GEMM_TRACE_UNIT_ISSUED = 7,
    AG_GEMM_TRACE_UNIT_LANDED = 8,
    AG_GEMM_TRACE_KB_WIDENED = 9,
    AG_GEMM_TRACE_KB_MMA = 10,
    AG_GEMM_TRACE_PIECE_DONE = 11,
    AG_GEMM_TRACE_COPY_START = 12,
    AG_GEMM_TRACE_ACC_READY = 13,
    AG_GEMM_TRACE_PARTS_READY = 14
} ag_gemm_trace_kind;

typedef struct {
    uint64_t t_ns;   /* the GPU's global nanosecond timer (%globaltimer) */
    uint32_t kind;   /* ag_gemm_trace_kind */
    uint32_t cta;    /* CTA index within its launch */
    uint32_t warp;   /* warp index within the CTA */
    uint32_t id;     /* per kind, see above */
    uint64_t aux;    /* per kind, see above */
} ag_gemm_trace_event;

/*
 * Turn tracing on (capacity > 0 events, at most 2^26; allocates
 * 32 + 32 * capacity bytes on the device) or off (capacity = 0, frees the
 * buffer).  Waits for the plan's last run.  Every later run clears the trace
 * and records its own events.  The capacity is split evenly between the
 * launch's CTAs, 32 warp slots each (an event is a plain store into its
 * warp's region, so tracing does not serialise the kernel on atomics); events
 * past a region's share are dropped and counted.
 */
int ag_gemm_plan_set_trace(ag_gemm_plan *plan, int64_t capacity);

/*
 * Wait for the plan's last run and copy up to max_events of its events,
 * sorted by time, to the HOST array out.  Returns the number of events the
 * run tried to record (kept + dropped), or a negative status
 * (AG_GEMM_ERR_STATE when tracing is off).
 */
int64_t ag_gemm_plan_trace(ag_gemm_plan *plan, ag_gemm_trace_event *out, int64_t max_events);

/*
 * Number of CTAs the fused kernel launches (fp16, bf16 and int8 plans with
 * M > 128): 0 = the default, one CTA per SM in CTA pairs; otherwise an even
 * number in [2, 4 * SMs].  Pair tiles are handed out at run time in schedule
 * order, so any grid computes the same C: a smaller grid simply has fewer
 * pairs, and a grid larger than the GPU holds at once leaves the extra pairs
 * to start as others finish (they find the tiles taken and exit) -- the
 * partial residency a GPU shared with other work can also cause.
 * AG_GEMM_ERR_UNSUPPORTED on the skinny int8 path (one CTA per SM, fixed).
 */
int ag_gemm_plan_set_grid(ag_gemm_plan *plan, int ctas);

/* Number of CTAs the plan's main kernel launches (one per SM unless set). */
int ag_gemm_plan_grid(const ag_gemm_plan *plan);

/* The ag_gemm_path the plan runs (fixed at creation by dtype and M); a
 * negative ag_gemm_status if plan is NULL. */
int ag_gemm_plan_path(const ag_gemm_plan *plan);

/*
 * fp16 AllGather+GEMM that allocates nothing (the pages have no counterpart
 * of this entry point).  It is for callers that are not allowed to call
 * cudaMalloc: for example a host application whose own allocator has already
 * reserved the device's memory, or a latency-critical path on which
 * cudaMalloc/cudaFree (which may synchronise the device and can take
 * unbounded time) are not acceptable.  It runs the same PIPELINED fused kernel
 * as ag_gemm_run with local rank 0, but the staging workspace, ready counters
 * and status word live in a fixed 64 MiB array inside the library's device
 * image, which every GPU that loads the library holds until the process
 * exits.  Arguments are as for ag_gemm_plan_create + ag_gemm_run
 * (chunk_rows = 0 picks the chunk size); the caller still provides the
 * shards, B and C.  status_out (device pointer, 2 x uint32, 8-byte aligned,
 * may be NULL) receives the status word of the run (0 = ok, low byte 1 or 2 =
 * a device wait timed out).
 *
 * Limits and behaviour:
 *  - the problem must need at most 64 MiB of scratch: 512 B + the counters
 *    ((n_shards-1) * chunks per source * 4 B, rounded to 256 B) + the staging
 *    workspace ((n_shards-1) * R * K * 2 B); larger problems are rejected with
 *    AG_GEMM_ERR_UNSUPPORTED and a message giving the size needed;
 *  - the first call on a device (with that device current) looks up the
 *    array's device address and prepares the kernel; make that first call
 *    before any stream capture;
 *  - every call clears the counters and status in the array on `stream`
 *    before its kernel; calls share the one array, so calls whose work
 *    overlaps on the GPU (different streams without ordering between them)
 *    race and give wrong results.
 */
int ag_gemm_run_noalloc(int n_shards, int64_t M, int64_t K, int64_t N,
                        int64_t chunk_rows, const void *const *shard_ptrs,
                        const void *B, float *C, uint32_t *status_out,
                        void *stream);

/* Thread-local code and text of the last error raised on this thread. */
int ag_gemm_last_error(void);
const char *ag_gemm_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* AG_GEMM_H */
