// schedule.h -- problem geometry, persistent tile order and producer copy
// items of the streamed AllGather+GEMM.  Used by the host plan code and by the
// device kernels, so that both walk exactly the same schedule.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define AGG_HD __host__ __device__ __forceinline__
#else
#define AGG_HD inline
#endif

namespace agg {

constexpr int kMaxShards = 64;
constexpr int kBlockM = 128;        // rows per CTA (one TMEM lane per row)
constexpr int kPairM = 256;         // rows of a CTA-pair tile (tcgen05 cta_group::2, M = 256)
constexpr int kBlockK = 64;         // fp16 elements per k-block: one 128-byte swizzle row
constexpr int kUmmaK = 16;          // K of one tcgen05.mma kind::f16
constexpr int kStages = 6;          // TMA -> MMA shared-memory ring depth
constexpr int kMaxBlockN = 256;
constexpr int kGroupM = 8;          // m-tiles per swizzle group
// int8 emulation: |a*b| <= 127^2 = 16129 and 16 k-blocks = 1024 terms keep every
// fp32 partial sum an integer below 2^24, hence exact.
constexpr int kSegBlocks = 16;
constexpr int64_t kPieceBytes = 32 * 1024;  // target source bytes per copy item
constexpr int64_t kMaxKI8 = 133000;

struct Geometry {
  int S;
  int dtype;             // 0 = f16, 1 = i8, 2 = bf16
  int64_t M, K, N, R;
  int64_t c;             // chunk rows
  int64_t Q;             // chunks per source
  int P;                 // copy items (pieces) per chunk
  int BN;                // block_n of a pair tile (each CTA loads BN / 2 columns of B)
  int64_t MT, NT;        // pair m-tiles (256 rows) per source, n-tiles
  int64_t tiles;
  int64_t KB;            // k-blocks
  int64_t items;         // producer copy items
  int64_t src_esize;     // bytes per source element (2 for f16, 1 for i8)
};

AGG_HD int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ComputeOptimalChunkSize analogue: 64..128 chunks per source.
AGG_HD int64_t choose_chunk_rows(int64_t R) {
  if (R < 1) return -1;
  if (R < 64) return 1;
  for (int64_t q = 64; q <= 128; ++q)
    if (R % q == 0) return R / q;
  int64_t best = 1;
  for (int64_t c = 1; c <= R / 64; ++c)
    if (R % c == 0) best = c;
  return best;
}

// Chunk rule of a plan with bounded staging: a chunk must lie inside one
// 256-row slot, so c divides 256 as well as R.  The unbounded rule's c when it
// does; else the largest common divisor of R and 256 that keeps >= 64 chunks
// per source; else 1.
AGG_HD int64_t choose_chunk_rows_bounded(int64_t R) {
  const int64_t c0 = choose_chunk_rows(R);
  if (c0 < 1 || kPairM % c0 == 0) return c0;
  int64_t best = 1;
  for (int64_t c = 1; c <= kPairM && c <= R / 64; c *= 2)
    if (R % c == 0) best = c;
  return best;
}

AGG_HD void make_geometry(Geometry& g, int S, int64_t M, int64_t K, int64_t N,
                          int dtype, int64_t chunk_rows) {
  g.S = S; g.dtype = dtype; g.M = M; g.K = K; g.N = N;
  g.R = M / S;
  g.c = chunk_rows > 0 ? chunk_rows : choose_chunk_rows(g.R);
  g.Q = g.R / g.c;
  g.src_esize = dtype == 1 ? 1 : 2;
  int64_t chunk_bytes = g.c * K * g.src_esize;
  int64_t p = ceil_div(chunk_bytes, kPieceBytes);
  int64_t vecs = chunk_bytes / 16;
  if (p > vecs) p = vecs;
  if (p < 1) p = 1;
  g.P = (int)p;
  g.BN = N <= 128 ? 128 : 256;
  g.MT = ceil_div(g.R, kPairM);
  g.NT = ceil_div(N, g.BN);
  g.tiles = (int64_t)S * g.MT * g.NT;
  g.KB = ceil_div(K, kBlockK);
  g.items = (int64_t)(S - 1) * g.Q * g.P;
}

// Tile t -> (consumption position, m-tile, n-tile).  Position 0 is the local
// shard; within a position, groups of kGroupM m-tiles are walked m-fastest.
// (32-bit arithmetic: a plan has fewer than 2^31 tiles, checked at validation.
// The kernels decode a tile at every tile boundary, where 64-bit divisions
// would delay the first loads of the next tile.)
AGG_HD void tile_coords(const Geometry& g, int64_t t, int& pos, int64_t& mt,
                        int64_t& nt) {
  const uint32_t MT = static_cast<uint32_t>(g.MT), NT = static_cast<uint32_t>(g.NT);
  const uint32_t per = MT * NT, t32 = static_cast<uint32_t>(t);
  const uint32_t p32 = t32 / per;
  const uint32_t u = t32 - p32 * per;
  const uint32_t group = static_cast<uint32_t>(kGroupM) * NT;
  const uint32_t gi = u / group;
  const uint32_t first_m = gi * static_cast<uint32_t>(kGroupM);
  const uint32_t gm = MT - first_m < static_cast<uint32_t>(kGroupM) ? MT - first_m
                                                                    : static_cast<uint32_t>(kGroupM);
  const uint32_t w = u - gi * group;
  const uint32_t n32 = w / gm;
  pos = static_cast<int>(p32);
  mt = first_m + (w - n32 * gm);
  nt = n32;
}

// Work items of the fused kernel: the first `full` tiles whole, then the
// remaining (tail) tiles in `split` parts along K -- the tiles that would
// leave most CTA pairs idle in the last round.  Tail items go part-major (the
// first part of every tail tile, then the second ...), so on the int8 path,
// where they are drawn, the last part of a tile, which adds the others'
// partial sums, is handed out after all of them.
// Item i -> tile t, part j of `parts`, and the part's k-blocks [kb0, kb1).
AGG_HD void work_item(const Geometry& g, int64_t full, int split, int64_t i, int64_t& t,
                      int& part, int& parts, int64_t& kb0, int64_t& kb1) {
  if (i < full) {
    t = i;
    part = 0;
    parts = 1;
    kb0 = 0;
    kb1 = g.KB;
    return;
  }
  // (32-bit: fewer than 2^31 tiles, K < 2^31 so KB * split < 2^32)
  const uint32_t tail = static_cast<uint32_t>(g.tiles - full);
  const uint32_t r = static_cast<uint32_t>(i - full);
  const uint32_t pj = r / tail;
  const uint32_t kb = static_cast<uint32_t>(g.KB), s = static_cast<uint32_t>(split);
  part = static_cast<int>(pj);
  t = full + (r - pj * tail);
  parts = split;
  kb0 = kb * pj / s;
  kb1 = kb * (pj + 1) / s;
}

// Parts per tail tile for `pairs` CTA pairs: tiles % pairs tiles are left for
// the last round.  When they fill at most half of the pairs, each is split in
// two along K, which halves that round -- worth it when a tile is long enough
// for the parts' extra work.  int8 parts hand partial sums to the last part
// (a store, a wait and an addition: a few microseconds whatever K; a half
// tile of 64 k-blocks saves only ~10 us), so only tiles of at least 128
// k-blocks (K >= 8192) are split.  fp16 / bf16 parts add into C blocks
// zeroed at the start of the run, with TMA reductions that cost what the
// plain store costs, so tiles of at least 32 k-blocks (K >= 2048) are.
inline int choose_split(const Geometry& g, int64_t pairs) {
  if (pairs < 2) return 1;
  const int64_t tail = g.tiles % pairs;
  const int64_t min_kb = g.dtype == 1 ? 128 : 32;  // int8 : fp16 / bf16
  if (tail == 0 || 2 * tail > pairs || g.KB < min_kb) return 1;
  return 2;
}

AGG_HD int source_of(const Geometry& g, int local, int pos) {
  return (local + pos) % g.S;
}

// Copy item i -> (consumption position >= 1, chunk q, piece p) and the
// 16-byte-vector range [v0, v1) of the source chunk it covers.
AGG_HD void item_coords(const Geometry& g, int64_t i, int& pos, int64_t& q,
                        int& piece, int64_t& v0, int64_t& v1) {
  int64_t per_pos = g.Q * g.P;
  pos = 1 + (int)(i / per_pos);
  int64_t r = i - (int64_t)(pos - 1) * per_pos;
  q = r / g.P;
  piece = (int)(r - q * g.P);
  int64_t vecs = g.c * g.K * g.src_esize / 16;
  v0 = vecs * piece / g.P;
  v1 = vecs * (piece + 1) / g.P;
}

// Bounded staging: row block b = (pos - 1) * MT + mt of the remote rows lives
// in slot b % W; before its use u = b / W (u >= 1) the slot's credit counter
// must reach base + u * NT, where base counts the credits of earlier runs:
// (epoch - 1) * (uses of the slot per run) * NT.
AGG_HD int64_t window_uses(const Geometry& g, int64_t W, int64_t slot) {
  const int64_t nb = (int64_t)(g.S - 1) * g.MT;
  return slot < nb ? (nb - slot + W - 1) / W : 0;
}
AGG_HD uint32_t window_target(const Geometry& g, int64_t W, int64_t b, uint32_t epoch) {
  const int64_t slot = b % W, use = b / W;
  return static_cast<uint32_t>((int64_t)(epoch - 1) * window_uses(g, W, slot) * g.NT +
                               use * g.NT);
}

// Chunks [q0, q1] of a source that the 128 rows starting at row0 touch;
// false if the rows lie past the end of the shard.
AGG_HD bool rows_chunks(const Geometry& g, int64_t row0, int64_t& q0, int64_t& q1) {
  if (row0 >= g.R) return false;
  int64_t r1 = row0 + kBlockM < g.R ? row0 + kBlockM : g.R;
  const uint32_t c = static_cast<uint32_t>(g.c);  // (R <= 2^31)
  q0 = static_cast<uint32_t>(row0) / c;
  q1 = static_cast<uint32_t>(r1 - 1) / c;
  return true;
}

// Skinny int8 path: the U (n-tile, 2-k-block) units are cut into G contiguous
// per-CTA ranges; CTA b takes [U b / G, U (b + 1) / G).
AGG_HD void skinny_cta_range(int64_t U, int64_t b, int64_t G, int64_t& lo, int64_t& hi) {
  lo = U * b / G;
  hi = U * (b + 1) / G;
}
// The CTA whose range holds unit x (the largest b with U b / G <= x).
AGG_HD int64_t skinny_owner(int64_t x, int64_t U, int64_t G) {
  return ((x + 1) * G + U - 1) / U - 1;
}
// Skinny int8 path, streamed gather: every unit reads all gathered rows, but
// only 128 k of them, so the remote rows are copied and released in k-parts
// and a unit waits only for the part that holds its k-slice.  np parts split
// the KQ units of an n-tile: part j covers units [KQ j / np, KQ (j + 1) / np)
// (k in [128 KQ j / np, 128 KQ (j + 1) / np), clipped at K).  A copy task is
// (part j, consumption position pos >= 1, chunk q): the c rows of the chunk
// over the part's k-range, released on counter (j (S - 1) + pos - 1) Q + q.
// Tasks are numbered part-major, then by position, then by chunk.
AGG_HD int skinny_parts(const Geometry& g, int64_t KQ) {
  int64_t np = ceil_div(g.c * g.K, 2048);  // ~2 KB of source per task
  if (np > 32) np = 32;
  if (np > KQ) np = KQ;
  return np < 1 ? 1 : static_cast<int>(np);
}
AGG_HD int skinny_part_of(int64_t qu, int64_t KQ, int np) {
  return static_cast<int>(((qu + 1) * np + KQ - 1) / KQ - 1);
}
// (32-bit arithmetic: a skinny plan has at most 127 remote rows, K <= 133000.)
AGG_HD void skinny_task(const Geometry& g, int64_t KQ, int np, int64_t t, int& j, int& pos,
                        int64_t& q, int64_t& k0, int64_t& k1) {
  const uint32_t Q = static_cast<uint32_t>(g.Q), per_part = static_cast<uint32_t>(g.S - 1) * Q;
  const uint32_t t32 = static_cast<uint32_t>(t), kq = static_cast<uint32_t>(KQ);
  j = static_cast<int>(t32 / per_part);
  const uint32_t r = t32 - static_cast<uint32_t>(j) * per_part;
  pos = 1 + static_cast<int>(r / Q);
  q = r - static_cast<uint32_t>(pos - 1) * Q;
  k0 = 128 * static_cast<int64_t>(kq * static_cast<uint32_t>(j) / static_cast<uint32_t>(np));
  k1 = 128 * static_cast<int64_t>(kq * static_cast<uint32_t>(j + 1) / static_cast<uint32_t>(np));
  if (k1 > g.K) k1 = g.K;
}
AGG_HD int64_t skinny_counter(const Geometry& g, int j, int pos, int64_t q) {
  return ((int64_t)j * (g.S - 1) + (pos - 1)) * g.Q + q;
}

// Most CTAs that share one n-tile of KQ units: the workspace slots per n-tile.
inline int64_t skinny_max_sharers(int64_t n_tiles, int64_t KQ, int64_t G) {
  const int64_t U = n_tiles * KQ;
  int64_t most = 1;
  for (int64_t nt = 0; nt < n_tiles; ++nt) {
    const int64_t c = skinny_owner((nt + 1) * KQ - 1, U, G) - skinny_owner(nt * KQ, U, G) + 1;
    if (c > most) most = c;
  }
  return most;
}

}  // namespace agg
