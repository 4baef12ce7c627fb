// Split-plan arithmetic shared by the host planner and the device planner, so
// that both cut every sequence into the same pieces (and the two paths give
// bit-identical results).  The occupancy rule is the NSPLIT fix of "The Build
// That Unlocked 3-6x Decode Speedup", section "Broader Significance": enough
// key pieces that the work units fill the GPU, chosen per sequence from its
// length.
#pragma once

#include <stdint.h>

#include "vmla_internal.h"

#ifdef __CUDACC__
#define VMLA_HD __host__ __device__ __forceinline__
#else
#define VMLA_HD inline
#endif

namespace vmla {

// Planner knobs of each kernel family.
VMLA_HD PlanShape plan_shape(int kernel) {
  PlanShape s;
  if (kernel == VMLA_KERNEL_SIMT) {
    s.rows_per_unit = 32;
    s.units_per_sm = 2;
    s.key_align = 32;
    s.min_chunk = 256;
    s.max_splits = 64;
  } else {
    // tensor-core kernel: one unit = 256 query rows on a cluster of four SMs
    // (a scorer pair and a mixer pair); the piece size is chosen per call among
    // candidates (plan_cand_chunk), two units per cluster being the default
    s.rows_per_unit = 256;
    s.units_per_sm = 2;  // per cluster of four SMs; the caller divides the SM count
    s.key_align = 128;   // the kernel's tile
    s.min_chunk = 128;   // one tile: a small workload is spread over every cluster
    s.max_splits = 64;
  }
  return s;
}

VMLA_HD int64_t plan_ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Status of one sequence's lengths (0 <= Q_b <= 64 drafts, N_b >= Q_b keys).
VMLA_HD int plan_check_seq(int64_t nq, int64_t nk) {
  return (nq < 0 || nq > VMLA_MAX_DRAFT || nk < nq) ? VMLA_ERR_SHAPE : VMLA_OK;
}

// Work of one sequence: (row blocks) x (keys); 0 when it has no queries.
VMLA_HD int64_t plan_seq_work(const PlanShape& sh, int64_t nq, int64_t nk, int num_heads) {
  return nq == 0 ? 0 : plan_ceil_div(nq * num_heads, sh.rows_per_unit) * nk;
}

// Row blocks of a sequence with nq drafts (rows_per_unit is a power of two).
VMLA_HD int64_t plan_row_blocks(const PlanShape& sh, int64_t nq, int num_heads) {
  // nq H <= 64 x 128: 32-bit arithmetic
  return ((uint32_t)(nq * num_heads) + (uint32_t)sh.rows_per_unit - 1u) / (uint32_t)sh.rows_per_unit;
}

// Keys per piece the planner aims at so that `slots` units run at once.
VMLA_HD int64_t plan_chunk_target(const PlanShape& sh, int64_t total_work, int64_t slots) {
  const int64_t per = plan_ceil_div(total_work > 1 ? total_work : 1, slots);
  return per > sh.min_chunk ? per : (int64_t)sh.min_chunk;
}

// Piece length and count of a sequence of nk >= 1 keys for a chunk target (or
// a forced count): the length is rounded up to the key alignment (a power of
// two in both kernel families), then the count is the one that leaves no
// piece empty.
VMLA_HD void plan_pieces(const PlanShape& sh, int64_t nk, int splits, int64_t chunk_target, int64_t* chunk,
                         int64_t* pieces) {
  // nk < 2^31 (int32 offsets), so every sum and quotient below fits 32 bits
  const uint32_t n = (uint32_t)nk, align = (uint32_t)sh.key_align;
  uint32_t p = splits > 0 ? (uint32_t)splits
               : chunk_target >= nk ? 1u
                                    : (n + (uint32_t)chunk_target - 1u) / (uint32_t)chunk_target;
  if (p > (uint32_t)sh.max_splits) p = (uint32_t)sh.max_splits;
  if (p < 1u) p = 1u;
  const uint32_t c = ((n + p - 1u) / p + align - 1u) & ~(align - 1u);
  *chunk = c;
  *pieces = (n + c - 1u) / c;
}

// Pieces of one sequence: fills n_rb, n_split and chunk of `s` (whose kv/q
// lengths are set) and returns its units; *part_rows / *merge_rows receive the
// fp32 partial rows and merge rows it needs.
VMLA_HD int64_t plan_split_seq(const PlanShape& sh, SeqPlan& s, int num_heads, int splits, int64_t chunk_target,
                               int64_t* part_rows, int64_t* merge_rows) {
  *part_rows = 0;
  *merge_rows = 0;
  if (s.n_q == 0) {
    s.n_rb = 0;
    s.n_split = 1;
    s.chunk = s.n_kv > 1 ? s.n_kv : 1;
    return 0;
  }
  const int64_t rows = (int64_t)s.n_q * num_heads;
  s.n_rb = (int32_t)plan_ceil_div(rows, sh.rows_per_unit);
  int64_t chunk = 0, pieces = 0;
  plan_pieces(sh, s.n_kv, splits, chunk_target, &chunk, &pieces);
  s.chunk = (int32_t)chunk;
  s.n_split = (int32_t)pieces;
  if (pieces > 1) {
    *part_rows = rows * pieces;
    *merge_rows = rows;
  }
  return (int64_t)s.n_rb * pieces;
}

// ---------------------------------------------------------------- piece size of the tensor-core kernel
// A unit's cost for the cluster schedule: its keys plus a fixed charge for
// loading Q, filling and draining the pipeline and writing the result (about
// three 128-key tiles' time, measured on the verify kernel).
constexpr int64_t kUnitFixedKeys = 384;

VMLA_HD int64_t plan_unit_cost(const SeqPlan& s, int unit) {
  const int64_t piece = (unit - s.unit_start) / s.n_rb;
  const int64_t lo = piece * s.chunk;
  const int64_t hi = lo + s.chunk < s.n_kv ? lo + s.chunk : (int64_t)s.n_kv;
  return (hi - lo) + kUnitFixedKeys;
}

// The planner picks the chunk target among kChunkCands candidates: candidate k
// aims at m_k / 16 units per cluster on average (m from 12 to 192; candidate
// kDefaultCand, m = 32, is two units per cluster).  Each candidate's units are
// scored by the longest cluster load of a snake deal of the units sorted by
// cost, plus the merge: its fp32 partial rows are written and read back at
// about a twentieth of a key's time each, and a merge launch costs a tile.  A
// candidate replaces the default only if it scores at least 3 % lower.
// Batches of more than kSearchMaxBatch sequences keep the default.
constexpr int kChunkCands = 32;
constexpr int kDefaultCand = 10;
constexpr int kSearchMaxBatch = 64;
constexpr int kRunsPerSeq = 2;  // a sequence's units: its full pieces and its last piece
constexpr int64_t kMergeRowsPerKey = 20;
constexpr int64_t kMergeLaunchKeys = 128;

VMLA_HD int64_t plan_merge_score(int64_t partial_rows) {
  return partial_rows / kMergeRowsPerKey + (partial_rows > 0 ? kMergeLaunchKeys : 0);
}

VMLA_HD int plan_cand_m(int k) {
  if (k < 10) return 12 + 2 * k;            // 12 .. 30
  if (k < 20) return 32 + 4 * (k - 10);     // 32 .. 68
  if (k < 28) return 72 + 8 * (k - 20);     // 72 .. 128
  return 144 + 16 * (k - 28);               // 144 .. 192
}

VMLA_HD int64_t plan_cand_chunk(const PlanShape& sh, int64_t total_work, int clusters, int k) {
  const int64_t ct = plan_ceil_div((total_work > 1 ? total_work : 1) * 16, (int64_t)clusters * plan_cand_m(k));
  return ct > sh.min_chunk ? ct : (int64_t)sh.min_chunk;
}

// The two runs of equal-cost units of one sequence under a chunk target:
// cost[0] x count[0] full pieces, cost[1] x count[1] last pieces (counts 0 for
// a sequence without queries); returns the sequence's fp32 partial rows.
// rb: the sequence's row blocks, ceil(nq H / rows_per_unit) (the caller computes it
// once for all candidates).
VMLA_HD int64_t plan_seq_runs(const PlanShape& sh, int64_t nq, int64_t nk, int num_heads, int64_t rb,
                              int64_t chunk_target, int64_t (&cost)[kRunsPerSeq], int64_t (&count)[kRunsPerSeq]) {
  cost[0] = cost[1] = 0;
  count[0] = count[1] = 0;
  if (nq == 0) return 0;
  int64_t chunk = 0, pieces = 0;
  plan_pieces(sh, nk, 0, chunk_target, &chunk, &pieces);
  cost[0] = chunk + kUnitFixedKeys;
  count[0] = rb * (pieces - 1);
  cost[1] = nk - (pieces - 1) * chunk + kUnitFixedKeys;
  count[1] = rb;
  return pieces > 1 ? nq * num_heads * pieces : 0;
}

// Units at positions p < x of a snake deal over C clusters (positions
// 0..C-1 go to clusters 0..C-1, positions C..2C-1 to clusters C-1..0, and so
// on) that land on cluster j.
VMLA_HD int64_t plan_snake_share(int64_t x, int j, int C) {
  // x <= kMaxTcUnits and 2C <= 2 kMaxClusters: 32-bit division (a 64-bit one is a
  // slow emulated sequence on the GPU, where this runs for every run and cluster)
  const uint32_t period = 2u * (uint32_t)C, xx = (uint32_t)x;
  const uint32_t q = xx / period, rem = xx - q * period;
  return 2 * (int64_t)q + (rem > (uint32_t)j ? 1 : 0) + (rem > period - 1u - (uint32_t)j ? 1 : 0);
}

// Sort position of run r among runs sorted by cost (descending), ties by run
// index: the units of all runs that come before it.
VMLA_HD bool plan_run_before(int64_t cost_a, int a, int64_t cost_b, int b) {
  return cost_a > cost_b || (cost_a == cost_b && a < b);
}

// The chosen candidate from the candidates' scores (-1: not a candidate).
VMLA_HD int plan_choose_cand(const int64_t* score) {
  int best = -1;
  for (int k = 0; k < kChunkCands; ++k)
    if (score[k] >= 0 && (best < 0 || score[k] < score[best])) best = k;
  const int64_t d = score[kDefaultCand];
  if (best < 0 || (d >= 0 && !(score[best] * 100 < d * 97))) best = kDefaultCand;
  return best;
}

// ---------------------------------------------------------------- lane plan of the tensor-core kernel
// The uniform plan deals equal pieces to the clusters; when the sequences'
// lengths do not divide into the clusters evenly its longest cluster load can
// sit well above the mean.  The lane plan instead cuts the work where the
// clusters' shares end (the wrap-around rule for splittable jobs on identical
// machines: lay the jobs end to end and cut every L): each stream (G row blocks
// of one sequence over all its key tiles) occupies its tiles plus a fixed
// charge in a cost space, and lane l takes [l L, (l + 1) L).  The G clusters of
// a lane take the G row blocks of the same stream pieces, so that they read the
// same key tiles at about the same time and share them through L2.  A stream
// cut into several pieces leaves fp32 partials that the merge combines; a
// stream within one lane writes its rows directly.
constexpr int kLaneMaxWidth = 4;
constexpr int64_t kUnitFixedTiles = kUnitFixedKeys / 128;
// A stream's fixed charge in the lane plan's cost space, in tiles.
constexpr int64_t kLaneStreamTiles = 5;

// Widths 2..kLaneMaxWidth that do not divide a sequence's row-block count (bit g).
VMLA_HD uint32_t plan_lane_misfit(int64_t n_rb) {
  uint32_t m = 0;
  if (n_rb > 0)
    for (int g = 2; g <= kLaneMaxWidth; ++g)
      if (n_rb % g != 0) m |= 1u << g;
  return m;
}

// Lane width: the largest g <= kLaneMaxWidth that divides every sequence's row
// blocks (the OR of their misfit masks), so that every stream has G row blocks.
VMLA_HD int plan_lane_width(uint32_t misfit) {
  for (int g = kLaneMaxWidth; g >= 2; --g)
    if (!(misfit & (1u << g))) return g;
  return 1;
}

VMLA_HD int64_t plan_seq_tiles(int64_t nk) { return (nk + 127) / 128; }

// Cost-space length of one stream of a sequence with nk keys: its tiles, then the fixed charge.
VMLA_HD int64_t plan_stream_span(int64_t nk) { return plan_seq_tiles(nk) + kLaneStreamTiles; }

// Pieces of a stream whose T tiles start at cost position a: the lanes of length L it meets.
// (a + T <= W <= INT32_MAX in a lane plan: 32-bit arithmetic.)
VMLA_HD int64_t plan_stream_pieces(int64_t a, int64_t T, int64_t L) {
  const uint32_t aa = (uint32_t)a, ll = (uint32_t)L;
  return (int64_t)((aa + (uint32_t)T - 1u) / ll - aa / ll) + 1;
}

// Lane length for total cost W over `lanes` lanes (at least one tile).
VMLA_HD int64_t plan_lane_tiles(int64_t W, int lanes) {
  const int64_t L = plan_ceil_div(W, lanes > 0 ? lanes : 1);
  return L > 0 ? L : 1;
}

// Query rows of stream g of a sequence with R rows (its last row block may be short).
VMLA_HD int64_t plan_stream_rows(int64_t g, int64_t rows_per_stream, int64_t R) {
  const int64_t hi = (g + 1) * rows_per_stream < R ? (g + 1) * rows_per_stream : R;
  return hi - g * rows_per_stream;
}

// Pieces (the most of any of its streams), partial rows and merge rows (the
// rows of its streams cut into more than one piece) of sequence b in a lane
// plan whose streams of b start at cost position c0: n_groups streams of span
// each, R = Q_b H query rows, rows_per_stream = G x 256.
VMLA_HD int64_t plan_lane_seq_split(int64_t c0, int64_t n_groups, int64_t nk, int64_t L, int64_t R,
                                    int64_t rows_per_stream, int64_t* part_rows, int64_t* merge_rows,
                                    int64_t* pieces_sum) {
  const int64_t T = plan_seq_tiles(nk), span = plan_stream_span(nk);
  int64_t most = 1, sum = 0, merge = 0;
  for (int64_t g = 0; g < n_groups; ++g) {
    const int64_t p = plan_stream_pieces(c0 + g * span, T, L);
    most = p > most ? p : most;
    sum += p;
    if (p > 1) merge += plan_stream_rows(g, rows_per_stream, R);
  }
  *part_rows = most > 1 ? R * most : 0;
  *merge_rows = merge;
  *pieces_sum = sum;
  return most;
}

// Score of a lane plan in the uniform plan's units (keys): a lane carries at
// most L plus the fixed charge of the stream it continues, and the merge.
VMLA_HD int64_t plan_lane_score(int64_t L, int64_t partial_rows) {
  return (L + kUnitFixedTiles) * 128 + plan_merge_score(partial_rows);
}

// The lane plan replaces the chosen uniform plan when it scores at least 3 % lower.
VMLA_HD bool plan_prefer_lanes(int64_t lane_score, int64_t uniform_score) {
  return uniform_score >= 0 && lane_score * 100 < uniform_score * 97;
}

}  // namespace vmla
