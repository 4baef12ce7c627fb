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
    // (a scorer pair and a mixer pair); about two units per cluster leave the
    // greedy schedule room to balance
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

// Keys per piece the planner aims at so that `slots` units run at once.
VMLA_HD int64_t plan_chunk_target(const PlanShape& sh, int64_t total_work, int64_t slots) {
  const int64_t per = plan_ceil_div(total_work > 1 ? total_work : 1, slots);
  return per > sh.min_chunk ? per : (int64_t)sh.min_chunk;
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
  int64_t pieces = splits > 0 ? (int64_t)splits : plan_ceil_div(s.n_kv, chunk_target);
  if (pieces > sh.max_splits) pieces = sh.max_splits;
  if (pieces < 1) pieces = 1;
  // piece length rounded to the key alignment, then the count that leaves no piece empty
  const int64_t chunk = plan_ceil_div(plan_ceil_div(s.n_kv, pieces), sh.key_align) * sh.key_align;
  pieces = plan_ceil_div(s.n_kv, chunk);
  s.chunk = (int32_t)chunk;
  s.n_split = (int32_t)pieces;
  if (pieces > 1) {
    *part_rows = rows * pieces;
    *merge_rows = rows;
  }
  return (int64_t)s.n_rb * pieces;
}

// Cost of a tensor-core work unit for the cluster schedule: its keys plus a
// fixed charge for filling and draining the pipeline.
VMLA_HD int64_t plan_unit_cost(const SeqPlan& s, int unit) {
  const int64_t piece = (unit - s.unit_start) / s.n_rb;
  const int64_t lo = piece * s.chunk;
  const int64_t hi = lo + s.chunk < s.n_kv ? lo + s.chunk : (int64_t)s.n_kv;
  return (hi - lo) + 256;
}

}  // namespace vmla
