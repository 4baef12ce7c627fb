// Host-side split planner and workspace layout.
//
// The key range of every sequence is cut into contiguous pieces so that the
// work units (query-row block x key piece) fill the GPU: the occupancy fix
// that raised NSPLIT in "The Build That Unlocked 3-6x Decode Speedup",
// section "Broader Significance", chosen here per sequence from its length
// and the SM count instead of one global constant.
#include <algorithm>
#include <cstring>
#include <vector>

#include "vmla_internal.h"

namespace vmla {

PlanShape plan_shape(int kernel) {
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
    s.min_chunk = 1024;
    s.max_splits = 64;
  }
  return s;
}

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

WorkspaceLayout workspace_layout(int64_t total_q, int64_t partial_rows, int64_t staged_rows) {
  auto up = [](size_t x) { return (x + VMLA_WORKSPACE_ALIGN - 1) / VMLA_WORKSPACE_ALIGN * VMLA_WORKSPACE_ALIGN; };
  WorkspaceLayout w;
  w.status_off = 0;
  w.masks_off = up(16);
  w.part_o_off = w.masks_off + up((size_t)total_q * 8);
  w.part_lse_off = w.part_o_off + up((size_t)partial_rows * kDv * 4);
  w.staged_off = w.part_lse_off + up((size_t)partial_rows * 4);
  w.total = w.staged_off + up((size_t)staged_rows * kRowBytes);
  return w;
}

int build_plan(int kernel, int batch, int num_heads, const int32_t* qo, const int32_t* kv, int splits, int num_sms,
               int tc_clusters, PlanParams* pp, vmla_plan_info* info) {
  if (!qo || !kv || !pp) return VMLA_ERR_NULL;
  if (kernel != VMLA_KERNEL_TC && kernel != VMLA_KERNEL_SIMT) return VMLA_ERR_SHAPE;
  if (batch < 0 || batch > VMLA_MAX_BATCH || num_heads < 1 || num_heads > VMLA_MAX_HEADS) return VMLA_ERR_SHAPE;
  if (splits < 0 || num_sms < 1) return VMLA_ERR_SHAPE;
  if (qo[0] != 0 || kv[0] != 0) return VMLA_ERR_SHAPE;
  for (int b = 0; b < batch; ++b) {
    int64_t nq = (int64_t)qo[b + 1] - qo[b];
    int64_t nk = (int64_t)kv[b + 1] - kv[b];
    if (nq < 0 || nq > VMLA_MAX_DRAFT || nk < nq) return VMLA_ERR_SHAPE;
  }
  const PlanShape sh = plan_shape(kernel);
  std::memset(pp, 0, sizeof(PlanParams));
  pp->batch = batch;
  pp->num_heads = num_heads;
  pp->rows_per_unit = sh.rows_per_unit;

  // slots: units that run at once
  const int clusters = tc_clusters > 0 ? tc_clusters : std::max(1, num_sms / 4);
  int64_t slots = kernel == VMLA_KERNEL_TC ? (int64_t)clusters * sh.units_per_sm : (int64_t)num_sms * sh.units_per_sm;
  int64_t total_work = 0;  // (row block) x (keys)
  for (int b = 0; b < batch; ++b) {
    int64_t nq = qo[b + 1] - qo[b], nk = kv[b + 1] - kv[b];
    if (nq == 0) continue;
    total_work += ceil_div(nq * num_heads, sh.rows_per_unit) * nk;
  }
  int64_t chunk_target = std::max<int64_t>(sh.min_chunk, ceil_div(std::max<int64_t>(total_work, 1), slots));

  int64_t unit = 0, part = 0, merge = 0;
  int max_s = 0;
  for (int b = 0; b < batch; ++b) {
    SeqPlan& s = pp->seq[b];
    s.kv_off = kv[b];
    s.n_kv = kv[b + 1] - kv[b];
    s.q_off = qo[b];
    s.n_q = qo[b + 1] - qo[b];
    s.unit_start = (int32_t)unit;
    s.merge_off = (int32_t)merge;
    s.part_off = (int32_t)part;
    if (s.n_q == 0) {
      s.n_rb = 0;
      s.n_split = 1;
      s.chunk = std::max(1, s.n_kv);
      continue;
    }
    int64_t rows = (int64_t)s.n_q * num_heads;
    s.n_rb = (int32_t)ceil_div(rows, sh.rows_per_unit);
    int64_t pieces;
    if (splits > 0) {
      pieces = splits;
    } else {
      pieces = ceil_div(s.n_kv, chunk_target);
    }
    pieces = std::max<int64_t>(1, std::min<int64_t>(pieces, sh.max_splits));
    // piece length rounded to the key alignment, then the count that leaves no piece empty
    int64_t chunk = ceil_div(ceil_div(s.n_kv, pieces), sh.key_align) * sh.key_align;
    pieces = ceil_div(s.n_kv, chunk);
    s.chunk = (int32_t)chunk;
    s.n_split = (int32_t)pieces;
    unit += (int64_t)s.n_rb * pieces;
    if (pieces > 1) {
      part += rows * pieces;
      merge += rows;
    }
    max_s = std::max<int>(max_s, (int)pieces);
  }
  if (unit > INT32_MAX || part > INT32_MAX / kDv) return VMLA_ERR_SHAPE;
  pp->total_units = (int32_t)unit;
  pp->merge_rows = (int32_t)merge;
  pp->max_splits = max_s;
  pp->partial_rows = (int32_t)part;
  if (info) {
    info->num_units = (int32_t)unit;
    info->max_splits = max_s;
    info->partial_rows = part;
    info->merge_rows = merge;
    info->workspace_bytes = workspace_layout(qo[batch], part, kernel == VMLA_KERNEL_TC ? kv[batch] : 0).total;
  }
  return VMLA_OK;
}

int build_tc_schedule(const PlanParams& plan, int num_clusters, int unit_begin, int unit_end, TcSched* sched) {
  if (!sched || num_clusters < 1) return VMLA_ERR_SHAPE;
  if (num_clusters > kMaxClusters) num_clusters = kMaxClusters;
  if (unit_begin < 0 || unit_end > plan.total_units || unit_end < unit_begin) return VMLA_ERR_SHAPE;
  const int U = unit_end - unit_begin;
  if (U > kMaxTcUnits) return VMLA_ERR_SHAPE;
  sched->num_clusters = num_clusters;
  sched->total_units = U;
  sched->unit_base = unit_begin;
  sched->pad = 0;
  // cost of a unit: its keys plus a fixed charge for filling and draining the pipeline
  struct Item { int64_t cost; int unit; };
  std::vector<Item> items;
  items.reserve(U);
  for (int b = 0; b < plan.batch; ++b) {
    const SeqPlan& s = plan.seq[b];
    for (int piece = 0; piece < s.n_split; ++piece) {
      const int64_t lo = (int64_t)piece * s.chunk;
      const int64_t hi = std::min<int64_t>(s.n_kv, lo + s.chunk);
      for (int rb = 0; rb < s.n_rb; ++rb) {
        const int u = s.unit_start + piece * s.n_rb + rb;
        if (u >= unit_begin && u < unit_end) items.push_back({(hi - lo) + 256, u});
      }
    }
  }
  // longest first, ties by unit id (deterministic)
  std::stable_sort(items.begin(), items.end(), [](const Item& x, const Item& y) { return x.cost > y.cost; });
  std::vector<int64_t> load(num_clusters, 0);
  std::vector<std::vector<int>> lists(num_clusters);
  for (const Item& it : items) {
    int best = 0;
    for (int c = 1; c < num_clusters; ++c)
      if (load[c] < load[best]) best = c;
    load[best] += it.cost;
    lists[best].push_back(it.unit);
  }
  int pos = 0;
  for (int c = 0; c < num_clusters; ++c) {
    sched->start[c] = (uint16_t)pos;
    // within a cluster, units of the same piece next to each other keep KV reuse in L2
    std::sort(lists[c].begin(), lists[c].end());
    for (int u : lists[c]) sched->order[pos++] = (uint16_t)(u - unit_begin);
  }
  sched->start[num_clusters] = (uint16_t)pos;
  return VMLA_OK;
}

}  // namespace vmla
