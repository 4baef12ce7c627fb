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
#include "vmla_plan_core.h"

namespace vmla {

// Host form of the piece-size choice.  The device planner scores every
// candidate with the closed form per (run, cluster) pair; here the candidates
// are scored best bound first and the rest pruned (which cannot change the
// choice), and the runs of a scored candidate are sorted and the snake shares
// summed by residue, which gives the same integer scores in O(R log R + C):
//   load_j = sum_r cost_r (F_j(end_r) - F_j(start_r)),
//   F_j(x) = 2 floor(x / 2C) + [x mod 2C > j] + [x mod 2C > 2C - 1 - j],
// so load_j = K + S(j) + S(2C - 1 - j) with K the whole-period part and S(x)
// the sum over residues v > x of (cost at end residue v) - (cost at start residue v).
// *chosen_score: the chosen candidate's score, or -1 when the search does not run.
static int64_t plan_pick_chunk_host(const PlanShape& sh, int batch, int num_heads, const int32_t* qo,
                                    const int32_t* kv, int clusters, int64_t total_work, int64_t* chosen_score) {
  const int64_t def = plan_cand_chunk(sh, total_work, clusters, kDefaultCand);
  *chosen_score = -1;
  if (batch > kSearchMaxBatch || batch < 1 || clusters < 1) return def;
  const int R = kRunsPerSeq * batch;
  const int64_t period = 2 * (int64_t)clusters;
  int64_t nq[kSearchMaxBatch], nk[kSearchMaxBatch], rbs[kSearchMaxBatch];
  for (int b = 0; b < batch; ++b) {
    nq[b] = (int64_t)qo[b + 1] - qo[b];
    nk[b] = (int64_t)kv[b + 1] - kv[b];
    rbs[b] = plan_row_blocks(sh, nq[b], num_heads);
  }
  // pass 1: every candidate's runs, partial rows and lower bound (some cluster carries at
  // least the mean load and one carries the largest unit)
  static thread_local int64_t cost[kChunkCands][kRunsPerSeq * kSearchMaxBatch];
  static thread_local int64_t count[kChunkCands][kRunsPerSeq * kSearchMaxBatch];
  int64_t score[kChunkCands], bound[kChunkCands], part[kChunkCands];
  for (int k = 0; k < kChunkCands; ++k) {
    const int64_t ct = plan_cand_chunk(sh, total_work, clusters, k);
    int64_t units = 0, prt = 0, total = 0, largest = 0;
    for (int b = 0; b < batch; ++b) {
      int64_t c2[kRunsPerSeq], n2[kRunsPerSeq];
      prt += plan_seq_runs(sh, nq[b], nk[b], num_heads, rbs[b], ct, c2, n2);
      for (int t = 0; t < kRunsPerSeq; ++t) {
        cost[k][kRunsPerSeq * b + t] = c2[t];
        count[k][kRunsPerSeq * b + t] = n2[t];
        units += n2[t];
        total += c2[t] * n2[t];
        if (n2[t] > 0 && c2[t] > largest) largest = c2[t];
      }
    }
    const int64_t mean = (total + clusters - 1) / clusters;
    part[k] = prt;
    bound[k] = (mean > largest ? mean : largest) + plan_merge_score(prt);
    score[k] = units > kMaxTcUnits ? -1 : -2;  // -1: not a candidate (more units than one launch holds)
  }
  // pass 2: exact scores, the default first, then the others by increasing bound (ties by
  // candidate); a candidate whose bound exceeds the best exact score so far cannot be chosen
  // (nor tie), so its bound stands in for its score, and so do those of all after it.  The
  // candidate with the lowest exact score, and every one that ties it, is always scored
  // exactly, so the choice is the one a full evaluation makes.
  int order[kChunkCands];
  int n_order = 0;
  if (score[kDefaultCand] == -2) order[n_order++] = kDefaultCand;
  for (int k = 0; k < kChunkCands; ++k)
    if (k != kDefaultCand && score[k] == -2) order[n_order++] = k;
  std::sort(order + (n_order > 0 && order[0] == kDefaultCand ? 1 : 0), order + n_order,
            [&](int x, int y) { return bound[x] < bound[y] || (bound[x] == bound[y] && x < y); });
  uint64_t key[kRunsPerSeq * kSearchMaxBatch];
  std::vector<int64_t> resid(period + 1);
  int64_t best = -1;  // lowest exact score so far
  for (int i = 0; i < n_order; ++i) {
    const int k = order[i];
    if (k != kDefaultCand && best >= 0 && bound[k] > best) {
      for (int i2 = i; i2 < n_order; ++i2) score[order[i2]] = bound[order[i2]];
      break;
    }
    const int64_t* cst = cost[k];
    const int64_t* cnt = count[k];
    // runs by cost, descending (costs are below 2^32, indexes below 2^8)
    for (int r = 0; r < R; ++r) key[r] = ((uint64_t)(0xFFFFFFFFll - cst[r]) << 8) | (uint64_t)r;
    std::sort(key, key + R);
    std::fill(resid.begin(), resid.end(), 0);
    // positions as quotient and residue modulo the period, advanced run by run
    int64_t whole = 0, q_lo = 0, r_lo = 0;
    for (int j2 = 0; j2 < R; ++j2) {
      const int r = (int)(key[j2] & 0xFFu);
      if (cnt[r] == 0) continue;
      const int64_t n = cnt[r];
      int64_t q_hi = q_lo + (n >= period ? n / period : 0), r_hi = r_lo + (n >= period ? n % period : n);
      if (r_hi >= period) {
        r_hi -= period;
        ++q_hi;
      }
      whole += cst[r] * 2 * (q_hi - q_lo);
      resid[r_hi] += cst[r];
      resid[r_lo] -= cst[r];
      q_lo = q_hi;
      r_lo = r_hi;
    }
    // suffix sums: resid[x] becomes the sum over residues v > x
    int64_t acc = 0;
    for (int64_t x = period - 1; x >= 0; --x) {
      const int64_t v = resid[x];
      resid[x] = acc;
      acc += v;
    }
    int64_t worst = 0;
    for (int j = 0; j < clusters; ++j) {
      const int64_t load = whole + resid[j] + resid[period - 1 - j];
      worst = load > worst ? load : worst;
    }
    score[k] = worst + plan_merge_score(part[k]);
    if (best < 0 || score[k] < best) best = score[k];
  }
  const int k = plan_choose_cand(score);
  *chosen_score = score[k];
  return plan_cand_chunk(sh, total_work, clusters, k);
}

// The lane plan (vmla_plan_core.h) of a tensor-core call, written into pp if it
// scores lower than the uniform plan's `uniform_score` (or, forced, whenever the
// lanes fit); returns whether it did.
static bool plan_lanes_host(const PlanShape& sh, int batch, int num_heads, const int32_t* qo, const int32_t* kv,
                            int clusters, int64_t uniform_score, bool forced, PlanParams* pp) {
  if (uniform_score < 0 && !forced) return false;
  uint32_t misfit = 0;
  for (int b = 0; b < batch; ++b) {
    const int64_t nq = (int64_t)qo[b + 1] - qo[b];
    if (nq > 0) misfit |= plan_lane_misfit(plan_ceil_div(nq * num_heads, sh.rows_per_unit));
  }
  const int G = plan_lane_width(misfit);
  const int lanes = clusters / G;
  if (lanes < 1 || lanes > sh.max_splits) return false;
  int64_t W = 0;
  for (int b = 0; b < batch; ++b) {
    const int64_t nq = (int64_t)qo[b + 1] - qo[b];
    if (nq > 0) W += plan_ceil_div(nq * num_heads, sh.rows_per_unit) / G * plan_stream_span((int64_t)kv[b + 1] - kv[b]);
  }
  if (W < 1 || W > INT32_MAX) return false;
  const int64_t L = plan_lane_tiles(W, lanes);
  int64_t c0 = 0, part = 0;
  for (int b = 0; b < batch; ++b) {
    const int64_t nq = (int64_t)qo[b + 1] - qo[b], nk = (int64_t)kv[b + 1] - kv[b];
    if (nq == 0) continue;
    const int64_t ng = plan_ceil_div(nq * num_heads, sh.rows_per_unit) / G;
    int64_t pr = 0, mr = 0, ps = 0;
    plan_lane_seq_split(c0, ng, nk, L, nq * num_heads, (int64_t)G * sh.rows_per_unit, &pr, &mr, &ps);
    part += pr;
    c0 += ng * plan_stream_span(nk);
  }
  if ((!forced && !plan_prefer_lanes(plan_lane_score(L, part), uniform_score)) || part > INT32_MAX / kDv)
    return false;
  // the plan: streams in sequence order, each sequence's partial rows and merge rows after the previous ones
  int64_t stream = 0, units = 0, merge = 0;
  int max_s = 0;
  c0 = 0;
  part = 0;
  for (int b = 0; b < batch; ++b) {
    SeqPlan& s = pp->seq[b];
    const int64_t nq = (int64_t)qo[b + 1] - qo[b], nk = (int64_t)kv[b + 1] - kv[b];
    s.unit_start = (int32_t)stream;
    s.lane_cost = (int32_t)c0;
    s.part_off = (int32_t)part;
    s.merge_off = (int32_t)merge;
    s.chunk = nk > 1 ? (int32_t)nk : 1;
    s.n_split = 1;
    s.n_rb = 0;
    if (nq == 0) continue;
    s.n_rb = (int32_t)plan_ceil_div(nq * num_heads, sh.rows_per_unit);
    const int64_t ng = s.n_rb / G;
    int64_t pr = 0, mr = 0, ps = 0;
    s.n_split =
        (int32_t)plan_lane_seq_split(c0, ng, nk, L, nq * num_heads, (int64_t)G * sh.rows_per_unit, &pr, &mr, &ps);
    part += pr;
    merge += mr;
    units += ps * G;
    stream += ng;
    c0 += ng * plan_stream_span(nk);
    max_s = std::max<int>(max_s, s.n_split);
  }
  pp->total_units = (int32_t)units;
  pp->merge_rows = (int32_t)merge;
  pp->max_splits = max_s;
  pp->partial_rows = (int32_t)part;
  pp->lane_width = G;
  pp->lane_tiles = (int32_t)L;
  pp->lane_total = (int32_t)W;
  pp->lane_count = (int32_t)plan_ceil_div(W, L);
  return true;
}

WorkspaceLayout workspace_layout(int64_t total_q, int64_t partial_rows, int64_t staged_rows) {
  auto up = [](size_t x) { return (x + VMLA_WORKSPACE_ALIGN - 1) / VMLA_WORKSPACE_ALIGN * VMLA_WORKSPACE_ALIGN; };
  WorkspaceLayout w;
  w.status_off = 0;
  w.masks_off = up(16);
  w.staged_off = w.masks_off + up((size_t)total_q * 8);
  w.part_o_off = w.staged_off + up((size_t)staged_rows * kRowBytes);
  w.part_lse_off = w.part_o_off + up((size_t)partial_rows * kDv * 4);
  w.total = w.part_lse_off + up((size_t)partial_rows * 4);
  return w;
}

int build_plan(int kernel, int batch, int num_heads, const int32_t* qo, const int32_t* kv, int splits, int num_sms,
               int tc_clusters, PlanParams* pp, vmla_plan_info* info) {
  if (!qo || !kv || !pp) return VMLA_ERR_NULL;
  if (kernel != VMLA_KERNEL_TC && kernel != VMLA_KERNEL_SIMT) return VMLA_ERR_SHAPE;
  if (batch < 0 || batch > VMLA_MAX_BATCH || num_heads < 1 || num_heads > VMLA_MAX_HEADS) return VMLA_ERR_SHAPE;
  if (splits < VMLA_SPLITS_LANES || num_sms < 1) return VMLA_ERR_SHAPE;
  const bool force_lanes = splits == VMLA_SPLITS_LANES;
  if (force_lanes) splits = 0;  // the uniform plan it falls back on is the planner's own
  if (qo[0] != 0 || kv[0] != 0) return VMLA_ERR_SHAPE;
  for (int b = 0; b < batch; ++b)
    if (plan_check_seq((int64_t)qo[b + 1] - qo[b], (int64_t)kv[b + 1] - kv[b]) != VMLA_OK) return VMLA_ERR_SHAPE;
  const PlanShape sh = plan_shape(kernel);
  std::memset(pp, 0, sizeof(PlanParams));
  pp->batch = batch;
  pp->num_heads = num_heads;
  pp->rows_per_unit = sh.rows_per_unit;

  // slots: units that run at once
  const int clusters = tc_clusters > 0 ? tc_clusters : std::max(1, num_sms / 4);
  int64_t slots = kernel == VMLA_KERNEL_TC ? (int64_t)clusters * sh.units_per_sm : (int64_t)num_sms * sh.units_per_sm;
  int64_t total_work = 0;  // (row block) x (keys)
  for (int b = 0; b < batch; ++b) total_work += plan_seq_work(sh, qo[b + 1] - qo[b], kv[b + 1] - kv[b], num_heads);
  // the tensor-core kernel's piece size is chosen by scoring candidate schedules
  int64_t uniform_score = -1;
  const int64_t chunk_target =
      kernel == VMLA_KERNEL_TC && splits == 0
          ? plan_pick_chunk_host(sh, batch, num_heads, qo, kv, clusters, total_work, &uniform_score)
          : plan_chunk_target(sh, total_work, slots);

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
    int64_t prows = 0, mrows = 0;
    unit += plan_split_seq(sh, s, num_heads, splits, chunk_target, &prows, &mrows);
    part += prows;
    merge += mrows;
    if (s.n_q > 0) max_s = std::max<int>(max_s, s.n_split);
  }
  if (unit > INT32_MAX || part > INT32_MAX / kDv) return VMLA_ERR_SHAPE;
  pp->total_units = (int32_t)unit;
  pp->merge_rows = (int32_t)merge;
  pp->max_splits = max_s;
  pp->partial_rows = (int32_t)part;
  // the tensor-core kernel may take the lane plan instead (it rewrites the pieces)
  if (kernel == VMLA_KERNEL_TC && splits == 0)
    plan_lanes_host(sh, batch, num_heads, qo, kv, clusters, uniform_score, force_lanes, pp);
  if (info) {
    info->num_units = pp->total_units;
    info->max_splits = pp->max_splits;
    info->partial_rows = pp->partial_rows;
    info->merge_rows = pp->merge_rows;
    info->workspace_bytes =
        workspace_layout(qo[batch], pp->partial_rows, kernel == VMLA_KERNEL_TC ? kv[batch] : 0).total;
    info->lane_width = pp->lane_width;
    info->lane_count = pp->lane_count;
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
  // cost of a unit: its keys plus a fixed charge for the unit's start and end
  struct Item { int64_t cost; int unit; };
  std::vector<Item> items;
  items.reserve(U);
  for (int b = 0; b < plan.batch; ++b) {
    const SeqPlan& s = plan.seq[b];
    for (int piece = 0; piece < s.n_split; ++piece)
      for (int rb = 0; rb < s.n_rb; ++rb) {
        const int u = s.unit_start + piece * s.n_rb + rb;
        if (u >= unit_begin && u < unit_end) items.push_back({plan_unit_cost(s, u), u});
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
