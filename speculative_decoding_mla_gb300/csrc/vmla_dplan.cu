// Device-side planner for stream-captured calls.
//
// The pages make the verify kernel CUDA-graph capture-safe after it first
// runs ("The Build That Unlocked 3-6x Decode Speedup", section "The Broader
// Significance").  A captured graph replays its launches with the parameters
// they were captured with, so a plan built on the host from one step's lengths
// would be stale at the next.  Here the plan is computed by a kernel from the
// device indptr arrays at run time: the same split arithmetic as the host
// planner (vmla_plan_core.h, so both give identical pieces and results), and
// a cluster schedule for the tensor-core kernel (units sorted by cost, dealt
// to the clusters in a snake order, then in unit order within each cluster).
// The piece size is the host planner's choice among the same candidates,
// scored with the same integer arithmetic, one block per candidate (the last
// block to finish makes the plan), and the lane plan replaces it under the
// host planner's rule (one thread per sequence, block-wide prefix sums for the
// streams' positions).
// The areas of the workspace are sized for caller-given upper bounds on the
// query and key totals.
#include <cuda_runtime.h>

#include "vmla_device.cuh"
#include "vmla_plan_core.h"

namespace vmla {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kSortKeys = 4096;  // power of two, at least kMaxTcUnits
constexpr int kCountedSchedule = 256;  // schedules of at most this many units are placed by counting
static_assert(kSortKeys >= kMaxTcUnits, "schedule sort size");
static_assert(VMLA_MAX_BATCH <= kPlanThreads, "one thread per sequence");
static_assert(4 * kRunsPerSeq * kSearchMaxBatch <= kSortKeys, "a candidate's scratch fits the sort keys");
static_assert(kMaxClusters <= kRunsPerSeq * kSearchMaxBatch, "cluster loads fit the scratch");
static_assert(kRunsPerSeq * kSearchMaxBatch <= kPlanThreads, "one thread per run");
static_assert(kCountedSchedule <= kPlanThreads, "one thread per counted unit");
static_assert(5 * VMLA_MAX_BATCH <= kSortKeys, "the lane plan's prefix sums fit the sort keys");

// Score of candidate k (plan_pick_chunk_host's) by a whole block: the longest
// cluster load of the snake deal of its units plus the merge's charge, or -1 when
// they exceed one launch.  Runs are ranked by cost (descending, ties by run), a
// run's sort position being the units of the runs before it; each (cluster, run)
// pair adds its cost times the run's units that land on the cluster.  Scratch:
// 4 x kRunsPerSeq x kSearchMaxBatch words of shared memory.
__device__ int64_t block_candidate_score(const PlanShape& sh, const int32_t* qo, const int32_t* kv, int batch,
                                         int num_heads, int clusters, int64_t total_work, int k, int64_t* scratch) {
  __shared__ unsigned long long s_units, s_part, s_worst;
  constexpr int kRuns = kRunsPerSeq * kSearchMaxBatch;
  int64_t* cost = scratch;
  int64_t* cnt = scratch + kRuns;
  int64_t* pos = scratch + 2 * kRuns;
  int64_t* load = scratch + 3 * kRuns;  // kMaxClusters <= kRuns entries
  const int tid = threadIdx.x;
  const int R = kRunsPerSeq * batch;
  const int64_t ct = plan_cand_chunk(sh, total_work, clusters, k);
  if (tid == 0) {
    s_units = 0;
    s_part = 0;
    s_worst = 0;
  }
  for (int j = tid; j < clusters; j += blockDim.x) load[j] = 0;
  __syncthreads();
  if (tid < batch) {
    int64_t c2[kRunsPerSeq], n2[kRunsPerSeq];
    const int64_t nq = (int64_t)qo[tid + 1] - qo[tid];
    const int64_t prt = plan_seq_runs(sh, nq, (int64_t)kv[tid + 1] - kv[tid], num_heads,
                                      plan_row_blocks(sh, nq, num_heads), ct, c2, n2);
    int64_t units = 0;
    for (int t = 0; t < kRunsPerSeq; ++t) {
      cost[kRunsPerSeq * tid + t] = c2[t];
      cnt[kRunsPerSeq * tid + t] = n2[t];
      units += n2[t];
    }
    atomicAdd(&s_units, (unsigned long long)units);
    atomicAdd(&s_part, (unsigned long long)prt);
  }
  __syncthreads();
  if (s_units > (unsigned long long)kMaxTcUnits) return -1;  // the same value in every thread
  if (tid < R) {
    const int64_t cr = cost[tid];
    int64_t p = 0;
    for (int r2 = 0; r2 < R; ++r2)
      if (plan_run_before(cost[r2], r2, cr, tid)) p += cnt[r2];
    pos[tid] = p;
  }
  __syncthreads();
  for (int q = tid; q < clusters * R; q += blockDim.x) {
    const int j = q / R, r = q - j * R;
    const int64_t n = cnt[r];
    if (n == 0) continue;
    const int64_t add = cost[r] * (plan_snake_share(pos[r] + n, j, clusters) - plan_snake_share(pos[r], j, clusters));
    if (add != 0) atomicAdd(reinterpret_cast<unsigned long long*>(&load[j]), (unsigned long long)add);
  }
  __syncthreads();
  if (tid < clusters) atomicMax(&s_worst, (unsigned long long)load[tid]);
  __syncthreads();
  return (int64_t)s_worst + plan_merge_score((int64_t)s_part);
}

// Ascending bitonic sort of the first n keys in shared memory (n a power of
// two, at most kSortKeys; whole block).
__device__ void block_sort(uint64_t* k, int n) {
  for (int size = 2; size <= n; size <<= 1)
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n / 2; i += blockDim.x) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool up = (lo & size) == 0;
        const uint64_t a = k[lo], b = k[hi];
        if ((a > b) == up) {
          k[lo] = b;
          k[hi] = a;
        }
      }
      __syncthreads();
    }
}

// Inclusive prefix sum of v[0, n) in place (whole block, n <= blockDim.x).
__device__ void block_scan(int64_t* v, int n) {
  for (int off = 1; off < n; off <<= 1) {
    int64_t t = 0;
    const int i = threadIdx.x;
    if (i < n && i >= off) t = v[i - off];
    __syncthreads();
    if (i < n && i >= off) v[i] += t;
    __syncthreads();
  }
}

// Lengths the plan cannot take: VMLA_ERR_SHAPE replaces whatever the gather, which runs
// beside the planner on the lengths it was given, recorded about their slots.
__device__ __forceinline__ void record_shape_error(uint32_t* status, uint32_t info) {
  atomicExch(status, (uint32_t)VMLA_ERR_SHAPE);
  status[1] = info;
}

__global__ void __launch_bounds__(kPlanThreads)
device_plan_kernel(const int32_t* __restrict__ qo, const int32_t* __restrict__ kv, int batch, int num_heads,
                   int splits, int clusters, int64_t max_total_q, int64_t max_total_kv, int64_t part_cap,
                   PlanParams* __restrict__ pp, TcSched* __restrict__ sched, uint32_t* status) {
  // the gather may start at once beside this grid (it reads no plan, and it waits for
  // this grid before it completes)
  grid_dependents_launch();
  // status[4]: blocks done with their candidate (zeroed before the launch, and again by
  // the last block); status[8..]: the candidates' scores (int64)
  unsigned int* done = status + 4;
  int64_t* scores = reinterpret_cast<int64_t*>(status + 8);
  __shared__ int64_t s_units[VMLA_MAX_BATCH], s_part[VMLA_MAX_BATCH], s_merge[VMLA_MAX_BATCH];
  __shared__ uint64_t keys[kSortKeys];
  __shared__ unsigned long long s_work;
  __shared__ int s_bad, s_maxs, s_cand, s_lanes, s_last;
  __shared__ unsigned int s_misfit;
  __shared__ int64_t s_score[kChunkCands];
  __shared__ int64_t s_chunk;
  const int tid = threadIdx.x;
  const PlanShape sh = plan_shape(VMLA_KERNEL_TC);
  if (tid == 0) {
    s_work = 0;
    s_bad = 0;
    s_maxs = 0;
    s_misfit = 0;
  }
  __syncthreads();
  // lengths: each thread checks one sequence and adds its work
  int64_t nq = 0, nk = 0;
  if (tid < batch) {
    nq = (int64_t)qo[tid + 1] - qo[tid];
    nk = (int64_t)kv[tid + 1] - kv[tid];
    if (plan_check_seq(nq, nk) != VMLA_OK)
      atomicOr(&s_bad, 1);
    else
      atomicAdd(&s_work, (unsigned long long)plan_seq_work(sh, nq, nk, num_heads));
  }
  if (tid == 0 && (qo[0] != 0 || kv[0] != 0 || (int64_t)qo[batch] > max_total_q || (int64_t)kv[batch] > max_total_kv))
    atomicOr(&s_bad, 2);
  __syncthreads();
  const bool lengths_ok = s_bad == 0;
  const int64_t total_work = (int64_t)s_work;
  const bool force_lanes = splits == VMLA_SPLITS_LANES;
  if (force_lanes) splits = 0;  // the uniform plan it falls back on is the planner's own
  const bool search = lengths_ok && splits == 0 && batch >= 1 && batch <= kSearchMaxBatch;
  // every block scores one candidate (the launch has kChunkCands blocks when a search
  // can run); the last block to finish reads all the scores and makes the plan
  if (search && blockIdx.x < kChunkCands) {
    const int64_t sc = block_candidate_score(sh, qo, kv, batch, num_heads, clusters, total_work, (int)blockIdx.x,
                                             reinterpret_cast<int64_t*>(keys));
    if (tid == 0) scores[blockIdx.x] = sc;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(done, 1u) == gridDim.x - 1 ? 1 : 0;
  __syncthreads();
  if (!s_last) return;
  if (tid == 0) *done = 0;  // ready for the next call (or graph replay)
  if (tid < kChunkCands) s_score[tid] = search && tid < (int)gridDim.x ? __ldcg(&scores[tid]) : -1;
  __syncthreads();
  if (tid == 0) {
    s_cand = search ? plan_choose_cand(s_score) : kDefaultCand;
    s_chunk = plan_cand_chunk(sh, total_work, clusters, s_cand);
  }
  __syncthreads();
  const int64_t chunk_target = s_chunk;

  // ---- the lane plan, weighed against the chosen uniform plan (plan_lanes_host's rule)
  const int64_t R = nq * num_heads;
  const int64_t n_rb = tid < batch && nq > 0 ? plan_ceil_div(R, sh.rows_per_unit) : 0;
  if (n_rb > 0) atomicOr(&s_misfit, plan_lane_misfit(n_rb));
  // prefix sums over the sequences in the sort keys' space (free until the schedule)
  int64_t* l_cost = reinterpret_cast<int64_t*>(keys);
  int64_t* l_stream = l_cost + VMLA_MAX_BATCH;
  int64_t* l_part = l_stream + VMLA_MAX_BATCH;
  int64_t* l_merge = l_part + VMLA_MAX_BATCH;
  int64_t* l_units = l_merge + VMLA_MAX_BATCH;
  __syncthreads();
  const int G = plan_lane_width(s_misfit);
  const int lanes = clusters / G;
  const int64_t ng = n_rb / G;
  const int64_t span = plan_stream_span(nk);
  if (tid < batch) {
    l_cost[tid] = ng * span;
    l_stream[tid] = ng;
  }
  __syncthreads();
  block_scan(l_cost, batch);
  block_scan(l_stream, batch);
  const int64_t W = batch > 0 ? l_cost[batch - 1] : 0;
  const int64_t Lt = plan_lane_tiles(W, lanes);
  const bool lane_fit =
      (search || (force_lanes && lengths_ok)) && lanes >= 1 && lanes <= sh.max_splits && W >= 1 && W <= INT32_MAX;
  int64_t lpr = 0, lmr = 0, lps = 0, lsplit = 1;
  if (lane_fit && n_rb > 0)
    lsplit = plan_lane_seq_split(l_cost[tid] - ng * span, ng, nk, Lt, R, (int64_t)G * sh.rows_per_unit, &lpr, &lmr,
                                 &lps);
  if (tid < batch) {
    l_part[tid] = lpr;
    l_merge[tid] = lmr;
    l_units[tid] = lps * G;
  }
  __syncthreads();
  block_scan(l_part, batch);
  block_scan(l_merge, batch);
  block_scan(l_units, batch);
  if (tid == 0) {
    const int64_t lpart = batch > 0 ? l_part[batch - 1] : 0;
    s_lanes = lane_fit && lpart <= INT32_MAX / kDv &&
              (force_lanes || plan_prefer_lanes(plan_lane_score(Lt, lpart), s_score[s_cand]));
  }
  __syncthreads();
  if (s_lanes) {
    if (tid < batch) {
      SeqPlan lp = {};
      lp.kv_off = kv[tid];
      lp.n_kv = (int32_t)nk;
      lp.q_off = qo[tid];
      lp.n_q = (int32_t)nq;
      lp.unit_start = (int32_t)(l_stream[tid] - ng);
      lp.lane_cost = (int32_t)(l_cost[tid] - ng * span);
      lp.part_off = (int32_t)(l_part[tid] - lpr);
      lp.merge_off = (int32_t)(l_merge[tid] - lmr);
      lp.chunk = nk > 1 ? (int32_t)nk : 1;
      lp.n_split = (int32_t)lsplit;
      lp.n_rb = (int32_t)n_rb;
      pp->seq[tid] = lp;
      if (n_rb > 0) atomicMax(&s_maxs, (int)lsplit);
    }
    __syncthreads();
    if (tid == 0) {
      const int64_t part = batch > 0 ? l_part[batch - 1] : 0;
      const bool ok = part <= part_cap;
      const int lane_count = (int)plan_ceil_div(W, Lt);
      pp->batch = batch;
      pp->num_heads = num_heads;
      pp->rows_per_unit = sh.rows_per_unit;
      pp->total_units = ok ? (int32_t)l_units[batch - 1] : 0;
      pp->merge_rows = ok ? (int32_t)l_merge[batch - 1] : 0;
      pp->max_splits = ok ? s_maxs : 0;
      pp->partial_rows = ok ? (int32_t)part : 0;
      pp->lane_width = G;
      pp->lane_tiles = (int32_t)Lt;
      pp->lane_total = (int32_t)W;
      pp->lane_count = ok ? lane_count : 0;
      pp->pad = 0;
      status[2] = ok ? (uint32_t)kv[batch] : 0u;
      status[3] = ok ? (uint32_t)qo[batch] : 0u;
      if (!ok) record_shape_error(status, 2u);
      sched->num_clusters = ok ? lane_count * G : 0;
      sched->total_units = ok ? (int32_t)l_units[batch - 1] : 0;
      sched->unit_base = 0;
      sched->pad = 0;
    }
    return;
  }
  __syncthreads();
  SeqPlan sp = {};
  int64_t u = 0, pr = 0, mr = 0;
  if (tid < batch) {
    sp.kv_off = kv[tid];
    sp.n_kv = (int32_t)nk;
    sp.q_off = qo[tid];
    sp.n_q = (int32_t)nq;
    if (lengths_ok) u = plan_split_seq(sh, sp, num_heads, splits, chunk_target, &pr, &mr);
    s_units[tid] = u;
    s_part[tid] = pr;
    s_merge[tid] = mr;
    if (lengths_ok && nq > 0) atomicMax(&s_maxs, sp.n_split);
  }
  __syncthreads();
  block_scan(s_units, batch);
  block_scan(s_part, batch);
  block_scan(s_merge, batch);
  const int64_t units = batch > 0 ? s_units[batch - 1] : 0;
  const int64_t part = batch > 0 ? s_part[batch - 1] : 0;
  const int64_t merge = batch > 0 ? s_merge[batch - 1] : 0;
  const bool ok = lengths_ok && units <= kMaxTcUnits && part <= part_cap;
  if (tid < batch) {
    sp.unit_start = (int32_t)(s_units[tid] - u);
    sp.part_off = (int32_t)(s_part[tid] - pr);
    sp.merge_off = (int32_t)(s_merge[tid] - mr);
    pp->seq[tid] = sp;
  }
  if (tid == 0) {
    pp->batch = batch;
    pp->num_heads = num_heads;
    pp->rows_per_unit = sh.rows_per_unit;
    pp->total_units = ok ? (int32_t)units : 0;
    pp->merge_rows = ok ? (int32_t)merge : 0;
    pp->max_splits = ok ? s_maxs : 0;
    pp->partial_rows = ok ? (int32_t)part : 0;
    pp->lane_width = 0;
    pp->lane_tiles = 0;
    pp->lane_total = 0;
    pp->lane_count = 0;
    pp->pad = 0;
    status[2] = ok ? (uint32_t)kv[batch] : 0u;  // key rows of the plan (diagnostic)
    status[3] = ok ? (uint32_t)qo[batch] : 0u;  // draft rows the mask kernel expands
    if (!ok) record_shape_error(status, lengths_ok ? 2u : (uint32_t)s_bad);
  }
  __syncthreads();
  // schedule: units by decreasing cost (ties by unit), dealt to the clusters
  // in a snake order, then in unit order within each cluster
  const int U = ok ? (int)units : 0;
  const int C = clusters;
  if (U <= kCountedSchedule) {
    // few units: each thread finds its unit's place by counting the keys before it (the
    // keys are distinct), which gives the sorts' order without their barriers
    uint64_t key = ~0ull;
    if (tid < U) {
      const int64_t cost = plan_unit_cost(pp->seq[seq_of_unit(*pp, tid)], tid);
      key = ((uint64_t)(0x7FFFFFFFll - cost) << 32) | (uint32_t)tid;
      keys[tid] = key;
    }
    __syncthreads();
    uint64_t key2 = ~0ull;
    if (tid < U) {
      int p = 0;
      for (int j = 0; j < U; ++j) p += keys[j] < key ? 1 : 0;
      const int round = p / C, j = p - round * C;
      const int c = (round & 1) ? C - 1 - j : j;
      key2 = ((uint64_t)c << 32) | (uint32_t)tid;
    }
    __syncthreads();
    if (tid < U) keys[tid] = key2;
    __syncthreads();
    if (tid < U) {
      int p = 0;
      for (int j = 0; j < U; ++j) p += keys[j] < key2 ? 1 : 0;
      sched->order[p] = (uint16_t)tid;
    }
    for (int c = tid; c <= C; c += blockDim.x) {
      int n = 0;  // units dealt to clusters before c
      for (int j = 0; j < U; ++j) n += (int)(keys[j] >> 32) < c ? 1 : 0;
      sched->start[c] = (uint16_t)n;
    }
    if (tid == 0) {
      sched->num_clusters = ok ? C : 0;
      sched->total_units = U;
      sched->unit_base = 0;
      sched->pad = 0;
    }
    return;
  }
  int n_sort = 2;  // sort only as many keys as there are units (rounded up to a power of two)
  while (n_sort < U) n_sort <<= 1;
  for (int k = tid; k < n_sort; k += blockDim.x) {
    uint64_t key = ~0ull;
    if (k < U) {
      const int64_t cost = plan_unit_cost(pp->seq[seq_of_unit(*pp, k)], k);
      key = ((uint64_t)(0x7FFFFFFFll - cost) << 32) | (uint32_t)k;
    }
    keys[k] = key;
  }
  __syncthreads();
  block_sort(keys, n_sort);
  for (int p = tid; p < U; p += blockDim.x) {
    const int round = p / C, j = p - round * C;
    const int c = (round & 1) ? C - 1 - j : j;
    keys[p] = ((uint64_t)c << 32) | (keys[p] & 0xFFFFFFFFull);
  }
  __syncthreads();
  block_sort(keys, n_sort);
  for (int p = tid; p < U; p += blockDim.x) sched->order[p] = (uint16_t)(keys[p] & 0xFFFFu);
  for (int c = tid; c <= C; c += blockDim.x) {
    int lo = 0, hi = U;  // first position whose cluster is >= c
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if ((int)(keys[mid] >> 32) < c) lo = mid + 1; else hi = mid;
    }
    sched->start[c] = (uint16_t)lo;
  }
  if (tid == 0) {
    sched->num_clusters = ok ? C : 0;
    sched->total_units = U;
    sched->unit_base = 0;
    sched->pad = 0;
  }
}

}  // namespace

DplanLayout dplan_layout(int batch, int num_heads, int64_t max_total_q, int64_t max_total_kv, int splits,
                         int clusters, bool staged) {
  auto up = [](size_t x) { return (x + VMLA_WORKSPACE_ALIGN - 1) / VMLA_WORKSPACE_ALIGN * VMLA_WORKSPACE_ALIGN; };
  const PlanShape sh = plan_shape(VMLA_KERNEL_TC);
  // units are at most clusters x m / 16 + (row blocks) with the planner's own
  // piece count (the largest candidate m; each sequence's pieces exceed its
  // share by less than one), or splits x (row blocks) when the count is
  // forced; 256 partial rows each.  A lane plan's partial rows are at most
  // 256 (clusters + 2 row blocks): a stream of T tiles has at most
  // (T - 1) / L + 2 pieces, and the streams' tiles times their row blocks sum
  // to at most G W <= clusters L.
  const int64_t row_blocks = plan_ceil_div(max_total_q * num_heads, sh.rows_per_unit) + batch;
  const int64_t units = splits > 0 ? (int64_t)splits * row_blocks
                                   : plan_ceil_div((int64_t)clusters * plan_cand_m(kChunkCands - 1), 16) +
                                         2 * row_blocks;
  int64_t cap = units * sh.rows_per_unit;
  const int64_t all = max_total_q * num_heads * sh.max_splits;
  if (cap > all) cap = all;
  DplanLayout L;
  L.status_off = 0;
  L.plan_off = up(32 + sizeof(int64_t) * kChunkCands);  // status words, the block counter, candidate scores
  L.sched_off = L.plan_off + up(sizeof(PlanParams));
  L.masks_off = L.sched_off + up(sizeof(TcSched));
  L.part_o_off = L.masks_off + up((size_t)max_total_q * 8);
  L.part_lse_off = L.part_o_off + up((size_t)cap * kDv * 4);
  L.staged_off = L.part_lse_off + up((size_t)cap * 4);
  L.total = L.staged_off + (staged ? up((size_t)max_total_kv * kRowBytes) : 0);
  L.part_cap = cap;
  return L;
}

int launch_device_plan(const int32_t* qo_indptr, const int32_t* kv_indptr, int batch, int num_heads, int splits,
                       int clusters, int64_t max_total_q, int64_t max_total_kv, int64_t part_cap,
                       PlanParams* plan, TcSched* sched, uint32_t* status, void* stream) {
  if (batch < 0 || batch > VMLA_MAX_BATCH || clusters < 1 || clusters > kMaxClusters) return VMLA_ERR_SHAPE;
  // one block per piece-size candidate when the candidate search can run (its lengths
  // are checked on the device), else one block
  const bool search = (splits == 0 || splits == VMLA_SPLITS_LANES) && batch >= 1 && batch <= kSearchMaxBatch;
  device_plan_kernel<<<search ? kChunkCands : 1, kPlanThreads, 0, (cudaStream_t)stream>>>(
      qo_indptr, kv_indptr, batch, num_heads, splits, clusters, max_total_q, max_total_kv, part_cap, plan, sched,
      status);
  return cudaGetLastError() == cudaSuccess ? VMLA_OK : VMLA_ERR_CUDA;
}

}  // namespace vmla
