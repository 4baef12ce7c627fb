// Split merge and draft-tree mask expansion.
//
// Merge: each split piece s of a query row left a normalised partial output
// o_s and its log-sum-exp (in a lane plan only the rows of streams cut into
// several pieces are merge rows: the others have their results already); the
// row's result is
//   lse = log sum_s exp(lse_s),  out = sum_s exp(lse_s - lse) * o_s,
// the combination of partial softmaxes that the NSPLIT split-KV of "The Build
// Script Edit", section "Context: The Long Road to a Custom sm_120 Kernel",
// implies.  A row takes one, two or four warps (each a share of its 512
// columns), chosen per launch so that every row's warps are resident at once
// without adding load rounds; each lane keeps twelve 16-byte loads in flight,
// the first batch issued together with the lse loads.  Every column sums its
// pieces in piece order whatever the split, so the result does not depend on
// it.  Pieces with lse = -inf carry no weight (their partial rows, which may
// hold anything, are read but never used).
//
// Tree masks: the q x q visibility matrix of "The Build That Bridged Design
// and Deployment", section "What This Build Achieves: The paged+bf16 Kernel",
// for a draft tree is each node's ancestor set plus itself; one thread per
// draft query walks its parent chain.
#include <cuda_runtime.h>

#include "vmla_device.cuh"
#include "vmla_plan_core.h"

namespace vmla {
namespace {

constexpr int kMergeWarps = 4;      // warps per block
constexpr int kMergeInFlight = 12;  // 16-byte loads a lane keeps in flight

// Warps per merge row: the count (4, 2 or 1) with the fewest rounds of the row's loads
// times waves of resident warps (64 per SM); ties go to more warps per row.
__host__ __device__ inline int merge_warps_per_row(int64_t rows, int max_pieces, int sms) {
  const int64_t resident = (int64_t)(sms > 0 ? sms : 1) * 64;
  int best = 4;
  int64_t best_cost = -1;
  for (int wpr = 4; wpr >= 1; wpr >>= 1) {
    const int64_t batch = kMergeInFlight / (4 / wpr);
    const int64_t rounds = (max_pieces + batch - 1) / batch;
    const int64_t waves = (rows * wpr + resident - 1) / resident;
    const int64_t cost = (rounds > 0 ? rounds : 1) * waves;
    if (best_cost < 0 || cost < best_cost) {
      best = wpr;
      best_cost = cost;
    }
  }
  return best;
}

// Sequence, row and piece count of merge row mrow (< plan.merge_rows); returns the
// sequence, with *S = 0 when the row is not a merge row of this plan.
__device__ __forceinline__ int merge_locate(const PlanParams& plan, int mrow, int* r_out, int* S_out) {
  // sequence owning merge row mrow: last b with merge_off <= mrow
  int lo = 0, hi = plan.batch;
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (plan.seq[mid].merge_off <= mrow) lo = mid; else hi = mid;
  }
  const SeqPlan& sp = plan.seq[lo];
  const int R = sp.n_q * plan.num_heads;
  int r = mrow - sp.merge_off;
  int S = sp.n_split;
  if (plan.lane_width > 0) {
    // lane plan: the sequence's merge rows are the rows of its streams cut into more than
    // one piece, stream by stream (a stream in one lane was written by the verify kernel)
    const int64_t T = plan_seq_tiles(sp.n_kv), per = (int64_t)plan.lane_width * plan.rows_per_unit;
    const int ng = sp.n_rb / plan.lane_width;
    int m = r;
    S = 0;
    for (int g = 0; g < ng; ++g) {
      const int p = (int)plan_stream_pieces(sp.lane_cost + g * (T + kLaneStreamTiles), T, plan.lane_tiles);
      if (p < 2) continue;
      const int rows = (int)plan_stream_rows(g, per, R);
      if (m < rows) {
        r = (int)(g * per) + m;
        S = p;
        break;
      }
      m -= rows;
    }
  }
  *r_out = r;
  *S_out = S;
  return lo;
}

// Part `part` of merge row mrow, merged by one warp: with WPR warps per row, the
// lane takes float4 columns (part F + f) 32 + lane of the row's 128, f < F = 4 / WPR.
template <int WPR>
__device__ __forceinline__ void merge_row(const PlanParams& plan, int mrow, int part, const float* __restrict__ part_o,
                                          const float* __restrict__ part_lse, int lse_is_log2,
                                          uint16_t* __restrict__ out, float* __restrict__ lse) {
  constexpr int F = 4 / WPR;
  constexpr int kBatch = kMergeInFlight / F;  // pieces loaded together
  const int lane = threadIdx.x & 31;
  int r = 0, S = 0;
  const SeqPlan& sp = plan.seq[merge_locate(plan, mrow, &r, &S)];
  if (S == 0) return;  // past the split streams' rows (not reached for a consistent plan)
  const int H = plan.num_heads;
  const int R = sp.n_q * H;
  const float to2 = lse_is_log2 ? 1.f : 1.4426950408889634f;
  const float4* src0 =
      reinterpret_cast<const float4*>(part_o + ((int64_t)sp.part_off + r) * kDv) + part * F * 32 + lane;
  const int64_t piece_stride = (int64_t)R * (kDv / 4);  // float4s between pieces of one row
  // the first batch of partial rows is in flight while the weights are worked out
  float4 v[kBatch][F];
#pragma unroll
  for (int b = 0; b < kBatch; ++b)
#pragma unroll
    for (int f = 0; f < F; ++f)
      v[b][f] = b < S ? __ldg(src0 + b * piece_stride + f * 32) : make_float4(0.f, 0.f, 0.f, 0.f);
  // lse of pieces lane and lane + 32 (S <= 64)
  float l0 = -INFINITY, l1 = -INFINITY;
  if (lane < S) l0 = part_lse[(int64_t)sp.part_off + (int64_t)lane * R + r] * to2;
  if (lane + 32 < S) l1 = part_lse[(int64_t)sp.part_off + (int64_t)(lane + 32) * R + r] * to2;
  const float M = warp_max(fmaxf(l0, l1));
  const int64_t orow = (int64_t)sp.q_off * H + r;
  uint2* dst = reinterpret_cast<uint2*>(out + orow * kDv) + part * F * 32 + lane;
  if (M == -INFINITY) {
#pragma unroll
    for (int f = 0; f < F; ++f) dst[f * 32] = make_uint2(0u, 0u);
    if (part == 0 && lane == 0) lse[orow] = -INFINITY;
    return;
  }
  const float w0 = exp2f(l0 - M), w1 = exp2f(l1 - M);
  const float W = warp_sum(w0 + w1);
  const float invW = 1.f / W;
  float4 acc[F];
#pragma unroll
  for (int f = 0; f < F; ++f) acc[f] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < S; s0 += kBatch) {
    if (s0 > 0) {
#pragma unroll
      for (int b = 0; b < kBatch; ++b)
#pragma unroll
        for (int f = 0; f < F; ++f)
          v[b][f] = s0 + b < S ? __ldg(src0 + (s0 + b) * piece_stride + f * 32) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int s = s0 + b;
      // every lane takes part in the shuffle; a piece without weight is skipped by a
      // select, so whatever its partial row holds never reaches the sum
      const float w = __shfl_sync(0xffffffffu, s < 32 ? w0 : w1, s & 31);
      if (s < S && w != 0.f) {
#pragma unroll
        for (int f = 0; f < F; ++f) {
          acc[f].x = fmaf(w, v[b][f].x, acc[f].x);
          acc[f].y = fmaf(w, v[b][f].y, acc[f].y);
          acc[f].z = fmaf(w, v[b][f].z, acc[f].z);
          acc[f].w = fmaf(w, v[b][f].w, acc[f].w);
        }
      }
    }
  }
#pragma unroll
  for (int f = 0; f < F; ++f)
    dst[f * 32] = make_uint2(pack_bf16x2(acc[f].x * invW, acc[f].y * invW), pack_bf16x2(acc[f].z * invW, acc[f].w * invW));
  if (part == 0 && lane == 0) lse[orow] = (M + log2f(W)) * 0.6931471805599453f;
}

// Each block merges kMergeWarps / WPR rows at a time: rows blockIdx.x (rows per block) + i,
// then a grid's worth further, and so on.
template <int WPR>
__device__ __forceinline__ void merge_body(const PlanParams& plan, const float* __restrict__ part_o,
                                           const float* __restrict__ part_lse, int lse_is_log2,
                                           uint16_t* __restrict__ out, float* __restrict__ lse) {
  constexpr int kRowsPerBlock = kMergeWarps / WPR;
  const int w = threadIdx.x >> 5;
  const int rows = plan.merge_rows;
  for (int mrow = blockIdx.x * kRowsPerBlock + w / WPR; mrow < rows; mrow += gridDim.x * kRowsPerBlock)
    merge_row<WPR>(plan, mrow, w % WPR, part_o, part_lse, lse_is_log2, out, lse);
}

template <int WPR>
__global__ void __launch_bounds__(kMergeWarps * 32)
merge_kernel(const __grid_constant__ PlanParams plan, const float* __restrict__ part_o,
             const float* __restrict__ part_lse, int lse_is_log2, uint16_t* __restrict__ out,
             float* __restrict__ lse) {
  // launched to start under the verify kernel's tail: its partials first
  grid_dependency_wait();
  merge_body<WPR>(plan, part_o, part_lse, lse_is_log2, out, lse);
}

// The plan in the workspace (device-planned calls), read past the wait; the grid is one
// wave of resident warps (`sms` SMs' worth), and the row split follows the same rule as
// the host-planned launch.
__global__ void __launch_bounds__(kMergeWarps * 32)
merge_kernel_dplan(const PlanParams* __restrict__ plan, int sms, const float* __restrict__ part_o,
                   const float* __restrict__ part_lse, uint16_t* __restrict__ out, float* __restrict__ lse) {
  grid_dependency_wait();
  const int wpr = merge_warps_per_row(plan->merge_rows, plan->max_splits, sms);
  if (wpr == 4) merge_body<4>(*plan, part_o, part_lse, 1, out, lse);
  else if (wpr == 2) merge_body<2>(*plan, part_o, part_lse, 1, out, lse);
  else merge_body<1>(*plan, part_o, part_lse, 1, out, lse);
}

__global__ void tree_mask_kernel(const int32_t* __restrict__ parent, const int32_t* __restrict__ qo_indptr,
                                 int batch, int total_q, const uint32_t* __restrict__ rows_dev,
                                 uint64_t* __restrict__ mask_out, uint32_t* status) {
  // device-planned calls start it early behind the gather: the planner's count first
  // (a launch after its predecessor has completed passes the wait at once)
  grid_dependents_launch();
  grid_dependency_wait();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (rows_dev) {  // device-planned call: the planner's count of draft rows (0 when the lengths are bad)
    const int r = (int)*rows_dev;
    total_q = r < total_q ? r : total_q;
  }
  if (t >= total_q) return;
  int lo = 0, hi = batch;
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (qo_indptr[mid] <= t) lo = mid; else hi = mid;
  }
  const int q0 = qo_indptr[lo];
  const int n = qo_indptr[lo + 1] - q0;
  const int i = t - q0;
  uint64_t bits = 0;
  int k = i;
  bool bad = n > VMLA_MAX_DRAFT;
  for (int steps = 0; k >= 0 && !bad; ++steps) {
    if (k >= n || steps > VMLA_MAX_DRAFT) { bad = true; break; }
    bits |= 1ull << k;
    const int p = parent[q0 + k];
    if (p >= k || p < -1) { bad = true; break; }
    k = p;
  }
  if (bad) {
    bits = 0;
    record_status(status, VMLA_ERR_PARENT, (uint32_t)t);
  }
  mask_out[t] = bits;
}

}  // namespace

int launch_merge(const PlanParams& plan, const float* part_o, const float* part_lse, int lse_is_log2,
                 uint16_t* out, float* lse, void* stream) {
  if (plan.merge_rows == 0) return VMLA_OK;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess)
    return VMLA_ERR_CUDA;
  const int wpr = merge_warps_per_row(plan.merge_rows, plan.max_splits, sms);
  const int rows_per_block = kMergeWarps / wpr;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1] = {early_start_attribute()};
  cfg.gridDim = dim3((unsigned)((plan.merge_rows + rows_per_block - 1) / rows_per_block), 1, 1);
  cfg.blockDim = dim3(kMergeWarps * 32, 1, 1);
  cfg.stream = (cudaStream_t)stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (wpr == 4) e = cudaLaunchKernelEx(&cfg, merge_kernel<4>, plan, part_o, part_lse, lse_is_log2, out, lse);
  else if (wpr == 2) e = cudaLaunchKernelEx(&cfg, merge_kernel<2>, plan, part_o, part_lse, lse_is_log2, out, lse);
  else e = cudaLaunchKernelEx(&cfg, merge_kernel<1>, plan, part_o, part_lse, lse_is_log2, out, lse);
  return e == cudaSuccess ? VMLA_OK : VMLA_ERR_CUDA;
}

int launch_tree_mask(const int32_t* parent, const int32_t* qo_indptr, int batch, int total_q, uint64_t* mask_out,
                     uint32_t* status, void* stream) {
  if (total_q == 0) return VMLA_OK;
  tree_mask_kernel<<<(total_q + 127) / 128, 128, 0, (cudaStream_t)stream>>>(parent, qo_indptr, batch, total_q,
                                                                             nullptr, mask_out, status);
  return cudaGetLastError() == cudaSuccess ? VMLA_OK : VMLA_ERR_CUDA;
}

int launch_merge_dplan(const PlanParams* plan, int64_t max_rows, const float* part_o, const float* part_lse,
                       uint16_t* out, float* lse, void* stream) {
  if (max_rows <= 0) return VMLA_OK;
  if (max_rows > INT32_MAX) return VMLA_ERR_SHAPE;
  // the merge rows are known only on the device: a grid that fills the GPU once (16
  // blocks of four warps per SM), each block taking every grid-th row, instead of a
  // block per row of the bound (most of which would find nothing to do)
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess)
    return VMLA_ERR_CUDA;
  const int64_t fill = (int64_t)sms * 16;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1] = {early_start_attribute()};
  cfg.gridDim = dim3((unsigned)(max_rows < fill ? max_rows : fill), 1, 1);
  cfg.blockDim = dim3(kMergeWarps * 32, 1, 1);
  cfg.stream = (cudaStream_t)stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, merge_kernel_dplan, plan, sms, part_o, part_lse, out, lse) != cudaSuccess)
    return VMLA_ERR_CUDA;
  return VMLA_OK;
}

int launch_tree_mask_dplan(const int32_t* parent, const int32_t* qo_indptr, int batch, int64_t max_total_q,
                           const uint32_t* rows_dev, uint64_t* mask_out, uint32_t* status, void* stream) {
  if (max_total_q <= 0) return VMLA_OK;
  if (max_total_q > INT32_MAX) return VMLA_ERR_SHAPE;
  const int total_q = (int)max_total_q;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1] = {early_start_attribute()};
  cfg.gridDim = dim3((unsigned)((total_q + 127) / 128), 1, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.stream = (cudaStream_t)stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, tree_mask_kernel, parent, qo_indptr, batch, total_q, rows_dev, mask_out, status) !=
      cudaSuccess)
    return VMLA_ERR_CUDA;
  return VMLA_OK;
}

}  // namespace vmla
