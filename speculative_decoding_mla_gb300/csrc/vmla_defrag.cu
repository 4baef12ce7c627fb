// Persistent KV defragmentation.
//
// "The Build That Unlocked 3-6x Decode Speedup" names the compaction of
// scattered page_size = 1 slots into contiguous runs as the plan's next phase
// (section "The Context: A Custom Kernel for an Unsupported Architecture"), so
// that the verify kernel streams a sequence's rows as plain tile loads.  The
// per-call gather (vmla_gather.cu) does this into the workspace at every call;
// this kernel does it once into the caller's pool: the rows of sequence b go
// to slots run_base[b] .. run_base[b] + N_b - 1, and the slots after the run up
// to a multiple of 128 are zeroed, because the verify kernel's last tile of a
// run reads them (with no weight) and stale contents could hold non-finite
// bf16 values.  verify_attn_mla_runs then reads the runs with no gather.
//
// One block per 128 rows of a run (grid rows are sequences), one warp per row
// at a time as in the gather: lane l moves 16-byte granules l, l+32 and l+64
// (< 72).  A source slot outside the pool records VMLA_ERR_INDEX and
// writes a zero row; a run outside the destination records VMLA_ERR_INDEX
// (with the sequence index) and is skipped.  With first_row (the append form,
// for a decode loop), rows j < first_row[b] are already in the run and are
// left alone; a first_row[b] outside [0, N_b] records VMLA_ERR_INDEX (with the
// sequence index) and that sequence is skipped.
#include <cuda_runtime.h>

#include "vmla_device.cuh"

namespace vmla {
namespace {

constexpr int kDefragWarps = 8;
constexpr int kRowU4 = kRowBytes / 16;  // 72
constexpr int kRunAlign = 128;          // rows one tile of the tensor-core kernel covers

__device__ __forceinline__ int64_t round_run(int64_t n) { return (n + kRunAlign - 1) / kRunAlign * kRunAlign; }

__device__ __forceinline__ bool run_ok(const int32_t* kv_indptr, const int32_t* run_base, int b, int64_t slots) {
  const int64_t n = (int64_t)kv_indptr[b + 1] - kv_indptr[b];
  const int64_t base = run_base[b];
  return n >= 0 && base >= 0 && base + n <= slots;
}

__device__ __forceinline__ bool first_ok(const int32_t* kv_indptr, const int32_t* first_row, int b) {
  if (!first_row) return true;
  const int64_t n = (int64_t)kv_indptr[b + 1] - kv_indptr[b];
  return first_row[b] >= 0 && first_row[b] <= n;
}

// Grid: x = blocks of kRunAlign rows of a run (its rows, then its zeroed tail),
// y = sequence.  A block below first_row[b] or past the run returns at once, so
// an append touches only the blocks that hold new rows.  With max_new > 0 the
// x blocks start at the kRunAlign boundary below first_row[b] (the grid then
// covers max_new new rows and the tail), and a sequence with more new rows
// records VMLA_ERR_INDEX and is skipped.
__global__ void __launch_bounds__(kDefragWarps * 32)
defrag_kernel(const uint4* __restrict__ src, int64_t src_slots, const int32_t* __restrict__ kv_indptr,
              const int32_t* __restrict__ kv_indices, uint4* __restrict__ dst, int64_t dst_slots,
              const int32_t* __restrict__ run_base, const int32_t* __restrict__ first_row, int64_t max_new,
              uint32_t* status) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = blockIdx.y;
  const int64_t n = (int64_t)kv_indptr[b + 1] - kv_indptr[b];
  const bool valid = run_ok(kv_indptr, run_base, b, dst_slots) && first_ok(kv_indptr, first_row, b);
  const int64_t first = first_row && valid ? first_row[b] : 0;
  const int64_t lo = (max_new > 0 ? first / kRunAlign * kRunAlign : 0) + (int64_t)blockIdx.x * kRunAlign;
  if (!valid || (max_new > 0 && n - first > max_new)) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && n > 0) record_status(status, VMLA_ERR_INDEX, (uint32_t)b);
    return;
  }
  if (lo >= round_run(n)) return;  // past this run and its tail
  if (lo + kRunAlign <= first && lo + kRunAlign <= n) return;  // rows already in the run, no tail here
  for (int64_t r = lo + warp; r < lo + kRunAlign; r += kDefragWarps) {
    const bool zero = r >= n;
    if (!zero && r < first) continue;  // already in the run (warp-uniform)
    const int64_t row = (int64_t)run_base[b] + r;
    if (row >= dst_slots) continue;  // a tail past the pool: the tile loads read zeros there
    uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0, v2 = v0;
    if (!zero) {
      const int64_t j = (int64_t)kv_indptr[b] + r;
      const int32_t slot = kv_indices[j];
      const bool ok = slot >= 0 && (int64_t)slot < src_slots;
      if (!ok && lane == 0) record_status(status, VMLA_ERR_INDEX, (uint32_t)j);
      if (ok) {
        const uint4* s = src + (int64_t)slot * kRowU4;
        v0 = s[lane];
        v1 = s[lane + 32];
        if (lane < kRowU4 - 64) v2 = s[lane + 64];
      }
    }
    uint4* d = dst + row * kRowU4;
    d[lane] = v0;
    d[lane + 32] = v1;
    if (lane < kRowU4 - 64) d[lane + 64] = v2;
  }
}

// Runs read by verify_attn_mla_runs must lie in the pool.
__global__ void run_check_kernel(const int32_t* __restrict__ kv_indptr, const int32_t* __restrict__ run_base,
                                 int batch, int64_t slots, uint32_t* status) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < batch && !run_ok(kv_indptr, run_base, b, slots)) record_status(status, VMLA_ERR_INDEX, (uint32_t)b);
  // started beside the device planner, this grid completes only after it (the verify kernel
  // after it reads the plan); launched after its predecessor has completed, the wait returns
  grid_dependency_wait();
}

}  // namespace

int launch_defrag(const uint16_t* src_pool, int64_t src_slots, const int32_t* kv_indptr, const int32_t* kv_indices,
                  const int32_t* kv_indptr_host, int batch, int64_t total_kv, uint16_t* dst_pool, int64_t dst_slots,
                  const int32_t* run_base, bool check_only, uint32_t* status, void* stream,
                  const int32_t* first_row, int64_t max_new, bool beside_planner) {
  if (batch == 0) return VMLA_OK;
  if (check_only) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1] = {early_start_attribute()};
    cfg.gridDim = dim3((unsigned)((batch + 127) / 128), 1, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.stream = (cudaStream_t)stream;
    cfg.attrs = attr;
    cfg.numAttrs = beside_planner ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, run_check_kernel, kv_indptr, run_base, batch, dst_slots, status) == cudaSuccess
               ? VMLA_OK
               : VMLA_ERR_CUDA;
  }
  // blocks of kRunAlign rows over the longest run with its tail, one grid row per sequence
  (void)total_kv;
  int64_t longest = 0;
  for (int b = 0; b < batch; ++b) {
    const int64_t len = (int64_t)kv_indptr_host[b + 1] - kv_indptr_host[b];
    longest = len > longest ? len : longest;
  }
  // all of the longest run, or (append with a bound) the new rows from the boundary below
  // first_row plus the tail: max_new + 2 (kRunAlign - 1) rows at most.  With a bound the
  // grid depends on nothing else, so a captured launch stays valid as the runs grow.
  const bool bounded = max_new > 0;
  const int64_t span = bounded ? max_new + 2 * (kRunAlign - 1) : longest;
  const int64_t xblocks = (span + kRunAlign - 1) / kRunAlign;
  if (xblocks == 0) return VMLA_OK;
  if (xblocks > INT32_MAX || batch > 65535) return VMLA_ERR_SHAPE;
  defrag_kernel<<<dim3((unsigned)xblocks, (unsigned)batch), kDefragWarps * 32, 0, (cudaStream_t)stream>>>(
      reinterpret_cast<const uint4*>(src_pool), src_slots, kv_indptr, kv_indices,
      reinterpret_cast<uint4*>(dst_pool), dst_slots, run_base, first_row, bounded ? max_new : 0, status);
  return cudaGetLastError() == cudaSuccess ? VMLA_OK : VMLA_ERR_CUDA;
}

}  // namespace vmla
