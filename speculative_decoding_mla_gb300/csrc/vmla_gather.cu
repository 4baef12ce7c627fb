// KV gather ("defragmentation"): copies every sequence's KV rows, read through
// kv_indices at page_size = 1, into one contiguous [total_kv, 576] bf16 area of
// the workspace, in sequence order.  Scattered 1152-byte rows are fetched once
// here, so the tensor-core kernel streams contiguous 64-row tiles with tiled
// TMA loads instead of row-by-row gathers.  This is the compaction of scattered
// page_size = 1 slots into contiguous runs that "The Build That Unlocked 3-6x
// Decode Speedup" names as the plan's next phase (section "The Context: A
// Custom Kernel for an Unsupported Architecture"), done per call.
//
// One warp per four rows at a time: lane l moves 16-byte granules l, l+32 and
// l+64 (< 72) of each, so every warp instruction reads and writes 512
// contiguous bytes; the four slots are read in one load and all twelve row
// loads are in flight before the stores, so a warp waits out one index read
// and one row read per four rows.  A slot outside [0, pool_slots) records
// VMLA_ERR_INDEX and stages a zero row.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "vmla_device.cuh"

namespace vmla {
namespace {

constexpr int kGatherWarps = 8;
constexpr int kRowU4 = kRowBytes / 16;  // 72
constexpr int kTileRows = 128;           // rows one tile of the tensor-core kernel covers

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

constexpr int kRowsPerWarp = 4;  // rows a gather warp has in flight

__global__ void __launch_bounds__(kGatherWarps * 32)
gather_rows_kernel(const uint4* __restrict__ pool, int64_t pool_slots, const int32_t* __restrict__ kv_indices,
                   int64_t total_kv, const int32_t* __restrict__ total_dev, uint4* __restrict__ staged,
                   uint32_t* status) {
  // the verify kernel may be scheduled as this grid's blocks retire (it waits for
  // the staged rows before it reads them)
  grid_dependents_launch();
  const int lane = threadIdx.x & 31;
  int64_t end = total_kv;
  if (total_dev) {
    // device-planned call: total_kv is the staged capacity and the rows are
    // kv_indptr[batch] of them (kv_indices holds the capacity's worth, so a count
    // the planner will reject still reads inside it); the tile after the last row
    // is zeroed too, as the tile loads' out-of-range fill would be, since it holds
    // an earlier call's rows
    const int64_t cap = total_kv, r = *total_dev > 0 ? *total_dev : 0;
    total_kv = r < cap ? r : cap;
    end = total_kv + kTileRows < cap ? total_kv + kTileRows : cap;
  }
  const int64_t warp0 = (int64_t)blockIdx.x * kGatherWarps + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * kGatherWarps;
  for (int64_t j = warp0 + total_kv; j < end; j += nwarps) {
    uint4* dst = staged + j * kRowU4;
    dst[lane] = make_uint4(0, 0, 0, 0);
    dst[lane + 32] = make_uint4(0, 0, 0, 0);
    if (lane < kRowU4 - 64) dst[lane + 64] = make_uint4(0, 0, 0, 0);
  }
  for (int64_t j0 = warp0 * kRowsPerWarp; j0 < total_kv; j0 += nwarps * kRowsPerWarp) {
    // lane k < kRowsPerWarp reads the slot of row j0 + k
    int32_t my = 0;
    if (lane < kRowsPerWarp && j0 + lane < total_kv) {
      my = kv_indices[j0 + lane];
      if (my < 0 || (int64_t)my >= pool_slots) {
        record_status(status, VMLA_ERR_INDEX, (uint32_t)(j0 + lane));
        my = -1;
      }
    }
    uint4 v[kRowsPerWarp][3];
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
      const int32_t slot = __shfl_sync(0xffffffffu, my, k);
      const bool ok = slot >= 0 && j0 + k < total_kv;
      const uint4* src = pool + (int64_t)(ok ? slot : 0) * kRowU4;
      v[k][0] = ok ? ld_stream(src + lane) : make_uint4(0, 0, 0, 0);
      v[k][1] = ok ? ld_stream(src + lane + 32) : make_uint4(0, 0, 0, 0);
      v[k][2] = (ok && lane < kRowU4 - 64) ? ld_stream(src + lane + 64) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
      if (j0 + k >= total_kv) break;
      uint4* dst = staged + (j0 + k) * kRowU4;
      dst[lane] = v[k][0];
      dst[lane + 32] = v[k][1];
      if (lane < kRowU4 - 64) dst[lane + 64] = v[k][2];
    }
  }
  // Started beside the device planner, this grid completes only after it (the kernels
  // after the gather read the plan); for a gather launched after its predecessor has
  // completed the wait returns at once.
  grid_dependency_wait();
}

// Two e4m3 codes (low byte first) -> two bf16 (low half first): exact to
// half precision, times the pool's scale in float32, rounded to bf16.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two_codes, float scale) {
  uint32_t h2;
  asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}" : "=r"(h2) : "r"(two_codes));
  const float lo = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
  const float hi = __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
  return pack_bf16x2(lo * scale, hi * scale);
}

// The same gather from a pool of e4m3 rows (576 bytes): lane l reads code
// granules l and, for l < 4, l + 32 (16 codes each) and writes their 16 bf16
// values as two granules of the staged row.
__global__ void __launch_bounds__(kGatherWarps * 32)
gather_rows_fp8_kernel(const uint4* __restrict__ pool, int64_t pool_slots, float scale,
                       const int32_t* __restrict__ kv_indices, int64_t total_kv, uint4* __restrict__ staged,
                       uint32_t* status) {
  grid_dependents_launch();
  constexpr int kCodeU4 = kDqk / 16;  // 36 granules of 16 codes
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (int64_t)blockIdx.x * kGatherWarps + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * kGatherWarps;
  for (int64_t j = warp0; j < total_kv; j += nwarps) {
    const int32_t slot = kv_indices[j];
    const bool ok = slot >= 0 && (int64_t)slot < pool_slots;
    if (!ok && lane == 0) record_status(status, VMLA_ERR_INDEX, (uint32_t)j);
    const uint4* src = pool + (int64_t)(ok ? slot : 0) * kCodeU4;
    uint4* dst = staged + j * kRowU4;
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
      const int g = lane + 32 * pass;
      if (g < kCodeU4) {
        const uint4 c = ok ? ld_stream(src + g) : make_uint4(0, 0, 0, 0);
        const uint32_t w[4] = {c.x, c.y, c.z, c.w};
        uint32_t o[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          o[2 * k] = e4m3x2_to_bf16x2(w[k] & 0xFFFFu, scale);
          o[2 * k + 1] = e4m3x2_to_bf16x2(w[k] >> 16, scale);
        }
        dst[2 * g] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[2 * g + 1] = make_uint4(o[4], o[5], o[6], o[7]);
      }
    }
  }
}

}  // namespace

namespace {
int launch_gather_impl(const RunArgs& a, const int32_t* total_dev, void* stream) {
  if (a.total_kv == 0) return VMLA_OK;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess)
    return VMLA_ERR_CUDA;
  const int64_t need = (a.total_kv + kGatherWarps * kRowsPerWarp - 1) / (kGatherWarps * kRowsPerWarp);
  // 8 blocks of 8 warps per SM keep enough rows in flight.  Beside the device planner the
  // blocks that find no room start as its blocks retire; a grid that left the planner's SMs
  // out would run the whole gather on fewer SMs, which costs more than the late start
  const int64_t cap = (int64_t)sms * 8;
  const int blocks = (int)(need < cap ? need : cap);
  if (a.kv_scale > 0.f) {
    if (total_dev) return VMLA_ERR_SHAPE;  // e4m3 pools are read by host-planned calls only
    gather_rows_fp8_kernel<<<blocks, kGatherWarps * 32, 0, (cudaStream_t)stream>>>(
        reinterpret_cast<const uint4*>(a.kv), a.pool_slots, a.kv_scale, a.kv_indices, a.total_kv,
        reinterpret_cast<uint4*>(a.staged), a.status);
    return cudaGetLastError() == cudaSuccess ? VMLA_OK : VMLA_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1] = {early_start_attribute()};
  cfg.gridDim = dim3(blocks, 1, 1);
  cfg.blockDim = dim3(kGatherWarps * 32, 1, 1);
  cfg.stream = (cudaStream_t)stream;
  cfg.attrs = attr;
  cfg.numAttrs = total_dev ? 1 : 0;  // early start only beside the device planner
  if (cudaLaunchKernelEx(&cfg, gather_rows_kernel, reinterpret_cast<const uint4*>(a.kv), a.pool_slots,
                         a.kv_indices, a.total_kv, total_dev, reinterpret_cast<uint4*>(a.staged), a.status) !=
      cudaSuccess)
    return VMLA_ERR_CUDA;
  return VMLA_OK;
}
}  // namespace

int launch_gather(const RunArgs& a, void* stream) { return launch_gather_impl(a, nullptr, stream); }

int launch_gather_dplan(const RunArgs& a, const int32_t* total_dev, void* stream) {
  return launch_gather_impl(a, total_dev, stream);
}

}  // namespace vmla
