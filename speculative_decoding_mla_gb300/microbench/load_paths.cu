// Microbenchmark: how fast one SM fills a two-stage shared-memory buffer of
// 64 KV rows x 576 bf16 columns (nine 128-byte-swizzled 64-column chunks, the
// layout the verify kernel's score MMAs read) when the rows are scattered
// 1152-byte pool rows (page_size = 1), by each load mechanism sm_103a offers:
//   tma_tile       tiled TMA loads of 64 contiguous rows (the staged layout)
//   gather4_lane0  TMA tile::gather4 (four rows x 64 columns), issued by lane 0 of each loader warp
//   gather4_all    the same, issued by every lane of the loader warps
//   ldgsts_noinc   16-byte cp.async by every lane, completion by cp.async.mbarrier.arrive.noinc
//   ldgsts_wait    16-byte cp.async, each warp waits for its own copies and arrives once
// One CTA per SM, W loader warps and one consumer thread that frees a stage
// after a fixed hold (0 or 1500 ns, standing in for the MMAs).  The slots of a
// load are read before the previous load's copies are issued.  Prints µs per
// 73,728-byte load per SM.  Two last sweeps repeat the tiled loads with the
// shared-memory request padded (unused bytes), which leaves the SM less L1, and
// with each CTA starting at its own phase of the hold (loads not in step).
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 \
//        -Ispeculative_decoding_mla_gb300/csrc -Iinclude -o /tmp/load_paths \
//        speculative_decoding_mla_gb300/microbench/load_paths.cu && /tmp/load_paths
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdio>
#include <cstdlib>
#include <vector>
#include <random>
#include <algorithm>
#include "vmla_sm100.cuh"
using namespace vmla::sm100;

constexpr int kStageBytes = 9 * 8192;
struct Smem {
  uint8_t kv[2][9][8192];
  uint64_t full[2], empty[2];
};

__device__ int g_err;

__device__ __forceinline__ bool bwait(uint64_t* bar, uint32_t par) {
  long long t0 = clock64();
  while (!mbar_try_wait(bar, par)) {
    if (clock64() - t0 > 4000000000LL) { atomicExch(&g_err, 1); return false; }
  }
  return true;
}

__device__ __forceinline__ void cp16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

template <int MODE>
__global__ void __launch_bounds__(416, 1) probe(const __grid_constant__ CUtensorMap tmap,
                                                const __grid_constant__ CUtensorMap gmap, const uint8_t* pool,
                                                const int* idx, int n_idx, int pool_rows, int tiles, int W,
                                                int delay_ns, int phase_ns) {
  extern __shared__ uint8_t raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.full[s], MODE == 3 ? W * 32 : (MODE == 4 ? W : 1));
      mbar_init(&sm.empty[s], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (warp < W) {
    if (phase_ns > 0) {  // this CTA's loads start at its own phase of the hold (bounded wait on the timer)
      const unsigned long long t0 = gtimer(), wait = (unsigned long long)((blockIdx.x * 97) % phase_ns);
      for (int k = 0; k < (1 << 22) && gtimer() - t0 < wait; ++k) {
      }
    }
    // slots of this tile's 64 rows: lane l holds rows l and l + 32 (prefetched one tile ahead)
    int s_lo;
    int s_hi = idx[(((long long)blockIdx.x * tiles) * 64 + lane + 32) % n_idx];
    s_lo = idx[(((long long)blockIdx.x * tiles) * 64 + lane) % n_idx];
    for (int it = 0; it < tiles; ++it) {
      const int s = it & 1;
      const long long base = ((long long)blockIdx.x * tiles + it) * 64;
      // next tile's slots, loaded before this tile's copies are issued
      const long long nb = base + 64;
      const int n_lo = idx[(nb + lane) % n_idx], n_hi = idx[(nb + lane + 32) % n_idx];
      if (!bwait(&sm.empty[s], ((it >> 1) & 1) ^ 1)) break;
      if (MODE == 0) {
        if (warp == 0 && lane == 0) {
          mbar_arrive_expect_tx(&sm.full[s], kStageBytes);
          const int y = (int)(base % (pool_rows - 64));
          for (int c = 0; c < 9; ++c) tma_load_2d(smem_u32(&sm.kv[s][c][0]), &tmap, 64 * c, y, smem_u32(&sm.full[s]));
        }
      } else if (MODE == 1 || MODE == 2) {
        if (warp == 0 && lane == 0) mbar_arrive_expect_tx(&sm.full[s], kStageBytes);
        const int nthr = MODE == 1 ? W : W * 32;
        const int me = MODE == 1 ? warp : warp * 32 + lane;
        // every lane takes part in the shuffles; only lanes with an op issue it
        for (int o0 = 0; o0 < 144; o0 += nthr) {
          const int o = o0 + me;
          const int g = o & 15;
          int y[4];
          for (int k = 0; k < 4; ++k) {
            const int r = 4 * g + k;
            const int v_lo = __shfl_sync(0xffffffffu, s_lo, r & 31);
            const int v_hi = __shfl_sync(0xffffffffu, s_hi, r & 31);
            y[k] = r < 32 ? v_lo : v_hi;
          }
          if (o < 144 && (MODE == 2 || lane == 0)) {
            const int c = o >> 4;
            tma_gather4(smem_u32(&sm.kv[s][c][0]) + g * 512, &gmap, 64 * c, y[0], y[1], y[2], y[3],
                        smem_u32(&sm.full[s]));
          }
        }
      } else {
        for (int f0 = 0; f0 < 64 * 72; f0 += W * 32) {
          const int f = f0 + warp * 32 + lane;
          const int r = (f < 64 * 72 ? f : 0) / 72;
          const int v_lo = __shfl_sync(0xffffffffu, s_lo, r & 31);
          const int v_hi = __shfl_sync(0xffffffffu, s_hi, r & 31);
          const int slot = r < 32 ? v_lo : v_hi;
          if (f < 64 * 72) {
            const int g = f - r * 72;
            const int c = g >> 3, gg = g & 7;
            const uint32_t dst = smem_u32(&sm.kv[s][c][0]) + r * 128 + ((gg ^ (r & 7)) << 4);
            cp16(dst, pool + (size_t)slot * 1152 + g * 16);
          }
        }
        if (MODE == 3) {
          cp_arrive_noinc(&sm.full[s]);
        } else {
          cp_commit();
          cp_wait_all();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.full[s]);
        }
      }
      s_lo = n_lo;
      s_hi = n_hi;
    }
  } else if (warp == W && lane == 0) {
    for (int it = 0; it < tiles; ++it) {
      const int s = it & 1;
      if (!bwait(&sm.full[s], (it >> 1) & 1)) break;
      fence_proxy_async_smem();
      if (delay_ns > 0) {
        unsigned long long t0 = gtimer();
        while (gtimer() - t0 < (unsigned long long)delay_ns) {
        }
      }
      mbar_arrive(&sm.empty[s]);
    }
  }
  __syncthreads();
}

typedef CUresult (*EncFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*, const cuuint64_t*,
                          const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                          CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

#define CK(x)                                                                          \
  do {                                                                                 \
    cudaError_t e = (x);                                                               \
    if (e != cudaSuccess) {                                                            \
      printf("CUDA error %s at %s:%d\n", cudaGetErrorString(e), __FILE__, __LINE__);   \
      exit(1);                                                                         \
    }                                                                                  \
  } while (0)

template <int MODE>
float run(const CUtensorMap& tm, const CUtensorMap& gm, const uint8_t* pool, const int* idx, int n_idx, int rows,
          int tiles, int W, int delay, int grid, size_t pad = 0, int phase = 0) {
  size_t smem = sizeof(Smem) + 1024 + pad;
  CK(cudaFuncSetAttribute(probe<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  cudaEvent_t a, b;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  probe<MODE><<<grid, (W + 1) * 32, smem>>>(tm, gm, pool, idx, n_idx, rows, tiles, W, delay, phase);
  CK(cudaGetLastError());
  CK(cudaDeviceSynchronize());
  cudaEventRecord(a);
  probe<MODE><<<grid, (W + 1) * 32, smem>>>(tm, gm, pool, idx, n_idx, rows, tiles, W, delay, phase);
  cudaEventRecord(b);
  CK(cudaDeviceSynchronize());
  float ms;
  cudaEventElapsedTime(&ms, a, b);
  int err = 0;
  CK(cudaMemcpyFromSymbol(&err, g_err, 4));
  if (err) printf("  (timeout flagged)\n");
  return ms;
}

int main() {
  const int rows = 200000;
  int sms = 0;
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  uint8_t* pool;
  CK(cudaMalloc(&pool, (size_t)rows * 1152));
  CK(cudaMemset(pool, 1, (size_t)rows * 1152));
  std::vector<int> h(rows);
  for (int i = 0; i < rows; ++i) h[i] = i;
  std::mt19937 rng(3);
  std::shuffle(h.begin(), h.end(), rng);
  int* idx;
  CK(cudaMalloc(&idx, rows * 4));
  CK(cudaMemcpy(idx, h.data(), rows * 4, cudaMemcpyHostToDevice));
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  CK(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q));
  EncFn enc = (EncFn)p;
  CUtensorMap tm, gm;
  cuuint64_t gdim[2] = {576, (cuuint64_t)rows};
  cuuint64_t gstr[1] = {1152};
  cuuint32_t box_t[2] = {64, 64}, box_g[2] = {64, 1}, es[2] = {1, 1};
  if (enc(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pool, gdim, gstr, box_t, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != 0 ||
      enc(&gm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pool, gdim, gstr, box_g, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != 0) {
    printf("encode failed\n");
    return 1;
  }
  const int tiles = 300;
  const char* names[] = {"tma_tile", "gather4_lane0", "gather4_all", "ldgsts_noinc", "ldgsts_wait"};
  for (int grid : {sms}) {
    for (int delay : {0, 1500}) {
      for (int mode = 0; mode < 5; ++mode) {
        for (int W : {1, 2, 4, 8, 12}) {
          if (mode == 0 && W > 1) continue;
          float ms = 0;
          switch (mode) {
            case 0: ms = run<0>(tm, gm, pool, idx, rows, rows, tiles, W, delay, grid); break;
            case 1: ms = run<1>(tm, gm, pool, idx, rows, rows, tiles, W, delay, grid); break;
            case 2: ms = run<2>(tm, gm, pool, idx, rows, rows, tiles, W, delay, grid); break;
            case 3: ms = run<3>(tm, gm, pool, idx, rows, rows, tiles, W, delay, grid); break;
            case 4: ms = run<4>(tm, gm, pool, idx, rows, rows, tiles, W, delay, grid); break;
          }
          const double us_tile = ms * 1e3 / tiles;
          const double gbs_sm = kStageBytes / (us_tile * 1e3);
          printf("grid %3d delay %4d %-14s W=%d  %.3f us/tile  %.1f GB/s/SM  %.0f GB/s total\n", grid, delay,
                 names[mode], W, us_tile, gbs_sm, gbs_sm * grid);
        }
      }
    }
  }
  // tiled loads with the shared-memory request padded to about 148, 196 and 225 KB
  for (int delay : {0, 1500})
    for (size_t pad : {(size_t)0, (size_t)49152, (size_t)77824}) {
      const float ms = run<0>(tm, gm, pool, idx, rows, rows, tiles, 1, delay, sms, pad);
      const double us_tile = ms * 1e3 / tiles;
      printf("smem %6zu B delay %4d tma_tile  %.3f us/tile  %.1f GB/s/SM\n", sizeof(Smem) + 1024 + pad, delay, us_tile,
             kStageBytes / (us_tile * 1e3));
    }
  // tiled loads under a 1.5 us hold with each CTA starting at its own phase (0 .. 1.5 us)
  for (int phase : {0, 1500}) {
    const float ms = run<0>(tm, gm, pool, idx, rows, rows, tiles, 1, 1500, sms, 0, phase);
    const double us_tile = ms * 1e3 / tiles;
    printf("phase spread %4d ns delay 1500 tma_tile  %.3f us/tile  %.1f GB/s/SM\n", phase, us_tile,
           kStageBytes / (us_tile * 1e3));
  }
  return 0;
}
