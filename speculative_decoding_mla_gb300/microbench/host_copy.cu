// Microbenchmark: a pinned host buffer moved to or from the device by the copy
// engine (one cudaMemcpyAsync) against a kernel that reads or writes it through
// its mapped device address, at the host-buffer call's sizes (long_185k's 740 KB
// of kv_indices, 1.2 MB of q, 1 MB of out).  Each transfer is timed on the host
// from its issue to the stream's synchronisation, median of 40; the empty
// synchronisation is printed beside them.
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O2 -o /tmp/host_copy \
//        speculative_decoding_mla_gb300/microbench/host_copy.cu && /tmp/host_copy
#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <cstdio>
#include <cstring>
#include <vector>

__global__ void copy_granules(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

template <class F>
double median_us(cudaStream_t st, F fn) {
  std::vector<double> v;
  for (int i = 0; i < 40; ++i) {
    cudaStreamSynchronize(st);
    const auto a = std::chrono::steady_clock::now();
    fn();
    cudaStreamSynchronize(st);
    v.push_back(std::chrono::duration<double, std::micro>(std::chrono::steady_clock::now() - a).count());
  }
  std::sort(v.begin(), v.end());
  return v[v.size() / 2];
}

int main() {
  const size_t sizes[] = {740064, 1179648, 1048576};
  cudaStream_t st;
  if (cudaStreamCreate(&st) != cudaSuccess) return 1;
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  for (size_t bytes : sizes) {
    void *h = nullptr, *d = nullptr, *hd = nullptr;
    if (cudaHostAlloc(&h, bytes, cudaHostAllocMapped) != cudaSuccess || cudaMalloc(&d, bytes) != cudaSuccess ||
        cudaHostGetDevicePointer(&hd, h, 0) != cudaSuccess) {
      std::printf("allocation failed: %s\n", cudaGetErrorString(cudaGetLastError()));
      return 1;
    }
    std::memset(h, 1, bytes);
    const size_t n = bytes / 16;
    const int grid = sms * 4;
    const double h2d_ce = median_us(st, [&] { cudaMemcpyAsync(d, h, bytes, cudaMemcpyHostToDevice, st); });
    const double h2d_k = median_us(st, [&] { copy_granules<<<grid, 256, 0, st>>>((const uint4*)hd, (uint4*)d, n); });
    const double d2h_ce = median_us(st, [&] { cudaMemcpyAsync(h, d, bytes, cudaMemcpyDeviceToHost, st); });
    const double d2h_k = median_us(st, [&] { copy_granules<<<grid, 256, 0, st>>>((const uint4*)d, (uint4*)hd, n); });
    const double sync = median_us(st, [] {});
    std::printf("%zu bytes: to device %.1f us (copy engine) / %.1f us (kernel on mapped memory); "
                "to host %.1f / %.1f us; synchronisation alone %.1f us\n",
                bytes, h2d_ce, h2d_k, d2h_ce, d2h_k, sync);
    cudaFreeHost(h);
    cudaFree(d);
  }
  const cudaError_t e = cudaGetLastError();
  std::printf("status: %s\n", cudaGetErrorString(e));
  return e == cudaSuccess ? 0 : 1;
}
