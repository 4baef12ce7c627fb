// Allocation-free entry point: the CUDA-core verify path with its scratch in a
// fixed array that lives in the library image on every device that loads it.
//
// Some callers cannot allocate device memory when they call in: code that runs
// under a memory pool or arena it does not own (a serving engine that has
// handed all free HBM to its KV cache), a custom allocator that must not be
// re-entered from inside a callback, or a plugin host that forbids cudaMalloc
// outside its own set-up phase.  They still own their inputs and outputs; this
// entry point only removes the workspace argument.
#include <cuda_runtime.h>

#include "vmla_internal.h"

namespace vmla {
namespace {

// Scratch for the status word, ancestor masks and split partials of one call.
__device__ __align__(256) unsigned char g_vmla_static_scratch[VMLA_STATIC_SCRATCH_BYTES];

// Device address of the scratch array on the current device.  It is looked up on
// every call (a host-side lookup in the loaded module): after a device reset the
// module is loaded again and the array may sit elsewhere, so no address is kept.
int static_scratch(void** ptr) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_vmla_static_scratch) != cudaSuccess || !p) return VMLA_ERR_CUDA;
  *ptr = p;
  return VMLA_OK;
}

}  // namespace
}  // namespace vmla

extern "C" int verify_attn_mla_simt_static_check(void* stream) {
  void* scratch = nullptr;
  int rc = vmla::static_scratch(&scratch);
  if (rc != VMLA_OK) return rc;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return VMLA_ERR_CUDA;
  // the status words open the scratch layout (offset 0), as they open a workspace
  uint32_t word[2] = {0, 0};
  if (cudaMemcpyFromSymbol(word, vmla::g_vmla_static_scratch, sizeof word, 0, cudaMemcpyDeviceToHost) != cudaSuccess)
    return VMLA_ERR_CUDA;
  return (int)(int32_t)word[0];
}

extern "C" int verify_attn_mla_simt_static(const void* q, const void* kv_pool, int64_t pool_slots,
                                           const int32_t* kv_indptr, const int32_t* kv_indices,
                                           const int32_t* qo_indptr, const uint64_t* draft_mask,
                                           const int32_t* parent, const int32_t* kv_indptr_host,
                                           const int32_t* qo_indptr_host, int batch, int num_heads, float sm_scale,
                                           int splits, void* out, float* lse, void* stream) {
  void* scratch = nullptr;
  int rc = vmla::static_scratch(&scratch);
  if (rc != VMLA_OK) return rc;
  // a plan that needs more than the array is refused (VMLA_ERR_WORKSPACE) before any launch
  return vmla::run_verify(VMLA_KERNEL_SIMT, q, kv_pool, pool_slots, 0.f, kv_indptr, kv_indices, nullptr, qo_indptr,
                          draft_mask,
                          parent, kv_indptr_host, qo_indptr_host, batch, num_heads, sm_scale, splits, out, lse,
                          scratch, VMLA_STATIC_SCRATCH_BYTES, stream);
}
