// Small device helpers shared by the library's kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "vmla_internal.h"

namespace vmla {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two floats -> packed bf16x2 (lo in bits 0-15), round to nearest even, one instruction.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// 2^x on the special-function unit (flushes denormal results to zero; 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start while the kernel before it in the stream still runs
// (once every block of that kernel has signalled, or exited); it must wait for
// that kernel's completion and memory before it reads anything the kernel
// wrote.  Without such a launch the wait returns at once.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// Launch attribute that lets a kernel start under the tail of the one before it
// (it then calls grid_dependency_wait before reading that kernel's output).
inline cudaLaunchAttribute early_start_attribute() {
  cudaLaunchAttribute a = {};
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

// First fault wins: records code and info in the workspace status word.
__device__ __forceinline__ void record_status(uint32_t* status, int code, uint32_t info) {
  if (!status) return;
  if (atomicCAS(status, 0u, (uint32_t)code) == 0u) status[1] = info;
}

// Visibility word of draft query i when no explicit word is given: bits 0..i.
__device__ __forceinline__ uint64_t causal_bits(int i) { return ~0ull >> (63 - i); }

// Sequence owning work unit `unit` (largest b with seq[b].unit_start <= unit and rows to do).
__device__ __forceinline__ int seq_of_unit(const PlanParams& p, int unit) {
  int lo = 0, hi = p.batch;
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (p.seq[mid].unit_start <= unit) lo = mid; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace vmla
