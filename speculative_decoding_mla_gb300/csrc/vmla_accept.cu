// Greedy acceptance of a verified draft tree.
//
// "The Build That Unlocked 3-6x Decode Speedup" lists a tree_accept kernel
// beside the verify kernels (section "The Context: A Custom Kernel for an
// Unsupported Architecture") without describing it.  This is the plain
// reading of greedy tree verification: draft node i proposes a token after its
// parent (the prefix for a root); it is accepted when its parent is accepted
// and its token equals the target model's greedy token after the parent.  The
// chosen path ends at the deepest accepted node, the smallest index among
// equally deep ones; the next token is the target's token after that node.
//
// One warp per sequence: the lanes stage its at most 64 parents and tokens in
// shared memory with coalesced loads, lane 0 walks the nodes in index order
// (parents come before their children; a 64-bit word of accepted nodes and
// each node's depth decide every node in one pass), and the lanes write the
// path back.
#include <cuda_runtime.h>

#include "vmla_device.cuh"

namespace vmla {
namespace {

constexpr int kAcceptWarps = 4;

__global__ void __launch_bounds__(kAcceptWarps * 32)
tree_accept_kernel(const int32_t* __restrict__ qo_indptr, const int32_t* __restrict__ parent,
                   const int32_t* __restrict__ draft, const int32_t* __restrict__ target,
                   const int32_t* __restrict__ root, int batch, int total_q, int32_t* __restrict__ accept_len,
                   int32_t* __restrict__ path, int32_t* __restrict__ next_token, uint32_t* status) {
  __shared__ int32_t s_par[kAcceptWarps][VMLA_MAX_DRAFT], s_draft[kAcceptWarps][VMLA_MAX_DRAFT],
      s_tgt[kAcceptWarps][VMLA_MAX_DRAFT], s_path[kAcceptWarps][VMLA_MAX_DRAFT];
  __shared__ uint8_t s_depth[kAcceptWarps][VMLA_MAX_DRAFT];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * kAcceptWarps + w;  // warp-uniform
  if (b >= batch) return;
  const int q0 = qo_indptr[b];
  const int n = qo_indptr[b + 1] - q0;
  const bool in_range = n >= 0 && n <= VMLA_MAX_DRAFT && q0 >= 0 && q0 + n <= total_q;
  const int m = in_range ? n : 0;
  for (int k = lane; k < m; k += 32) {
    s_par[w][k] = parent ? parent[q0 + k] : k - 1;
    s_draft[w][k] = draft[q0 + k];
    s_tgt[w][k] = target[q0 + k];
  }
  __syncwarp();
  int len = 0, best = -1, bad = in_range ? 0 : 1;
  if (lane == 0) {
    const int rt = root[b];
    uint64_t accepted = 0;
    int best_depth = -1;
    for (int i = 0; i < m; ++i) {
      const int p = s_par[w][i];
      if (p < -1 || p >= i) {
        bad = 1;
        break;
      }
      const int expected = p < 0 ? rt : s_tgt[w][p];
      const bool ok = (p < 0 || ((accepted >> p) & 1ull)) && s_draft[w][i] == expected;
      const int d = p < 0 ? 0 : s_depth[w][p] + 1;
      s_depth[w][i] = (uint8_t)d;
      if (ok) {
        accepted |= 1ull << i;
        if (d > best_depth) {
          best_depth = d;
          best = i;
        }
      }
    }
    if (bad) best = -1;
    len = best < 0 ? 0 : best_depth + 1;
    for (int k = len - 1, node = best; k >= 0; --k) {
      s_path[w][k] = node;
      node = s_par[w][node];
    }
    if (bad) record_status(status, VMLA_ERR_PARENT, (uint32_t)b);
    accept_len[b] = len;
    next_token[b] = best < 0 ? rt : s_tgt[w][best];
  }
  len = __shfl_sync(0xffffffffu, len, 0);
  __syncwarp();
  // the sequence's path entries, root first; -1 after the path
  for (int k = lane; k < m; k += 32) path[q0 + k] = k < len ? s_path[w][k] : -1;
}

}  // namespace

int launch_tree_accept(const int32_t* qo_indptr, const int32_t* parent, const int32_t* draft, const int32_t* target,
                       const int32_t* root, int batch, int total_q, int32_t* accept_len, int32_t* path,
                       int32_t* next_token, uint32_t* status, void* stream) {
  if (batch == 0) return VMLA_OK;
  tree_accept_kernel<<<(batch + kAcceptWarps - 1) / kAcceptWarps, kAcceptWarps * 32, 0, (cudaStream_t)stream>>>(
      qo_indptr, parent, draft, target, root, batch, total_q, accept_len, path, next_token, status);
  return cudaGetLastError() == cudaSuccess ? VMLA_OK : VMLA_ERR_CUDA;
}

}  // namespace vmla
