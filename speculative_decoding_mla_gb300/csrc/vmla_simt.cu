// Plain CUDA-core verify attention: a second, independent GPU implementation
// of the operation, used to cross-check the tensor-core kernel.
//
// One CTA = one work unit = 32 query rows (r = i*H + h) of one sequence over
// one contiguous piece of its key range.  8 warps x 4 rows.  Key tiles of 32
// rows are gathered through kv_indices into shared memory (page_size = 1, so
// every key is its own 1152-byte row) and shared by all 32 query rows of the
// CTA.  Scores use the streaming, online-softmax form of the flash-decode
// kernel of "The Build That Unlocked 3-6x Decode Speedup", section "The
// Context: A Custom Kernel for an Unsupported Architecture" (running max and
// sum, accumulator rescaled when the max grows), in base-2 exponent form.
#include <cuda_runtime.h>

#include "vmla_device.cuh"

namespace vmla {
namespace {

constexpr int kRows = 32;        // rows per CTA
constexpr int kWarps = 8;
constexpr int kRowsPerWarp = 4;
constexpr int kTile = 32;        // keys per shared-memory tile
constexpr int kThreads = kWarps * 32;
constexpr int kRowU4 = kRowBytes / 16;  // 72 uint4 per 576-element row
constexpr int kQPairs = kDqk / 64;      // 9 bf16 pairs of q per lane
constexpr int kOPairs = kDv / 64;       // 8 bf16 pairs of out per lane

__global__ void __launch_bounds__(kThreads, 1)
simt_verify_kernel(const __grid_constant__ PlanParams plan, const RunArgs a) {
  extern __shared__ __align__(16) uint4 tile_u4[];  // [kTile][kRowU4]
  __shared__ int32_t slot_s[kTile];
  __shared__ float p_s[kWarps][kRowsPerWarp][kTile];

  const int unit = blockIdx.x;
  const int b = seq_of_unit(plan, unit);
  const SeqPlan& sp = plan.seq[b];
  const int H = plan.num_heads;
  const int local = unit - sp.unit_start;
  const int rb = local % sp.n_rb;
  const int piece = local / sp.n_rb;
  const int R = sp.n_q * H;
  const int prefix = sp.n_kv - sp.n_q;
  const int k_lo = piece * sp.chunk;
  const int k_hi = min(sp.n_kv, k_lo + sp.chunk);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  float qv[kRowsPerWarp][2 * kQPairs];
  float o[kRowsPerWarp][2 * kOPairs];
  float m[kRowsPerWarp], l[kRowsPerWarp];
  uint64_t vis[kRowsPerWarp];
  bool active[kRowsPerWarp];
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const int r = rb * kRows + warp * kRowsPerWarp + rr;
    active[rr] = r < R;
    const int rc = active[rr] ? r : 0;
    const int i = rc / H, h = rc % H;
    const int t = sp.q_off + i;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(a.q + ((int64_t)t * H + h) * kDqk);
#pragma unroll
    for (int c = 0; c < kQPairs; ++c) {
      uint32_t w = active[rr] ? __ldg(qrow + c * 32 + lane) : 0u;
      qv[rr][2 * c] = bf16_lo(w);
      qv[rr][2 * c + 1] = bf16_hi(w);
    }
#pragma unroll
    for (int c = 0; c < 2 * kOPairs; ++c) o[rr][c] = 0.f;
    m[rr] = -INFINITY;
    l[rr] = 0.f;
    vis[rr] = a.masks ? a.masks[t] : causal_bits(i);
  }

  const uint4* pool = reinterpret_cast<const uint4*>(a.kv);
  for (int base = k_lo; base < k_hi; base += kTile) {
    if (threadIdx.x < kTile) {
      const int j = base + threadIdx.x;
      int32_t slot = -1;
      if (j < k_hi) {
        slot = a.kv_indices[sp.kv_off + j];
        if (slot < 0 || (int64_t)slot >= a.pool_slots) {
          record_status(a.status, VMLA_ERR_INDEX, (uint32_t)(sp.kv_off + j));
          slot = -1;
        }
      }
      slot_s[threadIdx.x] = slot;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < kTile * kRowU4; idx += kThreads) {
      const int row = idx / kRowU4, col = idx - row * kRowU4;
      const int32_t slot = slot_s[row];
      uint4 v = make_uint4(0, 0, 0, 0);
      if (slot >= 0) v = __ldg(pool + (int64_t)slot * kRowU4 + col);
      tile_u4[idx] = v;
    }
    __syncthreads();

    const uint32_t* tile_w = reinterpret_cast<const uint32_t*>(tile_u4);  // [kTile][288] words
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
      if (!active[rr]) continue;
      // partial dot products of this lane's 18 dims with every key of the tile
      float part[kTile];
#pragma unroll
      for (int j = 0; j < kTile; ++j) {
        const uint32_t* kr = tile_w + j * (kDqk / 2);
        float acc = 0.f;
#pragma unroll
        for (int c = 0; c < kQPairs; ++c) {
          const uint32_t w = kr[c * 32 + lane];
          acc = fmaf(qv[rr][2 * c], bf16_lo(w), acc);
          acc = fmaf(qv[rr][2 * c + 1], bf16_hi(w), acc);
        }
        part[j] = acc;
      }
      // butterfly reduce-scatter: afterwards this lane holds the full score of key `lane`
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int k = 0; k < off; ++k) {
          const float mine = upper ? part[k + off] : part[k];
          const float other = upper ? part[k] : part[k + off];
          part[k] = mine + __shfl_xor_sync(0xffffffffu, other, off);
        }
      }
      const int j = base + lane;
      // a slot outside the pool reads as a zero row (score 0, value 0) and stays visible,
      // as in the tensor-core kernel
      bool visible = j < k_hi;
      if (visible && j >= prefix) visible = ((vis[rr] >> (j - prefix)) & 1ull) != 0;
      const float s2 = visible ? part[0] * a.scale_log2 : -INFINITY;
      const float mx = warp_max(s2);
      const float m_new = fmaxf(m[rr], mx);
      float alpha = 1.f, p = 0.f;
      if (m_new != -INFINITY) {
        alpha = exp2f(m[rr] - m_new);
        p = visible ? exp2f(s2 - m_new) : 0.f;
      }
      m[rr] = m_new;
      l[rr] = l[rr] * alpha + p;
      p_s[warp][rr][lane] = p;
#pragma unroll
      for (int c = 0; c < 2 * kOPairs; ++c) o[rr][c] *= alpha;
    }
    __syncwarp();
    // o += p . V  (V = latent part of the tile rows), tile reads shared by the warp's rows
#pragma unroll 4
    for (int jj = 0; jj < kTile; ++jj) {
      const uint32_t* vr = tile_w + jj * (kDqk / 2);
      float pv[kRowsPerWarp];
#pragma unroll
      for (int rr = 0; rr < kRowsPerWarp; ++rr) pv[rr] = p_s[warp][rr][jj];
#pragma unroll
      for (int c = 0; c < kOPairs; ++c) {
        const uint32_t w = vr[c * 32 + lane];
        const float lo = bf16_lo(w), hi = bf16_hi(w);
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
          o[rr][2 * c] = fmaf(pv[rr], lo, o[rr][2 * c]);
          o[rr][2 * c + 1] = fmaf(pv[rr], hi, o[rr][2 * c + 1]);
        }
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const float lsum = warp_sum(l[rr]);
    if (!active[rr]) continue;
    const int r = rb * kRows + warp * kRowsPerWarp + rr;
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    const float lse2 = lsum > 0.f ? m[rr] + log2f(lsum) : -INFINITY;
    if (sp.n_split == 1) {
      const int64_t orow = (int64_t)sp.q_off * H + r;
      uint32_t* dst = reinterpret_cast<uint32_t*>(a.out + orow * kDv);
#pragma unroll
      for (int c = 0; c < kOPairs; ++c) dst[c * 32 + lane] = pack_bf16x2(o[rr][2 * c] * inv, o[rr][2 * c + 1] * inv);
      if (lane == 0) a.lse[orow] = lsum > 0.f ? lse2 * 0.6931471805599453f : -INFINITY;
    } else {
      const int64_t prow = (int64_t)sp.part_off + (int64_t)piece * R + r;
      float2* dst = reinterpret_cast<float2*>(a.part_o + prow * kDv);
#pragma unroll
      for (int c = 0; c < kOPairs; ++c) dst[c * 32 + lane] = make_float2(o[rr][2 * c] * inv, o[rr][2 * c + 1] * inv);
      if (lane == 0) a.part_lse[prow] = lse2;
    }
  }
}

}  // namespace

int launch_simt(const PlanParams& plan, const RunArgs& args, void* stream) {
  if (plan.total_units == 0) return VMLA_OK;
  const size_t smem = (size_t)kTile * kRowBytes;  // 36,864 B: under the 48 KB default
  simt_verify_kernel<<<plan.total_units, kThreads, smem, (cudaStream_t)stream>>>(plan, args);
  return cudaGetLastError() == cudaSuccess ? VMLA_OK : VMLA_ERR_CUDA;
}

}  // namespace vmla
