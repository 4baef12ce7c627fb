// C ABI of the verify attention: argument checks, planning, workspace carving
// and the launches, in stream order.  Exports are declared in
// include/verify_attn_mla.h.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "vmla_internal.h"

using namespace vmla;

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Checks shared by every run entry point; host arrays only.
int check_common(const int32_t* kv_indptr_host, const int32_t* qo_indptr_host, int batch, int num_heads,
                 int64_t pool_slots, int splits) {
  if (!kv_indptr_host || !qo_indptr_host) return VMLA_ERR_NULL;
  if (batch < 0 || batch > VMLA_MAX_BATCH || num_heads < 1 || num_heads > VMLA_MAX_HEADS) return VMLA_ERR_SHAPE;
  if (splits < VMLA_SPLITS_LANES || splits > 64 || pool_slots < 0 || pool_slots > INT32_MAX) return VMLA_ERR_SHAPE;
  if (kv_indptr_host[0] != 0 || qo_indptr_host[0] != 0) return VMLA_ERR_SHAPE;
  for (int b = 0; b < batch; ++b) {
    int64_t nq = (int64_t)qo_indptr_host[b + 1] - qo_indptr_host[b];
    int64_t nk = (int64_t)kv_indptr_host[b + 1] - kv_indptr_host[b];
    if (nq < 0 || nq > VMLA_MAX_DRAFT || nk < nq) return VMLA_ERR_SHAPE;
  }
  return VMLA_OK;
}

// Optional per-call kernel timing (see verify_attn_mla_timing_enable).
struct Timing {
  std::mutex mu;
  int cap = 0;
  int n = 0;
  std::vector<cudaEvent_t> ev;  // 6 per call: verify begin/end, merge begin/end, gather begin/end
  std::vector<char> merged;
};
Timing g_timing;
constexpr char kTimingFailed = 4;  // `merged` value of a call that failed after taking its slot

cudaEvent_t timing_event(int call, int k) { return g_timing.ev[(size_t)call * 6 + k]; }

int current_sm_count(int* sms, bool require_sm103) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return VMLA_ERR_DEVICE;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return VMLA_ERR_DEVICE;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return VMLA_ERR_DEVICE;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return VMLA_ERR_DEVICE;
  if (require_sm103 && !(major == 10 && minor == 3)) return VMLA_ERR_DEVICE;
  return VMLA_OK;
}

}  // namespace

namespace {
// failure-test settings of this thread (verify_attn_mla_test_fault)
thread_local int32_t g_test_fault = 0;
thread_local long long g_test_wait_cycles = 0;
}  // namespace

namespace vmla {

void test_fault_settings(int32_t* fault, long long* wait_cycles) {
  *fault = g_test_fault;
  *wait_cycles = g_test_wait_cycles > 0 ? g_test_wait_cycles : kWaitCyclesDefault;
}

int run_verify(int kernel, const void* q, const void* kv_pool, int64_t pool_slots, float kv_scale,
        const int32_t* kv_indptr, const int32_t* kv_indices, const int32_t* run_base, const int32_t* qo_indptr,
        const uint64_t* draft_mask, const int32_t* parent, const int32_t* kv_indptr_host,
        const int32_t* qo_indptr_host, int batch, int num_heads, float sm_scale, int splits, void* out, float* lse,
        void* workspace, size_t workspace_bytes, void* stream, void* q_ready, const PlanParams* plan_in,
        const vmla_plan_info* info_in) {
  int rc = check_common(kv_indptr_host, qo_indptr_host, batch, num_heads, pool_slots, splits);
  if (rc != VMLA_OK) return rc;
  // a positive finite scale (the kernels take row maxima over unscaled scores)
  if (!(sm_scale > 0.f) || !(sm_scale < INFINITY)) return VMLA_ERR_SHAPE;
  const int64_t total_q = qo_indptr_host[batch];
  const int64_t total_kv = kv_indptr_host[batch];
  if (!workspace) return VMLA_ERR_NULL;
  const bool runs = run_base != nullptr;  // rows in per-sequence pool runs: no gather
  if (runs && kernel != VMLA_KERNEL_TC) return VMLA_ERR_SHAPE;
  // an e4m3 pool (kv_scale > 0, finite) is dequantized by the gather of the tensor-core path
  if (kv_scale != 0.f && (!(kv_scale > 0.f) || !(kv_scale < INFINITY) || runs || kernel != VMLA_KERNEL_TC))
    return VMLA_ERR_SHAPE;
  if (total_q > 0 && (!q || !kv_pool || !kv_indptr || (!runs && !kv_indices) || !qo_indptr || !out || !lse))
    return VMLA_ERR_NULL;
  if (!aligned(run_base, 4)) return VMLA_ERR_ALIGN;
  if (total_kv > 0 && pool_slots == 0) return VMLA_ERR_SHAPE;
  if (!aligned(q, 16) || !aligned(kv_pool, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
      !aligned(workspace, VMLA_WORKSPACE_ALIGN) || !aligned(draft_mask, 8) || !aligned(parent, 4))
    return VMLA_ERR_ALIGN;
  int sms = 0;
  rc = current_sm_count(&sms, true);
  if (rc != VMLA_OK) return rc;
  int clusters = 0;
  if (kernel == VMLA_KERNEL_TC) {
    rc = tc_max_clusters(&clusters);
    if (rc != VMLA_OK) return rc;
  }
  static thread_local PlanParams own_plan;  // large (20 KB); kept off the stack
  vmla_plan_info info;
  const bool have_plan = plan_in && info_in;
  if (have_plan) info = *info_in;
  // The areas no plan sizes (status, masks, staged rows) lead the workspace, so the
  // kernels that fill them are queued first and the host builds the plan while they
  // run; without a plan in hand only that part of the size is checked before them.
  const int64_t staged_rows = kernel == VMLA_KERNEL_TC && !runs ? total_kv : 0;
  WorkspaceLayout L = workspace_layout(total_q, have_plan ? info.partial_rows : 0, staged_rows);
  if (workspace_bytes < L.total) return VMLA_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws + L.status_off);
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(status, 0, 8, st) != cudaSuccess) return VMLA_ERR_CUDA;
  if (total_q == 0) return VMLA_OK;

  const uint64_t* masks = draft_mask;
  if (!masks && parent) {
    uint64_t* m = reinterpret_cast<uint64_t*>(ws + L.masks_off);
    rc = launch_tree_mask(parent, qo_indptr, batch, (int)total_q, m, status, stream);
    if (rc != VMLA_OK) return rc;
    masks = m;
  }
  RunArgs a;
  test_fault_settings(&a.test_fault, &a.wait_cycles);
  a.q = static_cast<const uint16_t*>(q);
  a.kv = static_cast<const uint16_t*>(kv_pool);
  a.pool_slots = pool_slots;
  a.kv_indices = kv_indices;
  a.masks = masks;
  a.sm_scale = sm_scale;
  a.scale_log2 = sm_scale * 1.4426950408889634f;
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.out_rows = (int64_t)total_q * num_heads;
  a.staged = runs ? const_cast<uint16_t*>(static_cast<const uint16_t*>(kv_pool))
                  : reinterpret_cast<uint16_t*>(ws + L.staged_off);
  a.total_kv = runs ? pool_slots : total_kv;
  a.run_base = run_base;
  a.kv_scale = kv_scale;
  a.status = status;
  int slot = -1;
  {
    std::lock_guard<std::mutex> g(g_timing.mu);
    if (g_timing.n < g_timing.cap) slot = g_timing.n++;
  }
  // a call that fails past this point leaves its timing slot marked, and the readout skips it
  auto failed = [&](int code) {
    if (slot >= 0) g_timing.merged[slot] = kTimingFailed;
    return code;
  };
  if (runs) {
    // the runs must lie in the pool (the kernel reads whatever the tile loads
    // return; this check reports a run outside it)
    rc = launch_defrag(nullptr, 0, kv_indptr, nullptr, kv_indptr_host, batch, total_kv, nullptr, pool_slots, run_base,
                       true, status,
                       stream);
    if (rc != VMLA_OK) return failed(rc);
  } else if (kernel == VMLA_KERNEL_TC) {
    // KV rows of every sequence gathered once into a contiguous staging area, so
    // that the verify kernel streams them with tiled TMA loads
    if (slot >= 0) cudaEventRecord(timing_event(slot, 4), st);
    rc = launch_gather(a, stream);
    if (rc != VMLA_OK) return failed(rc);
    if (slot >= 0) cudaEventRecord(timing_event(slot, 5), st);
  }
  if (!have_plan) {
    // (the shapes passed check_common, so the plan itself does not fail; a workspace
    // too small for its partial rows is reported with the staged rows already queued)
    rc = build_plan(kernel, batch, num_heads, qo_indptr_host, kv_indptr_host, splits, sms, clusters, &own_plan,
                    &info);
    if (rc != VMLA_OK) return failed(rc);
    L = workspace_layout(total_q, info.partial_rows, staged_rows);
    if (workspace_bytes < L.total) return failed(VMLA_ERR_WORKSPACE);
  }
  const PlanParams& plan = have_plan ? *plan_in : own_plan;
  a.part_rows = plan.partial_rows;
  a.part_o = reinterpret_cast<float*>(ws + L.part_o_off);
  a.part_lse = reinterpret_cast<float*>(ws + L.part_lse_off);
  if (q_ready && cudaStreamWaitEvent(st, (cudaEvent_t)q_ready, 0) != cudaSuccess) return failed(VMLA_ERR_CUDA);
  if (slot >= 0) cudaEventRecord(timing_event(slot, 0), st);
  rc = kernel == VMLA_KERNEL_SIMT ? launch_simt(plan, a, stream) : launch_tc(plan, a, stream);
  if (rc != VMLA_OK) return failed(rc);
  if (slot >= 0) {
    cudaEventRecord(timing_event(slot, 1), st);
    g_timing.merged[slot] = (char)((plan.merge_rows > 0 ? 1 : 0) | (kernel == VMLA_KERNEL_TC ? 2 : 0));
    if (plan.merge_rows > 0) cudaEventRecord(timing_event(slot, 2), st);
  }
  rc = launch_merge(plan, a.part_o, a.part_lse, 1, a.out, a.lse, stream);
  if (rc != VMLA_OK) return failed(rc);
  if (slot >= 0 && plan.merge_rows > 0) cudaEventRecord(timing_event(slot, 3), st);
  return rc;
}

}  // namespace vmla

extern "C" {

int verify_attn_mla_plan(int kernel, int batch, int num_heads, const int32_t* qo_indptr_host,
                         const int32_t* kv_indptr_host, int splits, int num_sms, vmla_plan_info* info,
                         int32_t* splits_out) {
  if (!info) return VMLA_ERR_NULL;
  static thread_local PlanParams plan;
  int rc = build_plan(kernel, batch, num_heads, qo_indptr_host, kv_indptr_host, splits, num_sms, 0, &plan, info);
  if (rc == VMLA_OK && splits_out)
    for (int b = 0; b < batch; ++b) splits_out[b] = plan.seq[b].n_split;
  return rc;
}

int verify_attn_mla_workspace_size(int batch, int num_heads, const int32_t* qo_indptr_host,
                                   const int32_t* kv_indptr_host, int splits, size_t* bytes) {
  if (!bytes) return VMLA_ERR_NULL;
  int sms = 0;
  int rc = current_sm_count(&sms, false);
  if (rc != VMLA_OK) return rc;
  // the tensor-core plan with this device's co-resident cluster count, as a call would make it
  int clusters = 0;
  rc = vmla::tc_max_clusters(&clusters);
  if (rc != VMLA_OK) return rc;
  static thread_local vmla::PlanParams plan;
  vmla_plan_info info;
  rc = vmla::build_plan(VMLA_KERNEL_TC, batch, num_heads, qo_indptr_host, kv_indptr_host, splits, sms, clusters, &plan,
                        &info);
  if (rc != VMLA_OK) return rc;
  vmla_plan_info info2;
  rc = verify_attn_mla_plan(VMLA_KERNEL_SIMT, batch, num_heads, qo_indptr_host, kv_indptr_host, splits, sms, &info2,
                            nullptr);
  if (rc != VMLA_OK) return rc;
  // one size serves both kernels
  *bytes = info.workspace_bytes > info2.workspace_bytes ? info.workspace_bytes : info2.workspace_bytes;
  return VMLA_OK;
}

int verify_attn_mla(const void* q, const void* kv_pool, int64_t pool_slots, const int32_t* kv_indptr,
                    const int32_t* kv_indices, const int32_t* qo_indptr, const uint64_t* draft_mask,
                    const int32_t* parent, const int32_t* kv_indptr_host, const int32_t* qo_indptr_host, int batch,
                    int num_heads, float sm_scale, int splits, void* out, float* lse, void* workspace,
                    size_t workspace_bytes, void* stream) {
  return run_verify(VMLA_KERNEL_TC, q, kv_pool, pool_slots, 0.f, kv_indptr, kv_indices, nullptr, qo_indptr,
             draft_mask, parent, kv_indptr_host, qo_indptr_host, batch, num_heads, sm_scale, splits, out, lse,
             workspace, workspace_bytes, stream);
}

int verify_attn_mla_fp8(const void* q, const void* kv_pool_e4m3, int64_t pool_slots, float kv_scale,
                        const int32_t* kv_indptr, const int32_t* kv_indices, const int32_t* qo_indptr,
                        const uint64_t* draft_mask, const int32_t* parent, const int32_t* kv_indptr_host,
                        const int32_t* qo_indptr_host, int batch, int num_heads, float sm_scale, int splits, void* out,
                        float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (!(kv_scale > 0.f) || !(kv_scale < INFINITY)) return VMLA_ERR_SHAPE;
  return run_verify(VMLA_KERNEL_TC, q, kv_pool_e4m3, pool_slots, kv_scale, kv_indptr, kv_indices, nullptr, qo_indptr,
                    draft_mask, parent, kv_indptr_host, qo_indptr_host, batch, num_heads, sm_scale, splits, out, lse,
                    workspace, workspace_bytes, stream);
}

int verify_attn_mla_runs(const void* q, const void* kv_pool, int64_t pool_slots, const int32_t* kv_indptr,
                         const int32_t* run_base, const int32_t* qo_indptr, const uint64_t* draft_mask,
                         const int32_t* parent, const int32_t* kv_indptr_host, const int32_t* qo_indptr_host,
                         int batch, int num_heads, float sm_scale, int splits, void* out, float* lse,
                         void* workspace, size_t workspace_bytes, void* stream) {
  if (batch > 0 && !run_base) return VMLA_ERR_NULL;
  static const int32_t kNone = 0;  // any non-null pointer selects the runs mode when batch is 0
  return run_verify(VMLA_KERNEL_TC, q, kv_pool, pool_slots, 0.f, kv_indptr, nullptr, run_base ? run_base : &kNone,
                    qo_indptr, draft_mask, parent, kv_indptr_host, qo_indptr_host, batch, num_heads, sm_scale, splits,
                    out, lse, workspace, workspace_bytes, stream);
}

int verify_attn_mla_runs_workspace_size(int batch, int num_heads, const int32_t* qo_indptr_host,
                                        const int32_t* kv_indptr_host, int splits, size_t* bytes) {
  if (!bytes) return VMLA_ERR_NULL;
  int rc = check_common(kv_indptr_host, qo_indptr_host, batch, num_heads, 0, splits);
  if (rc != VMLA_OK) return rc;
  int sms = 0, clusters = 0;
  rc = current_sm_count(&sms, false);
  if (rc != VMLA_OK) return rc;
  rc = vmla::tc_max_clusters(&clusters);
  if (rc != VMLA_OK) return rc;
  static thread_local PlanParams plan;
  vmla_plan_info info;
  rc = build_plan(VMLA_KERNEL_TC, batch, num_heads, qo_indptr_host, kv_indptr_host, splits, sms, clusters, &plan,
                  &info);
  if (rc != VMLA_OK) return rc;
  *bytes = workspace_layout(qo_indptr_host[batch], info.partial_rows, 0).total;
  return VMLA_OK;
}

namespace {
int defrag_impl(const void* src_pool, int64_t src_slots, const int32_t* kv_indptr, const int32_t* kv_indices,
                const int32_t* kv_indptr_host, int batch, void* dst_pool, int64_t dst_slots, const int32_t* run_base,
                const int32_t* first_row, int64_t max_new, uint32_t* status_word, void* stream) {
  if (!kv_indptr_host) return VMLA_ERR_NULL;
  if (batch < 0 || batch > VMLA_MAX_BATCH || src_slots < 0 || src_slots > INT32_MAX || dst_slots < 0 ||
      dst_slots > INT32_MAX || kv_indptr_host[0] != 0)
    return VMLA_ERR_SHAPE;
  for (int b = 0; b < batch; ++b)
    if (kv_indptr_host[b + 1] < kv_indptr_host[b]) return VMLA_ERR_SHAPE;
  const int64_t total_kv = batch > 0 ? kv_indptr_host[batch] : 0;
  // nothing to copy; an append with a bound launches anyway (batch > 0), so that a captured
  // launch serves later replays whose runs are not empty
  if (total_kv == 0 && !(max_new > 0 && batch > 0)) return VMLA_OK;
  if (!src_pool || !dst_pool || !kv_indptr || !kv_indices || !run_base) return VMLA_ERR_NULL;
  if (!aligned(src_pool, 16) || !aligned(dst_pool, 16) || !aligned(status_word, 4) || !aligned(run_base, 4) ||
      !aligned(first_row, 4))
    return VMLA_ERR_ALIGN;
  int sms = 0;
  int rc = current_sm_count(&sms, true);
  if (rc != VMLA_OK) return rc;
  return launch_defrag(static_cast<const uint16_t*>(src_pool), src_slots, kv_indptr, kv_indices, kv_indptr_host,
                       batch, total_kv, static_cast<uint16_t*>(dst_pool), dst_slots, run_base, false, status_word,
                       stream, first_row, max_new);
}
}  // namespace

int verify_attn_mla_defrag(const void* src_pool, int64_t src_slots, const int32_t* kv_indptr,
                           const int32_t* kv_indices, const int32_t* kv_indptr_host, int batch, void* dst_pool,
                           int64_t dst_slots, const int32_t* run_base, uint32_t* status_word, void* stream) {
  return defrag_impl(src_pool, src_slots, kv_indptr, kv_indices, kv_indptr_host, batch, dst_pool, dst_slots,
                     run_base, nullptr, 0, status_word, stream);
}

int verify_attn_mla_defrag_append(const void* src_pool, int64_t src_slots, const int32_t* kv_indptr,
                                  const int32_t* kv_indices, const int32_t* kv_indptr_host, int batch,
                                  void* dst_pool, int64_t dst_slots, const int32_t* run_base,
                                  const int32_t* first_row, int64_t max_new_rows, uint32_t* status_word,
                                  void* stream) {
  if (batch > 0 && kv_indptr_host && (kv_indptr_host[batch] > 0 || max_new_rows > 0) && !first_row)
    return VMLA_ERR_NULL;
  if (max_new_rows < 0) return VMLA_ERR_SHAPE;
  return defrag_impl(src_pool, src_slots, kv_indptr, kv_indices, kv_indptr_host, batch, dst_pool, dst_slots,
                     run_base, first_row, max_new_rows, status_word, stream);
}

int verify_attn_mla_simt(const void* q, const void* kv_pool, int64_t pool_slots, const int32_t* kv_indptr,
                         const int32_t* kv_indices, const int32_t* qo_indptr, const uint64_t* draft_mask,
                         const int32_t* parent, const int32_t* kv_indptr_host, const int32_t* qo_indptr_host,
                         int batch, int num_heads, float sm_scale, int splits, void* out, float* lse,
                         void* workspace, size_t workspace_bytes, void* stream) {
  return run_verify(VMLA_KERNEL_SIMT, q, kv_pool, pool_slots, 0.f, kv_indptr, kv_indices, nullptr, qo_indptr, draft_mask,
             parent,
             kv_indptr_host, qo_indptr_host, batch, num_heads, sm_scale, splits, out, lse, workspace,
             workspace_bytes, stream);
}

int verify_attn_mla_merge(const float* o_parts, const float* lse_parts, int num_splits, int64_t rows, void* out,
                          float* lse, void* stream) {
  if (num_splits < 1 || num_splits > 64 || rows < 0 || rows > (INT32_MAX / 64)) return VMLA_ERR_SHAPE;
  if (rows == 0) return VMLA_OK;
  if (!o_parts || !lse_parts || !out || !lse) return VMLA_ERR_NULL;
  if (!aligned(o_parts, 16) || !aligned(out, 16) || !aligned(lse_parts, 4) || !aligned(lse, 4))
    return VMLA_ERR_ALIGN;
  int sms = 0;
  int rc = current_sm_count(&sms, true);
  if (rc != VMLA_OK) return rc;
  // one "sequence" whose rows are the given rows, split num_splits ways
  static thread_local PlanParams plan;
  std::memset(&plan, 0, sizeof plan);
  plan.batch = 1;
  plan.num_heads = 1;
  plan.merge_rows = (int32_t)rows;
  plan.seq[0].n_q = (int32_t)rows;
  plan.seq[0].n_split = num_splits;
  plan.seq[0].part_off = 0;
  plan.seq[0].merge_off = 0;
  plan.seq[0].q_off = 0;
  return launch_merge(plan, o_parts, lse_parts, 0, static_cast<uint16_t*>(out), lse, stream);
}

int verify_attn_mla_tree_mask(const int32_t* parent, const int32_t* qo_indptr, int batch, int total_q,
                              uint64_t* mask_out, uint32_t* status_word, void* stream) {
  if (batch < 0 || batch > VMLA_MAX_BATCH || total_q < 0) return VMLA_ERR_SHAPE;
  if (total_q == 0) return VMLA_OK;
  if (!parent || !qo_indptr || !mask_out) return VMLA_ERR_NULL;
  if (!aligned(mask_out, 8)) return VMLA_ERR_ALIGN;
  int sms = 0;
  int rc = current_sm_count(&sms, true);
  if (rc != VMLA_OK) return rc;
  return launch_tree_mask(parent, qo_indptr, batch, total_q, mask_out, status_word, stream);
}

int verify_attn_mla_check(const void* workspace, void* stream) {
  if (!workspace) return VMLA_ERR_NULL;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return VMLA_ERR_CUDA;
  uint32_t word[2] = {0, 0};
  if (cudaMemcpy(word, workspace, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return VMLA_ERR_CUDA;
  return (int)(int32_t)word[0];
}

namespace {
// Side stream, events and a pinned status slot of the host-buffer entry point,
// one set per thread and device.
struct HostSide {
  cudaStream_t side = nullptr;
  cudaEvent_t start = nullptr, q_done = nullptr;
  uint32_t* status = nullptr;  // pinned host copy of the workspace status words
};
int host_side(HostSide** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return VMLA_ERR_DEVICE;
  thread_local HostSide sides[64];
  HostSide& h = sides[dev];
  if (!h.side) {
    if (cudaStreamCreateWithFlags(&h.side, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&h.start, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&h.q_done, cudaEventDisableTiming) != cudaSuccess ||
        cudaMallocHost(reinterpret_cast<void**>(&h.status), 2 * sizeof(uint32_t)) != cudaSuccess) {
      h = HostSide();
      return VMLA_ERR_CUDA;
    }
  }
  *out = &h;
  return VMLA_OK;
}
}  // namespace

namespace {
// The host-buffer call's device buffer: q, the index arrays, the optional mask
// and parent arrays, out and lse, then the workspace (ws bytes), so that the
// inputs' places do not depend on the plan.
size_t host_buffer_bytes(size_t ws, const int32_t* qo_indptr_host, const int32_t* kv_indptr_host, int batch,
                         int num_heads, bool has_mask, bool has_parent) {
  auto up = [](size_t x) { return (x + VMLA_WORKSPACE_ALIGN - 1) / VMLA_WORKSPACE_ALIGN * VMLA_WORKSPACE_ALIGN; };
  const size_t T = (size_t)qo_indptr_host[batch], N = (size_t)kv_indptr_host[batch], B = (size_t)batch;
  size_t total = up(ws);
  total += up(T * num_heads * VMLA_D_QK * 2);  // q
  total += 2 * up((B + 1) * 4);                // indptr arrays
  total += up(N * 4);                          // kv_indices
  if (has_mask) total += up(T * 8);
  if (has_parent) total += up(T * 4);
  total += up(T * num_heads * VMLA_D_V * 2);   // out
  total += up(T * num_heads * 4);              // lse
  return total;
}
}  // namespace

int verify_attn_mla_host_buffer_size(int batch, int num_heads, const int32_t* qo_indptr_host,
                                     const int32_t* kv_indptr_host, int splits, int has_mask, int has_parent,
                                     size_t* bytes) {
  if (!bytes) return VMLA_ERR_NULL;
  int rc = check_common(kv_indptr_host, qo_indptr_host, batch, num_heads, 0, splits);
  if (rc != VMLA_OK) return rc;
  size_t ws = 0;
  rc = verify_attn_mla_workspace_size(batch, num_heads, qo_indptr_host, kv_indptr_host, splits, &ws);
  if (rc != VMLA_OK) return rc;
  *bytes = host_buffer_bytes(ws, qo_indptr_host, kv_indptr_host, batch, num_heads, has_mask != 0, has_parent != 0);
  return VMLA_OK;
}

int verify_attn_mla_host(const void* q_host, const void* kv_pool, int64_t pool_slots, const int32_t* kv_indptr_host,
                         const int32_t* kv_indices_host, const int32_t* qo_indptr_host,
                         const uint64_t* draft_mask_host, const int32_t* parent_host, int batch, int num_heads,
                         float sm_scale, int splits, void* out_host, float* lse_host, void* device_buffer,
                         size_t device_buffer_bytes, void* stream) {
  int rc = check_common(kv_indptr_host, qo_indptr_host, batch, num_heads, pool_slots, splits);
  if (rc != VMLA_OK) return rc;
  if (!device_buffer) return VMLA_ERR_NULL;
  if (!aligned(device_buffer, VMLA_WORKSPACE_ALIGN)) return VMLA_ERR_ALIGN;
  const size_t T = (size_t)qo_indptr_host[batch], N = (size_t)kv_indptr_host[batch], B = (size_t)batch;
  if (T > 0 && (!q_host || !kv_indices_host || !out_host || !lse_host || !kv_pool)) return VMLA_ERR_NULL;
  auto up = [](size_t x) { return (x + VMLA_WORKSPACE_ALIGN - 1) / VMLA_WORKSPACE_ALIGN * VMLA_WORKSPACE_ALIGN; };
  char* p = static_cast<char*>(device_buffer);
  char* d_q = p;             p += up(T * num_heads * VMLA_D_QK * 2);
  char* d_kvp = p;           p += up((B + 1) * 4);
  char* d_qop = p;           p += up((B + 1) * 4);
  char* d_kvi = p;           p += up(N * 4);
  char* d_mask = nullptr;
  if (draft_mask_host) { d_mask = p; p += up(T * 8); }
  char* d_par = nullptr;
  if (parent_host) { d_par = p; p += up(T * 4); }
  char* d_out = p;           p += up(T * num_heads * VMLA_D_V * 2);
  char* d_lse = p;           p += up(T * num_heads * 4);
  char* d_ws = p;  // the plan's workspace follows the inputs
  if (device_buffer_bytes < (size_t)(d_ws - static_cast<char*>(device_buffer))) return VMLA_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
  // q crosses on a side stream while the gather runs; only the kernels after the
  // gather read q, and they wait for its copy
  HostSide* hs = nullptr;
  if (T > 0) {
    rc = host_side(&hs);
    if (rc != VMLA_OK) return rc;
  }
  // The copies go out first; the plan is built on the host while they cross.  On staged
  // rows the kernels read no kv_indptr on the device (the plan carries the lengths) and
  // only the tree-mask kernel reads qo_indptr, so neither crosses unless needed.  Page-locked
  // indices are read by the gather itself through their mapped device address (4 bytes per
  // 2304 it moves); other host memory is copied first.
  const int32_t* kvi_dev = reinterpret_cast<const int32_t*>(d_kvi);
  bool kvi_mapped = false;
  if (T > 0 && N > 0) {
    cudaPointerAttributes pa;
    if (cudaPointerGetAttributes(&pa, kv_indices_host) == cudaSuccess && pa.type == cudaMemoryTypeHost &&
        pa.devicePointer) {
      kvi_dev = static_cast<const int32_t*>(pa.devicePointer);
      kvi_mapped = true;
    } else {
      cudaGetLastError();  // an unregistered pointer leaves an error to clear
    }
  }
  bool ok = true;
  if (d_par) ok = ok && cudaMemcpyAsync(d_qop, qo_indptr_host, (B + 1) * 4, h2d, st) == cudaSuccess;
  if (T > 0) {
    if (!kvi_mapped) ok = ok && cudaMemcpyAsync(d_kvi, kv_indices_host, N * 4, h2d, st) == cudaSuccess;
    if (d_mask) ok = ok && cudaMemcpyAsync(d_mask, draft_mask_host, T * 8, h2d, st) == cudaSuccess;
    if (d_par) ok = ok && cudaMemcpyAsync(d_par, parent_host, T * 4, h2d, st) == cudaSuccess;
  }
  if (hs) {
    // starts once the copies above have crossed, so that it shares the link with no other copy
    ok = ok && cudaEventRecord(hs->start, st) == cudaSuccess;
    ok = ok && cudaStreamWaitEvent(hs->side, hs->start, 0) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(d_q, q_host, T * num_heads * VMLA_D_QK * 2, h2d, hs->side) == cudaSuccess;
    ok = ok && cudaEventRecord(hs->q_done, hs->side) == cudaSuccess;
  }
  // the call queues its gather, then builds the plan on the host while the rows move
  // (the buffer's workspace part is checked against the plan there)
  if (ok)
    // (d_kvp is the kv_indptr slot of the buffer, left unfilled: nothing on this path reads it)
    rc = run_verify(VMLA_KERNEL_TC, d_q, kv_pool, pool_slots, 0.f, (const int32_t*)d_kvp, kvi_dev, nullptr,
                    (const int32_t*)d_qop, (const uint64_t*)d_mask, (const int32_t*)d_par, kv_indptr_host,
                    qo_indptr_host, batch, num_heads, sm_scale, splits, d_out, (float*)d_lse, d_ws,
                    device_buffer_bytes - (size_t)(d_ws - static_cast<char*>(device_buffer)), stream,
                    hs ? (void*)hs->q_done : nullptr);
  if (!ok || rc != VMLA_OK) {
    // the buffer is the caller's again when this returns: the copies already issued are waited for
    if (hs) cudaStreamSynchronize(hs->side);
    cudaStreamSynchronize(st);
    return ok ? rc : VMLA_ERR_CUDA;
  }
  if (!hs) return verify_attn_mla_check(d_ws, stream);  // nothing to compute
  // out, lse and the status words come back in stream order, then one synchronisation
  ok = ok && cudaMemcpyAsync(out_host, d_out, T * num_heads * VMLA_D_V * 2, d2h, st) == cudaSuccess;
  ok = ok && cudaMemcpyAsync(lse_host, d_lse, T * num_heads * 4, d2h, st) == cudaSuccess;
  ok = ok && cudaMemcpyAsync(hs->status, d_ws, 2 * sizeof(uint32_t), d2h, st) == cudaSuccess;
  ok = ok && cudaStreamSynchronize(st) == cudaSuccess;
  if (!ok) return VMLA_ERR_CUDA;
  return (int)(int32_t)hs->status[0];
}

namespace {
// Bounds of a device-planned call (host values only).
int check_dplan_bounds(int batch, int num_heads, int64_t max_total_q, int64_t max_total_kv, int splits) {
  if (batch < 0 || batch > VMLA_MAX_BATCH || num_heads < 1 || num_heads > VMLA_MAX_HEADS) return VMLA_ERR_SHAPE;
  if (splits < VMLA_SPLITS_LANES || splits > 64) return VMLA_ERR_SHAPE;
  if (max_total_q < 0 || max_total_q > (int64_t)batch * VMLA_MAX_DRAFT) return VMLA_ERR_SHAPE;
  if (max_total_kv < 0 || max_total_kv > INT32_MAX) return VMLA_ERR_SHAPE;
  return VMLA_OK;
}

int dplan_clusters(int* clusters) {
  int rc = tc_max_clusters(clusters);
  if (rc == VMLA_OK && *clusters > kMaxClusters) *clusters = kMaxClusters;
  return rc;
}
}  // namespace

namespace {
// Device-planned call on staged rows (kv_indices given, run_base NULL: the gather runs)
// or on pool runs (run_base given: no gather, a run check instead).
int device_plan_impl(const void* q, const void* kv_pool, int64_t pool_slots, const int32_t* kv_indptr,
                     const int32_t* kv_indices, const int32_t* run_base, const int32_t* qo_indptr,
                     const uint64_t* draft_mask, const int32_t* parent, int batch, int num_heads, int64_t max_total_q,
                     int64_t max_total_kv, float sm_scale, int splits, void* out, float* lse, void* workspace,
                     size_t workspace_bytes, void* stream) {
  const bool runs = run_base != nullptr;
  int rc = check_dplan_bounds(batch, num_heads, max_total_q, max_total_kv, splits);
  if (rc != VMLA_OK) return rc;
  if (pool_slots < 0 || pool_slots > INT32_MAX) return VMLA_ERR_SHAPE;
  if (!(sm_scale > 0.f) || !(sm_scale < INFINITY)) return VMLA_ERR_SHAPE;
  if (!workspace) return VMLA_ERR_NULL;
  if (batch > 0 && (!kv_indptr || !qo_indptr)) return VMLA_ERR_NULL;
  if (max_total_q > 0 && (!q || !kv_pool || (!runs && !kv_indices) || !out || !lse)) return VMLA_ERR_NULL;
  if (max_total_kv > 0 && pool_slots == 0) return VMLA_ERR_SHAPE;
  if (!aligned(q, 16) || !aligned(kv_pool, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
      !aligned(workspace, VMLA_WORKSPACE_ALIGN) || !aligned(draft_mask, 8) || !aligned(parent, 4) ||
      !aligned(run_base, 4))
    return VMLA_ERR_ALIGN;
  int sms = 0, clusters = 0;
  rc = current_sm_count(&sms, true);
  if (rc != VMLA_OK) return rc;
  rc = dplan_clusters(&clusters);
  if (rc != VMLA_OK) return rc;
  const DplanLayout L = dplan_layout(batch, num_heads, max_total_q, max_total_kv, splits, clusters, !runs);
  if (workspace_bytes < L.total) return VMLA_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws + L.status_off);
  PlanParams* plan = reinterpret_cast<PlanParams*>(ws + L.plan_off);
  TcSched* sched = reinterpret_cast<TcSched*>(ws + L.sched_off);
  cudaStream_t st = (cudaStream_t)stream;
  // status words 0-3 and the planner's block counter (word 4)
  if (cudaMemsetAsync(status, 0, 32, st) != cudaSuccess) return VMLA_ERR_CUDA;
  if (batch == 0 || max_total_q == 0) return VMLA_OK;
  rc = launch_device_plan(qo_indptr, kv_indptr, batch, num_heads, splits, clusters, max_total_q, max_total_kv,
                          L.part_cap, plan, sched, status, stream);
  if (rc != VMLA_OK) return rc;
  const uint64_t* masks = draft_mask;
  uint64_t* tree_masks = !masks && parent ? reinterpret_cast<uint64_t*>(ws + L.masks_off) : nullptr;
  if (tree_masks) masks = tree_masks;
  RunArgs a;
  test_fault_settings(&a.test_fault, &a.wait_cycles);
  a.q = static_cast<const uint16_t*>(q);
  a.kv = static_cast<const uint16_t*>(kv_pool);
  a.pool_slots = pool_slots;
  a.kv_indices = kv_indices;
  a.masks = masks;
  a.sm_scale = sm_scale;
  a.scale_log2 = sm_scale * 1.4426950408889634f;
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.out_rows = max_total_q * num_heads;
  a.part_rows = L.part_cap;
  a.part_o = reinterpret_cast<float*>(ws + L.part_o_off);
  a.part_lse = reinterpret_cast<float*>(ws + L.part_lse_off);
  // rows: the staged copy (its capacity; the gather stages kv_indptr[batch] of them) or the pool's runs
  a.staged = runs ? const_cast<uint16_t*>(static_cast<const uint16_t*>(kv_pool))
                  : reinterpret_cast<uint16_t*>(ws + L.staged_off);
  a.total_kv = runs ? pool_slots : max_total_kv;
  a.run_base = run_base;
  a.kv_scale = 0.f;
  a.status = status;
  // In stream order: the planner; the gather, started beside it (it reads no plan; it
  // waits for the planner before it completes); the tree masks (they
  // need the planner's count); the verify kernel, which reads the plan only once all of
  // that is complete; the merge.  On pool runs the check of the runs takes the gather's place
  // (also started beside the planner, and waiting for it before it completes).
  if (runs) {
    // the runs must lie in the pool (a run outside it is reported; its keys read the tile loads' zero fill)
    rc = launch_defrag(nullptr, 0, kv_indptr, nullptr, nullptr, batch, 0, nullptr, pool_slots, run_base, true, status,
                       stream, nullptr, 0, true);
  } else {
    rc = launch_gather_dplan(a, kv_indptr + batch, stream);
  }
  if (rc != VMLA_OK) return rc;
  if (tree_masks) {
    rc = launch_tree_mask_dplan(parent, qo_indptr, batch, max_total_q, status + 3, tree_masks, status, stream);
    if (rc != VMLA_OK) return rc;
  }
  rc = launch_tc_dplan(plan, sched, clusters, a, stream);
  if (rc != VMLA_OK) return rc;
  return launch_merge_dplan(plan, max_total_q * num_heads, a.part_o, a.part_lse, a.out, a.lse, stream);
}

int device_plan_workspace(int batch, int num_heads, int64_t max_total_q, int64_t max_total_kv, int splits, bool staged,
                          size_t* bytes) {
  if (!bytes) return VMLA_ERR_NULL;
  int rc = check_dplan_bounds(batch, num_heads, max_total_q, max_total_kv, splits);
  if (rc != VMLA_OK) return rc;
  int sms = 0, clusters = 0;
  rc = current_sm_count(&sms, true);
  if (rc != VMLA_OK) return rc;
  rc = dplan_clusters(&clusters);
  if (rc != VMLA_OK) return rc;
  *bytes = dplan_layout(batch, num_heads, max_total_q, max_total_kv, splits, clusters, staged).total;
  return VMLA_OK;
}
}  // namespace

int verify_attn_mla_device_plan_workspace_size(int batch, int num_heads, int64_t max_total_q, int64_t max_total_kv,
                                               int splits, size_t* bytes) {
  return device_plan_workspace(batch, num_heads, max_total_q, max_total_kv, splits, true, bytes);
}

int verify_attn_mla_device_plan(const void* q, const void* kv_pool, int64_t pool_slots, const int32_t* kv_indptr,
                                const int32_t* kv_indices, const int32_t* qo_indptr, const uint64_t* draft_mask,
                                const int32_t* parent, int batch, int num_heads, int64_t max_total_q,
                                int64_t max_total_kv, float sm_scale, int splits, void* out, float* lse,
                                void* workspace, size_t workspace_bytes, void* stream) {
  return device_plan_impl(q, kv_pool, pool_slots, kv_indptr, kv_indices, nullptr, qo_indptr, draft_mask, parent, batch,
                          num_heads, max_total_q, max_total_kv, sm_scale, splits, out, lse, workspace,
                          workspace_bytes, stream);
}

int verify_attn_mla_runs_device_plan_workspace_size(int batch, int num_heads, int64_t max_total_q,
                                                    int64_t max_total_kv, int splits, size_t* bytes) {
  return device_plan_workspace(batch, num_heads, max_total_q, max_total_kv, splits, false, bytes);
}

int verify_attn_mla_runs_device_plan(const void* q, const void* kv_pool, int64_t pool_slots, const int32_t* kv_indptr,
                                     const int32_t* run_base, const int32_t* qo_indptr, const uint64_t* draft_mask,
                                     const int32_t* parent, int batch, int num_heads, int64_t max_total_q,
                                     int64_t max_total_kv, float sm_scale, int splits, void* out, float* lse,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  if (batch > 0 && !run_base) return VMLA_ERR_NULL;
  static const int32_t kNone = 0;  // any non-null pointer selects the runs mode when batch is 0
  return device_plan_impl(q, kv_pool, pool_slots, kv_indptr, nullptr, run_base ? run_base : &kNone, qo_indptr,
                          draft_mask, parent, batch, num_heads, max_total_q, max_total_kv, sm_scale, splits, out, lse,
                          workspace, workspace_bytes, stream);
}

int verify_attn_mla_tree_accept(const int32_t* qo_indptr, const int32_t* parent, const int32_t* draft_token,
                                const int32_t* target_token, const int32_t* root_token, int batch, int total_q,
                                int32_t* accept_len, int32_t* accept_path, int32_t* next_token, uint32_t* status_word,
                                void* stream) {
  if (batch < 0 || batch > VMLA_MAX_BATCH || total_q < 0 || total_q > batch * VMLA_MAX_DRAFT) return VMLA_ERR_SHAPE;
  if (batch == 0) return VMLA_OK;
  if (!qo_indptr || !root_token || !accept_len || !next_token) return VMLA_ERR_NULL;
  if (total_q > 0 && (!draft_token || !target_token || !accept_path)) return VMLA_ERR_NULL;
  if (!aligned(qo_indptr, 4) || !aligned(parent, 4) || !aligned(draft_token, 4) || !aligned(target_token, 4) ||
      !aligned(root_token, 4) || !aligned(accept_len, 4) || !aligned(accept_path, 4) || !aligned(next_token, 4) ||
      !aligned(status_word, 4))
    return VMLA_ERR_ALIGN;
  int sms = 0;
  int rc = current_sm_count(&sms, true);
  if (rc != VMLA_OK) return rc;
  return launch_tree_accept(qo_indptr, parent, draft_token, target_token, root_token, batch, total_q, accept_len,
                            accept_path, next_token, status_word, stream);
}

int verify_attn_mla_test_fault(int fault, int64_t wait_cycles) {
  if ((fault != 0 && fault != kFaultNoQReady) || wait_cycles < 0) return VMLA_ERR_SHAPE;
  g_test_fault = fault;
  g_test_wait_cycles = wait_cycles;
  return VMLA_OK;
}

int verify_attn_mla_timing_enable(int capacity) {
  std::lock_guard<std::mutex> g(g_timing.mu);
  for (cudaEvent_t e : g_timing.ev) cudaEventDestroy(e);
  g_timing.ev.clear();
  g_timing.merged.clear();
  g_timing.cap = 0;
  g_timing.n = 0;
  if (capacity <= 0) return VMLA_OK;
  if (capacity > (1 << 20)) return VMLA_ERR_SHAPE;
  g_timing.ev.resize((size_t)capacity * 6);
  g_timing.merged.assign((size_t)capacity, 0);
  for (auto& e : g_timing.ev)
    if (cudaEventCreate(&e) != cudaSuccess) {
      e = nullptr;
      return VMLA_ERR_CUDA;
    }
  g_timing.cap = capacity;
  return VMLA_OK;
}

int verify_attn_mla_timing_read(float* gather_ms, float* verify_ms, float* merge_ms, int capacity, int* count) {
  if (!gather_ms || !verify_ms || !merge_ms || !count) return VMLA_ERR_NULL;
  std::lock_guard<std::mutex> g(g_timing.mu);
  int n = g_timing.n < capacity ? g_timing.n : capacity;
  auto elapsed = [](float* out, int call, int k0, int k1) {
    if (cudaEventSynchronize(timing_event(call, k1)) != cudaSuccess) return false;
    return cudaEventElapsedTime(out, timing_event(call, k0), timing_event(call, k1)) == cudaSuccess;
  };
  for (int i = 0; i < n; ++i) {
    merge_ms[i] = 0.f;
    gather_ms[i] = 0.f;
    verify_ms[i] = 0.f;
    if (g_timing.merged[i] == kTimingFailed) continue;  // a failed call: zeros
    if (!elapsed(&verify_ms[i], i, 0, 1)) return VMLA_ERR_CUDA;
    if ((g_timing.merged[i] & 1) && !elapsed(&merge_ms[i], i, 2, 3)) return VMLA_ERR_CUDA;
    if ((g_timing.merged[i] & 2) && !elapsed(&gather_ms[i], i, 4, 5)) return VMLA_ERR_CUDA;
  }
  *count = n;
  g_timing.n = 0;
  return VMLA_OK;
}

const char* verify_attn_mla_status_string(int status) {
  switch (status) {
    case VMLA_OK: return "ok";
    case VMLA_ERR_NULL: return "a required pointer is NULL";
    case VMLA_ERR_SHAPE: return "sizes out of range or inconsistent indptr arrays";
    case VMLA_ERR_ALIGN: return "a pointer misses its required alignment";
    case VMLA_ERR_WORKSPACE: return "workspace too small";
    case VMLA_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case VMLA_ERR_TIMEOUT: return "a kernel's bounded wait expired";
    case VMLA_ERR_INDEX: return "a kv slot index was outside the pool";
    case VMLA_ERR_DEVICE: return "no usable sm_103 device";
    case VMLA_ERR_PARENT: return "a draft parent index was malformed";
    default: return "unknown status";
  }
}

int verify_attn_mla_version(void) { return 100; }

}  // extern "C"
