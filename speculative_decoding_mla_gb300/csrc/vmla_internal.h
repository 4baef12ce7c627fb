// Internal declarations shared by the library's translation units (host and device).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "verify_attn_mla.h"

namespace vmla {

constexpr int kDqk = VMLA_D_QK;
constexpr int kDv = VMLA_D_V;
constexpr int kRowBytes = kDqk * 2;  // 1152 bytes per latent KV row / per query head

// Per-sequence entry of a split plan (passed to the kernels by value).
//
// Two forms.  Uniform plan (lane_width 0): sequence b's keys are cut into
// n_split pieces of `chunk` keys, and each (piece, row block) is a work unit
// that the cluster schedule deals out.  Lane plan (tensor-core kernel,
// lane_width G > 0): the clusters form lanes of G; each sequence's row blocks
// form n_rb / G streams of G row blocks over all its key tiles, laid end to
// end in a cost space (a stream spans its tiles plus kLaneStreamTiles); lane l
// takes the cost interval [l L, (l + 1) L) of every stream it meets, and
// cluster j of the lane takes row block g G + j of stream g.  A stream's pieces
// are the lanes it meets (vmla_plan_core.h).
struct SeqPlan {
  int32_t kv_off;      // kv_indptr[b]
  int32_t n_kv;        // N_b keys (prefix + drafts)
  int32_t q_off;       // qo_indptr[b]
  int32_t n_q;         // Q_b drafts
  int32_t unit_start;  // first work unit (uniform plan) or first stream (lane plan) of this sequence
  int32_t n_rb;        // row blocks (rows r = i*H + h, in blocks of rows_per_unit)
  int32_t n_split;     // key-range pieces (lane plan: the most of any of its streams)
  int32_t chunk;       // keys per piece (piece s covers [s*chunk, min(N_b, (s+1)*chunk))); uniform plan
  int32_t part_off;    // first partial row of this sequence (partial row = part_off + s*R_b + r)
  int32_t merge_off;   // first merge row (monotone over b; only split sequences own merge rows)
  int32_t lane_cost;   // lane plan: cost-space position of its first stream (monotone over b)
};

struct PlanParams {
  int32_t batch;
  int32_t num_heads;
  int32_t total_units;
  int32_t merge_rows;
  int32_t rows_per_unit;
  int32_t max_splits;
  int32_t partial_rows;
  int32_t lane_width;  // G of a lane plan, 0 for a uniform plan
  int32_t lane_tiles;  // L: cost-space length each lane takes
  int32_t lane_total;  // W: cost-space length of all streams
  int32_t lane_count;  // lanes with work (the launch has lane_count x G clusters)
  int32_t pad;
  SeqPlan seq[VMLA_MAX_BATCH];
};

// Work order of one tensor-core launch: cluster c processes the units
// order[start[c] .. start[c+1]) in that order (longest-first greedy balance).
// A plan with more units is run as several launches of at most kMaxTcUnits.
constexpr int kMaxTcUnits = 3072;
constexpr int kMaxClusters = 128;
struct TcSched {
  int32_t num_clusters;
  int32_t total_units;  // units of this launch
  int32_t unit_base;    // plan unit of order value 0
  int32_t pad;
  uint16_t start[kMaxClusters + 1];
  uint16_t order[kMaxTcUnits];  // plan unit = unit_base + order[k]
};

// Builds the per-cluster unit lists for the plan's units [unit_begin, unit_end)
// (at most kMaxTcUnits of them; host).  Returns a vmla_status.
int build_tc_schedule(const PlanParams& plan, int num_clusters, int unit_begin, int unit_end, TcSched* sched);

// Planner knobs of one kernel family.
struct PlanShape {
  int rows_per_unit;   // query rows one unit covers
  int units_per_sm;    // concurrent units per SM (fractional pairs expressed by the caller)
  int key_align;       // piece boundaries are multiples of this many keys
  int min_chunk;       // smallest piece the planner chooses on its own
  int max_splits;
};

// plan_shape(kernel): vmla_plan_core.h (host and device)

// Host planner: fills `pp` and `info`.  Returns a vmla_status.  For the
// tensor-core kernel the units fill `tc_clusters` four-SM clusters (the
// device's co-resident cluster count); tc_clusters <= 0 estimates it as
// num_sms / 4.
int build_plan(int kernel, int batch, int num_heads, const int32_t* qo_indptr_host,
               const int32_t* kv_indptr_host, int splits, int num_sms, int tc_clusters, PlanParams* pp,
               vmla_plan_info* info);

// Clusters of the tensor-core kernel that are co-resident on the current device.
int tc_max_clusters(int* out);

// Workspace layout (offsets in bytes from the workspace base, each 256 B aligned).
// The areas that do not depend on the plan come first, so that the kernels that
// fill them can be queued before the plan is built.
struct WorkspaceLayout {
  size_t status_off;  // uint32 status, uint32 info, 2 spare words
  size_t masks_off;   // uint64 [T_q] ancestor masks
  size_t staged_off;  // bf16 [staged_rows, 576]: every sequence's KV rows, contiguous (tensor-core kernel)
  size_t part_o_off;  // float [partial_rows, 512]
  size_t part_lse_off;// float [partial_rows]   (log2 domain)
  size_t total;
};
WorkspaceLayout workspace_layout(int64_t total_q, int64_t partial_rows, int64_t staged_rows);

// Bounded waits of the tensor-core kernel: about a second at 2 GHz, or the
// failure test's budget.
constexpr long long kWaitCyclesDefault = 2000000000LL;
// Failure test: the softmax warps never report Q ready, so a bounded wait expires.
constexpr int32_t kFaultNoQReady = 1;
// Failure-test settings for the calls that follow on this thread (verify_attn_mla_test_fault).
void test_fault_settings(int32_t* fault, long long* wait_cycles);

// Device-side entry points implemented in the .cu files (launch only; no sync).
struct RunArgs {
  const uint16_t* q;
  const uint16_t* kv;
  int64_t pool_slots;
  const int32_t* kv_indices;
  const uint64_t* masks;  // visibility words per query, or NULL for causal
  float scale_log2;       // sm_scale * log2(e)
  float sm_scale;
  uint16_t* out;
  float* lse;
  int64_t out_rows;         // rows of out and lse (query rows x heads, or their bound)
  int64_t part_rows;        // rows of part_o and part_lse (or their bound)
  float* part_o;
  float* part_lse;  // log2 domain
  uint16_t* staged; // contiguous copy of the gathered KV rows, [total_kv, 576] (tensor-core kernel),
                    // or the pool itself when the rows lie in runs
  int64_t total_kv; // rows of `staged`
  const int32_t* run_base;  // [batch] first pool slot of each sequence's run, or NULL (staged rows)
  long long wait_cycles;    // budget of every bounded wait in the tensor-core kernel (clock64 cycles)
  float kv_scale;           // 0: kv is bf16 [S, 576]; > 0: kv is e4m3 [S, 576] bytes, value = code * kv_scale
  int32_t test_fault;       // 0; kFaultNoQReady only in the failure test
  uint32_t* status;
};

// One verify call on a caller-provided workspace (argument checks, plan, launches).
// kv_indices NULL and run_base given: the rows of sequence b are the pool's
// slots run_base[b] .. run_base[b] + N_b - 1 (tensor-core kernel only).
// kv_scale > 0: kv_pool holds e4m3 codes; the gather dequantizes them (tensor-core kernel only).
// q_ready (a cudaEvent_t or NULL): the kernels that read q wait for it; the gather does not.
// plan_in / info_in: a plan the caller already built for these lengths with this
// device's SM and cluster counts (NULL: built here).
int run_verify(int kernel, const void* q, const void* kv_pool, int64_t pool_slots, float kv_scale,
               const int32_t* kv_indptr, const int32_t* kv_indices, const int32_t* run_base, const int32_t* qo_indptr,
               const uint64_t* draft_mask, const int32_t* parent,
               const int32_t* kv_indptr_host, const int32_t* qo_indptr_host, int batch, int num_heads,
               float sm_scale, int splits, void* out, float* lse, void* workspace, size_t workspace_bytes,
               void* stream, void* q_ready = nullptr, const PlanParams* plan_in = nullptr,
               const vmla_plan_info* info_in = nullptr);

// Device-planned calls (stream-capture safe): the plan and the cluster
// schedule are computed on the device from the device indptr arrays.  The
// workspace holds, after the status words, the plan, the schedule, and areas
// sized for upper bounds on the lengths fixed by the caller.
struct DplanLayout {
  size_t status_off;  // uint32 status, info, rows to gather, draft rows to mask; planner block counter
                      // (word 4) and candidate scores (int64 from word 8)
  size_t plan_off;    // PlanParams
  size_t sched_off;   // TcSched
  size_t masks_off;   // uint64 [max_total_q]
  size_t part_o_off;  // float [part_cap, 512]
  size_t part_lse_off;// float [part_cap]  (log2 domain)
  size_t staged_off;  // bf16 [max_total_kv, 576]
  size_t total;
  int64_t part_cap;   // partial rows the area holds
};
// staged = false: rows read from pool runs, no staging area.
DplanLayout dplan_layout(int batch, int num_heads, int64_t max_total_q, int64_t max_total_kv, int splits,
                         int clusters, bool staged = true);

// Planner kernel: reads qo_indptr / kv_indptr [batch+1] on the device, writes
// the plan and the schedule into the workspace, the gather and mask row counts
// into status words 2 and 3, and VMLA_ERR_SHAPE into the status word (with an
// empty plan) when the lengths are inconsistent or exceed the bounds.
int launch_device_plan(const int32_t* qo_indptr, const int32_t* kv_indptr, int batch, int num_heads, int splits,
                       int clusters, int64_t max_total_q, int64_t max_total_kv, int64_t part_cap,
                       PlanParams* plan, TcSched* sched, uint32_t* status, void* stream);
int launch_tc_dplan(const PlanParams* plan, const TcSched* sched, int clusters, const RunArgs& args, void* stream);
// Gather of the rows counted in *total_dev (kv_indptr[batch], clamped to [0, args.total_kv],
// the staged capacity), launched to start beside the planner kernel just queued; it waits
// for the planner before it completes.
int launch_gather_dplan(const RunArgs& args, const int32_t* total_dev, void* stream);
int launch_merge_dplan(const PlanParams* plan, int64_t max_rows, const float* part_o, const float* part_lse,
                       uint16_t* out, float* lse, void* stream);
int launch_tree_mask_dplan(const int32_t* parent, const int32_t* qo_indptr, int batch, int64_t max_total_q,
                           const uint32_t* rows_dev, uint64_t* mask_out, uint32_t* status, void* stream);

// Copies the rows of every sequence into its run of dst_pool and zeroes each
// run's tail up to a multiple of 128 rows; with check_only, records
// VMLA_ERR_INDEX for runs outside [0, dst_slots) without copying (beside_planner: the
// check starts beside the device planner kernel just queued and completes after it).
// first_row (device [batch], or NULL): rows below it are already in place and skipped.
int launch_defrag(const uint16_t* src_pool, int64_t src_slots, const int32_t* kv_indptr, const int32_t* kv_indices,
                  const int32_t* kv_indptr_host, int batch, int64_t total_kv, uint16_t* dst_pool, int64_t dst_slots,
                  const int32_t* run_base, bool check_only, uint32_t* status, void* stream,
                  const int32_t* first_row = nullptr, int64_t max_new = 0, bool beside_planner = false);

int launch_tree_accept(const int32_t* qo_indptr, const int32_t* parent, const int32_t* draft, const int32_t* target,
                       const int32_t* root, int batch, int total_q, int32_t* accept_len, int32_t* path,
                       int32_t* next_token, uint32_t* status, void* stream);

int launch_simt(const PlanParams& plan, const RunArgs& args, void* stream);
int launch_tc(const PlanParams& plan, const RunArgs& args, void* stream);
int launch_gather(const RunArgs& args, void* stream);
int launch_merge(const PlanParams& plan, const float* part_o, const float* part_lse, int lse_is_log2,
                 uint16_t* out, float* lse, void* stream);
int launch_tree_mask(const int32_t* parent, const int32_t* qo_indptr, int batch, int total_q, uint64_t* mask_out,
                     uint32_t* status, void* stream);

}  // namespace vmla
