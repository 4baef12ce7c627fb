/*
 * verify_attn_mla.h -- C ABI of the MLA speculative-decoding verify attention
 * for GB300 (sm_103a).
 *
 * The operation (the "verify attention" of "The Build That Unlocked 3-6x
 * Decode Speedup", section "The Context: A Custom Kernel for an Unsupported
 * Architecture"): every draft query of a sequence, per head, is scored against
 * that sequence's latent KV rows, masked, soft-maxed and used to weight the
 * latent rows.  The layout and the mask follow "The Build That Bridged Design
 * and Deployment", section "What This Build Achieves: The paged+bf16 Kernel":
 * bf16 rows read through a slot indirection at page_size = 1, several
 * requests per call, and a mask made of a prefix length plus a small q x q
 * visibility matrix over the draft tail.  Splitting the key range across
 * SMs and merging the partial softmaxes is the NSPLIT split-KV of "The Build
 * Script Edit", section "Context: The Long Road to a Custom sm_120 Kernel".
 *
 * Definition, for sequence b (N_b keys, Q_b drafts, prefix P_b = N_b - Q_b),
 * draft query i (token t = qo_indptr[b] + i) and head h:
 *   row_j  = kv_pool[kv_indices[kv_indptr[b] + j]]          576 bf16: [0,512) latent, [512,576) rope
 *   J      = { j < P_b } U { P_b + k : bit k of mask_i }
 *   mask_i = draft_mask[t] | ancestors-and-self from parent[] | causal bits 0..i
 *   s_j    = sm_scale * <q[t,h,0:576], row_j[0:576]>
 *   out[t,h,:] = sum_{j in J} softmax(s)_j * row_j[0:512]   (bf16, round-to-nearest-even)
 *   lse[t,h]   = ln sum_{j in J} exp(s_j)                    (fp32, natural log)
 * A query with no visible key gets out = 0 and lse = -inf.
 *
 * Conventions for every entry point:
 *   - Device pointers unless the name ends in _host.  bf16 data is passed as
 *     raw 16-bit patterns (`const void*`).  `stream` is a cudaStream_t (NULL =
 *     legacy default stream).  All device work is asynchronous on `stream`
 *     unless stated otherwise.
 *   - The caller owns every buffer.  The library keeps no pointer after a call
 *     returns and allocates no device memory in these entry points.
 *   - Errors are returned as a vmla_status (int); nothing throws.  Argument
 *     errors are detected on the host before any launch (one exception, a
 *     workspace short of the plan's partial rows, is described at
 *     verify_attn_mla).  Faults seen by a
 *     kernel (a slot index outside the pool, malformed parents, a bounded wait
 *     that ran out) are recorded in the workspace's status word and reported by
 *     verify_attn_mla_check().
 */
#ifndef VERIFY_ATTN_MLA_H
#define VERIFY_ATTN_MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define VMLA_D_QK 576     /* latent (512) + rope (64) per token and per query head */
#define VMLA_D_V 512      /* latent width; also the output width */
#define VMLA_MAX_DRAFT 64 /* draft positions per sequence (one 64-bit visibility word each) */
#define VMLA_MAX_BATCH 512
#define VMLA_MAX_HEADS 128
#define VMLA_WORKSPACE_ALIGN 256

typedef enum vmla_status {
  VMLA_OK = 0,
  VMLA_ERR_NULL = -1,      /* a required pointer is NULL */
  VMLA_ERR_SHAPE = -2,     /* sizes out of range or indptr arrays inconsistent */
  VMLA_ERR_ALIGN = -3,     /* a pointer misses its alignment (16 B for bf16 arrays, 256 B workspace) */
  VMLA_ERR_WORKSPACE = -4, /* workspace smaller than verify_attn_mla_workspace_size() */
  VMLA_ERR_CUDA = -5,      /* a CUDA runtime call or launch failed */
  VMLA_ERR_TIMEOUT = -6,   /* a kernel's bounded wait expired (kernel returned early) */
  VMLA_ERR_INDEX = -7,     /* a kv slot index was outside [0, pool_slots); that key still takes part,
                              with a row of zeros (score 0, value 0), in every kernel */
  VMLA_ERR_DEVICE = -8,    /* no usable sm_103 device for this library */
  VMLA_ERR_PARENT = -9     /* a parent index was not in [-1, i) (mask left empty) */
} vmla_status;

/* Description of the split plan a call would use (host only, no GPU needed). */
typedef struct vmla_plan_info {
  int32_t num_units;        /* work units (one CTA each; one four-CTA cluster each for the tensor-core kernel) */
  int32_t max_splits;       /* largest split count of any sequence */
  int64_t partial_rows;     /* fp32 partial (row, split) results kept in the workspace */
  int64_t merge_rows;       /* query rows whose splits the merge kernel combines */
  size_t workspace_bytes;   /* bytes verify_attn_mla needs in `workspace` */
  int32_t lane_width;       /* tensor-core kernel: 0 = equal pieces dealt to the clusters; G > 0 = the
                               lane plan (lanes of G clusters, each sequence's work cut where the
                               lanes' shares end) */
  int32_t lane_count;       /* lanes with work in a lane plan, else 0 */
} vmla_plan_info;

/* Kernel families a plan can be made for. */
#define VMLA_KERNEL_TC 0   /* tcgen05 / TMEM tensor-core kernel (what verify_attn_mla runs) */
#define VMLA_KERNEL_SIMT 1 /* plain CUDA-core kernel (verify_attn_mla_simt) */

/* `splits` value that makes the tensor-core planner take its lane plan
 * whenever the lanes fit (at most 64 of them), instead of only when it scores
 * lower; the CUDA-core kernel treats it as 0. */
#define VMLA_SPLITS_LANES (-1)

/* Split planner.  Splits each sequence's key range into contiguous pieces so
 * that the work units fill `num_sms` SMs (the NSPLIT occupancy fix of "The
 * Build That Unlocked 3-6x Decode Speedup", section "Broader Significance").
 * For the tensor-core kernel with splits = 0 the plan is made for num_sms / 4
 * clusters: either equal pieces per sequence, or (when it balances the
 * clusters better) the lane plan, whose pieces end where the lanes' shares of
 * all sequences' work end (info->lane_width > 0).
 *   qo_indptr_host, kv_indptr_host: host arrays [batch+1], starting at 0.
 *   splits: 0 = choose per sequence; k > 0 = k pieces for every sequence
 *           (capped so that no piece is empty); VMLA_SPLITS_LANES = the lane
 *           plan where it fits.
 *   splits_out: optional host array [batch] receiving each sequence's count
 *           (lane plan: the most pieces any of its row blocks has).
 * Returns VMLA_OK or VMLA_ERR_NULL / VMLA_ERR_SHAPE.  Pure host code. */
int verify_attn_mla_plan(int kernel, int batch, int num_heads, const int32_t* qo_indptr_host,
                         const int32_t* kv_indptr_host, int splits, int num_sms, vmla_plan_info* info,
                         int32_t* splits_out);

/* Workspace bytes verify_attn_mla needs for these lengths on the current
 * device (its SM count enters the plan).  Writes *bytes; returns a status. */
int verify_attn_mla_workspace_size(int batch, int num_heads, const int32_t* qo_indptr_host,
                                   const int32_t* kv_indptr_host, int splits, size_t* bytes);

/* The verify attention.  In stream order: the mask-expansion kernel when
 * `parent` is given; a gather kernel that copies every sequence's KV rows
 * (through kv_indices) into a contiguous area of the workspace, the
 * defragmentation step of "The Build That Unlocked 3-6x Decode Speedup",
 * section "The Context: A Custom Kernel for an Unsupported Architecture";
 * the tensor-core kernel; the merge kernel when a sequence is split.
 *   q           [T_q, H, 576] bf16, T_q = qo_indptr_host[batch]; 16 B aligned
 *   kv_pool     [pool_slots, 576] bf16 row-major (row stride 1152 B); 16 B aligned
 *   kv_indptr   [batch+1] int32; sequence b owns kv_indices[kv_indptr[b] .. kv_indptr[b+1])
 *   kv_indices  [kv_indptr[batch]] int32 slots; the LAST Q_b entries of each
 *               sequence are its draft tokens' rows, in draft order
 *   qo_indptr   [batch+1] int32; Q_b = qo_indptr[b+1] - qo_indptr[b] in [0, 64]
 *   draft_mask  [T_q] uint64 or NULL: bit k = query sees draft k of its sequence
 *   parent      [T_q] int32 or NULL: local parent of each draft (-1 = root;
 *               parent[i] < i).  Used only when draft_mask is NULL.  Both NULL
 *               means causal among the drafts.
 *   kv_indptr_host, qo_indptr_host: host copies of the two indptr arrays; read
 *               during the call to build the plan, not retained.
 *   sm_scale    score scale, finite and > 0 (1/sqrt(192) for the target model)
 *   splits      0 = planner's choice; k > 0 forces k pieces per sequence;
 *               VMLA_SPLITS_LANES takes the lane plan where it fits
 *   out         [T_q, H, 512] bf16 (16 B aligned);  lse [T_q, H] fp32
 *   workspace   >= verify_attn_mla_workspace_size() bytes, 256 B aligned.
 *               Holds the status word, ancestor masks, a contiguous copy of
 *               the gathered KV rows (1152 B per key) and split partials.
 *               Calls that share a workspace must be ordered on one stream.
 * The mask and gather kernels are queued before the plan is built (the host
 * plans while they run).  So a workspace large enough for the masks and rows
 * but not for the plan's partials returns VMLA_ERR_WORKSPACE with those kernels
 * queued: they write only inside the workspace, out and lse are untouched.
 * No host synchronisation and no allocation happen inside the call. */
int verify_attn_mla(const void* q, const void* kv_pool, int64_t pool_slots, const int32_t* kv_indptr,
                    const int32_t* kv_indices, const int32_t* qo_indptr, const uint64_t* draft_mask,
                    const int32_t* parent, const int32_t* kv_indptr_host, const int32_t* qo_indptr_host,
                    int batch, int num_heads, float sm_scale, int splits, void* out, float* lse, void* workspace,
                    size_t workspace_bytes, void* stream);

/* Stream-capture-safe form of verify_attn_mla.  The pages make the verify
 * kernel CUDA-graph capture-safe once it works ("The Build That Unlocked 3-6x
 * Decode Speedup", section "The Broader Significance"); a captured graph
 * replays every launch with its captured parameters, so here nothing depends
 * on host copies of the lengths: a planner kernel reads kv_indptr / qo_indptr
 * on the device at run time and writes the split plan (the same pieces as
 * verify_attn_mla's host planner, hence the same results bit for bit) and the
 * cluster schedule into the workspace, and every later kernel reads them from
 * there.  Capture one call per batch size; each replay may change the lengths,
 * the indices and the contents of every input buffer, within the bounds.
 *   batch, num_heads, sm_scale, splits, q .. lse: as for verify_attn_mla (the
 *               pointers are captured; their contents are read at replay)
 *   max_total_q   upper bound on qo_indptr[batch] at every replay, <= 64 * batch;
 *                 q holds max_total_q rows, out / lse hold max_total_q rows
 *   max_total_kv  upper bound on kv_indptr[batch] at every replay; kv_indices
 *                 holds max_total_kv entries
 *   workspace   >= verify_attn_mla_device_plan_workspace_size() bytes for the
 *               same batch, num_heads, bounds and splits, 256 B aligned.
 * Lengths that are inconsistent or exceed a bound are found by the planner on
 * the device: the call then computes nothing (out and lse keep their contents)
 * and verify_attn_mla_check returns VMLA_ERR_SHAPE.  Other argument errors are
 * returned before any launch.  No host synchronisation, allocation or host
 * read of device data happens inside the call. */
int verify_attn_mla_device_plan_workspace_size(int batch, int num_heads, int64_t max_total_q, int64_t max_total_kv,
                                               int splits, size_t* bytes);
int verify_attn_mla_device_plan(const void* q, const void* kv_pool, int64_t pool_slots, const int32_t* kv_indptr,
                                const int32_t* kv_indices, const int32_t* qo_indptr, const uint64_t* draft_mask,
                                const int32_t* parent, int batch, int num_heads, int64_t max_total_q,
                                int64_t max_total_kv, float sm_scale, int splits, void* out, float* lse,
                                void* workspace, size_t workspace_bytes, void* stream);

/* Persistent KV defragmentation ("The Build That Unlocked 3-6x Decode
 * Speedup" names the compaction of scattered page_size = 1 slots into
 * contiguous runs as the plan's next phase, section "The Context: A Custom
 * Kernel for an Unsupported Architecture").  Copies the rows of sequence b,
 * src_pool[kv_indices[kv_indptr[b] + j]] for j < N_b, to dst_pool slots
 * run_base[b] + j, and zeroes the run's following slots up to a multiple of
 * 128 rows (inside dst_slots), which verify_attn_mla_runs reads with no weight.
 *   src_pool [src_slots, 576] bf16, dst_pool [dst_slots, 576] bf16 (may be the
 *            same pool; a run must not overlap rows that are still being read)
 *   kv_indptr, kv_indices  device arrays as for verify_attn_mla;
 *   kv_indptr_host         host copy of kv_indptr (sizes the launch)
 *   run_base [batch] int32 device: each sequence's first destination slot;
 *            runs must not overlap one another
 *   status_word  optional: a source slot outside the pool or a run outside
 *            [0, dst_slots) records VMLA_ERR_INDEX (row or sequence index).
 * Argument errors return before the launch.  No host synchronisation. */
int verify_attn_mla_defrag(const void* src_pool, int64_t src_slots, const int32_t* kv_indptr,
                           const int32_t* kv_indices, const int32_t* kv_indptr_host, int batch, void* dst_pool,
                           int64_t dst_slots, const int32_t* run_base, uint32_t* status_word, void* stream);

/* The same copy for a decode loop that keeps its runs across steps: rows
 * j < first_row[b] of sequence b are already in place in its run (an earlier
 * defragmentation of the same run wrote them) and are left alone; rows
 * j >= first_row[b] are copied, and the run's tail is zeroed, as above.  A step
 * that accepted a_b tokens and drafts Q_b new ones passes the previous step's
 * accepted prefix length, so only the new rows cross.  The pages have no
 * counterpart; it is the persistent layout kept up to date per step.
 *   first_row [batch] int32 device: 0 <= first_row[b] <= N_b; a value outside
 *             records VMLA_ERR_INDEX (with the sequence index) in status_word
 *             and that sequence is skipped.
 *   max_new_rows  a bound on N_b - first_row[b] known to the caller (the launch
 *             then covers only that many rows past each first_row), or 0 for
 *             none; a sequence with more new rows records VMLA_ERR_INDEX and
 *             is skipped.  Negative: VMLA_ERR_SHAPE.  With a bound the launch
 *             depends on no host length (it is made even when the host copy
 *             says the runs are empty), so the call can be captured in a CUDA
 *             graph once and replayed as the runs grow (kv_indptr, kv_indices
 *             and first_row are read on the device at each replay).
 * Argument errors return before the launch.  No host synchronisation. */
int verify_attn_mla_defrag_append(const void* src_pool, int64_t src_slots, const int32_t* kv_indptr,
                                  const int32_t* kv_indices, const int32_t* kv_indptr_host, int batch,
                                  void* dst_pool, int64_t dst_slots, const int32_t* run_base,
                                  const int32_t* first_row, int64_t max_new_rows, uint32_t* status_word,
                                  void* stream);

/* verify_attn_mla on rows that lie in runs of the pool: the rows of sequence b
 * are kv_pool slots run_base[b] .. run_base[b] + N_b - 1 (its last Q_b rows
 * being the drafts), and the slots after each run up to a multiple of 128 hold
 * finite values (verify_attn_mla_defrag writes zeros there).  No gather runs:
 * the tensor-core kernel streams each run as tile loads straight from the pool.
 * Arguments as for verify_attn_mla with run_base [batch] int32 (device) in
 * place of kv_indices; workspace >= verify_attn_mla_runs_workspace_size()
 * bytes (no staged rows).  A run outside the pool records VMLA_ERR_INDEX
 * (sequence index) in the status word; its keys then read zeros. */
int verify_attn_mla_runs(const void* q, const void* kv_pool, int64_t pool_slots, const int32_t* kv_indptr,
                         const int32_t* run_base, const int32_t* qo_indptr, const uint64_t* draft_mask,
                         const int32_t* parent, const int32_t* kv_indptr_host, const int32_t* qo_indptr_host,
                         int batch, int num_heads, float sm_scale, int splits, void* out, float* lse,
                         void* workspace, size_t workspace_bytes, void* stream);
int verify_attn_mla_runs_workspace_size(int batch, int num_heads, const int32_t* qo_indptr_host,
                                        const int32_t* kv_indptr_host, int splits, size_t* bytes);

/* verify_attn_mla_runs for CUDA-graph capture: the plan is made on the device
 * from the device indptr arrays, as verify_attn_mla_device_plan makes it, and
 * the rows are read from their runs (no gather).  Arguments as for
 * verify_attn_mla_device_plan, with run_base [batch] int32 (device) in place
 * of kv_indices; max_total_kv bounds kv_indptr[batch] at every replay.  The
 * workspace holds no staged rows:
 * verify_attn_mla_runs_device_plan_workspace_size() bytes.  A decode loop can
 * capture this call after verify_attn_mla_defrag_append (with a bound on the
 * new rows) and replay both as its sequences grow.  Results equal
 * verify_attn_mla_runs' bit for bit.  Argument errors return before any
 * launch; lengths past the bounds make the call compute nothing and record
 * VMLA_ERR_SHAPE; a run outside the pool records VMLA_ERR_INDEX. */
int verify_attn_mla_runs_device_plan_workspace_size(int batch, int num_heads, int64_t max_total_q,
                                                    int64_t max_total_kv, int splits, size_t* bytes);
int verify_attn_mla_runs_device_plan(const void* q, const void* kv_pool, int64_t pool_slots, const int32_t* kv_indptr,
                                     const int32_t* run_base, const int32_t* qo_indptr, const uint64_t* draft_mask,
                                     const int32_t* parent, int batch, int num_heads, int64_t max_total_q,
                                     int64_t max_total_kv, float sm_scale, int splits, void* out, float* lse,
                                     void* workspace, size_t workspace_bytes, void* stream);

/* Failure test only.  For the calling thread's later calls of the tensor-core
 * entry points: fault 1 makes the kernel's softmax warps withhold the signal
 * that Q is in place, so no score MMA starts, a bounded wait expires, the
 * kernel records VMLA_ERR_TIMEOUT in the status word, stops every CTA of the
 * cluster and returns (no trap, no hang; the context stays usable); fault 0
 * restores normal operation.  wait_cycles sets the budget of every bounded
 * wait in clock cycles (0 = about a second).  Returns VMLA_ERR_SHAPE for other
 * values. */
int verify_attn_mla_test_fault(int fault, int64_t wait_cycles);

/* Greedy acceptance of the verified draft tree, the step after the verify
 * attention.  "The Build That Unlocked 3-6x Decode Speedup" lists a
 * tree_accept kernel (section "The Context: A Custom Kernel for an
 * Unsupported Architecture") without describing it; this is the plain reading:
 * draft node i of a sequence proposes draft_token[i] after its parent (the
 * prefix for a root) and is accepted when its parent is accepted and the token
 * equals the target model's greedy token after the parent.  The chosen path
 * ends at the deepest accepted node (the smallest index among equally deep
 * ones).  All arrays are device arrays; one warp per sequence.
 *   qo_indptr    [batch+1] int32; Q_b = qo_indptr[b+1] - qo_indptr[b] <= 64 nodes
 *   parent       [T_q] int32 local parent (-1 = root, parent[i] < i), or NULL for
 *                the chain parent[i] = i - 1
 *   draft_token  [T_q] int32: the token each node proposes
 *   target_token [T_q] int32: the target's greedy token after each node
 *   root_token   [batch] int32: the target's greedy token after the prefix
 *   accept_len   [batch] int32 out: nodes on the chosen path (0 .. Q_b)
 *   accept_path  [T_q] int32 out: from qo_indptr[b], the path's local node
 *                indices, root first, then -1 up to the sequence's end
 *   next_token   [batch] int32 out: the target's token after the path's last
 *                node, or root_token[b] when nothing is accepted
 *   status_word  optional (the first word of a workspace): a parent outside
 *                [-1, i) or a sequence outside [0, total_q) records
 *                VMLA_ERR_PARENT with the sequence index; that sequence
 *                accepts nothing.
 * Argument errors return before the launch.  No host synchronisation. */
int verify_attn_mla_tree_accept(const int32_t* qo_indptr, const int32_t* parent, const int32_t* draft_token,
                                const int32_t* target_token, const int32_t* root_token, int batch, int total_q,
                                int32_t* accept_len, int32_t* accept_path, int32_t* next_token, uint32_t* status_word,
                                void* stream);

/* verify_attn_mla on an fp8 latent pool: kv_pool_e4m3 [pool_slots, 576]
 * bytes, each an OCP FP8 E4M3 code (1 sign, 4 exponent bits with bias 7, 3
 * mantissa bits; codes S.1111.111 are NaN and must not occur), with one scale
 * for the pool: the value of a code is its e4m3 value times kv_scale, rounded
 * to float32 and then to bf16 (nearest even).  The pages do not describe an
 * fp8 cache; this is the plainest storage reading.  The gather dequantizes the
 * rows it copies into the workspace (the pool read is 576 B per key instead of
 * 1152), and everything after it is verify_attn_mla on those bf16 rows, so the
 * result equals verify_attn_mla on the dequantized pool bit for bit.
 * kv_scale: finite and > 0.  Workspace: verify_attn_mla_workspace_size(). */
int verify_attn_mla_fp8(const void* q, const void* kv_pool_e4m3, int64_t pool_slots, float kv_scale,
                        const int32_t* kv_indptr, const int32_t* kv_indices, const int32_t* qo_indptr,
                        const uint64_t* draft_mask, const int32_t* parent, const int32_t* kv_indptr_host,
                        const int32_t* qo_indptr_host, int batch, int num_heads, float sm_scale, int splits, void* out,
                        float* lse, void* workspace, size_t workspace_bytes, void* stream);

/* Fixed size of the scratch array behind verify_attn_mla_simt_static (32 MiB). */
#define VMLA_STATIC_SCRATCH_BYTES (32u << 20)

/* Same operation and arguments on the plain CUDA-core kernel (one warp per
 * four query rows, scores by FMA and warp shuffles).  A second, independent
 * GPU implementation used to cross-check the tensor-core kernel; its plan
 * and workspace come from verify_attn_mla_plan(VMLA_KERNEL_SIMT, ...). */
int verify_attn_mla_simt(const void* q, const void* kv_pool, int64_t pool_slots, const int32_t* kv_indptr,
                         const int32_t* kv_indices, const int32_t* qo_indptr, const uint64_t* draft_mask,
                         const int32_t* parent, const int32_t* kv_indptr_host, const int32_t* qo_indptr_host,
                         int batch, int num_heads, float sm_scale, int splits, void* out, float* lse,
                         void* workspace, size_t workspace_bytes, void* stream);

/* verify_attn_mla_simt without a workspace argument, for callers that cannot
 * allocate device memory at call time (an engine whose free HBM is all handed
 * to its KV cache, an allocator that must not be re-entered, a plugin host
 * that allows cudaMalloc only during its own set-up).  This entry point has no
 * counterpart in the pages; it exists only for such callers.
 * Scratch (status word, ancestor masks, split partials) comes from a fixed
 * VMLA_STATIC_SCRATCH_BYTES array in the library image, which every device
 * that loads the library holds until the process exits.  The entry point
 * allocates and frees nothing.  A plan whose workspace
 * (verify_attn_mla_plan(VMLA_KERNEL_SIMT, ...).workspace_bytes) exceeds the
 * array returns VMLA_ERR_WORKSPACE before any launch.  Each call looks up the
 * array's device address on the current device (cudaGetSymbolAddress, a host
 * query; the first one on a device loads the library's module there, so make
 * that first call before any stream capture).  Every call
 * on a device shares the one array and leaves its contents behind: calls that
 * may overlap on the GPU (different streams without ordering) race on it, so
 * order them on one stream.  Faults a kernel detects (a slot outside the pool,
 * malformed parents) are recorded in the array's status word, which
 * verify_attn_mla_simt_static_check() reads.  No address is kept between calls,
 * so the entry point stays usable after cudaDeviceReset (the module is loaded
 * again, possibly elsewhere, and the next call looks it up there). */
int verify_attn_mla_simt_static(const void* q, const void* kv_pool, int64_t pool_slots, const int32_t* kv_indptr,
                                const int32_t* kv_indices, const int32_t* qo_indptr, const uint64_t* draft_mask,
                                const int32_t* parent, const int32_t* kv_indptr_host,
                                const int32_t* qo_indptr_host, int batch, int num_heads, float sm_scale, int splits,
                                void* out, float* lse, void* stream);

/* Synchronises `stream` and returns the status word that the calls of
 * verify_attn_mla_simt_static on the current device left in the library's
 * scratch array (VMLA_OK when no kernel recorded a fault).  It copies 8 bytes
 * from the array to the host and allocates nothing.  Test and debugging aid;
 * it blocks the host. */
int verify_attn_mla_simt_static_check(void* stream);

/* The split merge on its own: o_parts [num_splits, rows, 512] fp32 (each part
 * already normalised by its own softmax sum), lse_parts [num_splits, rows]
 * fp32 (-inf = empty part).  Writes out [rows, 512] bf16 and lse [rows]:
 *   lse = ln sum_s exp(lse_s),  out = sum_s exp(lse_s - lse) * o_s.
 * 16 B aligned o_parts/out. */
int verify_attn_mla_merge(const float* o_parts, const float* lse_parts, int num_splits, int64_t rows, void* out,
                          float* lse, void* stream);

/* Expands draft-tree parents into per-query visibility words (bit k set for
 * k = i and every ancestor of i), the tree form of the q x q visibility
 * matrix.  parent [T_q] int32 local indices, qo_indptr [batch+1] device,
 * mask_out [T_q] uint64.  A malformed parent (not in [-1, i)) leaves that
 * query's word 0 and, if status_word (device uint32) is not NULL, records
 * VMLA_ERR_PARENT there. */
int verify_attn_mla_tree_mask(const int32_t* parent, const int32_t* qo_indptr, int batch, int total_q,
                              uint64_t* mask_out, uint32_t* status_word, void* stream);

/* Synchronises `stream`, reads the device status word of `workspace` left by
 * the last call that used it, and returns it (VMLA_OK when no kernel recorded
 * a fault).  Test and debugging aid; it blocks the host. */
int verify_attn_mla_check(const void* workspace, void* stream);

/* Host-buffer form for callers whose per-step inputs live in host memory.
 * Brings q, kv_indices and the optional mask/parent array (with qo_indptr for
 * a parent array) from host memory into `device_buffer`, runs verify_attn_mla
 * against the device-resident kv_pool, copies out and lse back into host
 * memory, and synchronises `stream` before returning (so the returned status
 * includes the device status word).  The indptr arrays are read on the host
 * for the plan.  Host buffers should be pinned for asynchronous copies; pinned
 * (page-locked) kv_indices are not copied but read in place by the gather
 * kernel through their mapped device address, so the call must not overlap a
 * change of them (it returns only when the stream is done).  q crosses on a
 * side stream after the other inputs, while the gather runs (the kernels after
 * the gather wait for it); out, lse and the status words return by
 * asynchronous copies on `stream` before its one synchronisation.  The
 * library keeps one such side stream, two events and an 8-byte pinned status
 * slot per calling thread and device, created at the first call.
 * device_buffer must hold verify_attn_mla_host_buffer_size() bytes (256 B
 * aligned). */
int verify_attn_mla_host_buffer_size(int batch, int num_heads, const int32_t* qo_indptr_host,
                                     const int32_t* kv_indptr_host, int splits, int has_mask, int has_parent,
                                     size_t* bytes);
int verify_attn_mla_host(const void* q_host, const void* kv_pool, int64_t pool_slots, const int32_t* kv_indptr_host,
                         const int32_t* kv_indices_host, const int32_t* qo_indptr_host,
                         const uint64_t* draft_mask_host, const int32_t* parent_host, int batch, int num_heads,
                         float sm_scale, int splits, void* out_host, float* lse_host, void* device_buffer,
                         size_t device_buffer_bytes, void* stream);

/* Measurement aid.  verify_attn_mla_timing_enable(n) creates host-side CUDA
 * events for the next n run calls (0 turns it off and frees them); while it is
 * on, every verify_attn_mla, _simt, _runs, _fp8 and _host call (not the
 * device-planned form) records events on its stream around each kernel it
 * launches.  verify_attn_mla_timing_read() waits
 * for those events and writes, per call in launch order, the device time in ms
 * of the KV gather kernel, the verify kernel and the merge kernel (0 for a
 * kernel the call did not launch) into arrays of `capacity` entries, sets
 * *count, and starts a new recording.  Not for concurrent use from several
 * host threads. */
int verify_attn_mla_timing_enable(int capacity);
int verify_attn_mla_timing_read(float* gather_ms, float* verify_ms, float* merge_ms, int capacity, int* count);

/* Human-readable name of a status code (static string). */
const char* verify_attn_mla_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int verify_attn_mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VERIFY_ATTN_MLA_H */
