/* CPU fp64 oracle for MLA speculative-decoding verify attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the package's smoke check and the bench's
 * CPU-baseline leg use it.  It shares no code with the GPU path; the only
 * thing both sides share is the seeded input generator.
 *
 * What it computes (plain definition, no tiling, no online softmax, no
 * splitting unless a split is asked for explicitly):
 *
 *   The operation is the verify attention described in "The Build That
 *   Unlocked 3-6x Decode Speedup", section "The Context: A Custom Kernel for an
 *   Unsupported Architecture" (draft queries scored against the MLA latent KV
 *   cache, softmax, weighted sum of the latent rows), with the data layout and
 *   the mask of "The Build That Bridged Design and Deployment", section "What
 *   This Build Achieves: The paged+bf16 Kernel": KV rows read through a slot
 *   indirection at page_size = 1, and a mask given as a prefix length (every
 *   prefix key visible) plus a small q x q visibility matrix over the draft
 *   tail.
 *
 *   For sequence b with N_b = kv_indptr[b+1] - kv_indptr[b] keys and
 *   Q_b = qo_indptr[b+1] - qo_indptr[b] draft queries, prefix P_b = N_b - Q_b,
 *   query i < Q_b (token t = qo_indptr[b] + i) and head h:
 *     row_j  = kv_pool[kv_indices[kv_indptr[b] + j], 0:576]       (bf16 -> f64)
 *     J      = { j < P_b } U { P_b + k : k < Q_b, bit k of mask_i }
 *     mask_i = draft_mask[t]                           if draft_mask is given
 *            = bits of i and of all its ancestors      if parent is given
 *            = bits 0..i (causal among drafts)         otherwise
 *     s_j    = sm_scale * sum_{d < 576} q[t,h,d] * row_j[d]
 *     m      = max_{j in J} s_j ,  l = sum_{j in J} exp(s_j - m)
 *     out    = sum_{j in J} exp(s_j - m) * row_j[0:512] / l
 *     lse    = m + ln l                                  (natural log)
 *   A query with no visible key gets out = 0 and lse = -inf.
 *
 * The split form (oracle_verify_split) cuts the key range [0, N_b) of each
 * sequence into contiguous pieces, evaluates each piece with the same
 * definition, and combines them with the log-sum-exp rule
 *     lse = ln sum_s exp(lse_s),  out = sum_s exp(lse_s - lse) * out_s,
 * the partial-softmax merge implied by the NSPLIT split-KV of "The Build
 * Script Edit", section "Context: The Long Road to a Custom sm_120 Kernel".
 * It exists to pin that identity, not to be fast.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_DQK 576
#define ORACLE_DV 512

static double bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Visibility bits of draft query i of one sequence over that sequence's drafts. */
static int draft_visibility(int i, int n_draft, const uint64_t* draft_mask_seq, const int32_t* parent_seq,
                            uint64_t* bits) {
  if (draft_mask_seq) {
    *bits = draft_mask_seq[i];
    return 0;
  }
  if (parent_seq) {
    uint64_t m = 0;
    int k = i, steps = 0;
    while (k >= 0) {
      if (k >= n_draft || steps > n_draft) return -1; /* not a forest with parents before children */
      m |= 1ULL << k;
      int p = parent_seq[k];
      if (p >= k) return -1;
      k = p;
      ++steps;
    }
    *bits = m;
    return 0;
  }
  uint64_t m = 0;
  for (int k = 0; k <= i; ++k) m |= 1ULL << k;
  *bits = m;
  return 0;
}

typedef struct {
  const uint16_t* q;
  const uint16_t* kv_pool;
  int64_t pool_slots;
  const int32_t* kv_indptr;
  const int32_t* kv_indices;
  const int32_t* qo_indptr;
  const uint64_t* draft_mask;
  const int32_t* parent;
  int batch, num_heads;
  double sm_scale;
} problem_t;

/* Evaluate query row (b, i, h) over the keys j in [j_lo, j_hi) of its sequence.
 * Writes out[0:512] and *lse.  Returns 0, or -1 on a bad index / mask. */
static int eval_row(const problem_t* P, int b, int i, int h, int j_lo, int j_hi, double* scores, double* out,
                    double* lse) {
  int kv0 = P->kv_indptr[b];
  int n_kv = P->kv_indptr[b + 1] - kv0;
  int q0 = P->qo_indptr[b];
  int n_q = P->qo_indptr[b + 1] - q0;
  int prefix = n_kv - n_q;
  int t = q0 + i;
  uint64_t bits;
  if (draft_visibility(i, n_q, P->draft_mask ? P->draft_mask + q0 : NULL, P->parent ? P->parent + q0 : NULL,
                       &bits) != 0)
    return -1;
  const uint16_t* qv = P->q + ((int64_t)t * P->num_heads + h) * ORACLE_DQK;
  double qd[ORACLE_DQK];
  for (int d = 0; d < ORACLE_DQK; ++d) qd[d] = bf16_to_f64(qv[d]);

  /* scores of the visible keys; -INFINITY marks an invisible one */
  double m = -INFINITY;
  for (int j = j_lo; j < j_hi; ++j) {
    int visible = (j < prefix) || ((bits >> (j - prefix)) & 1ULL);
    if (!visible) {
      scores[j - j_lo] = -INFINITY;
      continue;
    }
    int64_t slot = P->kv_indices[kv0 + j];
    if (slot < 0 || slot >= P->pool_slots) return -1;
    const uint16_t* row = P->kv_pool + slot * ORACLE_DQK;
    double s = 0.0;
    for (int d = 0; d < ORACLE_DQK; ++d) s += qd[d] * bf16_to_f64(row[d]);
    s *= P->sm_scale;
    scores[j - j_lo] = s;
    if (s > m) m = s;
  }
  for (int d = 0; d < ORACLE_DV; ++d) out[d] = 0.0;
  if (m == -INFINITY) {
    *lse = -INFINITY;
    return 0;
  }
  double l = 0.0;
  for (int j = j_lo; j < j_hi; ++j) {
    double s = scores[j - j_lo];
    if (s == -INFINITY) continue;
    double w = exp(s - m);
    l += w;
    const uint16_t* row = P->kv_pool + (int64_t)P->kv_indices[kv0 + j] * ORACLE_DQK;
    for (int d = 0; d < ORACLE_DV; ++d) out[d] += w * bf16_to_f64(row[d]);
  }
  for (int d = 0; d < ORACLE_DV; ++d) out[d] /= l;
  *lse = m + log(l);
  return 0;
}

/* ---- work distribution over (row) units ---- */

typedef struct {
  const problem_t* P;
  const int64_t* rows; /* global row ids t*H + h; NULL = all rows */
  int64_t n_rows;
  int splits; /* 0 = unsplit */
  double* out;
  double* lse;
  int64_t next;
  int error;
  pthread_mutex_t mu;
} work_t;

static int seq_of_token(const problem_t* P, int t) {
  int lo = 0, hi = P->batch; /* find b with qo_indptr[b] <= t < qo_indptr[b+1] */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (P->qo_indptr[mid] <= t) lo = mid; else hi = mid;
  }
  return lo;
}

static int eval_unit(const problem_t* P, int64_t row, int splits, double* scores, double* out, double* lse) {
  int t = (int)(row / P->num_heads), h = (int)(row % P->num_heads);
  int b = seq_of_token(P, t);
  int i = t - P->qo_indptr[b];
  int n_kv = P->kv_indptr[b + 1] - P->kv_indptr[b];
  if (splits <= 0) return eval_row(P, b, i, h, 0, n_kv, scores, out, lse);
  /* split form: contiguous pieces of [0, n_kv), then the log-sum-exp merge */
  int S = splits;
  double* o_s = (double*)malloc(sizeof(double) * ORACLE_DV * (size_t)S);
  double* l_s = (double*)malloc(sizeof(double) * (size_t)S);
  int rc = 0;
  for (int s = 0; s < S && rc == 0; ++s) {
    int lo = (int)(((int64_t)n_kv * s) / S), hi = (int)(((int64_t)n_kv * (s + 1)) / S);
    rc = eval_row(P, b, i, h, lo, hi, scores, o_s + (size_t)s * ORACLE_DV, &l_s[s]);
  }
  if (rc == 0) {
    double mx = -INFINITY;
    for (int s = 0; s < S; ++s) if (l_s[s] > mx) mx = l_s[s];
    for (int d = 0; d < ORACLE_DV; ++d) out[d] = 0.0;
    if (mx == -INFINITY) {
      *lse = -INFINITY;
    } else {
      double z = 0.0;
      for (int s = 0; s < S; ++s) z += exp(l_s[s] - mx);
      *lse = mx + log(z);
      for (int s = 0; s < S; ++s) {
        if (l_s[s] == -INFINITY) continue;
        double w = exp(l_s[s] - *lse);
        for (int d = 0; d < ORACLE_DV; ++d) out[d] += w * o_s[(size_t)s * ORACLE_DV + d];
      }
    }
  }
  free(o_s);
  free(l_s);
  return rc;
}

static void* worker(void* arg) {
  work_t* W = (work_t*)arg;
  int max_kv = 0;
  for (int b = 0; b < W->P->batch; ++b) {
    int n = W->P->kv_indptr[b + 1] - W->P->kv_indptr[b];
    if (n > max_kv) max_kv = n;
  }
  double* scores = (double*)malloc(sizeof(double) * (size_t)(max_kv > 0 ? max_kv : 1));
  for (;;) {
    pthread_mutex_lock(&W->mu);
    int64_t k = W->next++;
    pthread_mutex_unlock(&W->mu);
    if (k >= W->n_rows) break;
    int64_t row = W->rows ? W->rows[k] : k;
    if (eval_unit(W->P, row, W->splits, scores, W->out + k * ORACLE_DV, W->lse + k) != 0) {
      pthread_mutex_lock(&W->mu);
      W->error = 1;
      pthread_mutex_unlock(&W->mu);
    }
  }
  free(scores);
  return NULL;
}

static int check_problem(const problem_t* P) {
  if (!P->q || !P->kv_pool || !P->kv_indptr || !P->kv_indices || !P->qo_indptr) return -1;
  if (P->batch < 0 || P->num_heads <= 0) return -1;
  if (P->kv_indptr[0] != 0 || P->qo_indptr[0] != 0) return -1;
  for (int b = 0; b < P->batch; ++b) {
    int n_kv = P->kv_indptr[b + 1] - P->kv_indptr[b];
    int n_q = P->qo_indptr[b + 1] - P->qo_indptr[b];
    if (n_q < 0 || n_q > 64 || n_kv < n_q) return -1;
  }
  return 0;
}

static int run(const problem_t* P, const int64_t* rows, int64_t n_rows, int splits, double* out, double* lse,
               int num_threads) {
  if (check_problem(P) != 0) return -1;
  if (num_threads <= 0) num_threads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  if (num_threads < 1) num_threads = 1;
  if (num_threads > 1024) num_threads = 1024;
  if (n_rows < num_threads) num_threads = n_rows > 0 ? (int)n_rows : 1;
  work_t W;
  W.P = P;
  W.rows = rows;
  W.n_rows = n_rows;
  W.splits = splits;
  W.out = out;
  W.lse = lse;
  W.next = 0;
  W.error = 0;
  pthread_mutex_init(&W.mu, NULL);
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)num_threads);
  for (int k = 0; k < num_threads; ++k) pthread_create(&th[k], NULL, worker, &W);
  for (int k = 0; k < num_threads; ++k) pthread_join(th[k], NULL);
  free(th);
  pthread_mutex_destroy(&W.mu);
  return W.error ? -1 : 0;
}

#define PROBLEM_ARGS                                                                                      \
  const uint16_t *q, const uint16_t *kv_pool, int64_t pool_slots, const int32_t *kv_indptr,                \
      const int32_t *kv_indices, const int32_t *qo_indptr, const uint64_t *draft_mask, const int32_t *parent, \
      int batch, int num_heads, double sm_scale

#define PROBLEM_INIT \
  {q, kv_pool, pool_slots, kv_indptr, kv_indices, qo_indptr, draft_mask, parent, batch, num_heads, sm_scale}

/* Every query row: out [T_q, H, 512] f64, lse [T_q, H] f64. */
int oracle_verify(PROBLEM_ARGS, double* out, double* lse, int num_threads) {
  problem_t P = PROBLEM_INIT;
  if (check_problem(&P) != 0) return -1;
  int64_t n_rows = (int64_t)qo_indptr[batch] * num_heads;
  return run(&P, NULL, n_rows, 0, out, lse, num_threads);
}

/* A chosen subset of rows (global id t*H + h): out [n_rows, 512], lse [n_rows]. */
int oracle_verify_rows(PROBLEM_ARGS, const int64_t* rows, int64_t n_rows, double* out, double* lse,
                       int num_threads) {
  problem_t P = PROBLEM_INIT;
  if (check_problem(&P) != 0) return -1;
  int64_t total = (int64_t)qo_indptr[batch] * num_heads;
  for (int64_t k = 0; k < n_rows; ++k)
    if (rows[k] < 0 || rows[k] >= total) return -1;
  return run(&P, rows, n_rows, 0, out, lse, num_threads);
}

/* Split-and-merge form with `splits` contiguous key pieces per sequence (all rows). */
int oracle_verify_split(PROBLEM_ARGS, int splits, double* out, double* lse, int num_threads) {
  problem_t P = PROBLEM_INIT;
  if (splits < 1 || check_problem(&P) != 0) return -1;
  int64_t n_rows = (int64_t)qo_indptr[batch] * num_heads;
  return run(&P, NULL, n_rows, splits, out, lse, num_threads);
}

/* The log-sum-exp merge on its own: o_parts [S, R, D], lse_parts [S, R] -> o [R, D], lse [R].
 * A part with lse = -inf carries no weight; all parts -inf gives o = 0, lse = -inf. */
int oracle_merge(const double* o_parts, const double* lse_parts, int S, int64_t R, int D, double* o,
                 double* lse) {
  for (int64_t r = 0; r < R; ++r) {
    double mx = -INFINITY;
    for (int s = 0; s < S; ++s) if (lse_parts[(int64_t)s * R + r] > mx) mx = lse_parts[(int64_t)s * R + r];
    for (int d = 0; d < D; ++d) o[r * D + d] = 0.0;
    if (mx == -INFINITY) {
      lse[r] = -INFINITY;
      continue;
    }
    double z = 0.0;
    for (int s = 0; s < S; ++s) z += exp(lse_parts[(int64_t)s * R + r] - mx);
    lse[r] = mx + log(z);
    for (int s = 0; s < S; ++s) {
      double ls = lse_parts[(int64_t)s * R + r];
      if (ls == -INFINITY) continue;
      double w = exp(ls - lse[r]);
      for (int d = 0; d < D; ++d) o[r * D + d] += w * o_parts[((int64_t)s * R + r) * D + d];
    }
  }
  return 0;
}

/* Ancestor-closure visibility masks of every draft query from local parents. */
int oracle_tree_masks(const int32_t* parent, const int32_t* qo_indptr, int batch, uint64_t* mask_out) {
  for (int b = 0; b < batch; ++b) {
    int q0 = qo_indptr[b], n_q = qo_indptr[b + 1] - q0;
    if (n_q < 0 || n_q > 64) return -1;
    for (int i = 0; i < n_q; ++i)
      if (draft_visibility(i, n_q, NULL, parent + q0, &mask_out[q0 + i]) != 0) return -1;
  }
  return 0;
}

int oracle_num_cpus(void) { return (int)sysconf(_SC_NPROCESSORS_ONLN); }
