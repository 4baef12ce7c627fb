// Tensor-core verify attention for sm_103a: tcgen05 MMAs shared by pairs of
// SMs (cta_group::2) with TMEM accumulators, KV tiles streamed by tiled TMA.
//
// The method is the KV-split flash-decode of "The Build That Unlocked 3-6x
// Decode Speedup", section "The Context: A Custom Kernel for an Unsupported
// Architecture": KV tiles streamed through shared memory, online softmax, and
// one read of each KV tile shared by many query rows.  The pages share a tile
// across a head tile of 8 heads (section "Context: The Long Road to a Custom
// sm_120 Kernel" of "The Build Script Edit"); here a tile serves 256 query
// rows (heads x draft positions of one sequence) in one 2-SM MMA.  The KV rows
// are read from the contiguous copy the gather kernel made of each sequence's
// page_size = 1 slots, or from each sequence's run of the pool after a
// persistent defragmentation.
//
// A work unit is 256 query rows (r = i*H + h) of one sequence over one
// contiguous piece of its key range, and runs on a cluster of four CTAs:
//   ranks 0,1 ("scorer pair")  hold Q (latent part in tensor memory, rope part
//       in shared memory), each for its 128 rows.  Per 128-key tile each CTA
//       loads 64 of the keys (all 576 columns) and the pair computes
//       S = Q K^T as M256 x N128 MMAs: every CTA receives the scores of its
//       rows against all 128 keys.  Eight softmax warps per CTA run the online
//       softmax in two 64-key messages per tile; a sender thread ships each
//       message (P bf16 128 x 64, per-row rescale factors) to the matching
//       mixer CTA by a shared-memory bulk copy.
//   ranks 2,3 ("mixer pair")   hold O [128 x 512] fp32 in all 512 TMEM
//       columns each.  Per tile each CTA loads half of the 512 value columns
//       of all 128 keys and the pair computes O = alpha * O + P V as M256 x
//       N256 MMAs, then normalises and writes the result.
// Each SM thus streams half of every tile it needs; the split into scorer and
// mixer follows from tensor-memory capacity (O for 128 rows fills an SM's
// 512 columns).
//
// Warp roles (352 threads): warp 0 TMA producer (all ranks); warp 1: rank 0
// score MMA issuer, rank 1 forwarder of its S-buffer releases to rank 0,
// rank 2 P V issuer, rank 3 relay of its P arrivals to rank 2; scorer warps
// 2-9 softmax (two threads per row, 32 keys each per 64-key message), warp 10
// P sender; mixer warps 2-5 and 7-10 rescale/epilogue (two warps per TMEM
// lane quarter, each for half of the value columns), warp 6 P-slot release.
// Every wait is bounded; on expiry the kernel records VMLA_ERR_TIMEOUT in the
// status word, tells the other CTAs to stop, and every CTA leaves only after
// what was issued into it has landed (see the end of tc_verify_body), frees
// tensor memory and returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

#include <cstring>
#include <mutex>

#include "vmla_device.cuh"
#include "vmla_plan_core.h"
#include "vmla_sm100.cuh"

namespace vmla {
using namespace sm100;
namespace {

constexpr int kTileKeys = 128;         // keys per tile (N of the score MMA)
constexpr int kHalfKeys = 64;          // keys of a tile loaded by each scorer CTA
constexpr int kChunks = kDqk / 64;     // 9 column chunks of 64 bf16 (128 bytes) per row
constexpr int kQChunks = kDv / 64;     // 8 latent chunks (Q latent lives in TMEM columns 0..255)
constexpr int kVChunksCta = kDv / 128; // 4 value chunks per mixer CTA (half of the 8)
constexpr int kKBox = kHalfKeys * 128; // 8 KB: 64 rows x 128 bytes
constexpr int kVStages = 3;            // mixer V stages, one per 64-key message
static_assert(kVStages >= 2, "the scorer's two K stages use the first two stage barriers");
constexpr int kRowsCta = 128;
constexpr int kRowsUnit = 256;
constexpr int kSoftWarps = 8;          // scorer softmax warps: two per TMEM lane quarter
constexpr int kParts = kSoftWarps / 4; // threads per query row
constexpr int kPartKeys = 64 / kParts; // keys of a 64-key message per thread
constexpr int kSenderWarp = 2 + kSoftWarps;
constexpr int kThreadsTC = 32 * (kSenderWarp + 1);  // 11 warps
static_assert(kPartKeys == 16 || kPartKeys == 32, "TMEM load width per softmax thread");
constexpr int kClusterCtas = 4;
constexpr uint32_t kSCol = 256;        // S buffers at TMEM columns 256 and 384
constexpr float kTau = 8.0f;           // the running max is raised only when a tile exceeds it by 2^8
constexpr uint16_t kScorerMask = 0x3, kMixerMask = 0xC;
constexpr uint32_t kQBytes = 2 * kChunks * kKBox;  // a scorer CTA's 128 Q rows, all 576 columns

enum Cmd : uint32_t { kCmdRescale = 1, kCmdEpilogue = 2, kCmdExit = 3 };

// Optional pipeline trace (compile with -DVMLA_TRACE): global-timer stamps of
// each hand-off for the first kTraceTiles tiles of cluster 0, and (events 26-31)
// one stamp or count per cluster at the cluster's own index.
#ifdef VMLA_TRACE
constexpr int kTraceTiles = 256;
constexpr int kTraceEvents = 32;
__device__ uint64_t g_vmla_trace[kTraceEvents * kTraceTiles];
__device__ __forceinline__ void vtrace(int ev, int tile) {
  if (cluster_id_x() == 0 && ev >= 0 && ev < kTraceEvents && tile >= 0 && tile < kTraceTiles) {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    g_vmla_trace[ev * kTraceTiles + tile] = t;
  }
}
__device__ __forceinline__ void vtrace_cluster(int ev, uint64_t value, bool stamp) {
  const uint32_t c = cluster_id_x();
  if (ev >= 0 && ev < kTraceEvents && c < (uint32_t)kTraceTiles) {
    if (stamp) asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(value));
    g_vmla_trace[ev * kTraceTiles + c] = value;
  }
}
#define VTRACE(ev, tile) vtrace(ev, tile)
#define VTRACE_CLUSTER(ev) vtrace_cluster(ev, 0, true)
#define VTRACE_CLUSTER_VALUE(ev, v) vtrace_cluster(ev, v, false)
#else
#define VTRACE(ev, tile) ((void)0)
#define VTRACE_CLUSTER(ev) ((void)0)
#define VTRACE_CLUSTER_VALUE(ev, v) ((void)0)
#endif

// One P message covers half a tile (64 keys): two staging buffers of this
// size let one copy drain while the next half is computed, and the mixer
// starts its products as soon as each half has arrived.
constexpr int kMsgKeys = 64;
constexpr int kMsgsPerTile = kTileKeys / kMsgKeys;
constexpr int kPSlots = 6;  // mixer receive slots (an even count measured faster than an odd one)
constexpr int kStages = 2;  // scorer staging buffers (a copy drains while the next message is computed)
struct __align__(1024) PMsg {
  uint8_t p[kRowsCta * 128];  // P [128 rows][64 keys] bf16, K-major, 128-byte swizzle
  float alpha[kRowsCta];      // factor for O rows before this message's product (1 = unchanged)
  uint32_t flags;             // bit 0: some alpha differs from 1
  uint32_t pad[3];
};
constexpr uint32_t kMsgBytes = kRowsCta * 128 + kRowsCta * 4 + 16;  // bytes shipped per message
static_assert(offsetof(PMsg, pad) + 12 == kMsgBytes, "message layout");

struct __align__(16) Finals {
  float m[kRowsCta];  // running max (log2 units)
  float l[kRowsCta];  // softmax denominator relative to m
};

struct ScorerSmem {
  uint8_t kv[2][kChunks][kKBox];  // this CTA's 64 keys of each tile, 128-byte swizzled column chunks
  uint8_t qrope[kRowsCta * 128];  // Q rope part [128 rows x 64] bf16, K-major, 128-byte swizzle
  PMsg stage[kStages];            // P message staging
  Finals fin_stage[2];            // per-unit finals staging
  float pmax[2][kParts][kRowsCta];  // per message parity and part: partial row maxima
  float lpart[kParts - 1][kRowsCta]; // parts 1.. row sums at a unit's last message
};

struct MixerSmem {
  uint8_t v[kVStages][kVChunksCta][kKBox];  // this CTA's value columns of one message's 64 keys
  PMsg msg[kPSlots];                 // P receive slots
  Finals fin[2];                     // per-unit finals receive slots
  uint4 ep[8][32][4];                // epilogue: each warp's 32 rows x 64 bytes (16-byte granules, swizzled)
};

struct Ctl {
  uint64_t kfull[kVStages], kfree[kVStages];  // K stages (scorer: 2) or V stages (mixer: kVStages)
  uint64_t sfull[2], sfree[2];  // S buffers (scorer; sfree counts on rank 0)
  uint64_t sread[2];            // rank 1: its softmax warps have read S buffer s
  uint64_t staged[kStages], stgfree[kStages];  // scorer: P staging buffer written / free again
  uint64_t qfull;               // Q of both scorer CTAs written (rank 0)
  uint64_t qland, qfree;        // scorer: a unit's Q landed in the K stages / moved out of them
  uint64_t pfull[kPSlots], pfree[kPSlots], pdone[kPSlots];
  uint64_t finfull[2];          // mixer: unit finals received
  uint64_t finfree[2];          // scorer: the mixer's epilogue has read finals buffer f
  uint64_t cmd_full, cmd_done, obar;
  uint32_t cmd;
  uint32_t tmem_base;
  volatile int32_t abort_flag;
  long long wait_cycles;        // budget of every bounded wait (clock64 cycles)
  uint32_t warp_flags[kStages][kSoftWarps];  // per staging buffer: softmax warp w saw some alpha != 1
  uint32_t peer_flags[kPSlots];  // rank 2: flags of rank 3's half of message slot s
  volatile uint32_t wg_stop[4][2];  // scorer softmax warp pair (lane quarter): stop at this message (per parity)
  volatile uint32_t wg_cmd;   // mixer epilogue group: command broadcast
};

struct TcSmem {
  union {
    ScorerSmem s;
    MixerSmem m;
  } u;
  Ctl c;
};

// TMEM load of a softmax thread's columns (overloads by width).
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[32]) { tmem_ld32(taddr, r); }
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[16]) { tmem_ld16(taddr, r); }

// One work unit: row block rb of sequence b over keys [k_lo, k_hi), piece
// `piece` of the n_pieces that cover those rows' keys (one: the unit writes
// the rows' results, else fp32 partials for the merge).
struct UnitInfo {
  int b, rb, piece, n_pieces, R, prefix, k_lo, k_hi, n_tiles;
};

// Unit u of a uniform plan.
__device__ __forceinline__ UnitInfo decode_unit(const PlanParams& p, int u) {
  UnitInfo ui;
  ui.b = seq_of_unit(p, u);
  const SeqPlan& s = p.seq[ui.b];
  const int local = u - s.unit_start;
  ui.rb = local % s.n_rb;
  ui.piece = local / s.n_rb;
  ui.n_pieces = s.n_split;
  ui.R = s.n_q * p.num_heads;
  ui.prefix = s.n_kv - s.n_q;
  ui.k_lo = ui.piece * s.chunk;
  ui.k_hi = min(s.n_kv, ui.k_lo + s.chunk);
  ui.n_tiles = (ui.k_hi - ui.k_lo + kTileKeys - 1) / kTileKeys;
  return ui;
}

// Last sequence whose first stream starts at or before cost position x (a
// sequence without streams shares its position with the next one, so the
// search lands on one with streams for any x below the total).
__device__ __forceinline__ int lane_seq_at(const PlanParams& p, int64_t x) {
  int lo = 0, hi = p.batch;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.seq[mid].lane_cost <= x) lo = mid; else hi = mid;
  }
  return lo;
}

// Streams [*s_begin, *s_end) of a lane plan whose tiles meet lane l's interval
// [l L, (l + 1) L) of the cost space.
__device__ __forceinline__ void lane_streams(const PlanParams& p, int l, int* s_begin, int* s_end) {
  const int64_t L = p.lane_tiles, W = p.lane_total, P = (int64_t)l * L;
  *s_begin = *s_end = 0;
  if (P >= W) return;
  const int64_t Q = P + L < W ? P + L : W;
  const SeqPlan& s = p.seq[lane_seq_at(p, P)];
  const int64_t T = plan_seq_tiles(s.n_kv), g0 = (P - s.lane_cost) / (T + kLaneStreamTiles);
  int first = s.unit_start + (int)g0;
  if (P - s.lane_cost - g0 * (T + kLaneStreamTiles) >= T) ++first;  // P lies in that stream's fixed charge
  const SeqPlan& s2 = p.seq[lane_seq_at(p, Q - 1)];
  int64_t g2 = (Q - 1 - s2.lane_cost) / plan_stream_span(s2.n_kv);
  const int64_t ng2 = s2.n_rb / p.lane_width;
  if (g2 > ng2 - 1) g2 = ng2 - 1;
  const int last = s2.unit_start + (int)g2;
  *s_begin = first;
  *s_end = last + 1 > first ? last + 1 : first;
}

// Stream s of a lane plan as seen by cluster j of lane l: row block g G + j of
// the stream's sequence over the tiles of the stream that fall in the lane.
__device__ __forceinline__ UnitInfo decode_lane_unit(const PlanParams& p, int s, int l, int j) {
  UnitInfo ui;
  ui.b = seq_of_unit(p, s);
  const SeqPlan& sp = p.seq[ui.b];
  const int64_t g = s - sp.unit_start;
  const int64_t T = plan_seq_tiles(sp.n_kv), L = p.lane_tiles;
  const int64_t A = sp.lane_cost + g * (T + kLaneStreamTiles);  // cost position of the stream's first tile
  const int64_t P = (int64_t)l * L;
  const int64_t lo = (P > A ? P : A) - A;
  const int64_t hi = (P + L < A + T ? P + L : A + T) - A;
  ui.rb = (int)(g * p.lane_width + j);
  ui.piece = (int)(l - A / L);
  ui.n_pieces = (int)plan_stream_pieces(A, T, L);
  ui.R = sp.n_q * p.num_heads;
  ui.prefix = sp.n_kv - sp.n_q;
  ui.k_lo = (int)(lo * kTileKeys);
  ui.k_hi = min(sp.n_kv, (int)(hi * kTileKeys));
  ui.n_tiles = (int)(hi - lo);
  return ui;
}

// The k-th entry of this cluster's work list: an index of the schedule's order
// (uniform plan) or a stream index (lane plan).
__device__ __forceinline__ UnitInfo unit_at(const PlanParams& p, const TcSched& sched, int k) {
  if (p.lane_width == 0) return decode_unit(p, sched.unit_base + sched.order[k]);
  const int cid = (int)cluster_id_x();
  return decode_lane_unit(p, k, cid / p.lane_width, cid % p.lane_width);
}

// Sets the abort flag of every CTA of the cluster.
__device__ __noinline__ void abort_cluster(TcSmem& sm) {
  sm.c.abort_flag = 1;
  const uint32_t me = cluster_ctarank();
  const uint32_t local = smem_u32((const void*)const_cast<int32_t*>(&sm.c.abort_flag));
  for (uint32_t r = 0; r < kClusterCtas; ++r)
    if (r != me) st_cluster_u32(mapa(local, r), 1u);
}

// Bounded wait after a first try failed; false on expiry or when the cluster is aborting.
__device__ __noinline__ bool wait_bar_slow(TcSmem& sm, uint64_t* bar, uint32_t parity, uint32_t* status,
                                           int where) {
  const long long budget = sm.c.wait_cycles;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (sm.c.abort_flag) return false;
    if (clock64() - t0 > budget) {
      record_status(status, VMLA_ERR_TIMEOUT, (uint32_t)where);
      abort_cluster(sm);
      return false;
    }
  }
}

// Bounded wait; false on expiry or when the cluster is aborting.  The first try
// is inline (it suspends the thread until the phase completes or the hardware's
// time limit passes); the clocked loop is out of line.
__device__ __forceinline__ bool wait_bar(TcSmem& sm, uint64_t* bar, uint32_t parity, uint32_t* status, int where) {
  return mbar_try_wait_cluster(bar, parity) || wait_bar_slow(sm, bar, parity, status, where);
}

// Bounded wait that ignores the abort flag, for a phase that completes once
// what this CTA itself issued has landed (draining before exit).  Should the
// budget run out, the kernel records VMLA_ERR_TIMEOUT and aborts the cluster,
// so that every CTA waits out the settle period before it leaves.
__device__ __noinline__ void drain_bar(TcSmem& sm, uint64_t* bar, uint32_t parity, uint32_t* status, int where) {
  const long long budget = sm.c.wait_cycles;
  const long long t0 = clock64();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (clock64() - t0 > budget) {
      record_status(status, VMLA_ERR_TIMEOUT, (uint32_t)where);
      abort_cluster(sm);
      return;
    }
  }
}

// Bounded wait for a phase that another CTA's work completes; it may never
// come once the cluster is aborting (the settle period at the end of the
// kernel then covers whatever had been issued).
__device__ __noinline__ void drain_bar_live(TcSmem& sm, uint64_t* bar, uint32_t parity, uint32_t* status,
                                            int where) {
  const long long budget = sm.c.wait_cycles;
  const long long t0 = clock64();
  while (!mbar_try_wait_cluster(bar, parity) && !sm.c.abort_flag) {
    if (clock64() - t0 > budget) {
      record_status(status, VMLA_ERR_TIMEOUT, (uint32_t)where);
      abort_cluster(sm);
      return;
    }
  }
}

// After a failed wait: every CTA of the cluster has stopped issuing work, but
// tile loads, bulk copies, tensor-core commits and MMAs issued before may still
// be on their way into this CTA's shared and tensor memory.  Each of them takes
// microseconds; this waits half a millisecond of the global timer (and at most
// 2^26 reads of it).
__device__ __noinline__ void settle_after_abort() {
  uint64_t t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (int k = 0; k < (1 << 26); ++k) {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > 500000ull) break;
  }
}

__device__ __forceinline__ int total_tiles(const PlanParams& plan, const TcSched& sched, int u_begin, int u_end) {
  int total = 0;
  for (int k = u_begin; k < u_end; ++k) total += unit_at(plan, sched, k).n_tiles;
  return total;
}

// ------------------------------------------------------------------ producer (warp 0, lane 0, every CTA)
// Scorer CTA q loads keys [64q, 64q + 64) of each 128-key tile, all nine
// column chunks (one 3-D box: 64 rows x 9 chunks of 64 columns, chunk-major),
// into two tile stages; mixer CTA q loads value chunks {2q, 2q+1, 2q+4, 2q+5}
// of each 64-key message (two boxes of two chunks; the N halves the pair's P V
// MMAs expect) into kVStages message stages.  Both CTAs of
// a pair complete their bytes on the even CTA's barrier, which that CTA arms
// for the pair.  Rows past the piece's end belong to other keys (masked by the
// softmax) or lie outside the staged rows (zero fill).
// Before each unit's first tile a scorer CTA also loads the unit's Q rows (its
// 128) through both K stages: latent chunk c of row half h into stage h, chunk
// c; the rope chunk into qrope.  The softmax warps move the latent part into
// tensor memory and release the stages (qfree) before the first K tile loads.
__device__ void producer_role(TcSmem& sm, const CUtensorMap* map, const CUtensorMap* vmap, const CUtensorMap* qmap,
                              const PlanParams& plan, const TcSched& sched, const RunArgs& a, int u_begin, int u_end,
                              uint32_t rank) {
  const bool scorer = rank < 2;
  const uint32_t q = rank & 1;
  const uint32_t leader = rank & 2u;
  const int nst = scorer ? 2 : kVStages;
  const uint32_t pair_bytes = scorer ? 2u * kChunks * kKBox : 2u * kVChunksCta * kKBox;
  int it = 0;  // loads issued (tiles for the scorer, messages for the mixer)
  int uq = 0;  // Q loads issued (scorer)
  bool ok = true;
  // the kernel may start under the gather's tail: the staged rows are complete past this wait
  grid_dependency_wait();
  if (rank == 0) VTRACE_CLUSTER(28);  // the launch before this one is complete
  for (int ui_idx = u_begin; ui_idx < u_end && ok; ++ui_idx) {
    const UnitInfo ui = unit_at(plan, sched, ui_idx);
    const SeqPlan& sp = plan.seq[ui.b];
    // first row of the sequence in the tensor map: its staged offset, or its pool run
    // (a run outside the pool only reads the out-of-range fill; a check kernel reports it)
    const int row0 = a.run_base ? a.run_base[ui.b] : sp.kv_off;
    const int loads = scorer ? ui.n_tiles : ui.n_tiles * kMsgsPerTile;
    if (scorer) {
      // both stages free (the last two tiles' products are complete, and with them
      // every product that read the previous Q), then Q in, then wait until it has
      // been moved out; the tile loads below find these releases already complete
      for (int k = 0; k < 2 && ok; ++k)
        ok = wait_bar(sm, &sm.c.kfree[(it + k) % 2], (((it + k) / 2) & 1) ^ 1, a.status, 102);
      if (!ok) break;
      const int qy = sp.q_off * plan.num_heads + ui.rb * kRowsUnit + (int)q * kRowsCta;
      const uint32_t qbar = smem_u32(&sm.c.qland);
      mbar_arrive_expect_tx(&sm.c.qland, kQBytes);
#pragma unroll 1
      for (int h = 0; h < 2; ++h)
#pragma unroll 1
        for (int c = 0; c < kChunks; ++c) {
          const uint32_t dst = c < kQChunks ? smem_u32(&sm.u.s.kv[h][c][0]) : smem_u32(sm.u.s.qrope) + h * kKBox;
          tma_load_2d(dst, qmap, 64 * c, qy + 64 * h, qbar);
        }
      ++uq;
      if (!wait_bar(sm, &sm.c.qfree, (uq - 1) & 1, a.status, 103)) {
        ok = false;
        break;
      }
    }
    for (int n = 0; n < loads; ++n) {
      const int s = it % nst;
      if (!wait_bar(sm, &sm.c.kfree[s], ((it / nst) & 1) ^ 1, a.status, 100)) {
        ok = false;
        break;
      }
      if (rank != 3) VTRACE(scorer ? (q ? 10 : 0) : 5, it);
      const uint32_t bar = mapa(smem_u32(&sm.c.kfull[s]), leader);
      if (q == 0) mbar_arrive_expect_tx(&sm.c.kfull[s], pair_bytes);
      if (scorer) {
        // all nine column chunks of this CTA's 64 keys in one box (chunk-major in the stage)
        const int y = row0 + ui.k_lo + n * kTileKeys + kHalfKeys * (int)q;
        tma_load_3d_pair(smem_u32(&sm.u.s.kv[s][0][0]), map, 0, y, 0, bar);
      } else {
        // value chunks {2q, 2q+1} and {2q+4, 2q+5} of the message's 64 keys, two chunks per box
        const int y = row0 + ui.k_lo + n * kMsgKeys;
        tma_load_3d_pair(smem_u32(&sm.u.m.v[s][0][0]), vmap, 0, y, 2 * (int)q, bar);
        tma_load_3d_pair(smem_u32(&sm.u.m.v[s][2][0]), vmap, 0, y, 2 * (int)q + 4, bar);
      }
      ++it;
    }
  }
  // the even CTA drains its last loads (their barriers count both CTAs' bytes)
  if (q == 0)
    for (int k = 1; k <= nst && it - k >= 0; ++k)
      drain_bar_live(sm, &sm.c.kfull[(it - k) % nst], ((it - k) / nst) & 1, a.status, 120);
  // tail: the releases of the last stages arrive on this CTA's barriers from the
  // tensor core (a commit multicast to both CTAs of the pair); this CTA may not
  // exit while one is still in flight
  for (int k = 1; k <= nst && it - k >= 0; ++k)
    drain_bar_live(sm, &sm.c.kfree[(it - k) % nst], ((it - k) / nst) & 1, a.status, 121);
  // and the last Q load has landed (the softmax normally waited for it)
  if (scorer && uq > 0) drain_bar_live(sm, &sm.c.qland, (uq - 1) & 1, a.status, 122);
}

// ------------------------------------------------------------------ rank 0: score MMA issuer (warp 1, lane 0)
// Per tile: 32 M256 N128 K16 MMAs with A = Q latent from TMEM, then 4 with
// A = Q rope from shared memory; B = the pair's K rows (K-major).
__device__ void scorer_mma_role(TcSmem& sm, const PlanParams& plan, const TcSched& sched, const RunArgs& a,
                                uint32_t tbase, int u_begin, int u_end) {
  constexpr uint32_t idesc = idesc_bf16_f32(kRowsUnit, kTileKeys, 0, 0);
  ScorerSmem& S = sm.u.s;
  int it = 0, uu = 0;
  for (int ui_idx = u_begin; ui_idx < u_end; ++ui_idx, ++uu) {
    const UnitInfo ui = unit_at(plan, sched, ui_idx);
    if (!wait_bar(sm, &sm.c.qfull, uu & 1, a.status, 200)) break;
    tc_fence_after();
    bool ok = true;
    for (int t = 0; t < ui.n_tiles; ++t, ++it) {
      const int s = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      if (!wait_bar(sm, &sm.c.kfull[s], ph, a.status, 201)) {
        ok = false;
        break;
      }
      VTRACE(1, it);
      if (!wait_bar(sm, &sm.c.sfree[s], ph ^ 1, a.status, 202)) {
        ok = false;
        break;
      }
      VTRACE(12, it);
      tc_fence_after();
      const uint32_t d = tbase + kSCol + (uint32_t)s * kTileKeys;
#pragma unroll
      for (int c = 0; c < kQChunks; ++c) {
        const uint32_t kbase = smem_u32(&S.kv[s][c][0]);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_pair_ts(d, tbase + (uint32_t)(c * 32 + k * 8), smem_desc(kbase + k * 32, 16, 1024), idesc,
                      (c | k) != 0);
      }
      {
        const uint32_t kbase = smem_u32(&S.kv[s][kQChunks][0]);
        const uint32_t qbase = smem_u32(S.qrope);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_pair_ss(d, smem_desc(qbase + k * 32, 16, 1024), smem_desc(kbase + k * 32, 16, 1024), idesc, 1u);
      }
      mma_commit_pair(&sm.c.sfull[s], kScorerMask);
      mma_commit_pair(&sm.c.kfree[s], kScorerMask);
      VTRACE(2, it);
    }
    if (!ok) break;
  }
  // all issued MMAs complete before the CTA may exit (this arrive goes to rank 0
  // only: nothing in rank 1 waits for it)
  mma_commit_pair(&sm.c.obar, (uint16_t)0x1);
  drain_bar(sm, &sm.c.obar, 0, a.status, 204);
}

// ------------------------------------------------------------------ ranks 0,1: softmax (warps 2 .. 2+kSoftWarps-1)
// A tile's 128 scores per row are processed as two 64-key messages.  Thread
// (part, row): row = TMEM lane = query row of this CTA, keys
// [kPartKeys*part, kPartKeys*(part + 1)) of each message.  The parts of a row agree on
// the message max through shared memory (one barrier of the lane quarter's two
// warps per message; the four quarters run independently), so
// all keep the same running reference max m_ref (raised only when a message
// exceeds it by 2^kTau, which bounds P by 2^kTau and makes rescales rare).
// The P message is staged in shared memory; the sender thread ships it.
__device__ void scorer_softmax_role(TcSmem& sm, const PlanParams& plan, const TcSched& sched, const RunArgs& a,
                                    uint32_t tbase, int u_begin, int u_end, uint32_t rank) {
  constexpr int kPairThreads = 32 * kParts;  // the warps of one TMEM lane quarter (both parts of its rows)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sw = warp - 2;                 // 0 .. kSoftWarps-1
  const int wq = warp & 3;                 // TMEM lane quarter this warp may access
  const int part = sw >> 2;                // keys [kPartKeys*part, kPartKeys*(part + 1)) of a message
  const int row = wq * 32 + lane;          // query row within this CTA = TMEM lane
  const int tid = threadIdx.x - 64;        // 0 .. 32*kSoftWarps-1 within the softmax warps
  const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
  const int H = plan.num_heads;
  const float scale = a.scale_log2;
  ScorerSmem& S = sm.u.s;
  const uint32_t qfull_r = mapa(smem_u32(&sm.c.qfull), 0);
  int it = 0, uu = 0, msg = 0;
  bool stop = false;
  // q and the ancestor masks are read only once everything before the kernel in the
  // stream is complete (the kernel may start under the gather's tail)
  grid_dependency_wait();
  for (int ui_idx = u_begin; ui_idx < u_end && !stop; ++ui_idx, ++uu) {
    const UnitInfo ui = unit_at(plan, sched, ui_idx);
    const SeqPlan& sp = plan.seq[ui.b];
    const int r = ui.rb * kRowsUnit + (int)(rank & 1) * kRowsCta + row;
    const bool valid = r < ui.R;
    // Q of this unit, landed by the producer's TMA loads: latent chunk c of this
    // row in stage (row / 64), chunk c (128-byte swizzled rows) goes to TMEM
    // columns 32c .. 32c + 31 (two bf16 per column), each part its chunks; rows
    // past the unit's rows get zeros (also in their rope columns, which the
    // loads put into qrope).  The previous unit's products are complete (the
    // producer waited for the last two tiles' releases before loading).
    __syncwarp();
    if (tid == 0 && rank == 0) VTRACE(20, uu);  // Q of unit uu awaited
    wait_bar(sm, &sm.c.qland, uu & 1, a.status, 305);  // (a failed wait leaves garbage; the stop comes later)
    {
      const int lr = row & 63;
      const uint8_t* stage_rows = &S.kv[row >> 6][0][lr * 128];
#pragma unroll 1
      for (int c = part; c < kQChunks; c += kParts) {
        uint32_t v[32];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const uint4 x = valid ? *reinterpret_cast<const uint4*>(stage_rows + c * kKBox + ((g ^ (lr & 7)) << 4))
                                : make_uint4(0, 0, 0, 0);
          v[4 * g] = x.x;
          v[4 * g + 1] = x.y;
          v[4 * g + 2] = x.z;
          v[4 * g + 3] = x.w;
        }
        tmem_st32(tbase + lane_base + (uint32_t)(c * 32), v);
      }
      if (!valid)
#pragma unroll
        for (int g = (8 / kParts) * part; g < (8 / kParts) * (part + 1); ++g)
          *reinterpret_cast<uint4*>(S.qrope + row * 128 + ((g ^ (row & 7)) << 4)) = make_uint4(0, 0, 0, 0);
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (tid == 0 && rank == 0) VTRACE(21, uu);  // Q of unit uu written
      if (lane == 0) {
        mbar_arrive(&sm.c.qfree);  // the stages may take K tiles again
        // (the failure test withholds this signal: the score MMAs then never start and a
        // bounded wait expires)
        if (a.test_fault != kFaultNoQReady) {
          if (rank == 0) mbar_arrive(&sm.c.qfull);
          else mbar_arrive_remote(qfull_r);
        }
      }
    }
    const int i = valid ? r / H : 0;
    const uint64_t vis = a.masks ? a.masks[sp.q_off + i] : causal_bits(i);
    const int mask_from = min(ui.prefix, ui.k_hi);  // keys below this are visible to every valid row
    float m_ref = -INFINITY, l = 0.f;
    for (int t = 0; t < ui.n_tiles && !stop; ++t, ++it) {
      const int sb = it & 1;
      // a failed wait leaves garbage in this tile; each warp pair still meets at the
      // barrier of each message and stops together there
      wait_bar(sm, &sm.c.sfull[sb], (it >> 1) & 1, a.status, 300);
      if (tid == 0) VTRACE(rank ? 11 : 3, it);
#pragma unroll 1
      for (int j = 0; j < kMsgsPerTile; ++j, ++msg) {
        __syncwarp();
        tc_fence_after();
        uint32_t v[kPartKeys];
        {
          const uint32_t scol =
              tbase + lane_base + kSCol + (uint32_t)sb * kTileKeys + (uint32_t)(j * kMsgKeys + part * kPartKeys);
          tmem_ld_cols(scol, v);
        }
        tmem_wait_ld();
        if (j == kMsgsPerTile - 1) {
          // this warp has read its part of the S buffer
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(rank == 0 ? &sm.c.sfree[sb] : &sm.c.sread[sb]);
        }
        const int key0 = ui.k_lo + t * kTileKeys + j * kMsgKeys + part * kPartKeys;
        // raw scores; the scale (> 0) is applied in the exponent's fused multiply-add
        float x[kPartKeys];
#pragma unroll
        for (int k = 0; k < kPartKeys; ++k) x[k] = __uint_as_float(v[k]);
        if (!valid) {
#pragma unroll
          for (int k = 0; k < kPartKeys; ++k) x[k] = -INFINITY;
        } else if (key0 + kPartKeys > mask_from) {
#pragma unroll
          for (int k = 0; k < kPartKeys; ++k) {
            const int key = key0 + k;
            bool vis_k = key < ui.k_hi;
            if (vis_k && key >= ui.prefix) vis_k = ((vis >> (key - ui.prefix)) & 1ull) != 0;
            if (!vis_k) x[k] = -INFINITY;
          }
        }
        // row max over this thread's keys: four independent chains
        float mc[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
        for (int k = 4; k < kPartKeys; ++k) mc[k & 3] = fmaxf(mc[k & 3], x[k]);
        const float mh = fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3]));
        const int pb = msg & 1;  // double-buffered exchange slots (a thread may run one message ahead)
        S.pmax[pb][part][row] = mh;
        const bool last = t == ui.n_tiles - 1 && j == kMsgsPerTile - 1;
        const int sg = msg % kStages;  // staging buffer
        if (part == 0 && lane == 0) sm.c.wg_stop[wq][pb] = sm.c.abort_flag ? 1u : 0u;
        named_bar_sync(1 + wq, kPairThreads);  // the pair's partial maxima and stop decision visible
        if (sm.c.wg_stop[wq][pb]) {
          stop = true;
          break;
        }
        if (tid == 0 && j == 0) VTRACE(rank ? 15 : 14, it);
        float mraw = S.pmax[pb][0][row];
#pragma unroll
        for (int q = 1; q < kParts; ++q) mraw = fmaxf(mraw, S.pmax[pb][q][row]);
        const float mt = mraw * scale;
        float alpha = 1.f;
        if (mt > m_ref + kTau) {
          alpha = ex2_approx(m_ref - mt);  // 0 when m_ref = -inf
          l *= alpha;
          m_ref = mt;
        }
        // P of this thread's keys into registers (bf16 pairs) while the copy of message
        // msg - kStages may still be reading the staging buffer
        const float mref = m_ref == -INFINITY ? 0.f : m_ref;  // x = -inf there, so every p is 0
        uint32_t w[kPartKeys / 2];
        float ls[2] = {0.f, 0.f};
#pragma unroll
        for (int k = 0; k < kPartKeys / 2; ++k) {
          const float p0 = ex2_approx(fmaf(x[2 * k], scale, -mref));
          const float p1 = ex2_approx(fmaf(x[2 * k + 1], scale, -mref));
          ls[k & 1] += p0 + p1;
          w[k] = pack_bf16x2(p0, p1);
        }
        l += ls[0] + ls[1];
        // each warp waits for the staging buffer itself (lane 0); after a failed wait it
        // writes nothing, and its pair stops at the next message's barrier (the abort
        // flag is raised by the failed wait)
        bool free_ok = true;
        if (lane == 0 && msg >= kStages)
          free_ok = wait_bar(sm, &sm.c.stgfree[sg], ((msg - kStages) / kStages) & 1, a.status, 302);
        free_ok = __shfl_sync(0xffffffffu, free_ok ? 1 : 0, 0) != 0;
        if (free_ok) {
          // P row -> staging, 128-byte swizzle (16-byte granule g of row `row` at g ^ (row & 7));
          // this part owns granules kPartKeys/8 * part .. kPartKeys/8 * (part + 1) - 1
          uint8_t* prow = S.stage[sg].p + row * 128;
#pragma unroll
          for (int g = 0; g < kPartKeys / 8; ++g)
            *reinterpret_cast<uint4*>(prow + ((((kPartKeys / 8) * part + g) ^ (row & 7)) << 4)) =
                make_uint4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]);
          if (part == 0) S.stage[sg].alpha[row] = alpha;
        }
        const unsigned any = __ballot_sync(0xffffffffu, alpha != 1.f);
        if (lane == 0) sm.c.warp_flags[sg][sw] = any ? 1u : 0u;
        if (last) {
          // unit finals: running max and the row sum of all parts
          if (part > 0) S.lpart[part - 1][row] = l;
          named_bar_sync(1 + wq, kPairThreads);
          if (part == 0) {
            float lt = l;
#pragma unroll
            for (int q = 0; q < kParts - 1; ++q) lt += S.lpart[q][row];
            S.fin_stage[uu & 1].m[row] = m_ref;
            S.fin_stage[uu & 1].l[row] = lt;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.c.staged[sg]);
      }
    }
  }
}

// ------------------------------------------------------------------ ranks 0,1: P sender (warp 2+kSoftWarps, lane 0)
// Ships each staged message (and, after a unit's last message, the unit's
// finals) into the matching mixer CTA's receive slot, then reports when the
// copy has left the staging buffer.
__device__ void scorer_sender_role(TcSmem& sm, const PlanParams& plan, const TcSched& sched, const RunArgs& a,
                                   int u_begin, int u_end, uint32_t rank) {
  ScorerSmem& S = sm.u.s;
  const uint32_t mixer = rank + 2;
  int it = 0, uu = 0, msg = 0;
  for (int ui_idx = u_begin; ui_idx < u_end; ++ui_idx, ++uu) {
    const UnitInfo ui = unit_at(plan, sched, ui_idx);
    for (int t = 0; t < ui.n_tiles; ++t, ++it) {
      for (int j = 0; j < kMsgsPerTile; ++j, ++msg) {
        const int sg = msg % kStages;
        const int ms = msg % kPSlots;
        if (!wait_bar(sm, &sm.c.staged[sg], (msg / kStages) & 1, a.status, 310)) goto done;
        {
          uint32_t f = 0;
#pragma unroll
          for (int w = 0; w < kSoftWarps; ++w) f |= sm.c.warp_flags[sg][w];
          S.stage[sg].flags = f;
        }
        fence_proxy_async_smem();
        if (!wait_bar(sm, &sm.c.pfree[ms], ((msg / kPSlots) & 1) ^ 1, a.status, 311)) goto done;
        if (j == 0) VTRACE(rank ? 18 : 4, it);
        if (j == 1) VTRACE(rank ? 17 : 16, it);
        // into the mixer's receive slot (same offset in its view of shared memory)
        bulk_s2s_cluster(mapa(smem_u32(&sm.u.m.msg[ms]), mixer), smem_u32(&S.stage[sg]), kMsgBytes,
                         mapa(smem_u32(&sm.c.pfull[ms]), mixer));
        if (t == ui.n_tiles - 1 && j == kMsgsPerTile - 1) {
          // the mixer's finals buffer uu & 1 was read for unit uu - 2 (short units let this
          // thread run two units ahead of the mixer's epilogue)
          if (uu >= 2 && !wait_bar(sm, &sm.c.finfree[uu & 1], ((uu - 2) >> 1) & 1, a.status, 312)) {
            bulk_commit_group();
            goto done;
          }
          bulk_s2s_cluster(mapa(smem_u32(&sm.u.m.fin[uu & 1]), mixer), smem_u32(&S.fin_stage[uu & 1]),
                           sizeof(Finals), mapa(smem_u32(&sm.c.finfull[uu & 1]), mixer));
        }
        bulk_commit_group();
        if (msg >= kStages - 1) {
          // the copy issued kStages - 1 messages ago has finished reading its staging buffer
          bulk_wait_group_read<kStages - 1>();
          mbar_arrive(&sm.c.stgfree[(msg - (kStages - 1)) % kStages]);
        }
      }
    }
  }
done:
  // every copy this thread issued has been written into the mixer (not only read
  // from the staging buffer) before the CTA may reach the final cluster barrier
  bulk_wait_group<0>();
}

// ------------------------------------------------------------------ rank 1: S-buffer release forwarder (warp 1, lane 0)
// One remote arrive per tile on rank 0's S-buffer barrier once this CTA's
// softmax warps have read the buffer (keeps the cluster-scope release off the
// softmax warps).
__device__ void scorer_forward_role(TcSmem& sm, const RunArgs& a, int total) {
  for (int n = 0; n < total; ++n) {
    if (!wait_bar(sm, &sm.c.sread[n & 1], (n >> 1) & 1, a.status, 320)) return;
    mbar_arrive_remote(mapa(smem_u32(&sm.c.sfree[n & 1]), 0));
  }
}

// ------------------------------------------------------------------ rank 2: P V issuer (warp 1, lane 0)
// Per message (64 keys): 4 key steps x 2 value halves of M256 x N256 x K16
// MMAs, A = P (K-major, 128 rows in each mixer CTA), B = value columns of the
// message's 64 rows of the tile stage (MN-major view of the 128-byte-swizzled
// chunks: leading byte offset = chunk stride).
__device__ void mixer_mma_role(TcSmem& sm, const PlanParams& plan, const TcSched& sched, const RunArgs& a,
                               uint32_t tbase, int u_begin, int u_end) {
  constexpr uint32_t idesc = idesc_bf16_f32(kRowsUnit, 256, 0, 1);
  MixerSmem& M = sm.u.m;
  const uint32_t peer_cmd = mapa(smem_u32(&sm.c.cmd), 3);
  const uint32_t peer_cmd_full = mapa(smem_u32(&sm.c.cmd_full), 3);
  int it = 0, msg = 0, cmdn = 0, obn = 0;
  bool ok = true;
  auto post = [&](uint32_t c) {
    sm.c.cmd = c;
    st_cluster_u32(peer_cmd, c);
    mbar_arrive(&sm.c.cmd_full);
    mbar_arrive_remote(peer_cmd_full);
  };
  auto command = [&](uint32_t c) -> bool {
    post(c);
    const bool r = wait_bar(sm, &sm.c.cmd_done, cmdn & 1, a.status, 402);
    ++cmdn;
    return r;
  };
  auto quiesce = [&]() -> bool {
    mma_commit_pair(&sm.c.obar, kMixerMask);
    const bool r = wait_bar(sm, &sm.c.obar, obn & 1, a.status, 403);
    ++obn;
    return r;
  };
  for (int ui_idx = u_begin; ui_idx < u_end && ok; ++ui_idx) {
    const UnitInfo ui = unit_at(plan, sched, ui_idx);
    for (int t = 0; t < ui.n_tiles && ok; ++t, ++it) {
      for (int j = 0; j < kMsgsPerTile; ++j, ++msg) {
        const int s = msg % kVStages;  // V stage of this message
        if (!wait_bar(sm, &sm.c.kfull[s], (msg / kVStages) & 1, a.status, 400)) {
          ok = false;
          break;
        }
        if (j == 0) VTRACE(6, it);
        const int ps = msg % kPSlots;
        if (!wait_bar(sm, &sm.c.pfull[ps], (msg / kPSlots) & 1, a.status, 401)) {
          ok = false;
          break;
        }
        if (j == 0) VTRACE(7, it);
        if (j == 1) VTRACE(19, it);
        if ((t > 0 || j > 0) && ((M.msg[ps].flags | sm.c.peer_flags[ps]) & 1u)) {
          if (!quiesce() || !command(kCmdRescale | ((uint32_t)ps << 8))) {
            ok = false;
            break;
          }
        }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kMsgKeys / 16; ++k) {
          const uint64_t adesc = smem_desc(smem_u32(M.msg[ps].p) + k * 32, 16, 1024);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const uint64_t bdesc = smem_desc(smem_u32(&M.v[s][2 * hh][0]) + k * 16 * 128, kKBox, 1024);
            mma_pair_ss(tbase + (uint32_t)(256 * hh), adesc, bdesc, idesc, (t > 0 || j > 0 || k > 0) ? 1u : 0u);
          }
        }
        mma_commit_pair(&sm.c.pdone[ps], kMixerMask);
        mma_commit_pair(&sm.c.kfree[s], kMixerMask);
      }
      if (!ok) break;
      VTRACE(8, it);
    }
    if (!ok) break;
    // the epilogue group waits for this commit itself, so the command travels
    // while the unit's last products finish
    mma_commit_pair(&sm.c.obar, kMixerMask);
    ++obn;
    VTRACE(24, ui_idx - u_begin);  // epilogue command posted
    if (!command(kCmdEpilogue)) ok = false;
    VTRACE(25, ui_idx - u_begin);  // epilogue done
  }
  if (!ok) {
    // after a failed wait: the last commit goes to this CTA only and is waited for
    // regardless of the abort flag, so no arrival of this pair's earlier commits is
    // still travelling when the cluster leaves
    mma_commit_pair(&sm.c.obar, (uint16_t)0x4);
    drain_bar(sm, &sm.c.obar, obn & 1, a.status, 405);
  }
  post(kCmdExit);
}

// ------------------------------------------------------------------ rank 3: relay (warp 1, lane 0)
// Forwards each P arrival of this CTA (and its rescale flag) to rank 2, whose
// MMA reads both CTAs' halves of the message.
__device__ void mixer_relay_role(TcSmem& sm, const RunArgs& a, int total_msgs) {
  for (int n = 0; n < total_msgs; ++n) {
    const int s = n % kPSlots;
    if (!wait_bar(sm, &sm.c.pfull[s], (n / kPSlots) & 1, a.status, 700)) return;
    st_cluster_u32(mapa(smem_u32(&sm.c.peer_flags[s]), 2), sm.u.m.msg[s].flags);
    mbar_arrive_remote(mapa(smem_u32(&sm.c.pfull[s]), 2));
    VTRACE(13, n);
  }
}

// ------------------------------------------------------------------ ranks 2,3: P-slot release (warp 6, lane 0)
__device__ void mixer_release_role(TcSmem& sm, const RunArgs& a, int total_msgs, uint32_t rank) {
  const uint32_t scorer = rank - 2;
  for (int n = 0; n < total_msgs; ++n) {
    const int s = n % kPSlots;
    if (!wait_bar(sm, &sm.c.pdone[s], (n / kPSlots) & 1, a.status, 500)) return;
    if (rank == 2) VTRACE(9, n);
    if (n + kPSlots < total_msgs) {
      mbar_arrive_expect_tx(&sm.c.pfull[s], kMsgBytes);
      mbar_arrive_remote(mapa(smem_u32(&sm.c.pfree[s]), scorer));
    }
  }
}

// ------------------------------------------------------------------ ranks 2,3: rescale / epilogue (warps 2-5, 7-10)
// Two groups of four warps, one warp of each per TMEM lane quarter; group g
// owns value columns [256g, 256g + 256).  Thread 0 of group 0 takes each
// command and broadcasts it to the 256 threads.
constexpr int kEpiThreads = 256;
__device__ __forceinline__ int epi_gran(int row, int k) { return k ^ ((row >> 1) & 3); }  // conflict-free both ways

__device__ void mixer_epilogue_role(TcSmem& sm, const CUtensorMap* omap, const CUtensorMap* pmap,
                                    const PlanParams& plan, const TcSched& sched, const RunArgs& a, uint32_t tbase,
                                    int u_begin, int u_end, uint32_t rank) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp >= 7 ? 1 : 0;
  const int wq = warp & 3;
  const int row = wq * 32 + lane;
  const int tid = grp ? threadIdx.x - 224 + 128 : threadIdx.x - 64;
  const int ew = grp * 4 + (warp - (grp ? 7 : 2));  // epilogue warp 0..7 (its staging tile)
  const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
  const uint32_t col0 = (uint32_t)grp * (kDv / 2);
  const int H = plan.num_heads;
  MixerSmem& M = sm.u.m;
  const uint32_t lead_cmd_done = mapa(smem_u32(&sm.c.cmd_done), 2);
  int cmdn = 0, uu = 0, qn = 0;
  int ui_idx = u_begin;
  for (;;) {
    // thread 0 waits for the command, for the MMAs it follows (both CTAs'
    // tensor memory is written by rank 2's MMAs) and, for an epilogue, for the
    // unit's finals; the group learns the outcome at a barrier
    if (tid == 0) {
      uint32_t cmd = kCmdExit;
      if (wait_bar(sm, &sm.c.cmd_full, cmdn & 1, a.status, 600)) {
        cmd = sm.c.cmd;
        const uint32_t op = cmd & 0xFF;
        if (op == kCmdRescale || op == kCmdEpilogue) {
          if (!wait_bar(sm, &sm.c.obar, qn & 1, a.status, 602)) cmd = kCmdExit;
          ++qn;
        }
        if ((cmd & 0xFF) == kCmdEpilogue && ui_idx >= u_end) {
          // an epilogue with no unit left in this cluster's list: the command protocol is broken
          record_status(a.status, VMLA_ERR_TIMEOUT, 603u);
          cmd = kCmdExit;
        }
        if ((cmd & 0xFF) == kCmdEpilogue && !wait_bar(sm, &sm.c.finfull[uu & 1], (uu >> 1) & 1, a.status, 601))
          cmd = kCmdExit;
      }
      sm.c.wg_cmd = cmd;
    }
    ++cmdn;
    named_bar_sync(2, kEpiThreads);
    const uint32_t cmd = sm.c.wg_cmd;
    if ((cmd & 0xFF) == kCmdExit) {
      if (lane == 0) bulk_wait_group<0>();  // this warp's output stores are written before the CTA leaves
      if (tid == 0 && rank == 2) VTRACE_CLUSTER(29);  // the last unit's outputs written
      return;
    }
    __syncwarp();
    tc_fence_after();
    // tcgen05.ld / st are warp-collective: every branch around them is warp-uniform
    if ((cmd & 0xFF) == kCmdRescale) {
      const int s = (int)((cmd >> 8) & 0xFFu);
      const float alpha = M.msg[s].alpha[row];
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int c = 0; c < kDv / 64; ++c) {
          const uint32_t col = col0 + (uint32_t)(c * 32);
          uint32_t v[32];
          tmem_ld32(tbase + lane_base + col, v);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
          tmem_st32(tbase + lane_base + col, v);
        }
        tmem_wait_st();
      }
    } else {
      if (tid == 0 && rank == 2) VTRACE(22, uu);  // epilogue of unit uu starts
      // epilogue of unit ui_idx: O / l -> output row (or fp32 partial).  Each chunk
      // of the warp's 32 rows (64 bytes of each) goes through its shared-memory
      // tile, laid out as a 64-byte-swizzled box, and leaves as one tiled TMA
      // store; a group of 32 rows that runs past the unit's rows is stored by the
      // lanes instead (eight rows' 64 contiguous bytes per instruction), so that
      // nothing is written past them.
      const UnitInfo ui = unit_at(plan, sched, ui_idx);
      const SeqPlan& sp = plan.seq[ui.b];
      const int f = uu & 1;
      const float m = M.fin[f].m[row], lsum = M.fin[f].l[row];
      const int r = ui.rb * kRowsUnit + (int)(rank & 1) * kRowsCta + row;
      const bool valid = r < ui.R;
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
      const float lse2 = lsum > 0.f ? m + log2f(lsum) : -INFINITY;
      uint4(*tile)[4] = M.ep[ew];
      const uint32_t tile_s = smem_u32(&M.ep[ew][0][0]);
      const int r_w = ui.rb * kRowsUnit + (int)(rank & 1) * kRowsCta + wq * 32;  // query row of lane 0
      const bool whole = r_w + 32 <= ui.R;        // all 32 rows of the group belong to the unit
      const int sub = lane >> 2, k4 = lane & 3;  // lane store phase: rows 8i + sub, granule k4
      // the tile is rewritten only after the previous store has read it
      auto tile_free = [&]() {
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
      };
      auto tile_out = [&](const CUtensorMap* map, int x, int64_t y, auto* base) {
        fence_proxy_async_smem();
        __syncwarp();
        if (whole) {
          if (lane == 0) {
            tma_store_2d(map, tile_s, x, (int)y);
            bulk_commit_group();
          }
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int rr = 8 * i + sub;
            if (r_w + rr < ui.R)
              reinterpret_cast<uint4*>(base + (y + rr) * kDv + x)[k4] = tile[rr][epi_gran(rr, k4)];
          }
          __syncwarp();
        }
      };
      if (ui.n_pieces == 1) {
        const int64_t orow = (int64_t)sp.q_off * H + (valid ? r : 0);
        const int64_t orow_w = (int64_t)sp.q_off * H + r_w;
#pragma unroll 1
        for (int c = 0; c < kDv / 64; ++c) {  // 32 columns = 64 bytes of bf16 per row
          const uint32_t col = col0 + (uint32_t)(c * 32);
          uint32_t v[32];
          tmem_ld32(tbase + lane_base + col, v);
          tmem_wait_ld();
          tile_free();
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tile[lane][epi_gran(lane, k)] = make_uint4(
                pack_bf16x2(__uint_as_float(v[8 * k]) * inv, __uint_as_float(v[8 * k + 1]) * inv),
                pack_bf16x2(__uint_as_float(v[8 * k + 2]) * inv, __uint_as_float(v[8 * k + 3]) * inv),
                pack_bf16x2(__uint_as_float(v[8 * k + 4]) * inv, __uint_as_float(v[8 * k + 5]) * inv),
                pack_bf16x2(__uint_as_float(v[8 * k + 6]) * inv, __uint_as_float(v[8 * k + 7]) * inv));
          tile_out(omap, (int)col, orow_w, a.out);
        }
        if (valid && grp == 0) a.lse[orow] = lsum > 0.f ? lse2 * 0.6931471805599453f : -INFINITY;
      } else {
        const int64_t prow = (int64_t)sp.part_off + (int64_t)ui.piece * ui.R + (valid ? r : 0);
        const int64_t prow_w = (int64_t)sp.part_off + (int64_t)ui.piece * ui.R + r_w;
#pragma unroll 1
        for (int c = 0; c < kDv / 32; ++c) {  // 16 columns = 64 bytes of fp32 per row
          const uint32_t col = col0 + (uint32_t)(c * 16);
          uint32_t v[16];
          tmem_ld16(tbase + lane_base + col, v);
          tmem_wait_ld();
          tile_free();
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tile[lane][epi_gran(lane, k)] = make_uint4(__float_as_uint(__uint_as_float(v[4 * k]) * inv),
                                                       __float_as_uint(__uint_as_float(v[4 * k + 1]) * inv),
                                                       __float_as_uint(__uint_as_float(v[4 * k + 2]) * inv),
                                                       __float_as_uint(__uint_as_float(v[4 * k + 3]) * inv));
          tile_out(pmap, (int)col, prow_w, a.part_o);
        }
        if (valid && grp == 0) a.part_lse[prow] = lse2;
      }
      if (tid == 0 && rank == 2) VTRACE(23, uu);  // (thread 0's share of) the epilogue stored
      ++uu;
      ++ui_idx;
    }
    tc_fence_before();
    named_bar_sync(2, kEpiThreads);
    if (tid == 0) {
      // a finals buffer is re-armed for the unit two ahead once it has been read,
      // then handed back to the scorer
      if ((cmd & 0xFF) == kCmdEpilogue) {
        if (ui_idx + 1 < u_end) mbar_arrive_expect_tx(&sm.c.finfull[(uu + 1) & 1], sizeof(Finals));
        mbar_arrive_remote(mapa(smem_u32(&sm.c.finfree[(uu + 1) & 1]), rank - 2));
      }
      if (rank == 2) mbar_arrive(&sm.c.cmd_done);
      else mbar_arrive_remote(lead_cmd_done);
    }
  }
}

// The kernel body; `plan` and `sched` are kernel parameters (host-planned
// calls) or live in the workspace (device-planned calls).
__device__ __forceinline__ void tc_verify_body(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                               const CUtensorMap& qmap, const CUtensorMap& omap,
                                               const CUtensorMap& pmap, const PlanParams& plan,
                                               const TcSched& sched, const RunArgs& a) {
  extern __shared__ uint8_t smem_raw[];
  TcSmem& sm = *reinterpret_cast<TcSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cid = (int)cluster_id_x();
  // this cluster's work list: positions [u_begin, u_end) of the schedule's order,
  // or the streams its lane meets
  int u_begin = 0, u_end = 0;
  if (cid < sched.num_clusters) {
    if (plan.lane_width == 0) {
      u_begin = sched.start[cid];
      u_end = sched.start[cid + 1];
    } else {
      lane_streams(plan, cid / plan.lane_width, &u_begin, &u_end);
    }
  }
  if (threadIdx.x == 0 && rank == 0) VTRACE_CLUSTER(26);  // cluster entered

  if (threadIdx.x == 0) {
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&sm.c.kfull[s], 1);
      mbar_init(&sm.c.kfree[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.c.sfull[s], 1);
      mbar_init(&sm.c.sfree[s], kSoftWarps + 1);  // rank 0's softmax warps + rank 1's forwarder
      mbar_init(&sm.c.sread[s], kSoftWarps);
      mbar_init(&sm.c.finfull[s], 1);
      mbar_init(&sm.c.finfree[s], 1);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.c.staged[s], kSoftWarps);
      mbar_init(&sm.c.stgfree[s], 1);
    }
    for (int s = 0; s < kPSlots; ++s) {
      mbar_init(&sm.c.pfull[s], rank == 2 ? 2 : 1);  // rank 2: own arming + rank 3's relay
      mbar_init(&sm.c.pfree[s], 1);
      mbar_init(&sm.c.pdone[s], 1);
      sm.c.peer_flags[s] = 0;
    }
    mbar_init(&sm.c.qfull, 2 * kSoftWarps);  // every softmax warp of both scorer CTAs
    mbar_init(&sm.c.qland, 1);
    mbar_init(&sm.c.qfree, kSoftWarps);
    mbar_init(&sm.c.cmd_full, 1);
    mbar_init(&sm.c.cmd_done, 2);
    mbar_init(&sm.c.obar, 1);
    sm.c.abort_flag = 0;
    sm.c.wait_cycles = a.wait_cycles;
    fence_mbar_init();
    prefetch_tensormap(&kmap);
    if (rank >= 2) {
      prefetch_tensormap(&vmap);
      prefetch_tensormap(&omap);
      prefetch_tensormap(&pmap);
    } else {
      prefetch_tensormap(&qmap);
    }
  }
  __syncwarp();
  if (warp == 0) {
    tmem_alloc_pair(&sm.c.tmem_base, 512);
    tmem_relinquish_pair();
  }
  const int n_tiles_all = total_tiles(plan, sched, u_begin, u_end);
  const int total_msgs = kMsgsPerTile * n_tiles_all;
  // every barrier object is initialised before any thread of this CTA arms or
  // waits on one (the arming below runs in another warp than the initialisation)
  __syncthreads();
  if (rank >= 2 && threadIdx.x == 64) {  // thread 0 of the epilogue group
    // receive slots and finals buffers armed before the partner can send
    const int n_units = u_end - u_begin;
    for (int s = 0; s < kPSlots && s < total_msgs; ++s) mbar_arrive_expect_tx(&sm.c.pfull[s], kMsgBytes);
    for (int s = 0; s < 2 && s < n_units; ++s) mbar_arrive_expect_tx(&sm.c.finfull[s], sizeof(Finals));
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_arrive();
  cluster_wait();
  const uint32_t tbase = sm.c.tmem_base;
  if (threadIdx.x == 0 && rank == 0) {
    VTRACE_CLUSTER(27);  // set up (barriers, TMEM, receive slots armed)
    VTRACE_CLUSTER_VALUE(31, ((uint64_t)(u_end - u_begin) << 32) | (uint32_t)n_tiles_all);
  }

  if (warp == 0) {
    if (lane == 0) producer_role(sm, &kmap, &vmap, &qmap, plan, sched, a, u_begin, u_end, rank);
  } else if (warp == 1) {
    if (lane == 0) {
      if (rank == 0) scorer_mma_role(sm, plan, sched, a, tbase, u_begin, u_end);
      else if (rank == 2) mixer_mma_role(sm, plan, sched, a, tbase, u_begin, u_end);
      else if (rank == 3) mixer_relay_role(sm, a, total_msgs);
      else scorer_forward_role(sm, a, n_tiles_all);
    }
  } else if (rank < 2) {
    if (warp == kSenderWarp) {
      if (lane == 0) scorer_sender_role(sm, plan, sched, a, u_begin, u_end, rank);
    } else {
      scorer_softmax_role(sm, plan, sched, a, tbase, u_begin, u_end, rank);
    }
  } else if (warp == 6) {
    if (lane == 0) mixer_release_role(sm, a, total_msgs, rank);
  } else {
    mixer_epilogue_role(sm, &omap, &pmap, plan, sched, a, tbase, u_begin, u_end, rank);  // warps 2-5 and 7-10
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  // this CTA's work is done: the merge may be scheduled as CTAs retire (it waits
  // for the whole grid before it reads the partials)
  grid_dependents_launch();
  __syncwarp();
  // no CTA leaves while another may still address its shared or tensor memory.
  // Past this barrier no thread of the cluster issues anything.  On the normal
  // path every arrival into this CTA has been waited for by now (tile loads,
  // stage releases, P and finals copies, MMA commits).  After a failed wait some
  // of those waits were cut short, so the CTA first lets whatever was issued
  // land; all four CTAs read the same abort flag here, since a failed wait
  // raises it in every CTA of the cluster before the barrier.
  cluster_arrive();
  cluster_wait();
  if (threadIdx.x == 0 && rank == 0) VTRACE_CLUSTER(30);  // every role of the cluster finished
  if (sm.c.abort_flag) {
    if (threadIdx.x == 0) settle_after_abort();
    __syncthreads();
  }
  __syncwarp();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(tbase, 512);
  }
}

__global__ void __launch_bounds__(kThreadsTC, 1)
tc_verify_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                 const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
                 const __grid_constant__ CUtensorMap pmap, const __grid_constant__ PlanParams plan,
                 const __grid_constant__ TcSched sched, const RunArgs a) {
  tc_verify_body(kmap, vmap, qmap, omap, pmap, plan, sched, a);
}

// Same kernel with the plan and the cluster schedule read from the workspace,
// where the device planner wrote them (stream-capture-safe calls).
__global__ void __launch_bounds__(kThreadsTC, 1)
tc_verify_kernel_dplan(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                       const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
                       const __grid_constant__ CUtensorMap pmap, const PlanParams* __restrict__ plan,
                       const TcSched* __restrict__ sched, const RunArgs a) {
  // started early behind a kernel that itself may still wait for the planner: the plan
  // and the schedule are read only once everything before this launch is complete
  grid_dependency_wait();
  tc_verify_body(kmap, vmap, qmap, omap, pmap, *plan, *sched, a);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

constexpr size_t kSmemBytes = sizeof(TcSmem) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(sizeof(PlanParams) + sizeof(TcSched) + sizeof(RunArgs) + 5 * sizeof(CUtensorMap) < 32000,
              "kernel parameter budget");

// attr: room for two attributes (the cluster shape, and an early start under
// the previous kernel's tail when `early` is set)
cudaLaunchConfig_t cluster_config(int clusters, cudaLaunchAttribute* attr, bool early = false) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kClusterCtas * clusters, 1, 1);
  cfg.blockDim = dim3(kThreadsTC, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kClusterCtas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  if (early) attr[1] = early_start_attribute();
  cfg.attrs = attr;
  cfg.numAttrs = early ? 2 : 1;
  return cfg;
}

bool encode_rows(EncodeTiledFn enc, CUtensorMap* map, void* base, int64_t rows, uint32_t box_rows) {
  cuuint64_t gdim[2] = {(cuuint64_t)kDqk, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t gstride[1] = {(cuuint64_t)kRowBytes};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estride[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, gdim, gstride, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over staged rows [rows x 576 bf16] seen as (64 columns, row, column
// chunk) with strides 1152 B (row) and 128 B (chunk): a box of `box_rows` rows x
// `box_chunks` chunks lands chunk-major in shared memory, each chunk a
// 128-byte-swizzled [box_rows x 64] block, as the MMA descriptors expect.
bool encode_rows_chunks(EncodeTiledFn enc, CUtensorMap* map, void* base, int64_t rows, uint32_t box_rows,
                        uint32_t box_chunks) {
  cuuint64_t gdim[3] = {64, (cuuint64_t)(rows > 0 ? rows : 1), (cuuint64_t)kChunks};
  cuuint64_t gstride[2] = {(cuuint64_t)kRowBytes, 128};
  cuuint32_t box[3] = {64, box_rows, box_chunks};
  cuuint32_t estride[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, gdim, gstride, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output maps of the epilogue: [rows x 512] of bf16 outputs or fp32 partials,
// boxes of 32 rows x 64 bytes with 64-byte swizzle (the epilogue tiles' layout).
bool encode_out(EncodeTiledFn enc, CUtensorMap* map, void* base, int64_t rows, bool fp32) {
  cuuint64_t gdim[2] = {(cuuint64_t)kDv, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t gstride[1] = {(cuuint64_t)kDv * (fp32 ? 4 : 2)};
  cuuint32_t box[2] = {fp32 ? 16u : 32u, 32};
  cuuint32_t estride[2] = {1, 1};
  return enc(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, gdim, gstride,
             box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The five maps of a launch (staged KV rows for the scorer's K boxes and the
// mixer's V boxes, Q rows [query rows x heads x 576], outputs, partials);
// without partial rows the partial map repeats the output map (no unit of
// such a plan stores partials).
bool encode_maps(EncodeTiledFn enc, const RunArgs& a, CUtensorMap* kmap, CUtensorMap* vmap, CUtensorMap* qmap,
                 CUtensorMap* omap, CUtensorMap* pmap) {
  if (!encode_rows_chunks(enc, kmap, a.staged, a.total_kv, kHalfKeys, kChunks)) return false;
  if (!encode_rows_chunks(enc, vmap, a.staged, a.total_kv, kMsgKeys, 2)) return false;
  if (!encode_rows(enc, qmap, const_cast<uint16_t*>(a.q), a.out_rows, 64)) return false;
  if (!encode_out(enc, omap, a.out, a.out_rows, false)) return false;
  if (a.part_rows > 0 && a.part_o) return encode_out(enc, pmap, a.part_o, a.part_rows, true);
  *pmap = *omap;
  return true;
}

}  // namespace

int tc_max_clusters(int* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return VMLA_ERR_CUDA;
  static int cached[64] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> g(mu);
  if (dev < 64 && cached[dev] > 0) {
    *out = cached[dev];
    return VMLA_OK;
  }
  if (cudaFuncSetAttribute(tc_verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
          cudaSuccess ||
      cudaFuncSetAttribute(tc_verify_kernel_dplan, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
          cudaSuccess)
    return VMLA_ERR_CUDA;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = cluster_config(1, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, tc_verify_kernel, &cfg) != cudaSuccess || n < 1) return VMLA_ERR_CUDA;
  if (dev < 64) cached[dev] = n;
  *out = n;
  return VMLA_OK;
}

int launch_tc(const PlanParams& plan, const RunArgs& a, void* stream) {
  if (plan.total_units == 0) return VMLA_OK;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return VMLA_ERR_DEVICE;
  int clusters = 0;
  int rc = tc_max_clusters(&clusters);
  if (rc != VMLA_OK) return rc;
  clusters = clusters < kMaxClusters ? clusters : kMaxClusters;
  // 2-D map over the staged rows [total_kv x 576 bf16]: boxes of 64 rows x 64
  // columns with 128-byte swizzle (scorer half tiles, mixer message chunks),
  // and the epilogue's output maps
  CUtensorMap kmap, vmap, qmap, omap, pmap;
  if (!encode_maps(enc, a, &kmap, &vmap, &qmap, &omap, &pmap)) return VMLA_ERR_CUDA;
  static thread_local TcSched sched;
  if (plan.lane_width > 0) {
    // a lane plan: one launch of lane_count lanes, each cluster working out its own streams
    std::memset(&sched, 0, sizeof(sched));
    sched.num_clusters = plan.lane_count * plan.lane_width;
    sched.total_units = plan.total_units;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = cluster_config(sched.num_clusters, attr, true);
    cfg.stream = (cudaStream_t)stream;
    if (cudaLaunchKernelEx(&cfg, tc_verify_kernel, kmap, vmap, qmap, omap, pmap, plan, sched, a) != cudaSuccess)
      return VMLA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? VMLA_OK : VMLA_ERR_CUDA;
  }
  // units are independent: a plan with more than kMaxTcUnits runs as several launches
  for (int u0 = 0; u0 < plan.total_units; u0 += kMaxTcUnits) {
    const int u1 = plan.total_units - u0 < kMaxTcUnits ? plan.total_units : u0 + kMaxTcUnits;
    rc = build_tc_schedule(plan, clusters < u1 - u0 ? clusters : u1 - u0, u0, u1, &sched);
    if (rc != VMLA_OK) return rc;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = cluster_config(sched.num_clusters, attr, true);
    cfg.stream = (cudaStream_t)stream;
    if (cudaLaunchKernelEx(&cfg, tc_verify_kernel, kmap, vmap, qmap, omap, pmap, plan, sched, a) != cudaSuccess)
      return VMLA_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? VMLA_OK : VMLA_ERR_CUDA;
}

int launch_tc_dplan(const PlanParams* plan, const TcSched* sched, int clusters, const RunArgs& a, void* stream) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return VMLA_ERR_DEVICE;
  int dev_clusters = 0;
  int rc = tc_max_clusters(&dev_clusters);
  if (rc != VMLA_OK) return rc;
  if (clusters < 1 || clusters > dev_clusters || clusters > kMaxClusters) return VMLA_ERR_SHAPE;
  // the maps span the staged, output and partial areas' capacities; the planned
  // keys and rows lie inside them
  CUtensorMap kmap, vmap, qmap, omap, pmap;
  if (!encode_maps(enc, a, &kmap, &vmap, &qmap, &omap, &pmap)) return VMLA_ERR_CUDA;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = cluster_config(clusters, attr, true);
  cfg.stream = (cudaStream_t)stream;
  if (cudaLaunchKernelEx(&cfg, tc_verify_kernel_dplan, kmap, vmap, qmap, omap, pmap, plan, sched, a) != cudaSuccess)
    return VMLA_ERR_CUDA;
  return VMLA_OK;
}

}  // namespace vmla

#ifdef VMLA_TRACE
extern "C" int vmla_trace_read(uint64_t* host, int n) {
  const int total = vmla::kTraceEvents * vmla::kTraceTiles;
  if (n > total) n = total;
  return cudaMemcpyFromSymbol(host, vmla::g_vmla_trace, sizeof(uint64_t) * n) == cudaSuccess ? n : -1;
}
extern "C" int vmla_trace_clusters(void) {
  int n = 0;
  return vmla::tc_max_clusters(&n) == VMLA_OK ? n : -1;
}
extern "C" int vmla_trace_clear(void) {
  static uint64_t zeros[vmla::kTraceEvents * vmla::kTraceTiles] = {};
  return cudaMemcpyToSymbol(vmla::g_vmla_trace, zeros, sizeof zeros) == cudaSuccess ? 0 : -1;
}
#endif
