// Tensor-core verify attention for sm_103a: tcgen05 MMAs with TMEM
// accumulators, KV rows gathered by TMA (tile::gather4) at page_size = 1.
//
// The method is the KV-split flash-decode of "The Build That Unlocked 3-6x
// Decode Speedup", section "The Context: A Custom Kernel for an Unsupported
// Architecture": KV tiles streamed through shared memory, online softmax, and
// one read of each KV tile shared by many query rows.  The pages share a tile
// across a head tile of 8 heads (section "Context: The Long Road to a Custom
// sm_120 Kernel" of "The Build Script Edit"); here a tile serves 128 query
// rows (heads x draft positions of one sequence) in a single MMA.
//
// A work unit is 128 query rows (r = i*H + h) of one sequence over one
// contiguous piece of its key range, and runs on a cluster of two CTAs:
//   CTA 0 ("scorer")  keeps Q [128 x 576] in tensor memory (A operand),
//                     computes S = Q K^T for 64-key tiles into double-buffered
//                     TMEM columns, runs the online softmax (one thread per
//                     row), and ships P (bf16, 128 x 64) plus per-row rescale
//                     factors to CTA 1 by a shared-memory bulk copy.
//   CTA 1 ("mixer")   keeps O [128 x 512] fp32 in tensor memory and computes
//                     O = alpha * O + P V with V the latent part of the same
//                     gathered rows, then normalises and writes the result.
// The split of the work follows from tensor-memory capacity: O for 128 rows
// fills one SM's 512 TMEM columns, so Q and S live on the partner SM.
//
// Warp roles (320 threads): warp 0 TMA producer, warp 1 MMA issuer; CTA 0:
// warps 2-9 softmax, two threads per row (each 32 of the tile's 64 keys);
// CTA 1: warps 2-5 rescale/epilogue, warp 6 P-slot release.
// Every wait is bounded; on expiry the kernel records VMLA_ERR_TIMEOUT in the
// status word, tells the partner CTA to stop, drains its own copies and MMAs,
// frees tensor memory and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "vmla_device.cuh"
#include "vmla_sm100.cuh"

namespace vmla {
using namespace sm100;
namespace {

constexpr int kTileKeys = 64;
constexpr int kChunks = kDqk / 64;   // 9 column chunks of 64 bf16 (128 bytes) per row
constexpr int kVChunks = kDv / 64;   // 8 of them are the latent / value part
constexpr int kChunkBytes = kTileKeys * 128;
constexpr int kStages = 2;
constexpr int kRowsTC = 128;
constexpr int kThreadsTC = 320;      // 10 warps
constexpr uint32_t kSCol = 384;      // S buffers at TMEM columns 384 and 448 (Q uses 0..287)
constexpr float kTau = 8.0f;         // the running max is raised only when a tile exceeds it by 2^8
constexpr long long kWaitCycles = 2000000000LL;  // ~1 s at 2 GHz
constexpr int kPrefetchTiles = 6;  // tiles the scorer's producer prefetches into L2 ahead of its loads

enum Cmd : uint32_t { kCmdRescale = 1, kCmdEpilogue = 2, kCmdExit = 3 };

// Optional pipeline trace (compile with -DVMLA_TRACE): global-timer stamps of
// each hand-off for the first kTraceTiles tiles of cluster 0.
#ifdef VMLA_TRACE
constexpr int kTraceTiles = 256;
constexpr int kTraceEvents = 12;
__device__ uint64_t g_vmla_trace[kTraceEvents * kTraceTiles];
__device__ __forceinline__ void vtrace(int ev, int tile) {
  if (cluster_id_x() == 0 && tile < kTraceTiles) {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    g_vmla_trace[ev * kTraceTiles + tile] = t;
  }
}
#define VTRACE(ev, tile) vtrace(ev, tile)
#else
#define VTRACE(ev, tile) ((void)0)
#endif

struct __align__(1024) PMsg {
  uint8_t p[kRowsTC * 128];  // P [128 rows][64 keys] bf16, K-major, 128-byte swizzle
  float alpha[kRowsTC];      // factor for O rows before this tile's product (1 = unchanged)
  uint32_t flags;            // bit 0: some alpha differs from 1
  uint32_t pad[3];
};
constexpr uint32_t kMsgBytes = kRowsTC * 128 + kRowsTC * 4 + 16;  // bytes shipped per message

struct __align__(16) Finals {
  float m[kRowsTC];  // running max (log2 units)
  float l[kRowsTC];  // softmax denominator relative to m
};

struct TcSmem {
  uint8_t kv[kStages][kChunks][kChunkBytes];  // gathered rows, 128-byte swizzled chunks
  PMsg msg[2];                                // CTA 0: staging; CTA 1: receive slots
  Finals fin_stage[2];                        // CTA 0 staging of per-unit finals
  Finals fin[2];                              // CTA 1 receive
  uint64_t kfull[kStages], kfree[kStages];
  uint64_t sfull[2], sfree[2];
  uint64_t qfull;
  uint64_t pfull[2], pfree[2], pdone[2];
  uint64_t finfull[2];
  uint64_t cmd_full, cmd_done, obar;
  uint32_t cmd;
  uint32_t tmem_base;
  volatile int32_t abort_flag;
  uint32_t warp_flags[8];
  float pmax[2][kRowsTC];     // CTA 0: per-half partial row maxima of the current tile
  float lpart[kRowsTC];       // CTA 0: second half's row sums at a unit's last tile
  volatile uint32_t wg_stop;  // CTA 0 softmax group: stop after this tile
  volatile uint32_t wg_cmd;   // CTA 1 epilogue group: command broadcast
};

struct UnitInfo {
  int b, rb, piece, R, prefix, k_lo, k_hi, n_tiles;
};

__device__ __forceinline__ UnitInfo decode_unit(const PlanParams& p, int u) {
  UnitInfo ui;
  ui.b = seq_of_unit(p, u);
  const SeqPlan& s = p.seq[ui.b];
  const int local = u - s.unit_start;
  ui.rb = local % s.n_rb;
  ui.piece = local / s.n_rb;
  ui.R = s.n_q * p.num_heads;
  ui.prefix = s.n_kv - s.n_q;
  ui.k_lo = ui.piece * s.chunk;
  ui.k_hi = min(s.n_kv, ui.k_lo + s.chunk);
  ui.n_tiles = (ui.k_hi - ui.k_lo + kTileKeys - 1) / kTileKeys;
  return ui;
}

// Bounded wait; false on expiry or when the CTA is aborting.
__device__ __noinline__ bool wait_bar(TcSmem& sm, uint64_t* bar, uint32_t parity, uint32_t* status, int where,
                                      bool cluster_scope = false) {
  long long t0 = clock64();
  for (;;) {
    if (cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    if (sm.abort_flag) return false;
    if (clock64() - t0 > kWaitCycles) {
      record_status(status, VMLA_ERR_TIMEOUT, (uint32_t)where);
      sm.abort_flag = 1;
      // tell the partner CTA to stop too
      const uint32_t peer = cluster_ctarank() ^ 1u;
      const uint32_t remote = mapa(smem_u32((const void*)const_cast<int32_t*>(&sm.abort_flag)), peer);
      asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote), "r"(1) : "memory");
      return false;
    }
  }
}

// ------------------------------------------------------------------ producer (warp 0, lane 0, both CTAs)
// Loads each 64-key tile of the unit's key range from the contiguous staged
// copy of the KV rows: one 64-row x 64-column box (8 KB, 128-byte swizzle) per
// column chunk, 9 chunks for the scorer (K), 8 for the mixer (V).  Rows past
// the piece's end belong to other keys and are masked by the softmax.
__device__ void producer_role(TcSmem& sm, const CUtensorMap* map, const PlanParams& plan, const TcSched& sched,
                              const RunArgs& a, int u_begin, int u_end, int nch, bool prefetch) {
  int it = 0;
  bool ok = true;
  // L2 prefetch of the staged rows of tile t (contiguous: 64 rows x 1152 bytes), clamped to the staged area
  auto prefetch_tile = [&](const SeqPlan& sp, const UnitInfo& ui, int t) {
    if (!prefetch || t >= ui.n_tiles) return;
    const int64_t row0 = (int64_t)sp.kv_off + ui.k_lo + (int64_t)t * kTileKeys;
    int64_t rows = a.total_kv - row0;
    if (rows > kTileKeys) rows = kTileKeys;
    if (rows > 0) prefetch_l2_bulk(a.staged + row0 * kDqk, (uint32_t)(rows * kRowBytes));
  };
  for (int ui_idx = u_begin; ui_idx < u_end && ok; ++ui_idx) {
    const UnitInfo ui = decode_unit(plan, sched.order[ui_idx]);
    const SeqPlan& sp = plan.seq[ui.b];
    for (int t = 0; t < kPrefetchTiles && t < ui.n_tiles; ++t) prefetch_tile(sp, ui, t);
    for (int t = 0; t < ui.n_tiles; ++t) {
      const int s = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      if (!wait_bar(sm, &sm.kfree[s], ph ^ 1, a.status, 100)) {
        ok = false;
        break;
      }
      VTRACE(prefetch ? 0 : 6, it);
      const int y = sp.kv_off + ui.k_lo + t * kTileKeys;
      mbar_arrive_expect_tx(&sm.kfull[s], (uint32_t)(nch * kChunkBytes));
      const uint32_t bar = smem_u32(&sm.kfull[s]);
      for (int c = 0; c < nch; ++c) tma_load_2d(smem_u32(&sm.kv[s][c][0]), map, 64 * c, y, bar);
      prefetch_tile(sp, ui, t + kPrefetchTiles);
      ++it;
    }
  }
  // drain: the loads of the last two stages have landed before the CTA may exit
  for (int k = 1; k <= 2 && it - k >= 0; ++k) {
    const int j = it - k;
    long long t0 = clock64();
    while (!mbar_try_wait(&sm.kfull[j & 1], (j >> 1) & 1) && clock64() - t0 < kWaitCycles) {
    }
  }
}

// ------------------------------------------------------------------ CTA 0: QK^T issuer (warp 1, lane 0)
__device__ void scorer_mma_role(TcSmem& sm, const PlanParams& plan, const TcSched& sched, const RunArgs& a,
                                uint32_t tbase, int u_begin, int u_end) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, kTileKeys, 0, 0);
  int it = 0, uu = 0;
  for (int ui_idx = u_begin; ui_idx < u_end; ++ui_idx, ++uu) {
    const UnitInfo ui = decode_unit(plan, sched.order[ui_idx]);
    if (!wait_bar(sm, &sm.qfull, uu & 1, a.status, 200)) break;
    tc_fence_after();
    bool ok = true;
    for (int t = 0; t < ui.n_tiles; ++t, ++it) {
      const int s = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      if (!wait_bar(sm, &sm.kfull[s], ph, a.status, 201)) {
        ok = false;
        break;
      }
      VTRACE(1, it);
      if (!wait_bar(sm, &sm.sfree[s], ph ^ 1, a.status, 202)) {
        ok = false;
        break;
      }
      VTRACE(2, it);
      tc_fence_after();
      const uint32_t d = tbase + kSCol + (uint32_t)s * kTileKeys;
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        const uint32_t kbase = smem_u32(&sm.kv[s][c][0]);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ts(d, tbase + (uint32_t)(c * 32 + k * 8), smem_desc(kbase + k * 32, 16, 1024), idesc, (c | k) != 0);
      }
      mma_commit(&sm.sfull[s]);
      mma_commit(&sm.kfree[s]);
    }
    if (!ok) break;
  }
  // all issued MMAs complete before the CTA may exit
  mma_commit(&sm.obar);
  long long t0 = clock64();
  while (!mbar_try_wait(&sm.obar, 0) && clock64() - t0 < kWaitCycles) {
  }
}

// ------------------------------------------------------------------ CTA 0: softmax (warps 2-9)
// Thread (half, row): row = TMEM lane, keys [32*half, 32*half + 32) of each tile.
// The two halves of a row agree on the tile max through shared memory, so
// both keep the same running reference max m_ref (raised only when a tile
// exceeds it by 2^kTau, which bounds P by 2^kTau and makes rescales rare).
__device__ void scorer_softmax_role(TcSmem& sm, const PlanParams& plan, const TcSched& sched, const RunArgs& a,
                                    uint32_t tbase, int u_begin, int u_end) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wq = warp & 3;                 // TMEM lane quarter this warp may access
  const int half = (warp - 2) >> 2;        // 0: keys 0..31, 1: keys 32..63 of a tile
  const int row = wq * 32 + lane;          // query row within the unit = TMEM lane
  const int tid = threadIdx.x - 64;        // 0..255 within the softmax group
  const int wslot = warp - 2;              // 0..7
  const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
  const int H = plan.num_heads;
  const float scale = a.scale_log2;
  const uint32_t peer_pfull[2] = {mapa(smem_u32(&sm.pfull[0]), 1), mapa(smem_u32(&sm.pfull[1]), 1)};
  const uint32_t peer_msg[2] = {mapa(smem_u32(&sm.msg[0]), 1), mapa(smem_u32(&sm.msg[1]), 1)};
  int it = 0, uu = 0;
  for (int ui_idx = u_begin; ui_idx < u_end; ++ui_idx, ++uu) {
    const UnitInfo ui = decode_unit(plan, sched.order[ui_idx]);
    const SeqPlan& sp = plan.seq[ui.b];
    const int r = ui.rb * kRowsTC + row;
    const bool valid = r < ui.R;
    // Q rows of this unit into TMEM columns 0..287 (two bf16 per column); each
    // half of the group writes its own column chunks
    __syncwarp();
    {
      const uint4* qrow = reinterpret_cast<const uint4*>(a.q + ((int64_t)sp.q_off * H + (valid ? r : 0)) * kDqk);
#pragma unroll 1
      for (int c = half; c < kChunks; c += 2) {
        uint32_t v[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          uint4 x = valid ? __ldg(qrow + c * 8 + k) : make_uint4(0, 0, 0, 0);
          v[4 * k] = x.x;
          v[4 * k + 1] = x.y;
          v[4 * k + 2] = x.z;
          v[4 * k + 3] = x.w;
        }
        tmem_st32(tbase + lane_base + (uint32_t)(c * 32), v);
      }
      tmem_wait_st();
      tc_fence_before();
      named_bar_sync(1, 256);
      if (tid == 0) mbar_arrive(&sm.qfull);
    }
    const int i = valid ? r / H : 0;
    const uint64_t vis = a.masks ? a.masks[sp.q_off + i] : causal_bits(i);
    const int mask_from = min(ui.prefix, ui.k_hi);  // keys below this are visible to every valid row
    float m_ref = -INFINITY, l = 0.f;
    bool stop = false;
    for (int t = 0; t < ui.n_tiles; ++t, ++it) {
      const int s = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      // a failed wait leaves garbage in this tile; the group still meets at every
      // barrier below and stops together at the end of the tile
      wait_bar(sm, &sm.sfull[s], ph, a.status, 300);
      if (tid == 0) VTRACE(3, it);
      __syncwarp();
      tc_fence_after();
      uint32_t v[32];
      tmem_ld32(tbase + lane_base + kSCol + (uint32_t)s * kTileKeys + (uint32_t)half * 32, v);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&sm.sfree[s]);

      const int key0 = ui.k_lo + t * kTileKeys + half * 32;
      float x[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(v[j]) * scale;
      if (!valid) {
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = -INFINITY;
      } else if (key0 + 32 > mask_from) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int key = key0 + j;
          bool vis_j = key < ui.k_hi;
          if (vis_j && key >= ui.prefix) vis_j = ((vis >> (key - ui.prefix)) & 1ull) != 0;
          if (!vis_j) x[j] = -INFINITY;
        }
      }
      float mh = x[0];
#pragma unroll
      for (int j = 1; j < 32; ++j) mh = fmaxf(mh, x[j]);
      sm.pmax[half][row] = mh;
      const int ms = it & 1;  // message slot (one message per tile)
      const bool last = t == ui.n_tiles - 1;
      if (tid == 0) VTRACE(4, it);
      if (tid == 0 && it >= 2) bulk_wait_group_read<1>();
      named_bar_sync(1, 256);  // partial maxima visible; staging slot ms free
      const float mt = fmaxf(mh, sm.pmax[half ^ 1][row]);
      float alpha = 1.f;
      if (mt > m_ref + kTau) {
        alpha = ex2_approx(m_ref - mt);  // 0 when m_ref = -inf
        l *= alpha;
        m_ref = mt;
      }
      uint32_t pk[16];
      float lsum = 0.f;
      if (m_ref == -INFINITY) {
#pragma unroll
        for (int k = 0; k < 16; ++k) pk[k] = 0u;
      } else {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float p0 = ex2_approx(x[2 * k] - m_ref), p1 = ex2_approx(x[2 * k + 1] - m_ref);
          lsum += p0 + p1;
          pk[k] = pack_bf16x2(p0, p1);
        }
      }
      l += lsum;
      // P row -> staging, 128-byte swizzle (16-byte granule g of row `row` at g ^ (row & 7));
      // this half owns granules 4*half .. 4*half + 3
      uint8_t* prow = sm.msg[ms].p + row * 128;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int g = 4 * half + k;
        *reinterpret_cast<uint4*>(prow + ((g ^ (row & 7)) << 4)) =
            make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
      }
      if (half == 0) sm.msg[ms].alpha[row] = alpha;
      const unsigned any = __ballot_sync(0xffffffffu, alpha != 1.f);
      if (lane == 0) sm.warp_flags[wslot] = any ? 1u : 0u;
      if (last && half == 1) sm.lpart[row] = l;
      fence_proxy_async_smem();
      named_bar_sync(1, 256);
      if (last) {
        // unit finals: running max and the row sum of both halves
        if (half == 0) {
          sm.fin_stage[uu & 1].m[row] = m_ref;
          sm.fin_stage[uu & 1].l[row] = l + sm.lpart[row];
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 256);
      }
      if (tid == 0) {
        bool go = !sm.abort_flag;
        if (go) {
          uint32_t f = 0;
#pragma unroll
          for (int w = 0; w < 8; ++w) f |= sm.warp_flags[w];
          sm.msg[ms].flags = f;
          fence_proxy_async_smem();
          go = wait_bar(sm, &sm.pfree[ms], ((it >> 1) & 1) ^ 1, a.status, 301, true);
        }
        if (go) {
          VTRACE(5, it);
          bulk_s2s_cluster(peer_msg[ms], smem_u32(&sm.msg[ms]), kMsgBytes, peer_pfull[ms]);
          if (last)
            bulk_s2s_cluster(mapa(smem_u32(&sm.fin[uu & 1]), 1), smem_u32(&sm.fin_stage[uu & 1]), sizeof(Finals),
                             mapa(smem_u32(&sm.finfull[uu & 1]), 1));
          bulk_commit_group();
        }
        sm.wg_stop = go ? 0 : 1;
      }
      named_bar_sync(1, 256);
      if (sm.wg_stop) {
        stop = true;
        break;
      }
    }
    if (stop) break;
  }
  if (tid == 0) bulk_wait_group_read<0>();
}

// ------------------------------------------------------------------ CTA 1: P V issuer (warp 1, lane 0)
__device__ void mixer_mma_role(TcSmem& sm, const PlanParams& plan, const TcSched& sched, const RunArgs& a,
                               uint32_t tbase, int u_begin, int u_end) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 256, 0, 1);
  int it = 0, cmdn = 0, obn = 0;
  bool ok = true;
  auto command = [&](uint32_t c) -> bool {
    sm.cmd = c;
    mbar_arrive(&sm.cmd_full);
    const bool r = wait_bar(sm, &sm.cmd_done, cmdn & 1, a.status, 402);
    ++cmdn;
    return r;
  };
  auto quiesce = [&]() -> bool {
    mma_commit(&sm.obar);
    const bool r = wait_bar(sm, &sm.obar, obn & 1, a.status, 403);
    ++obn;
    return r;
  };
  for (int ui_idx = u_begin; ui_idx < u_end && ok; ++ui_idx) {
    const UnitInfo ui = decode_unit(plan, sched.order[ui_idx]);
    for (int t = 0; t < ui.n_tiles; ++t, ++it) {
      const int s = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      if (!wait_bar(sm, &sm.kfull[s], ph, a.status, 400)) {
        ok = false;
        break;
      }
      VTRACE(7, it);
      if (!wait_bar(sm, &sm.pfull[s], ph, a.status, 401, true)) {
        ok = false;
        break;
      }
      VTRACE(8, it);
      if (t > 0 && (sm.msg[s].flags & 1u)) {
        if (!quiesce() || !command(kCmdRescale | ((uint32_t)s << 8))) {
          ok = false;
          break;
        }
      }
      tc_fence_after();
      const uint32_t pbase = smem_u32(sm.msg[s].p);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t adesc = smem_desc(pbase + k * 32, 16, 1024);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint64_t bdesc = smem_desc(smem_u32(&sm.kv[s][4 * hh][0]) + k * 16 * 128, kChunkBytes, 1024);
          mma_ss(tbase + (uint32_t)(256 * hh), adesc, bdesc, idesc, (t > 0 || k > 0) ? 1u : 0u);
        }
      }
      mma_commit(&sm.kfree[s]);
      mma_commit(&sm.pdone[s]);
      VTRACE(9, it);
    }
    if (!ok) break;
    if (!quiesce() || !command(kCmdEpilogue)) ok = false;
  }
  if (!ok) quiesce();
  sm.cmd = kCmdExit;
  mbar_arrive(&sm.cmd_full);
}

// ------------------------------------------------------------------ CTA 1: P-slot release (warp 6, lane 0)
__device__ void mixer_release_role(TcSmem& sm, const PlanParams& plan, const TcSched& sched, const RunArgs& a,
                                   int u_begin, int u_end) {
  int total = 0;
  for (int ui_idx = u_begin; ui_idx < u_end; ++ui_idx) total += decode_unit(plan, sched.order[ui_idx]).n_tiles;
  const uint32_t peer_pfree[2] = {mapa(smem_u32(&sm.pfree[0]), 0), mapa(smem_u32(&sm.pfree[1]), 0)};
  for (int n = 0; n < total; ++n) {
    const int s = n & 1;
    if (!wait_bar(sm, &sm.pdone[s], (n >> 1) & 1, a.status, 500)) return;
    VTRACE(10, n);
    if (n + 2 < total) {
      mbar_arrive_expect_tx(&sm.pfull[s], kMsgBytes);
      mbar_arrive_remote(peer_pfree[s]);
    }
  }
}

// ------------------------------------------------------------------ CTA 1: rescale / epilogue (warps 2-5)
__device__ void mixer_epilogue_role(TcSmem& sm, const PlanParams& plan, const TcSched& sched, const RunArgs& a,
                                    uint32_t tbase, int u_begin, int u_end) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wq = warp & 3;
  const int row = wq * 32 + lane;
  const int tid = threadIdx.x - 64;
  const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
  const int H = plan.num_heads;
  int cmdn = 0, uu = 0;
  int ui_idx = u_begin;
  for (;;) {
    // thread 0 waits for the command (and, for an epilogue, the unit's finals);
    // the group learns it at a barrier, so a failed wait stops every thread
    if (tid == 0) {
      uint32_t cmd = kCmdExit;
      if (wait_bar(sm, &sm.cmd_full, cmdn & 1, a.status, 600)) {
        cmd = sm.cmd;
        if ((cmd & 0xFF) == kCmdEpilogue &&
            !wait_bar(sm, &sm.finfull[uu & 1], (uu >> 1) & 1, a.status, 601, true))
          cmd = kCmdExit;
      }
      sm.wg_cmd = cmd;
    }
    ++cmdn;
    named_bar_sync(2, 128);
    const uint32_t cmd = sm.wg_cmd;
    if ((cmd & 0xFF) == kCmdExit) return;
    __syncwarp();
    tc_fence_after();
    // tcgen05.ld / st are warp-collective: every branch around them is warp-uniform
    if ((cmd & 0xFF) == kCmdRescale) {
      const int s = (cmd >> 8) & 1;
      const float alpha = sm.msg[s].alpha[row];
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int c = 0; c < kDv / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tbase + lane_base + (uint32_t)(c * 32), v);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
          tmem_st32(tbase + lane_base + (uint32_t)(c * 32), v);
        }
        tmem_wait_st();
      }
    } else {
      // epilogue of unit ui_idx: O / l -> output row (or fp32 partial)
      const UnitInfo ui = decode_unit(plan, sched.order[ui_idx]);
      const SeqPlan& sp = plan.seq[ui.b];
      const int f = uu & 1;
      const float m = sm.fin[f].m[row], lsum = sm.fin[f].l[row];
      const int r = ui.rb * kRowsTC + row;
      const bool valid = r < ui.R;
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
      const float lse2 = lsum > 0.f ? m + log2f(lsum) : -INFINITY;
      if (sp.n_split == 1) {
        const int64_t orow = (int64_t)sp.q_off * H + (valid ? r : 0);
        uint4* dst = reinterpret_cast<uint4*>(a.out + orow * kDv);
#pragma unroll 1
        for (int c = 0; c < kDv / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tbase + lane_base + (uint32_t)(c * 32), v);
          tmem_wait_ld();
          if (valid) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              dst[c * 4 + k] = make_uint4(
                  pack_bf16x2(__uint_as_float(v[8 * k]) * inv, __uint_as_float(v[8 * k + 1]) * inv),
                  pack_bf16x2(__uint_as_float(v[8 * k + 2]) * inv, __uint_as_float(v[8 * k + 3]) * inv),
                  pack_bf16x2(__uint_as_float(v[8 * k + 4]) * inv, __uint_as_float(v[8 * k + 5]) * inv),
                  pack_bf16x2(__uint_as_float(v[8 * k + 6]) * inv, __uint_as_float(v[8 * k + 7]) * inv));
          }
          __syncwarp();
        }
        if (valid) a.lse[orow] = lsum > 0.f ? lse2 * 0.6931471805599453f : -INFINITY;
      } else {
        const int64_t prow = (int64_t)sp.part_off + (int64_t)ui.piece * ui.R + (valid ? r : 0);
        float4* dst = reinterpret_cast<float4*>(a.part_o + prow * kDv);
#pragma unroll 1
        for (int c = 0; c < kDv / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tbase + lane_base + (uint32_t)(c * 32), v);
          tmem_wait_ld();
          if (valid) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              dst[c * 8 + k] = make_float4(__uint_as_float(v[4 * k]) * inv, __uint_as_float(v[4 * k + 1]) * inv,
                                           __uint_as_float(v[4 * k + 2]) * inv, __uint_as_float(v[4 * k + 3]) * inv);
          }
          __syncwarp();
        }
        if (valid) a.part_lse[prow] = lse2;
      }
      ++uu;
      ++ui_idx;
    }
    tc_fence_before();
    named_bar_sync(2, 128);
    if (tid == 0) {
      // a finals buffer is re-armed for the unit two ahead once it has been read
      if ((cmd & 0xFF) == kCmdEpilogue && ui_idx + 1 < u_end)
        mbar_arrive_expect_tx(&sm.finfull[(uu + 1) & 1], sizeof(Finals));
      mbar_arrive(&sm.cmd_done);
    }
  }
}

__global__ void __launch_bounds__(kThreadsTC, 1)
tc_verify_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ PlanParams plan,
                 const __grid_constant__ TcSched sched, const RunArgs a) {
  extern __shared__ uint8_t smem_raw[];
  TcSmem& sm = *reinterpret_cast<TcSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cid = (int)cluster_id_x();
  const int u_begin = cid < sched.num_clusters ? sched.start[cid] : 0;
  const int u_end = cid < sched.num_clusters ? sched.start[cid + 1] : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.kfull[s], 1);
      mbar_init(&sm.kfree[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.sfull[s], 1);
      mbar_init(&sm.sfree[s], 256);
      mbar_init(&sm.pfull[s], 1);
      mbar_init(&sm.pfree[s], 1);
      mbar_init(&sm.pdone[s], 1);
      mbar_init(&sm.finfull[s], 1);
    }
    mbar_init(&sm.qfull, 1);
    mbar_init(&sm.cmd_full, 1);
    mbar_init(&sm.cmd_done, 1);
    mbar_init(&sm.obar, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&kv_map);
  }
  __syncwarp();
  if (warp == 0) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  if (rank == 1 && threadIdx.x == 64) {  // thread 0 of the epilogue group
    // receive slots and finals buffers armed before the partner can send
    int n_units = u_end - u_begin, total = 0;
    for (int k = u_begin; k < u_end; ++k) total += decode_unit(plan, sched.order[k]).n_tiles;
    for (int s = 0; s < 2 && s < total; ++s) mbar_arrive_expect_tx(&sm.pfull[s], kMsgBytes);
    for (int s = 0; s < 2 && s < n_units; ++s) mbar_arrive_expect_tx(&sm.finfull[s], sizeof(Finals));
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_arrive();
  cluster_wait();
  const uint32_t tbase = sm.tmem_base;

  if (warp == 0) {
    if (lane == 0)
      producer_role(sm, &kv_map, plan, sched, a, u_begin, u_end, rank == 0 ? kChunks : kVChunks, rank == 0);
  } else if (warp == 1) {
    if (lane == 0) {
      if (rank == 0) scorer_mma_role(sm, plan, sched, a, tbase, u_begin, u_end);
      else mixer_mma_role(sm, plan, sched, a, tbase, u_begin, u_end);
    }
  } else if (rank == 0) {
    scorer_softmax_role(sm, plan, sched, a, tbase, u_begin, u_end);
  } else if (warp < 6) {
    mixer_epilogue_role(sm, plan, sched, a, tbase, u_begin, u_end);
  } else if (warp == 6 && lane == 0) {
    mixer_release_role(sm, plan, sched, a, u_begin, u_end);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  // neither CTA leaves while the other may still address its shared memory
  cluster_arrive();
  cluster_wait();
  __syncwarp();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
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
static_assert(sizeof(PlanParams) + sizeof(TcSched) + sizeof(RunArgs) + sizeof(CUtensorMap) < 32000,
              "kernel parameter budget");

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
      cudaSuccess)
    return VMLA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreadsTC, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
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
  if (clusters > plan.total_units) clusters = plan.total_units;
  static thread_local TcSched sched;
  rc = build_tc_schedule(plan, clusters, &sched);
  if (rc != VMLA_OK) return rc;
  // 2-D map over the staged rows [total_kv x 576 bf16], boxes of 64 columns x 64 rows, 128-byte swizzle
  CUtensorMap map;
  cuuint64_t gdim[2] = {(cuuint64_t)kDqk, (cuuint64_t)(a.total_kv > 0 ? a.total_kv : 1)};
  cuuint64_t gstride[1] = {(cuuint64_t)kRowBytes};
  cuuint32_t box[2] = {64, (cuuint32_t)kTileKeys};
  cuuint32_t estride[2] = {1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.staged, gdim, gstride, box, estride,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return VMLA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * sched.num_clusters, 1, 1);
  cfg.blockDim = dim3(kThreadsTC, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, tc_verify_kernel, map, plan, sched, a) != cudaSuccess) return VMLA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? VMLA_OK : VMLA_ERR_CUDA;
}

}  // namespace vmla

#ifdef VMLA_TRACE
extern "C" int vmla_trace_read(uint64_t* host, int n) {
  const int total = vmla::kTraceEvents * vmla::kTraceTiles;
  if (n > total) n = total;
  return cudaMemcpyFromSymbol(host, vmla::g_vmla_trace, sizeof(uint64_t) * n) == cudaSuccess ? n : -1;
}
extern "C" int vmla_trace_clear(void) {
  static uint64_t zeros[vmla::kTraceEvents * vmla::kTraceTiles] = {};
  return cudaMemcpyToSymbol(vmla::g_vmla_trace, zeros, sizeof zeros) == cudaSuccess ? 0 : -1;
}
#endif
