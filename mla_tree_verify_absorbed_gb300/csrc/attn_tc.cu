// Tensor-core split-KV verify attention for sm_103a: tcgen05 MMAs issued for
// CTA pairs (cta_group::2) with TMEM accumulators, asynchronous gathers of the
// paged KV, a 4-CTA cluster per work item.
//
// Shape of the problem.  Per work item, 256 query rows (absorbed queries of
// (node, head) pairs; "Ground Truth in Silicon ...", section "Input Knowledge
// Required ...", item 2) attend over KV tiles of 64 tokens whose latent kv_c
// (512) and rope key k_pe (64) are shared by all rows ("Ground Truth in
// Silicon ...", section "The Message in Full").  Both products are dense
// contractions:  S = Q [256 x 576] . K^T [576 x 64]  and
// O += P [256 x 64] . V [64 x 512]  with V = kv_c.
//
// Why four CTAs.  An fp32 accumulator for 128 rows x 512 columns is exactly
// the 512 columns x 128 lanes of one SM's Tensor Memory, so O and S cannot
// share one SM; and the rate at which an SM can gather scattered pool rows,
// not the tensor cores, bounds this work, so every gathered byte should feed
// as many rows as possible.  A work item therefore runs on two CTA pairs:
//   * the score pair (cluster ranks 0, 1) holds the 256 query rows in TMEM,
//     128 per CTA (288 columns, bf16 pairs), as the A operand of
//     S = Q.K^T -- one M=256 MMA for both CTAs (TS form, N=64, K=576 in 36
//     steps), each CTA staging half of the tile's tokens (B is split along
//     N) -- double-buffers S in TMEM, and runs the online softmax of its
//     rows: one thread per row, base-2 exponent, the tree mask, and a lazy
//     running max (the max only moves when a tile beats it by more than
//     2^8, so rescaling O is rare);
//   * the value pair (ranks 2, 3) holds O for its 128 rows per CTA (512
//     columns) and runs O += P.V as M=256 MMAs (SS form, N=256 twice,
//     K=64), each CTA staging half of every kv_c row (V split along N) as
//     an MN-major operand.
// So each CTA reads half of every tile from L2 (the other half reaches its
// tensor core from the pair peer), and the smaller stages leave room for six
// in flight.  P (bf16) and the per-row rescale factors of score CTA c are
// staged in its own shared memory and moved to value CTA 2 + c by one thread
// with a bulk shared::cta -> shared::cluster copy whose bytes complete that
// CTA's barrier; the commit of the PV MMAs that read a P buffer arrives on
// both score CTAs' barriers directly, so P buffers come back without a relay
// thread.  The value CTAs rescale their own O rows when a factor differs from
// 1 and write the outputs.
//
// Data movement.  Eight producer warps per CTA gather the CTA's share of every
// tile with 16-byte cp.async copies written straight into the 128-byte
// swizzled layout the MMAs read; slot indices are fetched one tile ahead.
// cp.async completion can only signal a barrier of the issuing CTA, so a warp
// of each odd CTA relays "tile landed" to its pair's MMA-issuing CTA.  Each
// staged tile is reused by all 256 rows of the item -- the head-tile reuse of
// "The Critical Glue: Validating a Custom Flash Attention Kernel Through Test
// Infrastructure", section "What Came Before", widened to every (node, head)
// row.
//
// Signals between CTAs that hand over no data of the signalling thread (a
// buffer may be reused, a tile has landed, O is ready) use relaxed remote
// arrives: the data they guard has already been written and observed (cp.async
// and bulk-copy completion, tcgen05 wait::ld / wait::st) when they are sent,
// and a cluster-scope release arrive measured ~770 cycles per signal, more
// while the thread's earlier remote stores drained.  Only the row statistics handed to
// the value CTA (st.shared::cluster data) travel under a release arrive.
//
// Every wait is bounded; on timeout the kernel raises an abort flag in all
// four CTAs, sets MLA_DEVERR_TIMEOUT, stops issuing work, drains the MMAs it
// issued, frees TMEM and returns.
#include <mutex>

#include "common.cuh"
#include "sm100.cuh"

namespace mlav {
using namespace sm100;

namespace tc {

constexpr int kRG = 256;        // query rows per work item (pair MMA M)
constexpr int kRC = 128;        // query rows per CTA
constexpr int kTK = 64;         // tokens per KV tile (S MMA N)
constexpr int kStagesS = 5;     // KV tiles in flight, score pair
constexpr int kStagesV = 6;     // KV tiles in flight, value pair
constexpr int kStagesMax = kStagesV;
constexpr int kThreads = 576;   // 18 warps
constexpr int kClusterCtas = 4;
constexpr uint32_t kTmemCols = 512;

// warp roles
constexpr int kProducerWarps = 8;  // warps 0-7
constexpr int kProducerThreads = 32 * kProducerWarps;
// Row warps 8-15: two warpgroups, each covering the CTA's 128 rows (warp w
// reaches TMEM lanes 32 (w % 4) ..); warpgroup h takes columns half h.
constexpr int kWarpRows = 8, kRowWarps = 8, kRowThreads = 32 * kRowWarps;
constexpr int kWarpMma = 16;  // MMA issue (even CTAs) or tile-landed relay (odd CTAs)
constexpr int kWarpAux = 17;  // TMEM allocation; lane 0 of score CTAs: P bulk copies

// score CTA stage: its 32 tokens x 576 columns, as 9 chunks of 64 columns
// (chunks 0-7 kv_c, chunk 8 k_pe), each chunk 32 rows of 128 bytes
constexpr int kTokS = kTK / 2;
constexpr int kTokSPerWarp = kTokS / kProducerWarps;  // 4
constexpr int kChunkS = kTokS * 128;                  // 4 KB
constexpr int kStageS = 9 * kChunkS;                  // 36 KB
// value CTA stage: 64 tokens x its 256 kv_c columns, as 4 atoms of 64 columns
// (atom a covers columns 256 (a >> 1) + 128 half + 64 (a & 1) + [0, 64))
constexpr int kTokVPerWarp = kTK / kProducerWarps;  // 8
constexpr int kAtomV = kTK * 128;                   // 8 KB
constexpr int kStageV = 4 * kAtomV;                 // 32 KB
constexpr int kOffP = kStagesV * kStageV;           // value CTA: [2][16 KB]
constexpr int kPBytes = kRC * 128;                  // P tile [128 rows x 64 tokens] bf16
constexpr int kOffCtl = kOffP + 2 * kPBytes;
// score CTA, after its stages: P and its rescale factors are staged here
// ([2][16 KB], [2][128] floats) and bulk-copied to the value CTA; then the
// partial row maxima the two column halves of a row exchange per tile
// ([2 tiles][2 halves][128 rows]) and the partial sums per item ([128])
constexpr int kOffPStage = kStagesS * kStageS;
constexpr int kOffAStage = kOffPStage + 2 * kPBytes;
constexpr int kOffRed = kOffAStage + 2 * kRC * 4;
constexpr int kRedBytes = (2 * 2 * kRC + kRC) * 4;
constexpr uint32_t kPTxBytes = kPBytes + kRC * 4;   // P tile + alpha, per tile

constexpr uint32_t kIdescS = idesc_bf16_f32(kRG, kTK, 0, 0);  // A (Q, TMEM), B (K tile) K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(kRG, 256, 0, 1); // A (P) K-major, B (V) MN-major

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr uint64_t kDrainLimitNs = 20000000ull;   // 20 ms per drain wait on abort

struct alignas(16) Ctl {
  uint64_t full[kStagesMax];       // this CTA's share of a tile landed (kProducerThreads cp.async arrivals;
                                // even CTAs: + 1 relayed arrival for the odd CTA's share)
  uint64_t empty[kStagesMax];      // stage reusable: the pair MMAs reading it are complete
  uint64_t s_full[2];           // score: S tile in TMEM
  uint64_t s_free[2];           // score, rank 0: both CTAs' softmax warps loaded S (16 warp arrivals)
  uint64_t q_ready;             // score, rank 0: both CTAs' queries in TMEM (16 warp arrivals)
  uint64_t p_free[2];           // score: the value pair's PV MMAs that read this P buffer completed (commit)
  uint64_t fin_free;            // score: the value partner consumed lfin/mfin (256 arrivals)
  uint64_t xch[2];              // score: both halves' partial row maxima of a tile written (8 warp arrivals)
  uint64_t xfin;                // score: half 1's partial row sums of an item written (4 warp arrivals)
  uint64_t p_staged[2];         // score: P and alpha of a tile staged locally (8 warp arrivals)
  uint64_t p_full[2];           // value: P tile and alpha landed (bulk-copy bytes; armed by a row thread)
  uint64_t pv_done[2];          // value: PV MMAs of a tile complete
  uint64_t o_ready[2];          // value, rank 2: both CTAs' O ready for the tile's PV (16 warp arrivals)
  uint64_t fin_full;            // value: lfin/mfin written (128 remote arrivals)
  uint64_t drain;               // even CTAs: final MMA drain on abort
  uint64_t hold;                // self-test: never completed
  alignas(16) float alpha[2][kRC];  // value: per-row rescale of O before PV(j) (1 = unchanged; bulk-copy target)
  float lfin[kRC];              // value: final row sums of the weights
  float mfin[kRC];              // value: final running max (base-2 units)
  uint32_t tmem_base;
  int abort;
  int abort_site;
};
constexpr int kSmemBytes = kOffCtl + (int)sizeof(Ctl);
static_assert(offsetof(Ctl, alpha) % 16 == 0, "bulk-copy target alignment");
constexpr int kSmemAlloc = 232448;  // the per-CTA maximum; the base must be 1024-aligned
static_assert(kSmemBytes <= kSmemAlloc, "shared memory budget");
static_assert(kOffRed + kRedBytes <= kOffCtl, "score stages overlap the control block");
static_assert(kOffPStage % 1024 == 0 && kOffAStage % 16 == 0, "staging buffers: swizzle atoms and bulk-copy alignment");
static_assert(kWarpRows % 4 == 0 && kRowWarps == 8, "the row warps must form two warpgroups (TMEM lane quadrants)");
static_assert(kWarpAux < kThreads / 32, "warp roles exceed the CTA");

// Wait sites, recorded in the workspace's second error word when a wait gives
// up.  The numbers are part of the error report, so they stay fixed (13 was
// the wait of a P-release thread the MMA commit has replaced).
enum {
  kSiteEmpty = 1, kSiteQReady = 2, kSiteFullS = 3, kSiteSFree = 4, kSiteSFull = 5, kSitePFree = 6,
  kSiteFinFree = 7, kSiteFullV = 8, kSiteOReady = 9, kSitePFull = 10, kSitePvPrev = 11, kSitePvLast = 12,
  kSiteRelay = 14, kSiteFinFull = 15, kSiteXch = 16, kSitePStaged = 17, kSiteHold = 18
};

// Bounded wait on a barrier of this CTA.  Barriers that other CTAs (or pair
// MMA commits) arrive on are waited with cluster-scope acquire.  A wait that
// runs out of time records its site (waits that only see the abort flag
// record nothing) and tells every CTA of the cluster to stop.
__device__ __noinline__ void raise_abort(Ctl* c, int site, int j) {
  // a wait that gave up while no abort was raised ran out of time itself
  if (*reinterpret_cast<volatile int*>(&c->abort) == 0)
    atomicCAS(&c->abort_site, 0, (site & 0xff) | ((j & 0xffff) << 16));
  for (uint32_t rk = 0; rk < kClusterCtas; ++rk) st_cluster_u32(mapa_shared(smem_u32(&c->abort), rk), 1u);
}
__device__ __forceinline__ bool wait(uint64_t* bar, uint32_t parity, Ctl* c, int site, int j,
                                     bool cluster = true) {
  if (mbar_wait(bar, parity, &c->abort, kWaitLimitNs, cluster)) return true;
  raise_abort(c, site, j);
  return false;
}

// The same wait made by every lane of a warp; the result is warp-uniform and
// the warp is converged on return (the MMA roles issue with elect.sync).
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, Ctl* c, int site, int j) {
  return __all_sync(0xffffffffu, wait(bar, parity, c, site, j));
}

// 2^x by the hardware approximation (flushes results below 2^-126 to zero,
// which only drops weights negligible against the row max).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Calls f(slot, it) for the non-empty work units of this cluster (see Split),
// in order.  slot is the unit's partial-output slot, or -1 when the unit is a
// row group's only piece and writes the outputs itself.
template <class F>
__device__ __forceinline__ void for_items(const Params& p, const Split& sc, int cluster_id, int n_clusters, F&& f) {
  const int64_t n_units = sc.tail + (sc.n_items - sc.tail) * sc.P;
  for (int64_t u = cluster_id; u < n_units; u += n_clusters) {
    const bool piece = u >= sc.tail && sc.P > 1;
    const int64_t v = u - sc.tail;
    const int64_t item = piece ? sc.tail + v / sc.P : u;
    const int64_t slot = piece ? v : (sc.S > 1 ? u : -1);
    Item it = item_at(p, sc.S, item);
    if (piece) {
      const int64_t q = v % sc.P, a = it.t0, len = it.t1 - it.t0;
      it.t0 = (int)(a + q * len / sc.P);
      it.t1 = (int)(a + (q + 1) * len / sc.P);
    }
    if (it.t1 <= it.t0) continue;
    if (!f(slot, it)) return;
  }
}

// ---------------------------------------------------------------------------
// producers (all four CTAs)
// ---------------------------------------------------------------------------
// Stages this CTA's share of the KV tiles of its items, placing 16-byte piece
// q of a 128-byte row segment of token row r at  base + r * 128 + ((q ^ (r & 7)) * 16)
// -- the 128-byte swizzle of the operand layouts.
//   score CTA `half`: tokens [32 half, 32 half + 32) of each tile; warp pw
//     copies 4 of them: per token two instructions move the 1 KB kv_c row
//     (lane l moves pieces l and l + 32; chunk = piece / 8), and one more
//     instruction moves the four 128-byte k_pe rows into chunk 8;
//   value CTA `half`: all 64 tokens, kv_c columns [256 nh + 128 half, +128)
//     for nh = 0, 1; warp pw copies 8 tokens, one instruction per token (lane
//     l moves piece l & 15 of segment nh = l >> 4).
// Positions past the sequence read slot 0; the softmax gives them zero weight.
__device__ void producer(const Params& p, const Split sc, uint8_t* smem, Ctl* c, int pw, uint32_t rank, int cluster_id,
                         int n_clusters) {
  const int lane = threadIdx.x & 31;
  const bool score = rank < 2;
  const int half = (int)(rank & 1);
  const int ntok = score ? kTokSPerWarp : kTokVPerWarp;
  const int nst = score ? kStagesS : kStagesV;
  const int r0 = ntok * pw;                  // first token row of this warp within the CTA's share
  const int tok0 = score ? half * kTokS : 0;  // the share's first token within the tile
  const __nv_bfloat16* kvc_g = reinterpret_cast<const __nv_bfloat16*>(p.kv_c);
  const __nv_bfloat16* kpe_g = reinterpret_cast<const __nv_bfloat16*>(p.k_pe);
  const uint32_t sbase = smem_u32(smem);
  int j = 0;
  for_items(p, sc, cluster_id, n_clusters, [&](int64_t, const Item& it) {
    const int b = it.b;
    const int64_t N = (int64_t)p.prefix_lens[b] + p.Q;
    const int64_t idx0 = p.page_size == 1 ? (int64_t)p.kv_indptr[b] : 0;
    // slot of token row r0 + (lane % ntok) of tile t
    auto slot_of = [&](int t) -> int64_t {
      const int64_t pos = (int64_t)t * kTK + tok0 + r0 + (lane & (ntok - 1));
      if (pos >= N) return 0;
      int64_t sl;
      if (p.page_size == 1) {
        sl = p.kv_indices[idx0 + pos];
      } else {
        sl = (int64_t)p.block_table[(int64_t)b * p.max_pages + pos / p.page_size] * p.page_size +
             pos % p.page_size;
      }
      return (sl < 0 || sl >= p.pool_slots) ? 0 : sl;
    };
    int64_t next = slot_of(it.t0);
    for (int t = it.t0; t < it.t1; ++t, ++j) {
      const int s = j % nst;
      const int64_t slot = next;
      if (t + 1 < it.t1) next = slot_of(t + 1);  // index load for the next tile, in flight meanwhile
      bool ok = true;
      if (lane == 0) ok = wait(&c->empty[s], ((uint32_t)(j / nst) & 1u) ^ 1u, c, kSiteEmpty, j);
      if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
      if (score) {
        const uint32_t stage = sbase + s * kStageS;
#pragma unroll
        for (int tt = 0; tt < kTokSPerWarp; ++tt) {
          const int64_t sl = __shfl_sync(0xffffffffu, slot, tt);
          const int r = r0 + tt;
          const __nv_bfloat16* src = kvc_g + sl * p.kv_c_stride;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int g = lane + 32 * h;
            const int q = g & 7;
            cp_async_16(stage + (g >> 3) * kChunkS + r * 128 + ((q ^ (r & 7)) << 4), src + g * 8);
          }
        }
        const int tt = lane >> 3, q = lane & 7;
        const int64_t sl = __shfl_sync(0xffffffffu, slot, tt);
        const int r = r0 + tt;
        cp_async_16(stage + 8 * kChunkS + r * 128 + ((q ^ (r & 7)) << 4), kpe_g + sl * p.k_pe_stride + q * 8);
      } else {
        const uint32_t stage = sbase + s * kStageV;
        const int nh = lane >> 4, g = lane & 15, q = g & 7;
        const uint32_t dst0 = stage + (nh * 2 + (g >> 3)) * kAtomV;
        const int col = nh * 256 + half * 128 + g * 8;
#pragma unroll
        for (int tt = 0; tt < kTokVPerWarp; ++tt) {
          const int64_t sl = __shfl_sync(0xffffffffu, slot, tt);
          const int r = r0 + tt;
          cp_async_16(dst0 + r * 128 + ((q ^ (r & 7)) << 4), kvc_g + sl * p.kv_c_stride + col);
        }
      }
      cp_async_mbar_arrive(&c->full[s]);
    }
    return true;
  });
  // copies already issued must land before this CTA may exit
  cp_async_wait_all();
}

// Odd CTAs: tell the pair's MMA-issuing CTA when this CTA's share of a tile
// has landed (whole warp).
__device__ void relay(const Params& p, const Split sc, Ctl* c, uint32_t leader, int cluster_id, int n_clusters) {
  const int nst = leader == 0 ? kStagesS : kStagesV;
  int j = 0;
  for_items(p, sc, cluster_id, n_clusters, [&](int64_t, const Item& it) {
    for (int t = it.t0; t < it.t1; ++t, ++j) {
      const int s = j % nst;
      if (!wait_warp(&c->full[s], (uint32_t)(j / nst) & 1u, c, kSiteRelay, j)) return false;
      fence_proxy_async_smem();  // cp.async data, written through the generic proxy, feeds the MMA
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive_cluster_relaxed(&c->full[s], leader);
    }
    return true;
  });
}

// ---------------------------------------------------------------------------
// score pair
// ---------------------------------------------------------------------------
__device__ void score_mma(const Params& p, const Split sc, uint8_t* smem, Ctl* c, int cluster_id, int n_clusters) {
  // rank 0, whole warp; one elected lane issues each pair MMA.  While the
  // tensor pipe works through a tile's MMAs, the warp checks (without
  // blocking) whether the next tile can start, so the checks cost no pipe time.
  const uint32_t tS = c->tmem_base;        // columns [0, 128): two S buffers
  const uint32_t tQ = c->tmem_base + 128;  // columns [128, 416): queries, bf16 pairs
  int j = 0, seg = 0;
  // S(j) may start once its tile has landed in both CTAs and the softmax has
  // loaded S(j-2) from buffer j & 1 (the softmax loading S(j-1) from the other
  // buffer meanwhile does not delay these MMAs: measured, a TMEM load of other
  // columns completes in tens of cycles while MMAs run)
  if (p.hold_ns) {
    // failure-detection self-test: a wait that nothing completes, bounded by
    // hold_ns; giving up raises the abort in every CTA of the cluster
    if (!mbar_wait(&c->hold, 0u, &c->abort, p.hold_ns, true)) raise_abort(c, kSiteHold, 0);
    __syncwarp();
  }
  auto ready_test = [&](int jj) {
    const bool ok = mbar_test_wait_cluster(&c->full[jj % kStagesS], (uint32_t)(jj / kStagesS) & 1u) &&
                    (jj < 2 || mbar_test_wait_cluster(&c->s_free[jj & 1], (((uint32_t)jj >> 1) & 1u) ^ 1u));
    return __all_sync(0xffffffffu, ok);
  };
  for_items(p, sc, cluster_id, n_clusters, [&](int64_t, const Item& it) {
    if (!wait_warp(&c->q_ready, (uint32_t)seg & 1u, c, kSiteQReady, j)) return false;
    tc_fence_after();
    bool ready = false;
    for (int t = it.t0; t < it.t1; ++t, ++j) {
      const int s = j % kStagesS, sb = j & 1;
      if (!ready) {
        if (!wait_warp(&c->full[s], (uint32_t)(j / kStagesS) & 1u, c, kSiteFullS, j)) return false;
        if (j >= 2 && !wait_warp(&c->s_free[sb], (((uint32_t)j >> 1) & 1u) ^ 1u, c, kSiteSFree, j)) return false;
      }
      fence_proxy_async_smem();
      tc_fence_after();
      // descriptors differ only in the start-address field: add (offset >> 4)
      const uint64_t dk = smem_desc(smem_u32(smem + s * kStageS), 16, 1024, kLayoutSw128);
      const uint32_t ts = tS + sb * kTK;
#pragma unroll
      for (int kc = 0; kc < 9; ++kc) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_pair_ts_warp(ts, tQ + kc * 32 + kk * 8, dk + (uint64_t)((kc * kChunkS + kk * 32) >> 4), kIdescS,
                           (kc | kk) != 0);
        if (kc == 5) ready = (t + 1 < it.t1) && ready_test(j + 1);
      }
      mma_pair_commit_warp(&c->s_full[sb], 0x3);
      mma_pair_commit_warp(&c->empty[s], 0x3);
    }
    ++seg;
    return true;
  });
  if (__any_sync(0xffffffffu, c->abort != 0)) {
    // outstanding S MMAs must finish before TMEM is released
    mma_pair_commit_warp(&c->drain, 0x1);
    if ((threadIdx.x & 31) == 0) mbar_wait_drain(&c->drain, 0, kDrainLimitNs);
    __syncwarp();
  }
}

// Stages query row `row` of sequence b into Tensor Memory for row thread
// (quadrant of tQ, half h): columns [144 h, 144 h + 144), column c holding
// elements 2c, 2c+1 of the 576 (512 latent, then 64 rope).
__device__ __forceinline__ void stage_query_row(const Params& p, int b, int row, bool live, int h, uint32_t tQ) {
  const uint4* ql = reinterpret_cast<const uint4*>(p.q_lat) + ((int64_t)b * p.rows + row) * (kDl / 8);
  const uint4* qp = reinterpret_cast<const uint4*>(p.q_pe) + ((int64_t)b * p.rows + row) * (kDr / 8);
#pragma unroll 1
  for (int c0 = 144 * h; c0 < 144 * h + 144; c0 += 16) {
    uint32_t wv[16];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int col = c0 + 4 * v;  // 4 columns per 16-byte vector
      uint4 x = make_uint4(0, 0, 0, 0);
      if (live) x = col < 256 ? ql[col / 4] : qp[(col - 256) / 4];
      wv[4 * v + 0] = x.x;
      wv[4 * v + 1] = x.y;
      wv[4 * v + 2] = x.z;
      wv[4 * v + 3] = x.w;
    }
    __syncwarp();
    tmem_st_32x32b_x16(tQ + c0, wv);
  }
  tmem_wait_st();
}

// Online softmax of this CTA's 128 rows.  Each row is shared by two threads
// (warps w and w + 4 of the row warps) that take columns [32 h, 32 h + 32) of
// every tile: they exchange partial maxima per tile through shared memory, so
// both follow the same running max, and keep partial row sums that are added
// once per item.
__device__ void score_softmax(const Params& p, const Split sc, uint8_t* smem, Ctl* c, uint32_t rank, int cluster_id,
                              int n_clusters, int pre_g) {
  const int lane = threadIdx.x & 31;
  const int w = (threadIdx.x >> 5) - kWarpRows;     // 0..7
  const int wq = w & 3;                              // TMEM lane quadrant of this warp
  const int h = w >> 2;                              // column half
  const int r = wq * 32 + lane;                      // row within the CTA
  const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
  const uint32_t tS = c->tmem_base + lane_off + (uint32_t)(h * 32);
  const uint32_t tQ = c->tmem_base + 128 + lane_off;
  const uint32_t partner = rank + 2;                 // value CTA of these rows (row statistics)
  float* red_max = reinterpret_cast<float*>(smem + kOffRed);  // [2][2][kRC]
  float* red_l = red_max + 4 * kRC;                            // [kRC]
  const float sl2 = p.scale_log2;
  const int nq = p.Q;
  int j = 0, seg = 0;
  bool first = true;
  for_items(p, sc, cluster_id, n_clusters, [&](int64_t, const Item& it) {
    const int b = it.b;
    const int row = it.g * kRG + (int)rank * kRC + r;
    const bool live = row < p.rows;
    const int64_t P = p.prefix_lens[b];
    const uint64_t anc = live ? p.anc[(int64_t)b * p.Q + row / p.H] : 0ull;

    // stage this item's queries into TMEM (half h: columns [144 h, 144 h + 144)),
    // unless they were staged before the wait on the metadata kernel
    {
      if (!(first && b == 0 && it.g == pre_g)) stage_query_row(p, b, row, live, h, tQ);
      first = false;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(&c->q_ready, 0);
    }

    // m: running max of the scaled scores (base-2 units), the same in both
    // halves; l: this half's running sum of the weights 2^(score - m),
    // accumulated in fp32 before bf16 rounding
    float m = -INFINITY, l = 0.f;
    for (int t = it.t0; t < it.t1; ++t, ++j) {
      const int sb = j & 1;
      // tcgen05.ld is warp-collective: the warp-uniform wait leaves the warp converged
      if (!wait_warp(&c->s_full[sb], (uint32_t)(j >> 1) & 1u, c, kSiteSFull, j)) return false;
      tc_fence_after();
      uint32_t u[32];
      tmem_ld32_sync(tS + sb * kTK, u);
      // the tile is in registers: the next S MMA may overwrite this buffer
      // (relaxed: a release arrive would first wait for this thread's P
      // stores of the previous tile to reach the value CTA)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(&c->s_free[sb], 0);

      // prefix + tree mask on the raw scores.  Only tiles reaching the tree
      // tail need it; there the position relative to the first tree node lies
      // in (-64, Q + 64).  The branch is uniform across the warp (one tile,
      // one sequence), so it sits outside the loop.
      const int64_t pos0 = (int64_t)t * kTK + 32 * h;
      if (pos0 + 32 > P) {
        const int rel0 = (int)(pos0 - P);
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          const int rel = rel0 + q;  // < 0: prefix; [0, Q): tree node rel
          const bool vis = rel < 0 || (rel < nq && ((anc >> (rel & 63)) & 1ull));
          if (!vis) u[q] = 0xff800000u;  // -inf
        }
      }
      // partial row max of the raw scores in four independent chains
      float mx[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) mx[v] = __uint_as_float(u[v]);
#pragma unroll
      for (int q = 4; q < 32; ++q) mx[q & 3] = fmaxf(mx[q & 3], __uint_as_float(u[q]));
      const float pmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      // exchange with the other half of the row
      red_max[((j & 1) * 2 + h) * kRC + r] = pmax;
      __threadfence_block();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c->xch[j & 1]);
      if (!wait_warp(&c->xch[j & 1], (uint32_t)(j >> 1) & 1u, c, kSiteXch, j)) return false;
      // the scale is positive, so scaling the max equals the max of the scaled scores
      const float tmax = fmaxf(pmax, red_max[((j & 1) * 2 + (h ^ 1)) * kRC + r]) * sl2;
      // lazy running max: move it only when this tile beats it by > 8 (x 2^8)
      float alpha = 1.f;
      if (tmax > m + 8.f) {
        alpha = exp2f(m - tmax);  // 0 when m is -inf
        l *= alpha;
        m = tmax;
      }
      const float nmu = (m == -INFINITY) ? 0.f : -m;

      // wait until the value partner is done with this P buffer (and so with
      // the local staging buffer the bulk copy read it from)
      if (!wait_warp(&c->p_free[sb], ((uint32_t)(j >> 1) & 1u) ^ 1u, c, kSitePFree, j)) return false;
      uint8_t* pst = smem + kOffPStage + sb * kPBytes;
      // weights 2^(s * scale - m) as bf16, staged in the swizzled operand layout
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        uint32_t wv[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const float e0 = ex2_approx(fmaf(__uint_as_float(u[8 * q8 + 2 * v]), sl2, nmu));
          const float e1 = ex2_approx(fmaf(__uint_as_float(u[8 * q8 + 2 * v + 1]), sl2, nmu));
          ls[v] += e0 + e1;
          wv[v] = pack_bf16(e0, e1);
        }
        *reinterpret_cast<uint4*>(pst + sw128_offset(r, 32 * h + 8 * q8)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
      }
      l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      if (h == 0) reinterpret_cast<float*>(smem + kOffAStage)[sb * kRC + r] = alpha;  // one factor per row
      // the staged bytes are read by the bulk-copy engine (async proxy)
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c->p_staged[sb]);
    }

    // add the halves' row sums and hand the statistics to the value partner
    if (h == 1) {
      red_l[r] = l;
      __threadfence_block();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c->xfin);
    } else {
      if (!wait_warp(&c->xfin, (uint32_t)seg & 1u, c, kSiteXch, j)) return false;
      l += red_l[r];
      if (!wait_warp(&c->fin_free, ((uint32_t)seg & 1u) ^ 1u, c, kSiteFinFree, j)) return false;
      st_cluster_f32(mapa_shared(smem_u32(&c->lfin[r]), partner), l);
      st_cluster_f32(mapa_shared(smem_u32(&c->mfin[r]), partner), m);
      mbar_arrive_cluster(&c->fin_full, partner);
    }
    ++seg;
    return true;
  });
}

// Score CTAs, one thread: ships each staged P tile and its rescale factors to
// the value partner with two bulk copies whose bytes complete its p_full.
__device__ void p_copier(const Params& p, const Split sc, uint8_t* smem, Ctl* c, uint32_t rank, int cluster_id,
                         int n_clusters) {
  const uint32_t partner = rank + 2;
  int j = 0;
  for_items(p, sc, cluster_id, n_clusters, [&](int64_t, const Item& it) {
    for (int t = it.t0; t < it.t1; ++t, ++j) {
      const int sb = j & 1;
      if (!wait(&c->p_staged[sb], (uint32_t)(j >> 1) & 1u, c, kSitePStaged, j)) return false;
      const uint32_t bar = mapa_shared(smem_u32(&c->p_full[sb]), partner);
      bulk_copy_s2c(mapa_shared(smem_u32(smem + kOffP + sb * kPBytes), partner), smem + kOffPStage + sb * kPBytes,
                    kPBytes, bar);
      bulk_copy_s2c(mapa_shared(smem_u32(&c->alpha[sb][0]), partner), smem + kOffAStage + sb * kRC * 4, kRC * 4, bar);
      bulk_commit_group();
    }
    return true;
  });
  bulk_wait_group<0>();  // the copies have landed before this CTA may leave
}

// ---------------------------------------------------------------------------
// value pair
// ---------------------------------------------------------------------------
__device__ void value_mma(const Params& p, const Split sc, uint8_t* smem, Ctl* c, int cluster_id, int n_clusters) {
  // rank 2, whole warp; one elected lane issues each pair MMA, and checks
  // (without blocking) whether the next tile can start while these run
  const uint32_t tO = c->tmem_base;
  int j = 0;
  // PV(j) may start once its V tile has landed in both CTAs and P(j) has
  // landed in both with O holding the rescaled PV(0..j-1)
  auto ready_test = [&](int jj) {
    const bool ok = mbar_test_wait_cluster(&c->full[jj % kStagesV], (uint32_t)(jj / kStagesV) & 1u) &&
                    mbar_test_wait_cluster(&c->o_ready[jj & 1], (uint32_t)(jj >> 1) & 1u);
    return __all_sync(0xffffffffu, ok);
  };
  for_items(p, sc, cluster_id, n_clusters, [&](int64_t, const Item& it) {
    bool ready = false;
    for (int t = it.t0; t < it.t1; ++t, ++j) {
      const int s = j % kStagesV, pb = j & 1;
      if (!ready) {
        if (!wait_warp(&c->full[s], (uint32_t)(j / kStagesV) & 1u, c, kSiteFullV, j)) return false;
        if (!wait_warp(&c->o_ready[pb], (uint32_t)(j >> 1) & 1u, c, kSiteOReady, j)) return false;
      }
      fence_proxy_async_smem();
      tc_fence_after();
      const bool first = (t == it.t0);
      const uint64_t da = smem_desc(smem_u32(smem + kOffP + pb * kPBytes), 16, 1024, kLayoutSw128);
      // V: 64-column atoms 8 KB apart along N, 8-token groups 1 KB apart along K
      const uint64_t dv = smem_desc(smem_u32(smem + s * kStageV), kAtomV, 1024, kLayoutSw128);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
        for (int nh = 0; nh < 2; ++nh) {
          mma_pair_ss_warp(tO + nh * 256, da + (uint64_t)((kk * 32) >> 4),
                           dv + (uint64_t)((nh * 2 * kAtomV + kk * 16 * 128) >> 4), kIdescPV, !(first && kk == 0));
        }
        if (kk == 2) ready = (t + 1 < it.t1) && ready_test(j + 1);
      }
      mma_pair_commit_warp(&c->pv_done[pb], 0xC);
      // the same completion frees both score CTAs' P buffers (and the local
      // staging buffers their bulk copies read) without a relay
      mma_pair_commit_warp(&c->p_free[pb], 0x3);
      mma_pair_commit_warp(&c->empty[s], 0xC);
    }
    return true;
  });
  if (__any_sync(0xffffffffu, c->abort != 0)) {
    // outstanding PV MMAs must finish before TMEM is released
    mma_pair_commit_warp(&c->drain, 0x4);
    if ((threadIdx.x & 31) == 0) mbar_wait_drain(&c->drain, 0, kDrainLimitNs);
    __syncwarp();
  }
}

// Row warps of a value CTA (warpgroup h takes O columns [256 h, 256 h + 256)):
// per tile, wait for P, rescale this warp's O rows when a factor differs from
// 1, and tell the MMA-issuing CTA that O is ready; per item, normalise O and
// write the outputs (or the split partials).
__device__ void value_rows(const Params& p, const Split sc, Ctl* c, uint32_t rank, int cluster_id, int n_clusters) {
  const int lane = threadIdx.x & 31;
  const int w = (threadIdx.x >> 5) - kWarpRows;  // 0..7
  const int wq = w & 3;
  const int h = w >> 2;
  const int r = wq * 32 + lane;
  const int half = (int)(rank & 1);
  const int col0 = 256 * h;
  const uint32_t tO = c->tmem_base + ((uint32_t)(wq * 32) << 16) + (uint32_t)col0;
  const float ln2 = 0.69314718055994530942f;
  int j = 0, seg = 0;
  for_items(p, sc, cluster_id, n_clusters, [&](int64_t slot, const Item& it) {
    for (int t = it.t0; t < it.t1; ++t, ++j) {
      const int pb = j & 1;
      if (w == 0 && lane == 0) mbar_arrive_expect_tx(&c->p_full[pb], kPTxBytes);
      if (!wait_warp(&c->p_full[pb], (uint32_t)(j >> 1) & 1u, c, kSitePFull, j)) return false;
      if (t != it.t0) {
        const float a = c->alpha[pb][r];
        if (__any_sync(0xffffffffu, a != 1.f)) {
          // O must hold PV(j-1) in full before it is rescaled
          if (!wait_warp(&c->pv_done[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u, c, kSitePvPrev, j)) return false;
          tc_fence_after();
          // warp-collective TMEM traffic: every row takes part (factor 1 = unchanged)
#pragma unroll 1
          for (int c0 = 0; c0 < 256; c0 += 32) {
            uint32_t u[32];
            tmem_ld32_sync(tO + c0, u);
#pragma unroll
            for (int q = 0; q < 32; ++q) u[q] = __float_as_uint(__uint_as_float(u[q]) * a);
            tmem_st_32x32b_x32(tO + c0, u);
          }
          tmem_wait_st();
        }
      }
      fence_proxy_async_smem();  // the P bytes feed the MMA
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(&c->o_ready[pb], 2);
    }

    // epilogue of this item once its last PV is complete
    if (!wait_warp(&c->pv_done[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u, c, kSitePvLast, j)) return false;
    if (!wait_warp(&c->fin_full, (uint32_t)seg & 1u, c, kSiteFinFull, seg)) return false;
    tc_fence_after();
    const float l = c->lfin[r], m = c->mfin[r];
    mbar_arrive_cluster_relaxed(&c->fin_free, rank - 2);  // every row thread, 256 arrivals
    ++seg;
    const int row = it.g * kRG + half * kRC + r;
    const bool live = row < p.rows;  // TMEM loads stay warp-wide; only stores are per row
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse = l > 0.f ? (m + log2f(l)) * ln2 : -INFINITY;
    const int64_t orow = (int64_t)it.b * p.rows + row;
    if (slot < 0) {
      // bf16 row segments: 32-byte stores (whole sectors) when the caller's
      // array allows them, else 16-byte ones
      uint32_t* dst = reinterpret_cast<uint32_t*>(reinterpret_cast<__nv_bfloat16*>(p.out) + orow * kDl + col0);
      const bool wide = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0;
#pragma unroll 1
      for (int c0 = 0; c0 < 256; c0 += 32) {
        uint32_t u[32];
        __syncwarp();
        tmem_ld32_sync(tO + c0, u);
        if (live) {
          uint32_t w[16];
#pragma unroll
          for (int v = 0; v < 16; ++v)
            w[v] = pack_bf16(__uint_as_float(u[2 * v]) * inv, __uint_as_float(u[2 * v + 1]) * inv);
          if (wide) {
            st_global_v8(dst + c0 / 2, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
            st_global_v8(dst + c0 / 2 + 8, w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]);
          } else {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              reinterpret_cast<uint4*>(dst + c0 / 2)[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
          }
        }
      }
      if (live && p.lse && h == 0) p.lse[orow] = lse;
    } else {
      const int64_t prow = slot * kRG + half * kRC + r;
      // whole 32-byte sectors of the row (the workspace is 256-byte aligned)
      float* dst = p.part_o + prow * kDl + col0;
#pragma unroll 1
      for (int c0 = 0; c0 < 256; c0 += 32) {
        uint32_t u[32];
        __syncwarp();
        tmem_ld32_sync(tO + c0, u);
        if (live) {
#pragma unroll
          for (int v = 0; v < 4; ++v)
            st_global_v8(dst + c0 + 8 * v, __uint_as_float(u[8 * v + 0]) * inv, __uint_as_float(u[8 * v + 1]) * inv,
                         __uint_as_float(u[8 * v + 2]) * inv, __uint_as_float(u[8 * v + 3]) * inv,
                         __uint_as_float(u[8 * v + 4]) * inv, __uint_as_float(u[8 * v + 5]) * inv,
                         __uint_as_float(u[8 * v + 6]) * inv, __uint_as_float(u[8 * v + 7]) * inv);
        }
      }
      if (live && h == 0) p.part_lse[prow] = lse;
    }
    // the next item's first PV overwrites O: its o_ready follows these loads
    tc_fence_before();
    return true;
  });
}

__global__ void __cluster_dims__(kClusterCtas, 1, 1) __launch_bounds__(kThreads, 1) attn_tc_kernel(const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  const uint32_t rank = cluster_ctarank();
  const int warp = threadIdx.x >> 5;
  // The prologue (barriers, Tensor Memory, cluster sync, and for one sequence
  // the first item's queries) touches only this cluster's shared and Tensor
  // Memory and caller inputs, so it may overlap the end of the metadata
  // kernel; everything after grid_dep_wait() reads its results.
  Ctl* c = reinterpret_cast<Ctl*>(smem + kOffCtl);
  const bool leader = (rank & 1) == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesMax; ++s) {
      mbar_init(&c->full[s], kProducerThreads + (leader ? 1 : 0));
      mbar_init(&c->empty[s], 1);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(&c->s_full[q], 1);
      mbar_init(&c->s_free[q], 2 * kRowWarps);
      mbar_init(&c->xch[q], kRowWarps);
      mbar_init(&c->p_staged[q], kRowWarps);
      mbar_init(&c->p_free[q], 1);
      mbar_init(&c->p_full[q], 1);
      mbar_init(&c->pv_done[q], 1);
      mbar_init(&c->o_ready[q], 2 * kRowWarps);
    }
    mbar_init(&c->q_ready, 2 * kRowWarps);
    mbar_init(&c->fin_free, kRowThreads);
    mbar_init(&c->xfin, kRowWarps / 2);
    mbar_init(&c->fin_full, kRC);
    mbar_init(&c->drain, 1);
    mbar_init(&c->hold, 1);
    c->abort = 0;
    c->abort_site = 0;
    fence_mbar_init();
  }
  if (warp == kWarpAux) {
    tmem_alloc_pair(&c->tmem_base, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers of all CTAs initialised before any remote use
  tc_fence_after();
  // One sequence: a cluster's first work item has row group cluster mod G
  // whatever split count the metadata kernel picks, and queries are caller
  // inputs it does not write -- stage them while it runs.
  int pre_g = -1;
  if (p.B == 1 && rank < 2 && warp >= kWarpRows && warp < kWarpRows + kRowWarps) {
    const int w = warp - kWarpRows;
    const int r = (w & 3) * 32 + (threadIdx.x & 31);
    pre_g = (int)((blockIdx.x / kClusterCtas) % p.groups);
    const int row = pre_g * kRG + (int)rank * kRC + r;
    stage_query_row(p, 0, row, row < p.rows, w >> 2, c->tmem_base + 128 + ((uint32_t)((w & 3) * 32) << 16));
  }
  grid_dep_wait();
  // All CTAs of a cluster take the same branch here.  The validation bits are
  // final once the metadata kernel has completed; the timeout bit may be
  // raised by another cluster meanwhile, so it is not part of the test.
  if ((*p.err & ~MLA_DEVERR_TIMEOUT) || (smem_u32(smem) & 1023u)) {
    if (threadIdx.x == 0 && (smem_u32(smem) & 1023u)) set_err(p.err, MLA_DEVERR_LAYOUT);
    tc_fence_before();
    cluster_sync();
    if (warp == kWarpAux) tmem_dealloc_pair(c->tmem_base, kTmemCols);
    return;
  }

  const int cluster_id = blockIdx.x / kClusterCtas;
  const int n_clusters = gridDim.x / kClusterCtas;
  const Split sc = read_split(p);  // this call's work split, from the metadata kernel
  const bool score = rank < 2;
  if (warp < kProducerWarps) {
    producer(p, sc, smem, c, warp, rank, cluster_id, n_clusters);
  } else if (warp == kWarpMma) {
    if (!leader) relay(p, sc, c, rank & 2u, cluster_id, n_clusters);
    else if (score) score_mma(p, sc, smem, c, cluster_id, n_clusters);
    else value_mma(p, sc, smem, c, cluster_id, n_clusters);
  } else if (warp == kWarpAux) {
    if ((threadIdx.x & 31) == 0 && score) p_copier(p, sc, smem, c, rank, cluster_id, n_clusters);
  } else if (warp >= kWarpRows && warp < kWarpRows + kRowWarps) {
    if (score) score_softmax(p, sc, smem, c, rank, cluster_id, n_clusters, pre_g);
    else value_rows(p, sc, c, rank, cluster_id, n_clusters);
  }

  __syncwarp();
  grid_dep_launch();  // the LSE combine may start launching; it waits for this grid
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && c->abort) {
    set_err(p.err, MLA_DEVERR_TIMEOUT);
    if (c->abort_site) atomicCAS(p.err + 1, 0u, (uint32_t)c->abort_site | (rank << 8));
  }
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // no CTA leaves while a peer may still touch its shared memory
  if (warp == kWarpAux) tmem_dealloc_pair(c->tmem_base, kTmemCols);
}

}  // namespace tc

int tc_rows_per_group() { return tc::kRG; }
int tc_tokens_per_tile() { return tc::kTK; }
int tc_default_for(int dtype) { return dtype == MLA_BF16 ? MLA_ALGO_TC : MLA_ALGO_SIMT; }

// Clusters of four CTAs that can be resident at once on the current device
// (one CTA per SM), looked up once per device under a lock, so a process
// that drives GPUs of different kinds, or calls from several threads, gets
// each device's own figure.
int tc_clusters_per_gpu(int sm_count) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static int cached[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return sm_count / tc::kClusterCtas;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] > 0) return cached[dev];
  cudaFuncSetAttribute(tc::attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::kSmemAlloc);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tc::kClusterCtas * (sm_count / tc::kClusterCtas), 1, 1);
  cfg.blockDim = dim3(tc::kThreads, 1, 1);
  cfg.dynamicSmemBytes = tc::kSmemAlloc;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, tc::attn_tc_kernel, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = sm_count / tc::kClusterCtas;
  }
  cached[dev] = n;
  return n;
}

cudaError_t launch_attn_tc(const Params& p, cudaStream_t stream, bool pdl) {
  cudaError_t e = cudaFuncSetAttribute(tc::attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       tc::kSmemAlloc);
  if (e != cudaSuccess) return e;
  return launch_kernel(tc::attn_tc_kernel, dim3(tc::kClusterCtas * p.grid), dim3(tc::kThreads), tc::kSmemAlloc,
                       stream, pdl, p);
}

}  // namespace mlav
