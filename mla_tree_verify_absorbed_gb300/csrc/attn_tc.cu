// Tensor-core split-KV verify attention for sm_103a: tcgen05 MMAs with TMEM
// accumulators, asynchronous gathers of the paged KV, a 2-CTA cluster per work
// item.
//
// Shape of the problem.  Per work item, 128 query rows (absorbed queries of
// (node, head) pairs; "Ground Truth in Silicon ...", section "Input Knowledge
// Required ...", item 2) attend over KV tiles of 64 tokens whose latent kv_c
// (512) and rope key k_pe (64) are shared by all rows ("Ground Truth in
// Silicon ...", section "The Message in Full").  Both products are dense
// contractions:  S = Q [128 x 576] . K^T [576 x 64]  and
// O += P [128 x 64] . V [64 x 512]  with V = kv_c.
//
// Why two CTAs.  An fp32 accumulator for 128 rows x 512 columns is exactly
// the 512 columns x 128 lanes of one SM's Tensor Memory, so O and S cannot
// share one SM.  Each work item therefore runs on a cluster of two CTAs:
//   * the score CTA (rank 0) keeps the 128 query rows in TMEM (288 columns,
//     bf16 pairs) as the A operand of S = Q.K^T (TS form, M=128, N=64,
//     K=576 in 36 steps), double-buffers S in TMEM, and runs the online
//     softmax: one thread per row, base-2 exponent, the tree mask, and a
//     lazy running max (the max only moves when a tile beats it by more than
//     2^8, so rescaling O is rare);
//   * the value CTA (rank 1) keeps O (512 columns) in TMEM and runs
//     O += P.V (SS form, M=128, N=256 twice, K=64), with V read straight out
//     of the staged kv_c tile as an MN-major operand.
// P (bf16) and the per-row rescale factors travel from the score CTA's
// registers into the value CTA's shared memory as st.async stores whose bytes
// complete the value CTA's barrier.  The value CTA also writes the outputs.
//
// Data movement.  Each CTA stages its own 64-token KV tiles, three in flight:
// eight producer warps gather every token's pool row (kv_c, and k_pe in the
// score CTA) with 16-byte cp.async copies written straight into the 128-byte
// swizzled K-major layout the MMAs read, one 1 KB kv_c row per warp
// instruction pair so each instruction reads 512 contiguous bytes; slot
// indices are fetched one tile ahead.  Measured on GB300, the rate at which
// one SM can gather scattered rows grows with the number of warps issuing
// copies (outstanding requests per warp are limited): about 9 B/clk with two
// warps and 50 B/clk with eight when the rows sit in L2; a TMA tile::gather4
// version (four 128-byte rows per instruction) managed about 7 B/clk.  L2
// bandwidth is ample, so each CTA loading its own copy costs nothing that
// matters.  Each staged tile is reused by all 128 rows of the item -- the
// head-tile reuse of "The Critical Glue: Validating a Custom Flash Attention
// Kernel Through Test Infrastructure", section "What Came Before", widened to
// every (node, head) row.
//
// Every wait is bounded; on timeout the kernel sets MLA_DEVERR_TIMEOUT, stops
// issuing work, drains what it issued, frees TMEM and returns.
#include "common.cuh"
#include "sm100.cuh"

namespace mlav {
using namespace sm100;

namespace tc {

constexpr int kRG = 128;        // query rows per work item (MMA M)
constexpr int kTK = 64;         // tokens per KV tile
constexpr int kStages = 3;      // KV tiles in flight
constexpr int kThreads = 512;   // 16 warps
constexpr uint32_t kTmemCols = 512;

// warp roles
constexpr int kProducerWarps = 8;                  // warps 0-7
constexpr int kProducerThreads = 32 * kProducerWarps;
constexpr int kTokPerWarp = kTK / kProducerWarps;  // 8 tokens of each tile per producer warp
constexpr int kWarpMma = 8, kWarpRelease = 9, kWarpTmem = 10, kWarpRows = 12;  // rows: 12-15

constexpr int kChunk = kTK * 128;            // one 64-column bf16 chunk of a tile: 8 KB
constexpr int kKvcStage = 8 * kChunk;        // kv_c of one tile: 64 KB
constexpr int kOffKvc = 0;                   // [kStages][64 KB]
constexpr int kOffKpe = kStages * kKvcStage; // score CTA: [kStages][8 KB]
constexpr int kOffP = kStages * kKvcStage;   // value CTA: [2][16 KB]
constexpr int kPBytes = kRG * 128;           // P tile [128 rows x 64 tokens] bf16
constexpr int kOffCtl = kStages * kKvcStage + 2 * kPBytes;
constexpr uint32_t kKpeBytes = kTK * kDr * 2;      // 8192
constexpr uint32_t kPTxBytes = kPBytes + kRG * 4;  // P tile + alpha, per tile

// Byte strides of the MN-major V operand (tile chunk = 64 columns x 64 rows):
// between 64-column atoms along N, and between 8-row groups along K.
constexpr uint32_t kVAtomStrideN = kChunk;   // 8192
constexpr uint32_t kVGroupStrideK = 1024;

constexpr uint32_t kIdescS = idesc_bf16_f32(128, kTK, 0, 0);   // A (Q, TMEM), B (K tile) K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, 0, 1);  // A (P) K-major, B (V) MN-major

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr uint64_t kDrainLimitNs = 20000000ull;   // 20 ms per drain wait on abort

enum { kCmdRescale = 1, kCmdEpilogue = 2, kCmdExit = 3 };

struct alignas(16) Ctl {
  uint64_t full[kStages];   // KV tile landed (kProducerThreads cp.async arrivals)
  uint64_t empty[kStages];  // stage reusable: the MMAs reading it are complete
  uint64_t s_full[2];       // score: S tile in TMEM
  uint64_t s_free[2];       // score: softmax has read S (128 arrivals)
  uint64_t p_free[2];       // score: value CTA finished with its P buffer
  uint64_t q_ready;         // score: queries staged in TMEM (128 arrivals)
  uint64_t fin_free;        // score: value CTA consumed lfin/mfin (128 remote arrivals)
  uint64_t p_full[2];       // value: P tile and alpha landed (st.async bytes; armed by the MMA thread)
  uint64_t pv_done[2];      // value: PV MMAs of a tile complete
  uint64_t fin_full;        // value: lfin/mfin written (128 remote arrivals)
  uint64_t cmd_full;        // value: a command for the epilogue warps
  uint64_t cmd_done;        // value: command finished (128 arrivals)
  uint64_t drain;           // both: final MMA drain on abort
  float alpha[2][kRG];      // value: per-row rescale of O before PV(j) (1 = unchanged)
  float lfin[kRG];          // value: final row sums of the weights
  float mfin[kRG];          // value: final running max (base-2 units)
  uint32_t tmem_base;
  int abort;
  int abort_site;
  int cmd;
  int cmd_buf;
  long long cmd_item;
};
constexpr int kSmemBytes = kOffCtl + (int)sizeof(Ctl);
constexpr int kSmemAlloc = 232448;  // the per-CTA maximum; the base must be 1024-aligned
static_assert(kSmemBytes <= kSmemAlloc, "shared memory budget");
static_assert(kOffKpe + kStages * (int)kKpeBytes <= kOffCtl, "k_pe stages overlap control block");
static_assert(kWarpRows % 4 == 0, "the row warps must form a warpgroup (TMEM lane quadrants)");

// Wait sites, recorded in the workspace's second error word when a wait gives up.
enum {
  kSiteEmpty = 1, kSiteQReady, kSiteFullS, kSiteSFree, kSiteSFull, kSitePFree, kSiteFinFree,
  kSiteFullV, kSitePFull, kSitePvPrev, kSiteCmdDone, kSitePvLast, kSiteRelease, kSiteCmdFull, kSiteFinFull
};

__device__ __forceinline__ bool wait(uint64_t* bar, uint32_t parity, Ctl* c, int site, int j,
                                     bool cluster = false) {
  if (mbar_wait(bar, parity, &c->abort, kWaitLimitNs, cluster)) return true;
  // first site to give up in this CTA (others follow the abort flag)
  atomicCAS(&c->abort_site, 0, (site & 0xff) | ((j & 0xffff) << 16));
  return false;
}

// The same wait made by every lane of a warp; the result is warp-uniform and
// the warp is converged on return (the MMA roles issue with elect.sync).
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, Ctl* c, int site, int j,
                                          bool cluster = false) {
  return __all_sync(0xffffffffu, wait(bar, parity, c, site, j, cluster));
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

// ---------------------------------------------------------------------------
// producers (both CTAs)
// ---------------------------------------------------------------------------
// Stages the KV tiles of this CTA's items.  Producer warp pw copies tokens
// [8 pw, 8 pw + 8) of each tile: for every token, two warp instructions move
// its 1 KB kv_c row (lane l moves bytes 16l.. of each half), placing 16-byte
// piece q of 64-column chunk ch of token row r at
//   ch * kChunk + r * 128 + ((q ^ (r & 7)) * 16)
// -- the 128-byte swizzle of the K-major operand layout.  In the score CTA two
// more instructions move the 128-byte k_pe rows (four tokens each).  Positions
// past the sequence read slot 0; the softmax gives them zero weight.
__device__ void producer(const Params& p, uint8_t* smem, Ctl* c, int pw, bool with_kpe, int cluster_id,
                         int n_clusters) {
  const int lane = threadIdx.x & 31;
  const __nv_bfloat16* kvc_g = reinterpret_cast<const __nv_bfloat16*>(p.kv_c);
  const __nv_bfloat16* kpe_g = reinterpret_cast<const __nv_bfloat16*>(p.k_pe);
  const uint32_t sbase = smem_u32(smem);
  const int r0 = kTokPerWarp * pw;
  int j = 0;
  for (int64_t item = cluster_id; item < p.n_items; item += n_clusters) {
    const Item it = item_at(p, item);
    if (it.t1 <= it.t0) continue;
    const int b = it.b;
    const int64_t N = (int64_t)p.prefix_lens[b] + p.Q;
    const int64_t idx0 = p.page_size == 1 ? (int64_t)p.kv_indptr[b] : 0;
    // slot of token r0 + (lane % 8) of tile t
    auto slot_of = [&](int t) -> int64_t {
      const int64_t pos = (int64_t)t * kTK + r0 + (lane & (kTokPerWarp - 1));
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
      const int s = j % kStages;
      const int64_t slot = next;
      if (t + 1 < it.t1) next = slot_of(t + 1);  // index load for the next tile, in flight meanwhile
      bool ok = true;
      if (lane == 0) ok = wait(&c->empty[s], ((uint32_t)(j / kStages) & 1u) ^ 1u, c, kSiteEmpty, j);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const uint32_t stage = sbase + kOffKvc + s * kKvcStage;
#pragma unroll
      for (int tt = 0; tt < kTokPerWarp; ++tt) {
        const int64_t sl = __shfl_sync(0xffffffffu, slot, tt);
        const int r = r0 + tt;
        const __nv_bfloat16* src = kvc_g + sl * p.kv_c_stride;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int g = lane + 32 * h;  // 16-byte piece of the row
          const int ch = g >> 3, q = g & 7;
          cp_async_16(stage + ch * kChunk + r * 128 + ((q ^ (r & 7)) << 4), src + g * 8);
        }
      }
      if (with_kpe) {
        const uint32_t kst = sbase + kOffKpe + s * kKpeBytes;
#pragma unroll
        for (int gg = 0; gg < kTokPerWarp / 4; ++gg) {
          const int tt = gg * 4 + (lane >> 3), q = lane & 7;
          const int64_t sl = __shfl_sync(0xffffffffu, slot, tt);
          const int r = r0 + tt;
          cp_async_16(kst + r * 128 + ((q ^ (r & 7)) << 4), kpe_g + sl * p.k_pe_stride + q * 8);
        }
      }
      cp_async_mbar_arrive(&c->full[s]);
    }
  }
  // copies already issued must land before this CTA may exit
  cp_async_wait_all();
}

// ---------------------------------------------------------------------------
// score CTA roles
// ---------------------------------------------------------------------------
__device__ void score_mma(const Params& p, uint8_t* smem, Ctl* c, int cluster_id, int n_clusters) {
  // run by the whole warp; one elected lane issues each tcgen05 op
  const uint32_t tS = c->tmem_base;        // columns [0, 128): two S buffers
  const uint32_t tQ = c->tmem_base + 128;  // columns [128, 416): queries, bf16 pairs
  int j = 0, seg = 0;
  bool ok = true;
  for (int64_t item = cluster_id; item < p.n_items && ok; item += n_clusters) {
    const Item it = item_at(p, item);
    if (it.t1 <= it.t0) continue;
    if (!(ok = wait_warp(&c->q_ready, (uint32_t)seg & 1u, c, kSiteQReady, j))) break;
    tc_fence_after();
    for (int t = it.t0; t < it.t1; ++t, ++j) {
      const int s = j % kStages, sb = j & 1;
      if (!(ok = wait_warp(&c->full[s], (uint32_t)(j / kStages) & 1u, c, kSiteFullS, j))) break;
      // Issue S(j) only after the softmax has loaded S(j-1): a TMEM load waits
      // behind MMAs issued before it, so issuing S(j) first would hold the
      // softmax's load of S(j-1) until S(j) completes.  (This also implies
      // buffer sb, last read for S(j-2), is free.)
      if (j > 0 && !(ok = wait_warp(&c->s_free[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u, c, kSiteSFree, j)))
        break;
      fence_proxy_async_smem();  // cp.async data, written through the generic proxy, feeds the MMA
      tc_fence_after();
      // descriptors differ only in the start-address field: add (offset >> 4)
      const uint64_t dk = smem_desc(smem_u32(smem + kOffKvc + s * kKvcStage), 16, 1024, kLayoutSw128);
      const uint64_t dp = smem_desc(smem_u32(smem + kOffKpe + s * kKpeBytes), 16, 1024, kLayoutSw128);
      const uint32_t ts = tS + sb * kTK;
#pragma unroll
      for (int kc = 0; kc < 9; ++kc) {
        // chunks 0-7: the latent part in the kv_c stage; chunk 8: the rope part in the k_pe stage
        const uint64_t bd = kc < 8 ? dk + (uint64_t)((kc * kChunk) >> 4) : dp;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts_warp(ts, tQ + kc * 32 + kk * 8, bd + (uint64_t)((kk * 32) >> 4), kIdescS, (kc | kk) != 0);
      }
      mma_commit_warp(&c->s_full[sb]);
      mma_commit_warp(&c->empty[s]);
    }
    ++seg;
  }
  if (__any_sync(0xffffffffu, c->abort != 0)) {
    // outstanding S MMAs must finish before TMEM is released
    mma_commit_warp(&c->drain);
    if ((threadIdx.x & 31) == 0) mbar_wait_drain(&c->drain, 0, kDrainLimitNs);
    __syncwarp();
  }
}

__device__ void score_softmax(const Params& p, uint8_t* smem, Ctl* c, int cluster_id, int n_clusters) {
  const int wq = (threadIdx.x >> 5) & 3;            // TMEM lane quadrant of this warp
  const int r = wq * 32 + (threadIdx.x & 31);        // row within the item
  const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
  const uint32_t tS = c->tmem_base + lane_off;
  const uint32_t tQ = c->tmem_base + 128 + lane_off;
  const float sl2 = p.scale_log2;
  const int nq = p.Q;
  int j = 0, seg = 0;
  for (int64_t item = cluster_id; item < p.n_items; item += n_clusters) {
    const Item it = item_at(p, item);
    if (it.t1 <= it.t0) continue;
    const int b = it.b;
    const int row = it.g * kRG + r;
    const bool live = row < p.rows;
    const int64_t P = p.prefix_lens[b];
    const uint64_t anc = live ? p.anc[(int64_t)b * p.Q + row / p.H] : 0ull;

    // stage this item's queries into TMEM: column c holds elements 2c, 2c+1
    {
      const uint4* ql = reinterpret_cast<const uint4*>(p.q_lat) + ((int64_t)b * p.rows + row) * (kDl / 8);
      const uint4* qp = reinterpret_cast<const uint4*>(p.q_pe) + ((int64_t)b * p.rows + row) * (kDr / 8);
#pragma unroll 1
      for (int c0 = 0; c0 < 288; c0 += 16) {
        uint32_t w[16];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int col = c0 + 4 * v;  // 4 columns per 16-byte vector
          uint4 x = make_uint4(0, 0, 0, 0);
          if (live) x = col < 256 ? ql[col / 4] : qp[(col - 256) / 4];
          w[4 * v + 0] = x.x;
          w[4 * v + 1] = x.y;
          w[4 * v + 2] = x.z;
          w[4 * v + 3] = x.w;
        }
        __syncwarp();
        tmem_st_32x32b_x16(tQ + c0, w);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&c->q_ready);
    }

    // m: running max of the scaled scores (base-2 units); l: running sum of
    // the weights 2^(score - m), accumulated in fp32 before bf16 rounding
    float m = -INFINITY, l = 0.f;
    for (int t = it.t0; t < it.t1; ++t, ++j) {
      const int sb = j & 1;
      if (!wait(&c->s_full[sb], (uint32_t)(j >> 1) & 1u, c, kSiteSFull, j)) return;
      __syncwarp();  // tcgen05.ld is warp-collective: reconverge after the spin
      tc_fence_after();
      uint32_t u[kTK];
      tmem_ld64_sync(tS + sb * kTK, u);
      // the tile is in registers: the next S MMA may overwrite this buffer
      tc_fence_before();
      mbar_arrive(&c->s_free[sb]);

      // prefix + tree mask on the raw scores.  Only tiles reaching the tree
      // tail need it; there the position relative to the first tree node lies
      // in (-64, Q + 64).  The branch is uniform across the warp (one tile,
      // one sequence), so it sits outside the loop.
      const int64_t pos0 = (int64_t)t * kTK;
      if (pos0 + kTK > P) {
        const int rel0 = (int)(pos0 - P);
#pragma unroll
        for (int q = 0; q < kTK; ++q) {
          const int rel = rel0 + q;  // < 0: prefix; [0, Q): tree node rel
          const bool vis = rel < 0 || (rel < nq && ((anc >> (rel & 63)) & 1ull));
          if (!vis) u[q] = 0xff800000u;  // -inf
        }
      }
      // row max of the raw scores in eight independent chains; the scale is
      // positive, so scaling the max equals the max of the scaled scores
      float mx[8];
#pragma unroll
      for (int v = 0; v < 8; ++v) mx[v] = __uint_as_float(u[v]);
#pragma unroll
      for (int q = 8; q < kTK; ++q) mx[q & 7] = fmaxf(mx[q & 7], __uint_as_float(u[q]));
      const float tmax =
          fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) *
          sl2;
      // lazy running max: move it only when this tile beats it by > 8 (x 2^8)
      float alpha = 1.f;
      if (tmax > m + 8.f) {
        alpha = exp2f(m - tmax);  // 0 when m is -inf
        l *= alpha;
        m = tmax;
      }
      const float nmu = (m == -INFINITY) ? 0.f : -m;

      // wait until the value CTA is done with this P buffer
      if (!wait(&c->p_free[sb], ((uint32_t)(j >> 1) & 1u) ^ 1u, c, kSitePFree, j, true)) return;
      const uint32_t pbase = mapa_shared(smem_u32(smem + kOffP + sb * kPBytes), 1);
      const uint32_t pbar = mapa_shared(smem_u32(&c->p_full[sb]), 1);
      // weights 2^(s * scale - m) as bf16, shipped 16 bytes at a time
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q8 = 0; q8 < kTK / 8; ++q8) {
        uint32_t w[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const float e0 = ex2_approx(fmaf(__uint_as_float(u[8 * q8 + 2 * v]), sl2, nmu));
          const float e1 = ex2_approx(fmaf(__uint_as_float(u[8 * q8 + 2 * v + 1]), sl2, nmu));
          ls[v] += e0 + e1;
          w[v] = pack_bf16(e0, e1);
        }
        st_async_v4(pbase + sw128_offset(r, 8 * q8), w[0], w[1], w[2], w[3], pbar);
      }
      l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      // every row ships its factor; the bytes themselves complete p_full
      st_async_f32(mapa_shared(smem_u32(&c->alpha[sb][r]), 1), alpha, pbar);
    }

    // hand the row statistics to the value CTA for the epilogue
    if (!wait(&c->fin_free, ((uint32_t)seg & 1u) ^ 1u, c, kSiteFinFree, j, true)) return;
    st_cluster_f32(mapa_shared(smem_u32(&c->lfin[r]), 1), l);
    st_cluster_f32(mapa_shared(smem_u32(&c->mfin[r]), 1), m);
    mbar_arrive_cluster(&c->fin_full, 1);
    ++seg;
  }
}

// ---------------------------------------------------------------------------
// value CTA roles
// ---------------------------------------------------------------------------
__device__ void value_mma(const Params& p, uint8_t* smem, Ctl* c, int cluster_id, int n_clusters) {
  // run by the whole warp; one elected lane issues each tcgen05 op, lane 0
  // makes the single-count arrivals
  const uint32_t tO = c->tmem_base;
  const int lane = threadIdx.x & 31;
  int j = 0, ncmd = 0;
  bool ok = true;
  for (int64_t item = cluster_id; item < p.n_items && ok; item += n_clusters) {
    const Item it = item_at(p, item);
    if (it.t1 <= it.t0) continue;
    for (int t = it.t0; t < it.t1; ++t, ++j) {
      const int s = j % kStages, pb = j & 1;
      if (!(ok = wait_warp(&c->full[s], (uint32_t)(j / kStages) & 1u, c, kSiteFullV, j))) break;
      if (lane == 0) mbar_arrive_expect_tx(&c->p_full[pb], kPTxBytes);
      if (!(ok = wait_warp(&c->p_full[pb], (uint32_t)(j >> 1) & 1u, c, kSitePFull, j, true))) break;
      const bool first = (t == it.t0);
      bool rescale = false;
      if (!first) {
        const float4 a = reinterpret_cast<const float4*>(c->alpha[pb])[lane];  // 4 of the 128 rows per lane
        rescale = __any_sync(0xffffffffu, (a.x != 1.f) | (a.y != 1.f) | (a.z != 1.f) | (a.w != 1.f));
      }
      if (rescale) {
        // O must hold PV(j-1) in full before it is rescaled
        if (!(ok = wait_warp(&c->pv_done[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u, c, kSitePvPrev, j))) break;
        tc_fence_after();
        if (lane == 0) {
          c->cmd = kCmdRescale;
          c->cmd_buf = pb;
          mbar_arrive(&c->cmd_full);
        }
        if (!(ok = wait_warp(&c->cmd_done, (uint32_t)ncmd & 1u, c, kSiteCmdDone, j))) break;
        ++ncmd;
      }
      fence_proxy_async_smem();
      tc_fence_after();
      const uint64_t da = smem_desc(smem_u32(smem + kOffP + pb * kPBytes), 16, 1024, kLayoutSw128);
      const uint64_t dv = smem_desc(smem_u32(smem + kOffKvc + s * kKvcStage), kVAtomStrideN, kVGroupStrideK,
                                    kLayoutSw128);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
        for (int nh = 0; nh < 2; ++nh) {
          mma_ss_warp(tO + nh * 256, da + (uint64_t)((kk * 32) >> 4),
                      dv + (uint64_t)((nh * 4 * kChunk + kk * 16 * 128) >> 4), kIdescPV, !(first && kk == 0));
        }
      }
      mma_commit_warp(&c->pv_done[pb]);
      mma_commit_warp(&c->empty[s]);
    }
    if (!ok) break;
    // epilogue of this item once its last PV is complete
    if (!(ok = wait_warp(&c->pv_done[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u, c, kSitePvLast, j))) break;
    tc_fence_after();
    if (lane == 0) {
      c->cmd = kCmdEpilogue;
      c->cmd_item = item;
      mbar_arrive(&c->cmd_full);
    }
    if (!(ok = wait_warp(&c->cmd_done, (uint32_t)ncmd & 1u, c, kSiteCmdDone, j))) break;
    ++ncmd;
  }
  if (lane == 0) {
    c->cmd = kCmdExit;
    mbar_arrive(&c->cmd_full);
  }
  if (__any_sync(0xffffffffu, c->abort != 0)) {
    // outstanding PV MMAs must finish before TMEM is released
    mma_commit_warp(&c->drain);
    if (lane == 0) mbar_wait_drain(&c->drain, 0, kDrainLimitNs);
  }
  __syncwarp();
}

// Releases each tile's P buffer back to the score CTA once the PV MMAs that
// read it have completed.
__device__ void value_release(const Params& p, Ctl* c, int cluster_id, int n_clusters) {
  int j = 0;
  for (int64_t item = cluster_id; item < p.n_items; item += n_clusters) {
    const Item it = item_at(p, item);
    for (int t = it.t0; t < it.t1; ++t, ++j) {
      if (!wait(&c->pv_done[j & 1], (uint32_t)(j >> 1) & 1u, c, kSiteRelease, j)) return;
      mbar_arrive_cluster(&c->p_free[j & 1], 0);
    }
  }
}

__device__ void value_epilogue(const Params& p, Ctl* c) {
  const int wq = (threadIdx.x >> 5) & 3;
  const int r = wq * 32 + (threadIdx.x & 31);
  const uint32_t tO = c->tmem_base + ((uint32_t)(wq * 32) << 16);
  int ncmd = 0, seg = 0;
  const float ln2 = 0.69314718055994530942f;
  while (true) {
    if (!wait(&c->cmd_full, (uint32_t)ncmd & 1u, c, kSiteCmdFull, ncmd)) return;
    __syncwarp();
    ++ncmd;
    const int cmd = c->cmd;
    if (cmd == kCmdExit) return;
    tc_fence_after();
    if (cmd == kCmdRescale) {
      // warp-collective TMEM traffic: every row takes part (factor 1 = unchanged)
      const float a = c->alpha[c->cmd_buf][r];
#pragma unroll 1
      for (int c0 = 0; c0 < kDl; c0 += 32) {
        uint32_t u[32];
        tmem_ld32_sync(tO + c0, u);
#pragma unroll
        for (int q = 0; q < 32; ++q) u[q] = __float_as_uint(__uint_as_float(u[q]) * a);
        tmem_st_32x32b_x32(tO + c0, u);
      }
      tmem_wait_st();
    } else {  // kCmdEpilogue
      const Item it = item_at(p, c->cmd_item);
      if (!wait(&c->fin_full, (uint32_t)seg & 1u, c, kSiteFinFull, seg, true)) return;
      __syncwarp();
      const float l = c->lfin[r], m = c->mfin[r];
      mbar_arrive_cluster(&c->fin_free, 0);
      ++seg;
      const int row = it.g * kRG + r;
      const bool live = row < p.rows;  // TMEM loads stay warp-wide; only stores are per row
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse = l > 0.f ? (m + log2f(l)) * ln2 : -INFINITY;
      const int64_t orow = (int64_t)it.b * p.rows + row;
      if (p.splits == 1) {
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + orow * kDl);
#pragma unroll 1
        for (int c0 = 0; c0 < kDl; c0 += 32) {
          uint32_t u[32];
          __syncwarp();
          tmem_ld32_sync(tO + c0, u);
          if (live) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 o;
              o.x = pack_bf16(__uint_as_float(u[8 * v + 0]) * inv, __uint_as_float(u[8 * v + 1]) * inv);
              o.y = pack_bf16(__uint_as_float(u[8 * v + 2]) * inv, __uint_as_float(u[8 * v + 3]) * inv);
              o.z = pack_bf16(__uint_as_float(u[8 * v + 4]) * inv, __uint_as_float(u[8 * v + 5]) * inv);
              o.w = pack_bf16(__uint_as_float(u[8 * v + 6]) * inv, __uint_as_float(u[8 * v + 7]) * inv);
              dst[c0 / 8 + v] = o;
            }
          }
        }
        if (live && p.lse) p.lse[orow] = lse;
      } else {
        const int64_t prow = c->cmd_item * kRG + r;
        float4* dst = reinterpret_cast<float4*>(p.part_o + prow * kDl);
#pragma unroll 1
        for (int c0 = 0; c0 < kDl; c0 += 32) {
          uint32_t u[32];
          __syncwarp();
          tmem_ld32_sync(tO + c0, u);
          if (live) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[c0 / 4 + v] = make_float4(__uint_as_float(u[4 * v + 0]) * inv, __uint_as_float(u[4 * v + 1]) * inv,
                                            __uint_as_float(u[4 * v + 2]) * inv, __uint_as_float(u[4 * v + 3]) * inv);
          }
        }
        if (live) p.part_lse[prow] = lse;
      }
    }
    tc_fence_before();
    mbar_arrive(&c->cmd_done);
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) attn_tc_kernel(const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  const uint32_t rank = cluster_ctarank();
  const int warp = threadIdx.x >> 5;
  // Both CTAs of a cluster must take the same branch here.  The validation bits
  // were final before this kernel started; the timeout bit may be raised by
  // another cluster while this one starts, so it is not part of the test.
  if ((*p.err & ~MLA_DEVERR_TIMEOUT) || (smem_u32(smem) & 1023u)) {
    if (threadIdx.x == 0 && (smem_u32(smem) & 1023u)) set_err(p.err, MLA_DEVERR_LAYOUT);
    return;
  }
  Ctl* c = reinterpret_cast<Ctl*>(smem + kOffCtl);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&c->full[s], kProducerThreads);
      mbar_init(&c->empty[s], 1);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(&c->s_full[q], 1);
      mbar_init(&c->s_free[q], kRG);
      mbar_init(&c->p_free[q], 1);
      mbar_init(&c->p_full[q], 1);
      mbar_init(&c->pv_done[q], 1);
    }
    mbar_init(&c->q_ready, kRG);
    mbar_init(&c->fin_free, kRG);
    mbar_init(&c->fin_full, kRG);
    mbar_init(&c->cmd_full, 1);
    mbar_init(&c->cmd_done, kRG);
    mbar_init(&c->drain, 1);
    c->abort = 0;
    c->abort_site = 0;
    fence_mbar_init();
  }
  if (warp == kWarpTmem) {
    tmem_alloc(&c->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised before any remote use
  tc_fence_after();

  const int cluster_id = blockIdx.x >> 1;
  const int n_clusters = gridDim.x >> 1;
  if (warp < kProducerWarps) {
    producer(p, smem, c, warp, rank == 0, cluster_id, n_clusters);
  } else if (rank == 0) {
    if (warp == kWarpMma) score_mma(p, smem, c, cluster_id, n_clusters);
    else if (warp >= kWarpRows) score_softmax(p, smem, c, cluster_id, n_clusters);
  } else {
    if (warp == kWarpMma) value_mma(p, smem, c, cluster_id, n_clusters);
    else if (warp == kWarpRelease) { if ((threadIdx.x & 31) == 0) value_release(p, c, cluster_id, n_clusters); }
    else if (warp >= kWarpRows) value_epilogue(p, c);
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && c->abort) {
    set_err(p.err, MLA_DEVERR_TIMEOUT);
    atomicCAS(p.err + 1, 0u, (uint32_t)c->abort_site | (rank << 8));
  }
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // no CTA leaves while its peer may still touch its shared memory
  if (warp == kWarpTmem) tmem_dealloc(c->tmem_base, kTmemCols);
}

}  // namespace tc

int tc_rows_per_group() { return tc::kRG; }
int tc_tokens_per_tile() { return tc::kTK; }
int tc_default_for(int dtype) { return dtype == MLA_BF16 ? MLA_ALGO_TC : MLA_ALGO_SIMT; }

// Clusters of two CTAs that can be resident at once (one CTA per SM).
int tc_clusters_per_gpu(int sm_count) {
  static int cached = -1;
  if (cached > 0) return cached;
  cudaFuncSetAttribute(tc::attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::kSmemAlloc);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sm_count / 2), 1, 1);
  cfg.blockDim = dim3(tc::kThreads, 1, 1);
  cfg.dynamicSmemBytes = tc::kSmemAlloc;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, tc::attn_tc_kernel, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = sm_count / 2;
  }
  cached = n;
  return n;
}

cudaError_t launch_attn_tc(const Params& p, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(tc::attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       tc::kSmemAlloc);
  if (e != cudaSuccess) return e;
  tc::attn_tc_kernel<<<2 * p.grid, tc::kThreads, tc::kSmemAlloc, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mlav
