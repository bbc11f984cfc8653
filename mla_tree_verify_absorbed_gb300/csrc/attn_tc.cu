// Tensor-core split-KV verify attention for sm_103a: tcgen05 MMAs with TMEM
// accumulators, TMA gathers of the paged KV, a 2-CTA cluster per work item.
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
// P (bf16) travels from the score CTA's registers into the value CTA's
// shared memory through distributed shared memory; the rare rescale factors
// ride along.  The value CTA also writes the outputs.
//
// Data movement.  A producer warp in the score CTA gathers each 64-token tile
// with TMA tile::gather4 (four pool rows per instruction, 128-byte swizzle,
// 64-column boxes), kv_c multicast to both CTAs of the cluster, k_pe to the
// score CTA only; three stages in flight.  Each staged tile is reused by all
// 128 rows of the item -- the head-tile reuse of "The Critical Glue:
// Validating a Custom Flash Attention Kernel Through Test Infrastructure",
// section "What Came Before", widened to every (node, head) row.
//
// Every wait is bounded; on timeout the kernel sets MLA_DEVERR_TIMEOUT, stops
// issuing work, drains what it issued, frees TMEM and returns.
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "sm100.cuh"

namespace mlav {
using namespace sm100;

namespace tc {

constexpr int kRG = 128;        // query rows per work item (MMA M)
constexpr int kTK = 64;         // tokens per KV tile
constexpr int kStages = 3;      // KV tiles in flight
constexpr int kThreads = 256;   // 8 warps
constexpr uint32_t kTmemCols = 512;

constexpr int kChunk = kTK * 128;            // one 64-column bf16 chunk of a tile: 8 KB
constexpr int kKvcStage = 8 * kChunk;        // kv_c of one tile: 64 KB
constexpr int kOffKvc = 0;                   // [kStages][64 KB], same offset in both CTAs
constexpr int kOffKpe = kStages * kKvcStage; // score CTA: [kStages][8 KB]
constexpr int kOffP = kStages * kKvcStage;   // value CTA: [2][16 KB]
constexpr int kPBytes = kRG * 128;           // P tile [128 rows x 64 tokens] bf16
constexpr int kOffCtl = kStages * kKvcStage + 2 * kPBytes;
constexpr uint32_t kKvcBytes = kTK * kDl * 2;  // 65536
constexpr uint32_t kKpeBytes = kTK * kDr * 2;  // 8192

// Byte strides of the MN-major V operand (tile chunk = 64 columns x 64 rows):
// between 64-column atoms along N, and between 8-row groups along K.
constexpr uint32_t kVAtomStrideN = kChunk;   // 8192
constexpr uint32_t kVGroupStrideK = 1024;
#ifndef MLA_TC_V_LBO
#define MLA_TC_V_LBO kVAtomStrideN
#define MLA_TC_V_SBO kVGroupStrideK
#endif

constexpr uint32_t kIdescS = idesc_bf16_f32(128, kTK, 0, 0);   // A (Q, TMEM), B (K tile) K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, 0, 1);  // A (P) K-major, B (V) MN-major

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr uint64_t kDrainLimitNs = 20000000ull;   // 20 ms per drain wait on abort

enum { kCmdRescale = 1, kCmdEpilogue = 2, kCmdExit = 3 };

struct alignas(16) Ctl {
  uint64_t full[kStages];   // KV tile landed (score: kv_c + k_pe, value: kv_c)
  uint64_t empty[kStages];  // score: stage reusable (S MMA done + value CTA's PV done)
  uint64_t s_full[2];       // score: S tile in TMEM
  uint64_t s_free[2];       // score: softmax has read S (128 arrivals)
  uint64_t p_free[2];       // score: value CTA finished with its P buffer
  uint64_t q_ready;         // score: queries staged in TMEM (128 arrivals)
  uint64_t fin_free;        // score: value CTA consumed lfin/mfin (128 remote arrivals)
  uint64_t p_full[2];       // value: P, alpha and flag written (128 remote arrivals)
  uint64_t pv_done[2];      // value: PV MMAs of a tile complete
  uint64_t fin_full;        // value: lfin/mfin written (128 remote arrivals)
  uint64_t cmd_full;        // value: a command for the epilogue warps
  uint64_t cmd_done;        // value: command finished (128 arrivals)
  uint64_t drain;           // both: final MMA drain on abort
  float alpha[2][kRG];      // value: per-row rescale of O before PV(j)
  int flag[2];              // value: some row of tile j rescaled
  float lfin[kRG];          // value: final row sums of the bf16-rounded p (normalises out)
  float lxfin[kRG];         // value: final row sums of the unrounded p (gives lse)
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

__device__ __forceinline__ void red_or_cluster(uint32_t caddr, uint32_t v) {
  asm volatile("red.relaxed.cluster.shared::cluster.or.b32 [%0], %1;" ::"r"(caddr), "r"(v) : "memory");
}

__device__ __forceinline__ void tma_gather4_mc(void* dst, const CUtensorMap* map, int32_t x, int32_t y0,
                                               int32_t y1, int32_t y2, int32_t y3, uint64_t* bar,
                                               uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      ".multicast::cluster [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ---------------------------------------------------------------------------
// score CTA roles
// ---------------------------------------------------------------------------
__device__ void score_producer(const Params& p, const CUtensorMap* map_kvc, const CUtensorMap* map_kpe,
                               uint8_t* smem, Ctl* c, int cluster_id, int n_clusters) {
  const int lane = threadIdx.x & 31;
  int j = 0;
  for (int64_t item = cluster_id; item < p.n_items; item += n_clusters) {
    const Item it = item_at(p, item);
    const int b = it.b;
    const int64_t N = (int64_t)p.prefix_lens[b] + p.Q;
    for (int t = it.t0; t < it.t1; ++t, ++j) {
      const int s = j % kStages;
      const uint32_t ph = (uint32_t)(j / kStages) & 1u;
      bool ok = true;
      if (lane == 0) {
        ok = wait(&c->empty[s], ph ^ 1u, c, kSiteEmpty, j, true);
        if (ok) mbar_arrive_expect_tx(&c->full[s], kKvcBytes + kKpeBytes);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) return;
      if (lane < kTK / 4) {
        int32_t y[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int64_t pos = (int64_t)t * kTK + lane * 4 + q;
          y[q] = (int32_t)(pos < N ? resolve_slot(p, b, pos) : 0);
        }
        uint8_t* kvc = smem + kOffKvc + s * kKvcStage + lane * 512;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          tma_gather4_mc(kvc + ch * kChunk, map_kvc, ch * 64, y[0], y[1], y[2], y[3], &c->full[s], 0x3);
        tma_gather4(smem + kOffKpe + s * kKpeBytes + lane * 512, map_kpe, 0, y[0], y[1], y[2], y[3],
                    &c->full[s]);
      }
      __syncwarp();
    }
  }
  // drain: the last stages' copies must land before this CTA may exit
  if (lane == 0 && c->abort) {
    for (int q = j - kStages; q < j; ++q)
      if (q >= 0) mbar_wait_drain(&c->full[q % kStages], (uint32_t)(q / kStages) & 1u, kDrainLimitNs);
  }
}

__device__ void score_mma(const Params& p, uint8_t* smem, Ctl* c, int cluster_id, int n_clusters) {
  const uint32_t tS = c->tmem_base;        // columns [0, 128): two S buffers
  const uint32_t tQ = c->tmem_base + 128;  // columns [128, 416): queries, bf16 pairs
  int j = 0, seg = 0;
  for (int64_t item = cluster_id; item < p.n_items; item += n_clusters) {
    const Item it = item_at(p, item);
    if (it.t1 <= it.t0) continue;
    if (!wait(&c->q_ready, (uint32_t)seg & 1u, c, kSiteQReady, j)) return;
    tc_fence_after();
    for (int t = it.t0; t < it.t1; ++t, ++j) {
      const int s = j % kStages, sb = j & 1;
      if (!wait(&c->full[s], (uint32_t)(j / kStages) & 1u, c, kSiteFullS, j)) return;
      if (!wait(&c->s_free[sb], ((uint32_t)(j >> 1) & 1u) ^ 1u, c, kSiteSFree, j)) return;
      tc_fence_after();
      // descriptors differ only in the start-address field: add (offset >> 4)
      const uint64_t dk = smem_desc(smem_u32(smem + kOffKvc + s * kKvcStage), 16, 1024, kLayoutSw128);
      const uint64_t dp = smem_desc(smem_u32(smem + kOffKpe + s * kKpeBytes), 16, 1024, kLayoutSw128);
      const uint32_t ts = tS + sb * kTK;
#pragma unroll
      for (int kc = 0; kc < 9; ++kc) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t bd = (kc < 8 ? dk + (uint64_t)((kc * kChunk + kk * 32) >> 4) : dp + (uint64_t)((kk * 32) >> 4));
          mma_ts(ts, tQ + kc * 32 + kk * 8, bd, kIdescS, (kc | kk) != 0);
        }
      }
      mma_commit(&c->s_full[sb]);
      mma_commit(&c->empty[s]);
    }
    ++seg;
  }
}

__device__ void score_softmax(const Params& p, uint8_t* smem, Ctl* c, int cluster_id, int n_clusters) {
  const int wq = (threadIdx.x >> 5) & 3;            // TMEM lane quadrant of this warp
  const int r = wq * 32 + (threadIdx.x & 31);        // row within the item
  const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
  const uint32_t tS = c->tmem_base + lane_off;
  const uint32_t tQ = c->tmem_base + 128 + lane_off;
  int j = 0, seg = 0;
  for (int64_t item = cluster_id; item < p.n_items; item += n_clusters) {
    const Item it = item_at(p, item);
    if (it.t1 <= it.t0) continue;
    const int b = it.b;
    const int row = it.g * kRG + r;
    const bool live = row < p.rows;
    const int64_t P = p.prefix_lens[b];
    const int64_t N = P + p.Q;
    const uint64_t anc = live ? p.anc[(int64_t)b * p.Q + row / p.H] : 0ull;

    // stage this item's queries into TMEM: column c holds elements 2c, 2c+1
    {
      __syncwarp();
      const uint4* ql = reinterpret_cast<const uint4*>(p.q_lat) + ((int64_t)b * p.rows + row) * (kDl / 8);
      const uint4* qp = reinterpret_cast<const uint4*>(p.q_pe) + ((int64_t)b * p.rows + row) * (kDr / 8);
#pragma unroll 1
      for (int c0 = 0; c0 < 288; c0 += 32) {
        uint32_t w[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const int col = c0 + 4 * v;  // 4 columns per 16-byte vector
          uint4 x = make_uint4(0, 0, 0, 0);
          if (live) x = col < 256 ? ql[col / 4] : qp[(col - 256) / 4];
          w[4 * v + 0] = x.x;
          w[4 * v + 1] = x.y;
          w[4 * v + 2] = x.z;
          w[4 * v + 3] = x.w;
        }
        __syncwarp();
        tmem_st_32x32b_x32(tQ + c0, w);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&c->q_ready);
    }

    // l sums the bf16-rounded weights the value CTA multiplies by, so out is
    // normalised consistently; lx sums the unrounded weights for an exact lse
    float m = -INFINITY, l = 0.f, lx = 0.f;
    for (int t = it.t0; t < it.t1; ++t, ++j) {
      const int sb = j & 1;
      if (!wait(&c->s_full[sb], (uint32_t)(j >> 1) & 1u, c, kSiteSFull, j)) return;
      __syncwarp();  // tcgen05.ld is warp-collective: reconverge after the spin
      tc_fence_after();
      float x[kTK];
      {
        uint32_t u[32];
        tmem_ld_32x32b_x32(tS + sb * kTK, u);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 32; ++q) x[q] = __uint_as_float(u[q]);
        tmem_ld_32x32b_x32(tS + sb * kTK + 32, u);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 32; ++q) x[32 + q] = __uint_as_float(u[q]);
      }
      tc_fence_before();
      mbar_arrive(&c->s_free[sb]);

      // scale to base-2 units and apply the prefix + tree mask
      const int64_t pos0 = (int64_t)t * kTK;
      float tmax = -INFINITY;
      if (pos0 + kTK <= P) {
#pragma unroll
        for (int q = 0; q < kTK; ++q) {
          x[q] *= p.scale_log2;
          tmax = fmaxf(tmax, x[q]);
        }
      } else {
#pragma unroll
        for (int q = 0; q < kTK; ++q) {
          const int64_t pos = pos0 + q;
          const int64_t node = pos - P;
          const bool vis = pos < P || (pos < N && ((anc >> (node & 63)) & 1ull));
          x[q] = vis ? x[q] * p.scale_log2 : -INFINITY;
          tmax = fmaxf(tmax, x[q]);
        }
      }
      // lazy running max: move it only when this tile beats it by > 8 (x 2^8)
      float alpha = 1.f;
      const bool need = tmax > m + 8.f;
      if (need) {
        alpha = exp2f(m - tmax);  // 0 when m is -inf
        l *= alpha;
        lx *= alpha;
        m = tmax;
      }
      const float mu = (m == -INFINITY) ? 0.f : m;

      // wait until the value CTA is done with this P buffer
      if (!wait(&c->p_free[sb], ((uint32_t)(j >> 1) & 1u) ^ 1u, c, kSitePFree, j, true)) return;
      const uint32_t pbase = mapa_shared(smem_u32(smem + kOffP + sb * kPBytes), 1);
#pragma unroll
      for (int q8 = 0; q8 < 8; ++q8) {
        float e[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          e[u] = exp2f(x[8 * q8 + u] - mu);
          lx += e[u];
        }
        const uint32_t w0 = pack_bf16(e[0], e[1]), w1 = pack_bf16(e[2], e[3]);
        const uint32_t w2 = pack_bf16(e[4], e[5]), w3 = pack_bf16(e[6], e[7]);
        // the row sum uses the rounded values the value CTA multiplies by
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w0);
        float2 f0 = __bfloat1622float2(h[0]);
        l += f0.x + f0.y;
        f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w1));
        l += f0.x + f0.y;
        f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w2));
        l += f0.x + f0.y;
        f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w3));
        l += f0.x + f0.y;
        st_cluster_v4(pbase + sw128_offset(r, 8 * q8), w0, w1, w2, w3);
      }
      // every row ships its factor; rows that moved their max also raise the
      // tile's flag (the value CTA clears it when it releases the buffer)
      st_cluster_f32(mapa_shared(smem_u32(&c->alpha[sb][r]), 1), alpha);
      if (need) red_or_cluster(mapa_shared(smem_u32(&c->flag[sb]), 1), 1u);
      fence_proxy_async_cluster();
      mbar_arrive_cluster(&c->p_full[sb], 1);
    }

    // hand the row statistics to the value CTA for the epilogue
    if (!wait(&c->fin_free, ((uint32_t)seg & 1u) ^ 1u, c, kSiteFinFree, j, true)) return;
    st_cluster_f32(mapa_shared(smem_u32(&c->lfin[r]), 1), l);
    st_cluster_f32(mapa_shared(smem_u32(&c->lxfin[r]), 1), lx);
    st_cluster_f32(mapa_shared(smem_u32(&c->mfin[r]), 1), m);
    mbar_arrive_cluster(&c->fin_full, 1);
    ++seg;
  }
}

// ---------------------------------------------------------------------------
// value CTA roles
// ---------------------------------------------------------------------------
__device__ void value_mma(const Params& p, uint8_t* smem, Ctl* c, int cluster_id, int n_clusters) {
  const uint32_t tO = c->tmem_base;
  int j = 0, seg = 0, ncmd = 0;
  bool ok = true;
  for (int64_t item = cluster_id; item < p.n_items && ok; item += n_clusters) {
    const Item it = item_at(p, item);
    if (it.t1 <= it.t0) continue;
    for (int t = it.t0; t < it.t1; ++t, ++j) {
      const int s = j % kStages, pb = j & 1;
      mbar_arrive_expect_tx(&c->full[s], kKvcBytes);
      if (!(ok = wait(&c->full[s], (uint32_t)(j / kStages) & 1u, c, kSiteFullV, j))) break;
      if (!(ok = wait(&c->p_full[pb], (uint32_t)(j >> 1) & 1u, c, kSitePFull, j, true))) break;
      const bool first = (t == it.t0);
      if (!first && c->flag[pb]) {
        // O must hold PV(j-1) in full before it is rescaled
        if (!(ok = wait(&c->pv_done[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u, c, kSitePvPrev, j))) break;
        tc_fence_after();
        c->cmd = kCmdRescale;
        c->cmd_buf = pb;
        mbar_arrive(&c->cmd_full);
        if (!(ok = wait(&c->cmd_done, (uint32_t)ncmd & 1u, c, kSiteCmdDone, j))) break;
        ++ncmd;
      }
      tc_fence_after();
      const uint64_t da = smem_desc(smem_u32(smem + kOffP + pb * kPBytes), 16, 1024, kLayoutSw128);
      const uint64_t dv = smem_desc(smem_u32(smem + kOffKvc + s * kKvcStage), MLA_TC_V_LBO, MLA_TC_V_SBO,
                                    kLayoutSw128);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
        for (int nh = 0; nh < 2; ++nh) {
          mma_ss(tO + nh * 256, da + (uint64_t)((kk * 32) >> 4),
                 dv + (uint64_t)((nh * 4 * kChunk + kk * 16 * 128) >> 4), kIdescPV, !(first && kk == 0));
        }
      }
      mma_commit(&c->pv_done[pb]);
    }
    if (!ok) break;
    // epilogue of this item once its last PV is complete
    if (!(ok = wait(&c->pv_done[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u, c, kSitePvLast, j))) break;
    tc_fence_after();
    c->cmd = kCmdEpilogue;
    c->cmd_item = item;
    mbar_arrive(&c->cmd_full);
    if (!(ok = wait(&c->cmd_done, (uint32_t)ncmd & 1u, c, kSiteCmdDone, j))) break;
    ++ncmd;
    ++seg;
  }
  c->cmd = kCmdExit;
  mbar_arrive(&c->cmd_full);
  if (c->abort) {
    // drain: outstanding MMAs and multicast copies into this CTA
    mma_commit(&c->drain);
    mbar_wait_drain(&c->drain, 0, kDrainLimitNs);
    for (int q = j - kStages + 1; q <= j; ++q)
      if (q >= 0) mbar_wait_drain(&c->full[q % kStages], (uint32_t)(q / kStages) & 1u, kDrainLimitNs);
  }
}

// Releases each tile's stage and P buffer back to the score CTA once the PV
// MMAs that read them have completed.
__device__ void value_release(const Params& p, Ctl* c, int cluster_id, int n_clusters) {
  int j = 0;
  for (int64_t item = cluster_id; item < p.n_items; item += n_clusters) {
    const Item it = item_at(p, item);
    for (int t = it.t0; t < it.t1; ++t, ++j) {
      if (!wait(&c->pv_done[j & 1], (uint32_t)(j >> 1) & 1u, c, kSiteRelease, j)) return;
      c->flag[j & 1] = 0;  // ordered before the release below
      mbar_arrive_cluster(&c->empty[j % kStages], 0);
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
        tmem_ld_32x32b_x32(tO + c0, u);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 32; ++q) u[q] = __float_as_uint(__uint_as_float(u[q]) * a);
        tmem_st_32x32b_x32(tO + c0, u);
      }
      tmem_wait_st();
    } else {  // kCmdEpilogue
      const Item it = item_at(p, c->cmd_item);
      if (!wait(&c->fin_full, (uint32_t)seg & 1u, c, kSiteFinFull, seg, true)) return;
      __syncwarp();
      const float l = c->lfin[r], lx = c->lxfin[r], m = c->mfin[r];
      mbar_arrive_cluster(&c->fin_free, 0);
      ++seg;
      const int row = it.g * kRG + r;
      const bool live = row < p.rows;  // TMEM loads stay warp-wide; only stores are per row
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse = lx > 0.f ? (m + log2f(lx)) * ln2 : -INFINITY;
      const int64_t orow = (int64_t)it.b * p.rows + row;
      if (p.splits == 1) {
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + orow * kDl);
#pragma unroll 1
        for (int c0 = 0; c0 < kDl; c0 += 32) {
          uint32_t u[32];
          __syncwarp();
          tmem_ld_32x32b_x32(tO + c0, u);
          tmem_wait_ld();
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
          tmem_ld_32x32b_x32(tO + c0, u);
          tmem_wait_ld();
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

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const Params p, const __grid_constant__ CUtensorMap map_kvc,
                   const __grid_constant__ CUtensorMap map_kpe) {
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
      mbar_init(&c->full[s], 1);
      mbar_init(&c->empty[s], 2);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(&c->s_full[q], 1);
      mbar_init(&c->s_free[q], kRG);
      mbar_init(&c->p_free[q], 1);
      mbar_init(&c->p_full[q], kRG);
      mbar_init(&c->pv_done[q], 1);
      c->flag[q] = 0;
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
  if (warp == 2) {
    tmem_alloc(&c->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 64 && rank == 0) {
    prefetch_tmap(&map_kvc);
    prefetch_tmap(&map_kpe);
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised before any remote use
  tc_fence_after();

  const int cluster_id = blockIdx.x >> 1;
  const int n_clusters = gridDim.x >> 1;
  if (rank == 0) {
    if (warp == 0) score_producer(p, &map_kvc, &map_kpe, smem, c, cluster_id, n_clusters);
    else if (warp == 1) { if ((threadIdx.x & 31) == 0) score_mma(p, smem, c, cluster_id, n_clusters); }
    else if (warp >= 4) score_softmax(p, smem, c, cluster_id, n_clusters);
  } else {
    if (warp == 1) { if ((threadIdx.x & 31) == 0) value_mma(p, smem, c, cluster_id, n_clusters); }
    else if (warp == 2) { if ((threadIdx.x & 31) == 0) value_release(p, c, cluster_id, n_clusters); }
    else if (warp >= 4) value_epilogue(p, c);
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (rank == 0 && threadIdx.x == 0 && c->abort) {
    // outstanding S MMAs must finish before TMEM is released
    mma_commit(&c->drain);
    mbar_wait_drain(&c->drain, 0, kDrainLimitNs);
  }
  if (threadIdx.x == 0 && c->abort) {
    set_err(p.err, MLA_DEVERR_TIMEOUT);
    atomicCAS(p.err + 1, 0u, (uint32_t)c->abort_site | (rank << 8));
    // let multicast copies issued by the peer before it stopped land here
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < kDrainLimitNs) {
    }
  }
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // no CTA leaves while its peer may still touch its shared memory
  if (warp == 2) tmem_dealloc(c->tmem_base, kTmemCols);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// Rows of a pool tensor as a 2-D map: width columns, 64-column boxes, one row
// per box (the shape tile::gather4 expects), 128-byte swizzle.
bool make_row_map(CUtensorMap* m, const void* base, int64_t width, int64_t stride_elems, int64_t rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)stride_elems * 2};
  cuuint32_t box[2] = {64, 1};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
  CUtensorMap map_kvc, map_kpe;
  if (!tc::make_row_map(&map_kvc, p.kv_c, kDl, p.kv_c_stride, p.pool_slots) ||
      !tc::make_row_map(&map_kpe, p.k_pe, kDr, p.k_pe_stride, p.pool_slots))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(tc::attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       tc::kSmemAlloc);
  if (e != cudaSuccess) return e;
  tc::attn_tc_kernel<<<2 * p.grid, tc::kThreads, tc::kSmemAlloc, stream>>>(p, map_kvc, map_kpe);
  return cudaGetLastError();
}

}  // namespace mlav
