// Metadata kernels: ancestor-or-self masks of every draft tree, per-sequence
// tile counts (which the work items of the attention kernels cut into
// chunks), and validation of every device-resident table entry.
//
// The mask rule follows "Reading the Reference: How a Single File-Read Message
// Anchored a Complex CUDA Kernel Implementation", section "Output Knowledge
// Created by This Message" (prefix visibility + tree-tail visibility) and
// "Ground Truth in Silicon ...", section "Input Knowledge Required ...",
// item 3: node i sees tree node t when t is i or an ancestor of i.  One thread
// per (sequence, node) walks the node's parent links and sets a bit for each
// ancestor; parents precede their nodes, so the walk takes at most i steps, and
// a link that breaks that rule ends the walk (its own node reports it).
#include "common.cuh"

namespace mlav {

constexpr int kMetaThreads = 1024;
static_assert(kMetaThreads / 32 == 32, "the block scan combines 32 warp totals in one warp");

// Block-wide inclusive scan of one value per thread (kMetaThreads threads):
// a shuffle scan inside each warp, then one warp scans the 32 warp totals --
// two block barriers instead of one pair per doubling step.  sh holds at
// least kMetaThreads / 32 entries.
__device__ int64_t block_inclusive_scan(int64_t v, int64_t* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  if (lane == 31) sh[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int64_t t = sh[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t u = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += u;
    }
    sh[lane] = t;  // inclusive prefix over the warps
  }
  __syncthreads();
  const int64_t r = v + (warp > 0 ? sh[warp - 1] : 0);
  __syncthreads();  // sh may be reused by the caller's next round
  return r;
}

// Split plan of the tensor-core kernel when the caller leaves the split count
// to the library.  The host sizes the workspace for S_max = p.splits chunks per
// row group (the count that fills the clusters in whole waves, from B, H and Q
// alone) and for at least one partial slot per cluster; once the tile counts
// T_b are known, every S in [1, S_max] is scored by the time it would take and
// the cheapest is used (the smaller S on a tie).  The persistent clusters take
// work units round-robin (unit u runs on cluster u mod grid), so the attention
// time is the most loaded cluster's sum over its non-empty units of (fixed
// cost + tiles); S > 1 adds the combine kernel's pass over the fp32 partials.
// For S = 1 a second form is scored too: when the items fill W >= 1 whole
// waves and r more items remain, each of those r items runs as
// P = grid / r >= 2 pieces of its tile range (one unit per idle cluster), and
// the combine merges just those rows.  The constants are GB300 measurements of
// this library's kernels: ~1 us per 64-token tile per cluster, ~14 tiles'
// worth of fixed cost per unit (query staging, pipeline fill and drain, the
// epilogue), and a combine moving ~3 TB/s plus ~3 us of launch and tail.
// Integer arithmetic throughout, so the same lengths always give the same
// plan.  One warp scores one candidate at a time; its lanes add unit costs
// into the warp's per-cluster totals in shared memory.
constexpr int kPlanMaxClusters = 64;
constexpr int kPlanMaxSplits = 64;
constexpr int kPlanSharedSeqs = 2048;  // the plan is made for batches whose tile counts fit shared memory
constexpr uint32_t kPlanUnitTiles = 14;
constexpr int64_t kPlanTileNs = 1000;
constexpr int64_t kPlanCombineBytesPerNs = 3000;
constexpr int64_t kPlanCombineFixedNs = 3000;

// Tiles of chunk k when T tiles are cut into n chunks: floor((k+1) T / n) -
// floor(k T / n), in 32-bit arithmetic (T = q n + rem, rem < n <= 4096).
__device__ __forceinline__ uint32_t plan_chunk_tiles(uint32_t T, uint32_t n, uint32_t k) {
  const uint32_t q = T / n, rem = T - q * n;
  return q + ((k + 1) * rem) / n - (k * rem) / n;
}

// The warp's largest per-cluster total, in ns.  Totals are 32-bit tile counts:
// one that wrapped could only make the plan slower, never wrong, since every
// plan computes the same attention.
__device__ __forceinline__ int64_t plan_makespan_ns(const uint32_t* ld, int C) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  uint32_t mx = 0u;
  for (int c = lane; c < C; c += 32) mx = max(mx, ld[c]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  return (int64_t)mx * kPlanTileNs;
}

// cost[S - 1] and pieces[S - 1] (1: no split tail) for S in [1, S_max];
// tiles_sh holds every T_b (B <= kPlanSharedSeqs).  Item counts are below
// 2^26 (the host refuses larger plans), so unit indices fit 32 bits.
__device__ void plan_scores(const Params& p, const int32_t* tiles_sh, uint32_t* load, int64_t* cost, int* pieces) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  auto tiles = [&](int b) -> uint32_t { return (uint32_t)tiles_sh[b]; };
  const int C = p.grid, G = p.groups;
  uint32_t* ld = load + warp * kPlanMaxClusters;
  const int64_t rows_bytes = (int64_t)p.rows * (kDl * 4);  // fp32 partial bytes of one sequence's rows
  for (int S = warp + 1; S <= p.splits; S += kMetaThreads / 32) {
    for (int c = lane; c < C; c += 32) ld[c] = 0u;
    __syncwarp();
    const int n = p.B * G * S;
    // chunk bk = b S + k: its G items are units bk G .. bk G + G - 1, dealt
    // to consecutive clusters from (bk G) mod C
    for (int bk = lane; bk < p.B * S; bk += 32) {
      const int b = bk / S;
      const uint32_t t = plan_chunk_tiles(tiles(b), (uint32_t)S, (uint32_t)(bk - b * S));
      if (t == 0) continue;
      int c = (int)(((int64_t)bk * G) % C);
      for (int g = 0; g < G; ++g) {
        atomicAdd(&ld[c], kPlanUnitTiles + t);
        if (++c == C) c = 0;
      }
    }
    int64_t best = plan_makespan_ns(ld, C);
    if (S > 1) best += (int64_t)p.B * S * rows_bytes / kPlanCombineBytesPerNs + kPlanCombineFixedNs;
    int best_p = 1;
    const int full = (n / C) * C, r = n - full;
    if (S == 1 && full > 0 && r > 0 && C / r >= 2) {
      // the same items, the last r cut into P pieces each
      const int P = C / r;
      __syncwarp();
      for (int c = lane; c < C; c += 32) ld[c] = 0u;
      __syncwarp();
      for (int b = lane; b * G < full; b += 32) {
        const uint32_t T = tiles(b);
        if (T == 0) continue;
        int c = (int)(((int64_t)b * G) % C);
        for (int g = 0; g < G && b * G + g < full; ++g) {
          atomicAdd(&ld[c], kPlanUnitTiles + T);
          if (++c == C) c = 0;
        }
      }
      for (int v = lane; v < r * P; v += 32) {
        const uint32_t t = plan_chunk_tiles(tiles((full + v / P) / G), (uint32_t)P, (uint32_t)(v % P));
        if (t > 0) atomicAdd(&ld[v], kPlanUnitTiles + t);
      }
      const int64_t ns = plan_makespan_ns(ld, C) +
                         (int64_t)r * P * p.rg * (kDl * 4) / kPlanCombineBytesPerNs + kPlanCombineFixedNs;
      if (ns < best) {
        best = ns;
        best_p = P;
      }
    }
    if (lane == 0) {
      cost[S - 1] = best;
      pieces[S - 1] = best_p;
    }
    __syncwarp();
  }
}

// One block.  Clears the error word, validates prefix_lens / kv_indptr /
// page capacity, computes T_b = ceil(N_b / tk) and the prefix sums
// seq_kv_base of N_b (a thread per sequence), fixes the call's split count,
// then validates the parents and builds anc (a thread per node).
__global__ void __launch_bounds__(kMetaThreads) meta_seq_kernel(Params p) {
  __shared__ int64_t sh[kMetaThreads / 32];
  __shared__ int64_t carry_kv;
  __shared__ uint32_t plan_load[(kMetaThreads / 32) * kPlanMaxClusters];
  __shared__ int64_t plan_cost[kPlanMaxSplits];
  __shared__ int plan_pieces[kPlanMaxSplits];
  __shared__ int32_t tiles_sh[kPlanSharedSeqs];
  const int tid = threadIdx.x;
  grid_dep_launch();  // the slot pass may start launching; it waits for this kernel
  if (tid == 0) {
    p.err[0] = 0u;
    p.err[1] = 0u;  // where a bounded wait gave up, if one did
    carry_kv = 0;
    p.seq_kv_base[0] = 0;
  }
  __syncthreads();

  for (int b0 = 0; b0 < p.B; b0 += kMetaThreads) {
    const int b = b0 + tid;
    int64_t nkv = 0;
    if (b < p.B) {
      int64_t P = p.prefix_lens[b];
      uint32_t e = 0;
      if (P < 0) { e |= MLA_DEVERR_PREFIX; P = 0; }
      const int64_t N = P + p.Q;
      if (p.page_size == 1) {
        const int64_t lo = p.kv_indptr[b], hi = p.kv_indptr[b + 1];
        // with kv_indptr[0] == 0 and every span equal to N_b, all reads stay in
        // kv_indices[0 .. kv_indptr[B])
        if ((b == 0 && lo != 0) || lo < 0 || hi - lo != N) e |= MLA_DEVERR_INDPTR;
      } else if (N > (int64_t)p.max_pages * p.page_size) {
        e |= MLA_DEVERR_PAGES;
      }
      if (e) set_err(p.err, e);
      const int64_t T = (N + p.tk - 1) / p.tk;
      p.seq_tiles[b] = (int32_t)T;
      if (b < kPlanSharedSeqs) tiles_sh[b] = (int32_t)T;
      nkv = N;
    }
    const int64_t k_inc = block_inclusive_scan(nkv, sh);
    if (b < p.B) {
      p.seq_kv_base[b + 1] = carry_kv + k_inc;
    }
    __syncthreads();
    if (tid == kMetaThreads - 1) {
      carry_kv += k_inc;
    }
    __syncthreads();
  }

  // the work split of this call (the tile counts above are visible to the
  // whole block after the loop's last barrier): S, the grid assumed, the first
  // item of a tail cut into pieces, pieces per tail item
  // (a batch of more than kPlanSharedSeqs sequences has far more row groups
  // than clusters, where the wave-filling S_max is the plan)
  if (p.auto_plan && p.B <= kPlanSharedSeqs && p.splits >= 1 && p.splits <= kPlanMaxSplits && p.grid >= 1 &&
      p.grid <= kPlanMaxClusters && p.part_slots >= p.grid) {
    plan_scores(p, tiles_sh, plan_load, plan_cost, plan_pieces);
    __syncthreads();
    if (tid < 32) {
      // the cheapest S (the smaller on a tie): lane l looks at S = l + 1, l + 33
      int64_t bc = INT64_MAX;
      int bs = 0;
      for (int S = tid + 1; S <= p.splits; S += 32)
        if (plan_cost[S - 1] < bc) {
          bc = plan_cost[S - 1];
          bs = S;
        }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const int64_t oc = __shfl_xor_sync(0xffffffffu, bc, o);
        const int os = __shfl_xor_sync(0xffffffffu, bs, o);
        if (oc < bc || (oc == bc && os < bs)) {
          bc = oc;
          bs = os;
        }
      }
      if (tid == 0) {
        const int best = bs;
        const int64_t n = (int64_t)p.B * p.groups * best;
        const int P = plan_pieces[best - 1];
        p.plan[0] = best;
        p.plan[1] = p.grid;
        p.plan[2] = (int32_t)(P > 1 ? (n / p.grid) * p.grid : n);
        p.plan[3] = P;
      }
    }
  } else if (tid == 0) {
    p.plan[0] = p.splits;
    p.plan[1] = p.grid;
    p.plan[2] = (int32_t)p.n_items;
    p.plan[3] = 1;
  }

  // ancestor-or-self masks
  const int64_t nodes = (int64_t)p.B * p.Q;
  uint32_t e = 0;
  for (int64_t k = tid; k < nodes; k += kMetaThreads) {
    const int i = (int)(k % p.Q);
    const int32_t* par = p.tree_parent + (k - i);
    int j = par[i];
    if (j < -1 || j >= i) e |= MLA_DEVERR_PARENT;
    uint64_t m = 1ull << i;
    int cur = i;
    while (j >= 0 && j < cur) {
      m |= 1ull << j;
      cur = j;
      j = par[j];
    }
    p.anc[k] = m;
  }
  if (e) set_err(p.err, e);
}

// Grid-stride pass over every (sequence, position): checks that each resolved
// slot lies in the pool and, when slots_out is given, records it.  Skips all
// table reads if the sequence-level checks already failed (an inconsistent
// indptr would make the index arithmetic itself unsafe).
__global__ void meta_slots_kernel(Params p, int32_t* slots_out, int64_t capacity) {
  grid_dep_wait();    // reads the sequence metadata and error word of meta_seq_kernel
  grid_dep_launch();  // the attention kernel may start its prologue meanwhile
  if (*p.err & (MLA_DEVERR_PREFIX | MLA_DEVERR_INDPTR | MLA_DEVERR_PAGES)) return;
  const int64_t total = p.seq_kv_base[p.B];
  uint32_t e = 0;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < total;
       k += (int64_t)gridDim.x * blockDim.x) {
    const int b = seq_of(p.seq_kv_base, p.B, k);
    const int64_t pos = k - p.seq_kv_base[b];
    int64_t s;
    if (p.page_size == 1) {
      s = p.kv_indices[(int64_t)p.kv_indptr[b] + pos];
    } else {
      s = (int64_t)p.block_table[(int64_t)b * p.max_pages + pos / p.page_size] * p.page_size +
          pos % p.page_size;
    }
    if (s < 0 || s >= p.pool_slots) e |= MLA_DEVERR_SLOT;
    if (slots_out) {
      if (k < capacity) slots_out[k] = (int32_t)s;
      else e |= MLA_DEVERR_CAPACITY;
    }
  }
  if (e) set_err(p.err, e);
}

__global__ void copy_anc_kernel(Params p, uint64_t* anc_out) {
  const int64_t n = (int64_t)p.B * p.Q;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n;
       k += (int64_t)gridDim.x * blockDim.x)
    anc_out[k] = p.anc[k];
}

cudaError_t launch_meta(const Params& p, int sm_count, int32_t* slots_out, int64_t capacity,
                        uint64_t* anc_out, cudaStream_t stream) {
  meta_seq_kernel<<<1, kMetaThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_kernel(meta_slots_kernel, dim3(2 * sm_count), dim3(256), 0, stream, true, p, slots_out, capacity);
  if (e != cudaSuccess) return e;
  if (anc_out) {
    copy_anc_kernel<<<64, 256, 0, stream>>>(p, anc_out);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace mlav
