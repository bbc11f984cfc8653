// LSE combine of split-KV pieces (flash-decoding merge).
//
// A row group whose KV range was cut into several chunks has one normalised
// partial output o_s and log-sum-exp lse_s per non-empty chunk.  Exactly:
//   lse = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) * o_s,
// because each piece's softmax over its own tokens, reweighted by its share
// of the total exponent mass, is the softmax over the union.  When a call
// keeps one chunk per row group the attention kernel writes the results
// directly: this kernel is then not launched, or (the split count being chosen
// on the device) returns at once -- unless the plan cut the items of a last,
// partial wave into pieces, whose rows alone it then merges.
#include "common.cuh"

namespace mlav {

constexpr int kCombineThreads = 256;  // 8 warps

// WR warps share an output row, warp c taking columns [c 512/WR, (c+1) 512/WR):
// lane l holds columns c 512/WR + 4 (l + 32 q) .. + 3, q < 4/WR, of every
// piece, so each access of the warp covers 512 contiguous bytes; BATCH pieces
// are in flight at a time.  One warp per row, four pieces deep, when a call has
// few pieces per row (its many rows keep the GPU busy); four warps per row,
// eight pieces deep, when it may have many pieces and few rows.
template <int WR, int BATCH>
struct RowMerge {
  static constexpr int kQ = 4 / WR;     // float4 per lane per piece
  static constexpr int kBatch = BATCH;  // pieces whose rows are loaded together
  static_assert(32 % BATCH == 0, "a batch never straddles 32 pieces");

  // Merges the n pieces of output row `orow`, column block `cb`.  Piece k
  // holds tiles [k T / n, (k+1) T / n) of its row group's range of T tiles
  // (empty ones were skipped by the attention kernel: their slots hold stale
  // bytes and are never read) in partial row prow0 + k pstride.
  __device__ __forceinline__ static void run(const Params& p, int64_t orow, int cb, int n, int64_t prow0,
                                             int64_t pstride, int64_t T) {
    const int lane = threadIdx.x & 31;
    const int col0 = cb * (kDl / WR);
    // which of pieces k0 .. k0 + 31 were computed, one bit each (lane k tests
    // piece k0 + k)
    auto live_mask = [&](int k0) {
      const int64_t k = k0 + lane;
      return __ballot_sync(0xffffffffu, k < n && ((k + 1) * T) / n > (k * T) / n);
    };
    float4 v[kBatch][kQ];
    auto load_batch = [&](int k0, uint32_t lm) {
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if ((lm >> ((k0 + u) & 31)) & 1u) {
          const float4* src = reinterpret_cast<const float4*>(p.part_o + (prow0 + (k0 + u) * pstride) * kDl + col0);
#pragma unroll
          for (int q = 0; q < kQ; ++q) v[u][q] = src[lane + 32 * q];
        }
      }
    };
    // the first pieces' rows are in flight while the largest lse is found
    uint32_t lm = live_mask(0);
    load_batch(0, lm);
    float M = -INFINITY;
    for (int k0 = 0; k0 < n; k0 += 32) {
      const uint32_t m = k0 == 0 ? lm : live_mask(k0);
      if ((m >> lane) & 1u) M = fmaxf(M, p.part_lse[prow0 + (int64_t)(k0 + lane) * pstride]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    // weights exp(lse_k - M) <= 1, summed in piece order; pieces with weight
    // 0 (empty, or an lse of -inf) add nothing
    float L = 0.f;
    float4 acc[kQ];
#pragma unroll
    for (int q = 0; q < kQ; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
#pragma unroll 1
      for (int k0 = 0; k0 < n; k0 += kBatch) {
        if (k0 > 0) {
          if ((k0 & 31) == 0) lm = live_mask(k0);  // batches never straddle 32 pieces
          load_batch(k0, lm);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          if (!((lm >> ((k0 + u) & 31)) & 1u)) continue;
          const float w = __expf(p.part_lse[prow0 + (int64_t)(k0 + u) * pstride] - M);
          if (w == 0.f) continue;
          L += w;
#pragma unroll
          for (int q = 0; q < kQ; ++q) {
            acc[q].x = fmaf(w, v[u][q].x, acc[q].x);
            acc[q].y = fmaf(w, v[u][q].y, acc[q].y);
            acc[q].z = fmaf(w, v[u][q].z, acc[q].z);
            acc[q].w = fmaf(w, v[u][q].w, acc[q].w);
          }
        }
      }
    }
    const float inv = (L > 0.f) ? 1.f / L : 0.f;
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
      const int64_t d = col0 + (int64_t)4 * (lane + 32 * q);
      if (p.dtype == MLA_BF16) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc[q].x * inv, acc[q].y * inv);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc[q].z * inv, acc[q].w * inv);
        uint2 w2;
        w2.x = *reinterpret_cast<uint32_t*>(&lo);
        w2.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) + orow * kDl + d) = w2;
      } else {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + orow * kDl + d) =
            make_float4(acc[q].x * inv, acc[q].y * inv, acc[q].z * inv, acc[q].w * inv);
      }
    }
    if (cb == 0 && lane == 0 && p.lse) p.lse[orow] = (L > 0.f) ? M + logf(L) : -INFINITY;
  }
};

template <int WR, int BATCH>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(Params p) {
  grid_dep_wait();  // the attention kernel's partials and error word
  if (*p.err) return;
  const Split sp = read_split(p);
  // nothing to merge when every row group was one piece (the attention kernel
  // wrote the outputs itself)
  if (sp.S == 1 && sp.P == 1) return;
  // one task (output row, column block) per warp: every row when S > 1, else
  // the rows of the pieced tail items only
  const int64_t gw = (int64_t)blockIdx.x * (kCombineThreads / 32) + (threadIdx.x >> 5);
  const int64_t w = gw / WR;
  const int cb = (int)(gw % WR);
  if (sp.S > 1) {
    // S chunks; chunk k of row group g of sequence b is item slot (b S + k) G + g
    if (w >= (int64_t)p.B * p.rows) return;
    const int b = (int)(w / p.rows);
    const int row = (int)(w % p.rows);
    const int g = row / p.rg;
    const int r = row - g * p.rg;
    const int S = sp.S;
    RowMerge<WR, BATCH>::run(p, w, cb, S, ((int64_t)b * S * p.groups + g) * p.rg + r, (int64_t)p.groups * p.rg,
                             p.seq_tiles[b]);
  } else {
    // P pieces of item tail + j in slots j P .. j P + P - 1 (S = 1: item
    // b G + g covers all of sequence b's tiles)
    const int64_t j = w / p.rg;
    const int r = (int)(w % p.rg);
    if (j >= sp.n_items - sp.tail) return;
    const int64_t item = sp.tail + j;
    const int g = (int)(item % p.groups);
    const int b = (int)(item / p.groups);
    const int row = g * p.rg + r;
    if (row >= p.rows) return;
    const int P = sp.P;
    RowMerge<WR, BATCH>::run(p, (int64_t)b * p.rows + row, cb, P, j * P * p.rg + r, p.rg, p.seq_tiles[b]);
  }
}

cudaError_t launch_combine(const Params& p, cudaStream_t stream, bool pdl) {
  // rows to cover: every row (S > 1) or the rows of at most one item per
  // cluster (pieced tail); warps past the chosen plan's tasks return at once
  int64_t rows = (int64_t)p.B * p.rows;
  if (p.auto_plan && (int64_t)p.grid * p.rg > rows) rows = (int64_t)p.grid * p.rg;
  // four warps per row only when a call can have many chunks per row
  const bool wide = p.splits > 16;
  const int64_t warps = rows * (wide ? 4 : 1);
  const int64_t blocks = (warps + (kCombineThreads / 32) - 1) / (kCombineThreads / 32);
  if (blocks == 0) return cudaSuccess;
  if (wide) return launch_kernel(combine_kernel<4, 8>, dim3((unsigned)blocks), dim3(kCombineThreads), 0, stream, pdl, p);
  return launch_kernel(combine_kernel<1, 4>, dim3((unsigned)blocks), dim3(kCombineThreads), 0, stream, pdl, p);
}

}  // namespace mlav
