// LSE combine of split-KV pieces (flash-decoding merge).
//
// A row group whose KV range was cut into several chunks has one normalised
// partial output o_s and log-sum-exp lse_s per non-empty chunk.  Exactly:
//   lse = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) * o_s,
// because each piece's softmax over its own tokens, reweighted by its share
// of the total exponent mass, is the softmax over the union.  When a call
// keeps one chunk per row group the attention kernel writes the results
// directly: this kernel is then not launched, or (the split count being chosen
// on the device) returns at once.
#include "common.cuh"

namespace mlav {

constexpr int kCombineThreads = 256;  // 8 warps; one warp per output row
constexpr int kPieceBatch = 4;        // pieces whose partial rows are loaded together

// Merges the n pieces of output row `orow` (lane l holds columns
// 4 (l + 32 q) .. + 3, q = 0..3, so every access of the warp covers 512
// contiguous bytes).  prow(k): partial row of piece k; live(k): piece k was
// computed (an empty piece's slot holds stale bytes and is never read).
template <class PRow, class Live>
__device__ __forceinline__ void merge_row(const Params& p, int64_t orow, int n, PRow prow, Live live) {
  const int lane = threadIdx.x & 31;
  float4 v[kPieceBatch][4];
  auto load_batch = [&](int k0) {
#pragma unroll
    for (int u = 0; u < kPieceBatch; ++u) {
      if (k0 + u < n && live(k0 + u)) {
        const float4* src = reinterpret_cast<const float4*>(p.part_o + prow(k0 + u) * kDl);
#pragma unroll
        for (int q = 0; q < 4; ++q) v[u][q] = src[lane + 32 * q];
      }
    }
  };
  // the first pieces' rows are in flight while the largest lse is found
  load_batch(0);
  float M = -INFINITY;
  for (int k = lane; k < n; k += 32)
    if (live(k)) M = fmaxf(M, p.part_lse[prow(k)]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  // weights exp(lse_k - M) <= 1, summed in piece order; pieces with weight 0
  // (empty, or an lse of -inf) add nothing
  float L = 0.f;
  float4 acc[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    for (int k0 = 0; k0 < n; k0 += kPieceBatch) {
      if (k0 > 0) load_batch(k0);
#pragma unroll
      for (int u = 0; u < kPieceBatch; ++u) {
        if (k0 + u >= n || !live(k0 + u)) continue;
        const float w = __expf(p.part_lse[prow(k0 + u)] - M);
        if (w == 0.f) continue;
        L += w;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
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
  for (int q = 0; q < 4; ++q) {
    const int64_t d = (int64_t)4 * (lane + 32 * q);
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
  if (lane == 0 && p.lse) p.lse[orow] = (L > 0.f) ? M + logf(L) : -INFINITY;
}

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(Params p) {
  grid_dep_wait();  // the attention kernel's partials and error word
  if (*p.err) return;
  const Split sp = read_split(p);
  // nothing to merge when every row group was one piece (the attention kernel
  // wrote the outputs itself)
  if (sp.S == 1 && sp.P == 1) return;
  const int64_t w = (int64_t)blockIdx.x * (kCombineThreads / 32) + (threadIdx.x >> 5);
  if (sp.S > 1) {
    // every row: S chunks, chunk k of row group g of sequence b in item slot
    // (b S + k) G + g
    if (w >= (int64_t)p.B * p.rows) return;
    const int b = (int)(w / p.rows);
    const int row = (int)(w % p.rows);
    const int g = row / p.rg;
    const int r = row - g * p.rg;
    const int64_t T = p.seq_tiles[b];
    const int S = sp.S;
    merge_row(
        p, w, S, [&](int k) { return (((int64_t)b * S + k) * p.groups + g) * p.rg + r; },
        [&](int k) { return ((int64_t)(k + 1) * T) / S > ((int64_t)k * T) / S; });
  } else {
    // the rows of the tail items only: P pieces of item tail + j in slots
    // j P .. j P + P - 1 (S = 1: item = b G + g covers all of sequence b's tiles)
    const int64_t j = w / p.rg;
    const int r = (int)(w % p.rg);
    if (j >= sp.n_items - sp.tail) return;
    const int64_t item = sp.tail + j;
    const int g = (int)(item % p.groups);
    const int b = (int)(item / p.groups);
    const int row = g * p.rg + r;
    if (row >= p.rows) return;
    const int64_t T = p.seq_tiles[b];
    const int P = sp.P;
    merge_row(
        p, (int64_t)b * p.rows + row, P, [&](int k) { return (j * P + k) * p.rg + r; },
        [&](int k) { return ((int64_t)(k + 1) * T) / P > ((int64_t)k * T) / P; });
  }
}

cudaError_t launch_combine(const Params& p, cudaStream_t stream, bool pdl) {
  // every row (S > 1), or the rows of at most one item per cluster (tail pieces)
  int64_t warps = (int64_t)p.B * p.rows;
  if ((int64_t)p.grid * p.rg > warps) warps = (int64_t)p.grid * p.rg;
  const int64_t blocks = (warps + (kCombineThreads / 32) - 1) / (kCombineThreads / 32);
  if (blocks == 0) return cudaSuccess;
  return launch_kernel(combine_kernel, dim3((unsigned)blocks), dim3(kCombineThreads), 0, stream, pdl, p);
}

}  // namespace mlav
