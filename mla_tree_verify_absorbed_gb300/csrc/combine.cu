// LSE combine of split-KV pieces (flash-decoding merge).
//
// A row group whose KV range was cut into several chunks has one normalised
// partial output o_s and log-sum-exp lse_s per non-empty chunk.  Exactly:
//   lse = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) * o_s,
// because each piece's softmax over its own tokens, reweighted by its share
// of the total exponent mass, is the softmax over the union.  With one chunk
// per row group the attention kernel wrote the results directly and this
// kernel is not launched.
#include "common.cuh"

namespace mlav {

constexpr int kCombineThreads = 256;  // 8 warps; one warp per (row, quarter of the 512 columns)
constexpr int kQuarters = 4;          // 128 columns per warp: one float4 per lane

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(Params p) {
  grid_dep_wait();  // the attention kernel's partials and error word
  if (*p.err) return;
  const int lane = threadIdx.x & 31;
  const int64_t gw = (int64_t)blockIdx.x * (kCombineThreads / 32) + (threadIdx.x >> 5);
  const int64_t total_rows = (int64_t)p.B * p.rows;
  if (gw >= total_rows * kQuarters) return;
  const int64_t grow = gw / kQuarters;
  const int quarter = (int)(gw % kQuarters);
  const int b = (int)(grow / p.rows);
  const int row = (int)(grow % p.rows);
  const int g = row / p.rg;
  const int64_t T = p.seq_tiles[b];
  const int S = p.splits;
  const int r = row - g * p.rg;
  auto item_of = [&](int k) { return ((int64_t)b * S + k) * p.groups + g; };
  auto nonempty = [&](int k) { return ((int64_t)(k + 1) * T) / S > ((int64_t)k * T) / S; };
  // pass 1: the lanes read the pieces' lse in parallel; warp max
  float M = -INFINITY;
  for (int k = lane; k < S; k += 32)
    if (nonempty(k)) M = fmaxf(M, p.part_lse[item_of(k) * p.rg + r]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  // pass 2: weights exp(lse_k - M) (lane k % 32 holds piece k's), warp sum, and
  // the weighted sum of the pieces' outputs in piece order.  The loads of
  // kBatch pieces are issued before any is used; a piece with weight 0 (empty,
  // or beyond S) loads from piece k0, which is always allocated, and its value
  // is never used, so nothing it holds reaches the sum.
  constexpr int kBatch = 8;
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    for (int k0 = 0; k0 < S; k0 += 32) {
      const int k = k0 + lane;
      const float wk = (k < S && nonempty(k)) ? __expf(p.part_lse[item_of(k) * p.rg + r] - M) : 0.f;
      float wsum = wk;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
      L += wsum;
      const int n = S - k0 < 32 ? S - k0 : 32;
      for (int q0 = 0; q0 < n; q0 += kBatch) {
        float w[kBatch];
        float4 v[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          w[u] = __shfl_sync(0xffffffffu, wk, (q0 + u) & 31);
          if (q0 + u >= n) w[u] = 0.f;
          const int kk = w[u] != 0.f ? k0 + q0 + u : k0;
          v[u] = reinterpret_cast<const float4*>(p.part_o + (item_of(kk) * p.rg + r) * kDl)[quarter * 32 + lane];
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          if (w[u] != 0.f) {
            acc.x = fmaf(w[u], v[u].x, acc.x);
            acc.y = fmaf(w[u], v[u].y, acc.y);
            acc.z = fmaf(w[u], v[u].z, acc.z);
            acc.w = fmaf(w[u], v[u].w, acc.w);
          }
        }
      }
    }
  }
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
  const int64_t orow = (int64_t)b * p.rows + row;
  const int64_t d = (int64_t)4 * (quarter * 32 + lane);
  if (p.dtype == MLA_BF16) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    uint2 w2;
    w2.x = *reinterpret_cast<uint32_t*>(&lo);
    w2.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) + orow * kDl + d) = w2;
  } else {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + orow * kDl + d) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  }
  if (quarter == 0 && lane == 0 && p.lse) p.lse[orow] = (L > 0.f) ? M + logf(L) : -INFINITY;
}

cudaError_t launch_combine(const Params& p, cudaStream_t stream, bool pdl) {
  const int64_t warps = (int64_t)p.B * p.rows * kQuarters;
  const int64_t blocks = (warps + (kCombineThreads / 32) - 1) / (kCombineThreads / 32);
  if (blocks == 0) return cudaSuccess;
  return launch_kernel(combine_kernel, dim3((unsigned)blocks), dim3(kCombineThreads), 0, stream, pdl, p);
}

}  // namespace mlav
