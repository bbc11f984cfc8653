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

constexpr int kCombineThreads = 256;  // one warp per row

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(Params p) {
  if (*p.err) return;
  const int lane = threadIdx.x & 31;
  const int64_t gw = (int64_t)blockIdx.x * (kCombineThreads / 32) + (threadIdx.x >> 5);
  const int64_t total_rows = (int64_t)p.B * p.rows;
  if (gw >= total_rows) return;
  const int b = (int)(gw / p.rows);
  const int row = (int)(gw % p.rows);
  const int g = row / p.rg;
  const int64_t T = p.seq_tiles[b];
  const int S = p.splits;
  const int r = row - g * p.rg;
  auto item_of = [&](int k) { return ((int64_t)b * S + k) * p.groups + g; };
  auto nonempty = [&](int k) { return ((int64_t)(k + 1) * T) / S > ((int64_t)k * T) / S; };
  float M = -INFINITY;
  for (int k = 0; k < S; ++k)
    if (nonempty(k)) M = fmaxf(M, p.part_lse[item_of(k) * p.rg + r]);
  float L = 0.f;
  float4 acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    for (int k = 0; k < S; ++k) {
      if (!nonempty(k)) continue;
      const int64_t prow = item_of(k) * p.rg + r;
      const float w = __expf(p.part_lse[prow] - M);
      L += w;
      const float4* o = reinterpret_cast<const float4*>(p.part_o + prow * kDl);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 v = o[lane + 32 * q];
        acc[q].x = fmaf(w, v.x, acc[q].x);
        acc[q].y = fmaf(w, v.y, acc[q].y);
        acc[q].z = fmaf(w, v.z, acc[q].z);
        acc[q].w = fmaf(w, v.w, acc[q].w);
      }
    }
  }
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
  const int64_t orow = (int64_t)b * p.rows + row;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int64_t d = 4 * (lane + 32 * k);
    store_out(p.out, p.dtype, orow * kDl + d + 0, acc[k].x * inv);
    store_out(p.out, p.dtype, orow * kDl + d + 1, acc[k].y * inv);
    store_out(p.out, p.dtype, orow * kDl + d + 2, acc[k].z * inv);
    store_out(p.out, p.dtype, orow * kDl + d + 3, acc[k].w * inv);
  }
  if (lane == 0 && p.lse) p.lse[orow] = (L > 0.f) ? M + logf(L) : -INFINITY;
}

cudaError_t launch_combine(const Params& p, cudaStream_t stream) {
  const int64_t total_rows = (int64_t)p.B * p.rows;
  const int64_t blocks = (total_rows + (kCombineThreads / 32) - 1) / (kCombineThreads / 32);
  if (blocks == 0) return cudaSuccess;
  combine_kernel<<<(unsigned)blocks, kCombineThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mlav
