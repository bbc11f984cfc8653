// CUDA-core split-KV verify attention (fp32 products, fp32 accumulation).
//
// It is the kernel for the fp32 cache (a 1e-4 relative tolerance needs fp32
// products, which the bf16 tensor-core path cannot give) and an explicit
// alternative for bf16.  Structure: CTAs take work items (sequence, KV chunk,
// row group) round-robin; for each item a CTA keeps the
// group's 16 absorbed query rows in shared memory, stages 32-token KV tiles
// (kv_c and k_pe of each token, gathered through the slot table) once, and
// reuses each staged tile for every row of the group -- the head-tile reuse
// idea of "The Critical Glue: Validating a Custom Flash Attention Kernel
// Through Test Infrastructure", section "What Came Before", widened from 8
// heads to every (node, head) row.  Softmax is online in base 2 with a
// running max and sum per row ("Reading the Reference ...", section "Why This
// File Matters": streaming online softmax, prefix and tree tail masked in one
// pass).
#include "common.cuh"

namespace mlav {

constexpr int kSimtRG = 16;          // rows per row group
constexpr int kSimtTK = 32;          // tokens per KV tile (one per lane)
constexpr int kSimtThreads = 256;    // 8 warps x 2 rows
constexpr int kSimtKvStride = kDk + 1;  // padded smem row: lanes read different rows conflict-free
constexpr int kSimtSmem = (kSimtRG * kDk + kSimtTK * kSimtKvStride) * 4 + kSimtTK * 8;

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__global__ void __launch_bounds__(kSimtThreads, 2) attn_simt_kernel(Params p) {
  if (*p.err) return;  // bad tables: do nothing, the host reports the error
  extern __shared__ float4 smem_f4[];
  float* q_s = reinterpret_cast<float*>(smem_f4);          // [16][576]
  float* kv_s = q_s + kSimtRG * kDk;                        // [32][577]
  int64_t* slot_s = reinterpret_cast<int64_t*>(kv_s + kSimtTK * kSimtKvStride);  // [32]

  const T* q_lat = reinterpret_cast<const T*>(p.q_lat);
  const T* q_pe = reinterpret_cast<const T*>(p.q_pe);
  const T* kv_c = reinterpret_cast<const T*>(p.kv_c);
  const T* k_pe = reinterpret_cast<const T*>(p.k_pe);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t item = blockIdx.x; item < p.n_items; item += gridDim.x) {
    const Item sg = item_at(p, p.splits, item);
    if (sg.t1 <= sg.t0) continue;  // empty chunk (sequence shorter than the split count)
    const int b = sg.b;
    const int64_t P = p.prefix_lens[b];
    const int64_t N = P + p.Q;
    const int row0 = sg.g * kSimtRG;

    // stage the group's query rows (zeros past the last row)
    __syncthreads();
    for (int k = threadIdx.x; k < kSimtRG * kDk; k += kSimtThreads) {
      const int r = k / kDk, d = k % kDk;
      const int row = row0 + r;
      float v = 0.f;
      if (row < p.rows) {
        const int64_t qrow = (int64_t)b * p.rows + row;
        v = d < kDl ? to_f(q_lat[qrow * kDl + d]) : to_f(q_pe[qrow * kDr + (d - kDl)]);
      }
      q_s[k] = v;
    }

    // per-warp rows and their tree masks
    const int rA = row0 + 2 * warp, rB = rA + 1;
    const uint64_t ancA = (rA < p.rows) ? p.anc[(int64_t)b * p.Q + rA / p.H] : 0ull;
    const uint64_t ancB = (rB < p.rows) ? p.anc[(int64_t)b * p.Q + rB / p.H] : 0ull;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
    float oA[16], oB[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) { oA[k] = 0.f; oB[k] = 0.f; }

    for (int t = sg.t0; t < sg.t1; ++t) {
      const int64_t pos0 = (int64_t)t * kSimtTK;
      __syncthreads();  // previous tile fully consumed (and q_s written)
      if (threadIdx.x < kSimtTK) {
        const int64_t pos = pos0 + threadIdx.x;
        slot_s[threadIdx.x] = (pos < N) ? resolve_slot(p, b, pos) : -1;
      }
      __syncthreads();
      for (int k = threadIdx.x; k < kSimtTK * kDk; k += kSimtThreads) {
        const int j = k / kDk, d = k % kDk;
        const int64_t s = slot_s[j];
        float v = 0.f;
        if (s >= 0) v = d < kDl ? to_f(kv_c[s * p.kv_c_stride + d]) : to_f(k_pe[s * p.k_pe_stride + (d - kDl)]);
        kv_s[j * kSimtKvStride + d] = v;
      }
      __syncthreads();

      // scores: lane = token
      const float* kr = kv_s + lane * kSimtKvStride;
      const float* qa = q_s + (2 * warp) * kDk;
      const float* qb = qa + kDk;
      float sA = 0.f, sB = 0.f;
#pragma unroll 8
      for (int d = 0; d < kDk; ++d) {
        const float kv = kr[d];
        sA = fmaf(qa[d], kv, sA);
        sB = fmaf(qb[d], kv, sB);
      }
      const int64_t pos = pos0 + lane;
      bool visA = false, visB = false;
      if (pos < N) {
        if (pos < P) { visA = true; visB = true; }
        else {
          const int node = (int)(pos - P);
          visA = (ancA >> node) & 1ull;
          visB = (ancB >> node) & 1ull;
        }
      }
      sA = visA ? sA * p.scale_log2 : -INFINITY;
      sB = visB ? sB * p.scale_log2 : -INFINITY;

      // online softmax (base 2)
      float tA = sA, tB = sB;
#pragma unroll
      for (int off = 16; off; off >>= 1) {
        tA = fmaxf(tA, __shfl_xor_sync(0xffffffffu, tA, off));
        tB = fmaxf(tB, __shfl_xor_sync(0xffffffffu, tB, off));
      }
      const float mA2 = fmaxf(mA, tA), mB2 = fmaxf(mB, tB);
      const float baseA = (mA2 == -INFINITY) ? 0.f : mA2;
      const float baseB = (mB2 == -INFINITY) ? 0.f : mB2;
      const float aA = exp2f(mA - baseA), aB = exp2f(mB - baseB);
      const float pA = exp2f(sA - baseA), pB = exp2f(sB - baseB);
      float sumA = pA, sumB = pB;
#pragma unroll
      for (int off = 16; off; off >>= 1) {
        sumA += __shfl_xor_sync(0xffffffffu, sumA, off);
        sumB += __shfl_xor_sync(0xffffffffu, sumB, off);
      }
      lA = lA * aA + sumA;
      lB = lB * aB + sumB;
      mA = mA2;
      mB = mB2;
#pragma unroll
      for (int k = 0; k < 16; ++k) { oA[k] *= aA; oB[k] *= aB; }
      // values: lane owns d = lane + 32k
#pragma unroll 4
      for (int j = 0; j < kSimtTK; ++j) {
        const float wA = __shfl_sync(0xffffffffu, pA, j);
        const float wB = __shfl_sync(0xffffffffu, pB, j);
        const float* vr = kv_s + j * kSimtKvStride + lane;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float v = vr[32 * k];
          oA[k] = fmaf(wA, v, oA[k]);
          oB[k] = fmaf(wB, v, oB[k]);
        }
      }
    }

    // write this piece: final output if it is the whole row group, else a partial
    const float ln2 = 0.69314718055994530942f;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int row = rr ? rB : rA;
      if (row >= p.rows) continue;
      const float l = rr ? lB : lA, m = rr ? mB : mA;
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      const float lse = (l > 0.f) ? (m + log2f(l)) * ln2 : -INFINITY;
      const float* o = rr ? oB : oA;
      if (p.splits == 1) {
        const int64_t orow = (int64_t)b * p.rows + row;
#pragma unroll
        for (int k = 0; k < 16; ++k) store_out(p.out, p.dtype, orow * kDl + lane + 32 * k, o[k] * inv);
        if (lane == 0 && p.lse) p.lse[orow] = lse;
      } else {
        const int64_t prow = item * kSimtRG + (row - row0);
#pragma unroll
        for (int k = 0; k < 16; ++k) p.part_o[prow * kDl + lane + 32 * k] = o[k] * inv;
        if (lane == 0) p.part_lse[prow] = lse;
      }
    }
  }
}

cudaError_t launch_attn_simt(const Params& p, cudaStream_t stream) {
  const int grid = p.grid;
  if (p.dtype == MLA_BF16) {
    cudaFuncSetAttribute(attn_simt_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSimtSmem);
    attn_simt_kernel<__nv_bfloat16><<<grid, kSimtThreads, kSimtSmem, stream>>>(p);
  } else {
    cudaFuncSetAttribute(attn_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSimtSmem);
    attn_simt_kernel<float><<<grid, kSimtThreads, kSimtSmem, stream>>>(p);
  }
  return cudaGetLastError();
}

int simt_rows_per_group() { return kSimtRG; }
int simt_ctas_per_gpu(int sm_count) { return 2 * sm_count; }  // two resident CTAs per SM
int simt_tokens_per_tile() { return kSimtTK; }

}  // namespace mlav
