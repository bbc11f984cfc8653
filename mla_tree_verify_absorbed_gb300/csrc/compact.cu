// KV compaction: rewrites the cache rows a batch of sequences reads, scattered
// over the pool, into one contiguous run of slots, and writes the page_size=1
// index table of the new layout.
//
// The pages name KV-cache defragmentation as a phase of the work ("Ground
// Truth in Silicon ...", section "Why This Message Was Written": defragmentation
// in two tiers; "The Critical Glue ...", section "What Came Before") because
// a 200k context whose slots are scattered over the pool reads its KV row by
// row.  This is the device step of that: for every sequence b and logical
// position p in [0, prefix_lens[b] + Q) (prefix first, then the tree nodes in
// order, the order the verify call reads them), the kv_c and k_pe rows of the
// slot that position resolves to are copied to destination slot
// dst_slot0 + (sum of earlier sequences' lengths) + p.  Rows are copied whole,
// bit for bit; the verify call on the new layout reads the same values in the
// same order.
//
// It runs after the metadata kernel, which has validated every table entry
// and built the per-sequence offsets; when that found a bad table the copy
// touches nothing.  Each warp moves two rows per step with 16-byte vector
// loads and stores: the copy is bound by HBM (each row read once, written
// once).
#include "common.cuh"

namespace mlav {

constexpr int kCompactThreads = 256;

// Row k of the flat order: its destination slot (or -1 when it does not fit)
// and the source slot it resolves to.
__device__ __forceinline__ int64_t compact_dst(const Params& p, int64_t k, int64_t dst_slot0, int64_t dst_slots,
                                               int64_t* src) {
  const int64_t d = dst_slot0 + k;
  if (d >= dst_slots) return -1;
  const int b = seq_of(p.seq_kv_base, p.B, k);
  *src = resolve_slot(p, b, k - p.seq_kv_base[b]);
  return d;
}

// One warp moves two rows per step: every lane loads its 16-byte pieces of
// both rows into registers first, then stores them (up to 4 kv_c pieces and
// 1 k_pe piece per lane and row: 2048 + 256 bytes for fp32 caches).
__global__ void __launch_bounds__(kCompactThreads) compact_kernel(Params p, uint8_t* dst_kvc, uint8_t* dst_kpe,
                                                                  int64_t dkvc_stride, int64_t dkpe_stride,
                                                                  int64_t dst_slot0, int64_t dst_slots,
                                                                  int32_t* new_idx, int32_t* new_indptr) {
  if (*p.err) return;  // a table failed validation: write nothing
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t total = p.seq_kv_base[p.B];
  const int el = p.dtype == MLA_BF16 ? 2 : 4;
  const int kvc_vec = kDl * el / 16, kpe_vec = kDr * el / 16;  // 16-byte pieces per row
  const uint8_t* __restrict__ src_kvc = static_cast<const uint8_t*>(p.kv_c);
  const uint8_t* __restrict__ src_kpe = static_cast<const uint8_t*>(p.k_pe);
  uint32_t e = 0;
  if (new_indptr && warp == 0)
    for (int b = lane; b <= p.B; b += 32) new_indptr[b] = (int32_t)p.seq_kv_base[b];
  for (int64_t k0 = 2 * warp; k0 < total; k0 += 2 * nwarps) {
    int64_t s[2] = {0, 0}, d[2];
    uint4 va[2][4], vr[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      d[h] = (k0 + h < total) ? compact_dst(p, k0 + h, dst_slot0, dst_slots, &s[h]) : -2;
      if (d[h] == -1) e |= MLA_DEVERR_CAPACITY;
      const uint4* a = reinterpret_cast<const uint4*>(src_kvc + s[h] * p.kv_c_stride * el);
      const uint4* r = reinterpret_cast<const uint4*>(src_kpe + s[h] * p.k_pe_stride * el);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int v = lane + 32 * q;
        if (d[h] >= 0 && v < kvc_vec) va[h][q] = a[v];
      }
      if (d[h] >= 0 && lane < kpe_vec) vr[h] = r[lane];
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (d[h] < 0) continue;
      uint4* da = reinterpret_cast<uint4*>(dst_kvc + d[h] * dkvc_stride * el);
      uint4* dr = reinterpret_cast<uint4*>(dst_kpe + d[h] * dkpe_stride * el);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int v = lane + 32 * q;
        if (v < kvc_vec) da[v] = va[h][q];
      }
      if (lane < kpe_vec) dr[lane] = vr[h];
      if (lane == 0) new_idx[k0 + h] = (int32_t)d[h];
    }
  }
  if (e && lane == 0) set_err(p.err, e);
}

cudaError_t launch_compact(const Params& p, int sm_count, void* dst_kvc, void* dst_kpe, int64_t dkvc_stride,
                           int64_t dkpe_stride, int64_t dst_slot0, int64_t dst_slots, int32_t* new_idx,
                           int32_t* new_indptr, cudaStream_t stream) {
  compact_kernel<<<8 * sm_count, kCompactThreads, 0, stream>>>(
      p, static_cast<uint8_t*>(dst_kvc), static_cast<uint8_t*>(dst_kpe), dkvc_stride, dkpe_stride, dst_slot0,
      dst_slots, new_idx, new_indptr);
  return cudaGetLastError();
}

}  // namespace mlav
