// Shared device-side definitions of the verify-attention kernels: the launch
// parameter block, the workspace layout, slot resolution, and the linear
// work partition that the attention and combine kernels agree on.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/mla_verify.h"

namespace mlav {

constexpr int kDl = 512;
constexpr int kDr = 64;
constexpr int kDk = kDl + kDr;

// Everything a kernel needs, passed by value.
struct Params {
  int B, Q, H;
  int rows;          // H * Q rows per sequence; row r = node (r / H), head (r % H)
  int dtype;         // MLA_BF16 / MLA_FP32
  const void* q_lat;
  const void* q_pe;
  const void* kv_c;
  const void* k_pe;
  int64_t kv_c_stride, k_pe_stride, pool_slots;
  int page_size;
  const int32_t* kv_indptr;
  const int32_t* kv_indices;
  const int32_t* block_table;
  int max_pages;
  const int32_t* prefix_lens;
  const int32_t* tree_parent;
  float scale;       // natural-log score scale
  float scale_log2;  // scale * log2(e): scores in base-2 units
  void* out;
  float* lse;

  // partition
  int rg;            // rows per row group
  int groups;        // G = ceil(rows / rg)
  int tk;            // tokens per tile
  int units;         // U: work units the linear tile space is cut into

  // workspace views
  uint32_t* err;
  uint64_t* anc;           // [B][Q]
  int32_t* seq_tiles;      // [B]   T_b = ceil(N_b / tk)
  int64_t* seq_base;       // [B+1] cumulative G * T_b  (linear work positions)
  int64_t* seq_kv_base;    // [B+1] cumulative N_b
  float* part_lse;         // [slots][rg]  (natural log)
  float* part_o;           // [slots][rg][512], normalised partial outputs
};

// ---------------------------------------------------------------------------
// Workspace layout: fixed regions, each 256-byte aligned.
// ---------------------------------------------------------------------------
struct WsLayout {
  size_t err, anc, seq_tiles, seq_base, seq_kv_base, part_lse, part_o, total;
  int64_t part_slots;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline WsLayout ws_layout(int B, int Q, int rg, int64_t part_slots) {
  WsLayout L;
  size_t o = 0;
  L.err = o;          o = align256(o + 16);
  L.anc = o;          o = align256(o + sizeof(uint64_t) * (size_t)B * (size_t)Q + 8);
  L.seq_tiles = o;    o = align256(o + sizeof(int32_t) * (size_t)B + 4);
  L.seq_base = o;     o = align256(o + sizeof(int64_t) * ((size_t)B + 1));
  L.seq_kv_base = o;  o = align256(o + sizeof(int64_t) * ((size_t)B + 1));
  L.part_lse = o;     o = align256(o + sizeof(float) * (size_t)part_slots * rg);
  L.part_o = o;       o = align256(o + sizeof(float) * (size_t)part_slots * rg * kDl);
  L.total = o;
  L.part_slots = part_slots;
  return L;
}

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void set_err(uint32_t* err, uint32_t bits) { atomicOr(err, bits); }

// Pool slot of logical position `pos` of sequence b.  The metadata kernel has
// validated every table entry before any attention kernel runs; the clamps
// below only keep a bad table from ever producing an address outside the pool.
__device__ __forceinline__ int64_t resolve_slot(const Params& p, int b, int64_t pos) {
  int64_t s;
  if (p.page_size == 1) {
    s = p.kv_indices[(int64_t)p.kv_indptr[b] + pos];
  } else {
    int64_t pg = pos / p.page_size;
    if (pg >= p.max_pages) pg = p.max_pages - 1;
    s = (int64_t)p.block_table[(int64_t)b * p.max_pages + pg] * p.page_size + pos % p.page_size;
  }
  if (s < 0 || s >= p.pool_slots) s = 0;
  return s;
}

__device__ __forceinline__ float load_elem(const void* base, int dtype, int64_t idx) {
  if (dtype == MLA_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
  return reinterpret_cast<const float*>(base)[idx];
}

// Linear work space: position x in [0, W) with W = seq_base[B]; sequence b
// owns [seq_base[b], seq_base[b+1]) = G row groups x T_b tiles, row-group
// major.  Unit c owns [floor(c*W/U), floor((c+1)*W/U)).
__device__ __forceinline__ int64_t unit_lo(int64_t c, int64_t W, int64_t U) { return (c * W) / U; }

// The unit whose range contains position x (W >= 1).
__device__ __forceinline__ int64_t unit_of(int64_t x, int64_t W, int64_t U) {
  return ((x + 1) * U - 1) / W;
}

// Sequence owning linear position x (binary search over seq_base).
__device__ __forceinline__ int seq_of(const int64_t* seq_base, int B, int64_t x) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (seq_base[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Partial-output slot of unit c's piece of row group (b, g).  Units meeting a
// row group are consecutive, so c + (b*G + g) never collides; it stays below
// U + B*G.
__device__ __forceinline__ int64_t part_slot(int64_t c, int b, int g, int G) {
  return c + (int64_t)b * G + g;
}

// One contiguous piece of a unit's range inside one row group.
struct Segment {
  int b, g;
  int t0, t1;      // tiles [t0, t1) of sequence b
  int T;           // T_b
  bool whole;      // the piece is the row group's whole KV range
};

__device__ __forceinline__ Segment segment_at(const Params& p, int64_t x, int64_t hi) {
  Segment s;
  s.b = seq_of(p.seq_base, p.B, x);
  s.T = p.seq_tiles[s.b];
  int64_t off = x - p.seq_base[s.b];
  s.g = (int)(off / s.T);
  s.t0 = (int)(off % s.T);
  int64_t group_end = p.seq_base[s.b] + (int64_t)(s.g + 1) * s.T;
  int64_t end = hi < group_end ? hi : group_end;
  s.t1 = s.t0 + (int)(end - x);
  s.whole = (s.t0 == 0 && s.t1 == s.T);
  return s;
}

// bf16 / fp32 store of one output element.
__device__ __forceinline__ void store_out(void* out, int dtype, int64_t idx, float v) {
  if (dtype == MLA_BF16) reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  else reinterpret_cast<float*>(out)[idx] = v;
}

}  // namespace mlav
