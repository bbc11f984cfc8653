// Shared device-side definitions of the verify-attention kernels: the launch
// parameter block, the workspace layout, slot resolution, and the work-item
// partition that the attention and combine kernels agree on.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

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

  // partition: work item i = (b * S + k) * groups + g covers row group g of
  // sequence b over KV chunk k (tiles [k*T_b/S, (k+1)*T_b/S)), S the split
  // count of the call (*plan).  Chunk-major order puts the row groups of one
  // chunk next to each other, so items running at the same time read the same
  // KV from L2.
  int rg;            // rows per row group
  int groups;        // G = ceil(rows / rg)
  int tk;            // tokens per tile
  int splits;        // S_max: the workspace holds partials for B * S_max * G items
  int64_t n_items;   // B * S_max * G
  int grid;          // CTAs (or clusters) taking items round-robin
  int auto_plan;     // 1: the metadata kernel picks S in [1, S_max]; 0: S = S_max

  // workspace views
  uint32_t* err;
  int32_t* plan;           // [4] written by the metadata kernel: S, the grid it assumed, the first
                           // item of a tail cut into pieces, pieces per tail item (1: none)
  uint64_t* anc;           // [B][Q]
  int32_t* seq_tiles;      // [B]   T_b = ceil(N_b / tk)
  int64_t* seq_kv_base;    // [B+1] cumulative N_b
  float* part_lse;         // [part_slots][rg]  (natural log)
  float* part_o;           // [part_slots][rg][512], normalised partial outputs
  int64_t part_slots;      // partial slots the workspace holds (items, or pieces of a split tail)

  // failure-detection self-test only (0 otherwise): the tensor-core kernel
  // first waits, at most this many ns, on a barrier nothing completes
  uint64_t hold_ns;
};

// ---------------------------------------------------------------------------
// Workspace layout: fixed regions, each 256-byte aligned; the error words sit
// at offset 0 and the split count at offset 256 of every layout.
// ---------------------------------------------------------------------------
struct WsLayout {
  size_t err, plan, anc, seq_tiles, seq_kv_base, part_lse, part_o, total;
  int64_t part_slots;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline WsLayout ws_layout(int B, int Q, int rg, int64_t part_slots) {
  WsLayout L;
  size_t o = 0;
  L.err = o;          o = align256(o + 16);
  L.plan = o;         o = align256(o + 16);
  L.anc = o;          o = align256(o + sizeof(uint64_t) * (size_t)B * (size_t)Q + 8);
  L.seq_tiles = o;    o = align256(o + sizeof(int32_t) * (size_t)B + 4);
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

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start while the kernel before it in the stream is still
// running; grid_dep_wait() blocks until that kernel has completed and its
// writes are visible (it returns at once when the launch had no such
// dependency).  grid_dep_launch() lets the next kernel start launching once
// every CTA of this grid has called it or exited.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch with or without programmatic stream serialization.
template <class... KArgs, class... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                 bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

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

// One work item: row group g of sequence b over KV tiles [t0, t1).
struct Item {
  int b, g, k;
  int t0, t1;
};

// Item i of a call that cuts each row group's KV into S chunks.
__device__ __forceinline__ Item item_at(const Params& p, int S, int64_t i) {
  Item it;
  it.g = (int)(i % p.groups);
  const int64_t bk = i / p.groups;
  it.k = (int)(bk % S);
  it.b = (int)(bk / S);
  const int64_t T = p.seq_tiles[it.b];
  it.t0 = (int)((it.k * T) / S);
  it.t1 = (int)(((it.k + 1) * T) / S);
  return it;
}

// The work split of a call, as the metadata kernel fixed it: S KV chunks per
// row group give B * G * S items; with P > 1 (only when S = 1), each item from
// index `tail` on -- the last, partial wave of the persistent grid -- runs as
// P pieces of its tile range, so that wave keeps every cluster busy.  Work
// unit u < tail is item u; unit tail + v is piece v % P of item tail + v / P
// and writes partial slot v.  Words out of range fall back to S_max without
// pieces: the metadata kernel always writes them, and the checks only keep
// every index inside the workspace.
struct Split {
  int S, P;
  int64_t tail, n_items;
};

__device__ __forceinline__ Split read_split(const Params& p) {
  Split sp;
  sp.S = p.plan[0];
  if (sp.S < 1 || sp.S > p.splits) sp.S = p.splits;
  sp.n_items = (int64_t)p.B * p.groups * sp.S;
  sp.tail = p.plan[2];
  sp.P = p.plan[3];
  if (sp.S != 1 || sp.P < 2 || sp.P > p.grid || sp.tail < 0 || sp.tail > sp.n_items ||
      (sp.n_items - sp.tail) * sp.P > p.part_slots) {
    sp.P = 1;
    sp.tail = sp.n_items;
  }
  return sp;
}

// Sequence owning flat position k of the per-sequence prefix sums `base`.
__device__ __forceinline__ int seq_of(const int64_t* base, int B, int64_t k) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (base[mid] <= k) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// bf16 / fp32 store of one output element.
__device__ __forceinline__ void store_out(void* out, int dtype, int64_t idx, float v) {
  if (dtype == MLA_BF16) reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  else reinterpret_cast<float*>(out)[idx] = v;
}

}  // namespace mlav
