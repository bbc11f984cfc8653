// C ABI of the verify-attention library: argument validation, the work
// partition, workspace carving and the launch sequence
//   metadata kernel -> split-KV attention kernel -> LSE combine
// on the caller's stream.  Nothing here allocates device memory or
// synchronises the host (mla_verify_check excepted, by design).
#include <cmath>
#include <cstring>

#include "common.cuh"

namespace mlav {
cudaError_t launch_meta(const Params& p, int sm_count, int32_t* slots_out, int64_t capacity,
                        uint64_t* anc_out, cudaStream_t stream);
cudaError_t launch_attn_simt(const Params& p, cudaStream_t stream);
cudaError_t launch_combine(const Params& p, cudaStream_t stream, bool pdl);
int simt_rows_per_group();
int simt_tokens_per_tile();
cudaError_t launch_attn_tc(const Params& p, cudaStream_t stream, bool pdl);
int tc_rows_per_group();
int tc_tokens_per_tile();
int tc_clusters_per_gpu(int sm_count);
int simt_ctas_per_gpu(int sm_count);
int tc_default_for(int dtype);
cudaError_t launch_compact(const Params& p, int sm_count, void* dst_kvc, void* dst_kpe, int64_t dkvc_stride,
                           int64_t dkpe_stride, int64_t dst_slot0, int64_t dst_slots, int32_t* new_idx,
                           int32_t* new_indptr, cudaStream_t stream);
}  // namespace mlav

using namespace mlav;

namespace {

struct Plan {
  int algo;        // MLA_ALGO_SIMT or MLA_ALGO_TC (resolved)
  int rg, tk, groups;
  int splits;      // KV chunks per row group (S_max when auto_plan)
  int64_t items;   // B * splits * groups
  bool auto_plan;  // the metadata kernel picks the split count in [1, splits]
  int grid;        // CTAs (SIMT) or clusters (TC), persistent over items
  int sm_count;
  WsLayout L;
  bool noop;
};

int device_sm_count(int* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  *out = n;
  return 0;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// Shape-level checks: everything the workspace size depends on.
mla_status validate_shape(const mla_verify_args* a) {
  if (!a) return MLA_ERR_INVALID_ARG;
  if (a->B < 0 || a->Q < 0 || a->H < 1) return MLA_ERR_INVALID_ARG;
  if (a->Q > MLA_MAX_Q) return MLA_ERR_UNSUPPORTED;
  if (a->dtype != MLA_BF16 && a->dtype != MLA_FP32) return MLA_ERR_INVALID_ARG;
  if (a->algo != MLA_ALGO_AUTO && a->algo != MLA_ALGO_SIMT && a->algo != MLA_ALGO_TC)
    return MLA_ERR_INVALID_ARG;
  if (a->algo == MLA_ALGO_TC && a->dtype != MLA_BF16) return MLA_ERR_UNSUPPORTED;
  if ((int64_t)a->H * a->Q > (int64_t)1 << 24) return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

// Table-level checks shared by every call that reads the KV tables.
mla_status validate_tables(const mla_verify_args* a) {
  if (!a->prefix_lens || !a->tree_parent) return MLA_ERR_INVALID_ARG;
  if (a->kv_c_stride < MLA_DL || a->k_pe_stride < MLA_DR || a->pool_slots < 1 ||
      a->pool_slots > INT32_MAX)
    return MLA_ERR_INVALID_ARG;
  if (a->page_size < 1) return MLA_ERR_INVALID_ARG;
  if (a->page_size == 1) {
    if (!a->kv_indptr || !a->kv_indices) return MLA_ERR_INVALID_ARG;
  } else {
    if (!a->block_table || a->max_pages < 1) return MLA_ERR_INVALID_ARG;
    if ((int64_t)a->max_pages * a->page_size > INT32_MAX) return MLA_ERR_INVALID_ARG;
  }
  return MLA_OK;
}

// Everything the attention itself reads or writes.
mla_status validate_call(const mla_verify_args* a) {
  mla_status st = validate_tables(a);
  if (st != MLA_OK) return st;
  if (!a->q_lat || !a->q_pe || !a->kv_c || !a->k_pe || !a->prefix_lens || !a->tree_parent || !a->out)
    return MLA_ERR_INVALID_ARG;
  const int el = a->dtype == MLA_BF16 ? 2 : 4;
  if ((a->kv_c_stride * el) % 16 || (a->k_pe_stride * el) % 16) return MLA_ERR_INVALID_ARG;
  if (!aligned16(a->q_lat) || !aligned16(a->q_pe) || !aligned16(a->kv_c) || !aligned16(a->k_pe) ||
      !aligned16(a->out))
    return MLA_ERR_INVALID_ARG;
  // the kernels take the running maximum on raw scores and scale it after,
  // which needs a positive scale (masked scores are -inf: a zero scale would
  // turn them into NaN)
  if (!std::isfinite(a->scale) || !(a->scale > 0.f)) return MLA_ERR_INVALID_ARG;
  if (a->profile_events && (!a->profile_events[0] || !a->profile_events[1])) return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

// Smallest split count whose items fill `slots` concurrent workers to at
// least 90% over whole waves; failing that, the best fill for S <= 64.
int auto_splits(int64_t row_groups, int64_t slots) {
  int best = 1;
  double best_eff = -1.0;
  for (int S = 1; S <= 64; ++S) {
    const int64_t items = row_groups * S;
    const int64_t waves = (items + slots - 1) / slots;
    const double eff = (double)items / (double)(waves * slots);
    if (items >= slots && eff >= 0.9) return S;
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = S;
    }
  }
  return best;
}

// num_splits: 0 = auto (needs a device), > 0 = exactly that many KV chunks per
// row group.
mla_status make_plan(const mla_verify_args* a, int num_splits, Plan* pl) {
  mla_status st = validate_shape(a);
  if (st != MLA_OK) return st;
  if (num_splits < 0 || num_splits > 4096) return MLA_ERR_INVALID_ARG;
  std::memset(pl, 0, sizeof(*pl));
  pl->noop = (a->B == 0 || a->Q == 0);
  int algo = a->algo;
  if (algo == MLA_ALGO_AUTO) algo = tc_default_for(a->dtype);
  pl->algo = algo;
  if (algo == MLA_ALGO_TC) {
    pl->rg = tc_rows_per_group();
    pl->tk = tc_tokens_per_tile();
  } else {
    pl->rg = simt_rows_per_group();
    pl->tk = simt_tokens_per_tile();
  }
  const int64_t rows = (int64_t)a->H * a->Q;
  pl->groups = (int)((rows + pl->rg - 1) / pl->rg);
  if (pl->noop) {
    pl->L = ws_layout(0, 0, pl->rg, 0);
    return MLA_OK;
  }
  const int64_t row_groups = (int64_t)a->B * pl->groups;
  int64_t slots = 0;
  if (num_splits == 0) {
    if (device_sm_count(&pl->sm_count) != 0) return MLA_ERR_CUDA;
    slots = (algo == MLA_ALGO_TC) ? tc_clusters_per_gpu(pl->sm_count) : simt_ctas_per_gpu(pl->sm_count);
    if (slots < 1) slots = 1;
    pl->splits = auto_splits(row_groups, slots);
    // the tensor-core kernel's split count is then fixed on the device, from
    // the sequences' lengths, within [1, splits]
    pl->auto_plan = (algo == MLA_ALGO_TC);
  } else {
    pl->splits = num_splits;
  }
  pl->items = row_groups * pl->splits;
  if (pl->items > ((int64_t)1 << 26)) return MLA_ERR_UNSUPPORTED;
  int64_t part_slots = pl->splits > 1 ? pl->items : 0;
  // an automatic plan may keep one chunk per row group and cut the items of a
  // partial last wave into pieces, at most one per cluster
  if (pl->auto_plan && part_slots < slots) part_slots = slots;
  pl->L = ws_layout(a->B, a->Q, pl->rg, part_slots);
  return MLA_OK;
}

Params make_params(const mla_verify_args* a, const Plan& pl, void* ws) {
  Params p;
  std::memset(&p, 0, sizeof(p));
  p.B = a->B;
  p.Q = a->Q;
  p.H = a->H;
  p.rows = a->H * a->Q;
  p.dtype = a->dtype;
  p.q_lat = a->q_lat;
  p.q_pe = a->q_pe;
  p.kv_c = a->kv_c;
  p.k_pe = a->k_pe;
  p.kv_c_stride = a->kv_c_stride;
  p.k_pe_stride = a->k_pe_stride;
  p.pool_slots = a->pool_slots;
  p.page_size = a->page_size;
  p.kv_indptr = a->kv_indptr;
  p.kv_indices = a->kv_indices;
  p.block_table = a->block_table;
  p.max_pages = a->max_pages;
  p.prefix_lens = a->prefix_lens;
  p.tree_parent = a->tree_parent;
  p.scale = a->scale;
  p.scale_log2 = (float)((double)a->scale * 1.4426950408889634);
  p.out = a->out;
  p.lse = a->lse;
  p.rg = pl.rg;
  p.groups = pl.groups;
  p.tk = pl.tk;
  p.splits = pl.splits;
  p.n_items = pl.items;
  p.grid = pl.grid;
  p.auto_plan = pl.auto_plan ? 1 : 0;
  char* base = static_cast<char*>(ws);
  p.err = reinterpret_cast<uint32_t*>(base + pl.L.err);
  p.plan = reinterpret_cast<int32_t*>(base + pl.L.plan);
  p.anc = reinterpret_cast<uint64_t*>(base + pl.L.anc);
  p.seq_tiles = reinterpret_cast<int32_t*>(base + pl.L.seq_tiles);
  p.seq_kv_base = reinterpret_cast<int64_t*>(base + pl.L.seq_kv_base);
  p.part_lse = reinterpret_cast<float*>(base + pl.L.part_lse);
  p.part_o = reinterpret_cast<float*>(base + pl.L.part_o);
  p.part_slots = pl.L.part_slots;
  return p;
}

mla_status check_ws(const Plan& pl, const void* ws, size_t ws_bytes) {
  if (!ws) return MLA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return MLA_ERR_WORKSPACE;
  if (ws_bytes < pl.L.total) return MLA_ERR_WORKSPACE;
  return MLA_OK;
}

}  // namespace

namespace mlav {
// The split count a call with these arguments and num_splits would use
// (num_splits itself when > 0), or -1 when the arguments are invalid.
int plan_splits(const mla_verify_args* a, int num_splits) {
  Plan pl;
  if (make_plan(a, num_splits, &pl) != MLA_OK) return -1;
  return pl.noop ? 1 : pl.splits;
}
}  // namespace mlav

extern "C" {

size_t mla_verify_workspace_size(const mla_verify_args* a, int num_splits) {
  Plan pl;
  if (make_plan(a, num_splits, &pl) != MLA_OK) return 0;
  return pl.L.total;
}

}  // extern "C"

namespace {
mla_status run_attn(const mla_verify_args* a, void* workspace, size_t ws_bytes, int num_splits,
                    mla_stream_t stream, uint64_t hold_ns) {
  Plan pl;
  mla_status st = make_plan(a, num_splits, &pl);
  if (st != MLA_OK) return st;
  if (pl.noop) return MLA_OK;
  st = validate_call(a);
  if (st != MLA_OK) return st;
  st = check_ws(pl, workspace, ws_bytes);
  if (st != MLA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (pl.sm_count == 0 && device_sm_count(&pl.sm_count) != 0) return MLA_ERR_CUDA;
  {
    const int64_t cap = (pl.algo == MLA_ALGO_TC) ? tc_clusters_per_gpu(pl.sm_count) : simt_ctas_per_gpu(pl.sm_count);
    pl.grid = (int)(pl.items < cap ? pl.items : cap);
    if (pl.grid < 1) pl.grid = 1;
  }
  Params p = make_params(a, pl, workspace);
  p.hold_ns = hold_ns;
  if (launch_meta(p, pl.sm_count, nullptr, 0, nullptr, s) != cudaSuccess) return MLA_ERR_CUDA;
  // Consecutive kernels overlap launch and prologue with the previous kernel's
  // tail (programmatic dependent launch), except around the caller's profiling
  // events, which must see each kernel start and end on its own.
  const bool pdl = a->profile_events == nullptr;
  if (a->profile_events && cudaEventRecord((cudaEvent_t)a->profile_events[0], s) != cudaSuccess)
    return MLA_ERR_CUDA;
  cudaError_t e = (pl.algo == MLA_ALGO_TC) ? launch_attn_tc(p, s, pdl) : launch_attn_simt(p, s);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  if (a->profile_events && cudaEventRecord((cudaEvent_t)a->profile_events[1], s) != cudaSuccess)
    return MLA_ERR_CUDA;
  // the combine returns at once when the device plan kept every row group whole
  if ((pl.splits > 1 || pl.auto_plan) && launch_combine(p, s, pdl) != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}
}  // namespace

extern "C" {

mla_status mla_verify_attn(const mla_verify_args* a, void* workspace, size_t ws_bytes, int num_splits,
                           mla_stream_t stream) {
  return run_attn(a, workspace, ws_bytes, num_splits, stream, 0);
}

mla_status mla_verify_selftest_timeout(const mla_verify_args* a, void* workspace, size_t ws_bytes,
                                       uint64_t hold_ns, mla_stream_t stream) {
  if (!a) return MLA_ERR_INVALID_ARG;
  if (hold_ns == 0 || hold_ns > 1000000000ull) return MLA_ERR_INVALID_ARG;
  if (a->dtype != MLA_BF16 || (a->algo != MLA_ALGO_AUTO && a->algo != MLA_ALGO_TC)) return MLA_ERR_UNSUPPORTED;
  mla_verify_args t = *a;
  t.algo = MLA_ALGO_TC;
  if (t.B == 0 || t.Q == 0) return MLA_ERR_INVALID_ARG;  // the self-test needs a launch
  return run_attn(&t, workspace, ws_bytes, 0, stream, hold_ns);
}

mla_status mla_kv_compact(const mla_verify_args* a, void* workspace, size_t ws_bytes, void* dst_kv_c,
                          void* dst_k_pe, int64_t dst_kv_c_stride, int64_t dst_k_pe_stride, int64_t dst_slot0,
                          int64_t dst_slots, int32_t* new_kv_indices, int32_t* new_kv_indptr,
                          mla_stream_t stream) {
  Plan pl;
  mla_status st = make_plan(a, 1, &pl);
  if (st != MLA_OK) return st;
  st = validate_tables(a);
  if (st != MLA_OK) return st;
  if (!dst_kv_c || !dst_k_pe || !new_kv_indices) return MLA_ERR_INVALID_ARG;
  const int64_t el = a->dtype == MLA_BF16 ? 2 : 4;
  if (!aligned16(dst_kv_c) || !aligned16(dst_k_pe)) return MLA_ERR_INVALID_ARG;
  // source rows are read with 16-byte vector loads too
  if (!a->kv_c || !a->k_pe || !aligned16(a->kv_c) || !aligned16(a->k_pe) || (a->kv_c_stride * el) % 16 ||
      (a->k_pe_stride * el) % 16)
    return MLA_ERR_INVALID_ARG;
  if (dst_kv_c_stride < 512 || dst_k_pe_stride < 64 || (dst_kv_c_stride * el) % 16 || (dst_k_pe_stride * el) % 16)
    return MLA_ERR_INVALID_ARG;
  if (dst_slot0 < 0 || dst_slots < 0 || dst_slots > INT32_MAX) return MLA_ERR_INVALID_ARG;
  if (pl.noop) return MLA_OK;
  st = check_ws(pl, workspace, ws_bytes);
  if (st != MLA_OK) return st;
  if (device_sm_count(&pl.sm_count) != 0) return MLA_ERR_CUDA;
  const Params p = make_params(a, pl, workspace);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (launch_meta(p, pl.sm_count, nullptr, 0, nullptr, s) != cudaSuccess) return MLA_ERR_CUDA;
  if (launch_compact(p, pl.sm_count, dst_kv_c, dst_k_pe, dst_kv_c_stride, dst_k_pe_stride, dst_slot0, dst_slots,
                     new_kv_indices, new_kv_indptr, s) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

mla_status mla_verify_build_meta(const mla_verify_args* a, void* workspace, size_t ws_bytes, uint64_t* anc,
                                 int32_t* slots, int64_t slots_capacity, mla_stream_t stream) {
  Plan pl;
  mla_status st = make_plan(a, 1, &pl);
  if (st != MLA_OK) return st;
  if (pl.noop) return MLA_OK;
  st = validate_tables(a);
  if (st != MLA_OK) return st;
  if (!anc || !slots || slots_capacity < 0) return MLA_ERR_INVALID_ARG;
  st = check_ws(pl, workspace, ws_bytes);
  if (st != MLA_OK) return st;
  if (device_sm_count(&pl.sm_count) != 0) return MLA_ERR_CUDA;
  const Params p = make_params(a, pl, workspace);
  if (launch_meta(p, pl.sm_count, slots, slots_capacity, anc, reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

mla_status mla_verify_check(const void* workspace, mla_stream_t stream, uint32_t* bits) {
  if (!workspace) return MLA_ERR_WORKSPACE;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return MLA_ERR_CUDA;
  uint32_t v = 0;
  // the error word sits at offset 0 of every workspace layout
  if (cudaMemcpy(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ERR_CUDA;
  if (bits) *bits = v;
  return v ? MLA_ERR_DEVICE_CHECK : MLA_OK;
}

mla_status mla_verify_splits_used(const void* workspace, mla_stream_t stream, int32_t* splits) {
  if (!workspace) return MLA_ERR_WORKSPACE;
  if (!splits) return MLA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return MLA_ERR_CUDA;
  // the split count sits at offset 256 of every workspace layout
  int32_t v = 0;
  if (cudaMemcpy(&v, static_cast<const char*>(workspace) + 256, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MLA_ERR_CUDA;
  *splits = v;
  return MLA_OK;
}

const char* mla_status_str(mla_status s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
    case MLA_ERR_DEVICE_CHECK: return "MLA_ERR_DEVICE_CHECK";
  }
  return "MLA_ERR_UNKNOWN";
}

int mla_verify_abi_version(void) { return MLA_VERIFY_ABI_VERSION; }

}  // extern "C"
