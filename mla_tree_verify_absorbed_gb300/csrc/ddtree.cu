// DDTree draft-tree construction and greedy token acceptance, with their C
// ABI (include/mla_ddtree.h).
//
// The pages name both steps as kernels of the DFlash / DDTree project next to
// tree-verify attention ("Reading the Reference: How a Single File-Read
// Message Anchored a Complex CUDA Kernel Implementation", section "Input
// Knowledge Required to Understand This Message", item 1); the rules
// implemented are the readings stated in the header.
//
// Both are latency-bound: a sequence is a few hundred bytes of input and its
// selection is a chain of `budget` dependent steps, so each sequence gets one
// warp and the whole working set lives in registers and shared memory.
//
// Construction, per warp.  Key of a draft node: (score, higher first; then
// rank sequence, lexicographically smaller first).  Rank sequences are packed
// four bits per depth, depth 1 in the top nibble, with the depths below the
// node's own left at zero; comparing (packed value, depth) then orders rank
// sequences exactly lexicographically with a prefix before its extensions.
// Every node has at most two successors in the left-child / right-sibling
// view of the tree: its first child (rank 0 one depth down) and its next
// sibling (rank + 1 at its own depth).  Neither outranks the node (a
// log-probability is <= 0 and each depth's list is best first; float32
// rounding is monotone), so selecting the best node of a frontier that starts
// at the best depth-1 node, and replacing each selected node by its two
// successors, yields the nodes in exactly the ranking order.  The frontier
// never holds more than budget + 1 <= 64 nodes.  A single warp has nothing to
// hide the latency of dependent instructions, so a step is kept short: the
// frontier lives in shared memory (one entry per slot) and each lane holds
// only the score keys of its two slots; one redux.sync max and two ballots
// name the winner (five butterfly rounds on (rank sequence, depth) only when
// several slots tie on score); every lane reads the winner's entry and
// computes its successors, so the arithmetic is uniform and only the writes
// are predicated.  The tree is staged in shared memory and written out with
// coalesced stores at the end.
#include <math.h>

#include "common.cuh"
#include "../../include/mla_ddtree.h"

namespace mlav {
namespace {

constexpr int kTreeWarps = 4;  // sequences per CTA
constexpr int kMaxDepth = MLA_DDTREE_MAX_DEPTH;
constexpr int kMaxCand = MLA_DDTREE_MAX_CAND;

static_assert(kMaxDepth * 4 <= 64 && kMaxCand <= 16, "rank sequences are packed 4 bits per depth");

// Larger float (scores are <= 0 or -inf) -> larger key; +0 and -0 the same
// key, as they compare equal.  0 is below every key of a valid node.
__device__ __forceinline__ uint32_t score_key(float s) {
  if (s == 0.0f) s = 0.0f;
  const uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int rank_shift(int depth) { return 4 * (kMaxDepth - depth); }

// The frontier of one sequence, one entry per slot (64 slots), in shared
// memory; each lane keeps the score keys of its two slots (lane, 32 + lane) in
// registers.
struct Frontier {
  float score[MLA_MAX_Q];
  float pscore[MLA_MAX_Q];  // the parent's score
  uint64_t packed[MLA_MAX_Q];
  int32_t depth[MLA_MAX_Q];
  int32_t rank[MLA_MAX_Q];
  int32_t parent[MLA_MAX_Q];
};

struct BuildParams {
  int B, L, K, budget;
  const int32_t* root_token;
  const int32_t* cand_token;
  const float* cand_logp;
  int32_t* tree_parent;
  int32_t* tree_token;
  int32_t* tree_depth;
  float* tree_score;
  uint32_t* err;
};

__global__ void __launch_bounds__(kTreeWarps * 32) ddtree_build_kernel(BuildParams p) {
  __shared__ float s_lp[kTreeWarps][kMaxDepth * kMaxCand];
  __shared__ int32_t s_tok[kTreeWarps][kMaxDepth * kMaxCand];
  __shared__ int32_t s_par[kTreeWarps][MLA_MAX_Q], s_ntok[kTreeWarps][MLA_MAX_Q], s_dep[kTreeWarps][MLA_MAX_Q];
  __shared__ float s_sc[kTreeWarps][MLA_MAX_Q];
  __shared__ Frontier s_fr[kTreeWarps];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int b = blockIdx.x * kTreeWarps + w;
  if (b >= p.B) return;  // whole warp
  const int LK = p.L * p.K, Q = p.budget + 1;
  float* lp = s_lp[w];
  int32_t* tok = s_tok[w];
  Frontier& fr = s_fr[w];
  const float* glp = p.cand_logp + (int64_t)b * LK;
  const int32_t* gtok = p.cand_token + (int64_t)b * LK;
  for (int i = lane; i < LK; i += 32) {
    lp[i] = glp[i];
    tok[i] = gtok[i];
  }
  __syncwarp();
  bool bad = false;
  for (int i = lane; i < LK; i += 32) {
    const float v = lp[i];
    bad |= isnan(v) || v > 0.0f || (i % p.K != 0 && v > lp[i - 1]);
  }
  if (__any_sync(0xffffffffu, bad)) {
    if (lane == 0) set_err(p.err, MLA_DEVERR_DRAFT);
    return;
  }

  int32_t* o_par = s_par[w];
  int32_t* o_tok = s_ntok[w];
  int32_t* o_dep = s_dep[w];
  float* o_sc = s_sc[w];
  if (lane == 0) {
    o_par[0] = -1;
    o_tok[0] = p.root_token[b];
    o_dep[0] = 0;
    o_sc[0] = 0.0f;
    // slot 0: the best depth-1 node
    fr.score[0] = 0.0f + lp[0];
    fr.pscore[0] = 0.0f;
    fr.packed[0] = 0;
    fr.depth[0] = 1;
    fr.rank[0] = 0;
    fr.parent[0] = 0;
  }
  // score keys of slots lane and 32 + lane (0 = empty).  A selected node's
  // first child reuses its slot; its next sibling takes slot `next_free`,
  // which only grows: 1 + (one per step) <= 1 + budget <= 64.
  uint32_t k0 = 0, k1 = 0;
  if (lane == 0) k0 = score_key(0.0f + lp[0]);
  __syncwarp();
  int next_free = 1;
  for (int n = 1; n < Q; ++n) {
    const uint32_t lk = k0 > k1 ? k0 : k1;
    const uint32_t top = __reduce_max_sync(0xffffffffu, lk);
    if (top == 0) {  // frontier exhausted: the host check on budget rules this out
      if (lane == 0) set_err(p.err, MLA_DEVERR_DRAFT);
      return;
    }
    const unsigned t0 = __ballot_sync(0xffffffffu, k0 == top);
    const unsigned t1 = __ballot_sync(0xffffffffu, k1 == top);
    int win;  // slot of the selected node
    if (__popc(t0) + __popc(t1) == 1) {
      win = t0 ? __ffs(t0) - 1 : 32 + __ffs(t1) - 1;
    } else {
      // equal scores: the smallest (rank sequence, depth) wins
      uint64_t bp = ~0ull;
      int bd = 0x7fffffff, bi = 64;
      if (k0 == top) {
        bp = fr.packed[lane];
        bd = fr.depth[lane];
        bi = lane;
      }
      if (k1 == top) {
        const uint64_t p1 = fr.packed[32 + lane];
        const int d1 = fr.depth[32 + lane];
        if (p1 < bp || (p1 == bp && d1 < bd)) {
          bp = p1;
          bd = d1;
          bi = 32 + lane;
        }
      }
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) {
        const uint64_t p2 = __shfl_xor_sync(0xffffffffu, bp, m);
        const int d2 = __shfl_xor_sync(0xffffffffu, bd, m);
        const int i2 = __shfl_xor_sync(0xffffffffu, bi, m);
        if (p2 < bp || (p2 == bp && (d2 < bd || (d2 == bd && i2 < bi)))) {
          bp = p2;
          bd = d2;
          bi = i2;
        }
      }
      win = bi;
    }
    // every lane reads the winner and computes its successors (uniform values)
    const float wsc = fr.score[win], wps = fr.pscore[win];
    const uint64_t wpk = fr.packed[win];
    const int wd = fr.depth[win], wr = fr.rank[win], wpar = fr.parent[win];
    const bool has_child = wd < p.L, has_sib = wr + 1 < p.K;
    const float csc = has_child ? wsc + lp[wd * p.K] : 0.0f;
    const float ssc = has_sib ? wps + lp[(wd - 1) * p.K + wr + 1] : 0.0f;
    const uint32_t ckey = has_child ? score_key(csc) : 0u;
    const uint32_t skey = has_sib ? score_key(ssc) : 0u;
    const int sslot = next_free;
    __syncwarp();  // all reads of the winner's entry precede the writes below
    if (lane == 0) {
      o_par[n] = wpar;
      o_tok[n] = tok[(wd - 1) * p.K + wr];
      o_dep[n] = wd;
      o_sc[n] = wsc;
      if (has_child) {
        fr.score[win] = csc;
        fr.pscore[win] = wsc;
        fr.depth[win] = wd + 1;
        fr.rank[win] = 0;
        fr.parent[win] = n;  // packed unchanged: rank 0 at the new depth
      }
      if (has_sib) {
        fr.score[sslot] = ssc;
        fr.pscore[sslot] = wps;
        fr.packed[sslot] = wpk + (1ull << rank_shift(wd));
        fr.depth[sslot] = wd;
        fr.rank[sslot] = wr + 1;
        fr.parent[sslot] = wpar;
      }
    }
    if (lane == (win & 31)) {
      if (win >> 5) k1 = ckey; else k0 = ckey;
    }
    if (has_sib) {
      if (lane == (sslot & 31)) {
        if (sslot >> 5) k1 = skey; else k0 = skey;
      }
      ++next_free;
    }
    __syncwarp();  // the frontier writes are visible to the next step's reads
  }
  __syncwarp();
  const int64_t o = (int64_t)b * Q;
  for (int j = lane; j < Q; j += 32) {
    p.tree_parent[o + j] = o_par[j];
    p.tree_token[o + j] = o_tok[j];
    if (p.tree_depth) p.tree_depth[o + j] = o_dep[j];
    if (p.tree_score) p.tree_score[o + j] = o_sc[j];
  }
}

struct AcceptParams {
  int B, Q;
  const int32_t* tree_parent;
  const int32_t* tree_token;
  const int32_t* target_token;
  const int32_t* node_slot;
  int32_t* accept_len;
  int32_t* accept_nodes;
  int32_t* accept_slots;
  int32_t* next_token;
  uint32_t* err;
};

// One warp per sequence; node j sits in lane j & 31, register j >> 5.
__global__ void __launch_bounds__(kTreeWarps * 32) ddtree_accept_kernel(AcceptParams p) {
  __shared__ int32_t s_path[kTreeWarps][MLA_MAX_Q];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int b = blockIdx.x * kTreeWarps + w;
  if (b >= p.B) return;
  const int64_t o = (int64_t)b * p.Q;
  int par[2], tk[2], tg[2];
  bool bad = false;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int j = lane + 32 * h;
    const bool in = j < p.Q;
    par[h] = in ? p.tree_parent[o + j] : -2;
    tk[h] = in ? p.tree_token[o + j] : 0;
    tg[h] = in ? p.target_token[o + j] : 0;
    if (in) bad |= (j == 0) ? par[h] != -1 : (par[h] < 0 || par[h] >= j);
  }
  if (__any_sync(0xffffffffu, bad)) {
    if (lane == 0) set_err(p.err, MLA_DEVERR_PARENT);
    return;
  }
  int32_t* path = s_path[w];
  int cur = 0, len = 1;
  if (lane == 0) path[0] = 0;
  // parents precede children, so cur grows every step and the walk ends
  for (;;) {
    const int want = __shfl_sync(0xffffffffu, cur < 32 ? tg[0] : tg[1], cur & 31);
    const unsigned m0 = __ballot_sync(0xffffffffu, par[0] == cur && tk[0] == want);
    const unsigned m1 = __ballot_sync(0xffffffffu, par[1] == cur && tk[1] == want);
    if (!(m0 | m1)) break;
    cur = m0 ? __ffs(m0) - 1 : 32 + __ffs(m1) - 1;
    if (lane == 0) path[len] = cur;
    ++len;
  }
  __syncwarp();
  const int bonus = __shfl_sync(0xffffffffu, cur < 32 ? tg[0] : tg[1], cur & 31);
  for (int j = lane; j < p.Q; j += 32) {
    const int v = j < len ? path[j] : -1;
    p.accept_nodes[o + j] = v;
    if (p.accept_slots) p.accept_slots[o + j] = j < len ? p.node_slot[o + v] : -1;
  }
  if (lane == 0) {
    p.accept_len[b] = len;
    p.next_token[b] = bonus;
  }
}

bool aligned4(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 3u) == 0; }

mla_status check_ws(void* ws, size_t bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || bytes < MLA_DDTREE_WORKSPACE_BYTES)
    return MLA_ERR_WORKSPACE;
  return MLA_OK;
}

// K + K^2 + ... + K^L, saturated above the largest budget
int64_t draft_nodes(int L, int K) {
  int64_t total = 0, pw = 1;
  for (int d = 1; d <= L; ++d) {
    pw *= K;
    total += pw;
    if (total > MLA_DDTREE_MAX_BUDGET) return total;
  }
  return total;
}

}  // namespace
}  // namespace mlav

using namespace mlav;

extern "C" mla_status mla_ddtree_build(const mla_ddtree_build_args* a, void* ws, size_t ws_bytes,
                                       mla_stream_t stream) {
  if (!a || a->B < 0) return MLA_ERR_INVALID_ARG;
  if (a->L < 1 || a->L > kMaxDepth || a->K < 1 || a->K > kMaxCand) return MLA_ERR_INVALID_ARG;
  if (a->budget < 1 || a->budget > MLA_DDTREE_MAX_BUDGET || a->budget > draft_nodes(a->L, a->K))
    return MLA_ERR_INVALID_ARG;
  const mla_status wst = check_ws(ws, ws_bytes);
  if (wst != MLA_OK) return wst;
  if (a->B == 0) return MLA_OK;
  if (!a->root_token || !a->cand_token || !a->cand_logp || !a->tree_parent || !a->tree_token)
    return MLA_ERR_INVALID_ARG;
  const void* ptrs[] = {a->root_token, a->cand_token, a->cand_logp, a->tree_parent,
                        a->tree_token, a->tree_depth, a->tree_score};
  for (const void* q : ptrs)
    if (!aligned4(q)) return MLA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, 16, st) != cudaSuccess) return MLA_ERR_CUDA;
  BuildParams p;
  p.B = a->B;
  p.L = a->L;
  p.K = a->K;
  p.budget = a->budget;
  p.root_token = a->root_token;
  p.cand_token = a->cand_token;
  p.cand_logp = a->cand_logp;
  p.tree_parent = a->tree_parent;
  p.tree_token = a->tree_token;
  p.tree_depth = a->tree_depth;
  p.tree_score = a->tree_score;
  p.err = static_cast<uint32_t*>(ws);
  const int grid = (a->B + kTreeWarps - 1) / kTreeWarps;
  ddtree_build_kernel<<<grid, kTreeWarps * 32, 0, st>>>(p);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

extern "C" mla_status mla_ddtree_accept(const mla_ddtree_accept_args* a, void* ws, size_t ws_bytes,
                                        mla_stream_t stream) {
  if (!a || a->B < 0 || a->Q < 1 || a->Q > MLA_MAX_Q) return MLA_ERR_INVALID_ARG;
  if (a->accept_slots && !a->node_slot) return MLA_ERR_INVALID_ARG;
  const mla_status wst = check_ws(ws, ws_bytes);
  if (wst != MLA_OK) return wst;
  if (a->B == 0) return MLA_OK;
  if (!a->tree_parent || !a->tree_token || !a->target_token || !a->accept_len || !a->accept_nodes ||
      !a->next_token)
    return MLA_ERR_INVALID_ARG;
  const void* ptrs[] = {a->tree_parent, a->tree_token, a->target_token, a->node_slot,
                        a->accept_len,  a->accept_nodes, a->accept_slots, a->next_token};
  for (const void* q : ptrs)
    if (!aligned4(q)) return MLA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, 16, st) != cudaSuccess) return MLA_ERR_CUDA;
  AcceptParams p;
  p.B = a->B;
  p.Q = a->Q;
  p.tree_parent = a->tree_parent;
  p.tree_token = a->tree_token;
  p.target_token = a->target_token;
  p.node_slot = a->node_slot;
  p.accept_len = a->accept_len;
  p.accept_nodes = a->accept_nodes;
  p.accept_slots = a->accept_slots;
  p.next_token = a->next_token;
  p.err = static_cast<uint32_t*>(ws);
  const int grid = (a->B + kTreeWarps - 1) / kTreeWarps;
  ddtree_accept_kernel<<<grid, kTreeWarps * 32, 0, st>>>(p);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
