/*
 * mla_ddtree.h -- C ABI of the DDTree draft-tree construction and greedy
 * token-acceptance kernels that surround the verify attention of
 * mla_verify.h in a speculative-decoding step.
 *
 * The pages name both steps as kernels of the DFlash / DDTree project, next
 * to tree-verify attention ("Reading the Reference: How a Single File-Read
 * Message Anchored a Complex CUDA Kernel Implementation", section "Input
 * Knowledge Required to Understand This Message", item 1) and describe
 * neither.  The readings implemented here:
 *
 *   Construction.  A block drafter gives, for each depth d = 1..L below the
 *   root, its K best candidate tokens with log-probabilities, best first.  A
 *   draft node is a sequence of candidate ranks (k_1..k_d); its token is
 *   cand_token[d-1][k_d]; its score is the float32 sum, root first, of its
 *   positions' log-probabilities.  The tree is the `budget` highest-scoring
 *   nodes; equal scores go to the lexicographically smaller rank sequence (a
 *   prefix before its extensions).  Node 0 is the root (root_token, parent
 *   -1); nodes 1..budget follow in ranking order, so every parent index is
 *   smaller than its child's -- the tree_parent format mla_verify_attn takes,
 *   with Q = budget + 1.
 *
 *   Acceptance (greedy).  target_token[i] is the target model's next-token
 *   choice after node i.  From the root, the walk moves to the lowest-index
 *   child of the current node whose token equals the target's choice at the
 *   current node, while there is one.  Accepted: the root and every node
 *   walked to; the target's choice at the last one is the next (bonus) token.
 *
 * Conventions as in mla_verify.h: DEVICE pointers owned by the caller,
 * asynchronous on `stream`, nothing allocated, host-visible argument errors
 * returned before any launch.  The workspace holds only the error word: at
 * least MLA_DDTREE_WORKSPACE_BYTES of device memory, 256-byte aligned (a
 * verify workspace will do); each call clears its error word first, and
 * mla_verify_check reads it.  A sequence whose device-resident inputs break
 * a rule below sets the MLA_DEVERR_* bit named there and leaves that
 * sequence's outputs unwritten; the other sequences are processed.
 */
#ifndef MLA_DDTREE_H
#define MLA_DDTREE_H

#include "mla_verify.h"

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_DDTREE_MAX_DEPTH 16          /* L: drafted positions below the root */
#define MLA_DDTREE_MAX_CAND 16           /* K: candidates per depth */
#define MLA_DDTREE_MAX_BUDGET (MLA_MAX_Q - 1) /* draft nodes; the root makes Q = budget + 1 <= 64 */
#define MLA_DDTREE_WORKSPACE_BYTES 256u

#define MLA_DEVERR_DRAFT 0x100u /* a log-probability is NaN or > 0, or a depth's list is not best first */

typedef struct {
    int B;                    /* sequences, >= 0 (0 = no-op) */
    int L;                    /* depths, 1..MLA_DDTREE_MAX_DEPTH */
    int K;                    /* candidates per depth, 1..MLA_DDTREE_MAX_CAND */
    int budget;               /* draft nodes, 1..MLA_DDTREE_MAX_BUDGET and <= K + K^2 + ... + K^L */
    const int32_t *root_token;/* [B] */
    const int32_t *cand_token;/* [B][L][K], contiguous */
    const float *cand_logp;   /* [B][L][K], contiguous; per depth non-increasing in k, each <= 0
                                 (-inf allowed), not NaN -- else MLA_DEVERR_DRAFT */
    int32_t *tree_parent;     /* out [B][budget+1]: -1 for node 0, else the parent's index (< node) */
    int32_t *tree_token;      /* out [B][budget+1] */
    int32_t *tree_depth;      /* out [B][budget+1], 0 for the root; may be NULL */
    float *tree_score;        /* out [B][budget+1], the node's score (0 for the root); may be NULL */
} mla_ddtree_build_args;

/* Builds the draft tree of every sequence (one warp per sequence, best-first
 * selection of `budget` nodes).  Returns MLA_ERR_INVALID_ARG for a NULL
 * required pointer, a pointer not 4-byte aligned, or L, K, budget outside
 * the ranges above; MLA_ERR_WORKSPACE for a NULL, misaligned or too small
 * workspace; MLA_ERR_CUDA when the launch fails. */
mla_status mla_ddtree_build(const mla_ddtree_build_args *args, void *workspace, size_t ws_bytes,
                            mla_stream_t stream);

typedef struct {
    int B;                      /* sequences, >= 0 (0 = no-op) */
    int Q;                      /* tree nodes per sequence, 1..MLA_MAX_Q */
    const int32_t *tree_parent; /* [B][Q]: parent[0] == -1 and 0 <= parent[i] < i for i >= 1 --
                                   else MLA_DEVERR_PARENT */
    const int32_t *tree_token;  /* [B][Q] */
    const int32_t *target_token;/* [B][Q]: the target's next-token choice after each node */
    const int32_t *node_slot;   /* [B][Q] pool slot of each node's KV row; may be NULL */
    int32_t *accept_len;        /* out [B]: accepted nodes, root included (>= 1) */
    int32_t *accept_nodes;      /* out [B][Q]: accepted node indices root first, then -1 */
    int32_t *accept_slots;      /* out [B][Q]: node_slot of those nodes, then -1; may be NULL,
                                   needs node_slot */
    int32_t *next_token;        /* out [B]: the target's choice at the last accepted node */
} mla_ddtree_accept_args;

/* Greedy acceptance of every sequence (one warp per sequence).  With
 * page_size = 1 tables, appending accept_slots[b][0..accept_len[b]) to
 * sequence b's slot list commits the accepted nodes' KV rows without moving
 * them.  Returns MLA_ERR_INVALID_ARG for a NULL required pointer, a pointer
 * not 4-byte aligned, Q outside 1..MLA_MAX_Q, or accept_slots without
 * node_slot; MLA_ERR_WORKSPACE and MLA_ERR_CUDA as for mla_ddtree_build. */
mla_status mla_ddtree_accept(const mla_ddtree_accept_args *args, void *workspace, size_t ws_bytes,
                             mla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DDTREE_H */
