"""CPU oracle for DDTree draft-tree construction and greedy token acceptance.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers.  Nothing in the CUDA
library or its Python binding imports this module, and it imports nothing
from them.  Plain Python loops: it is meant for small batches.

Source.  "Reading the Reference: How a Single File-Read Message Anchored a
Complex CUDA Kernel Implementation", section "Input Knowledge Required to
Understand This Message", item 1, names tree construction and token
acceptance as kernels of the DFlash / DDTree speculative-decoding project,
next to tree-verify attention, and says nothing more about them.  The
readings taken here (the plainest ones the rest of the pages support):

* The drafter (DFlash drafts a block of future positions in one pass) gives,
  for every depth d = 1..L below the root, its K best candidate tokens with
  log-probabilities, best first: cand_token[d-1][k], cand_logp[d-1][k].
* A draft node is a sequence of candidate ranks (k_1, ..., k_d); its token is
  cand_token[d-1][k_d] and its score is the log of the product of its
  positions' draft probabilities, accumulated in float32 from the root down:
  score(k_1..k_d) = score(k_1..k_{d-1}) + cand_logp[d-1][k_d], score(root) = 0.
* Under a budget of `budget` draft nodes the tree is the `budget` nodes with
  the highest score; equal scores go to the lexicographically smaller rank
  sequence (a prefix before its extensions).  Because log-probabilities are
  <= 0 a node never outscores its parent, so the chosen set always contains
  every chosen node's parent.
* Output order is the order of that ranking, after node 0 = the root (the
  last committed token, parent -1).  A node's parent therefore always has a
  smaller index, which is the tree format the verify attention takes.
* Acceptance is greedy: target_token[i] is the target model's next-token
  choice after node i (from the verify pass).  Starting at the root, the walk
  moves to the child of the current node whose token equals the target's
  choice at the current node (the lowest-index such child), as long as there
  is one.  The accepted nodes are the root and every node walked to; the
  target's choice at the last one is the bonus token.

Each function below states its check of the inputs; a violated requirement
raises ValueError.
"""
from __future__ import annotations

from typing import List, Optional, Tuple

import numpy as np

MAX_DEPTH = 16
MAX_CAND = 16
MAX_BUDGET = 63


def node_count(L: int, K: int) -> int:
    """Draft nodes that exist at all: K + K^2 + ... + K^L."""
    return sum(K ** d for d in range(1, L + 1))


def check_draft(cand_logp: np.ndarray) -> None:
    """Every log-probability is a number <= 0 and each depth's list is best first."""
    lp = np.asarray(cand_logp, dtype=np.float32)
    if np.isnan(lp).any() or (lp > 0).any():
        raise ValueError("log-probabilities must be <= 0 and not NaN")
    if (lp[..., 1:] > lp[..., :-1]).any():
        raise ValueError("candidates must be sorted best first")


def build_tree_one(root_token: int, cand_token: np.ndarray, cand_logp: np.ndarray, budget: int):
    """The DDTree for one sequence.

    Returns (parent, token, depth, score) of the 1 + budget nodes, node 0 the
    root.  The selection follows the definition directly: the chosen set grows
    one node at a time, each time taking the best node (highest score, then
    smallest rank sequence) among the children of the nodes chosen so far.
    Since no node outscores its parent, the node taken at each step is the
    best node not chosen yet, so the order is the ranking itself.
    """
    cand_token = np.asarray(cand_token)
    lp = np.asarray(cand_logp, dtype=np.float32)
    L, K = lp.shape
    check_draft(lp)
    if not 1 <= budget <= node_count(L, K):
        raise ValueError("budget outside 1 .. number of draft nodes")

    parent: List[int] = [-1]
    token: List[int] = [int(root_token)]
    depth: List[int] = [0]
    score: List[np.float32] = [np.float32(0.0)]
    ranks: List[Tuple[int, ...]] = [()]

    def children(i: int):
        d = depth[i]
        if d == L:
            return []
        return [(np.float32(score[i] + lp[d, k]), ranks[i] + (k,), i) for k in range(K)]

    frontier = children(0)
    while len(parent) < 1 + budget:
        best = min(frontier, key=lambda c: (-c[0], c[1]))
        frontier.remove(best)
        s, r, par = best
        parent.append(par)
        token.append(int(cand_token[len(r) - 1, r[-1]]))
        depth.append(len(r))
        score.append(s)
        ranks.append(r)
        frontier.extend(children(len(parent) - 1))
    return (np.asarray(parent, dtype=np.int32), np.asarray(token, dtype=np.int32),
            np.asarray(depth, dtype=np.int32), np.asarray(score, dtype=np.float32))


def build_tree(root_token, cand_token, cand_logp, budget: int):
    """Batched build_tree_one: inputs [B], [B][L][K], [B][L][K]; outputs [B][1+budget]."""
    root_token = np.asarray(root_token)
    B = root_token.shape[0]
    outs = [build_tree_one(root_token[b], cand_token[b], cand_logp[b], budget) for b in range(B)]
    if B == 0:
        z = np.zeros((0, budget + 1))
        return (z.astype(np.int32), z.astype(np.int32), z.astype(np.int32), z.astype(np.float32))
    return tuple(np.stack([o[j] for o in outs]) for j in range(4))


def check_tree(tree_parent: np.ndarray) -> None:
    """Node 0 is the only root; every other node's parent has a smaller index."""
    tp = np.asarray(tree_parent)
    if tp.shape[0] < 1 or tp[0] != -1:
        raise ValueError("node 0 must be the root (parent -1)")
    for i in range(1, tp.shape[0]):
        if not 0 <= tp[i] < i:
            raise ValueError("parent must precede its node")


def accept_one(tree_parent, tree_token, target_token, node_slot=None):
    """Greedy acceptance for one sequence.

    Returns (accepted node indices, bonus token, accepted nodes' slots or
    None).  The walk starts at the root and moves to the lowest-index child of
    the current node whose token is the target's choice at the current node.
    """
    tp = np.asarray(tree_parent)
    tt = np.asarray(tree_token)
    tg = np.asarray(target_token)
    check_tree(tp)
    path = [0]
    cur = 0
    while True:
        nxt = None
        for j in range(tp.shape[0]):
            if tp[j] == cur and tt[j] == tg[cur]:
                nxt = j
                break
        if nxt is None:
            break
        path.append(nxt)
        cur = nxt
    slots = None if node_slot is None else [int(node_slot[j]) for j in path]
    return path, int(tg[cur]), slots


def accept(tree_parent, tree_token, target_token, node_slot: Optional[np.ndarray] = None):
    """Batched accept_one.  Returns accept_len [B], accept_nodes [B][Q] (-1 after
    the path), next_token [B], accept_slots [B][Q] (-1 padded) or None."""
    tp = np.asarray(tree_parent)
    B, Q = tp.shape
    n_len = np.zeros(B, dtype=np.int32)
    nodes = np.full((B, Q), -1, dtype=np.int32)
    nxt = np.zeros(B, dtype=np.int32)
    slots = None if node_slot is None else np.full((B, Q), -1, dtype=np.int32)
    for b in range(B):
        path, bonus, sl = accept_one(tp[b], tree_token[b], target_token[b],
                                     None if node_slot is None else node_slot[b])
        n_len[b] = len(path)
        nodes[b, :len(path)] = path
        nxt[b] = bonus
        if slots is not None:
            slots[b, :len(path)] = sl
    return n_len, nodes, nxt, slots
