"""Seeded synthetic inputs for DDTree tree construction and acceptance.

This module only draws inputs: the drafter's per-depth candidate lists (token
ids with log-probabilities, best first), root tokens, and the target model's
next-token choices at the tree's nodes.  It holds none of the construction or
acceptance arithmetic, so the CUDA path and the CPU oracle can both be fed
from it.  No model or logits are available, so the draws stand in for a block
drafter's output:

* Per (sequence, depth) the drafter's distribution is a softmax over 256
  N(0, 2^2) logits in which one token gets a bonus of ``6 * exp(-d / 6)`` at
  depth d (1-based): the drafter is confident near the root and less so deep
  in the block.  The K largest probabilities, best first, give
  ``cand_logp = float32(log p)``; the K token ids are distinct draws from a
  vocabulary of 163,840 ids (the size of a Kimi / DeepSeek-V3 vocabulary).
* ``mode="ties"`` replaces the log-probabilities by multiples of -1/2 in
  [-1.5, 0] (sorted), so equal scores, zero log-probabilities (a node that
  scores the same as its parent) and equal siblings are common.
* ``mode="zeros"`` sets every rank past the second to -inf at a third of the
  depths (candidates with probability 0).
* Target choices: at a node of depth d < L the target picks, with probability
  ``p_follow``, the drafter's rank-r candidate for depth d + 1, r drawn
  geometrically (rank 0 most likely), else a random vocabulary id; at depth L
  always a random id.  Node depths come from the parent array alone.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

VOCAB = 163840


@dataclasses.dataclass
class Draft:
    name: str
    B: int
    L: int
    K: int
    budget: int
    root_token: np.ndarray  # [B] int32
    cand_token: np.ndarray  # [B][L][K] int32
    cand_logp: np.ndarray   # [B][L][K] float32, best first

    @property
    def Q(self) -> int:
        return self.budget + 1


def make_draft(*, name: str, B: int, L: int, K: int, budget: int, seed: int,
               mode: str = "softmax") -> Draft:
    rng = np.random.default_rng(seed)
    root = rng.integers(0, VOCAB, size=B, dtype=np.int64).astype(np.int32)
    tok = np.zeros((B, L, K), dtype=np.int32)
    lp = np.zeros((B, L, K), dtype=np.float32)
    for b in range(B):
        for d in range(L):
            tok[b, d] = rng.choice(VOCAB, size=K, replace=False).astype(np.int32)
            if mode == "ties":
                v = -0.5 * rng.integers(0, 4, size=K)
                lp[b, d] = np.sort(v)[::-1].astype(np.float32)
                continue
            z = 2.0 * rng.standard_normal(256)
            z[0] += 6.0 * np.exp(-(d + 1) / 6.0)
            z -= z.max()
            p = np.exp(z)
            p /= p.sum()
            top = np.sort(p)[::-1][:K]
            lp[b, d] = np.log(top).astype(np.float32)
            if mode == "zeros" and rng.random() < 1.0 / 3.0 and K > 2:
                lp[b, d, 2:] = -np.inf
    return Draft(name=name, B=B, L=L, K=K, budget=budget, root_token=root, cand_token=tok, cand_logp=lp)


def node_depths(tree_parent: np.ndarray) -> np.ndarray:
    """Depth of every node (root 0) from the parent array [B][Q]."""
    tp = np.asarray(tree_parent)
    dep = np.zeros(tp.shape, dtype=np.int32)
    for b in range(tp.shape[0]):
        for i in range(tp.shape[1]):
            dep[b, i] = 0 if tp[b, i] < 0 else dep[b, tp[b, i]] + 1
    return dep


def make_targets(draft: Draft, tree_parent: np.ndarray, seed: int, p_follow: float = 0.8,
                 p_rank: float = 0.6) -> np.ndarray:
    """The target model's next-token choice at every node, [B][Q] int32."""
    rng = np.random.default_rng(seed)
    dep = node_depths(tree_parent)
    B, Q = dep.shape
    out = np.zeros((B, Q), dtype=np.int32)
    for b in range(B):
        for i in range(Q):
            d = dep[b, i]
            if d < draft.L and rng.random() < p_follow:
                r = min(int(rng.geometric(p_rank)) - 1, draft.K - 1)
                out[b, i] = draft.cand_token[b, d, r]
            else:
                out[b, i] = rng.integers(0, VOCAB)
    return out


def make_node_slots(B: int, Q: int, seed: int, pool_slots: int = 1 << 20) -> np.ndarray:
    """Distinct pool slots holding the tree nodes' KV rows, [B][Q] int32."""
    rng = np.random.default_rng(seed)
    return rng.choice(pool_slots, size=B * Q, replace=False).astype(np.int32).reshape(B, Q)


# Named workloads: one sequence with the 64-node tree of the verify benchmark,
# and a batch of such sequences.
DRAFT_CONFIGS = {
    "tree_b1": dict(B=1, L=16, K=8, budget=63, seed=21),
    "tree_b256": dict(B=256, L=16, K=8, budget=63, seed=22),
}


def make_draft_config(name: str, seed: Optional[int] = None, mode: str = "softmax") -> Draft:
    cfg = dict(DRAFT_CONFIGS[name])
    if seed is not None:
        cfg["seed"] = seed
    return make_draft(name=name, mode=mode, **cfg)


def random_rooted_tree(B: int, Q: int, seed: int, vocab: int = VOCAB):
    """Trees of Q nodes with node 0 the only root (parent[i] uniform in [0, i-1])
    and tokens drawn from ``vocab`` ids (a small vocab makes equal sibling
    tokens common).  Returns (tree_parent, tree_token) [B][Q] int32."""
    rng = np.random.default_rng(seed)
    tp = np.zeros((B, Q), dtype=np.int32)
    tt = rng.integers(0, vocab, size=(B, Q)).astype(np.int32)
    tp[:, 0] = -1
    for i in range(1, Q):
        tp[:, i] = rng.integers(0, i, size=B)
    return tp, tt
