"""Pins of the DDTree construction / acceptance oracle to facts other than itself.

Each pin takes the oracle module (``oracle.ddtree`` or a planted mutant of it)
and raises on a mismatch.  What pins it:

* hand-worked trees whose probabilities are far apart, expected values written
  out by hand from the reading stated in the oracle (top-``budget`` nodes by
  product of per-depth draft probabilities, ties to the smaller rank sequence,
  node 0 the root);
* brute force: every rank sequence up to depth L enumerated, scored, sorted,
  cut at the budget (tiny L and K only);
* special cases with a closed form: one candidate per depth gives a chain,
  one depth gives the root's children in rank order;
* acceptance against a different statement of the same rule (a node is
  accepted when its parent is and its token is the target's choice at its
  parent) and against hand-worked walks.
"""
import itertools

import numpy as np

from mla_tree_verify_absorbed_gb300 import draft_inputs as DI

F32 = np.float32


def _hand_draft():
    # depth 1: p = .6 / .4 (tokens 11, 12); depth 2: p = .7 / .3 (tokens 21, 22)
    tok = np.asarray([[11, 12], [21, 22]], dtype=np.int32)
    lp = np.log(np.asarray([[0.6, 0.4], [0.7, 0.3]])).astype(np.float32)
    return tok, lp


def pin_hand_example(dd):
    tok, lp = _hand_draft()
    # products: (0) .6, (0,0) .42, (1) .4, (1,0) .28, (0,1) .18, (1,1) .12
    parent, token, depth, score = dd.build_tree_one(5, tok, lp, 6)
    assert parent.tolist() == [-1, 0, 1, 0, 3, 1, 3], parent
    assert token.tolist() == [5, 11, 21, 12, 21, 22, 22], token
    assert depth.tolist() == [0, 1, 2, 1, 2, 2, 2], depth
    want = [1.0, 0.6, 0.42, 0.4, 0.28, 0.18, 0.12]
    assert np.allclose(np.exp(score.astype(np.float64)), want, rtol=1e-6), score
    parent3, token3, _, _ = dd.build_tree_one(5, tok, lp, 3)
    assert parent3.tolist() == [-1, 0, 1, 0] and token3.tolist() == [5, 11, 21, 12]


def pin_hand_ties(dd):
    # every probability 1 (log 0): all nodes tie, so rank sequences decide:
    # (0), (0,0), (0,1), (1), (1,0), (1,1) -- prefix first, then lexicographic
    tok = np.asarray([[1, 2], [3, 4]], dtype=np.int32)
    lp = np.zeros((2, 2), dtype=np.float32)
    parent, token, depth, _ = dd.build_tree_one(0, tok, lp, 6)
    assert parent.tolist() == [-1, 0, 1, 1, 0, 4, 4], parent
    assert token.tolist() == [0, 1, 3, 4, 2, 3, 4], token
    assert depth.tolist() == [0, 1, 2, 2, 1, 2, 2]


def _brute(root, tok, lp, budget):
    L, K = lp.shape
    nodes = []
    for d in range(1, L + 1):
        for r in itertools.product(range(K), repeat=d):
            s = F32(0.0)
            for i, k in enumerate(r):
                s = F32(s + lp[i, k])
            nodes.append((s, r))
    nodes.sort(key=lambda n: (-float(n[0]), n[1]))
    chosen = nodes[:budget]
    index = {(): 0}
    for i, (_, r) in enumerate(chosen):
        index[r] = i + 1
    parent = [-1] + [index[r[:-1]] for _, r in chosen]
    token = [root] + [int(tok[len(r) - 1, r[-1]]) for _, r in chosen]
    depth = [0] + [len(r) for _, r in chosen]
    score = [F32(0.0)] + [s for s, _ in chosen]
    return parent, token, depth, score


def pin_brute_force(dd):
    cases = [(3, 3, "softmax", 1), (4, 2, "softmax", 2), (3, 3, "ties", 3), (2, 4, "zeros", 4),
             (4, 3, "zeros", 5), (5, 2, "ties", 6)]
    for L, K, mode, seed in cases:
        d = DI.make_draft(name="pin", B=3, L=L, K=K, budget=1, seed=seed, mode=mode)
        total = dd.node_count(L, K)
        for b in range(d.B):
            for budget in sorted({1, 2, 5, min(total, 17), min(total, 63)}):
                got = dd.build_tree_one(d.root_token[b], d.cand_token[b], d.cand_logp[b], budget)
                want = _brute(int(d.root_token[b]), d.cand_token[b], d.cand_logp[b], budget)
                assert got[0].tolist() == want[0], (L, K, mode, budget)
                assert got[1].tolist() == want[1]
                assert got[2].tolist() == want[2]
                assert [float(x) for x in got[3]] == [float(x) for x in want[3]]


def pin_chain(dd):
    # one candidate per depth: the tree is the chain of the drafted block
    d = DI.make_draft(name="pin", B=2, L=16, K=1, budget=1, seed=7)
    for b in range(d.B):
        for budget in (1, 9, 16):
            parent, token, depth, _ = dd.build_tree_one(d.root_token[b], d.cand_token[b], d.cand_logp[b], budget)
            assert parent.tolist() == list(range(-1, budget))
            assert token.tolist() == [int(d.root_token[b])] + d.cand_token[b, :budget, 0].tolist()
            assert depth.tolist() == list(range(budget + 1))


def pin_single_depth(dd):
    # one depth: the root's children, best first (candidates are sorted already)
    d = DI.make_draft(name="pin", B=2, L=1, K=16, budget=1, seed=8)
    for b in range(d.B):
        parent, token, _, score = dd.build_tree_one(d.root_token[b], d.cand_token[b], d.cand_logp[b], 16)
        assert parent.tolist() == [-1] + [0] * 16
        assert token.tolist() == [int(d.root_token[b])] + d.cand_token[b, 0].tolist()
        assert [float(x) for x in score[1:]] == [float(x) for x in d.cand_logp[b, 0]]


def pin_tree_invariants(dd):
    d = DI.make_draft(name="pin", B=4, L=16, K=8, budget=63, seed=9)
    parent, token, depth, score = dd.build_tree(d.root_token, d.cand_token, d.cand_logp, 63)
    for b in range(d.B):
        assert parent[b, 0] == -1 and depth[b, 0] == 0 and score[b, 0] == 0
        for i in range(1, 64):
            p = parent[b, i]
            assert 0 <= p < i and depth[b, i] == depth[b, p] + 1
            # the score is the parent's plus the log-probability of the node's own candidate
            k = int(np.nonzero(d.cand_token[b, depth[b, i] - 1] == token[b, i])[0][0])
            assert score[b, i] == F32(score[b, p] + d.cand_logp[b, depth[b, i] - 1, k])
            assert score[b, i] <= score[b, i - 1] or i == 1
        for i in range(64):  # siblings carry distinct tokens
            kids = [token[b, j] for j in range(64) if parent[b, j] == i]
            assert len(kids) == len(set(kids))


def pin_rejects_bad_drafts(dd):
    tok, lp = _hand_draft()
    for bad in (np.asarray([[np.nan, -1.0], [-0.1, -0.2]]), np.asarray([[0.1, -1.0], [-0.1, -0.2]]),
                np.asarray([[-1.0, -0.5], [-0.1, -0.2]])):
        try:
            dd.build_tree_one(0, tok, bad.astype(np.float32), 2)
        except ValueError:
            continue
        raise AssertionError("bad draft accepted")
    try:
        dd.build_tree_one(0, tok, lp, 7)  # only 6 draft nodes exist
    except ValueError:
        return
    raise AssertionError("budget above the node count accepted")


def pin_accept_hand(dd):
    tok, lp = _hand_draft()
    parent, token, _, _ = dd.build_tree_one(5, tok, lp, 6)
    # tree: 0 root; 1 (11) <- 0; 2 (21) <- 1; 3 (12) <- 0; 4 (21) <- 3; 5 (22) <- 1; 6 (22) <- 3
    tgt = np.asarray([11, 22, 7, 21, 8, 99, 9], dtype=np.int32)
    path, bonus, _ = dd.accept_one(parent, token, tgt)
    assert path == [0, 1, 5] and bonus == 99
    tgt2 = np.asarray([12, 0, 0, 21, 42, 0, 0], dtype=np.int32)
    path, bonus, _ = dd.accept_one(parent, token, tgt2)
    assert path == [0, 3, 4] and bonus == 42
    tgt3 = np.asarray([13, 21, 0, 0, 0, 0, 0], dtype=np.int32)
    path, bonus, slots = dd.accept_one(parent, token, tgt3, node_slot=np.arange(100, 107))
    assert path == [0] and bonus == 13 and slots == [100]


def pin_accept_matches_flags(dd):
    # a node is accepted iff its parent is and its token is the target's choice
    # at the parent; with distinct sibling tokens the accepted nodes form a path
    d = DI.make_draft(name="pin", B=24, L=16, K=8, budget=63, seed=10)
    parent, token, _, _ = dd.build_tree(d.root_token, d.cand_token, d.cand_logp, 63)
    lens = []
    for p_follow in (0.0, 0.5, 0.9, 1.0):
        tgt = DI.make_targets(d, parent, seed=11, p_follow=p_follow)
        slots = DI.make_node_slots(d.B, 64, seed=12)
        n_len, nodes, nxt, acc_slots = dd.accept(parent, token, tgt, slots)
        for b in range(d.B):
            ok = [True] + [False] * 63
            for i in range(1, 64):
                ok[i] = ok[parent[b, i]] and token[b, i] == tgt[b, parent[b, i]]
            want = [i for i in range(64) if ok[i]]
            assert sorted(nodes[b, :n_len[b]].tolist()) == want
            assert (nodes[b, n_len[b]:] == -1).all()
            last = nodes[b, n_len[b] - 1]
            assert nxt[b] == tgt[b, last]
            assert acc_slots[b, :n_len[b]].tolist() == [int(slots[b, j]) for j in nodes[b, :n_len[b]]]
            lens.append(int(n_len[b]))
    assert max(lens) >= 4 and min(lens) == 1  # the cases walk somewhere


def pin_accept_chain(dd):
    # a chain whose every token is the target's choice is accepted whole
    Q = 17
    parent = np.arange(-1, Q - 1, dtype=np.int32)
    token = np.arange(100, 100 + Q, dtype=np.int32)
    tgt = np.append(token[1:], 555).astype(np.int32)
    path, bonus, _ = dd.accept_one(parent, token, tgt)
    assert path == list(range(Q)) and bonus == 555
    tgt[7] = -1
    path, bonus, _ = dd.accept_one(parent, token, tgt)
    assert path == list(range(8)) and bonus == -1


def pin_accept_rejects_bad_trees(dd):
    for tp in ([0, 0], [-1, 1], [-1, 0, -1]):
        try:
            dd.accept_one(np.asarray(tp), np.zeros(len(tp)), np.zeros(len(tp)))
        except ValueError:
            continue
        raise AssertionError(f"bad tree accepted: {tp}")


ALL_PINS = [pin_hand_example, pin_hand_ties, pin_brute_force, pin_chain, pin_single_depth,
            pin_tree_invariants, pin_rejects_bad_drafts, pin_accept_hand, pin_accept_matches_flags,
            pin_accept_chain, pin_accept_rejects_bad_trees]
