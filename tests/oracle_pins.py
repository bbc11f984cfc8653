"""Pins that tie the CPU oracle to facts other than itself.

Each ``pin_*`` takes an ``oracle.Oracle`` handle and raises AssertionError (or
ValueError) when the oracle disagrees with:

* the absorb identity: non-absorbed MLA with random per-head W_UK / W_UV
  ("Ground Truth in Silicon ...", section "Input Knowledge Required ...",
  item 2: the absorbed form pre-computes the query's contribution);
* plain causal attention, which a chain-shaped draft tree must reduce to;
* a dense masked-softmax implementation whose mask comes from walking parent
  pointers, with lse from scipy's logsumexp;
* closed forms (equal value rows, zero queries, a lone visible token);
* invariance under a permutation of the pool's slots;
* hand-worked tables (tests/golden/tiny_tree_anc.txt, a small page table);
* exact widening of bf16 inputs.

They are plain functions so that tests/test_oracle_mutations.py can run them
against copies of the oracle with a planted mistake.
"""
from __future__ import annotations

import os

import numpy as np
from scipy.special import logsumexp

from mla_tree_verify_absorbed_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------------------
# helpers (independent of the oracle)
# ----------------------------------------------------------------------------
def ancestors_by_walk(parent) -> list:
    """Set of ancestor-or-self node ids per node, by following parent links."""
    out = []
    for i in range(len(parent)):
        s, j = set(), i
        while j >= 0:
            s.add(j)
            j = int(parent[j])
        out.append(s)
    return out


def visible_positions(p: I.Problem, b: int, i: int) -> list:
    P = int(p.prefix_lens[b])
    anc = ancestors_by_walk(p.tree_parent[b])[i]
    return list(range(P)) + [P + t for t in sorted(anc)]


def widened(p: I.Problem):
    """q_lat, q_pe, kv_c, k_pe as float64 arrays."""
    def f(x):
        if p.dtype == "bf16":
            return I.bf16_bits_to_f32(x).astype(np.float64)
        return np.asarray(x, dtype=np.float64)
    pool = f(p.pool)
    return f(p.q_lat), f(p.q_pe), pool[:, :I.DL], pool[:, I.DL:]


def f64_problem(seed, B=2, Q=5, H=3, prefix=(7, 4), trees=None, layout="scattered",
                pool_slots=None, page_size=1, n_pages=None):
    kw = dict(name="pin", dtype="fp64", B=B, H=H, Q=Q, prefix_lens=list(prefix), seed=seed,
              trees=trees, layout=layout, page_size=page_size)
    if layout == "paged":
        kw["n_pages"] = n_pages
    elif pool_slots is not None:
        kw["pool_slots"] = pool_slots
    return I.make_problem(**kw)


# ----------------------------------------------------------------------------
# pins
# ----------------------------------------------------------------------------
def pin_tree_anc_golden(orc):
    rows = []
    with open(os.path.join(GOLDEN, "tiny_tree_anc.txt")) as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                node, mask, vis = line.split()
                rows.append((int(node), int(mask, 16), int(vis)))
    tree = np.asarray([I.TINY_TREE], dtype=np.int32)
    anc = orc.tree_anc(tree)[0]
    for node, mask, _ in rows:
        assert int(anc[node]) == mask, (node, hex(int(anc[node])), hex(mask))
    # visible counts through the full attention call
    p = I.make_config("tiny")
    r = np.asarray([(0, n, 0) for n, _, _ in rows], dtype=np.int32)
    _, _, nvis = orc.verify_rows(p, r)
    assert [int(x) for x in nvis] == [v for _, _, v in rows], nvis


def pin_tree_anc_walk(orc):
    rng = np.random.default_rng(11)
    trees = np.stack([I.random_tree(rng, 64, depth_cap=d) for d in (1, 2, 8, 64)])
    anc = orc.tree_anc(trees)
    for b in range(trees.shape[0]):
        walk = ancestors_by_walk(trees[b])
        for i in range(64):
            want = sum(1 << t for t in walk[i])
            assert int(anc[b, i]) == want, (b, i)


def pin_slots_paged_hand(orc):
    # page_size 4; sequence 0 has 6+1 positions on pages [2, 0]; sequence 1 has
    # 2+1 positions on page [1].  Worked by hand: page k holds slots 4k..4k+3.
    p = f64_problem(0, B=2, Q=1, H=1, prefix=(6, 2), trees=[[-1], [-1]], layout="paged",
                    page_size=4, n_pages=3)
    p.block_table = np.asarray([[2, 0], [1, -1]], dtype=np.int32)
    got = orc.resolve_slots(p)
    assert list(got) == [8, 9, 10, 11, 0, 1, 2, 4, 5, 6], list(got)


def pin_slots_tables(orc):
    # page_size=1: the slot list is the index table itself, sequence by sequence.
    p = f64_problem(1, B=3, Q=4, H=1, prefix=(5, 0, 9), layout="scattered", pool_slots=64)
    assert np.array_equal(orc.resolve_slots(p), p.kv_indices)
    # paged: each sequence's slots are its pages' slot ranges laid end to end,
    # and no two sequences share a slot.
    p = f64_problem(2, B=3, Q=3, H=1, prefix=(13, 1, 30), layout="paged", page_size=8,
                    n_pages=12)
    got = orc.resolve_slots(p)
    k = 0
    for b in range(p.B):
        n = int(p.kv_lens[b])
        pages = [int(x) for x in p.block_table[b] if x >= 0]
        want = np.concatenate([np.arange(pg * 8, pg * 8 + 8) for pg in pages])[:n]
        assert np.array_equal(got[k:k + n], want), b
        k += n
    assert len(set(got.tolist())) == len(got)


def pin_absorb_identity(orc):
    """Absorbed attention == non-absorbed MLA with per-head projections."""
    rng = np.random.default_rng(5)
    p = f64_problem(3, B=2, Q=6, H=3, prefix=(9, 3), layout="scattered", pool_slots=40)
    dn = 128
    w_uk = rng.standard_normal((p.H, I.DL, dn)) / np.sqrt(I.DL)
    w_uv = rng.standard_normal((p.H, I.DL, dn)) / np.sqrt(I.DL)
    q_nope = rng.standard_normal((p.B, p.Q, p.H, dn))
    # the absorbed query q_lat_h = W_UK_h q_nope_h
    p.q_lat = np.einsum("hdn,bqhn->bqhd", w_uk, q_nope)
    rows = I.all_rows(p)
    out, lse, _ = orc.verify_rows(p, rows)
    _, q_pe, kv_c, k_pe = widened(p)
    for r, (b, i, h) in enumerate(rows):
        pos = visible_positions(p, b, i)
        slots = [p.slot_of(b, x) for x in pos]
        keys = np.concatenate([kv_c[slots] @ w_uk[h], k_pe[slots]], axis=1)   # [n, 128+64]
        vals = kv_c[slots] @ w_uv[h]                                         # [n, 128]
        q = np.concatenate([q_nope[b, i, h], q_pe[b, i, h]])
        s = p.scale * (keys @ q)
        w = np.exp(s - s.max())
        w /= w.sum()
        o_head = w @ vals
        np.testing.assert_allclose(w_uv[h].T @ out[r], o_head, rtol=1e-10, atol=1e-12)
        assert abs(lse[r] - logsumexp(s)) < 1e-10


def pin_chain_is_causal(orc):
    """A chain-shaped tree makes the verify step plain causal attention."""
    Q, P = 7, 10
    p = f64_problem(4, B=1, Q=Q, H=2, prefix=(P,), trees=[list(range(-1, Q - 1))],
                    layout="scattered", pool_slots=30)
    rows = I.all_rows(p)
    out, lse, _ = orc.verify_rows(p, rows)
    q_lat, q_pe, kv_c, k_pe = widened(p)
    N = P + Q
    slots = [p.slot_of(0, x) for x in range(N)]
    K = np.concatenate([kv_c[slots], k_pe[slots]], axis=1)       # keys by position
    V = kv_c[slots]
    for r, (b, i, h) in enumerate(rows):
        qpos = P + i                                             # query's own position
        q = np.concatenate([q_lat[b, i, h], q_pe[b, i, h]])
        s = p.scale * (K @ q)
        s[qpos + 1:] = -np.inf                                   # causal: nothing after itself
        w = np.exp(s - s.max())
        w /= w.sum()
        np.testing.assert_allclose(out[r], w @ V, rtol=1e-11, atol=1e-13)
        assert abs(lse[r] - logsumexp(s)) < 1e-11


def pin_dense_bruteforce(orc):
    """Dense [rows x N] masked softmax on a random tree, several layouts."""
    cases = [
        f64_problem(6, B=2, Q=9, H=2, prefix=(12, 0), layout="scattered", pool_slots=50),
        f64_problem(7, B=3, Q=5, H=1, prefix=(3, 17, 1), layout="paged", page_size=4,
                    n_pages=16),
        f64_problem(8, B=1, Q=64, H=1, prefix=(5,), layout="contiguous"),
    ]
    for p in cases:
        rows = I.all_rows(p)
        out, lse, nvis = orc.verify_rows(p, rows)
        q_lat, q_pe, kv_c, k_pe = widened(p)
        for b in range(p.B):
            N = int(p.kv_lens[b])
            slots = [p.slot_of(b, x) for x in range(N)]
            K = np.concatenate([kv_c[slots], k_pe[slots]], axis=1)
            Qm = np.concatenate([q_lat[b], q_pe[b]], axis=-1).reshape(p.Q * p.H, -1)
            S = p.scale * (Qm @ K.T)                              # [Q*H, N]
            mask = np.zeros((p.Q, N), dtype=bool)
            P = int(p.prefix_lens[b])
            walk = ancestors_by_walk(p.tree_parent[b])
            for i in range(p.Q):
                mask[i, :P] = True
                for t in walk[i]:
                    mask[i, P + t] = True
            mask = np.repeat(mask, p.H, axis=0)
            S = np.where(mask, S, -np.inf)
            L = logsumexp(S, axis=1)
            W = np.exp(S - L[:, None])
            O = W @ kv_c[slots]
            sel = rows[:, 0] == b
            np.testing.assert_allclose(out[sel], O, rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(lse[sel], L, rtol=1e-12, atol=1e-12)
            assert np.array_equal(nvis[sel], mask.sum(axis=1))


def pin_permutation_invariance(orc):
    p = f64_problem(9, B=2, Q=6, H=2, prefix=(11, 4), layout="scattered", pool_slots=64)
    rows = I.all_rows(p)
    out0, lse0, _ = orc.verify_rows(p, rows)
    perm = np.random.default_rng(3).permutation(p.pool_slots)   # new slot of old slot s
    pool = np.empty_like(p.pool)
    pool[perm] = p.pool
    p.pool = pool
    p.kv_indices = perm[p.kv_indices].astype(np.int32)
    out1, lse1, _ = orc.verify_rows(p, rows)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def pin_closed_forms(orc):
    # (a) every kv_c row equal to v: the output is v whatever the weights.
    p = f64_problem(10, B=2, Q=4, H=2, prefix=(6, 2), layout="scattered", pool_slots=20)
    v = np.random.default_rng(1).standard_normal(I.DL)
    p.pool[:, :I.DL] = v
    out, _, _ = orc.verify_rows(p, I.all_rows(p))
    np.testing.assert_allclose(out, np.broadcast_to(v, out.shape), rtol=1e-13, atol=1e-13)

    # (b) zero queries: uniform weights, out = mean of visible rows, lse = ln |V|.
    p = f64_problem(11, B=2, Q=5, H=1, prefix=(8, 0), layout="scattered", pool_slots=20)
    p.q_lat[:] = 0.0
    p.q_pe[:] = 0.0
    rows = I.all_rows(p)
    out, lse, nvis = orc.verify_rows(p, rows)
    _, _, kv_c, _ = widened(p)
    for r, (b, i, h) in enumerate(rows):
        pos = visible_positions(p, b, i)
        mean = kv_c[[p.slot_of(b, x) for x in pos]].mean(axis=0)
        np.testing.assert_allclose(out[r], mean, rtol=1e-13, atol=1e-14)
        assert abs(lse[r] - np.log(len(pos))) < 1e-14 and nvis[r] == len(pos)

    # (c) empty prefix and a root node: only the node itself is visible, so
    #     out = its own kv_c row and lse = its own score, here scale * a * c.
    p = f64_problem(12, B=1, Q=3, H=1, prefix=(0,), trees=[[-1, -1, 0]], layout="scattered",
                    pool_slots=8)
    a, c, e = 1.5, -2.25, 0.75
    p.q_lat[0, 1, 0, :] = 0.0
    p.q_lat[0, 1, 0, 3] = a
    p.q_pe[0, 1, 0, :] = 0.0
    p.q_pe[0, 1, 0, 7] = e
    s1 = p.slot_of(0, 1)
    p.pool[s1, :] = 0.0
    p.pool[s1, 3] = c
    p.pool[s1, I.DL + 7] = 2.0
    out, lse, nvis = orc.verify_rows(p, np.asarray([[0, 1, 0]], dtype=np.int32))
    assert nvis[0] == 1
    assert np.array_equal(out[0], p.pool[s1, :I.DL])
    assert abs(lse[0] - p.scale * (a * c + e * 2.0)) < 1e-15


def pin_bf16_widening(orc):
    """bf16 inputs read exactly as the float64 values they encode."""
    p = I.make_problem(name="w", dtype="bf16", B=1, H=2, Q=3, prefix_lens=[9], seed=13,
                       layout="scattered", pool_slots=16)
    rows = I.all_rows(p)
    out_b, lse_b, _ = orc.verify_rows(p, rows)
    q_lat, q_pe, kv_c, k_pe = widened(p)
    p.dtype = "fp64"
    p.q_lat, p.q_pe = q_lat, q_pe
    p.pool = np.concatenate([kv_c, k_pe], axis=1)
    out_d, lse_d, _ = orc.verify_rows(p, rows)
    assert np.array_equal(out_b, out_d) and np.array_equal(lse_b, lse_d)
    # and the widening itself: a few bit patterns with known values
    probe = np.asarray([0x3F80, 0xC000, 0x3E80, 0x0000, 0x7F7F], dtype=np.uint16)
    want = [1.0, -2.0, 0.25, 0.0, 3.3895313892515355e38]
    p2 = I.make_problem(name="w2", dtype="bf16", B=1, H=1, Q=1, prefix_lens=[0], seed=1,
                        layout="contiguous")
    for bits, val in zip(probe, want):
        p2.q_lat[:] = 0
        p2.q_pe[:] = 0
        p2.pool[:] = 0
        p2.pool[0, 0] = bits
        out, lse, _ = orc.verify_rows(p2, np.asarray([[0, 0, 0]], dtype=np.int32))
        assert out[0, 0] == val and lse[0] == 0.0, (hex(int(bits)), out[0, 0])


ALL_PINS = [
    pin_tree_anc_golden, pin_tree_anc_walk, pin_slots_paged_hand, pin_slots_tables,
    pin_absorb_identity, pin_chain_is_causal, pin_dense_bruteforce,
    pin_permutation_invariance, pin_closed_forms, pin_bf16_widening,
]
