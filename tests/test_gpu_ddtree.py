"""DDTree construction and greedy acceptance through the C ABI (needs a GPU).

Every output is compared bit for bit with the oracle on the same seeded
inputs: parents, tokens, depths, accepted paths and bonus tokens exactly, and
the float32 node scores bit-exactly (both sides add the same float32
log-probabilities in the same order, root first).
"""
import numpy as np
import pytest

from oracle import ddtree as dd
from mla_tree_verify_absorbed_gb300 import api
from mla_tree_verify_absorbed_gb300 import draft_inputs as DI

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MLA_DEVERR_PARENT = 0x8
MLA_DEVERR_DRAFT = 0x100


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.load()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def build_both(d):
    want = dd.build_tree(d.root_token, d.cand_token, d.cand_logp, d.budget)
    parent, token, depth, score, ws = api.ddtree_build(dev(d.root_token), dev(d.cand_token), dev(d.cand_logp),
                                                       d.budget)
    assert api.check(ws) == 0
    got = tuple(t.cpu().numpy() for t in (parent, token, depth, score))
    return got, want


def assert_same_tree(got, want):
    for g, w, name in zip(got[:3], want[:3], ("parent", "token", "depth")):
        assert np.array_equal(g, w), name
    assert np.array_equal(got[3].view(np.uint32), want[3].view(np.uint32)), "score bits"


@pytest.mark.parametrize("name", sorted(DI.DRAFT_CONFIGS))
@pytest.mark.parametrize("mode", ["softmax", "ties", "zeros"])
def test_build_matches_oracle(name, mode):
    d = DI.make_draft_config(name, mode=mode)
    got, want = build_both(d)
    assert_same_tree(got, want)


@pytest.mark.parametrize("L,K,budget,mode", [
    (1, 16, 16, "softmax"),   # one depth: the root's children in rank order
    (16, 1, 16, "softmax"),   # one candidate per depth: a chain of the whole block
    (3, 3, 39, "softmax"),    # every draft node there is
    (2, 2, 6, "ties"),
    (16, 16, 63, "softmax"),  # widest lists, largest budget
    (16, 16, 63, "ties"),
    (5, 4, 1, "zeros"),       # a single draft node
    (7, 2, 63, "zeros"),
])
def test_build_edge_shapes(L, K, budget, mode):
    d = DI.make_draft(name="edge", B=37, L=L, K=K, budget=budget, seed=L * 100 + K, mode=mode)
    got, want = build_both(d)
    assert_same_tree(got, want)


def test_build_rejects_bad_drafts_per_sequence():
    d = DI.make_draft(name="bad", B=9, L=8, K=4, budget=20, seed=3)
    lp = d.cand_logp.copy()
    lp[1, 2, 1] = np.nan
    lp[4, 0, 0] = 0.25                  # a probability above 1
    lp[7, 5, 2] = lp[7, 5, 1] + 0.5     # not best first
    parent, token, depth, score, ws = api.ddtree_build(dev(d.root_token), dev(d.cand_token), dev(lp), d.budget)
    assert api.check(ws) == MLA_DEVERR_DRAFT
    good = [b for b in range(d.B) if b not in (1, 4, 7)]
    want = dd.build_tree(d.root_token[good], d.cand_token[good], lp[good], d.budget)
    got = tuple(t.cpu().numpy() for t in (parent, token, depth, score))
    assert_same_tree(tuple(g[good] for g in got), want)
    for b in (1, 4, 7):  # untouched
        assert (got[0][b] == -7).all() and (got[1][b] == -7).all() and np.isnan(got[3][b]).all()


def test_build_then_verify_format():
    # the built tree is a valid tree_parent table for the verify call (Q = budget + 1)
    d = DI.make_draft_config("tree_b256")
    got, _ = build_both(d)
    parent = got[0]
    assert parent.shape[1] == 64 and (parent[:, 0] == -1).all()
    idx = np.arange(64)[None, :]
    assert ((parent[:, 1:] >= 0) & (parent[:, 1:] < idx[:, 1:])).all()


@pytest.mark.parametrize("p_follow", [0.0, 0.6, 0.9, 1.0])
def test_accept_matches_oracle_on_built_trees(p_follow):
    d = DI.make_draft_config("tree_b256")
    parent, token, _, _ = dd.build_tree(d.root_token, d.cand_token, d.cand_logp, d.budget)
    tgt = DI.make_targets(d, parent, seed=31, p_follow=p_follow)
    slots = DI.make_node_slots(d.B, d.Q, seed=32)
    want = dd.accept(parent, token, tgt, slots)
    n_len, nodes, nxt, acc_slots, ws = api.ddtree_accept(dev(parent), dev(token), dev(tgt), dev(slots))
    assert api.check(ws) == 0
    assert np.array_equal(n_len.cpu().numpy(), want[0])
    assert np.array_equal(nodes.cpu().numpy(), want[1])
    assert np.array_equal(nxt.cpu().numpy(), want[2])
    assert np.array_equal(acc_slots.cpu().numpy(), want[3])


@pytest.mark.parametrize("Q", [1, 2, 31, 32, 33, 63, 64])
def test_accept_random_trees_with_equal_sibling_tokens(Q):
    # tokens from 3 ids: equal siblings are common and the lowest index must win
    tp, tt = DI.random_rooted_tree(B=300, Q=Q, seed=40 + Q, vocab=3)
    rng = np.random.default_rng(50 + Q)
    tgt = rng.integers(0, 3, size=(300, Q)).astype(np.int32)
    want = dd.accept(tp, tt, tgt)
    n_len, nodes, nxt, acc_slots, ws = api.ddtree_accept(dev(tp), dev(tt), dev(tgt))
    assert api.check(ws) == 0 and acc_slots is None
    assert np.array_equal(n_len.cpu().numpy(), want[0])
    assert np.array_equal(nodes.cpu().numpy(), want[1])
    assert np.array_equal(nxt.cpu().numpy(), want[2])
    if Q > 8:
        assert want[0].max() >= 4


def test_accept_rejects_bad_trees_per_sequence():
    tp, tt = DI.random_rooted_tree(B=6, Q=20, seed=60)
    tgt = np.zeros_like(tt)
    tp[2, 0] = 0       # node 0 not a root
    tp[4, 9] = 9       # a node its own parent
    tp[5, 13] = -1     # a second root
    n_len, nodes, nxt, _, ws = api.ddtree_accept(dev(tp), dev(tt), dev(tgt))
    assert api.check(ws) == MLA_DEVERR_PARENT
    got_len = n_len.cpu().numpy()
    good = [0, 1, 3]
    want = dd.accept(tp[good], tt[good], tgt[good])
    assert np.array_equal(got_len[good], want[0])
    assert np.array_equal(nodes.cpu().numpy()[good], want[1])
    assert (got_len[[2, 4, 5]] == -7).all() and (nodes.cpu().numpy()[[2, 4, 5]] == -7).all()


def test_build_accept_chain_on_device_and_in_a_graph():
    # build -> accept on one stream with no host step between, then the same
    # two calls captured in a CUDA graph and replayed on new inputs
    d = DI.make_draft_config("tree_b256")
    parent_o, token_o, _, _ = dd.build_tree(d.root_token, d.cand_token, d.cand_logp, d.budget)
    tgt = DI.make_targets(d, parent_o, seed=71, p_follow=0.9)
    want = dd.accept(parent_o, token_o, tgt)
    root, ctok, clp, dtgt = dev(d.root_token), dev(d.cand_token), dev(d.cand_logp), dev(tgt)
    B, Q = d.B, d.Q
    i32 = dict(dtype=torch.int32, device="cuda")
    parent, token = torch.empty((B, Q), **i32), torch.empty((B, Q), **i32)
    n_len, nodes, nxt = torch.empty((B,), **i32), torch.empty((B, Q), **i32), torch.empty((B,), **i32)
    ws_b = api.alloc_workspace(api.DDTREE_WORKSPACE_BYTES)
    ws_a = api.alloc_workspace(api.DDTREE_WORKSPACE_BYTES)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        api.ddtree_build_into(root, ctok, clp, d.budget, parent, token, ws_b, stream=s)
        api.ddtree_accept_into(parent, token, dtgt, n_len, nodes, nxt, ws_a, stream=s)
    s.synchronize()
    assert np.array_equal(n_len.cpu().numpy(), want[0]) and np.array_equal(nodes.cpu().numpy(), want[1])
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        api.ddtree_build_into(root, ctok, clp, d.budget, parent, token, ws_b, stream=s)
        api.ddtree_accept_into(parent, token, dtgt, n_len, nodes, nxt, ws_a, stream=s)
    d2 = DI.make_draft_config("tree_b256", seed=99)
    p2, t2, _, _ = dd.build_tree(d2.root_token, d2.cand_token, d2.cand_logp, d2.budget)
    tgt2 = DI.make_targets(d2, p2, seed=72, p_follow=0.9)
    want2 = dd.accept(p2, t2, tgt2)
    root.copy_(dev(d2.root_token))
    ctok.copy_(dev(d2.cand_token))
    clp.copy_(dev(d2.cand_logp))
    dtgt.copy_(dev(tgt2))
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(parent.cpu().numpy(), p2) and np.array_equal(token.cpu().numpy(), t2)
    assert np.array_equal(n_len.cpu().numpy(), want2[0]) and np.array_equal(nodes.cpu().numpy(), want2[1])
    assert np.array_equal(nxt.cpu().numpy(), want2[2])
    assert api.check(ws_b) == 0 and api.check(ws_a) == 0
