"""CUDA path against the CPU oracle, through the C ABI (needs a GPU)."""
import numpy as np
import pytest

import oracle
from mla_tree_verify_absorbed_gb300 import api
from mla_tree_verify_absorbed_gb300 import inputs as I
from tests import parity as PT

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ALGOS_BF16 = ["simt", "tc"]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.load()


def run(p, algo="auto", num_splits=0, separate_pools=False, **kw):
    di = api.device_inputs(p, separate_pools=separate_pools)
    out, lse = api.verify_attn(di, num_splits=num_splits, algo=algo, **kw)
    torch.cuda.synchronize()
    return di, out, lse


# ---------------------------------------------------------------------------
# a1 / a2: tree masks and slot resolution, bit-exact
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", I.CONFIG_NAMES)
def test_meta_bitexact(name):
    p = PT.workload(name)
    di = api.device_inputs(p)
    anc, slots, ws = api.build_meta(di)
    assert api.check(ws) == 0
    want_anc = oracle.get().tree_anc(p.tree_parent)
    got_anc = anc.cpu().numpy().view(np.uint64)
    assert np.array_equal(got_anc, want_anc)
    want_slots = oracle.get().resolve_slots(p)
    assert np.array_equal(slots.cpu().numpy(), want_slots)


# ---------------------------------------------------------------------------
# small problems: every output element against the oracle
# ---------------------------------------------------------------------------
def mid_problem(seed=21, layout="scattered"):
    kw = dict(name="mid", dtype="bf16", B=2, H=64, Q=16, prefix_lens=[300, 777], seed=seed)
    if layout == "paged":
        kw.update(layout="paged", page_size=64, n_pages=40)
    else:
        kw.update(layout="scattered", pool_slots=2048)
    return I.make_problem(**kw)


def ragged_problem():
    # rows = 5 heads x 7 nodes = 35 (not a multiple of any row group), tiny and
    # empty prefixes, paged with page_size 16
    return I.make_problem(name="ragged", dtype="bf16", B=3, H=5, Q=7, prefix_lens=[0, 1, 130],
                          seed=22, layout="paged", page_size=16, n_pages=20)


def check_all_rows(p, out, lse, what):
    rows = I.all_rows(p)
    ro, rl = PT.oracle_rows(p, rows)
    go, gl = PT.gather_rows(out, lse, rows)
    PT.assert_close(go, ro, p.dtype, what + " out")
    PT.assert_close(gl, rl, p.dtype, what + " lse")


def test_tiny_fp32():
    p = PT.workload("tiny")
    _, out, lse = run(p)
    check_all_rows(p, out, lse, "tiny")


@pytest.mark.parametrize("algo", ALGOS_BF16)
@pytest.mark.parametrize("maker", [mid_problem, ragged_problem,
                                   lambda: mid_problem(23, "paged")],
                         ids=["mid_scattered", "ragged_paged", "mid_paged"])
def test_full_rows_bf16(algo, maker):
    p = maker()
    _, out, lse = run(p, algo=algo)
    check_all_rows(p, out, lse, f"{p.name}/{algo}")


def test_tiny_fp32_via_simt_bf16_shape():
    # the same tiny tree through the bf16 cache and both kernel families
    p = I.make_problem(name="tiny_bf16", dtype="bf16", B=1, H=16, Q=8, prefix_lens=[256], seed=0,
                       trees=[I.TINY_TREE])
    for algo in ALGOS_BF16:
        _, out, lse = run(p, algo=algo)
        check_all_rows(p, out, lse, f"tiny_bf16/{algo}")


def ragged_batch_problem(seed=28):
    # four sequences of very different lengths (1 to 40 tiles): chunks of
    # one split count differ in size between sequences, some are empty
    return I.make_problem(name="ragged_batch", dtype="bf16", B=4, H=64, Q=16, prefix_lens=[2500, 0, 700, 33],
                          seed=seed, layout="scattered", pool_slots=4096)


@pytest.mark.parametrize("algo", ALGOS_BF16)
@pytest.mark.parametrize("maker", [mid_problem, ragged_batch_problem], ids=["mid", "ragged_batch"])
def test_split_invariance(algo, maker):
    p = maker(24)
    rows = I.all_rows(p)
    ro, rl = PT.oracle_rows(p, rows)
    results = []
    # 20 and 40 chunks: more chunks than most sequences have tiles (empty
    # chunks), the combine's four-warps-per-row form, and (40) more than 32
    # pieces per row
    for ns in (1, 2, 7, 20, 40, 0):
        _, out, lse = run(p, algo=algo, num_splits=ns)
        go, gl = PT.gather_rows(out, lse, rows)
        PT.assert_close(go, ro, "bf16", f"splits={ns} out")
        PT.assert_close(gl, rl, "bf16", f"splits={ns} lse")
        results.append((go, gl))
    for go, gl in results[1:]:
        # pieces only change fp32 summation order: a couple of bf16 ulps at most
        assert np.abs(go - results[0][0]).max() <= 2e-2 * np.abs(results[0][0]).max()
        assert np.abs(gl - results[0][1]).max() <= 1e-4 * np.abs(results[0][1]).max() + 1e-5


@pytest.mark.parametrize("num_splits", [9, 7, 0])
def test_one_sequence_with_empty_leading_chunks(num_splits):
    # one sequence of 5 tiles (16 row groups): cut 9 ways, chunk 0 is empty,
    # so a cluster's first real work item is not the row group whose queries
    # it staged while the metadata kernel ran -- it must stage them again
    p = I.make_problem(name="one_seq_short", dtype="bf16", B=1, H=64, Q=64, prefix_lens=[256], seed=29,
                       layout="scattered", pool_slots=1024)
    _, out, lse = run(p, algo="tc", num_splits=num_splits)
    check_all_rows(p, out, lse, f"one short sequence, splits={num_splits}")


@pytest.mark.parametrize("num_splits", [1, 2])
def test_output_16_byte_aligned_only(num_splits):
    # the API asks for 16-byte aligned outputs; the tensor-core kernel writes
    # whole 32-byte sectors only where the array allows them, so an output 16
    # bytes past a 32-byte boundary takes the narrow stores: same bytes
    p = mid_problem(27)
    di = api.device_inputs(p)
    ref_out, ref_lse = api.verify_attn(di, num_splits=num_splits, algo="tc")
    n = p.B * p.Q * p.H * 512
    buf = torch.empty(n + 8, dtype=torch.bfloat16, device="cuda")
    out = buf[8:].view(p.B, p.Q, p.H, 512)
    assert out.data_ptr() % 32 == 16
    out, lse = api.verify_attn(di, out=out, num_splits=num_splits, algo="tc")
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)
    assert torch.equal(lse, ref_lse)


@pytest.mark.parametrize("algo", ALGOS_BF16)
@pytest.mark.parametrize("page_size,H,Q,lens", [
    (8, 16, 13, [500, 9, 1200]),        # 208 rows: one ragged row group per sequence
    (32, 24, 5, [0, 700]),              # 120 rows, an empty prefix
    (128, 128, 1, [900, 2000, 31]),     # 128 heads, one node, pages wider than a tile
    (32, 16, 64, [300]),                # 1024 rows, a 64-node tree over a short prefix
], ids=["p8_H16_Q13", "p32_H24_Q5", "p128_H128_Q1", "p32_H16_Q64"])
def test_page_sizes_and_head_counts(algo, page_size, H, Q, lens):
    n_pages = sum(-(-(int(P) + Q) // page_size) for P in lens) + 3
    p = I.make_problem(name="pages_heads", dtype="bf16", B=len(lens), H=H, Q=Q, prefix_lens=lens, seed=30,
                       layout="paged", page_size=page_size, n_pages=n_pages)
    _, out, lse = run(p, algo=algo)
    check_all_rows(p, out, lse, f"page {page_size} H {H} Q {Q}")


@pytest.mark.parametrize("algo", ALGOS_BF16)
def test_padded_pool_rows(algo):
    # the cache rows inside a wider array: kv_c at columns [0, 512), k_pe at
    # [640, 704) of 704-element rows -- the gathers follow the row strides, so
    # the results are the packed pool's bytes, and the compaction copies the
    # same rows
    import dataclasses
    p = mid_problem(31)
    di = api.device_inputs(p)
    ref_out, ref_lse = api.verify_attn(di, algo=algo, num_splits=3)
    wide = torch.zeros((di.pool.shape[0], 704), dtype=di.pool.dtype, device=di.pool.device)
    wide[:, :512] = di.pool[:, :512]
    wide[:, 640:704] = di.pool[:, 512:576]
    dw = dataclasses.replace(di, kv_c=wide[:, :512], k_pe=wide[:, 640:704], pool=None)
    out, lse = api.verify_attn(dw, algo=algo, num_splits=3)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)
    assert torch.equal(lse, ref_lse)
    total = int(np.sum(np.asarray(p.prefix_lens, dtype=np.int64) + p.Q))
    d_ref = torch.empty((total, 576), dtype=di.pool.dtype, device=di.pool.device)
    d_wide = torch.empty_like(d_ref)
    api.kv_compact(di, d_ref)
    api.kv_compact(dw, d_wide)
    torch.cuda.synchronize()
    assert torch.equal(d_ref, d_wide)


@pytest.mark.parametrize("algo", ALGOS_BF16)
@pytest.mark.parametrize("scale", [1.0, 1e-3], ids=["sharp", "flat"])
def test_score_scales(algo, scale):
    # scale 1 puts the scores' spread near 24 (a row's weights move the lazy
    # running max tile after tile); scale 1e-3 makes the softmax nearly
    # uniform over up to ~800 tokens
    p = I.make_problem(name="scales", dtype="bf16", B=2, H=64, Q=16, prefix_lens=[300, 777], seed=32,
                       layout="scattered", pool_slots=2048, scale=scale)
    _, out, lse = run(p, algo=algo)
    check_all_rows(p, out, lse, f"scale {scale}")


@pytest.mark.parametrize("algo", ALGOS_BF16)
@pytest.mark.parametrize("num_splits", [1, 3, 0])
def test_lse_may_be_null(algo, num_splits):
    # lse is optional: with a NULL pointer the outputs are the same bytes
    import ctypes
    p = mid_problem(33)
    di = api.device_inputs(p)
    ref_out, _ = api.verify_attn(di, algo=algo, num_splits=num_splits)
    out = torch.empty_like(ref_out)
    a = api.make_args(di, out=out, lse=None, algo=algo)
    assert not a.lse
    lib = api.load()
    n = lib.mla_verify_workspace_size(ctypes.byref(a), num_splits)
    ws = api.alloc_workspace(n)
    st = lib.mla_verify_attn(ctypes.byref(a), ctypes.c_void_p(ws.data_ptr()), ctypes.c_size_t(n), num_splits,
                             api._stream(None))
    assert st == api.MLA_OK
    assert api.check(ws) == 0
    assert torch.equal(out, ref_out)


def test_two_streams_at_once():
    # calls on two streams with their own workspaces share no device state:
    # launched back to back without a synchronisation they give the bytes of
    # the same calls made one after the other
    probs = [mid_problem(34), ragged_batch_problem(35)]
    dis = [api.device_inputs(p) for p in probs]
    refs = [api.verify_attn(d, algo="tc") for d in dis]
    torch.cuda.synchronize()
    outs = [(torch.empty_like(o), torch.empty_like(l)) for o, l in refs]
    wss = [api.alloc_workspace(api.workspace_size(d, 0, algo="tc")) for d in dis]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s_ in streams:
        s_.wait_stream(torch.cuda.current_stream())
    for _ in range(3):
        for d, (o, l), w, s_ in zip(dis, outs, wss, streams):
            api.verify_attn(d, out=o, lse=l, workspace=w, algo="tc", stream=s_)
    torch.cuda.synchronize()
    for (o, l), (ro, rl), w in zip(outs, refs, wss):
        assert api.check(w) == 0
        assert torch.equal(o, ro) and torch.equal(l, rl)


@pytest.mark.parametrize("algo", ALGOS_BF16)
def test_needles(algo):
    p = mid_problem(25)
    I.plant_needles(p, seed=5)
    _, out, lse = run(p, algo=algo)
    rows = I.all_rows(p)
    ro, rl = PT.oracle_rows(p, rows)
    go, gl = PT.gather_rows(out, lse, rows)
    # the softmax is peaked: outputs are O(1), a wrong gather or mask moves them by O(1)
    assert np.abs(ro).max() > 1.0
    PT.assert_close(go, ro, "bf16", "needle out")
    PT.assert_close(gl, rl, "bf16", "needle lse")


@pytest.mark.parametrize("algo", ALGOS_BF16)
def test_separate_pools(algo):
    p = mid_problem(26)
    _, out, lse = run(p, algo=algo, separate_pools=True)
    check_all_rows(p, out, lse, "separate pools")


@pytest.mark.parametrize("algo", ALGOS_BF16)
def test_edge_trees(algo):
    # every node a root over an empty prefix: each row sees only itself
    p = I.make_problem(name="roots", dtype="bf16", B=2, H=4, Q=5, prefix_lens=[0, 0], seed=27,
                       trees=[[-1] * 5, [-1, 0, -1, 2, 3]])
    _, out, lse = run(p, algo=algo)
    check_all_rows(p, out, lse, "roots")
    # a 64-node chain: the last node's mask uses bit 63
    p = I.make_problem(name="chain64", dtype="bf16", B=1, H=2, Q=64, prefix_lens=[10], seed=28,
                       trees=[list(range(-1, 63))])
    _, out, lse = run(p, algo=algo)
    check_all_rows(p, out, lse, "chain64")
    # a single node, a single head
    p = I.make_problem(name="q1", dtype="bf16", B=3, H=1, Q=1, prefix_lens=[5, 0, 64], seed=29)
    _, out, lse = run(p, algo=algo)
    check_all_rows(p, out, lse, "q1")


# ---------------------------------------------------------------------------
# full-size workloads, in the launch configuration the benchmark times
# (num_splits = 0, default kernel family): sampled rows against the oracle
# ---------------------------------------------------------------------------
def test_lse_single_needle_c3():
    # one planted token that every row of the 200k-prefix workload sees: its
    # weight dominates every row's normaliser (score ~35 against ln Z ~14 for
    # the other 200k tokens), so a wrong gather of that one slot, or a wrong
    # scale on it, moves lse by several units -- far above the tolerance --
    # and the recorded margin shows how close the kernel really is
    p = I.make_config("c3")
    I.plant_needles(p, seed=7, n_prefix=1, strength=60.0)
    _, out, lse = run(p)
    rows = I.sample_rows(p, 2, seed=33)
    ro, rl = PT.oracle_rows(p, rows)
    go, gl = PT.gather_rows(out, lse, rows)
    assert rl.min() > 18.0, rl.min()  # the needle dominates every sampled row
    PT.assert_close(go, ro, "bf16", "c3 single-needle out")
    PT.assert_close(gl, rl, "bf16", "c3 single-needle lse")


@pytest.mark.parametrize("name,heads,needles", [
    ("c2", 8, False), ("c2", 4, True), ("c3", 2, False), ("c3", 2, True),
    ("c4", 2, False), ("c5", 2, False), ("c6", 8, False), ("c6", 8, True),
])
def test_full_size_sampled(name, heads, needles):
    p = PT.workload(name, needles)
    _, out, lse = run(p)
    rows = I.sample_rows(p, heads, seed=31)
    ro, rl = PT.oracle_rows(p, rows)
    go, gl = PT.gather_rows(out, lse, rows)
    PT.assert_close(go, ro, p.dtype, f"{name} out")
    PT.assert_close(gl, rl, p.dtype, f"{name} lse")
    # properties that hold at any size: finite everywhere, lse >= max visible score bound
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


# ---------------------------------------------------------------------------
# device-side table checks (bad contents never reach an address; the
# error word reports them and outputs are left untouched)
# ---------------------------------------------------------------------------
def _poisoned(p, field):
    di = api.device_inputs(p)
    if field == "slot":
        di.kv_indices[5] = di.pool_slots          # one past the pool
        want = 0x4
    elif field == "parent":
        di.tree_parent[0, 3] = 3                  # a node may not be its own parent
        want = 0x8
    elif field == "indptr":
        di.kv_indptr[1] += 1                      # span disagrees with prefix_lens + Q
        want = 0x2
    elif field == "prefix":
        di.prefix_lens[0] = -4
        want = 0x1
    return di, want


@pytest.mark.parametrize("field", ["slot", "parent", "indptr", "prefix"])
def test_device_table_errors(field):
    p = mid_problem(30)
    di, want = _poisoned(p, field)
    out = torch.full((p.B, p.Q, p.H, 512), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((p.B, p.Q, p.H), 7.0, dtype=torch.float32, device="cuda")
    ws = api.alloc_workspace(api.workspace_size(di, 0))
    api.verify_attn(di, out=out, lse=lse, workspace=ws)
    bits = api.check(ws)
    assert bits & want, hex(bits)
    assert (out.float() == 7.0).all() and (lse == 7.0).all()
    # the same workspace is clean again after a good call
    di2 = api.device_inputs(p)
    api.verify_attn(di2, workspace=ws)
    assert api.check(ws) == 0


def test_noop_shapes():
    p = I.make_problem(name="empty", dtype="bf16", B=1, H=4, Q=0, prefix_lens=[12], seed=1)
    di = api.device_inputs(p)
    out, lse = api.verify_attn(di)
    assert out.numel() == 0
