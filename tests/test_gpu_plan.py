"""The automatic split count, chosen on the device from the sequences' lengths
(needs a GPU).

With num_splits = 0 the host sizes the workspace for S_max, the count whose
work items fill the clusters in whole waves (from B, H, Q and the SM count
alone), and the metadata kernel picks the tensor-core kernel's count S in
[1, S_max] once it has read prefix_lens, by a cost model of the kernels.
Checked here:
  * the device's choice equals the same model restated plainly on the host
    (items dealt round-robin to the clusters, each cluster's load the sum of
    (fixed cost + tiles) over its items, the most loaded cluster's time plus,
    for S > 1, the combine's pass over the fp32 partials; integer ns);
  * an automatic call gives the same bytes as an explicit call with the count
    it chose (same kernels, same chunks) and matches the oracle;
  * the choice follows the lengths: equal B, H, Q pick different counts for
    a short and a long prefix;
  * a pieced tail (S = 1, the last partial wave's items cut into pieces)
    leaves every whole item's bytes as the explicit call's and matches the
    oracle on the tail's rows;
  * the SIMT kernel keeps S_max.
"""
import ctypes

import numpy as np
import pytest

from mla_tree_verify_absorbed_gb300 import api
from mla_tree_verify_absorbed_gb300 import inputs as I
from tests import parity as PT

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

# the model's constants (GB300 measurements of the kernels): ns per 64-token
# tile on one cluster, fixed cost per item in tiles, combine bytes per ns and
# its fixed ns
TILE_NS, ITEM_TILES, COMBINE_BYTES_PER_NS, COMBINE_NS = 1000, 14, 3000, 3000
TK, RG_TC = 64, 256


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.load()


def model_choice(prefix_lens, Q, H, s_max, grid):
    """(S, P): the split count and the pieces per tail item (1: none)."""
    T = [-(-(int(P) + Q) // TK) for P in prefix_lens]
    B, rows = len(T), H * Q
    G = -(-rows // RG_TC)
    best = None
    for S in range(1, s_max + 1):
        load = [0] * grid
        n = B * G * S
        for i in range(n):
            bk = i // G
            k, b = bk % S, bk // S
            t = (k + 1) * T[b] // S - k * T[b] // S
            if t > 0:
                load[i % grid] += ITEM_TILES + t
        ns = max(load) * TILE_NS
        if S > 1:
            ns += B * S * rows * 512 * 4 // COMBINE_BYTES_PER_NS + COMBINE_NS
        cand = (ns, S, 1)
        full = (n // grid) * grid
        r = n - full
        if S == 1 and full > 0 and r > 0 and grid // r >= 2:
            # the last r items cut into P pieces, one per otherwise idle cluster
            P = grid // r
            load = [0] * grid
            for i in range(full):
                if T[i // G] > 0:
                    load[i % grid] += ITEM_TILES + T[i // G]
            for v in range(r * P):
                Tb = T[(full + v // P) // G]
                q = v % P
                t = (q + 1) * Tb // P - q * Tb // P
                if t > 0:
                    load[v] += ITEM_TILES + t
            tns = max(load) * TILE_NS + r * P * RG_TC * 512 * 4 // COMBINE_BYTES_PER_NS + COMBINE_NS
            if tns < ns:
                cand = (tns, S, P)
        if best is None or cand[0] < best[0]:
            best = cand
    return best[1], best[2]


def ws_size(di, splits, algo):
    a = api.make_args(di, algo=algo, check=False)
    return int(api.load().mla_verify_workspace_size(ctypes.byref(a), int(splits)))


def s_max_of(di, algo):
    """The count the workspace of an automatic call is sized for: the explicit
    count with the same workspace, or 1 when there is none (an automatic
    tensor-core plan with S_max = 1 still holds one partial slot per cluster
    for a pieced tail, which an explicit single chunk does not)."""
    want = ws_size(di, 0, algo)
    hits = [k for k in range(1, 65) if ws_size(di, k, algo) == want]
    if not hits:
        assert algo == "tc" and ws_size(di, 1, algo) < want < ws_size(di, 2, algo)
        return 1
    assert len(hits) == 1, hits
    return hits[0]


def auto_call(di, algo="tc"):
    """(out, lse, S used, grid the plan assumed, first tail item, pieces per
    tail item) -- the plan words follow S at workspace offset 256."""
    ws = api.alloc_workspace(ws_size(di, 0, algo))
    out, lse = api.verify_attn(di, num_splits=0, algo=algo, workspace=ws)
    used = api.splits_used(ws)
    words = ws[256:272].cpu().numpy().view(np.int32)
    return out, lse, used, int(words[1]), int(words[2]), int(words[3])


SHAPES = {
    # name: (B, H, Q, prefix_lens, layout)
    "one_seq_4k": (1, 64, 64, [4096], "scattered"),
    "one_seq_65k": (1, 64, 64, [65536], "scattered"),
    "ragged4": (4, 64, 32, [100, 5000, 20000, 700], "scattered"),
    "many_heads_paged": (8, 128, 16, [2048, 1500, 3000, 64, 2048, 900, 2500, 2048], "paged"),
    "small_mid": (2, 64, 16, [300, 777], "scattered"),
    # 80 items on 36 clusters: two whole waves and a tail of 8 items
    "tail_split": (10, 128, 16, [2048] * 10, "paged"),
}


def make(name, seed=61):
    B, H, Q, lens, layout = SHAPES[name]
    total = sum(int(P) + Q for P in lens)
    kw = dict(name=name, dtype="bf16", B=B, H=H, Q=Q, prefix_lens=lens, seed=seed)
    if layout == "paged":
        kw.update(layout="paged", page_size=64, n_pages=sum(-(-(int(P) + Q) // 64) for P in lens) + 8)
    else:
        kw.update(layout="scattered", pool_slots=total + 1024)
    return I.make_problem(**kw)


@pytest.mark.parametrize("name", list(SHAPES))
def test_device_choice_equals_the_model(name):
    p = make(name)
    di = api.device_inputs(p)
    s_max = s_max_of(di, "tc")
    out, lse, used, grid, tail, pieces = auto_call(di)
    assert 1 <= used <= s_max
    assert grid >= 1
    want = model_choice(p.prefix_lens, p.Q, p.H, s_max, grid)
    assert (used, pieces) == want, (used, pieces, s_max, grid)
    n_items = p.B * (-(-p.H * p.Q // RG_TC)) * used
    ref_out, ref_lse = api.verify_attn(di, num_splits=used, algo="tc")
    torch.cuda.synchronize()
    if pieces == 1:
        # the same bytes as the explicit count
        assert tail == n_items
        assert torch.equal(out, ref_out)
        assert torch.equal(lse, ref_lse)
    else:
        # whole items give the explicit call's bytes; the rows of the pieced
        # tail are merged from pieces (compared with the oracle elsewhere)
        assert tail == (n_items // grid) * grid and 0 < n_items - tail < grid
        G = -(-p.H * p.Q // RG_TC)
        whole = np.ones((p.B, p.Q * p.H), dtype=bool)
        for item in range(tail, n_items):
            b, g = item // G, item % G
            whole[b, g * RG_TC:(g + 1) * RG_TC] = False
        m = torch.as_tensor(whole.reshape(p.B, p.Q, p.H), device=out.device)
        assert torch.equal(out[m], ref_out[m])
        assert torch.equal(lse[m], ref_lse[m])
        assert not bool(m.all())


@pytest.mark.parametrize("name", ["ragged4", "small_mid", "many_heads_paged", "tail_split"])
def test_automatic_count_matches_oracle(name):
    p = make(name, seed=62)
    di = api.device_inputs(p)
    out, lse, used, _, _, pieces = auto_call(di)
    rows = I.sample_rows(p, 2, seed=5) if name != "small_mid" else I.all_rows(p)
    if name == "tail_split":
        assert pieces > 1
        rows = rows[rows[:, 0] == p.B - 1]  # the last sequence's row groups are the tail
    ro, rl = PT.oracle_rows(p, rows)
    go, gl = PT.gather_rows(out, lse, rows)
    PT.assert_close(go, ro, "bf16", f"{name} auto S={used} P={pieces} out")
    PT.assert_close(gl, rl, "bf16", f"{name} auto S={used} P={pieces} lse")


def test_choice_follows_the_lengths():
    # equal B, H, Q (so equal S_max and workspace): a 4k prefix is best cut in
    # few chunks, a 100k prefix in S_max
    short = api.device_inputs(I.make_problem(name="short", dtype="bf16", B=1, H=64, Q=64, prefix_lens=[4096],
                                             seed=63, layout="scattered", pool_slots=8192))
    long_ = api.device_inputs(I.make_problem(name="long", dtype="bf16", B=1, H=64, Q=64, prefix_lens=[100000],
                                             seed=64, layout="scattered", pool_slots=131072))
    s_max = s_max_of(short, "tc")
    assert s_max_of(long_, "tc") == s_max
    _, _, s_short, grid, _, _ = auto_call(short)
    _, _, s_long, _, _, _ = auto_call(long_)
    assert s_short == model_choice([4096], 64, 64, s_max, grid)[0]
    assert s_long == model_choice([100000], 64, 64, s_max, grid)[0]
    assert s_short < s_long


def test_simt_keeps_the_wave_count():
    p = make("small_mid", seed=65)
    di = api.device_inputs(p)
    _, _, used, _, tail, pieces = auto_call(di, algo="simt")
    assert used == s_max_of(di, "simt")
    assert pieces == 1


def test_batches_beyond_the_plan_keep_the_wave_count():
    # the plan is made for up to 2048 sequences (their tile counts in shared
    # memory); a larger batch keeps S_max -- here 1: 2100 row groups fill the
    # clusters -- and no pieced tail
    B = 2100
    lens = np.random.default_rng(66).integers(0, 200, size=B)
    p = I.make_problem(name="many_seqs", dtype="bf16", B=B, H=16, Q=1, prefix_lens=lens, seed=66,
                       layout="scattered", pool_slots=int(lens.sum()) + B + 64)
    di = api.device_inputs(p)
    out, lse, used, _, _, pieces = auto_call(di)
    assert used == s_max_of(di, "tc") == 1
    assert pieces == 1
    rows = I.sample_rows(p, 2, seed=7)[::8]
    ro, rl = PT.oracle_rows(p, rows)
    go, gl = PT.gather_rows(out, lse, rows)
    PT.assert_close(go, ro, "bf16", "2100 sequences out")
    PT.assert_close(gl, rl, "bf16", "2100 sequences lse")
