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
    T = [-(-(int(P) + Q) // TK) for P in prefix_lens]
    B, rows = len(T), H * Q
    G = -(-rows // RG_TC)
    best, best_ns = None, None
    for S in range(1, s_max + 1):
        load = [0] * grid
        for i in range(B * G * S):
            bk = i // G
            k, b = bk % S, bk // S
            t = (k + 1) * T[b] // S - k * T[b] // S
            if t > 0:
                load[i % grid] += ITEM_TILES + t
        ns = max(load) * TILE_NS
        if S > 1:
            ns += B * rows * S * 512 * 4 // COMBINE_BYTES_PER_NS + COMBINE_NS
        if best_ns is None or ns < best_ns:
            best, best_ns = S, ns
    return best


def ws_size(di, splits, algo):
    a = api.make_args(di, algo=algo, check=False)
    return int(api.load().mla_verify_workspace_size(ctypes.byref(a), int(splits)))


def s_max_of(di, algo):
    """The count the workspace of an automatic call is sized for."""
    want = ws_size(di, 0, algo)
    hits = [k for k in range(1, 65) if ws_size(di, k, algo) == want]
    assert len(hits) == 1, hits
    return hits[0]


def auto_call(di, algo="tc"):
    ws = api.alloc_workspace(ws_size(di, 0, algo))
    out, lse = api.verify_attn(di, num_splits=0, algo=algo, workspace=ws)
    used = api.splits_used(ws)
    grid = int(ws[260:264].cpu().numpy().view(np.int32)[0])  # the cluster count the plan assumed
    return out, lse, used, grid


SHAPES = {
    # name: (B, H, Q, prefix_lens, layout)
    "one_seq_4k": (1, 64, 64, [4096], "scattered"),
    "one_seq_65k": (1, 64, 64, [65536], "scattered"),
    "ragged4": (4, 64, 32, [100, 5000, 20000, 700], "scattered"),
    "many_heads_paged": (8, 128, 16, [2048, 1500, 3000, 64, 2048, 900, 2500, 2048], "paged"),
    "small_mid": (2, 64, 16, [300, 777], "scattered"),
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
    out, lse, used, grid = auto_call(di)
    assert 1 <= used <= s_max
    assert grid >= 1
    assert used == model_choice(p.prefix_lens, p.Q, p.H, s_max, grid), (used, s_max, grid)
    # the same bytes as the explicit count
    ref_out, ref_lse = api.verify_attn(di, num_splits=used, algo="tc")
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)
    assert torch.equal(lse, ref_lse)


@pytest.mark.parametrize("name", ["ragged4", "small_mid", "many_heads_paged"])
def test_automatic_count_matches_oracle(name):
    p = make(name, seed=62)
    di = api.device_inputs(p)
    out, lse, used, _ = auto_call(di)
    rows = I.sample_rows(p, 2, seed=5) if name != "small_mid" else I.all_rows(p)
    ro, rl = PT.oracle_rows(p, rows)
    go, gl = PT.gather_rows(out, lse, rows)
    PT.assert_close(go, ro, "bf16", f"{name} auto S={used} out")
    PT.assert_close(gl, rl, "bf16", f"{name} auto S={used} lse")


def test_choice_follows_the_lengths():
    # equal B, H, Q (so equal S_max and workspace): a 4k prefix is best cut in
    # few chunks, a 100k prefix in S_max
    short = api.device_inputs(I.make_problem(name="short", dtype="bf16", B=1, H=64, Q=64, prefix_lens=[4096],
                                             seed=63, layout="scattered", pool_slots=8192))
    long_ = api.device_inputs(I.make_problem(name="long", dtype="bf16", B=1, H=64, Q=64, prefix_lens=[100000],
                                             seed=64, layout="scattered", pool_slots=131072))
    s_max = s_max_of(short, "tc")
    assert s_max_of(long_, "tc") == s_max
    _, _, s_short, grid = auto_call(short)
    _, _, s_long, _ = auto_call(long_)
    assert s_short == model_choice([4096], 64, 64, s_max, grid)
    assert s_long == model_choice([100000], 64, 64, s_max, grid)
    assert s_short < s_long


def test_simt_keeps_the_wave_count():
    p = make("small_mid", seed=65)
    di = api.device_inputs(p)
    _, _, used, _ = auto_call(di, algo="simt")
    assert used == s_max_of(di, "simt")
