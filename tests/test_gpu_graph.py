"""The verify call captured in a CUDA graph (needs a GPU).

The call makes no host synchronisation and no allocation when the caller
passes the outputs and the workspace, so it can be captured once and replayed
for every verify step of a decode loop.  A replay must give the same bytes as
an eager call on the same inputs (same partition, same kernels), and must pick
up inputs updated in place between replays.
"""
import numpy as np
import pytest

from mla_tree_verify_absorbed_gb300 import api
from mla_tree_verify_absorbed_gb300 import inputs as I
from tests import parity as PT

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.load()


def _problem(seed):
    return I.make_problem(name="graph", dtype="bf16", B=2, H=64, Q=16, prefix_lens=[900, 2100], seed=seed,
                          layout="scattered", pool_slots=4096)


@pytest.mark.parametrize("algo", ["tc", "simt"])
def test_graph_replay_matches_eager(algo):
    p = _problem(51)
    di = api.device_inputs(p)
    out0, lse0 = api.verify_attn(di, algo=algo)
    torch.cuda.synchronize()

    out = torch.empty_like(out0)
    lse = torch.empty_like(lse0)
    ws = api.alloc_workspace(api.workspace_size(di, 0, algo=algo))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture
        api.verify_attn(di, out=out, lse=lse, workspace=ws, algo=algo)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        api.verify_attn(di, out=out, lse=lse, workspace=ws, algo=algo)
    out.zero_()
    lse.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, out0) and torch.equal(lse, lse0)
    assert api.check(ws) == 0

    # new queries written into the captured buffers: the replay follows them
    p2 = _problem(52)
    di.q_lat.copy_(torch.as_tensor(p2.q_lat.view(np.int16)).view(torch.bfloat16).to(di.q_lat.device)
                   .reshape(di.q_lat.shape))
    di.q_pe.copy_(torch.as_tensor(p2.q_pe.view(np.int16)).view(torch.bfloat16).to(di.q_pe.device)
                  .reshape(di.q_pe.shape))
    g.replay()
    torch.cuda.synchronize()
    p.q_lat, p.q_pe = p2.q_lat, p2.q_pe
    rows = I.all_rows(p)
    ro, rl = PT.oracle_rows(p, rows)
    go, gl = PT.gather_rows(out, lse, rows)
    PT.assert_close(go, ro, "bf16", f"graph/{algo} out")
    PT.assert_close(gl, rl, "bf16", f"graph/{algo} lse")


@pytest.mark.parametrize("algo", ["tc", "simt"])
def test_overlapped_launches_match_plain_launches(algo):
    # Without profiling events the metadata, attention and combine kernels
    # are launched with programmatic stream serialization (each may start
    # while the previous one finishes); with events they are plain launches.
    # Both must give the same bytes, back to back on one stream, many times.
    p = I.make_problem(name="pdl", dtype="bf16", B=3, H=16, Q=8, prefix_lens=[3000, 17, 1200], seed=81,
                       layout="scattered", pool_slots=8192)
    di = api.device_inputs(p)
    ref_o, ref_l = api.verify_attn(di, algo=algo, num_splits=3)
    evs = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    for e in evs:
        e.record()
    plain_o, plain_l = api.verify_attn(di, algo=algo, num_splits=3, profile_events=evs)
    torch.cuda.synchronize()
    assert torch.equal(plain_o, ref_o) and torch.equal(plain_l, ref_l)
    ws = api.alloc_workspace(api.workspace_size(di, 3, algo))
    outs = []
    for _ in range(20):
        o, l = api.verify_attn(di, algo=algo, num_splits=3, workspace=ws)
        outs.append((o, l))
    torch.cuda.synchronize()
    assert api.check(ws) == 0
    for o, l in outs:
        assert torch.equal(o, ref_o) and torch.equal(l, ref_l)


def test_graph_replay_follows_new_lengths():
    # the split count is chosen on the device from prefix_lens, so a captured
    # call re-plans when the caller shortens a sequence between replays (a
    # plan fixed on the host at capture time could not)
    p = I.make_problem(name="graph_len", dtype="bf16", B=1, H=64, Q=64, prefix_lens=[8000], seed=53,
                       layout="scattered", pool_slots=9000)
    di = api.device_inputs(p)
    out = torch.empty((1, 64, 64, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, 64, 64), dtype=torch.float32, device="cuda")
    ws = api.alloc_workspace(api.workspace_size(di, 0, algo="tc"))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        api.verify_attn(di, out=out, lse=lse, workspace=ws, algo="tc")
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        api.verify_attn(di, out=out, lse=lse, workspace=ws, algo="tc")
    g.replay()
    long_splits = api.splits_used(ws)

    # 300 prefix tokens: the tree nodes now sit at positions 300..363 of the
    # same index table
    di.prefix_lens.fill_(300)
    di.kv_indptr[1] = 300 + 64
    g.replay()
    short_splits = api.splits_used(ws)
    assert api.check(ws) == 0
    assert long_splits > short_splits >= 1, (long_splits, short_splits)
    p.prefix_lens = np.array([300], dtype=np.int32)
    p.kv_indptr = np.array([0, 364], dtype=np.int32)
    rows = I.all_rows(p)
    ro, rl = PT.oracle_rows(p, rows)
    go, gl = PT.gather_rows(out, lse, rows)
    PT.assert_close(go, ro, "bf16", "graph after shortening out")
    PT.assert_close(gl, rl, "bf16", "graph after shortening lse")
