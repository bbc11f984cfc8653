"""mla_verify_attn_noalloc against mla_verify_attn (needs a GPU).

The no-allocation entry point serves callers that may not allocate device
memory at call time (a plugin inside an engine that owns the device memory
pool, a decode loop that must avoid cudaMalloc's synchronisation).  It runs
the same kernels with the same split count on a scratch array held by the
library, so its results must be the same bytes as the regular entry point's
-- and stay the same on a second call, when the shared scratch still holds the
first call's contents.  Collected last on purpose (file name).
"""
import ctypes

import numpy as np
import pytest

from mla_tree_verify_absorbed_gb300 import api
from mla_tree_verify_absorbed_gb300 import inputs as I

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.load()


def _ws_size(di, splits, algo):
    a = api.make_args(di, algo=algo, check=False)
    return int(api.load().mla_verify_workspace_size(ctypes.byref(a), int(splits)))


@pytest.mark.parametrize("case", ["bf16_tc", "fp32_simt"])
def test_noalloc_matches_regular_entry_point_twice(case):
    if case == "bf16_tc":
        p = I.make_problem(name="noalloc", dtype="bf16", B=2, H=64, Q=16, prefix_lens=[300, 777],
                           seed=41, layout="scattered", pool_slots=2048)
        splits, algo = 2, "tc"
    else:
        p = I.make_config("tiny")
        splits, algo = 3, "simt"
    di = api.device_inputs(p)
    ref_out, ref_lse = api.verify_attn(di, num_splits=splits, algo=algo)
    torch.cuda.synchronize()
    for call in range(2):
        out, lse = api.verify_attn_noalloc(di, num_splits=splits, algo=algo, check_device=True)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out), f"call {call}: out differs from mla_verify_attn"
        assert torch.equal(lse, ref_lse), f"call {call}: lse differs from mla_verify_attn"


def test_noalloc_automatic_splits_fit_the_scratch():
    # 64 heads x 64 nodes: the automatic split count of mla_verify_attn needs
    # more workspace than the scratch holds, so the no-allocation call lowers
    # it to the largest count that fits -- and equals mla_verify_attn run with
    # that count, byte for byte, on two calls in a row
    p = I.make_problem(name="noalloc_auto", dtype="bf16", B=1, H=64, Q=64, prefix_lens=[2000],
                       seed=43, layout="scattered", pool_slots=4096)
    di = api.device_inputs(p)
    auto_bytes = _ws_size(di, 0, "tc")
    assert auto_bytes > api.NOALLOC_SCRATCH_BYTES
    s_auto = next(s for s in range(1, 4097) if _ws_size(di, s, "tc") == auto_bytes)
    fit = max(s for s in range(1, s_auto + 1) if _ws_size(di, s, "tc") <= api.NOALLOC_SCRATCH_BYTES)
    assert 1 <= fit < s_auto
    ref_out, ref_lse = api.verify_attn(di, num_splits=fit, algo="tc")
    for call in range(2):
        out, lse = api.verify_attn_noalloc(di, num_splits=0, algo="tc", check_device=True)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out), f"call {call}: out differs from mla_verify_attn with {fit} splits"
        assert torch.equal(lse, ref_lse), f"call {call}: lse differs"


def test_noalloc_reports_device_table_errors():
    # a slot one past the pool: the metadata kernel rejects it before any KV
    # access, the attention writes nothing, and the error word in the
    # library's scratch says why; the next good call is clean again
    p = I.make_problem(name="noalloc_bad", dtype="bf16", B=2, H=16, Q=8, prefix_lens=[200, 37],
                       seed=44, layout="scattered", pool_slots=600)
    di = api.device_inputs(p)
    good_out, good_lse = api.verify_attn(di, num_splits=1, algo="tc")
    di.kv_indices[5] = di.pool_slots
    out = torch.full((p.B, p.Q, p.H, 512), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((p.B, p.Q, p.H), 7.0, dtype=torch.float32, device="cuda")
    api.verify_attn_noalloc(di, out=out, lse=lse, num_splits=1, algo="tc")
    bits = api.noalloc_check()
    assert bits & 0x4, hex(bits)  # MLA_DEVERR_SLOT
    assert (out.float() == 7.0).all() and (lse == 7.0).all()
    with pytest.raises(api.MlaError) as e:
        api.verify_attn_noalloc(di, out=out, lse=lse, num_splits=1, algo="tc", check_device=True)
    assert e.value.status == api.MLA_ERR_DEVICE_CHECK
    di2 = api.device_inputs(p)
    out2, lse2 = api.verify_attn_noalloc(di2, num_splits=1, algo="tc", check_device=True)
    assert api.noalloc_check() == 0
    assert torch.equal(out2, good_out) and torch.equal(lse2, good_lse)


def test_noalloc_rejects_oversized_work():
    p = I.make_problem(name="big", dtype="bf16", B=2, H=64, Q=16, prefix_lens=[300, 777],
                       seed=42, layout="scattered", pool_slots=2048)
    di = api.device_inputs(p)
    need = _ws_size(di, 64, "tc")
    assert need > api.NOALLOC_SCRATCH_BYTES
    with pytest.raises(api.MlaError) as e:
        api.verify_attn_noalloc(di, num_splits=64, algo="tc")
    assert e.value.status == api.MLA_ERR_WORKSPACE
