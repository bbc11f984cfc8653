"""mla_verify_attn_noalloc against mla_verify_attn (needs a GPU).

The no-allocation entry point serves callers that may not allocate device
memory at call time (a plugin inside an engine that owns the device memory
pool, a decode loop that must avoid cudaMalloc's synchronisation).  It runs
the same kernels on a scratch array held by the library, so its results must
match the regular entry point's within the parity tolerance -- and keep
matching on a second call, when the shared scratch still holds the first
call's contents.  Collected last on purpose (file name).
"""
import ctypes

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


def _as_np(out, lse):
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


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
    ro, rl = _as_np(ref_out, ref_lse)
    for call in range(2):
        out, lse = api.verify_attn_noalloc(di, num_splits=splits, algo=algo)
        torch.cuda.synchronize()
        go, gl = _as_np(out, lse)
        PT.assert_close(go, ro, p.dtype, f"call {call} out")
        PT.assert_close(gl, rl, p.dtype, f"call {call} lse")


def test_noalloc_rejects_oversized_work():
    p = I.make_problem(name="big", dtype="bf16", B=2, H=64, Q=16, prefix_lens=[300, 777],
                       seed=42, layout="scattered", pool_slots=2048)
    di = api.device_inputs(p)
    # placeholders: only the workspace size is asked for
    a = api.make_args(di, torch.empty(1, device="cuda"), torch.empty(1, device="cuda"), "tc", check=False)
    need = api.load().mla_verify_workspace_size(ctypes.byref(a), 64)
    assert need > api.NOALLOC_SCRATCH_BYTES
    with pytest.raises(api.MlaError) as e:
        api.verify_attn_noalloc(di, num_splits=64, algo="tc")
    assert e.value.status == api.MLA_ERR_WORKSPACE
