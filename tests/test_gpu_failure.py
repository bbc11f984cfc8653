"""Failure detection on the GPU without a fault (needs a GPU).

mla_verify_selftest_timeout runs the tensor-core call with one device wait
that nothing completes, bounded by a short limit.  The kernel must give up,
stop every CTA of the cluster, free its Tensor Memory and finish; the host
reads MLA_DEVERR_TIMEOUT and the wait site from the workspace; the outputs
are untouched; and the next ordinary call on the same context and workspace
runs clean and correct.
"""
import time

import pytest

from mla_tree_verify_absorbed_gb300 import api
from mla_tree_verify_absorbed_gb300 import inputs as I
from tests import parity as PT

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MLA_DEVERR_TIMEOUT = 0x40
SITE_HOLD = 18  # the self-test wait's site number in the second error word


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.load()


def test_timeout_is_reported_and_the_context_recovers():
    p = I.make_problem(name="hold", dtype="bf16", B=2, H=64, Q=16, prefix_lens=[900, 2100], seed=61,
                       layout="scattered", pool_slots=4096)
    di = api.device_inputs(p)
    out = torch.full((p.B, p.Q, p.H, 512), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((p.B, p.Q, p.H), 7.0, dtype=torch.float32, device="cuda")
    ws = api.alloc_workspace(api.workspace_size(di, 0, algo="tc"))

    t0 = time.monotonic()
    api.selftest_timeout(di, out, lse, ws, hold_ns=50_000_000)
    bits = api.check(ws)
    elapsed = time.monotonic() - t0
    assert bits & MLA_DEVERR_TIMEOUT, hex(bits)
    site = int(ws[:8].view(torch.int32)[1].item())
    assert site & 0xFF == SITE_HOLD and (site >> 8) & 0xFF == 0, hex(site)  # score leader CTA
    assert elapsed < 10.0, elapsed
    assert (out.float() == 7.0).all() and (lse == 7.0).all()

    # the same context and workspace: an ordinary call runs clean and correct
    out2, lse2 = api.verify_attn(di, workspace=ws)
    assert api.check(ws) == 0
    rows = I.all_rows(p)
    ro, rl = PT.oracle_rows(p, rows)
    go, gl = PT.gather_rows(out2, lse2, rows)
    PT.assert_close(go, ro, "bf16", "after timeout out")
    PT.assert_close(gl, rl, "bf16", "after timeout lse")
