"""KV compaction through the C ABI (needs a GPU).

mla_kv_compact copies every sequence's rows, in the order the verify call
reads them, into one contiguous run of destination slots and writes the
page_size=1 tables of the new layout.  Checked bit for bit against the rows
the oracle resolves, and by the verify call itself: on the compacted layout it
must give the same bytes as on the original.
"""
import dataclasses

import numpy as np
import pytest

import oracle
from mla_tree_verify_absorbed_gb300 import api
from mla_tree_verify_absorbed_gb300 import inputs as I

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MLA_DEVERR_SLOT = 0x4
MLA_DEVERR_CAPACITY = 0x20


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.load()


def scattered():
    return I.make_problem(name="cs", dtype="bf16", B=3, H=16, Q=8, prefix_lens=[700, 0, 1500], seed=71,
                          layout="scattered", pool_slots=4096)


def paged():
    return I.make_problem(name="cp", dtype="bf16", B=2, H=16, Q=8, prefix_lens=[333, 1000], seed=72,
                          layout="paged", page_size=16, n_pages=120)


def pool_rows(p):
    """The pool as int16 bit patterns [slots][576] (exact comparison)."""
    return np.asarray(p.pool).view(np.int16)


@pytest.mark.parametrize("maker", [scattered, paged], ids=["scattered", "paged"])
def test_compaction_copies_rows_and_tables(maker):
    p = maker()
    di = api.device_inputs(p)
    src = oracle.get().resolve_slots(p)  # flat, sequence by sequence
    total = len(src)
    slot0 = 37
    dst = torch.full((slot0 + total + 5, 576), -3.0, dtype=torch.bfloat16, device="cuda")
    new_idx, new_indptr, ws = api.kv_compact(di, dst, dst_slot0=slot0)
    assert api.check(ws) == 0
    assert np.array_equal(new_idx.cpu().numpy(), slot0 + np.arange(total))
    lens = np.asarray(p.prefix_lens, dtype=np.int64) + p.Q
    assert np.array_equal(new_indptr.cpu().numpy(), np.concatenate([[0], np.cumsum(lens)]))
    got = dst.cpu().view(torch.int16).numpy()
    assert np.array_equal(got[slot0:slot0 + total], pool_rows(p)[src])
    # nothing outside the destination run is touched
    untouched = np.full((576,), np.array([-3.0], dtype=np.float32).view(np.int32)[0] >> 16, dtype=np.int16)
    assert (got[:slot0] == untouched).all() and (got[slot0 + total:] == untouched).all()


@pytest.mark.parametrize("maker", [scattered, paged], ids=["scattered", "paged"])
@pytest.mark.parametrize("algo", ["tc", "simt"])
def test_verify_on_compacted_layout_is_identical(maker, algo):
    p = maker()
    di = api.device_inputs(p)
    out0, lse0 = api.verify_attn(di, algo=algo)
    total = int((np.asarray(p.prefix_lens) + p.Q).sum())
    dst = torch.zeros((total, 576), dtype=torch.bfloat16, device="cuda")
    new_idx, new_indptr, ws = api.kv_compact(di, dst)
    assert api.check(ws) == 0
    dc = dataclasses.replace(di, kv_c=dst[:, :512], k_pe=dst[:, 512:], pool=dst, page_size=1,
                             kv_indptr=new_indptr, kv_indices=new_idx, block_table=None)
    out1, lse1 = api.verify_attn(dc, algo=algo)
    torch.cuda.synchronize()
    assert torch.equal(out1, out0) and torch.equal(lse1, lse0)


def test_capacity_overflow_is_reported():
    p = scattered()
    di = api.device_inputs(p)
    src = oracle.get().resolve_slots(p)
    cap = len(src) // 2
    dst = torch.zeros((cap, 576), dtype=torch.bfloat16, device="cuda")
    new_idx, _, ws = api.kv_compact(di, dst)
    assert api.check(ws) & MLA_DEVERR_CAPACITY
    # the rows that fit are there
    got = dst.cpu().view(torch.int16).numpy()
    assert np.array_equal(got, pool_rows(p)[src[:cap]])


def test_bad_table_copies_nothing():
    p = scattered()
    di = api.device_inputs(p)
    di.kv_indices[11] = p.pool.shape[0]  # one past the pool
    total = int((np.asarray(p.prefix_lens) + p.Q).sum())
    dst = torch.full((total, 576), 5.0, dtype=torch.bfloat16, device="cuda")
    _, _, ws = api.kv_compact(di, dst)
    assert api.check(ws) & MLA_DEVERR_SLOT
    assert (dst.float() == 5.0).all()
