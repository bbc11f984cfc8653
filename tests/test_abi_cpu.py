"""The C-ABI library without a GPU: it loads, exports every declared symbol,
and rejects malformed arguments on the host before touching CUDA."""
import ctypes
import glob
import os
import re

import pytest

from mla_tree_verify_absorbed_gb300 import api, build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return api.load()


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(mla_\w+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(api.EXPORTS), names
    for n in names:
        assert hasattr(lib, n), n


def test_abi_version_and_status_strings(lib):
    assert lib.mla_verify_abi_version() == 1
    assert api.status_str(0) == "MLA_OK"
    assert api.status_str(5) == "MLA_ERR_DEVICE_CHECK"


def test_struct_layout_matches_header(lib):
    # offsets of a few fields under the C ABI on LP64 (natural alignment)
    A = api.MlaVerifyArgs
    assert A.q_lat.offset == 16 and A.kv_c_stride.offset == 48 and A.page_size.offset == 72
    assert A.kv_indptr.offset == 80 and A.max_pages.offset == 104
    assert A.scale.offset == 128 and A.out.offset == 136 and A.algo.offset == 152
    assert A.profile_events.offset == 160 and ctypes.sizeof(A) == 168


def fake_args(**kw):
    """Well-formed arguments with fake (never dereferenced on the host) pointers."""
    a = api.MlaVerifyArgs()
    a.B, a.Q, a.H, a.dtype = 2, 8, 16, api.MLA_BF16
    p = 0x10000
    for f in ("q_lat", "q_pe", "kv_c", "k_pe", "kv_indptr", "kv_indices", "prefix_lens",
              "tree_parent", "out", "lse"):
        setattr(a, f, p)
        p += 0x10000
    a.kv_c_stride, a.k_pe_stride, a.pool_slots = 576, 576, 1000
    a.page_size, a.scale, a.algo = 1, 0.07, api.ALGO["simt"]
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def attn(lib, a, ws=0x100000, nbytes=1 << 40, splits=1):
    return lib.mla_verify_attn(ctypes.byref(a), ctypes.c_void_p(ws), ctypes.c_size_t(nbytes), splits, None)


@pytest.mark.parametrize("field,value,status", [
    ("B", -1, api.MLA_ERR_INVALID_ARG),
    ("H", 0, api.MLA_ERR_INVALID_ARG),
    ("Q", 65, api.MLA_ERR_UNSUPPORTED),
    ("dtype", 7, api.MLA_ERR_INVALID_ARG),
    ("algo", 9, api.MLA_ERR_INVALID_ARG),
])
def test_shape_validation(lib, field, value, status):
    a = fake_args(**{field: value})
    assert attn(lib, a) == status
    assert lib.mla_verify_workspace_size(ctypes.byref(a), 1) == 0


@pytest.mark.parametrize("field,value,status", [
    ("q_lat", None, api.MLA_ERR_INVALID_ARG),
    ("out", None, api.MLA_ERR_INVALID_ARG),
    ("kv_indices", None, api.MLA_ERR_INVALID_ARG),
    ("kv_c_stride", 511, api.MLA_ERR_INVALID_ARG),
    ("kv_c_stride", 516, api.MLA_ERR_INVALID_ARG),      # 1032 bytes: not a multiple of 16
    ("k_pe_stride", 60, api.MLA_ERR_INVALID_ARG),
    ("pool_slots", 0, api.MLA_ERR_INVALID_ARG),
    ("page_size", 0, api.MLA_ERR_INVALID_ARG),
    ("kv_c", 0x10008, api.MLA_ERR_INVALID_ARG),         # not 16-byte aligned
    ("scale", float("nan"), api.MLA_ERR_INVALID_ARG),
    ("scale", 0.0, api.MLA_ERR_INVALID_ARG),
    ("scale", -0.07, api.MLA_ERR_INVALID_ARG),
    ("scale", float("inf"), api.MLA_ERR_INVALID_ARG),
])
def test_call_validation(lib, field, value, status):
    # the workspace size depends on shapes only; the call itself rejects these
    a = fake_args(**{field: value})
    assert attn(lib, a) == status
    assert lib.mla_verify_workspace_size(ctypes.byref(a), 1) == \
        lib.mla_verify_workspace_size(ctypes.byref(fake_args()), 1)


def test_tc_requires_bf16(lib):
    a = fake_args(dtype=api.MLA_FP32, algo=api.ALGO["tc"])
    assert attn(lib, a) == api.MLA_ERR_UNSUPPORTED


def test_paged_needs_block_table(lib):
    a = fake_args(page_size=64, kv_indptr=None, kv_indices=None)
    assert attn(lib, a) == api.MLA_ERR_INVALID_ARG
    a = fake_args(page_size=64, block_table=0x900000, max_pages=0)
    assert attn(lib, a) == api.MLA_ERR_INVALID_ARG


def test_noop_shapes(lib):
    for kw in (dict(B=0), dict(Q=0)):
        a = fake_args(**kw)
        assert attn(lib, a, ws=0, nbytes=0) == api.MLA_OK


def test_workspace_checks(lib):
    a = fake_args()
    need = lib.mla_verify_workspace_size(ctypes.byref(a), 1)
    assert need > 0
    assert attn(lib, a, ws=0) == api.MLA_ERR_WORKSPACE
    assert attn(lib, a, ws=0x100010) == api.MLA_ERR_WORKSPACE          # not 256-byte aligned
    assert attn(lib, a, nbytes=need - 1) == api.MLA_ERR_WORKSPACE
    # more splits never need less workspace; one split needs no partials
    assert lib.mla_verify_workspace_size(ctypes.byref(a), 4) > need
    assert lib.mla_verify_workspace_size(ctypes.byref(a), 4) >= 4 * 2 * 8 * 16 * 513 * 4
    b = fake_args(algo=api.ALGO["tc"])
    assert lib.mla_verify_workspace_size(ctypes.byref(b), 3) > 0
    assert lib.mla_verify_workspace_size(ctypes.byref(a), -1) == 0
    assert lib.mla_verify_workspace_size(ctypes.byref(a), 5000) == 0


def test_splits_used_argument_checks(lib):
    # both checks come before any CUDA call
    v = ctypes.c_int32(-7)
    assert lib.mla_verify_splits_used(None, None, ctypes.byref(v)) == api.MLA_ERR_WORKSPACE
    assert lib.mla_verify_splits_used(ctypes.c_void_p(0x100000), None, None) == api.MLA_ERR_INVALID_ARG
    assert v.value == -7


def test_build_meta_validation(lib):
    a = fake_args()
    st = lib.mla_verify_build_meta(ctypes.byref(a), ctypes.c_void_p(0x100000), ctypes.c_size_t(1 << 40),
                                   None, ctypes.c_void_p(0x200000), ctypes.c_int64(10), None)
    assert st == api.MLA_ERR_INVALID_ARG


def test_selftest_timeout_argument_checks(lib):
    # rejected on the host, before any device call
    a = fake_args()
    ws = ctypes.c_void_p(0x100000)
    assert lib.mla_verify_selftest_timeout(ctypes.byref(a), ws, 1 << 20, 0, None) == api.MLA_ERR_INVALID_ARG
    assert lib.mla_verify_selftest_timeout(ctypes.byref(a), ws, 1 << 20, 2_000_000_000, None) == \
        api.MLA_ERR_INVALID_ARG
    f = fake_args(dtype=api.MLA_FP32)
    assert lib.mla_verify_selftest_timeout(ctypes.byref(f), ws, 1 << 20, 1000, None) == api.MLA_ERR_UNSUPPORTED
    s = fake_args(algo=api.ALGO["simt"])
    assert lib.mla_verify_selftest_timeout(ctypes.byref(s), ws, 1 << 20, 1000, None) == api.MLA_ERR_UNSUPPORTED


def test_kv_compact_argument_checks(lib):
    a = fake_args()
    ws = ctypes.c_void_p(0x100000)
    good = dict(dst_kv_c=0x200000, dst_k_pe=0x200400, s1=576, s2=576, slot0=0, slots=1 << 20, idx=0x300000)

    def call(**kw):
        c = dict(good, **kw)
        return lib.mla_kv_compact(ctypes.byref(a), ws, 1 << 24, c["dst_kv_c"], c["dst_k_pe"], c["s1"], c["s2"],
                                  c["slot0"], c["slots"], c["idx"], None, None)
    assert call(dst_kv_c=None) == api.MLA_ERR_INVALID_ARG
    assert call(idx=None) == api.MLA_ERR_INVALID_ARG
    assert call(dst_k_pe=0x200408) == api.MLA_ERR_INVALID_ARG   # not 16-byte aligned
    assert call(s1=500) == api.MLA_ERR_INVALID_ARG              # a destination row must hold 512 elements
    assert call(s2=60) == api.MLA_ERR_INVALID_ARG
    assert call(s1=577) == api.MLA_ERR_INVALID_ARG              # row stride not a multiple of 16 bytes
    assert call(slot0=-1) == api.MLA_ERR_INVALID_ARG
    assert call(slots=1 << 40) == api.MLA_ERR_INVALID_ARG


def fake_build_args(**kw):
    a = api.MlaDdtreeBuildArgs()
    a.B, a.L, a.K, a.budget = 4, 16, 8, 63
    p = 0x10000
    for f in ("root_token", "cand_token", "cand_logp", "tree_parent", "tree_token", "tree_depth", "tree_score"):
        setattr(a, f, p)
        p += 0x10000
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def fake_accept_args(**kw):
    a = api.MlaDdtreeAcceptArgs()
    a.B, a.Q = 4, 64
    p = 0x10000
    for f in ("tree_parent", "tree_token", "target_token", "node_slot", "accept_len", "accept_nodes",
              "accept_slots", "next_token"):
        setattr(a, f, p)
        p += 0x10000
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_ddtree_struct_layout(lib):
    A = api.MlaDdtreeBuildArgs
    assert A.root_token.offset == 16 and A.tree_score.offset == 64 and ctypes.sizeof(A) == 72
    C = api.MlaDdtreeAcceptArgs
    assert C.tree_parent.offset == 8 and C.next_token.offset == 64 and ctypes.sizeof(C) == 72


@pytest.mark.parametrize("field,value", [
    ("B", -1), ("L", 0), ("L", 17), ("K", 0), ("K", 17), ("budget", 0), ("budget", 64),
    ("root_token", 0), ("cand_token", 0), ("cand_logp", 0), ("tree_parent", 0), ("tree_token", 0),
    ("cand_logp", 0x10002), ("tree_depth", 0x10001),
])
def test_ddtree_build_argument_checks(lib, field, value):
    a = fake_build_args(**{field: value})
    st = lib.mla_ddtree_build(ctypes.byref(a), ctypes.c_void_p(0x100000), ctypes.c_size_t(256), None)
    assert st == api.MLA_ERR_INVALID_ARG


def test_ddtree_build_budget_above_node_count(lib):
    # K = 1, L = 4: only four draft nodes exist
    a = fake_build_args(K=1, L=4, budget=5)
    assert lib.mla_ddtree_build(ctypes.byref(a), ctypes.c_void_p(0x100000), 256, None) == api.MLA_ERR_INVALID_ARG
    # K = 2, L = 2: 6 nodes
    a = fake_build_args(K=2, L=2, budget=7)
    assert lib.mla_ddtree_build(ctypes.byref(a), ctypes.c_void_p(0x100000), 256, None) == api.MLA_ERR_INVALID_ARG


def test_ddtree_workspace_checks(lib):
    a = fake_build_args()
    for ws, n in ((0, 256), (0x100080, 256), (0x100000, 255)):
        assert lib.mla_ddtree_build(ctypes.byref(a), ctypes.c_void_p(ws), n, None) == api.MLA_ERR_WORKSPACE
    c = fake_accept_args()
    for ws, n in ((0, 256), (0x100080, 256), (0x100000, 16)):
        assert lib.mla_ddtree_accept(ctypes.byref(c), ctypes.c_void_p(ws), n, None) == api.MLA_ERR_WORKSPACE


def test_ddtree_empty_batch_is_noop(lib):
    a = fake_build_args(B=0)
    assert lib.mla_ddtree_build(ctypes.byref(a), ctypes.c_void_p(0x100000), 256, None) == api.MLA_OK
    c = fake_accept_args(B=0)
    assert lib.mla_ddtree_accept(ctypes.byref(c), ctypes.c_void_p(0x100000), 256, None) == api.MLA_OK


@pytest.mark.parametrize("field,value", [
    ("B", -1), ("Q", 0), ("Q", 65), ("tree_parent", 0), ("tree_token", 0), ("target_token", 0),
    ("accept_len", 0), ("accept_nodes", 0), ("next_token", 0), ("node_slot", 0), ("accept_nodes", 0x10002),
])
def test_ddtree_accept_argument_checks(lib, field, value):
    c = fake_accept_args(**{field: value})
    st = lib.mla_ddtree_accept(ctypes.byref(c), ctypes.c_void_p(0x100000), ctypes.c_size_t(256), None)
    assert st == api.MLA_ERR_INVALID_ARG


def test_headers_are_plain_c(tmp_path):
    # The boundary is a C ABI: both headers compile as C99 on their own (no
    # CUDA or C++ headers), and every declared function can be referenced.
    names = declared_functions()
    src = "#include <mla_verify.h>\n#include <mla_ddtree.h>\n"
    src += "typedef void (*mla_any_fn)(void);\n"
    src += "mla_any_fn mla_abi_table[] = {\n" + ",\n".join(f"  (mla_any_fn)&{n}" for n in names) + "\n};\n"
    src += "int mla_abi_sizes(void) { return (int)(sizeof(mla_verify_args) + sizeof(mla_ddtree_build_args)"
    src += " + sizeof(mla_ddtree_accept_args)); }\n"
    c = tmp_path / "abi.c"
    c.write_text(src)
    import subprocess
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-c", str(c),
                        "-I", os.path.join(ROOT, "include"), "-o", str(tmp_path / "abi.o")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_ddtree_binding_rejects_wrong_tensors(lib):
    # checks the binding makes before any pointer reaches the library
    torch = pytest.importorskip("torch")
    ws = torch.zeros(256, dtype=torch.uint8)
    B, L, K = 2, 4, 3
    root = torch.zeros(B, dtype=torch.int32)
    tok = torch.zeros(B, L, K, dtype=torch.int32)
    lp = torch.zeros(B, L, K, dtype=torch.float32)
    par = torch.zeros(B, 6, dtype=torch.int32)
    tt = torch.zeros(B, 6, dtype=torch.int32)
    with pytest.raises(ValueError, match="dtype"):
        api.ddtree_build_into(root, tok, lp.double(), 5, par, tt, ws)
    with pytest.raises(ValueError, match="dtype"):
        api.ddtree_build_into(root.long(), tok, lp, 5, par, tt, ws)
    with pytest.raises(ValueError, match="shape"):
        api.ddtree_build_into(root, tok, lp, 4, par, tt, ws)  # outputs sized for budget 5
    with pytest.raises(ValueError, match="contiguous"):
        api.ddtree_build_into(root, tok.transpose(1, 2).contiguous().transpose(1, 2), lp, 5, par, tt, ws)
    with pytest.raises(ValueError, match="CUDA"):
        api.ddtree_build_into(root, tok, lp, 5, par, tt, ws)  # CPU tensors
    n = torch.zeros(B, dtype=torch.int32)
    with pytest.raises(ValueError, match="dtype"):
        api.ddtree_accept_into(par, tt, tt.long(), n, par, n, ws)
    with pytest.raises(ValueError, match="shape"):
        api.ddtree_accept_into(par, tt, tt, n[:1], par, n, ws)


def test_device_inputs_check_catches_wrong_tensors():
    torch = pytest.importorskip("torch")
    import dataclasses
    from mla_tree_verify_absorbed_gb300 import inputs as I
    p = I.make_problem(name="chk", dtype="bf16", B=2, H=4, Q=3, prefix_lens=[5, 9], seed=1,
                       layout="scattered", pool_slots=64)
    di = api.device_inputs(p, device="cpu")
    with pytest.raises(ValueError, match="CUDA"):
        di.check()  # everything right but the device
    with pytest.raises(ValueError, match="prefix_lens"):
        dataclasses.replace(di, prefix_lens=di.prefix_lens.long()).check()
    with pytest.raises(ValueError, match="q_lat"):
        dataclasses.replace(di, q_lat=di.q_lat.float()).check()
    with pytest.raises(ValueError, match="kv_c"):
        dataclasses.replace(di, kv_c=di.pool[:, :256]).check()
    with pytest.raises(ValueError, match="kv_indices"):
        dataclasses.replace(di, kv_indices=di.kv_indices.long()).check()
    with pytest.raises(ValueError, match="out"):
        api.make_args(di, out=torch.zeros(2, 3, 4, 256, dtype=torch.bfloat16))
