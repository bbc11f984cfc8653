"""ctypes binding of the C ABI in include/mla_verify.h and include/mla_ddtree.h.

Argument marshalling only: torch tensors give device pointers, sizes and
strides; every step of the computation runs in the CUDA library.  The library
is loaded on first use and a missing build raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libmla_verify.so")

MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_CUDA, MLA_ERR_WORKSPACE, \
    MLA_ERR_DEVICE_CHECK = range(6)
MLA_BF16, MLA_FP32 = 0, 1
ALGO = {"auto": 0, "simt": 1, "tc": 2}

DEVERR = {
    0x1: "PREFIX", 0x2: "INDPTR", 0x4: "SLOT", 0x8: "PARENT", 0x10: "PAGES",
    0x20: "CAPACITY", 0x40: "TIMEOUT", 0x80: "LAYOUT", 0x100: "DRAFT",
}

# every symbol include/*.h declares
EXPORTS = ("mla_verify_workspace_size", "mla_verify_attn", "mla_verify_attn_noalloc", "mla_verify_noalloc_check",
           "mla_verify_build_meta", "mla_verify_check", "mla_verify_splits_used", "mla_status_str",
           "mla_verify_abi_version",
           "mla_verify_selftest_timeout", "mla_kv_compact", "mla_ddtree_build", "mla_ddtree_accept")
NOALLOC_SCRATCH_BYTES = 32 << 20
DDTREE_WORKSPACE_BYTES = 256


class MlaVerifyArgs(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("Q", ctypes.c_int), ("H", ctypes.c_int),
        ("dtype", ctypes.c_int),
        ("q_lat", ctypes.c_void_p), ("q_pe", ctypes.c_void_p),
        ("kv_c", ctypes.c_void_p), ("k_pe", ctypes.c_void_p),
        ("kv_c_stride", ctypes.c_int64), ("k_pe_stride", ctypes.c_int64),
        ("pool_slots", ctypes.c_int64),
        ("page_size", ctypes.c_int),
        ("kv_indptr", ctypes.c_void_p), ("kv_indices", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p), ("max_pages", ctypes.c_int),
        ("prefix_lens", ctypes.c_void_p), ("tree_parent", ctypes.c_void_p),
        ("scale", ctypes.c_float),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("algo", ctypes.c_int),
        ("profile_events", ctypes.c_void_p),
    ]


class MlaDdtreeBuildArgs(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("L", ctypes.c_int), ("K", ctypes.c_int), ("budget", ctypes.c_int),
        ("root_token", ctypes.c_void_p), ("cand_token", ctypes.c_void_p), ("cand_logp", ctypes.c_void_p),
        ("tree_parent", ctypes.c_void_p), ("tree_token", ctypes.c_void_p),
        ("tree_depth", ctypes.c_void_p), ("tree_score", ctypes.c_void_p),
    ]


class MlaDdtreeAcceptArgs(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("Q", ctypes.c_int),
        ("tree_parent", ctypes.c_void_p), ("tree_token", ctypes.c_void_p), ("target_token", ctypes.c_void_p),
        ("node_slot", ctypes.c_void_p),
        ("accept_len", ctypes.c_void_p), ("accept_nodes", ctypes.c_void_p), ("accept_slots", ctypes.c_void_p),
        ("next_token", ctypes.c_void_p),
    ]


class MlaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_str(status)}")


_lib = None


def load(path: Optional[str] = None):
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library not built: {p} (run __graft_entry__.build())")
    lib = ctypes.CDLL(p)
    lib.mla_verify_workspace_size.restype = ctypes.c_size_t
    lib.mla_verify_workspace_size.argtypes = [ctypes.POINTER(MlaVerifyArgs), ctypes.c_int]
    lib.mla_verify_attn.restype = ctypes.c_int
    lib.mla_verify_attn.argtypes = [ctypes.POINTER(MlaVerifyArgs), ctypes.c_void_p, ctypes.c_size_t,
                                    ctypes.c_int, ctypes.c_void_p]
    lib.mla_verify_attn_noalloc.restype = ctypes.c_int
    lib.mla_verify_attn_noalloc.argtypes = [ctypes.POINTER(MlaVerifyArgs), ctypes.c_int, ctypes.c_void_p]
    lib.mla_verify_noalloc_check.restype = ctypes.c_int
    lib.mla_verify_noalloc_check.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]
    lib.mla_verify_splits_used.restype = ctypes.c_int
    lib.mla_verify_splits_used.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]
    lib.mla_verify_build_meta.restype = ctypes.c_int
    lib.mla_verify_build_meta.argtypes = [ctypes.POINTER(MlaVerifyArgs), ctypes.c_void_p, ctypes.c_size_t,
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                          ctypes.c_void_p]
    lib.mla_verify_selftest_timeout.restype = ctypes.c_int
    lib.mla_verify_selftest_timeout.argtypes = [ctypes.POINTER(MlaVerifyArgs), ctypes.c_void_p, ctypes.c_size_t,
                                                ctypes.c_uint64, ctypes.c_void_p]
    lib.mla_kv_compact.restype = ctypes.c_int
    lib.mla_kv_compact.argtypes = [ctypes.POINTER(MlaVerifyArgs), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.mla_ddtree_build.restype = ctypes.c_int
    lib.mla_ddtree_build.argtypes = [ctypes.POINTER(MlaDdtreeBuildArgs), ctypes.c_void_p, ctypes.c_size_t,
                                     ctypes.c_void_p]
    lib.mla_ddtree_accept.restype = ctypes.c_int
    lib.mla_ddtree_accept.argtypes = [ctypes.POINTER(MlaDdtreeAcceptArgs), ctypes.c_void_p, ctypes.c_size_t,
                                      ctypes.c_void_p]
    lib.mla_verify_check.restype = ctypes.c_int
    lib.mla_verify_check.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]
    lib.mla_status_str.restype = ctypes.c_char_p
    lib.mla_status_str.argtypes = [ctypes.c_int]
    lib.mla_verify_abi_version.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def status_str(s: int) -> str:
    return load().mla_status_str(int(s)).decode()


# ----------------------------------------------------------------------------
# torch marshalling
# ----------------------------------------------------------------------------
def _ptr(t) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


@dataclass
class DeviceInputs:
    """Device tensors of one verify problem (see inputs.Problem)."""
    B: int
    Q: int
    H: int
    dtype: str
    scale: float
    q_lat: object
    q_pe: object
    kv_c: object            # [pool_slots, >=512] view (row stride = pool row)
    k_pe: object            # [pool_slots, >=64] view
    prefix_lens: object
    tree_parent: object
    page_size: int
    kv_indptr: object = None
    kv_indices: object = None
    block_table: object = None
    pool: object = None     # owning tensor of kv_c / k_pe

    @property
    def pool_slots(self) -> int:
        return int(self.kv_c.shape[0])

    def check(self):
        """What the C ABI cannot see from pointers: element types, shapes,
        layouts and the device of every tensor.  Raises ValueError."""
        self.check_layout()
        _on_cuda(**self.tensors())

    def tensors(self):
        return dict(q_lat=self.q_lat, q_pe=self.q_pe, kv_c=self.kv_c, k_pe=self.k_pe, prefix_lens=self.prefix_lens,
                    tree_parent=self.tree_parent, kv_indptr=self.kv_indptr, kv_indices=self.kv_indices,
                    block_table=self.block_table)

    def check_layout(self):
        import torch
        el = torch.bfloat16 if self.dtype == "bf16" else torch.float32
        B, Q, H = self.B, self.Q, self.H
        _need(self.q_lat, "q_lat", el, (B, Q, H, 512))
        _need(self.q_pe, "q_pe", el, (B, Q, H, 64))
        for t, name, w in ((self.kv_c, "kv_c", 512), (self.k_pe, "k_pe", 64)):
            if t is None or t.dtype != el or t.dim() != 2 or t.shape[1] != w or t.stride(1) != 1:
                raise ValueError(f"{name} must be a [slots][{w}] {el} view with unit column stride")
        if self.k_pe.shape[0] != self.kv_c.shape[0]:
            raise ValueError("kv_c and k_pe must cover the same pool slots")
        _need(self.prefix_lens, "prefix_lens", torch.int32, (B,))
        _need(self.tree_parent, "tree_parent", torch.int32, (B, Q))
        if self.page_size == 1:
            _need(self.kv_indptr, "kv_indptr", torch.int32, (B + 1,))
            if self.kv_indices is None or self.kv_indices.dtype != torch.int32 or self.kv_indices.dim() != 1 \
                    or not self.kv_indices.is_contiguous():
                raise ValueError("kv_indices must be a contiguous 1-D int32 tensor")
        else:
            if self.block_table is None or self.block_table.dtype != torch.int32 or self.block_table.dim() != 2 \
                    or self.block_table.shape[0] != B or not self.block_table.is_contiguous():
                raise ValueError("block_table must be a contiguous [B][max_pages] int32 tensor")


def device_inputs(problem, device="cuda", separate_pools: bool = False) -> DeviceInputs:
    """Copy a numpy inputs.Problem to the device (packed [slot][576] pool by
    default; separate kv_c / k_pe arrays with ``separate_pools``)."""
    import torch

    def t(x, dt=None):
        if x is None:
            return None
        a = np.ascontiguousarray(x)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
        tt = torch.from_numpy(a).to(device)
        return tt if dt is None else tt.to(dt)

    pool = t(problem.pool)
    if separate_pools:
        kv_c = pool[:, :512].contiguous()
        k_pe = pool[:, 512:].contiguous()
        owner = None
    else:
        kv_c, k_pe, owner = pool[:, :512], pool[:, 512:], pool
    return DeviceInputs(
        B=problem.B, Q=problem.Q, H=problem.H, dtype=problem.dtype, scale=problem.scale,
        q_lat=t(problem.q_lat), q_pe=t(problem.q_pe), kv_c=kv_c, k_pe=k_pe,
        prefix_lens=t(problem.prefix_lens.astype(np.int32)),
        tree_parent=t(problem.tree_parent.astype(np.int32)),
        page_size=problem.page_size,
        kv_indptr=t(problem.kv_indptr), kv_indices=t(problem.kv_indices),
        block_table=t(problem.block_table), pool=owner)


def make_args(di: DeviceInputs, out=None, lse=None, algo: str = "auto",
              profile_events=None, check: bool = True) -> MlaVerifyArgs:
    if check:
        import torch
        di.check_layout()
        odt = torch.bfloat16 if di.dtype == "bf16" else torch.float32
        if out is not None:
            _need(out, "out", odt, (di.B, di.Q, di.H, 512))
        if lse is not None:
            _need(lse, "lse", torch.float32, (di.B, di.Q, di.H))
        _on_cuda(out=out, lse=lse, **di.tensors())
    a = MlaVerifyArgs()
    a.B, a.Q, a.H = di.B, di.Q, di.H
    a.dtype = MLA_BF16 if di.dtype == "bf16" else MLA_FP32
    a.q_lat, a.q_pe = _ptr(di.q_lat), _ptr(di.q_pe)
    a.kv_c, a.k_pe = _ptr(di.kv_c), _ptr(di.k_pe)
    a.kv_c_stride = int(di.kv_c.stride(0))
    a.k_pe_stride = int(di.k_pe.stride(0))
    a.pool_slots = di.pool_slots
    a.page_size = di.page_size
    a.kv_indptr, a.kv_indices = _ptr(di.kv_indptr), _ptr(di.kv_indices)
    a.block_table = _ptr(di.block_table)
    a.max_pages = 0 if di.block_table is None else int(di.block_table.shape[1])
    a.prefix_lens, a.tree_parent = _ptr(di.prefix_lens), _ptr(di.tree_parent)
    a.scale = di.scale
    a.out, a.lse = _ptr(out), _ptr(lse)
    a.algo = ALGO[algo]
    if profile_events is not None:
        # keep the pointer array alive as long as the struct
        a._ev = (ctypes.c_void_p * 2)(int(profile_events[0].cuda_event), int(profile_events[1].cuda_event))
        a.profile_events = ctypes.cast(a._ev, ctypes.c_void_p)
    return a


def workspace_size(di: DeviceInputs, num_splits: int = 0, algo: str = "auto") -> int:
    a = make_args(di, algo=algo, check=False)
    n = load().mla_verify_workspace_size(ctypes.byref(a), int(num_splits))
    if n == 0 and di.B > 0 and di.Q > 0:
        raise MlaError(MLA_ERR_INVALID_ARG, "mla_verify_workspace_size")
    return int(n)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream))


def alloc_workspace(nbytes: int, device="cuda"):
    import torch
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def verify_attn(di: DeviceInputs, out=None, lse=None, num_splits: int = 0, algo: str = "auto",
                workspace=None, stream=None, profile_events=None, check: bool = True):
    """Run mla_verify_attn; returns (out [B,Q,H,512], lse [B,Q,H] fp32).
    check=False skips the tensor checks (a loop that already passed them)."""
    import torch
    dev = di.q_lat.device
    odt = torch.bfloat16 if di.dtype == "bf16" else torch.float32
    if out is None:
        out = torch.empty((di.B, di.Q, di.H, 512), dtype=odt, device=dev)
    if lse is None:
        lse = torch.empty((di.B, di.Q, di.H), dtype=torch.float32, device=dev)
    a = make_args(di, out, lse, algo, profile_events, check)
    lib = load()
    need = lib.mla_verify_workspace_size(ctypes.byref(a), int(num_splits))
    if workspace is None:
        workspace = alloc_workspace(need, dev)
    st = lib.mla_verify_attn(ctypes.byref(a), ctypes.c_void_p(_ptr(workspace)),
                             ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                             int(num_splits), _stream(stream))
    if st != MLA_OK:
        raise MlaError(st, "mla_verify_attn")
    return out, lse


def verify_attn_noalloc(di: DeviceInputs, out=None, lse=None, num_splits: int = 0, algo: str = "auto",
                        stream=None, check_device: bool = False):
    """Run mla_verify_attn_noalloc (library-held scratch, no workspace); returns
    (out, lse).  Output tensors are created here when not given -- the library
    call itself allocates nothing.  check_device=True synchronises the stream
    and raises MlaError(MLA_ERR_DEVICE_CHECK) when the device found bad table
    contents (noalloc_check)."""
    import torch
    dev = di.q_lat.device
    odt = torch.bfloat16 if di.dtype == "bf16" else torch.float32
    if out is None:
        out = torch.empty((di.B, di.Q, di.H, 512), dtype=odt, device=dev)
    if lse is None:
        lse = torch.empty((di.B, di.Q, di.H), dtype=torch.float32, device=dev)
    a = make_args(di, out, lse, algo)
    st = load().mla_verify_attn_noalloc(ctypes.byref(a), int(num_splits), _stream(stream))
    if st != MLA_OK:
        raise MlaError(st, "mla_verify_attn_noalloc")
    if check_device and noalloc_check(stream) != 0:
        raise MlaError(MLA_ERR_DEVICE_CHECK, "mla_verify_attn_noalloc")
    return out, lse


def noalloc_check(stream=None) -> int:
    """Synchronise and return the device error bits the last
    mla_verify_attn_noalloc call on the current device left."""
    bits = ctypes.c_uint32(0)
    st = load().mla_verify_noalloc_check(_stream(stream), ctypes.byref(bits))
    if st not in (MLA_OK, MLA_ERR_DEVICE_CHECK):
        raise MlaError(st, "mla_verify_noalloc_check")
    return int(bits.value)


def selftest_timeout(di: DeviceInputs, out, lse, workspace, hold_ns: int, stream=None):
    """Run mla_verify_selftest_timeout: the tensor-core call with one device
    wait that gives up after hold_ns; read the outcome with check()."""
    a = make_args(di, out, lse, "tc")
    st = load().mla_verify_selftest_timeout(ctypes.byref(a), ctypes.c_void_p(_ptr(workspace)),
                                            ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                                            ctypes.c_uint64(int(hold_ns)), _stream(stream))
    if st != MLA_OK:
        raise MlaError(st, "mla_verify_selftest_timeout")


def kv_compact(di: DeviceInputs, dst_pool, dst_slot0: int = 0, workspace=None, stream=None):
    """Run mla_kv_compact into ``dst_pool`` ([slots][576] of the cache dtype:
    kv_c columns 0-511, k_pe 512-575); returns (new_kv_indices [sum N_b] int32,
    new_kv_indptr [B+1] int32, workspace)."""
    import torch
    dev = di.q_lat.device
    a = make_args(di)
    lib = load()
    need = lib.mla_verify_workspace_size(ctypes.byref(a), 1)
    if workspace is None:
        workspace = alloc_workspace(need, dev)
    total = int((di.prefix_lens.to(torch.int64) + di.Q).sum().item())
    new_idx = torch.full((max(total, 1),), -1, dtype=torch.int32, device=dev)
    new_indptr = torch.zeros((di.B + 1,), dtype=torch.int32, device=dev)
    kv_compact_into(di, dst_pool, new_idx, new_indptr, workspace, dst_slot0, stream)
    return new_idx[:total], new_indptr, workspace


def kv_compact_into(di: DeviceInputs, dst_pool, new_idx, new_indptr, workspace, dst_slot0: int = 0, stream=None):
    """mla_kv_compact with caller-provided output tables (no host synchronisation)."""
    a = make_args(di)
    lib = load()
    st = lib.mla_kv_compact(ctypes.byref(a), ctypes.c_void_p(_ptr(workspace)),
                            ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                            ctypes.c_void_p(_ptr(dst_pool)), ctypes.c_void_p(_ptr(dst_pool[:, 512:])),
                            ctypes.c_int64(dst_pool.stride(0)), ctypes.c_int64(dst_pool.stride(0)),
                            ctypes.c_int64(dst_slot0), ctypes.c_int64(dst_pool.shape[0]),
                            ctypes.c_void_p(_ptr(new_idx)), ctypes.c_void_p(_ptr(new_indptr)), _stream(stream))
    if st != MLA_OK:
        raise MlaError(st, "mla_kv_compact")


def build_meta(di: DeviceInputs, workspace=None, stream=None):
    """Run mla_verify_build_meta; returns (anc [B,Q] uint64 as int64, slots [sum N_b] int32)."""
    import torch
    dev = di.q_lat.device
    a = make_args(di)
    lib = load()
    need = lib.mla_verify_workspace_size(ctypes.byref(a), 1)
    if workspace is None:
        workspace = alloc_workspace(need, dev)
    total = int((di.prefix_lens.to(torch.int64) + di.Q).sum().item())
    anc = torch.zeros((di.B, di.Q), dtype=torch.int64, device=dev)
    slots = torch.full((max(total, 1),), -7, dtype=torch.int32, device=dev)
    st = lib.mla_verify_build_meta(ctypes.byref(a), ctypes.c_void_p(_ptr(workspace)),
                                   ctypes.c_size_t(workspace.numel()), ctypes.c_void_p(_ptr(anc)),
                                   ctypes.c_void_p(_ptr(slots)), ctypes.c_int64(total), _stream(stream))
    if st != MLA_OK:
        raise MlaError(st, "mla_verify_build_meta")
    return anc, slots[:total], workspace


def check(workspace, stream=None) -> int:
    """Synchronise and return the device error bits of the last call on this workspace."""
    bits = ctypes.c_uint32(0)
    st = load().mla_verify_check(ctypes.c_void_p(_ptr(workspace)), _stream(stream), ctypes.byref(bits))
    if st not in (MLA_OK, MLA_ERR_DEVICE_CHECK):
        raise MlaError(st, "mla_verify_check")
    return int(bits.value)


def splits_used(workspace, stream=None) -> int:
    """Synchronise and return the split count the last verify_attn call on
    this workspace used (the library's choice when num_splits was 0)."""
    v = ctypes.c_int32(0)
    st = load().mla_verify_splits_used(ctypes.c_void_p(_ptr(workspace)), _stream(stream), ctypes.byref(v))
    if st != MLA_OK:
        raise MlaError(st, "mla_verify_splits_used")
    return int(v.value)



# ----------------------------------------------------------------------------
# DDTree construction and acceptance (include/mla_ddtree.h)
# ----------------------------------------------------------------------------
def _ws_bytes(workspace) -> int:
    return workspace.numel() * workspace.element_size()


def _need(t, name: str, dtype, shape):
    """The C ABI sees only a pointer: check what it cannot (dtype, shape,
    contiguity, device) before handing it over."""
    import torch
    if t is None:
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _on_cuda(**tensors):
    for name, t in tensors.items():
        if t is not None and t.device.type != "cuda":
            raise ValueError(f"{name} must be a CUDA tensor")


def _check_build(root_token, cand_token, cand_logp, B, L, K, Q, tree_parent, tree_token, tree_depth, tree_score,
                 workspace):
    import torch
    _need(cand_logp, "cand_logp", torch.float32, (B, L, K))
    _need(cand_token, "cand_token", torch.int32, (B, L, K))
    _need(root_token, "root_token", torch.int32, (B,))
    for t, name in ((tree_parent, "tree_parent"), (tree_token, "tree_token")):
        _need(t, name, torch.int32, (B, Q))
    if tree_depth is not None:
        _need(tree_depth, "tree_depth", torch.int32, (B, Q))
    if tree_score is not None:
        _need(tree_score, "tree_score", torch.float32, (B, Q))
    _on_cuda(cand_logp=cand_logp, cand_token=cand_token, root_token=root_token, tree_parent=tree_parent,
             tree_token=tree_token, tree_depth=tree_depth, tree_score=tree_score, workspace=workspace)


def _check_accept(tree_parent, tree_token, target_token, accept_len, accept_nodes, next_token, node_slot,
                  accept_slots, workspace, B, Q):
    import torch
    for t, name in ((tree_parent, "tree_parent"), (tree_token, "tree_token"), (target_token, "target_token"),
                    (accept_nodes, "accept_nodes")):
        _need(t, name, torch.int32, (B, Q))
    for t, name in ((accept_len, "accept_len"), (next_token, "next_token")):
        _need(t, name, torch.int32, (B,))
    if node_slot is not None:
        _need(node_slot, "node_slot", torch.int32, (B, Q))
    if accept_slots is not None:
        _need(accept_slots, "accept_slots", torch.int32, (B, Q))
    _on_cuda(tree_parent=tree_parent, tree_token=tree_token, target_token=target_token, accept_nodes=accept_nodes,
             accept_len=accept_len, next_token=next_token, node_slot=node_slot, accept_slots=accept_slots,
             workspace=workspace)


def ddtree_build_into(root_token, cand_token, cand_logp, budget: int, tree_parent, tree_token, workspace,
                      tree_depth=None, tree_score=None, stream=None, check: bool = True):
    """mla_ddtree_build into caller-provided [B][budget+1] outputs (no host
    synchronisation).  check=False skips the tensor checks, for a loop that
    passes tensors it has already passed once with checking on."""
    if cand_logp.dim() != 3:
        raise ValueError("cand_logp must be [B][L][K]")
    B, L, K = cand_logp.shape
    Q = int(budget) + 1
    if check:
        _check_build(root_token, cand_token, cand_logp, B, L, K, Q, tree_parent, tree_token, tree_depth, tree_score,
                     workspace)
    a = MlaDdtreeBuildArgs()
    a.B, a.L, a.K, a.budget = B, L, K, int(budget)
    a.root_token, a.cand_token, a.cand_logp = _ptr(root_token), _ptr(cand_token), _ptr(cand_logp)
    a.tree_parent, a.tree_token = _ptr(tree_parent), _ptr(tree_token)
    a.tree_depth, a.tree_score = _ptr(tree_depth), _ptr(tree_score)
    st = load().mla_ddtree_build(ctypes.byref(a), ctypes.c_void_p(_ptr(workspace)),
                                 ctypes.c_size_t(_ws_bytes(workspace)), _stream(stream))
    if st != MLA_OK:
        raise MlaError(st, "mla_ddtree_build")


def ddtree_build(root_token, cand_token, cand_logp, budget: int, workspace=None, stream=None):
    """Build the draft trees; inputs are device tensors [B] int32, [B][L][K] int32,
    [B][L][K] float32.  Returns (parent, token, depth, score) [B][budget+1] and the workspace."""
    import torch
    dev = cand_logp.device
    B = cand_logp.shape[0]
    Q = int(budget) + 1
    if workspace is None:
        workspace = alloc_workspace(DDTREE_WORKSPACE_BYTES, dev)
    parent = torch.full((B, Q), -7, dtype=torch.int32, device=dev)
    token = torch.full((B, Q), -7, dtype=torch.int32, device=dev)
    depth = torch.full((B, Q), -7, dtype=torch.int32, device=dev)
    score = torch.full((B, Q), float("nan"), dtype=torch.float32, device=dev)
    ddtree_build_into(root_token, cand_token, cand_logp, budget, parent, token, workspace, depth, score, stream)
    return parent, token, depth, score, workspace


def ddtree_accept_into(tree_parent, tree_token, target_token, accept_len, accept_nodes, next_token, workspace,
                       node_slot=None, accept_slots=None, stream=None, check: bool = True):
    """mla_ddtree_accept into caller-provided outputs (no host synchronisation);
    check as for ddtree_build_into."""
    if tree_parent.dim() != 2:
        raise ValueError("tree_parent must be [B][Q]")
    B, Q = tree_parent.shape
    if check:
        _check_accept(tree_parent, tree_token, target_token, accept_len, accept_nodes, next_token, node_slot,
                      accept_slots, workspace, B, Q)
    a = MlaDdtreeAcceptArgs()
    a.B, a.Q = B, Q
    a.tree_parent, a.tree_token, a.target_token = _ptr(tree_parent), _ptr(tree_token), _ptr(target_token)
    a.node_slot = _ptr(node_slot)
    a.accept_len, a.accept_nodes, a.accept_slots = _ptr(accept_len), _ptr(accept_nodes), _ptr(accept_slots)
    a.next_token = _ptr(next_token)
    st = load().mla_ddtree_accept(ctypes.byref(a), ctypes.c_void_p(_ptr(workspace)),
                                  ctypes.c_size_t(_ws_bytes(workspace)), _stream(stream))
    if st != MLA_OK:
        raise MlaError(st, "mla_ddtree_accept")


def ddtree_accept(tree_parent, tree_token, target_token, node_slot=None, workspace=None, stream=None):
    """Greedy acceptance; inputs are device int32 tensors [B][Q].  Returns
    (accept_len [B], accept_nodes [B][Q], next_token [B], accept_slots [B][Q] or None, workspace)."""
    import torch
    dev = tree_parent.device
    B, Q = tree_parent.shape
    if workspace is None:
        workspace = alloc_workspace(DDTREE_WORKSPACE_BYTES, dev)
    n_len = torch.full((B,), -7, dtype=torch.int32, device=dev)
    nodes = torch.full((B, Q), -7, dtype=torch.int32, device=dev)
    nxt = torch.full((B,), -7, dtype=torch.int32, device=dev)
    slots = None if node_slot is None else torch.full((B, Q), -7, dtype=torch.int32, device=dev)
    ddtree_accept_into(tree_parent, tree_token, target_token, n_len, nodes, nxt, workspace, node_slot, slots, stream)
    return n_len, nodes, nxt, slots, workspace
