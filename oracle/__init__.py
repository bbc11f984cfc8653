"""CPU float64 oracle for DDTree verify attention (MLA, absorbed form).

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers.  Nothing in the CUDA
library or its Python binding imports this package, and this package imports
nothing from them.

The arithmetic lives in ``mla_oracle.c`` (plain C, float64, OpenMP across
rows); this module compiles it with gcc and marshals numpy arrays into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "mla_oracle.c")
LIB_DIR = os.path.join(_HERE, "lib")
LIB = os.path.join(LIB_DIR, "libmla_oracle.so")

DL, DR = 512, 64
_DTYPE = {"bf16": 0, "fp32": 1, "fp64": 2}


class OracleProblem(ctypes.Structure):
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
        ("scale", ctypes.c_double),
    ]


def build(src: str = SRC, out: str = LIB, extra_flags=()) -> str:
    """Compile the oracle into a shared library (gcc, -O2, OpenMP)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11",
           *extra_flags, src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


class Oracle:
    """ctypes handle on one build of the oracle library."""

    def __init__(self, lib_path: Optional[str] = None):
        path = lib_path or LIB
        if lib_path is None and (not os.path.exists(path) or
                                 os.path.getmtime(path) < os.path.getmtime(SRC)):
            build()
        self.lib = ctypes.CDLL(path)
        self.lib.oracle_tree_anc.restype = ctypes.c_int
        self.lib.oracle_tree_anc.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                             ctypes.c_void_p]
        self.lib.oracle_resolve_slots.restype = ctypes.c_int64
        self.lib.oracle_resolve_slots.argtypes = [ctypes.POINTER(OracleProblem), ctypes.c_void_p]
        self.lib.oracle_verify_rows.restype = ctypes.c_int
        self.lib.oracle_verify_rows.argtypes = [ctypes.POINTER(OracleProblem), ctypes.c_int,
                                                ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_void_p, ctypes.c_void_p]
        self.lib.oracle_num_threads.restype = ctypes.c_int

    # -- a1 -----------------------------------------------------------------
    def tree_anc(self, tree_parent: np.ndarray) -> np.ndarray:
        tp = np.ascontiguousarray(tree_parent, dtype=np.int32)
        B, Q = tp.shape
        anc = np.zeros((B, Q), dtype=np.uint64)
        rc = self.lib.oracle_tree_anc(B, Q, tp.ctypes.data, anc.ctypes.data)
        if rc != 0:
            raise ValueError("invalid tree")
        return anc

    # -- problem marshalling --------------------------------------------------
    def _problem(self, p, keep: list) -> OracleProblem:
        def arr(x, dt=None):
            if x is None:
                return None
            a = np.ascontiguousarray(x if dt is None else x.astype(dt, copy=False))
            keep.append(a)
            return a.ctypes.data

        pool = np.ascontiguousarray(p.pool)
        keep.append(pool)
        width = pool.shape[1]
        el = pool.itemsize
        pr = OracleProblem()
        pr.B, pr.Q, pr.H = p.B, p.Q, p.H
        pr.dtype = _DTYPE[p.dtype]
        pr.q_lat = arr(p.q_lat)
        pr.q_pe = arr(p.q_pe)
        pr.kv_c = pool.ctypes.data
        pr.k_pe = pool.ctypes.data + DL * el
        pr.kv_c_stride = width
        pr.k_pe_stride = width
        pr.pool_slots = pool.shape[0]
        pr.page_size = p.page_size
        pr.kv_indptr = arr(p.kv_indptr, np.int32)
        pr.kv_indices = arr(p.kv_indices, np.int32)
        pr.block_table = arr(p.block_table, np.int32)
        pr.max_pages = p.max_pages
        pr.prefix_lens = arr(p.prefix_lens, np.int32)
        pr.tree_parent = arr(p.tree_parent, np.int32)
        pr.scale = p.scale
        return pr

    # -- a2 -----------------------------------------------------------------
    def resolve_slots(self, p) -> np.ndarray:
        keep: list = []
        pr = self._problem(p, keep)
        total = int(p.kv_lens.sum())
        slots = np.zeros(total + 1, dtype=np.int32)
        n = self.lib.oracle_resolve_slots(ctypes.byref(pr), slots.ctypes.data)
        if n < 0:
            raise ValueError("slot table entry out of range")
        return slots[:n]

    # -- a3..a9 (the definition) ----------------------------------------------
    def verify_rows(self, p, rows: np.ndarray):
        """Return (out [n, 512] f64, lse [n] f64, n_visible [n] i64) for rows (b, i, h)."""
        keep: list = []
        pr = self._problem(p, keep)
        rows = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 3)
        n = rows.shape[0]
        out = np.zeros((n, DL), dtype=np.float64)
        lse = np.zeros(n, dtype=np.float64)
        nvis = np.zeros(n, dtype=np.int64)
        rc = self.lib.oracle_verify_rows(ctypes.byref(pr), n, rows.ctypes.data,
                                         out.ctypes.data, lse.ctypes.data, nvis.ctypes.data)
        if rc != 0:
            raise ValueError("oracle rejected the problem")
        return out, lse, nvis

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())


_default: Optional[Oracle] = None


def get() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
