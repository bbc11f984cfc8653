"""Seeded synthetic inputs for DDTree verify attention (MLA, absorbed form).

This module only draws inputs: queries, the latent KV pool, draft trees,
prefix lengths and the slot / page tables that place each sequence's tokens
in the pool.  It holds none of the attention arithmetic, so both the CUDA
path and the CPU oracle can be fed from it without sharing any part of the
method.

Shapes follow the workloads of "Ground Truth in Silicon: The Role of the
Python Reference in Custom CUDA Kernel Development" (section "The Message in
Full": a per-token latent ``kv_c`` of width 512 and a rope key ``k_pe`` of
width 64, shared by every head) and "The Critical Glue: Validating a Custom
Flash Attention Kernel Through Test Infrastructure" (section "The Context":
a 200k-token context whose KV lives at scattered page_size=1 slots).

Conventions (the plainest reading where the pages are silent):

* Logical positions of sequence ``b`` are ``0 .. N_b-1`` with
  ``N_b = prefix_len[b] + Q``; the committed prefix occupies ``0 .. P_b-1``
  and draft-tree node ``t`` sits at position ``P_b + t``.
* ``page_size == 1``: position ``p`` of sequence ``b`` lives at pool slot
  ``kv_indices[kv_indptr[b] + p]``.
* ``page_size > 1``: position ``p`` lives at slot
  ``block_table[b][p // page_size] * page_size + p % page_size``.
* N(0,1) draws are made in float64, rounded to float32, and for bf16
  workloads rounded again to bf16 (round to nearest, ties to even).
* A random draft tree draws ``parent[i]`` uniformly from ``[-1, i-1]`` and
  redraws while the node would sit deeper than the depth cap (a root has
  depth 1).  ``-1`` always satisfies the cap, so the draw terminates.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence

import numpy as np

DL = 512  # latent width (kv_lora_rank)
DR = 64   # decoupled rope key width (qk_rope_head_dim)
DK = DL + DR
DEFAULT_SCALE = 1.0 / math.sqrt(192.0)


# ----------------------------------------------------------------------------
# bf16 storage helpers (input preparation only)
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return the bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


_STORAGE = {"bf16": np.uint16, "fp32": np.float32, "fp64": np.float64}


def _normal_block(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float64)
    if dtype == "fp64":          # oracle-only pins
        return x
    x = x.astype(np.float32)
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    return x


def _normal_rows(rng: np.random.Generator, n_rows: int, width: int, dtype: str,
                 chunk: int = 16384) -> np.ndarray:
    out = np.empty((n_rows, width), dtype=_STORAGE[dtype])
    for r0 in range(0, n_rows, chunk):
        r1 = min(n_rows, r0 + chunk)
        out[r0:r1] = _normal_block(rng, (r1 - r0, width), dtype)
    return out


def random_tree(rng: np.random.Generator, q: int, depth_cap: int = 8) -> np.ndarray:
    """Draw a draft tree (forest) of ``q`` nodes in topological order."""
    parent = np.empty(q, dtype=np.int32)
    depth = np.zeros(q, dtype=np.int64)
    for i in range(q):
        while True:
            p = int(rng.integers(-1, i)) if i > 0 else -1   # uniform in [-1, i-1]
            d = 1 if p < 0 else int(depth[p]) + 1
            if d <= depth_cap:
                break
        parent[i] = p
        depth[i] = d
    return parent


# ----------------------------------------------------------------------------
# Problem container
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class Problem:
    name: str
    dtype: str                 # "bf16" or "fp32" ("fp64" only for oracle pins)
    B: int
    Q: int
    H: int
    scale: float
    prefix_lens: np.ndarray    # int32 [B]
    tree_parent: np.ndarray    # int32 [B, Q]
    q_lat: np.ndarray          # [B, Q, H, 512] (uint16 bf16 bits, or float32)
    q_pe: np.ndarray           # [B, Q, H, 64]
    pool: np.ndarray           # [pool_slots, 576]: kv_c in columns 0..511, k_pe in 512..575
    page_size: int
    kv_indptr: Optional[np.ndarray] = None    # int32 [B+1]   (page_size == 1)
    kv_indices: Optional[np.ndarray] = None   # int32 [sum N_b] (page_size == 1)
    block_table: Optional[np.ndarray] = None  # int32 [B, max_pages] (page_size > 1)
    seed: int = 0
    notes: str = ""

    @property
    def pool_slots(self) -> int:
        return int(self.pool.shape[0])

    @property
    def rows_per_seq(self) -> int:
        return self.H * self.Q

    @property
    def n_rows(self) -> int:
        return self.B * self.H * self.Q

    @property
    def kv_lens(self) -> np.ndarray:
        return (self.prefix_lens.astype(np.int64) + self.Q)

    @property
    def max_pages(self) -> int:
        return 0 if self.block_table is None else int(self.block_table.shape[1])

    def slot_of(self, b: int, p: int) -> int:
        """Pool slot of logical position ``p`` of sequence ``b`` (table lookup)."""
        if self.page_size == 1:
            return int(self.kv_indices[int(self.kv_indptr[b]) + p])
        ps = self.page_size
        return int(self.block_table[b, p // ps]) * ps + p % ps

    def kv_bytes_touched(self) -> int:
        el = 2 if self.dtype == "bf16" else 4
        return int(self.kv_lens.sum()) * DK * el


# ----------------------------------------------------------------------------
# Builders
# ----------------------------------------------------------------------------
def make_problem(*, name: str, dtype: str, B: int, H: int, Q: int,
                 prefix_lens: Sequence[int], seed: int,
                 trees: Optional[Sequence[Sequence[int]]] = None,
                 depth_cap: int = 8,
                 layout: str = "contiguous",   # "contiguous" | "scattered" | "paged"
                 pool_slots: Optional[int] = None,
                 page_size: int = 1,
                 n_pages: Optional[int] = None,
                 scale: float = DEFAULT_SCALE) -> Problem:
    rng = np.random.default_rng(seed)
    prefix = np.asarray(prefix_lens, dtype=np.int32).reshape(B)
    if trees is None:
        parent = np.stack([random_tree(rng, Q, depth_cap) for _ in range(B)]) if Q > 0 \
            else np.zeros((B, 0), dtype=np.int32)
    else:
        parent = np.asarray(trees, dtype=np.int32).reshape(B, Q)
    n = prefix.astype(np.int64) + Q

    kv_indptr = kv_indices = block_table = None
    if layout in ("contiguous", "scattered"):
        assert page_size == 1
        total = int(n.sum())
        if pool_slots is None:
            pool_slots = total
        assert pool_slots >= total
        kv_indptr = np.zeros(B + 1, dtype=np.int32)
        kv_indptr[1:] = np.cumsum(n)
        if layout == "contiguous":
            kv_indices = np.arange(total, dtype=np.int32)
        else:
            perm = rng.permutation(pool_slots).astype(np.int32)
            kv_indices = perm[:total].copy()
    elif layout == "paged":
        assert page_size > 1
        pages_per_seq = [int(math.ceil(int(x) / page_size)) for x in n]
        max_pages = max(pages_per_seq) if pages_per_seq else 0
        if n_pages is None:
            n_pages = sum(pages_per_seq)
        assert n_pages >= sum(pages_per_seq)
        perm = rng.permutation(n_pages).astype(np.int32)
        block_table = np.full((B, max(max_pages, 1)), -1, dtype=np.int32)
        off = 0
        for b, k in enumerate(pages_per_seq):
            block_table[b, :k] = perm[off:off + k]
            off += k
        pool_slots = n_pages * page_size
    else:
        raise ValueError(layout)

    q_lat = _normal_rows(rng, B * Q * H, DL, dtype).reshape(B, Q, H, DL)
    q_pe = _normal_rows(rng, B * Q * H, DR, dtype).reshape(B, Q, H, DR)
    pool = _normal_rows(rng, int(pool_slots), DK, dtype)
    return Problem(name=name, dtype=dtype, B=B, Q=Q, H=H, scale=float(scale),
                   prefix_lens=prefix, tree_parent=parent.astype(np.int32),
                   q_lat=q_lat, q_pe=q_pe, pool=pool, page_size=page_size,
                   kv_indptr=kv_indptr, kv_indices=kv_indices,
                   block_table=block_table, seed=seed)


TINY_TREE = [-1, 0, 1, 1, 2, 3, 4, 4]


def make_config(name: str, seed: Optional[int] = None) -> Problem:
    """The five workloads: tiny fp32, and four bf16 shapes up to a 200k prefix.

    ``tiny``  B=1 H=16 prefix 256, fixed 8-node tree, fp32, contiguous slots.
    ``c2``    B=1 H=64 prefix 4096, random 64-node tree, bf16, contiguous.
    ``c3``    B=1 H=64 prefix 200,000, 64-node tree, bf16, page_size=1 slots
              drawn from a seeded permutation of a 262,144-slot pool.
    ``c4``    B=8 H=64 prefix ~U[1024, 32768], 32-node trees, bf16, disjoint
              page_size=1 slots in a shared 393,216-slot pool.
    ``c5``    B=32 H=128 prefix 8192, 16-node trees, bf16, page_size=64 with
              pages permuted in a 4,200-page pool.
    ``c6``    B=1 H=64 prefix 200,000, a 4-node chain (a linear draft), bf16,
              page_size=1 slots as in c3: 256 query rows, the regime where the
              KV read, not the products, bounds the call.
    """
    if name == "tiny":
        p = make_problem(name=name, dtype="fp32", B=1, H=16, Q=8, prefix_lens=[256],
                         seed=0 if seed is None else seed, trees=[TINY_TREE])
    elif name == "c2":
        p = make_problem(name=name, dtype="bf16", B=1, H=64, Q=64, prefix_lens=[4096],
                         seed=1 if seed is None else seed)
    elif name == "c3":
        p = make_problem(name=name, dtype="bf16", B=1, H=64, Q=64, prefix_lens=[200000],
                         seed=2 if seed is None else seed, layout="scattered",
                         pool_slots=262144)
    elif name == "c4":
        s = 3 if seed is None else seed
        lens = np.random.default_rng(s + 1000).integers(1024, 32768, size=8, endpoint=True)
        p = make_problem(name=name, dtype="bf16", B=8, H=64, Q=32, prefix_lens=lens,
                         seed=s, layout="scattered", pool_slots=393216)
    elif name == "c5":
        p = make_problem(name=name, dtype="bf16", B=32, H=128, Q=16, prefix_lens=[8192] * 32,
                         seed=4 if seed is None else seed, layout="paged", page_size=64,
                         n_pages=4200)
    elif name == "c6":
        p = make_problem(name=name, dtype="bf16", B=1, H=64, Q=4, prefix_lens=[200000],
                         seed=5 if seed is None else seed, layout="scattered", pool_slots=262144,
                         trees=[[-1, 0, 1, 2]])
    else:
        raise ValueError(f"unknown workload {name!r}")
    return p


CONFIG_NAMES = ("tiny", "c2", "c3", "c4", "c5", "c6")


# ----------------------------------------------------------------------------
# Needles: a few keys planted so the softmax peaks on known tokens
# ----------------------------------------------------------------------------
def plant_needles(p: Problem, seed: int = 99, n_prefix: int = 3, strength: float = 40.0,
                  q_bias: float = 8.0) -> Dict[int, List[int]]:
    """Bias every query of a sequence toward a shared direction ``u`` and write
    keys ``strength*u + noise`` at ``n_prefix`` random prefix positions and at
    one random draft-tree node.  Rows then put most of their softmax weight on
    those tokens, so a gather from a wrong slot or a wrong tail mask moves the
    output by O(1) instead of hiding under a near-uniform average.

    Edits ``p`` in place; returns {b: [positions planted]}.
    """
    rng = np.random.default_rng(seed)
    planted: Dict[int, List[int]] = {}
    for b in range(p.B):
        u = rng.standard_normal(DL)
        u /= np.linalg.norm(u)
        if p.dtype == "bf16":
            ql = bf16_bits_to_f32(p.q_lat[b]).astype(np.float64)
        else:
            ql = p.q_lat[b].astype(np.float64)
        ql = ql + q_bias * u
        ql32 = ql.astype(np.float32)
        p.q_lat[b] = f32_to_bf16_bits(ql32) if p.dtype == "bf16" else ql32
        P = int(p.prefix_lens[b])
        pos = []
        if P > 0:
            k = min(n_prefix, P)
            pos += [int(x) for x in rng.choice(P, size=k, replace=False)]
        if p.Q > 0:
            pos.append(P + int(rng.integers(0, p.Q)))
        for pp in pos:
            v = strength * u + 0.5 * rng.standard_normal(DL)
            row = np.concatenate([v, rng.standard_normal(DR)]).astype(np.float32)
            p.pool[p.slot_of(b, pp)] = f32_to_bf16_bits(row) if p.dtype == "bf16" else row
        planted[b] = pos
    p.notes += " needles"
    return planted


# ----------------------------------------------------------------------------
# Row subsets for sampled parity at full size
# ----------------------------------------------------------------------------
def sample_rows(p: Problem, heads_per_node: int, seed: int = 7) -> np.ndarray:
    """Every (b, node) with ``heads_per_node`` seeded heads each.

    Returns int32 [n, 3] of (b, i, h), sorted.
    """
    rng = np.random.default_rng(seed)
    out = []
    k = min(heads_per_node, p.H)
    for b in range(p.B):
        for i in range(p.Q):
            for h in sorted(rng.choice(p.H, size=k, replace=False)):
                out.append((b, i, int(h)))
    return np.asarray(out, dtype=np.int32).reshape(-1, 3)


def all_rows(p: Problem) -> np.ndarray:
    b, i, h = np.meshgrid(np.arange(p.B), np.arange(p.Q), np.arange(p.H), indexing="ij")
    return np.stack([b.ravel(), i.ravel(), h.ravel()], axis=1).astype(np.int32)
