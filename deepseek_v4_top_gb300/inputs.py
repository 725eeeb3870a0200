"""Seeded synthetic inputs for top-k sparse attention.

This module only draws numbers: it holds none of the attention arithmetic.
Both the CPU oracle (via the tests and the bench's CPU leg) and the CUDA path
consume exactly the arrays produced here, so the two sides see identical
bits.

Shapes follow the DeepSeek-V4.1 sparse-attention pages: 64 heads in total
(TensorFold PR #1206, "What changes", 16 heads a rank at world 4), a latent
KV row of 512 values processed as sixteen 32-wide column groups (akol1
TensorFold PR #4, first commit message), k = 640 selected keys (same PR,
second commit message: "exact sums at k 640"), 2048-row prefill segments and
4096 / 32K caches (PR #1206, flashosophy's runs).  No dataset is involved;
the pages' own workloads are whole-model prompts on weights that are not
available, and these synthetic arrays stand in for them.

Conventions
-----------
* ``q``    : [R, H, 512]  float32 array, or uint16 array of bf16 bits.
* ``kv``   : prefill [N, 512], decode [B, N, 512] (slot b is row b's cache).
* ``idx``  : int32 [R, k_max]; entries at and beyond ``n_sel[r]`` hold the
             poison value -1 and must never be used.
* ``n_sel``: int32 [R].
* ``sink`` : float32 [H].
* ``scale``: python float (1/sqrt(512) unless a case says otherwise).

bf16 values are produced by round-to-nearest-even from float32 draws.
"""

from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import math
from typing import List, Optional

import numpy as np

D = 512
POISON = -1
SEED_BASE = 0xD5A0

F32 = "f32"
BF16 = "bf16"

BF16_NAN = 0x7FC0
BF16_PINF = 0x7F80
BF16_NINF = 0xFF80


# --------------------------------------------------------------------------
# bf16 helpers (bit conversions only)
# --------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); NaN stays a quiet NaN."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = ((u[nan] >> np.uint32(16)) | np.uint32(0x40)).astype(np.uint16)
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------
# Case container
# --------------------------------------------------------------------------
@dataclasses.dataclass
class Case:
    name: str
    mode: str            # "decode" or "prefill"
    dtype: str           # "f32" or "bf16"
    R: int               # query rows (decode: slots B)
    H: int
    N: int               # cache positions (per slot in decode)
    k_max: int
    q: np.ndarray
    kv: np.ndarray
    idx: np.ndarray
    n_sel: np.ndarray
    sink: np.ndarray
    scale: float
    note: str = ""
    rows_per_slot: int = 1   # decode: query rows sharing a slot (row r reads slot r // rows_per_slot)

    @property
    def B(self) -> int:
        """Slots of a decode case (rows of a prefill case)."""
        return self.R // self.rows_per_slot if self.mode == "decode" else self.R

    def as_f32(self, a: np.ndarray) -> np.ndarray:
        """Input array widened to float32 (exact for bf16 bits)."""
        return bf16_bits_to_f32(a) if self.dtype == BF16 else a

    def kv_rows_of(self, r: int) -> np.ndarray:
        """The cache that row r selects from (widened to float32)."""
        base = self.kv[r // self.rows_per_slot] if self.mode == "decode" else self.kv
        return self.as_f32(base)

    def gathered_bytes(self) -> int:
        esz = 2 if self.dtype == BF16 else 4
        return int(np.clip(self.n_sel, 0, self.k_max).sum()) * D * esz


# --------------------------------------------------------------------------
# Drawing primitives
# --------------------------------------------------------------------------
def _normal(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    return f32_to_bf16_bits(x) if dtype == BF16 else x


def _normal_parallel(seed_seq: np.random.SeedSequence, n_blocks: int, block_shape,
                     dtype: str) -> np.ndarray:
    """Draw n_blocks independent blocks, each from its own child generator.

    The result does not depend on thread scheduling: block i always comes
    from child i of ``seed_seq``.
    """
    children = seed_seq.spawn(n_blocks)
    esz = np.uint16 if dtype == BF16 else np.float32
    out = np.empty((n_blocks,) + tuple(block_shape), dtype=esz)

    def work(i):
        out[i] = _normal(np.random.default_rng(children[i]), block_shape, dtype)

    with _cf.ThreadPoolExecutor(max_workers=min(16, n_blocks)) as ex:
        list(ex.map(work, range(n_blocks)))
    return out


def _distinct(rng: np.random.Generator, n: int, k: int) -> np.ndarray:
    return rng.choice(n, size=k, replace=False).astype(np.int32)


def _empty_idx(R: int, k_max: int) -> np.ndarray:
    return np.full((R, k_max), POISON, dtype=np.int32)


# --------------------------------------------------------------------------
# The five workload configurations
# --------------------------------------------------------------------------
def tiny(seed: Optional[int] = None, mode: str = "prefill") -> Case:
    """2 query rows, 8 heads, fp32, a 256-position cache, k = 64 distinct."""
    rng = np.random.default_rng(SEED_BASE + 0 if seed is None else seed)
    R, H, N, k = 2, 8, 256, 64
    q = _normal(rng, (R, H, D), F32)
    kv = _normal(rng, (R, N, D) if mode == "decode" else (N, D), F32)
    idx = _empty_idx(R, k)
    for r in range(R):
        idx[r] = _distinct(rng, N, k)
    sink = rng.standard_normal(H, dtype=np.float32)
    return Case("tiny", mode, F32, R, H, N, k, q, kv, idx,
                np.full(R, k, np.int32), sink, 1.0 / math.sqrt(D))


def single_decode(seed: Optional[int] = None) -> Case:
    """One decode row: 64 heads, bf16, 4096 positions, 640 sorted distinct keys."""
    rng = np.random.default_rng(SEED_BASE + 1 if seed is None else seed)
    R, H, N, k = 1, 64, 4096, 640
    q = _normal(rng, (R, H, D), BF16)
    kv = _normal(rng, (R, N, D), BF16)
    idx = _empty_idx(R, k)
    idx[0] = np.sort(_distinct(rng, N, k))
    sink = rng.standard_normal(H, dtype=np.float32)
    return Case("single_decode", "decode", BF16, R, H, N, k, q, kv, idx,
                np.full(R, k, np.int32), sink, 1.0 / math.sqrt(D))


def batched_decode(seed: Optional[int] = None, B: int = 8, N: int = 32768) -> Case:
    """B slots x 1 row, 64 heads, bf16, each slot its own N-position cache, k = 640."""
    s = SEED_BASE + 2 if seed is None else seed
    rng = np.random.default_rng(s)
    H, k = 64, 640
    q = _normal(rng, (B, H, D), BF16)
    idx = _empty_idx(B, k)
    for b in range(B):
        idx[b] = _distinct(rng, N, k)
    sink = rng.standard_normal(H, dtype=np.float32)
    kv = _normal_parallel(np.random.SeedSequence([s, 1]), B, (N, D), BF16)
    return Case("batched_decode", "decode", BF16, B, H, N, k, q, kv, idx,
                np.full(B, k, np.int32), sink, 1.0 / math.sqrt(D))


def prefill(seed: Optional[int] = None, rows: int = 2048, N: int = 4096,
            first_pos: Optional[int] = None) -> Case:
    """Causal prefill segment: rows at positions first_pos.. of an N-position cache.

    A row at position p selects min(p+1, 640) distinct positions in [0, p]:
    the top-k of fresh N(0,1) scores, kept in descending-score order (the
    order an indexer emits).
    """
    s = SEED_BASE + 3 if seed is None else seed
    rng = np.random.default_rng(s)
    H, k = 64, 640
    p0 = N - rows if first_pos is None else first_pos
    q = _normal_parallel(np.random.SeedSequence([s, 1]), rows, (H, D), BF16)
    kv = _normal(rng, (N, D), BF16)
    idx = _empty_idx(rows, k)
    n_sel = np.zeros(rows, np.int32)
    for i in range(rows):
        p = p0 + i
        m = min(p + 1, k)
        sc = rng.standard_normal(p + 1, dtype=np.float32)
        top = np.argpartition(-sc, m - 1)[:m] if m < p + 1 else np.arange(p + 1)
        top = top[np.argsort(-sc[top], kind="stable")]
        idx[i, :m] = top.astype(np.int32)
        n_sel[i] = m
    sink = rng.standard_normal(H, dtype=np.float32)
    return Case("prefill", "prefill", BF16, rows, H, N, k, q, kv, idx, n_sel,
                sink, 1.0 / math.sqrt(D))


def multi_row_decode(seed: Optional[int] = None, B: int = 8, T: int = 2, N: int = 32768,
                     k: int = 640, dtype: str = BF16, H: int = 64) -> Case:
    """Decode with T query rows a slot (a step's draft tokens verified together).

    Slot b's rows b*T .. b*T+T-1 read cache kv[b].  Row 0 of a slot selects k
    distinct random positions; each later row of the slot keeps about 90% of
    them and replaces the rest with other positions, so the rows' selections
    overlap as those of neighbouring tokens do.
    """
    s = SEED_BASE + 7 if seed is None else seed
    rng = np.random.default_rng(s)
    R = B * T
    q = _normal(rng, (R, H, D), dtype)
    kv = _normal(rng, (B, N, D), dtype)
    idx = _empty_idx(R, k)
    for b in range(B):
        base = _distinct(rng, N, k)
        for t in range(T):
            row = base.copy()
            if t > 0:
                swap = rng.random(k) < 0.1
                fresh = np.setdiff1d(_distinct(rng, N, min(N, 2 * k)), base)[:int(swap.sum())]
                row[np.nonzero(swap)[0][:len(fresh)]] = fresh
            idx[b * T + t] = row
    sink = rng.standard_normal(H, dtype=np.float32)
    return Case("multi_row_decode", "decode", dtype, R, H, N, k, q, kv, idx,
                np.full(R, k, np.int32), sink, 1.0 / math.sqrt(D), rows_per_slot=T)


def indexer_scores(mode: str = "prefill", seed: Optional[int] = None, rows: Optional[int] = None,
                   N: Optional[int] = None):
    """Index scores for the top-k selection: N(0,1) float32 per (row, position).

    prefill: 2048 rows at positions N-2048 .. N-1 of an N = 4096 cache; row i
    has n_valid = p + 1 candidates (its causal prefix).  decode: 8 rows, each
    over its own 32768-position cache (n_valid = N).  Returns
    (scores [rows, N], n_valid [rows]).
    """
    s = SEED_BASE + (5 if mode == "prefill" else 6) if seed is None else seed
    rng = np.random.default_rng(s)
    if mode == "prefill":
        rows = 2048 if rows is None else rows
        N = 4096 if N is None else N
        n_valid = (np.arange(rows) + (N - rows) + 1).astype(np.int32)
    else:
        rows = 8 if rows is None else rows
        N = 32768 if N is None else N
        n_valid = np.full(rows, N, np.int32)
    scores = rng.standard_normal((rows, N), dtype=np.float32)
    return scores, n_valid


EDGE_HEADS = (16, 32, 64)
EDGE_KS = (1, 7, 63, 64, 65, 127, 640)
EDGE_SPECIALS = ("q_nan", "q_pinf", "q_ninf", "kv_nan", "kv_pinf", "kv_ninf",
                 "unselected_nan", "sink_ninf", "sink_zero")


def _edge_base(rng, name, dtype, H, k, mode, R=None, N=None, k_extra=None) -> Case:
    R = int(rng.integers(1, 4)) if R is None else R
    N = int(rng.integers(max(64, k), 8193)) if N is None else N
    k_extra = int(rng.integers(0, 3)) if k_extra is None else k_extra
    k_max = k + k_extra
    q = _normal(rng, (R, H, D), dtype)
    kv = _normal(rng, (R, N, D) if mode == "decode" else (N, D), dtype)
    idx = _empty_idx(R, k_max)
    n_sel = np.zeros(R, np.int32)
    for r in range(R):
        # ragged rows: the last rows of a multi-row case select fewer keys
        m = k if r == 0 else max(1, k - r * (k // 3 + 1))
        idx[r, :m] = _distinct(rng, N, m)
        n_sel[r] = m
    sink = rng.standard_normal(H, dtype=np.float32)
    return Case(name, mode, dtype, R, H, N, k_max, q, kv, idx, n_sel, sink,
                1.0 / math.sqrt(D))


def _put(case: Case, arr: np.ndarray, where, kind: str):
    if case.dtype == BF16:
        arr[where] = {"nan": BF16_NAN, "pinf": BF16_PINF, "ninf": BF16_NINF}[kind]
    else:
        arr[where] = {"nan": np.nan, "pinf": np.inf, "ninf": -np.inf}[kind]


def edge_special(name: str, seed: int) -> Case:
    """One of the nine special edge cases (nonfinite injection, sink extremes)."""
    rng = np.random.default_rng(seed)
    i = EDGE_SPECIALS.index(name)
    dtype = BF16 if i % 2 == 0 else F32
    mode = "decode" if i % 3 == 0 else "prefill"
    c = _edge_base(rng, "edge_" + name, dtype, 32, 65, mode, R=2, N=512, k_extra=1)
    kvr = (lambda r: c.kv[r]) if mode == "decode" else (lambda r: c.kv)
    if name.startswith("q_"):
        _put(c, c.q, (0, 3, 17), name[2:])
        _put(c, c.q, (1, 30, 500), name[2:])
    elif name.startswith("kv_"):
        # a row selected by row 0 (its 10th pick) and one selected by row 1
        _put(c, kvr(0), (int(c.idx[0, 10]), 40), name[3:])
        _put(c, kvr(1), (int(c.idx[1, 64]), 7), name[3:])
    elif name == "unselected_nan":
        for r in range(c.R):
            rows = np.ones(c.N, bool)
            sel = c.idx[r, :c.n_sel[r]]
            if mode == "prefill":
                for rr in range(c.R):
                    rows[c.idx[rr, :c.n_sel[rr]]] = False
            else:
                rows[sel] = False
            _put(c, kvr(r), (rows, slice(None)), "nan")
    elif name == "sink_ninf":
        c.sink[:] = -np.inf
    elif name == "sink_zero":
        c.sink[:] = 0.0
    c.note = name
    return c


def edge_sweep(seed: int = SEED_BASE + 4) -> List[Case]:
    """The 51-shape edge sweep: 42 ordinary shapes plus 9 special cases."""
    rng = np.random.default_rng(seed)
    cases = []
    n = 0
    for dtype in (F32, BF16):
        for H in EDGE_HEADS:
            for k in EDGE_KS:
                mode = "decode" if n % 2 == 0 else "prefill"
                cases.append(_edge_base(rng, f"edge_{dtype}_h{H}_k{k}", dtype, H, k, mode))
                n += 1
    for j, name in enumerate(EDGE_SPECIALS):
        cases.append(edge_special(name, seed * 131 + j))
    return cases


# --------------------------------------------------------------------------
# Extra structured cases (test-only shapes)
# --------------------------------------------------------------------------
def rising_scores(seed: int = 77, dtype: str = BF16, mode: str = "prefill", k: int = 640,
                  H: int = 64, step: float = 32.0) -> Case:
    """Scores that climb by a large step from one 128-key block to the next.

    Every head gets q[h, 0] = 4 and the key at selection position j gets
    kv[., 0] = step * (j // 128), so each later block of selected keys
    scores about 4*step*scale higher than the one before: a running-max
    softmax must rescale what it has accumulated.
    """
    rng = np.random.default_rng(seed)
    c = _edge_base(rng, "rising_scores", dtype, H, k, mode, R=2, N=max(1024, 2 * k), k_extra=0)
    c.n_sel[:] = k
    # the two rows select disjoint keys, so a shared (prefill) cache keeps
    # each row's ramp intact
    both = _distinct(rng, c.N, 2 * k)
    c.idx[0, :k] = both[:k]
    c.idx[1, :k] = both[k:]
    four = f32_to_bf16_bits(np.float32([4.0]))[0] if dtype == BF16 else np.float32(4.0)
    c.q[:, :, 0] = four
    for r in range(c.R):
        cache = c.kv[r] if mode == "decode" else c.kv
        for j in range(k):
            v = np.float32(step * (j // 128))
            cache[c.idx[r, j], 0] = f32_to_bf16_bits(np.float32([v]))[0] if dtype == BF16 else v
    c.note = "rising block maxima"
    return c


def config(cid: int, **kw):
    """The workload configurations by number (1-based, as listed in the spec)."""
    return {1: tiny, 2: single_decode, 3: batched_decode, 4: prefill}[cid](**kw)
