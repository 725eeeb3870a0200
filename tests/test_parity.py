"""GPU parity: the C-ABI kernels against the fp64 oracle, element by element.

Tolerances (stated for the workload): fp32 inputs |g-o| <= 1e-6 + 1e-5|o|;
bf16 inputs |g-o| <= 3e-3 * max|o| over the (row, head).  Nonfinite classes
must match exactly.  Guards of 4 KiB around every output must be untouched
and the device error word must stay 0 for valid inputs (the pages' kernel
contract gates: nonfinite classes against float64, five byte-identical
repeats with untouched guards, exact sums at k 640 -- akol1 TensorFold PR #4,
second commit message; the 51-shape sweep -- first commit message).
"""

import math

import numpy as np
import pytest

import oracle
from deepseek_v4_top_gb300 import inputs as I

from gpu_helpers import compare, run, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    import torch
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)


def _check_full(case):
    got, code = run(case)
    assert code == 0, "device error word %#x" % code
    ref, _ = oracle.attn(case)
    return compare(case, got, ref)


@pytest.mark.parametrize("mode", ["decode", "prefill"])
def test_tiny_fp32(mode):
    _check_full(I.tiny(mode=mode))


def test_single_decode_row():
    _check_full(I.single_decode())


def test_batched_decode_full_size():
    """8 slots x 32768 positions, k = 640: every output against the oracle."""
    _check_full(I.batched_decode())


def test_prefill_full_size_every_pair():
    """2048 rows at positions 2048..4095 of a 4096-position cache, k = 640:
    every (row, head) output against the oracle (131,072 pairs)."""
    _check_full(I.prefill())


@pytest.mark.parametrize("first_pos,rows,N", [(0, 131, 512), (560, 90, 1024)])
def test_prefill_ragged_causal_rows(first_pos, rows, N):
    """Rows with n_sel = p+1 crossing the 128-key tile edge and the 640 cap."""
    _check_full(I.prefill(rows=rows, N=N, first_pos=first_pos))


_SWEEP = I.edge_sweep()


@pytest.mark.parametrize("i", range(len(_SWEEP)), ids=[c.name for c in _SWEEP])
def test_edge_sweep(i):
    _check_full(_SWEEP[i])


@pytest.mark.parametrize("mode", ["decode", "prefill"])
def test_rescaling_when_later_tiles_score_higher(mode):
    """Block maxima climbing by ~5.7 per 128 keys force the running reference
    maximum to move, so the accumulated value sum and row sum are rescaled."""
    _check_full(I.rising_scores(mode=mode))
    # blocks that climb by ~41 log2 units each: every later tile passes the
    # lag the kernel allows its reference maxima, so every one rescales
    _check_full(I.rising_scores(mode=mode, step=160.0))


@pytest.mark.parametrize("mode", ["decode", "prefill"])
def test_exact_sums_at_k640(mode):
    """Small-integer rows, q = 0, sink = -inf: every weight is 1 and the
    value sums are exact integers; out = sum/640 to within one ulp."""
    rng = np.random.default_rng(21)
    N, k = 2048, 640
    c = I.prefill(rows=2, N=N, first_pos=N - 2) if mode == "prefill" else I.batched_decode(B=2, N=N)
    vals = rng.integers(-8, 9, size=c.kv.shape).astype(np.float32)
    c.kv = I.f32_to_bf16_bits(vals)
    c.q[:] = 0
    c.sink[:] = -np.inf
    got, code = run(c)
    assert code == 0
    for r in range(c.R):
        cache = vals[r] if mode == "decode" else vals
        s = cache[c.idx[r, :k]].astype(np.float64).sum(axis=0)
        exact = s / 640.0
        ulp = np.spacing(np.abs(exact).astype(np.float32)).astype(np.float64)
        for h in range(c.H):
            assert np.all(np.abs(got[r, h] - exact) <= ulp), (r, h)


_REPEAT_CASES = {
    "single_decode_bf16": lambda: I.single_decode(),
    "prefill_200_bf16": lambda: I.prefill(rows=200, N=2048, first_pos=1500),
    "tiny_decode_fp32": lambda: I.tiny(mode="decode"),
    "tiny_prefill_fp32": lambda: I.tiny(mode="prefill"),
    "batched_decode_b8_full_size": lambda: I.batched_decode(),
}
for _j, _name in enumerate(I.EDGE_SPECIALS):
    _REPEAT_CASES["special_" + _name] = (lambda n=_name, j=_j: I.edge_special(n, (I.SEED_BASE + 4) * 131 + j))


@pytest.mark.parametrize("name", sorted(_REPEAT_CASES))
def test_five_repeats_are_bit_identical(name):
    """Five calls on the same inputs give the same bytes (akol1 TensorFold
    PR #4, second commit message: five byte-identical repeats), on both
    kernels (fp32 and bf16), through the split decode with its combine step,
    and for every nonfinite special case of the edge sweep."""
    c = _REPEAT_CASES[name]()
    d = to_device(c)
    first, code = run(c, d)
    assert code == 0
    for _ in range(4):
        again, code = run(c, d)
        assert code == 0
        assert np.array_equal(first.view(np.uint32), again.view(np.uint32))


def test_rows_do_not_depend_on_their_batch():
    """A row gives the same bits alone and among others (decode and prefill)."""
    c = I.batched_decode(B=5, N=4096)
    full, _ = run(c)
    for b in (0, 3):
        one = I.Case("one", "decode", c.dtype, 1, c.H, c.N, c.k_max, c.q[b:b + 1], c.kv[b:b + 1],
                     c.idx[b:b + 1], c.n_sel[b:b + 1], c.sink, c.scale)
        alone, _ = run(one)
        assert np.array_equal(alone[0].view(np.uint32), full[b].view(np.uint32))
    p = I.prefill(rows=300, N=2048, first_pos=1000)
    full, _ = run(p)
    for lo, hi in ((0, 1), (17, 170), (299, 300)):
        part = I.Case("part", "prefill", p.dtype, hi - lo, p.H, p.N, p.k_max, p.q[lo:hi], p.kv,
                      p.idx[lo:hi], p.n_sel[lo:hi], p.sink, p.scale)
        got, _ = run(part)
        assert np.array_equal(got.view(np.uint32), full[lo:hi].view(np.uint32))


@pytest.mark.parametrize("dtype", [I.F32, I.BF16])
@pytest.mark.parametrize("mode", ["decode", "prefill"])
def test_out_of_range_selection_sets_error_and_nan_row(dtype, mode):
    from deepseek_v4_top_gb300 import dsa
    rng = np.random.default_rng(8)
    c = I._edge_base(rng, "bad", dtype, 32, 300, mode, R=5, N=1000, k_extra=0)
    for r in range(c.R):
        c.idx[r] = rng.choice(c.N, c.k_max, replace=False)
    c.n_sel[:] = c.k_max
    c.idx[1, 5] = c.N            # index == N
    c.idx[2, 299] = -3           # negative index, in the last partial tile
    c.n_sel[3] = c.k_max + 1     # n_sel beyond k_max
    got, code = run(c)
    assert code == (dsa.DSA_DEVERR_IDX_RANGE | dsa.DSA_DEVERR_NSEL_RANGE)
    assert np.isnan(got[1:4]).all()
    assert np.isfinite(got[0]).all() and np.isfinite(got[4]).all()
    ref, _ = oracle.attn(c)
    compare(c, got, ref)          # the oracle's contract gives the same NaN rows
    assert dsa.dsa_get_device_error() == 0      # reading cleared the word


@pytest.mark.parametrize("dtype", [I.F32, I.BF16])
@pytest.mark.parametrize("mode", ["decode", "prefill"])
def test_empty_selection_and_infinite_sinks(dtype, mode):
    rng = np.random.default_rng(9)
    c = I._edge_base(rng, "empty", dtype, 16, 200, mode, R=3, N=700, k_extra=5)
    c.n_sel[1] = 0
    c.sink[:4] = np.inf
    c.sink[4:8] = -np.inf
    _check_full(c)


def test_negative_scale():
    c = I.single_decode()
    c.scale = -0.75 / math.sqrt(512)
    _check_full(c)
