"""Pins for the fp64 oracle (CPU only).

The oracle is checked against things other than itself: a dense masked
softmax written independently (scores over the whole cache, a multiplicity
mask, a library softmax), closed forms, exact integer sums at k = 640 (the
pages' "exact sums at k 640" gate, akol1 TensorFold PR #4, second commit
message), IEEE special cases and invariances.  Each test names the mistake
it is there to catch.
"""

import math
from fractions import Fraction

import numpy as np
import pytest
import scipy.special

from deepseek_v4_top_gb300 import inputs as I

D = 512


def _case(dtype, mode, R=2, H=4, N=96, k=13, k_max=None, seed=5):
    rng = np.random.default_rng(seed)
    k_max = k if k_max is None else k_max
    q = I._normal(rng, (R, H, D), dtype)
    kv = I._normal(rng, (R, N, D) if mode == "decode" else (N, D), dtype)
    idx = np.full((R, k_max), I.POISON, np.int32)
    n_sel = np.zeros(R, np.int32)
    for r in range(R):
        m = k if r == 0 else max(1, k - 3 * r)
        idx[r, :m] = rng.choice(N, m, replace=False)
        n_sel[r] = m
    sink = rng.standard_normal(H).astype(np.float32)
    return I.Case("t", mode, dtype, R, H, N, k_max, q, kv, idx, n_sel, sink, 1 / math.sqrt(D))


def dense_reference(c):
    """Dense masked attention over the whole cache (independent routine).

    Scores every cache position with one matrix product, weights each by how
    many times the row selected it (0 for unselected positions), appends the
    sink as one extra logit with no value row, and normalises with
    scipy's logsumexp.
    """
    out = np.zeros((c.R, c.H, D))
    q = c.as_f32(c.q).astype(np.float64)
    for r in range(c.R):
        X = c.kv_rows_of(r).astype(np.float64)              # [N, D]
        mult = np.bincount(c.idx[r, :c.n_sel[r]], minlength=c.N).astype(np.float64)
        S = (X @ q[r].T) * float(np.float32(c.scale))      # [N, H]
        for h in range(c.H):
            sel = mult > 0
            logits = np.concatenate([[float(c.sink[h])], S[sel, h] + np.log(mult[sel])])
            lse = scipy.special.logsumexp(logits)
            w = np.zeros(c.N)
            w[sel] = np.exp(S[sel, h] + np.log(mult[sel]) - lse)
            out[r, h] = w @ X
    return out


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(1e-300, np.max(np.abs(b)))


@pytest.mark.parametrize("dtype", [I.F32, I.BF16])
@pytest.mark.parametrize("mode", ["decode", "prefill"])
def test_matches_dense_masked_attention(oracle_lib, dtype, mode):
    """Catches a wrong index, slot, scale, operand role or dropped sink term."""
    c = _case(dtype, mode, R=3, H=5, N=200, k=37, k_max=40)
    got, _ = oracle_lib.attn(c)
    ref = dense_reference(c)
    assert _rel(got, ref) < 1e-12


def test_duplicate_indices_count_twice(oracle_lib):
    """A position selected twice is weighted twice (the plain sum)."""
    c = _case(I.F32, "prefill", R=1, H=3, N=50, k=6)
    c.idx[0, :6] = [4, 9, 4, 17, 4, 30]
    got, _ = oracle_lib.attn(c)
    assert _rel(got, dense_reference(c)) < 1e-12


def test_k1_without_sink_returns_the_row_exactly(oracle_lib):
    c = _case(I.BF16, "decode", R=2, H=3, N=64, k=1)
    c.sink[:] = -np.inf
    got, _ = oracle_lib.attn(c)
    for r in range(c.R):
        x = c.kv_rows_of(r)[c.idx[r, 0]].astype(np.float64)
        for h in range(c.H):
            assert np.array_equal(got[r, h], x)


def test_k1_with_sink_is_a_logistic_weight(oracle_lib):
    """q = a*e_0, x_0[0] = b: s_0 = scale*a*b exactly; out = x_0 / (1 + e^(sink - s_0)).

    Catches a sink that is scaled, dropped, or added to the numerator.
    """
    c = _case(I.F32, "prefill", R=1, H=2, N=32, k=1)
    c.q[:] = 0
    c.q[0, :, 0] = [3.0, -2.0]
    c.kv[c.idx[0, 0], 0] = 4.0
    c.scale = 0.25
    c.sink[:] = [1.5, 0.75]
    got, _ = oracle_lib.attn(c)
    x = c.kv[c.idx[0, 0]].astype(np.float64)
    s = [0.25 * 3.0 * 4.0, 0.25 * -2.0 * 4.0]
    for h in range(2):
        expect = x / (1.0 + math.exp(float(c.sink[h]) - s[h]))
        np.testing.assert_allclose(got[0, h], expect, rtol=1e-15, atol=0)
    # sink equal to the score: exactly half of the row
    c.sink[:] = [3.0, -2.0]
    got, _ = oracle_lib.attn(c)
    assert np.array_equal(got[0, 0], x / 2)
    assert np.array_equal(got[0, 1], x / 2)


def test_sink_minus_inf_is_plain_softmax(oracle_lib):
    """With sink = -inf the result is textbook softmax attention (scipy softmax)."""
    c = _case(I.BF16, "prefill", R=2, H=3, N=120, k=50)
    c.sink[:] = -np.inf
    got, _ = oracle_lib.attn(c)
    q = c.as_f32(c.q).astype(np.float64)
    for r in range(c.R):
        X = c.kv_rows_of(r)[c.idx[r, :c.n_sel[r]]].astype(np.float64)
        for h in range(c.H):
            w = scipy.special.softmax((X @ q[r, h]) * float(np.float32(c.scale)))
            np.testing.assert_allclose(got[r, h], w @ X, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("sink", [-np.inf, 0.0, 1.25])
def test_constant_score_gives_the_mean(oracle_lib, sink):
    """q = 0: every score is 0, so out = K/(K + e^sink) * mean of the rows."""
    c = _case(I.F32, "decode", R=2, H=2, N=80, k=21)
    c.q[:] = 0
    c.sink[:] = sink
    got, _ = oracle_lib.attn(c)
    for r in range(c.R):
        K = int(c.n_sel[r])
        X = c.kv[r][c.idx[r, :K]].astype(np.float64)
        expect = X.mean(axis=0) * (K / (K + math.exp(sink)))
        for h in range(c.H):
            np.testing.assert_allclose(got[r, h], expect, rtol=1e-13, atol=1e-15)


def test_all_equal_rows_return_that_row(oracle_lib):
    """Every selected row equal to v: out = v * (1 - w_sink)."""
    c = _case(I.BF16, "prefill", R=1, H=3, N=64, k=9)
    v = I.f32_to_bf16_bits(np.random.default_rng(3).standard_normal(D).astype(np.float32))
    for p in c.idx[0, :9]:
        c.kv[p] = v
    vf = I.bf16_bits_to_f32(v).astype(np.float64)
    c.sink[:] = [-np.inf, 0.0, 2.0]
    got, _ = oracle_lib.attn(c)
    assert np.array_equal(got[0, 0], vf)
    q = I.bf16_bits_to_f32(c.q).astype(np.float64)
    for h in (1, 2):
        s = float(np.float32(c.scale)) * (q[0, h] @ vf)
        w_sink = 1.0 / (1.0 + 9.0 * math.exp(s - float(c.sink[h])))
        np.testing.assert_allclose(got[0, h], vf * (1 - w_sink), rtol=1e-13)


def test_exact_integer_sums_at_k640(oracle_lib):
    """Small-integer rows, q = 0, sink = -inf: out = (integer column sum)/640, correctly rounded."""
    rng = np.random.default_rng(11)
    N, k = 1024, 640
    vals = rng.integers(-8, 9, size=(N, D)).astype(np.float32)
    c = _case(I.BF16, "prefill", R=1, H=2, N=N, k=k)
    c.kv = I.f32_to_bf16_bits(vals)
    c.q[:] = 0
    c.sink[:] = -np.inf
    got, _ = oracle_lib.attn(c)
    sums = vals[c.idx[0, :k]].astype(np.int64).sum(axis=0)
    expect = np.array([float(Fraction(int(s), 640)) for s in sums])
    assert np.array_equal(got[0, 0], expect)
    assert np.array_equal(got[0, 1], expect)


def test_permutation_invariance(oracle_lib):
    c = _case(I.F32, "decode", R=2, H=4, N=300, k=77)
    a, _ = oracle_lib.attn(c)
    rng = np.random.default_rng(2)
    for r in range(c.R):
        m = c.n_sel[r]
        c.idx[r, :m] = c.idx[r, rng.permutation(m)]
    b, _ = oracle_lib.attn(c)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-15)


def test_power_of_two_rescaling_is_exact(oracle_lib):
    """kv * 2^5 with q * 2^-5 leaves every score unchanged and scales out by 2^5 exactly."""
    c = _case(I.F32, "prefill", R=2, H=3, N=90, k=33)
    a, _ = oracle_lib.attn(c)
    c.kv = c.kv * np.float32(32.0)
    c.q = c.q * np.float32(1 / 32.0)
    b, _ = oracle_lib.attn(c)
    assert np.array_equal(b, a * 32.0)


def test_rows_use_their_own_slot_in_decode(oracle_lib):
    """Changing slot 1's cache changes row 1 only."""
    c = _case(I.F32, "decode", R=3, H=2, N=64, k=10)
    a, _ = oracle_lib.attn(c)
    c.kv[1] = c.kv[1] * np.float32(0.5)
    b, _ = oracle_lib.attn(c)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[2], b[2])
    assert not np.array_equal(a[1], b[1])


def test_entries_past_n_sel_are_never_read(oracle_lib):
    """Poison (-1) beyond n_sel must not turn the row into the NaN contract row."""
    c = _case(I.F32, "prefill", R=2, H=2, N=64, k=10, k_max=16)
    got, _ = oracle_lib.attn(c)
    assert np.isfinite(got).all()


def test_batch_independence(oracle_lib):
    c = _case(I.BF16, "decode", R=3, H=3, N=70, k=20)
    full, _ = oracle_lib.attn(c)
    for r in range(c.R):
        one = I.Case("one", "decode", c.dtype, 1, c.H, c.N, c.k_max, c.q[r:r + 1], c.kv[r:r + 1],
                     c.idx[r:r + 1], c.n_sel[r:r + 1], c.sink, c.scale)
        got, _ = oracle_lib.attn(one)
        assert np.array_equal(got[0], full[r])


def test_pairs_and_rowhead_agree_with_full(oracle_lib):
    c = _case(I.BF16, "prefill", R=3, H=4, N=100, k=30)
    full, _ = oracle_lib.attn(c)
    rows = np.array([2, 0, 1], np.int32)
    heads = np.array([3, 1, 0], np.int32)
    got, _ = oracle_lib.pairs(c, rows, heads)
    for i in range(3):
        assert np.array_equal(got[i], full[rows[i], heads[i]])
        assert np.array_equal(oracle_lib.rowhead(c, int(rows[i]), int(heads[i])), got[i])


# ---------------------------------------------------------------- nonfinite
def test_nan_in_q_poisons_only_that_head(oracle_lib):
    c = _case(I.F32, "prefill", R=2, H=3, N=64, k=12)
    c.q[0, 1, 7] = np.nan
    got, _ = oracle_lib.attn(c)
    assert np.isnan(got[0, 1]).all()
    assert np.isfinite(got[0, 0]).all() and np.isfinite(got[0, 2]).all() and np.isfinite(got[1]).all()


def test_plus_inf_score_gives_nan(oracle_lib):
    c = _case(I.F32, "prefill", R=1, H=2, N=64, k=12)
    c.q[0, 0, :] = 0
    c.q[0, 0, 5] = np.inf
    c.kv[c.idx[0, 3], 5] = 1.0      # +inf * 1 -> +inf score for that key
    got, _ = oracle_lib.attn(c)
    assert np.isnan(got[0, 0]).all()


def test_minus_inf_score_has_zero_weight(oracle_lib):
    """A -inf score removes the key; column c is NaN only where that key's value is infinite."""
    c = _case(I.F32, "prefill", R=1, H=2, N=64, k=12)
    p = c.idx[0, 4]
    base, _ = oracle_lib.attn(c)
    c.kv[p, 9] = -np.inf   # head scores with q[.,9] > 0 become -inf, others +inf
    got, _ = oracle_lib.attn(c)
    for h in range(2):
        if c.q[0, h, 9] > 0:
            assert np.isnan(got[0, h, 9])
            keep = np.ones(D, bool)
            keep[9] = False
            assert np.isfinite(got[0, h, keep]).all()
            # equals the result with key 4 removed
            c2 = _case(I.F32, "prefill", R=1, H=2, N=64, k=12)
            c2.idx[0, :11] = np.delete(c2.idx[0, :12], 4)
            c2.n_sel[0] = 11
            ref, _ = oracle_lib.attn(c2)
            np.testing.assert_allclose(got[0, h, keep], ref[0, h, keep], rtol=1e-13, atol=1e-15)
        else:
            assert np.isnan(got[0, h]).all()


def test_nonfinite_in_unselected_rows_has_no_effect(oracle_lib):
    c = _case(I.BF16, "decode", R=2, H=2, N=64, k=10)
    a, _ = oracle_lib.attn(c)
    for r in range(c.R):
        mask = np.ones(c.N, bool)
        mask[c.idx[r, :c.n_sel[r]]] = False
        c.kv[r][mask] = I.BF16_NAN
    b, _ = oracle_lib.attn(c)
    assert np.array_equal(a, b)


def test_sink_extremes_and_empty_selection(oracle_lib):
    c = _case(I.F32, "prefill", R=1, H=3, N=64, k=8)
    c.sink[:] = [np.inf, -np.inf, 0.5]
    got, _ = oracle_lib.attn(c)
    assert np.array_equal(got[0, 0], np.zeros(D))          # the sink takes all the weight
    c.n_sel[0] = 0
    got, _ = oracle_lib.attn(c)
    assert np.array_equal(got[0, 0], np.zeros(D))
    assert np.isnan(got[0, 1]).all()                       # 0 / 0
    assert np.array_equal(got[0, 2], np.zeros(D))          # 0 / e^sink


def test_out_of_range_selection_gives_nan_row(oracle_lib):
    c = _case(I.F32, "prefill", R=3, H=2, N=64, k=8)
    c.idx[1, 2] = 64          # == N
    c.n_sel[2] = c.k_max + 1
    got, _ = oracle_lib.attn(c)
    assert np.isfinite(got[0]).all()
    assert np.isnan(got[1]).all() and np.isnan(got[2]).all()


def test_threads_do_not_change_bits(oracle_lib):
    c = _case(I.BF16, "prefill", R=3, H=8, N=128, k=40)
    a, _ = oracle_lib.attn(c, threads=1)
    b, used = oracle_lib.attn(c, threads=0)
    assert used >= 1
    assert np.array_equal(a, b)


def test_golden_closed_forms(oracle_lib):
    """Hand-derived fixtures in tests/golden/closed_forms.json."""
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")
    for g in json.load(open(path))["cases"]:
        H, N = g["H"], g["N"]
        q = np.zeros((1, H, D), np.float32)
        for h, vec in enumerate(g["q"]):
            for d, v in vec.items():
                q[0, h, int(d)] = v
        kv = np.zeros((N, D), np.float32)
        for row, vec in g["kv"].items():
            for d, v in vec.items():
                kv[int(row), int(d)] = v
        k = len(g["idx"])
        c = I.Case(g["name"], "prefill", I.F32, 1, H, N, k, q, kv,
                   np.array([g["idx"]], np.int32), np.array([k], np.int32),
                   np.array([float(s) for s in g["sink"]], np.float32), g["scale"])
        got, _ = oracle_lib.attn(c)
        for h, vec in enumerate(g["expected"]):
            expect = np.zeros(D)
            for d, v in vec.items():
                expect[int(d)] = float(Fraction(v))
            np.testing.assert_allclose(got[0, h], expect, rtol=4e-16, atol=0, err_msg=g["name"])


@pytest.mark.parametrize("T", [2, 3])
def test_rows_sharing_a_slot_read_that_slot(oracle_lib, T):
    # catches: a row reading slot r instead of slot r // T
    c = I.multi_row_decode(B=2, T=T, N=300, k=40, dtype=I.F32, H=4, seed=31)
    got, _ = oracle_lib.attn(c)
    kv_each = np.stack([c.kv[r // T] for r in range(c.R)])
    plain = I.Case("plain", "decode", c.dtype, c.R, c.H, c.N, c.k_max, c.q, kv_each, c.idx, c.n_sel,
                   c.sink, c.scale)
    ref, _ = oracle_lib.attn(plain)
    assert np.array_equal(got, ref)
    assert c.B == 2
