"""Pins for the oracle's output projection (CPU only).

The C oracle (plain triple loop in fp64) is checked against routes written
independently here: numpy's float64 matmul, closed forms (an identity
matrix, one-hot rows), linearity, and the bound its |a||w| sum must obey.
Each test names the mistake it is there to catch.
"""

import numpy as np
import pytest

import oracle


def to_bf16_bits(x):
    """float32 -> bf16 bit patterns by round to nearest even (numpy only)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def widen(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def test_matches_numpy_matmul_on_a_non_square_case():
    # a transposed operand, a dropped or misplaced term, or a wrong stride
    # shows up against an independent float64 matmul on R != K != d_out
    rng = np.random.default_rng(7000)
    R, K, d_out = 5, 96, 40
    a = rng.standard_normal((R, K))
    w = to_bf16_bits(rng.standard_normal((K, d_out)).astype(np.float32))
    out, absv = oracle.oproj(a, w)
    ref = a @ widen(w)
    assert np.allclose(out, ref, rtol=0, atol=1e-12 * (np.abs(a) @ np.abs(widen(w))).max())
    assert np.allclose(absv, np.abs(a) @ np.abs(widen(w)), rtol=1e-13, atol=0)


def test_identity_matrix_returns_the_rows():
    # the projection by I is the input, bit for bit (every product is exact)
    rng = np.random.default_rng(7001)
    K = 64
    a = rng.standard_normal((3, K))
    w = to_bf16_bits(np.eye(K, dtype=np.float32))
    out, _ = oracle.oproj(a, w)
    assert np.array_equal(out, a)


def test_one_hot_rows_pick_rows_of_w():
    # a one-hot a[r] = e_k selects row k of w: catches a row/column swap of w
    rng = np.random.default_rng(7002)
    K, d_out = 32, 24
    w = to_bf16_bits(rng.standard_normal((K, d_out)).astype(np.float32))
    ks = [0, 5, 31]
    a = np.zeros((len(ks), K), np.float32)
    for r, k in enumerate(ks):
        a[r, k] = 1.0
    out, absv = oracle.oproj(to_bf16_bits(a), w)
    for r, k in enumerate(ks):
        assert np.array_equal(out[r], widen(w[k]))
        assert np.array_equal(absv[r], np.abs(widen(w[k])))


def test_bf16_rows_equal_their_widened_doubles():
    # the two input forms are the same numbers: same sums, same order, same bits
    rng = np.random.default_rng(7003)
    a16 = to_bf16_bits(rng.standard_normal((4, 48)).astype(np.float32))
    w = to_bf16_bits(rng.standard_normal((48, 16)).astype(np.float32))
    o1, b1 = oracle.oproj(a16, w)
    o2, b2 = oracle.oproj(widen(a16), w)
    assert np.array_equal(o1, o2) and np.array_equal(b1, b2)


def test_linear_in_the_rows_and_bounded_by_the_abs_sum():
    rng = np.random.default_rng(7004)
    K, d_out = 80, 12
    w = to_bf16_bits(rng.standard_normal((K, d_out)).astype(np.float32))
    a1, a2 = rng.standard_normal((2, K)), rng.standard_normal((2, K))
    o1, b1 = oracle.oproj(a1, w)
    o2, b2 = oracle.oproj(a2, w)
    o12, _ = oracle.oproj(a1 + a2, w)
    assert np.allclose(o12, o1 + o2, rtol=0, atol=1e-12 * (b1 + b2).max())
    assert (np.abs(o1) <= b1 * (1 + 1e-15)).all()


def test_rejects_bad_arguments():
    w = np.zeros((8, 8), np.uint16)
    with pytest.raises(ValueError):
        oracle.oproj(np.zeros((2, 7)), w)            # K mismatch
    with pytest.raises(TypeError):
        oracle.oproj(np.zeros((2, 8), np.float32), w)
