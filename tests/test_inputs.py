"""The seeded input generator (CPU only)."""

import numpy as np

from deepseek_v4_top_gb300 import inputs as I


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.00390625, 1.005859375, -2.5, 3.0e38, np.inf, -np.inf], np.float32)
    b = I.f32_to_bf16_bits(x)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa (1.0) wins
    assert b[0] == 0x3F80 and b[1] == 0x3F80
    # 1 + 1.5*2^-8 rounds up to 1 + 2^-7
    assert b[2] == 0x3F81
    assert b[3] == 0xC020
    assert b[5] == I.BF16_PINF and b[6] == I.BF16_NINF
    assert np.isnan(I.bf16_bits_to_f32(I.f32_to_bf16_bits(np.array([np.nan], np.float32))))[0]
    back = I.bf16_bits_to_f32(b[:4])
    assert np.array_equal(back, np.array([1.0, 1.0, 1.0078125, -2.5], np.float32))


def test_tiny_is_deterministic_and_distinct():
    a, b = I.tiny(), I.tiny()
    assert np.array_equal(a.q, b.q) and np.array_equal(a.idx, b.idx)
    for r in range(a.R):
        assert len(set(a.idx[r].tolist())) == 64
        assert a.idx[r].min() >= 0 and a.idx[r].max() < a.N


def test_single_decode_is_sorted():
    c = I.single_decode()
    assert c.q.dtype == np.uint16 and c.kv.shape == (1, 4096, 512)
    assert np.all(np.diff(c.idx[0]) > 0)


def test_prefill_rows_are_causal_top_k():
    c = I.prefill(rows=6, N=700, first_pos=600)
    for i in range(c.R):
        p = 600 + i
        m = min(p + 1, 640)
        assert c.n_sel[i] == m
        sel = c.idx[i, :m]
        assert len(set(sel.tolist())) == m and sel.min() >= 0 and sel.max() <= p
        assert np.all(c.idx[i, m:] == I.POISON)


def test_batched_decode_small_is_deterministic():
    a = I.batched_decode(B=3, N=1024)
    b = I.batched_decode(B=3, N=1024)
    assert a.kv.shape == (3, 1024, 512)
    assert np.array_equal(a.kv, b.kv)
    assert not np.array_equal(a.kv[0], a.kv[1])


def test_edge_sweep_has_51_shapes():
    cases = I.edge_sweep()
    assert len(cases) == 51
    hs = {c.H for c in cases[:42]}
    ks = {int(c.n_sel[0]) for c in cases[:42]}
    assert hs == {16, 32, 64} and ks == {1, 7, 63, 64, 65, 127, 640}
    assert {c.dtype for c in cases} == {"f32", "bf16"}
    assert {c.mode for c in cases} == {"decode", "prefill"}
    for c in cases:
        assert c.n_sel.max() <= c.k_max
        for r in range(c.R):
            sel = c.idx[r, :c.n_sel[r]]
            assert sel.min() >= 0 and sel.max() < c.N
            assert np.all(c.idx[r, c.n_sel[r]:] == I.POISON)


def test_rising_scores_ramp():
    c = I.rising_scores(k=256, H=4)
    f = I.bf16_bits_to_f32(c.kv)
    for r in range(c.R):
        assert f[c.idx[r, 0], 0] == 0.0 and f[c.idx[r, 200], 0] == 32.0
