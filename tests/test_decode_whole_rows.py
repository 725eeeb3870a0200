"""Decode without the key split (dsa_sparse_attn_decode_whole_rows): GPU
parity against the oracle, bit-identity with the prefill call over the
slots' caches viewed as one cache, independence from the batch, and the
split decode with more units than SMs keeping the bits its rows have in
small batches."""

import numpy as np
import pytest

import oracle
from deepseek_v4_top_gb300 import inputs as I

from gpu_helpers import GUARD, SENTINEL, compare, run, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    import torch
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)


def _whole(c, d=None, out_dtype="float32"):
    """Run case c through dsa_sparse_attn_decode_whole_rows into a guarded
    buffer; returns (out as float32 [R,H,512], error word)."""
    import torch
    from deepseek_v4_top_gb300 import dsa
    d = d if d is not None else to_device(c)
    T = max(c.rows_per_slot, 1)
    n = c.R * c.H * 512
    if out_dtype == "float32":
        buf = torch.empty(n + 2 * GUARD, dtype=torch.int32, device="cuda:0")
        buf.fill_(int(SENTINEL.view(np.int32)))
        out = buf[GUARD:GUARD + n].view(torch.float32).view(c.R, c.H, 512)
    else:
        out = torch.empty((c.R, c.H, 512), dtype=torch.bfloat16, device="cuda:0")
    dsa.dsa_sparse_attn_decode_whole_rows(d["q"], d["kv"], d["idx"], d["n_sel"], d["sink"], c.scale, out, T)
    code = dsa.dsa_get_device_error()
    if out_dtype != "float32":
        return out.view(torch.int16).cpu().numpy().view(np.uint16), code
    host = buf.cpu().numpy().view(np.uint32)
    assert np.all(host[:GUARD] == SENTINEL) and np.all(host[GUARD + n:] == SENTINEL), "guard written"
    assert not np.any(host[GUARD:GUARD + n] == SENTINEL), "some outputs were not written"
    return host[GUARD:GUARD + n].view(np.float32).reshape(c.R, c.H, 512).copy(), code


def _ragged(c, seed):
    """Give the rows n_sel of every kind (empty, one key, tile edges, full)."""
    rng = np.random.default_rng(seed)
    pick = np.array([0, 1, 127, 128, 129, 255, 256, 383, 500, c.k_max])
    c.n_sel = np.minimum(pick[rng.integers(0, len(pick), c.R)], c.k_max).astype(np.int32)
    c.n_sel[0] = c.k_max
    return c


@pytest.mark.parametrize("B,T", [(3, 1), (2, 2), (4, 3)])
def test_whole_rows_match_the_oracle(B, T):
    c = _ragged(I.multi_row_decode(B=B, T=T, N=3000, k=640, seed=700 + 10 * B + T), 701)
    got, code = _whole(c)
    assert code == 0
    ref, _ = oracle.attn(c)
    compare(c, got, ref)


@pytest.mark.parametrize("H,k,T", [(16, 77, 1), (32, 2048, 2), (64, 1, 1), (16, 129, 3)])
def test_whole_rows_other_head_counts_and_selection_sizes(H, k, T):
    """16 and 32 heads, one key, a partial tile, and 2048 keys (16 tiles a
    row): parity with the oracle and bit-identity with the prefill call over
    the flattened caches."""
    c = I.multi_row_decode(B=3, T=T, N=max(2 * k, 300), k=k, H=H, seed=790 + k + H)
    c.n_sel[-1] = max(k // 2, 1)
    got, code = _whole(c)
    assert code == 0
    ref, _ = oracle.attn(c)
    compare(c, got, ref)
    slot = np.arange(c.R) // T
    idx = c.idx.copy()
    for r in range(c.R):
        idx[r, :c.n_sel[r]] += slot[r] * c.N
    flat = I.Case("flat", "prefill", c.dtype, c.R, c.H, c.kv.shape[0] * c.N, c.k_max, c.q,
                  c.kv.reshape(-1, 512), idx, c.n_sel, c.sink, c.scale)
    want, code = run(flat)
    assert code == 0
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_whole_rows_fp32_inputs_give_the_decode_rows_bits():
    c = I.multi_row_decode(B=2, T=2, N=600, k=200, dtype=I.F32, H=16, seed=720)
    got, code = _whole(c)
    assert code == 0
    want, _ = run(c)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    ref, _ = oracle.attn(c)
    compare(c, got, ref)


@pytest.mark.parametrize("T", [1, 2])
def test_whole_rows_equal_prefill_over_the_flattened_caches(T):
    """The same kernel path as a prefill row: the slots' caches viewed as one
    [slots * N, 512] cache, each row's indices offset by its slot times N."""
    c = _ragged(I.multi_row_decode(B=5, T=T, N=2000, k=640, seed=730 + T), 731)
    got, code = _whole(c)
    assert code == 0
    slot = np.arange(c.R) // T
    idx = c.idx.copy()
    for r in range(c.R):
        idx[r, :c.n_sel[r]] += slot[r] * c.N
    flat = I.Case("flat", "prefill", c.dtype, c.R, c.H, c.kv.shape[0] * c.N, c.k_max, c.q,
                  c.kv.reshape(-1, 512), idx, c.n_sel, c.sink, c.scale)
    want, code = run(flat)
    assert code == 0
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_whole_rows_do_not_depend_on_the_batch_and_repeat():
    """More rows than SMs (the row queue hands them out): each row's bits
    equal those of the row run alone, and five runs give the same bits."""
    c = _ragged(I.batched_decode(B=200, N=700, seed=740), 741)
    d = to_device(c)
    got, code = _whole(c, d)
    assert code == 0
    for _ in range(4):
        again, code = _whole(c, d)
        assert code == 0 and np.array_equal(again.view(np.uint32), got.view(np.uint32))
    for r in (0, 1, 57, 151, 152, 199):
        one = I.Case("one", "decode", c.dtype, 1, c.H, c.N, c.k_max, c.q[r:r + 1], c.kv[r:r + 1],
                     c.idx[r:r + 1], c.n_sel[r:r + 1], c.sink, c.scale)
        alone, code = _whole(one)
        assert code == 0
        assert np.array_equal(alone[0].view(np.uint32), got[r].view(np.uint32)), r
    ref, _ = oracle.attn(I.Case("some", "decode", c.dtype, 8, c.H, c.N, c.k_max, c.q[:8], c.kv[:8],
                                c.idx[:8], c.n_sel[:8], c.sink, c.scale))
    compare(c, got[:8], ref)


def test_whole_rows_bf16_output_is_the_rounded_fp32_output():
    c = _ragged(I.multi_row_decode(B=3, T=2, N=1500, k=640, seed=750), 751)
    d = to_device(c)
    f32, code = _whole(c, d)
    assert code == 0
    b16, code = _whole(c, d, out_dtype="bfloat16")
    assert code == 0
    assert np.array_equal(b16, I.f32_to_bf16_bits(f32))


def test_whole_rows_unused_index_entries_may_hold_anything():
    """Entries at or past a row's n_sel are never read."""
    c = _ragged(I.batched_decode(B=160, N=900, seed=760), 761)
    d = to_device(c)
    clean, code = _whole(c, d)
    assert code == 0
    rng = np.random.default_rng(762)
    for r in range(c.R):
        tail = c.idx[r, c.n_sel[r]:]
        tail[:] = rng.choice(np.array([-7, 2 ** 31 - 1, -2 ** 31, c.N, 10 * c.N], np.int32), tail.shape)
    d = to_device(c)
    dirty, code = _whole(c, d)
    assert code == 0
    assert np.array_equal(dirty.view(np.uint32), clean.view(np.uint32))


def test_whole_rows_flag_bad_selections_like_the_decode():
    """An out-of-range index gives that row NaN and sets the error bit; a bad
    n_sel gives NaN and its own bit.  The other rows keep their bits."""
    from deepseek_v4_top_gb300 import dsa
    c = I.batched_decode(B=4, N=800, seed=770)
    d = to_device(c)
    good, code = _whole(c, d)
    assert code == 0
    c.idx[1, 300] = c.N
    c.n_sel[2] = c.k_max + 1
    bad, code = _whole(c)
    assert code & dsa.DSA_DEVERR_IDX_RANGE and code & dsa.DSA_DEVERR_NSEL_RANGE
    assert np.isnan(bad[1]).all() and np.isnan(bad[2]).all()
    for r in (0, 3):
        assert np.array_equal(bad[r].view(np.uint32), good[r].view(np.uint32))


def test_split_decode_with_more_units_than_sms_keeps_its_bits():
    """64 rows x 5 chunks = 320 units: every CTA runs more than one unit.
    Each row has the bits it has in a batch of 8 (one unit a CTA)."""
    c = I.batched_decode(B=64, N=2048, seed=780)
    c.n_sel[::7] = 300
    d = to_device(c)
    big, code = run(c, d)
    assert code == 0
    for b0 in (0, 24, 56):
        part = I.Case("part", "decode", c.dtype, 8, c.H, c.N, c.k_max, c.q[b0:b0 + 8], c.kv[b0:b0 + 8],
                      c.idx[b0:b0 + 8], c.n_sel[b0:b0 + 8], c.sink, c.scale)
        small, code = run(part)
        assert code == 0
        assert np.array_equal(small.view(np.uint32), big[b0:b0 + 8].view(np.uint32))
    ref, _ = oracle.attn(I.Case("some", "decode", c.dtype, 8, c.H, c.N, c.k_max, c.q[:8], c.kv[:8],
                                c.idx[:8], c.n_sel[:8], c.sink, c.scale))
    compare(c, big[:8], ref)


def test_full_size_batch_sampled_against_the_oracle():
    """The bench's large decode batch in its own launch configuration (608
    slots of 32768 positions, k = 640, inputs drawn on the device): sampled
    rows of the whole-row call and of the split call against the oracle.
    Each sampled row's selected KV rows are copied out in index order, so
    the oracle reads exactly the rows the kernels gathered, in that order."""
    import torch
    from deepseek_v4_top_gb300 import dsa
    B, N, K, H, D = 608, 32768, 640, 64, 512
    dev = torch.device("cuda:0")
    g = torch.Generator(device=dev)
    g.manual_seed(0xD5A0 + 29)
    kv = torch.empty((B, N, D), dtype=torch.bfloat16, device=dev)
    for b0 in range(0, B, 64):
        kv[b0:b0 + 64].normal_(generator=g)
    q = torch.randn((B, H, D), generator=g, device=dev).to(torch.bfloat16)
    sink = torch.randn(H, generator=g, device=dev)
    idx = torch.stack([torch.randperm(N, generator=g, device=dev)[:K] for _ in range(B)]).to(torch.int32)
    n_sel = torch.full((B,), K, dtype=torch.int32, device=dev)
    n_sel[5] = 0
    n_sel[300] = 129
    whole = torch.empty((B, H, D), dtype=torch.float32, device=dev)
    split = torch.empty_like(whole)
    scale = 1.0 / np.sqrt(D)
    dsa.dsa_sparse_attn_decode_whole_rows(q, kv, idx, n_sel, sink, scale, whole)
    dsa.dsa_sparse_attn_decode(q, kv, idx, n_sel, sink, scale, split)
    assert dsa.dsa_get_device_error() == 0
    rows = [0, 5, 151, 152, 300, 455, 607]
    sel = idx[rows].long()
    gathered = torch.stack([kv[r][sel[i]] for i, r in enumerate(rows)])      # [rows, K, D] in index order
    bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    c = I.Case("b608_sample", "decode", I.BF16, len(rows), H, K, K, bits(q[rows]), bits(gathered),
               np.tile(np.arange(K, dtype=np.int32), (len(rows), 1)), n_sel[rows].cpu().numpy(),
               sink.cpu().numpy(), scale)
    ref, _ = oracle.attn(c)
    compare(c, whole[rows].cpu().numpy(), ref)
    compare(c, split[rows].cpu().numpy(), ref)
    del kv
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", I.EDGE_SPECIALS)
def test_whole_rows_nonfinite_specials_match_the_oracle_and_repeat(name):
    """The edge sweep's nine special cases (NaN and infinities in q or in a
    selected row, NaN in every unselected row, -inf and zero sinks) as
    decode batches through the whole-row call: the oracle's classes and
    tolerance, and five runs with the same bits.  A prefill case becomes a
    decode batch whose slots each hold a copy of its cache."""
    c = I.edge_special(name, (I.SEED_BASE + 4) * 131 + 700 + I.EDGE_SPECIALS.index(name))
    if c.mode == "prefill":
        kv = np.ascontiguousarray(np.broadcast_to(c.kv, (c.R,) + c.kv.shape))
        c = I.Case(c.name, "decode", c.dtype, c.R, c.H, c.N, c.k_max, c.q, kv, c.idx, c.n_sel, c.sink, c.scale)
    d = to_device(c)
    got, code = _whole(c, d)
    assert code == 0
    ref, _ = oracle.attn(c)
    compare(c, got, ref)
    for _ in range(4):
        again, code = _whole(c, d)
        assert code == 0 and np.array_equal(again.view(np.uint32), got.view(np.uint32))
