"""GPU parity of decode with several query rows a slot (row r reads slot
r // T) against the oracle, and bit-identity with the same rows run one a
slot, each over its own copy of the cache."""

import numpy as np
import pytest

import oracle
from deepseek_v4_top_gb300 import inputs as I

from gpu_helpers import compare, run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    import torch
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("B,T", [(1, 2), (3, 2), (2, 4), (8, 2)])
def test_bf16_rows_sharing_slots_match_the_oracle(B, T):
    c = I.multi_row_decode(B=B, T=T, N=4096, k=640, seed=600 + 10 * B + T)
    got, code = run(c)
    assert code == 0
    ref, _ = oracle.attn(c)
    compare(c, got, ref)


def test_fp32_rows_sharing_slots_match_the_oracle():
    c = I.multi_row_decode(B=2, T=3, N=512, k=100, dtype=I.F32, H=16, seed=650)
    got, code = run(c)
    assert code == 0
    ref, _ = oracle.attn(c)
    compare(c, got, ref)


@pytest.mark.parametrize("dtype", [I.BF16, I.F32])
def test_same_bits_as_one_row_a_slot(dtype):
    c = I.multi_row_decode(B=3, T=2, N=1024, k=300, dtype=dtype, H=32, seed=660)
    got, _ = run(c)
    kv_each = np.stack([c.kv[r // c.rows_per_slot] for r in range(c.R)])
    plain = I.Case("plain", "decode", c.dtype, c.R, c.H, c.N, c.k_max, c.q, kv_each, c.idx, c.n_sel,
                   c.sink, c.scale)
    ref, _ = run(plain)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
