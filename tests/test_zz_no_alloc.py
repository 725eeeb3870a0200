"""The decode entry point that allocates no device memory.

Some callers of this library must not allocate device memory: engines that
reserve all of it at start-up and forbid allocation afterwards, and callers
on a latency-critical path where cudaMalloc / cudaFree would synchronise the
device.  dsa_sparse_attn_decode_noalloc() serves them from a fixed static
device array.  These tests call it through the C ABI and check it against
dsa_sparse_attn_decode(), which allocates its scratch, on two calls in a
row with different shapes, so a call cannot lean on what the one before it
left in the shared array.  This file is collected last on purpose.
"""

import numpy as np
import pytest

from deepseek_v4_top_gb300 import inputs as I

from gpu_helpers import compare, to_device

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    import torch
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)

def _call(name, case, d):
    """One decode call through the C ABI with raw device addresses."""
    import torch
    from deepseek_v4_top_gb300 import dsa
    out = torch.full((case.R, case.H, 512), float("nan"), dtype=torch.float32, device="cuda:0")
    st = dsa.call_raw(name, d["q"].data_ptr(), d["kv"].data_ptr(), d["idx"].data_ptr(),
                      d["n_sel"].data_ptr(), d["sink"].data_ptr(), case.scale, out.data_ptr(),
                      case.R, case.H, case.N, case.k_max, dsa.DSA_BF16,
                      torch.cuda.current_stream().cuda_stream)
    assert st == dsa.DSA_OK, dsa.status_string(st)
    torch.cuda.synchronize()
    return out.cpu().numpy()

def test_noalloc_decode_matches_the_allocating_decode_twice_in_a_row():
    first = I.batched_decode(B=8, N=8192)                 # 8 rows x 5 chunks = 40 units
    rng = np.random.default_rng(12)
    second = I._edge_base(rng, "second", I.BF16, 32, 300, "decode", R=3, N=2000, k_extra=20)
    for case in (first, second):
        d = to_device(case)
        ref = _call("dsa_sparse_attn_decode", case, d).astype(np.float64)
        got = _call("dsa_sparse_attn_decode_noalloc", case, d)
        assert np.isfinite(got).all()
        compare(case, got, ref)

def test_noalloc_rejects_batches_beyond_its_fixed_scratch():
    from deepseek_v4_top_gb300 import dsa
    fake = 1 << 20
    # 13 rows x ceil(640/128) = 65 units > 64
    st = dsa.call_raw("dsa_sparse_attn_decode_noalloc", fake, fake, fake, fake, fake, 0.1, fake,
                      13, 64, 4096, 640, dsa.DSA_BF16, 0)
    assert st == dsa.DSA_ERR_UNSUPPORTED
    st = dsa.call_raw("dsa_sparse_attn_decode_noalloc", fake, fake, fake, fake, fake, 0.1, fake,
                      2, 64, 4096, 640, dsa.DSA_F32, 0)
    assert st == dsa.DSA_ERR_UNSUPPORTED
