"""The decode entry point that allocates no device memory.

Some callers of this library must not allocate device memory: engines that
reserve all of it at start-up and forbid allocation afterwards, and callers
on a latency-critical path where cudaMalloc / cudaFree would synchronise the
device.  dsa_sparse_attn_decode_noalloc() serves them from a fixed static
device array.  These tests call it through the C ABI and check it against
dsa_sparse_attn_decode(), which allocates its scratch.  Both run the same
kernels with the same key chunking, so the outputs must be the same bytes.
Calls follow one another with different shapes, so a call cannot lean on
what the one before it left in the shared array.  This file is collected
last on purpose.
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


def _both(case):
    """The allocating decode, its device error word, then the no-allocation
    decode on the same device inputs."""
    from deepseek_v4_top_gb300 import dsa
    d = to_device(case)
    ref = _call("dsa_sparse_attn_decode", case, d)
    code = dsa.dsa_get_device_error()
    got = _call("dsa_sparse_attn_decode_noalloc", case, d)
    assert dsa.dsa_get_device_error() == 0     # this entry point reports no error bits
    return ref, code, got


def _cases():
    rng = np.random.default_rng(12)
    return [
        # 8 rows x 5 key chunks = 40 units: partials and the combine step
        I.batched_decode(B=8, N=8192),
        # ragged rows over three chunks of up to 128 keys
        I._edge_base(rng, "three_chunks", I.BF16, 32, 300, "decode", R=3, N=2000, k_extra=20),
        # k_max <= 128: one chunk a row, written straight to the output
        I._edge_base(rng, "one_chunk", I.BF16, 64, 100, "decode", R=5, N=1500, k_extra=28),
        # exactly DSA_NOALLOC_MAX_UNITS units: 8 rows x ceil(1024 / 128)
        I._edge_base(rng, "max_units", I.BF16, 64, 1024, "decode", R=8, N=3000, k_extra=0),
    ]


def test_noalloc_decode_is_bit_identical_to_the_allocating_decode_call_after_call():
    from deepseek_v4_top_gb300 import dsa
    cases = _cases()
    assert cases[3].R * -(-cases[3].k_max // 128) == dsa.DSA_NOALLOC_MAX_UNITS
    for case in cases:
        ref, code, got = _both(case)
        assert code == 0
        assert np.isfinite(got).all(), case.name
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), case.name
        compare(case, got, ref.astype(np.float64))


def test_noalloc_out_of_range_selection_gives_a_nan_row():
    """A selected index >= N makes that row NaN (the error bit is lost on this
    entry point); the other rows are the allocating decode's bytes."""
    from deepseek_v4_top_gb300 import dsa
    rng = np.random.default_rng(13)
    case = I._edge_base(rng, "bad_index", I.BF16, 64, 400, "decode", R=4, N=2500, k_extra=0)
    case.idx[2, 50] = case.N            # row 2 selects its first 132 entries
    ref, code, got = _both(case)
    assert code == dsa.DSA_DEVERR_IDX_RANGE
    assert np.isnan(got[2]).all()
    for r in (0, 1, 3):
        assert np.isfinite(got[r]).all()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


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


def test_noalloc_after_shutdown_looks_its_array_up_again():
    """dsa_shutdown() releases the library's device state and forgets the
    array's looked-up address; the next call looks it up again and gives the
    same bytes as before."""
    import torch
    from deepseek_v4_top_gb300 import dsa
    case = I.batched_decode(B=4, N=4096)
    d = to_device(case)
    before = _call("dsa_sparse_attn_decode_noalloc", case, d)
    torch.cuda.synchronize()
    dsa.dsa_shutdown()
    after = _call("dsa_sparse_attn_decode_noalloc", case, d)
    again = _call("dsa_sparse_attn_decode", case, d)
    assert np.array_equal(before.view(np.uint32), after.view(np.uint32))
    assert np.array_equal(before.view(np.uint32), again.view(np.uint32))
    assert dsa.dsa_get_device_error() == 0
