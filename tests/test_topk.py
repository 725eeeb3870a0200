"""GPU parity of the top-k selection against the oracle (bit-exact: the
outputs are positions and counts), including the sizes the bench times,
ties, signed zeros, infinities and NaNs, short rows, padding, bad counts,
and the selection feeding the attention."""

import numpy as np
import pytest

import oracle
from deepseek_v4_top_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    import torch
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)


def gpu_topk(scores, n_valid, k, k_max=None):
    import torch
    from deepseek_v4_top_gb300 import dsa
    k_max = k if k_max is None else k_max
    R = scores.shape[0]
    s = torch.from_numpy(np.ascontiguousarray(scores, dtype=np.float32)).cuda()
    nv = torch.from_numpy(np.ascontiguousarray(n_valid, dtype=np.int32)).cuda()
    idx = torch.full((R, k_max), 12345, dtype=torch.int32, device="cuda")
    n_sel = torch.full((R,), 12345, dtype=torch.int32, device="cuda")
    dsa.dsa_topk_select(s, nv, k, idx, n_sel)
    code = dsa.dsa_get_device_error()
    return idx.cpu().numpy(), n_sel.cpu().numpy(), code


def check(scores, n_valid, k, k_max=None):
    got_idx, got_n, code = gpu_topk(scores, n_valid, k, k_max)
    ref_idx, ref_n, bad = oracle.topk(scores, n_valid, k, k_max)
    assert np.array_equal(got_n, ref_n)
    assert np.array_equal(got_idx, ref_idx)
    return code, bad


def special_scores(rng, shape):
    s = rng.integers(-4, 5, shape).astype(np.float32)
    s[rng.random(shape) < 0.1] = -0.0
    s[rng.random(shape) < 0.03] = np.inf
    s[rng.random(shape) < 0.03] = -np.inf
    s[rng.random(shape) < 0.03] = np.nan
    return s


def test_prefill_rows_full_size():
    scores, n_valid = I.indexer_scores("prefill")
    code, _ = check(scores, n_valid, 640)
    assert code == 0


def test_decode_rows_full_size():
    scores, n_valid = I.indexer_scores("decode")
    code, _ = check(scores, n_valid, 640)
    assert code == 0


@pytest.mark.parametrize("k", [1, 7, 64, 640, 2048])
def test_ties_signed_zeros_infinities_and_nans(k):
    rng = np.random.default_rng(5000 + k)
    R, ld = 9, 3000
    scores = special_scores(rng, (R, ld))
    n_valid = np.array([0, 1, 2, k - 1 if k > 1 else 0, k, k + 1, 1000, 2999, 3000], np.int32)
    n_valid = np.minimum(n_valid, ld)
    code, _ = check(scores, n_valid, k, k + 3)
    assert code == 0


@pytest.mark.parametrize("k", [7, 640, 2048])
def test_specials_on_long_rows(k):
    # rows over 8192 positions (selected in two steps: each 8192-position
    # share, then the shares' picks): ties, signed zeros, infinities and NaNs
    # whose runs cross the shares
    rng = np.random.default_rng(5050 + k)
    R, ld = 6, 9000
    scores = special_scores(rng, (R, ld))
    n_valid = np.array([k - 1, k + 1, 8192, 8193, 8999, 9000], np.int32)
    code, _ = check(scores, n_valid, k, k + 5)
    assert code == 0


@pytest.mark.parametrize("ld", [1024, 20000])
def test_all_scores_equal_and_all_nan(ld):
    scores = np.zeros((3, ld), np.float32)
    scores[1] = np.nan
    scores[2, ::2] = -0.0
    code, _ = check(scores, np.array([ld, ld, ld - 247], np.int32), 640)
    assert code == 0


def test_long_rows_and_row_stride():
    rng = np.random.default_rng(5100)
    scores = rng.standard_normal((4, 32768), dtype=np.float32)
    scores[:, 1000:1100] = 7.0        # ties at the top
    code, _ = check(scores, np.array([32768, 30000, 641, 640], np.int32), 640, 700)
    assert code == 0


@pytest.mark.parametrize("ld", [3000, 4092, 4096, 4100, 5000, 8188, 8192, 8196, 12000, 28676])
def test_row_strides_and_ragged_tails(ld):
    # row strides on both sides of 4096 (one 256-thread CTA below, one of
    # 512 threads above) and of 8192 (one step below, two steps above),
    # candidate counts ending at every offset within a float4 and within a
    # thread's run
    rng = np.random.default_rng(5150 + ld)
    scores = rng.standard_normal((8, ld), dtype=np.float32)
    scores[:, 5:40] = 1.5             # ties straddling the threshold
    n_valid = np.array([ld, ld - 1, ld - 2, ld - 3, ld - 17, 641, 700, 3], np.int32)
    code, _ = check(scores, n_valid, 640)
    assert code == 0


def test_bad_counts_set_the_error_bit_and_select_nothing():
    from deepseek_v4_top_gb300 import dsa
    rng = np.random.default_rng(5200)
    scores = rng.standard_normal((3, 256), dtype=np.float32)
    idx, n_sel, code = gpu_topk(scores, np.array([257, -3, 100], np.int32), 16)
    assert code & dsa.DSA_DEVERR_NVALID_RANGE
    assert list(n_sel[:2]) == [0, 0] and (idx[:2] == -1).all()
    ref_idx, ref_n, _ = oracle.topk(scores, np.array([257, -3, 100], np.int32), 16)
    assert np.array_equal(idx, ref_idx) and np.array_equal(n_sel, ref_n)


@pytest.mark.parametrize("ld", [1028, 4096])
def test_more_rows_than_fit_at_once(ld):
    # more rows than the GPU runs CTAs at once, with bad counts, rows whose
    # entries are all picks, empty rows, ragged tails and specials interleaved
    from deepseek_v4_top_gb300 import dsa
    rng = np.random.default_rng(5300 + ld)
    R = 1500
    scores = rng.standard_normal((R, ld), dtype=np.float32)
    scores[::7] = special_scores(rng, scores[::7].shape)
    n_valid = rng.integers(1, ld + 1, R).astype(np.int32)
    n_valid[::11] = rng.integers(0, 101, n_valid[::11].shape)   # all picks (k = 100), some empty
    n_valid[5::13] = ld + 1 + rng.integers(0, 4, n_valid[5::13].shape)
    n_valid[9::17] = -1
    n_valid[-1] = ld
    got_idx, got_n, code = gpu_topk(scores, n_valid, 100, 130)
    ref_idx, ref_n, bad = oracle.topk(scores, n_valid, 100, 130)
    assert np.array_equal(got_n, ref_n) and np.array_equal(got_idx, ref_idx)
    assert bad.any() and code & dsa.DSA_DEVERR_NVALID_RANGE


def test_repeats_are_identical():
    scores, n_valid = I.indexer_scores("prefill", rows=256)
    first = gpu_topk(scores, n_valid, 640)
    for _ in range(4):
        again = gpu_topk(scores, n_valid, 640)
        assert np.array_equal(first[0], again[0]) and np.array_equal(first[1], again[1])


def test_selection_feeds_the_attention():
    # the GPU picks drive the prefill attention; the result matches the
    # oracle's attention over the oracle's picks
    import torch
    from deepseek_v4_top_gb300 import dsa
    from gpu_helpers import compare
    case = I.prefill(rows=48, N=1024, first_pos=900)
    scores, n_valid = I.indexer_scores("prefill", rows=48, N=1024)
    idx, n_sel, code = gpu_topk(scores, n_valid, case.k_max)
    assert code == 0
    ref_idx, ref_n, _ = oracle.topk(scores, n_valid, case.k_max)
    picked = I.Case("picked", "prefill", case.dtype, case.R, case.H, case.N, case.k_max, case.q, case.kv,
                    ref_idx, ref_n, case.sink, case.scale)
    t = lambda a: torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.empty((case.R, case.H, 512), dtype=torch.float32, device="cuda")
    dsa.dsa_sparse_attn_prefill(t(case.q), t(case.kv), torch.from_numpy(idx).cuda(),
                                torch.from_numpy(n_sel).cuda(), torch.from_numpy(case.sink).cuda(),
                                case.scale, out)
    assert dsa.dsa_get_device_error() == 0
    ref, _ = oracle.attn(picked)
    compare(picked, out.cpu().numpy(), ref)
