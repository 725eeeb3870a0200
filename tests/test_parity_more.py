"""More GPU parity: launch shapes the main parity file does not reach.

- decode batches with more work units than SMs, so a CTA runs several units
  and the combine merges chunk partials written in different rounds;
- decode rows longer than 1024 keys (16 key chunks a row);
- prefill rows whose unit count is not a multiple of the SM count;
- the same calls captured into a CUDA graph, and issued on a side stream,
  must give the same bits as direct calls on the current stream;
- index entries past n_sel holding arbitrary values (extremes included)
  change no output bit and raise no error.

Tolerances as in test_parity.py: bf16 |g-o| <= 3e-3 * max|o| over the
(row, head), nonfinite classes exact.
"""

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


def _check(case):
    got, code = run(case)
    assert code == 0, "device error word %#x" % code
    ref, _ = oracle.attn(case)
    return compare(case, got, ref)


def test_decode_more_units_than_sms():
    # 48 rows x 5 chunks = 240 units on at most 152 SMs
    rng = np.random.default_rng(4101)
    _check(I._edge_base(rng, "decode_b48", I.BF16, 64, 640, "decode", R=48, N=2048, k_extra=0))


@pytest.mark.parametrize("k", [1024, 1025, 2048])
def test_decode_long_rows(k):
    # 8, 9 and 16 key chunks a row, rows ragged below k
    rng = np.random.default_rng(4200 + k)
    _check(I._edge_base(rng, "decode_k%d" % k, I.BF16, 64, k, "decode", R=3, N=4096, k_extra=1))


def test_prefill_rows_not_a_multiple_of_the_grid():
    # 157 rows: the last round of the persistent grid is 5 rows
    rng = np.random.default_rng(4300)
    _check(I._edge_base(rng, "prefill_r157", I.BF16, 64, 640, "prefill", R=157, N=1024, k_extra=0))


def _calls(d, case, out, stream):
    from deepseek_v4_top_gb300 import dsa
    fn = dsa.dsa_sparse_attn_decode if case.mode == "decode" else dsa.dsa_sparse_attn_prefill
    fn(d["q"], d["kv"], d["idx"], d["n_sel"], d["sink"], case.scale, out, stream)


@pytest.mark.parametrize("mode", ["decode", "prefill"])
def test_graph_replay_and_side_stream_match_direct_calls(mode):
    import torch
    from deepseek_v4_top_gb300 import dsa
    rng = np.random.default_rng(4400)
    case = I._edge_base(rng, "graph_" + mode, I.BF16, 64, 300, mode, R=6, N=2048, k_extra=2)
    d = to_device(case)
    shape = (case.R, case.H, 512)
    direct = torch.empty(shape, dtype=torch.float32, device="cuda")
    _calls(d, case, direct, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_error() == 0

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    on_side = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(side):
        _calls(d, case, on_side, side)
    side.synchronize()

    replayed = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            _calls(d, case, replayed, torch.cuda.current_stream())
        replayed.fill_(float("nan"))
        g.replay()
        g.replay()
    side.synchronize()
    assert dsa.dsa_get_device_error() == 0

    a = direct.cpu().numpy().view(np.uint32)
    assert np.array_equal(a, on_side.cpu().numpy().view(np.uint32))
    assert np.array_equal(a, replayed.cpu().numpy().view(np.uint32))
    ref, _ = oracle.attn(case)
    compare(case, direct.cpu().numpy(), ref)


@pytest.mark.parametrize("mode", ["decode", "prefill"])
def test_sinks_far_above_every_score(mode):
    # Heads 0-15 carry a sink logit of +80: every score of theirs lies more
    # than 100 log2 units below it, so weights taken against the sink would
    # fall to the bottom of the fp32 range.  The outputs of those heads are
    # tiny (about e^-80 times a mean of V) and must still match relatively.
    rng = np.random.default_rng(4500)
    case = I._edge_base(rng, "sink_high_" + mode, I.BF16, 64, 640, mode, R=3, N=2048, k_extra=0)
    case.sink[:16] = 80.0
    _check(case)


@pytest.mark.parametrize("mode", ["decode", "prefill"])
def test_scores_far_above_the_sinks(mode):
    # Sinks of -60: the first tile's scores pass the sinks by about 86 log2
    # units, more than a reference may lag.
    rng = np.random.default_rng(4600)
    case = I._edge_base(rng, "sink_low_" + mode, I.BF16, 64, 640, mode, R=3, N=2048, k_extra=0)
    case.sink[:] = -60.0
    _check(case)


def test_decode_rows_match_across_combine_paths():
    # 40 rows x 5 chunks = 200 units: more than SMs, so CTAs run several
    # units and the combine merges partials written in different rounds.  The
    # first 20 rows alone (100 units) and the first 5 alone (25 units) run one
    # unit a CTA.  A row must give the same bits in every launch.
    rng = np.random.default_rng(4700)
    big = I._edge_base(rng, "decode_b40", I.BF16, 64, 640, "decode", R=40, N=2048, k_extra=0)
    full, code = run(big)
    assert code == 0
    ref, _ = oracle.attn(big)
    compare(big, full, ref)
    for n in (20, 5):
        sub = I.Case("sub%d" % n, "decode", big.dtype, n, big.H, big.N, big.k_max, big.q[:n], big.kv[:n],
                     big.idx[:n], big.n_sel[:n], big.sink, big.scale)
        got, code = run(sub)
        assert code == 0
        assert np.array_equal(got.view(np.uint32), full[:n].view(np.uint32))


@pytest.mark.parametrize("mode", ["decode", "prefill"])
@pytest.mark.parametrize("H", [1, 13])
def test_fp32_head_counts_off_the_warp_groups(mode, H):
    # the fp32 kernel gives each CTA 8 heads (one warp each) of one row; head
    # counts that leave a group partly empty
    rng = np.random.default_rng(4800 + H)
    _check(I._edge_base(rng, "f32_h%d_%s" % (H, mode), I.F32, H, 70, mode, R=3, N=600, k_extra=3))


def _garbage_tail(case, seed):
    """The same case with every idx entry past n_sel[r] replaced by arbitrary
    int32 values, the extremes included (the header lets those entries hold
    anything)."""
    import copy
    c = copy.copy(case)
    c.idx = case.idx.copy()
    rng = np.random.default_rng(seed)
    for r in range(c.R):
        tail = c.idx[r, max(int(c.n_sel[r]), 0):]
        tail[:] = rng.integers(-2**31, 2**31, tail.shape, dtype=np.int64).astype(np.int32)
        if tail.size >= 2:
            tail[0], tail[-1] = np.iinfo(np.int32).max, np.iinfo(np.int32).min
    return c


@pytest.mark.parametrize("which", ["decode", "prefill", "decode_rows", "fp32_decode"])
def test_unused_index_entries_may_hold_anything(which):
    rng = np.random.default_rng(77)
    if which == "decode":
        case = I._edge_base(rng, "tail_decode", I.BF16, 64, 500, "decode", R=6, N=3000, k_extra=140)
    elif which == "prefill":
        case = I._edge_base(rng, "tail_prefill", I.BF16, 64, 300, "prefill", R=200, N=2000, k_extra=40)
    elif which == "decode_rows":
        case = I.multi_row_decode(B=3, T=2, N=2048, k=300)
        case.n_sel[1::2] = case.n_sel[1::2] // 2          # half-used rows leave long tails
    else:
        case = I._edge_base(rng, "tail_fp32", I.F32, 16, 200, "decode", R=3, N=1000, k_extra=60)
    want, code = run(case)
    assert code == 0
    got, code = run(_garbage_tail(case, 78))
    assert code == 0, "device error word %#x" % code
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
