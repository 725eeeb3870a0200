"""Calls on different streams at once.

A decode batch and a prefill segment are independent calls, and a serving
step may issue them on two streams so that they overlap on the GPU (the
bench's step does).  The library keeps no state that two such calls share
except the sticky error word: the decode's split partials have their own
scratch, and each stream has its own prefill row queue.  These tests run the
two calls on two streams at once, several times over, and check the bytes
against the same calls run one after the other on one stream."""

import numpy as np
import pytest

from deepseek_v4_top_gb300 import inputs as I

from gpu_helpers import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    import torch
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)


def _calls(dec, d_dec, pre, d_pre):
    import torch
    from deepseek_v4_top_gb300 import dsa
    o_dec = torch.empty((dec.R, dec.H, 512), dtype=torch.float32, device="cuda:0")
    o_pre = torch.empty((pre.R, pre.H, 512), dtype=torch.float32, device="cuda:0")

    def run_dec(s):
        dsa.dsa_sparse_attn_decode(d_dec["q"], d_dec["kv"], d_dec["idx"], d_dec["n_sel"], d_dec["sink"],
                                   dec.scale, o_dec, s)

    def run_pre(s):
        dsa.dsa_sparse_attn_prefill(d_pre["q"], d_pre["kv"], d_pre["idx"], d_pre["n_sel"], d_pre["sink"],
                                    pre.scale, o_pre, s)
    return o_dec, o_pre, run_dec, run_pre


@pytest.mark.parametrize("prefill_rows", [300, 2048])
def test_decode_and_prefill_on_two_streams_give_the_one_stream_bytes(prefill_rows):
    import torch
    from deepseek_v4_top_gb300 import dsa
    dec = I.batched_decode(B=8, N=8192)
    pre = I.prefill(rows=prefill_rows, N=4096)
    d_dec, d_pre = to_device(dec), to_device(pre)
    o_dec, o_pre, run_dec, run_pre = _calls(dec, d_dec, pre, d_pre)
    main = torch.cuda.current_stream()
    run_dec(main)
    run_pre(main)
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_error() == 0
    want_dec, want_pre = o_dec.clone(), o_pre.clone()
    side = torch.cuda.Stream()
    for order in range(4):
        o_dec.fill_(float("nan"))
        o_pre.fill_(float("nan"))
        side.wait_stream(main)
        if order % 2 == 0:
            run_dec(side)
            run_pre(main)
        else:
            run_pre(main)
            run_dec(side)
        main.wait_stream(side)
        torch.cuda.synchronize()
        assert dsa.dsa_get_device_error() == 0
        assert torch.equal(o_dec.view(torch.int32), want_dec.view(torch.int32))
        assert torch.equal(o_pre.view(torch.int32), want_pre.view(torch.int32))


def test_two_prefill_segments_on_two_streams_use_their_own_row_queues():
    """Two prefill calls with more rows than SMs, each on its own stream at
    once: each stream's row queue hands out that call's rows only."""
    import torch
    from deepseek_v4_top_gb300 import dsa
    a = I.prefill(seed=41, rows=700, N=4096)
    b = I.prefill(seed=42, rows=500, N=2048, first_pos=1000)
    da, db = to_device(a), to_device(b)
    oa = torch.empty((a.R, a.H, 512), dtype=torch.float32, device="cuda:0")
    ob = torch.empty((b.R, b.H, 512), dtype=torch.float32, device="cuda:0")

    def run(c, d, o, s):
        dsa.dsa_sparse_attn_prefill(d["q"], d["kv"], d["idx"], d["n_sel"], d["sink"], c.scale, o, s)
    main = torch.cuda.current_stream()
    run(a, da, oa, main)
    run(b, db, ob, main)
    torch.cuda.synchronize()
    want_a, want_b = oa.clone(), ob.clone()
    side = torch.cuda.Stream()
    for _ in range(3):
        oa.fill_(float("nan"))
        ob.fill_(float("nan"))
        side.wait_stream(main)
        run(a, da, oa, main)
        run(b, db, ob, side)
        main.wait_stream(side)
        torch.cuda.synchronize()
        assert dsa.dsa_get_device_error() == 0
        assert torch.equal(oa.view(torch.int32), want_a.view(torch.int32))
        assert torch.equal(ob.view(torch.int32), want_b.view(torch.int32))
