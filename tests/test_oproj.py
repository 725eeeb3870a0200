"""GPU: the bf16 output of the attention and the output projection.

- A bf16 output is the float32 output of the same call rounded to nearest
  even, bit for bit, on every kernel path (tensor-core prefill, with and
  without the row queue; split decode and its combine; several rows a slot;
  the fp32-input kernel).
- dsa_oproj (the library's tensor-core GEMM) against the oracle's fp64
  product of the same bf16 inputs, within the float32-accumulation bound
  K * 2^-24 * sum_k |a||w|, on ragged tiles and on more tiles than SMs;
  repeated calls give the same bits.
- dsa_sparse_attn_prefill_oproj against the oracle's attention followed by
  the oracle's projection, within the bound that the attention's parity bar,
  the bf16 rounding and the accumulation give together.
"""

import numpy as np
import pytest

import oracle
from deepseek_v4_top_gb300 import inputs as I

pytestmark = pytest.mark.gpu

ATTN_BAR = 3e-3          # the bf16 attention parity bar (per element, x the (row, head) max)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    import torch
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)


def _run_both(case):
    """The case through dsa_sparse_attn twice: float32 out and bf16 out."""
    import torch
    from deepseek_v4_top_gb300 import dsa
    from gpu_helpers import to_device
    d = to_device(case)
    T = case.rows_per_slot if case.mode == "decode" else 0
    o32 = torch.empty((case.R, case.H, 512), dtype=torch.float32, device="cuda")
    o16 = torch.empty((case.R, case.H, 512), dtype=torch.bfloat16, device="cuda")
    dsa.dsa_sparse_attn(d["q"], d["kv"], d["idx"], d["n_sel"], d["sink"], case.scale, o32, T)
    dsa.dsa_sparse_attn(d["q"], d["kv"], d["idx"], d["n_sel"], d["sink"], case.scale, o16, T)
    assert dsa.dsa_get_device_error() == 0
    return o32, o16


def _rne_bits(o32):
    """float32 -> bf16 bit patterns, round to nearest even, in numpy."""
    u = o32.cpu().numpy().view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


@pytest.mark.parametrize("which", ["prefill_48", "prefill_queue_300", "decode_b4", "decode_rows_3x2",
                                   "fp32_prefill", "fp32_decode", "kv_pinf"])
def test_bf16_out_is_the_rounded_fp32_out(which):
    import torch
    case = {
        "prefill_48": lambda: I.prefill(rows=48, N=1024, first_pos=900),
        "prefill_queue_300": lambda: I.prefill(rows=300, N=1024, first_pos=700),
        "decode_b4": lambda: I.batched_decode(B=4, N=4096),
        "decode_rows_3x2": lambda: I.multi_row_decode(B=3, T=2, N=4096),
        "fp32_prefill": lambda: I.tiny(),
        "fp32_decode": lambda: I.tiny(mode="decode"),
        "kv_pinf": lambda: I.edge_special("kv_pinf", 91),
    }[which]()
    o32, o16 = _run_both(case)
    want = _rne_bits(o32)
    got = o16.view(torch.int16).cpu().numpy().view(np.uint16)
    nan32 = np.isnan(o32.cpu().numpy())
    nan16 = ((got & 0x7F80) == 0x7F80) & ((got & 0x7F) != 0)
    assert np.array_equal(nan32, nan16)
    assert np.array_equal(np.where(nan32, 0, got), np.where(nan32, 0, want))


def _bf16_bits(rng, shape, scale=1.0):
    return I.f32_to_bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


@pytest.mark.parametrize("R,K,d_out", [(48, 4096, 256), (16, 32768, 512), (5, 1024, 8),
                                       # ragged M, K and N tiles; one partial K slice
                                       (300, 72, 264), (130, 8, 520),
                                       # 224 output tiles: CTAs run several, both accumulators
                                       (1024, 128, 7168)])
def test_oproj_matches_the_oracle(R, K, d_out):
    import torch
    from deepseek_v4_top_gb300 import dsa
    rng = np.random.default_rng(7100 + K + d_out)
    a = _bf16_bits(rng, (R, K))
    w = _bf16_bits(rng, (K, d_out), 1.0 / np.sqrt(K))
    ta = torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    tw = torch.from_numpy(w.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.full((R, d_out), float("nan"), dtype=torch.float32, device="cuda")
    dsa.dsa_oproj(ta, tw, out)
    got = out.cpu().numpy().astype(np.float64)
    ref, absv = oracle.oproj(a, w)
    lim = K * 2.0 ** -24 * absv
    assert np.isfinite(got).all()
    assert (np.abs(got - ref) <= lim).all(), float(np.max(np.abs(got - ref) / lim))
    again = torch.empty_like(out)
    dsa.dsa_oproj(ta, tw, again)
    assert torch.equal(out, again)           # no split-K: the same bits every call


def test_prefill_with_output_projection_matches_the_oracle():
    import torch
    from deepseek_v4_top_gb300 import dsa
    from gpu_helpers import to_device
    case = I.prefill(rows=24, N=1024, first_pos=900)
    R, H = case.R, case.H
    K, d_out = H * 512, 256
    rng = np.random.default_rng(7200)
    w = _bf16_bits(rng, (K, d_out), 1.0 / np.sqrt(K))
    d = to_device(case)
    tw = torch.from_numpy(w.view(np.int16)).cuda().view(torch.bfloat16)
    attn = torch.empty((R, H, 512), dtype=torch.bfloat16, device="cuda")
    out = torch.full((R, d_out), float("nan"), dtype=torch.float32, device="cuda")
    dsa.dsa_sparse_attn_prefill_oproj(d["q"], d["kv"], d["idx"], d["n_sel"], d["sink"], case.scale, tw,
                                      attn, out)
    assert dsa.dsa_get_device_error() == 0
    got = out.cpu().numpy().astype(np.float64)
    o, _ = oracle.attn(case)                                   # [R, H, 512] fp64
    ref, absv = oracle.oproj(o.reshape(R, K), w)
    # attention error per (row, head): ATTN_BAR * max|o|, then the bf16
    # rounding (2^-9 of a value within that bar), then the accumulation
    e_rh = (ATTN_BAR + 2.0 ** -9 * (1 + ATTN_BAR)) * np.abs(o).max(axis=-1)         # [R, H]
    w_abs = np.abs(I.bf16_bits_to_f32(w).astype(np.float64)).reshape(H, 512, d_out).sum(axis=1)  # [H, d_out]
    lim = e_rh @ w_abs + K * 2.0 ** -24 * absv * (1 + 2 * ATTN_BAR)
    assert (np.abs(got - ref) <= lim).all(), float(np.max(np.abs(got - ref) / lim))
    # the attention rows handed to the GEMM are the bf16 output of the attention alone
    o16 = torch.empty_like(attn)
    dsa.dsa_sparse_attn(d["q"], d["kv"], d["idx"], d["n_sel"], d["sink"], case.scale, o16, 0)
    assert torch.equal(o16.view(torch.int16), attn.view(torch.int16))
