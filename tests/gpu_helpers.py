"""Shared helpers for the GPU tests: upload a Case, run it through the C ABI
with guard regions around the output, compare with the oracle."""

import numpy as np

from deepseek_v4_top_gb300 import inputs as I

GUARD = 1024                       # floats (4 KiB) before and after out
SENTINEL = np.uint32(0x7FBADBAD)   # a NaN payload no kernel writes
TOL_F32_REL, TOL_F32_ABS = 1e-5, 1e-6
TOL_BF16 = 3e-3


def to_device(case, dev="cuda:0"):
    import torch
    if case.dtype == I.BF16:
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    return dict(q=t(case.q), kv=t(case.kv), idx=torch.from_numpy(case.idx).to(dev),
                n_sel=torch.from_numpy(case.n_sel).to(dev), sink=torch.from_numpy(case.sink).to(dev))


def run(case, dev_inputs=None, dev="cuda:0", check_guards=True):
    """Run one case through the C ABI; returns (out float32 [R,H,512], error word)."""
    import torch
    from deepseek_v4_top_gb300 import dsa
    d = dev_inputs if dev_inputs is not None else to_device(case, dev)
    n = case.R * case.H * 512
    buf = torch.empty(n + 2 * GUARD, dtype=torch.int32, device=dev)
    buf.fill_(int(SENTINEL.view(np.int32)))
    out = buf[GUARD:GUARD + n].view(torch.float32).view(case.R, case.H, 512)
    if case.mode == "decode" and case.rows_per_slot > 1:
        dsa.dsa_sparse_attn_decode_rows(d["q"], d["kv"], d["idx"], d["n_sel"], d["sink"], case.scale, out,
                                        case.rows_per_slot)
    else:
        fn = dsa.dsa_sparse_attn_decode if case.mode == "decode" else dsa.dsa_sparse_attn_prefill
        fn(d["q"], d["kv"], d["idx"], d["n_sel"], d["sink"], case.scale, out)
    code = dsa.dsa_get_device_error()
    host = buf.cpu().numpy().view(np.uint32)
    if check_guards:
        assert np.all(host[:GUARD] == SENTINEL), "guard before out was written"
        assert np.all(host[GUARD + n:] == SENTINEL), "guard after out was written"
    res = host[GUARD:GUARD + n].view(np.float32).reshape(case.R, case.H, 512)
    assert not np.any(host[GUARD:GUARD + n] == SENTINEL), "some outputs were not written"
    return res.copy(), code


def classes_match(got, ref):
    """Nonfinite classes must agree element by element (NaN, +inf, -inf, finite)."""
    g = got.astype(np.float64)
    for name, f in (("nan", np.isnan), ("+inf", lambda a: a == np.inf), ("-inf", lambda a: a == -np.inf)):
        bad = f(g) != f(ref)
        if bad.any():
            i = tuple(np.argwhere(bad)[0])
            return False, "%s class differs at %s: gpu %r oracle %r" % (name, i, g[i], ref[i])
    return True, ""


def compare(case, got, ref):
    """Assert the stated tolerance: fp32 |g-o| <= 1e-6 + 1e-5|o|; bf16
    |g-o| <= 3e-3 * max|o| over the finite outputs of the same (row, head).
    Returns the worst error as a fraction of its limit."""
    ok, msg = classes_match(got, ref)
    assert ok, "%s: %s" % (case.name, msg)
    fin = np.isfinite(ref)
    g = got.astype(np.float64)
    err = np.where(fin, np.abs(g - np.where(fin, ref, 0.0)), 0.0)
    if case.dtype == I.F32:
        lim = TOL_F32_ABS + TOL_F32_REL * np.abs(np.where(fin, ref, 0.0))
    else:
        norm = np.max(np.where(fin, np.abs(ref), 0.0), axis=-1, keepdims=True)
        lim = TOL_BF16 * norm
    bad = err > lim
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError("%s: %d outputs out of tolerance; first at %s: gpu %r oracle %r (limit %g)"
                             % (case.name, int(bad.sum()), i, g[i], ref[i], lim[i]))
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(lim > 0, err / lim, 0.0)
    return float(np.max(r)) if r.size else 0.0
