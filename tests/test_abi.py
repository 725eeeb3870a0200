"""The C-ABI library: it loads, exports every declared symbol, and rejects
bad host-side arguments before touching the GPU (CPU only)."""

import os
import re
import subprocess

import pytest

from deepseek_v4_top_gb300 import dsa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from deepseek_v4_top_gb300 import build
    build.build()
    return dsa.load()


def _declared_functions():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:DSA_API\s+)?(?:const\s+)?\w+[\s\*]+(dsa_\w+)\s*\(",
                                text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert "dsa_sparse_attn_decode" in names and "dsa_sparse_attn_prefill" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(dsa.EXPORTS)


def test_only_the_c_abi_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", dsa.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    ours = {n for n in exported if n.startswith("dsa")}
    assert ours == set(dsa.EXPORTS)


def test_status_strings(lib):
    assert dsa.status_string(0) == "DSA_OK"
    assert dsa.status_string(1) == "DSA_ERR_INVALID_ARG"
    assert dsa.status_string(2) == "DSA_ERR_UNSUPPORTED"
    assert dsa.status_string(3) == "DSA_ERR_CUDA"
    assert dsa.status_string(4) == "DSA_ERR_DEVICE_CHECK"
    assert dsa.status_string(99) == "DSA_UNKNOWN_STATUS"


FAKE = 1 << 20     # a 16-byte-aligned non-null address; never dereferenced


@pytest.mark.parametrize("name", ["dsa_sparse_attn_decode", "dsa_sparse_attn_prefill"])
def test_host_validation_before_any_launch(lib, name):
    good = dict(q=FAKE, kv=FAKE, idx=FAKE, n_sel=FAKE, sink=FAKE, scale=0.1, out=FAKE,
                R=2, H=64, N=100, k_max=8, dtype=dsa.DSA_BF16)

    def call(**kw):
        a = dict(good)
        a.update(kw)
        return dsa.call_raw(name, a["q"], a["kv"], a["idx"], a["n_sel"], a["sink"], a["scale"],
                            a["out"], a["R"], a["H"], a["N"], a["k_max"], a["dtype"])

    for ptr in ("q", "kv", "idx", "n_sel", "sink", "out"):
        assert call(**{ptr: 0}) == dsa.DSA_ERR_INVALID_ARG
    assert call(q=FAKE + 8) == dsa.DSA_ERR_INVALID_ARG        # misaligned
    assert call(out=FAKE + 4) == dsa.DSA_ERR_INVALID_ARG
    assert call(R=-1) == dsa.DSA_ERR_INVALID_ARG
    assert call(N=0) == dsa.DSA_ERR_INVALID_ARG
    assert call(k_max=0) == dsa.DSA_ERR_INVALID_ARG
    assert call(H=0) == dsa.DSA_ERR_INVALID_ARG
    for h in (65, 128):
        assert call(H=h) == dsa.DSA_ERR_UNSUPPORTED
    assert call(dtype=7) == dsa.DSA_ERR_UNSUPPORTED
    # nothing to do: returns before any device work
    assert call(R=0, q=0, out=0) == dsa.DSA_OK


def test_device_error_query_rejects_null(lib):
    assert lib.dsa_get_device_error(None, None) == dsa.DSA_ERR_INVALID_ARG


def test_topk_host_validation_before_any_launch(lib):
    good = dict(scores=FAKE, ld=64, n_valid=FAKE, R=3, k=8, idx=FAKE, k_max=8, n_sel=FAKE)

    def call(**kw):
        a = dict(good)
        a.update(kw)
        return lib.dsa_topk_select(a["scores"], a["ld"], a["n_valid"], a["R"], a["k"], a["idx"],
                                   a["k_max"], a["n_sel"], None)

    for ptr in ("scores", "n_valid", "idx", "n_sel"):
        assert call(**{ptr: 0}) == dsa.DSA_ERR_INVALID_ARG
    assert call(scores=FAKE + 4) == dsa.DSA_ERR_INVALID_ARG     # misaligned rows
    assert call(ld=62) == dsa.DSA_ERR_INVALID_ARG                # not a multiple of 4
    assert call(ld=0) == dsa.DSA_ERR_INVALID_ARG
    assert call(k=0) == dsa.DSA_ERR_INVALID_ARG
    assert call(k=9) == dsa.DSA_ERR_INVALID_ARG                 # k > k_max
    assert call(R=-1) == dsa.DSA_ERR_INVALID_ARG
    assert call(k=2049, k_max=4096) == dsa.DSA_ERR_UNSUPPORTED
    assert call(ld=32772) == dsa.DSA_ERR_UNSUPPORTED
    assert call(R=0, scores=0) == dsa.DSA_OK


def test_general_call_and_projection_host_validation(lib):
    def attn(**kw):
        a = dict(q=FAKE, kv=FAKE, idx=FAKE, n_sel=FAKE, sink=FAKE, out=FAKE, R=4, T=0, out_dtype=dsa.DSA_BF16)
        a.update(kw)
        return lib.dsa_sparse_attn(a["q"], a["kv"], a["idx"], a["n_sel"], a["sink"], 0.1, a["out"], a["R"],
                                   a["T"], 64, 100, 8, dsa.DSA_BF16, a["out_dtype"], None)
    assert attn(T=3) == dsa.DSA_ERR_INVALID_ARG                # rows not a multiple of rows_per_slot
    assert attn(T=-1) == dsa.DSA_ERR_INVALID_ARG
    assert attn(out_dtype=7) == dsa.DSA_ERR_UNSUPPORTED
    assert attn(out=FAKE + 2) == dsa.DSA_ERR_INVALID_ARG       # misaligned out
    assert attn(R=0, q=0, out=0) == dsa.DSA_OK

    def whole(**kw):
        a = dict(q=FAKE, kv=FAKE, idx=FAKE, n_sel=FAKE, sink=FAKE, out=FAKE, R=4, T=1, out_dtype=dsa.DSA_F32)
        a.update(kw)
        return lib.dsa_sparse_attn_decode_whole_rows(a["q"], a["kv"], a["idx"], a["n_sel"], a["sink"], 0.1,
                                                     a["out"], a["R"], a["T"], 64, 100, 8, dsa.DSA_BF16,
                                                     a["out_dtype"], None)
    assert whole(T=0) == dsa.DSA_ERR_INVALID_ARG               # decode needs rows_per_slot >= 1
    assert whole(T=3) == dsa.DSA_ERR_INVALID_ARG               # rows not a multiple of rows_per_slot
    assert whole(R=-1) == dsa.DSA_ERR_INVALID_ARG
    for ptr in ("q", "kv", "idx", "n_sel", "sink", "out"):
        assert whole(**{ptr: 0}) == dsa.DSA_ERR_INVALID_ARG
    assert whole(out_dtype=7) == dsa.DSA_ERR_UNSUPPORTED
    assert whole(R=0, q=0, out=0) == dsa.DSA_OK

    def proj(**kw):
        a = dict(attn=FAKE, w=FAKE, out=FAKE, R=4, K=512, d_out=64)
        a.update(kw)
        return lib.dsa_oproj(a["attn"], a["w"], a["out"], a["R"], a["K"], a["d_out"], None)
    for ptr in ("attn", "w", "out"):
        assert proj(**{ptr: 0}) == dsa.DSA_ERR_INVALID_ARG
    assert proj(K=0) == dsa.DSA_ERR_INVALID_ARG
    assert proj(K=12) == dsa.DSA_ERR_INVALID_ARG               # not a multiple of 8
    assert proj(d_out=6) == dsa.DSA_ERR_INVALID_ARG
    assert proj(w=FAKE + 8) == dsa.DSA_ERR_INVALID_ARG
    assert proj(R=-1) == dsa.DSA_ERR_INVALID_ARG
    assert proj(R=0, attn=0, w=0, out=0) == dsa.DSA_OK

    def fused(**kw):
        a = dict(w=FAKE, attn=FAKE, out=FAKE, d_out=64)
        a.update(kw)
        return lib.dsa_sparse_attn_prefill_oproj(FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, a["w"], a["attn"], a["out"],
                                                 4, 64, 100, 8, a["d_out"], None)
    assert fused(w=0) == dsa.DSA_ERR_INVALID_ARG
    assert fused(attn=0) == dsa.DSA_ERR_INVALID_ARG
    assert fused(d_out=4) == dsa.DSA_ERR_INVALID_ARG


def test_decode_rows_host_validation(lib):
    def call(B=2, T=2, **kw):
        a = dict(q=FAKE, kv=FAKE, idx=FAKE, n_sel=FAKE, sink=FAKE, out=FAKE)
        a.update(kw)
        return lib.dsa_sparse_attn_decode_rows(a["q"], a["kv"], a["idx"], a["n_sel"], a["sink"], 0.1,
                                               a["out"], B, T, 64, 100, 8, dsa.DSA_BF16, None)
    assert call(T=0) == dsa.DSA_ERR_INVALID_ARG
    assert call(B=-1) == dsa.DSA_ERR_INVALID_ARG
    assert call(B=1 << 20, T=1 << 12) == dsa.DSA_ERR_INVALID_ARG     # rows beyond int range
    assert call(q=0) == dsa.DSA_ERR_INVALID_ARG
    assert call(B=0, q=0, out=0) == dsa.DSA_OK


def test_decode_cache_limit_counts_slots_not_rows(lib):
    # 2 slots x 16384 rows a slot over 65536 positions: rows x N reaches 2^31,
    # slots x N does not, so the call passes the host checks (on a machine
    # without a GPU it then fails at the device, not on its arguments)
    st = lib.dsa_sparse_attn_decode_rows(FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, FAKE, 2, 1 << 14, 64, 1 << 16, 8,
                                         dsa.DSA_BF16, None)
    assert st != dsa.DSA_ERR_INVALID_ARG
    st = lib.dsa_sparse_attn_decode_rows(FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, FAKE, 1 << 15, 1, 64, 1 << 16, 8,
                                         dsa.DSA_BF16, None)
    assert st == dsa.DSA_ERR_INVALID_ARG          # 32768 slots x 65536 positions


def test_head_shard_kernels_host_validation(lib):
    def shard(**kw):
        a = dict(q=FAKE, sink=FAKE, ql=FAKE, sl=FAKE, R=4, H=64, world=4, rank=1, dtype=dsa.DSA_BF16)
        a.update(kw)
        return lib.dsa_shard_heads(a["q"], a["sink"], a["ql"], a["sl"], a["R"], a["H"], a["world"], a["rank"],
                                   a["dtype"], None)
    for ptr in ("q", "sink", "ql", "sl"):
        assert shard(**{ptr: 0}) == dsa.DSA_ERR_INVALID_ARG
    assert shard(q=FAKE + 8) == dsa.DSA_ERR_INVALID_ARG
    assert shard(R=-1) == dsa.DSA_ERR_INVALID_ARG
    assert shard(rank=4) == dsa.DSA_ERR_INVALID_ARG
    assert shard(world=0) == dsa.DSA_ERR_INVALID_ARG
    assert shard(H=300, world=2) == dsa.DSA_ERR_UNSUPPORTED   # 150 heads a rank
    assert shard(dtype=7) == dsa.DSA_ERR_UNSUPPORTED
    assert shard(R=0, q=0, sink=0, ql=0, sl=0) == dsa.DSA_OK

    def unshard(**kw):
        a = dict(g=FAKE, out=FAKE, R=4, H=64, world=4, dtype=dsa.DSA_F32)
        a.update(kw)
        return lib.dsa_unshard_heads(a["g"], a["out"], a["R"], a["H"], a["world"], a["dtype"], None)
    assert unshard(g=0) == dsa.DSA_ERR_INVALID_ARG
    assert unshard(out=0) == dsa.DSA_ERR_INVALID_ARG
    assert unshard(out=FAKE + 4) == dsa.DSA_ERR_INVALID_ARG
    assert unshard(R=-1) == dsa.DSA_ERR_INVALID_ARG
    assert unshard(world=-2) == dsa.DSA_ERR_INVALID_ARG
    assert unshard(dtype=5) == dsa.DSA_ERR_UNSUPPORTED
    assert unshard(R=0, g=0, out=0) == dsa.DSA_OK


def test_binding_refuses_tensors_and_streams_of_another_device(monkeypatch):
    """The library launches on the current device; the binding refuses a
    tensor or a stream that lives on another one (its addresses would not be
    valid there) before anything reaches the C ABI."""
    import types

    import torch
    from deepseek_v4_top_gb300 import dsa
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    here = types.SimpleNamespace(device=types.SimpleNamespace(index=0))
    there = types.SimpleNamespace(device=types.SimpleNamespace(index=1))
    dsa._same_device(("a", here), ("b", here))
    with pytest.raises(ValueError, match="cuda:1"):
        dsa._same_device(("a", here), ("b", there))
    stream = types.SimpleNamespace(device=types.SimpleNamespace(index=1), cuda_stream=1234)
    with pytest.raises(ValueError, match="stream"):
        dsa._stream_handle(stream)
    ok = types.SimpleNamespace(device=types.SimpleNamespace(index=0), cuda_stream=1234)
    assert dsa._stream_handle(ok) == 1234
    assert dsa._stream_handle(5678) == 5678
