"""Python binding of libdsa.so: the C ABI of include/dsa.h under the same names.

Argument marshalling only.  Every step of the attention runs in the CUDA
kernels of libdsa.so; PyTorch provides device memory and the current stream.
There is no fallback: if the library is missing or the GPU is unsupported,
the calls raise.
"""

from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdsa.so")

DSA_OK = 0
DSA_ERR_INVALID_ARG = 1
DSA_ERR_UNSUPPORTED = 2
DSA_ERR_CUDA = 3
DSA_ERR_DEVICE_CHECK = 4

DSA_F32 = 0
DSA_BF16 = 1

DSA_DEVERR_IDX_RANGE = 0x1
DSA_DEVERR_NSEL_RANGE = 0x2
DSA_DEVERR_TIMEOUT = 0x4
DSA_DEVERR_LAYOUT = 0x8
DSA_DEVERR_NVALID_RANGE = 0x10

# Every function declared in include/dsa.h.
EXPORTS = ("dsa_sparse_attn_decode", "dsa_sparse_attn_decode_rows", "dsa_sparse_attn_prefill",
           "dsa_sparse_attn", "dsa_sparse_attn_decode_whole_rows", "dsa_oproj", "dsa_sparse_attn_prefill_oproj",
           "dsa_sparse_attn_decode_noalloc",
           "dsa_topk_select", "dsa_head_shard", "dsa_shard_heads", "dsa_unshard_heads",
           "dsa_selftest_wait_limit", "dsa_get_device_error", "dsa_status_string", "dsa_shutdown")
DSA_NOALLOC_MAX_UNITS = 64

_lib = None
_lock = threading.Lock()


class HeadShardPlan(ctypes.Structure):
    """dsa_head_shard_plan of include/dsa.h."""
    _fields_ = [("heads_per_rank", ctypes.c_int), ("padded_heads", ctypes.c_int),
                ("first_head", ctypes.c_int), ("real_heads", ctypes.c_int)]


class DsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s returned %s" % (where, status_string(status)))


def load():
    """Load libdsa.so (it must have been built; see __graft_entry__.build)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("libdsa.so is not built: run __graft_entry__.build() first")
            lib = ctypes.CDLL(LIB_PATH)
            P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            sig = [P, P, P, P, P, F, P, I, I, I, I, I, P]
            for name in ("dsa_sparse_attn_decode", "dsa_sparse_attn_prefill",
                         "dsa_sparse_attn_decode_noalloc"):
                fn = getattr(lib, name)
                fn.argtypes = sig
                fn.restype = I
            lib.dsa_sparse_attn_decode_rows.argtypes = [P, P, P, P, P, F, P, I, I, I, I, I, I, P]
            lib.dsa_sparse_attn_decode_rows.restype = I
            lib.dsa_sparse_attn.argtypes = [P, P, P, P, P, F, P, I, I, I, I, I, I, I, P]
            lib.dsa_sparse_attn.restype = I
            lib.dsa_sparse_attn_decode_whole_rows.argtypes = [P, P, P, P, P, F, P, I, I, I, I, I, I, I, P]
            lib.dsa_sparse_attn_decode_whole_rows.restype = I
            lib.dsa_oproj.argtypes = [P, P, P, I, I, I, P]
            lib.dsa_oproj.restype = I
            lib.dsa_sparse_attn_prefill_oproj.argtypes = [P, P, P, P, P, F, P, P, P, I, I, I, I, I, P]
            lib.dsa_sparse_attn_prefill_oproj.restype = I
            lib.dsa_topk_select.argtypes = [P, I, P, I, I, P, I, P, P]
            lib.dsa_topk_select.restype = I
            lib.dsa_head_shard.argtypes = [I, I, I, ctypes.POINTER(HeadShardPlan)]
            lib.dsa_head_shard.restype = I
            lib.dsa_shard_heads.argtypes = [P, P, P, P, I, I, I, I, I, P]
            lib.dsa_shard_heads.restype = I
            lib.dsa_unshard_heads.argtypes = [P, P, I, I, I, I, P]
            lib.dsa_unshard_heads.restype = I
            lib.dsa_selftest_wait_limit.argtypes = [P]
            lib.dsa_selftest_wait_limit.restype = I
            lib.dsa_get_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
            lib.dsa_get_device_error.restype = I
            lib.dsa_status_string.argtypes = [I]
            lib.dsa_status_string.restype = ctypes.c_char_p
            lib.dsa_shutdown.argtypes = []
            lib.dsa_shutdown.restype = I
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().dsa_status_string(int(status)).decode()


# ------------------------------------------------------------- raw pointers
def call_raw(name: str, q: int, kv: int, idx: int, n_sel: int, sink: int, scale: float, out: int,
             R: int, H: int, N: int, k_max: int, dtype: int, stream: int = 0) -> int:
    """Call an entry point with integer device addresses; returns the status."""
    fn = getattr(load(), name)
    return int(fn(q, kv, idx, n_sel, sink, ctypes.c_float(scale), out, R, H, N, k_max, dtype,
                  stream))


# ------------------------------------------------------------ torch tensors
def _same_device(*pairs):
    """Every tensor must be on the current CUDA device: the library launches
    there, and another device's addresses are not valid in its kernels."""
    import torch
    cur = torch.cuda.current_device()
    for name, t in pairs:
        if t.device.index != cur:
            raise ValueError("%s is on cuda:%s, but the calls run on the current device cuda:%d "
                             "(torch.cuda.set_device)" % (name, t.device.index, cur))


def _dtype_code(t):
    import torch
    if t.dtype == torch.float32:
        return DSA_F32
    if t.dtype == torch.bfloat16:
        return DSA_BF16
    raise TypeError("q and kv_cache must be float32 or bfloat16, got %s" % t.dtype)


def _check(q, kv, idx, n_sel, sink, out, decode, rows_per_slot=1, out_dtype=None):
    import torch
    for name, t in (("q", q), ("kv_cache", kv), ("idx", idx), ("n_sel", n_sel), ("sink", sink),
                    ("out", out)):
        if not isinstance(t, torch.Tensor):
            raise TypeError("%s must be a torch.Tensor" % name)
        if not t.is_cuda:
            raise ValueError("%s must be a CUDA tensor" % name)
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % name)
    _same_device(("q", q), ("kv_cache", kv), ("idx", idx), ("n_sel", n_sel), ("sink", sink), ("out", out))
    if kv.dtype != q.dtype:
        raise TypeError("q and kv_cache must have the same dtype")
    if idx.dtype != torch.int32 or n_sel.dtype != torch.int32:
        raise TypeError("idx and n_sel must be int32")
    if sink.dtype != torch.float32:
        raise TypeError("sink must be float32")
    if out.dtype != (torch.float32 if out_dtype is None else out_dtype):
        raise TypeError("out must be %s" % ("float32" if out_dtype is None else out_dtype))
    if q.dim() != 3 or q.shape[2] != 512:
        raise ValueError("q must be [rows, heads, 512]")
    R, H = q.shape[0], q.shape[1]
    if decode:
        if kv.dim() != 3 or kv.shape[0] * rows_per_slot != R or kv.shape[2] != 512:
            raise ValueError("decode kv_cache must be [slots, N, 512] with slots * rows_per_slot = rows")
        N = kv.shape[1]
    else:
        if kv.dim() != 2 or kv.shape[1] != 512:
            raise ValueError("prefill kv_cache must be [N, 512]")
        N = kv.shape[0]
    if idx.dim() != 2 or idx.shape[0] != R:
        raise ValueError("idx must be [rows, k_max]")
    if tuple(n_sel.shape) != (R,) or tuple(sink.shape) != (H,) or tuple(out.shape) != (R, H, 512):
        raise ValueError("n_sel [rows], sink [heads] and out [rows, heads, 512] expected")
    return R, H, N, idx.shape[1]


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    if hasattr(stream, "device") and getattr(stream.device, "index", None) is not None:
        if stream.device.index != torch.cuda.current_device():
            raise ValueError("the stream belongs to cuda:%d, but the calls run on the current device cuda:%d"
                             % (stream.device.index, torch.cuda.current_device()))
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _run(name, decode, q, kv_cache, idx, n_sel, sink, scale, out, stream):
    R, H, N, k_max = _check(q, kv_cache, idx, n_sel, sink, out, decode)
    st = call_raw(name, q.data_ptr(), kv_cache.data_ptr(), idx.data_ptr(), n_sel.data_ptr(),
                  sink.data_ptr(), float(scale), out.data_ptr(), R, H, N, k_max,
                  _dtype_code(q), _stream_handle(stream))
    if st != DSA_OK:
        raise DsaError(st, name)
    return out


def dsa_sparse_attn_decode(q, kv_cache, idx, n_sel, sink, scale, out, stream=None):
    """Decode attention: q [B,H,512], kv_cache [B,N,512], out [B,H,512] fp32."""
    return _run("dsa_sparse_attn_decode", True, q, kv_cache, idx, n_sel, sink, scale, out, stream)


def dsa_sparse_attn_decode_rows(q, kv_cache, idx, n_sel, sink, scale, out, rows_per_slot, stream=None):
    """Decode with T = rows_per_slot query rows a slot: q [B*T,H,512], kv_cache [B,N,512],
    idx [B*T,k_max], n_sel [B*T], out [B*T,H,512] fp32; row r reads slot r // T."""
    T = int(rows_per_slot)
    if T < 1:
        raise ValueError("rows_per_slot must be >= 1")
    if kv_cache.dim() != 3 or q.dim() != 3 or q.shape[0] != kv_cache.shape[0] * T:
        raise ValueError("q must be [slots * rows_per_slot, heads, 512] for kv_cache [slots, N, 512]")
    R, H, N, k_max = _check(q, kv_cache, idx, n_sel, sink, out, decode=True, rows_per_slot=T)
    st = load().dsa_sparse_attn_decode_rows(q.data_ptr(), kv_cache.data_ptr(), idx.data_ptr(),
                                            n_sel.data_ptr(), sink.data_ptr(), ctypes.c_float(float(scale)),
                                            out.data_ptr(), R // T, T, H, N, k_max, _dtype_code(q),
                                            _stream_handle(stream))
    if st != DSA_OK:
        raise DsaError(st, "dsa_sparse_attn_decode_rows")
    return out


def dsa_sparse_attn_prefill(q, kv_cache, idx, n_sel, sink, scale, out, stream=None):
    """Prefill attention: q [R,H,512], kv_cache [N,512], out [R,H,512] fp32."""
    return _run("dsa_sparse_attn_prefill", False, q, kv_cache, idx, n_sel, sink, scale, out, stream)


def dsa_sparse_attn(q, kv_cache, idx, n_sel, sink, scale, out, rows_per_slot=0, stream=None):
    """Attention with the output type taken from `out` (float32 or bfloat16):
    rows_per_slot 0 is prefill (kv_cache [N,512]), T >= 1 decode with T rows a
    slot (kv_cache [R/T,N,512]).  A bf16 out holds the float32 result rounded
    to nearest even."""
    import torch
    T = int(rows_per_slot)
    if T < 0:
        raise ValueError("rows_per_slot must be >= 0")
    if not isinstance(out, torch.Tensor) or out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out must be a float32 or bfloat16 tensor")
    R, H, N, k_max = _check(q, kv_cache, idx, n_sel, sink, out, decode=T > 0, rows_per_slot=max(T, 1),
                            out_dtype=out.dtype)
    st = load().dsa_sparse_attn(q.data_ptr(), kv_cache.data_ptr(), idx.data_ptr(), n_sel.data_ptr(),
                                sink.data_ptr(), ctypes.c_float(float(scale)), out.data_ptr(), R, T, H, N,
                                k_max, _dtype_code(q), _dtype_code(out), _stream_handle(stream))
    if st != DSA_OK:
        raise DsaError(st, "dsa_sparse_attn")
    return out


def dsa_sparse_attn_decode_whole_rows(q, kv_cache, idx, n_sel, sink, scale, out, rows_per_slot=1, stream=None):
    """Decode without the key split (each row whole in one CTA, no partials):
    q [B*T,H,512], kv_cache [B,N,512], idx [B*T,k_max], n_sel [B*T], out
    [B*T,H,512] float32 or bfloat16; row r reads slot r // T (T =
    rows_per_slot).  For batches of about as many rows as SMs or more."""
    import torch
    T = int(rows_per_slot)
    if T < 1:
        raise ValueError("rows_per_slot must be >= 1")
    if not isinstance(out, torch.Tensor) or out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("out must be a float32 or bfloat16 tensor")
    if kv_cache.dim() != 3 or q.dim() != 3 or q.shape[0] != kv_cache.shape[0] * T:
        raise ValueError("q must be [slots * rows_per_slot, heads, 512] for kv_cache [slots, N, 512]")
    R, H, N, k_max = _check(q, kv_cache, idx, n_sel, sink, out, decode=True, rows_per_slot=T, out_dtype=out.dtype)
    st = load().dsa_sparse_attn_decode_whole_rows(q.data_ptr(), kv_cache.data_ptr(), idx.data_ptr(),
                                                  n_sel.data_ptr(), sink.data_ptr(), ctypes.c_float(float(scale)),
                                                  out.data_ptr(), R, T, H, N, k_max, _dtype_code(q),
                                                  _dtype_code(out), _stream_handle(stream))
    if st != DSA_OK:
        raise DsaError(st, "dsa_sparse_attn_decode_whole_rows")
    return out


def _check_oproj(attn, w_o, out):
    import torch
    for name, t in (("attn", attn), ("w_o", w_o), ("out", out)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA tensor" % name)
    _same_device(("attn", attn), ("w_o", w_o), ("out", out))
    if attn.dtype != torch.bfloat16 or w_o.dtype != torch.bfloat16 or out.dtype != torch.float32:
        raise TypeError("attn and w_o must be bfloat16, out float32")
    if w_o.dim() != 2 or out.dim() != 2:
        raise ValueError("w_o [K, d_out] and out [rows, d_out] expected")
    R, K, d_out = attn.shape[0], w_o.shape[0], w_o.shape[1]
    if attn.numel() != R * K or tuple(out.shape) != (R, d_out):
        raise ValueError("attn [rows, K] (or [rows, H, 512] with H*512 = K) and out [rows, d_out] expected")
    return R, K, d_out


def dsa_oproj(attn, w_o, out, stream=None):
    """Output projection: out [R,d_out] fp32 = attn [R,K] bf16 . w_o [K,d_out] bf16."""
    R, K, d_out = _check_oproj(attn, w_o, out)
    st = load().dsa_oproj(attn.data_ptr(), w_o.data_ptr(), out.data_ptr(), R, K, d_out, _stream_handle(stream))
    if st != DSA_OK:
        raise DsaError(st, "dsa_oproj")
    return out


def dsa_sparse_attn_prefill_oproj(q, kv_cache, idx, n_sel, sink, scale, w_o, attn, out, stream=None):
    """Prefill attention (bf16 q/kv) into attn [R,H,512] bf16, then
    out [R,d_out] fp32 = attn . w_o [H*512,d_out] bf16."""
    R, H, N, k_max = _check(q, kv_cache, idx, n_sel, sink, attn, decode=False, out_dtype=attn.dtype)
    R2, K, d_out = _check_oproj(attn, w_o, out)
    if K != H * 512 or R2 != R:
        raise ValueError("w_o must be [heads * 512, d_out]")
    st = load().dsa_sparse_attn_prefill_oproj(q.data_ptr(), kv_cache.data_ptr(), idx.data_ptr(), n_sel.data_ptr(),
                                              sink.data_ptr(), ctypes.c_float(float(scale)), w_o.data_ptr(),
                                              attn.data_ptr(), out.data_ptr(), R, H, N, k_max, d_out,
                                              _stream_handle(stream))
    if st != DSA_OK:
        raise DsaError(st, "dsa_sparse_attn_prefill_oproj")
    return out


def dsa_sparse_attn_decode_noalloc(q, kv_cache, idx, n_sel, sink, scale, out, stream=None):
    """Decode attention that allocates no device memory (fixed static scratch;
    see include/dsa.h for its size limit and its sharing rules)."""
    return _run("dsa_sparse_attn_decode_noalloc", True, q, kv_cache, idx, n_sel, sink, scale, out,
                stream)


def dsa_topk_select(scores, n_valid, k, idx, n_sel, stream=None):
    """Top-k selection of each row of scores [R, ld] (float32) among positions
    [0, n_valid[r]) into idx [R, k_max] and n_sel [R] (int32)."""
    import torch
    for name, t in (("scores", scores), ("n_valid", n_valid), ("idx", idx), ("n_sel", n_sel)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA tensor" % name)
    _same_device(("scores", scores), ("n_valid", n_valid), ("idx", idx), ("n_sel", n_sel))
    if scores.dtype != torch.float32 or scores.dim() != 2:
        raise TypeError("scores must be a float32 [rows, ld] tensor")
    if n_valid.dtype != torch.int32 or idx.dtype != torch.int32 or n_sel.dtype != torch.int32:
        raise TypeError("n_valid, idx and n_sel must be int32")
    R, ld = scores.shape
    if tuple(n_valid.shape) != (R,) or tuple(n_sel.shape) != (R,) or idx.dim() != 2 or idx.shape[0] != R:
        raise ValueError("n_valid [rows], idx [rows, k_max] and n_sel [rows] expected")
    st = load().dsa_topk_select(scores.data_ptr(), ld, n_valid.data_ptr(), R, int(k), idx.data_ptr(),
                                idx.shape[1], n_sel.data_ptr(), _stream_handle(stream))
    if st != DSA_OK:
        raise DsaError(st, "dsa_topk_select")
    return idx, n_sel


# ------------------------------------------------- head-sharded parallelism
def dsa_head_shard(H: int, world: int, rank: int) -> HeadShardPlan:
    """Which heads rank `rank` of `world` owns (host only; see include/dsa.h)."""
    plan = HeadShardPlan()
    st = load().dsa_head_shard(int(H), int(world), int(rank), ctypes.byref(plan))
    if st != DSA_OK:
        raise DsaError(st, "dsa_head_shard")
    return plan


def dsa_shard_heads(q, sink, q_local, sink_local, world: int, rank: int, stream=None):
    """q_local [R,hpr,512], sink_local [hpr] = rank's heads of q [R,H,512],
    sink [H] (zero for padding heads)."""
    import torch
    for name, t in (("q", q), ("sink", sink), ("q_local", q_local), ("sink_local", sink_local)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA tensor" % name)
    _same_device(("q", q), ("sink", sink), ("q_local", q_local), ("sink_local", sink_local))
    if q.dim() != 3 or q.shape[2] != 512 or q_local.dtype != q.dtype:
        raise ValueError("q [rows, heads, 512] and q_local of the same dtype expected")
    R, H = q.shape[0], q.shape[1]
    plan = dsa_head_shard(H, world, rank)
    if tuple(q_local.shape) != (R, plan.heads_per_rank, 512) or tuple(sink.shape) != (H,) \
            or tuple(sink_local.shape) != (plan.heads_per_rank,):
        raise ValueError("q_local [rows, heads_per_rank, 512], sink [heads], sink_local [heads_per_rank] expected")
    if sink.dtype != torch.float32 or sink_local.dtype != torch.float32:
        raise TypeError("sinks must be float32")
    st = load().dsa_shard_heads(q.data_ptr(), sink.data_ptr(), q_local.data_ptr(), sink_local.data_ptr(),
                                R, H, int(world), int(rank), _dtype_code(q), _stream_handle(stream))
    if st != DSA_OK:
        raise DsaError(st, "dsa_shard_heads")
    return q_local, sink_local


def dsa_unshard_heads(gathered, out, world: int, stream=None):
    """out [R,H,512] from gathered [world,R,hpr,512] (padding heads dropped)."""
    import torch
    for name, t in (("gathered", gathered), ("out", out)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA tensor" % name)
    _same_device(("gathered", gathered), ("out", out))
    if out.dim() != 3 or out.shape[2] != 512 or gathered.dtype != out.dtype:
        raise ValueError("out [rows, heads, 512] and gathered of the same dtype expected")
    R, H = out.shape[0], out.shape[1]
    plan = dsa_head_shard(H, world, 0)
    if tuple(gathered.shape) != (world, R, plan.heads_per_rank, 512):
        raise ValueError("gathered must be [world, rows, heads_per_rank, 512]")
    st = load().dsa_unshard_heads(gathered.data_ptr(), out.data_ptr(), R, H, int(world), _dtype_code(out),
                                  _stream_handle(stream))
    if st != DSA_OK:
        raise DsaError(st, "dsa_unshard_heads")
    return out


def tp_sparse_attn(q_local, kv_cache, idx, n_sel, sink_local, scale, out_local, gathered, out, group=None,
                   rows_per_slot=0, stream=None):
    """One rank's step of head-sharded attention, all on one stream (torch's
    current one unless `stream` is given): the attention call over the rank's
    heads into out_local [R,hpr,512], an all-gather of every rank's out_local
    into gathered [world,R,hpr,512] (torch.distributed on `group`; NCCL on
    GPUs), then the gathered outputs laid out as out [R,H,512].  With one
    rank, out_local itself is the gathered array."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group) if dist.is_available() and dist.is_initialized() else 1
    with torch.cuda.stream(stream if stream is not None else torch.cuda.current_stream()):
        dsa_sparse_attn(q_local, kv_cache, idx, n_sel, sink_local, scale, out_local,
                        rows_per_slot=rows_per_slot)
        if world > 1:
            dist.all_gather_into_tensor(gathered.view(-1), out_local.view(-1), group=group)
            src = gathered
        else:
            src = out_local.view((1,) + tuple(out_local.shape))
        return dsa_unshard_heads(src, out, world)


def tp_oproj_weights(w_o, H: int, world: int, rank: int):
    """The rank's rows of the output projection w_o [H*512, d_out] (bf16) for
    tp_sparse_attn_oproj: its heads' 512-row blocks, then zero blocks for its
    padding heads, whose attention outputs (q = 0, sink = 0) must not reach
    the projection.  One-time weight preparation: a view of w_o when the rank
    has no padding heads, else a padded copy."""
    import torch
    if not isinstance(w_o, torch.Tensor) or w_o.dim() != 2 or w_o.shape[0] != H * 512:
        raise ValueError("w_o must be a [heads * 512, d_out] tensor")
    plan = dsa_head_shard(H, world, rank)
    lo, n = plan.first_head * 512, plan.real_heads * 512
    if plan.real_heads == plan.heads_per_rank:
        return w_o[lo:lo + n]
    local = torch.zeros((plan.heads_per_rank * 512, w_o.shape[1]), dtype=w_o.dtype, device=w_o.device)
    local[:n].copy_(w_o[lo:lo + n])
    return local


def tp_sparse_attn_oproj(q_local, kv_cache, idx, n_sel, sink_local, scale, w_o_local, attn_local, out,
                         group=None, rows_per_slot=0, stream=None, scatter_out=None):
    """One rank's step of head-sharded attention followed by the output
    projection, row-parallel, all on one stream (torch's current one unless
    `stream` is given): the attention over the rank's heads into attn_local
    [R,hpr,512] (bf16), the rank's share of the projection out [R,d_out] fp32
    = attn_local . w_o_local (w_o_local from tp_oproj_weights), then a sum
    of every rank's share over `group` (torch.distributed all-reduce; NCCL on
    GPUs), so that every rank holds the whole projection.  Against
    tp_sparse_attn followed by the projection, the ranks exchange the
    projected rows (R x d_out fp32) instead of the attention outputs
    (R x H x 512 bf16).  The shares are summed in the collective's order, so
    the result differs from the one-GPU projection by fp32 rounding.

    With `scatter_out` ([R / world, d_out] float32, R a multiple of the world
    size) the sum is reduce-scattered instead: rank w receives rows
    [w R / world, (w + 1) R / world) of the projection in scatter_out, and
    `out` keeps the rank's own unsummed share.  Returns the tensor that holds
    the summed rows."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group) if dist.is_available() and dist.is_initialized() else 1
    if attn_local.dtype != torch.bfloat16:
        raise TypeError("attn_local must be bfloat16 (the projection's A operand)")
    R = attn_local.shape[0]
    if scatter_out is not None:
        if (not isinstance(scatter_out, torch.Tensor) or scatter_out.dtype != torch.float32
                or not scatter_out.is_contiguous() or R % world != 0
                or tuple(scatter_out.shape) != (R // world, out.shape[-1])):
            raise ValueError("scatter_out must be a contiguous float32 [rows / world, d_out] tensor, "
                             "rows a multiple of the world size")
        _same_device(("out", out), ("scatter_out", scatter_out))
    with torch.cuda.stream(stream if stream is not None else torch.cuda.current_stream()):
        dsa_sparse_attn(q_local, kv_cache, idx, n_sel, sink_local, scale, attn_local,
                        rows_per_slot=rows_per_slot)
        dsa_oproj(attn_local.view(R, -1), w_o_local, out)
        if scatter_out is not None:
            if world > 1:
                dist.reduce_scatter_tensor(scatter_out, out, op=dist.ReduceOp.SUM, group=group)
            else:
                scatter_out.copy_(out)
            return scatter_out
        if world > 1:
            dist.all_reduce(out, op=dist.ReduceOp.SUM, group=group)
        return out


def dsa_selftest_wait_limit(stream=None) -> None:
    """Queue the bounded-wait self-test (sets DSA_DEVERR_TIMEOUT after ~2 s)."""
    st = load().dsa_selftest_wait_limit(_stream_handle(stream))
    if st != DSA_OK:
        raise DsaError(st, "dsa_selftest_wait_limit")


def dsa_get_device_error(stream=None) -> int:
    """Synchronise the stream, return and clear the device error word."""
    code = ctypes.c_uint32(0)
    st = load().dsa_get_device_error(_stream_handle(stream), ctypes.byref(code))
    if st != DSA_OK:
        raise DsaError(st, "dsa_get_device_error")
    return int(code.value)


def dsa_shutdown() -> None:
    st = load().dsa_shutdown()
    if st != DSA_OK:
        raise DsaError(st, "dsa_shutdown")
