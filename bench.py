"""Benchmark of the top-k sparse-attention hot path on GB300.

One step = one batched decode call (8 slots x 32768-position caches) and one
prefill call (2048 rows at positions 2048..4095 of a 4096-position cache), both
with 64 heads, 512-wide latent rows, k = 640 selected keys, bf16 inputs; the
two independent calls are issued on two streams at once.  Metric: row*heads
per second (whole job), plus each call's own time and gathered-KV GB/s, timed
one call after the other on one stream.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs the same per-GPU workload (weak scaling); the
step time is the maximum over ranks.  --impl reference times the fp64 CPU
oracle on the host cores on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from deepseek_v4_top_gb300 import inputs as I  # noqa: E402

H, D, K = 64, 512, 640
E2E_CHUNKS = 8                              # prefill row chunks in the end-to-end step
OPROJ_D_OUT = 7168                          # output projection width timed (DeepSeek-V3's model width;
                                            # the pages give none for V4.1)
DEC_B, DEC_N = 8, 32768
DEC_BIG_B = 608                             # a decode batch that fills the GPU: four rows an SM
PRE_R, PRE_N = 2048, 4096
METRIC = "sparse-attn row·heads/s and HBM GB/s at H=64,d=512,k=640 (decode B=8, prefill 2048)"
WORKLOAD = ("decode B=8 x 1 row (N=32768 per slot) + prefill 2048 rows (positions 2048..4095, "
            "N=4096); H=64, d=512, k=640, bf16 q/kv, fp32 out")
UNITS_PER_STEP = (DEC_B + PRE_R) * H        # row*heads
FLOPS_PER_ROW = 4 * H * D * K              # q.k and p.v, one row, all heads


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "of measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "of fallback"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def compulsory_bytes(rows: int, kv_bytes: int) -> int:
    """Bytes a call must move to or from HBM at least: q (bf16) and idx in,
    out (fp32) back, and the KV rows it reads (decode: the gathered rows,
    each slot's cache being far larger than L2; prefill: the whole 4 MiB
    cache, which then stays in L2)."""
    return rows * H * D * 2 + rows * K * 4 + rows * H * D * 4 + kv_bytes


def reduce_max(value: float, world: int) -> float:
    """Maximum of a per-rank float over the process group (identity when alone)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        rows = [s for (t, s) in self.samples if t0 <= t <= t1 + 0.05] or [s for (_, s) in self.samples]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if len(r) > 1 and num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if len(r) > 2 and num(r[2]) is not None]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if len(r) > 5 + i and r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- traffic
def recorded_traffic():
    """DRAM bytes per prefill launch from the committed ncu summary, if the
    kernel source is still the one the counters were taken on."""
    path = os.path.join(ROOT, "profiles", "dsa_tc_kernel_prefill2048.md")
    src = os.path.join(ROOT, "deepseek_v4_top_gb300", "csrc", "dsa_tc.cu")
    try:
        text = open(path).read()
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.e+]+)", text)
    if not m_sha or not m_b or m_sha.group(1) != sha:
        return None
    return float(m_b.group(1))


# ------------------------------------------------------------ CPU oracle
def host_cores():
    """(cores this process may run on, cores the host has online)."""
    try:
        usable = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        usable = os.cpu_count() or 1
    try:
        online = os.sysconf("SC_NPROCESSORS_ONLN")
    except (AttributeError, ValueError, OSError):
        online = os.cpu_count() or usable
    return usable, online


def oracle_sample(pre, dec, target_s: float, rows_cap: int = PRE_R):
    """Time the fp64 oracle on whole rows (all 64 heads) of both workloads,
    growing the sample until it takes about target_s on all threads, then on
    one thread for about a fifth of that.  Returns a dict: row*heads/s on all
    threads and on one, the threads used, the host's cores, and a description."""
    import oracle
    oracle.build()

    def timed(n_pre, n_dec, threads):
        t0 = time.perf_counter()
        used = 1
        if n_pre:
            rows = np.repeat(np.arange(n_pre, dtype=np.int32), H)
            heads = np.tile(np.arange(H, dtype=np.int32), n_pre)
            _, used = oracle.pairs(pre, rows, heads, threads)
        if n_dec:
            rows = np.repeat(np.arange(n_dec, dtype=np.int32), H)
            heads = np.tile(np.arange(H, dtype=np.int32), n_dec)
            _, used = oracle.pairs(dec, rows, heads, threads)
        return time.perf_counter() - t0, used

    dt, used = timed(1, 1, 0)
    n = max(1, min(rows_cap, int(target_s / max(dt, 1e-6))))
    n_dec = min(n, dec.R)
    dt, used = timed(n, n_dec, 0)
    all_rate = (n + n_dec) * H / dt
    # one thread: one decode and one prefill row at a time, ~target_s / 5 in all
    dt1, _ = timed(1, 1, 1)
    n1 = max(1, min(rows_cap, int(target_s / 5 / max(dt1, 1e-6) / 2)))
    dt1, _ = timed(n1, min(n1, dec.R), 1)
    one_rate = (n1 + min(n1, dec.R)) * H / dt1
    usable, online = host_cores()
    desc = ("%d prefill rows + %d decode rows x 64 heads (k=640 each), fp64 oracle, %d OpenMP threads on "
            "%d usable of %d online host cores; single thread: %d + %d rows"
            % (n, n_dec, used, usable, online, n1, min(n1, dec.R)))
    return {"value": all_rate, "threads": used, "cores": online, "cores_usable": usable,
            "single_thread_value": one_rate, "sample": desc}


# ------------------------------------------------------------------ ours
SUS_CALLS, SUS_SETS = 128, 128


def decode_sustained(dsa, d, case, dev):
    """Milliseconds per decode call when SUS_CALLS calls run back to back from
    one CUDA graph, each over its own set of q, idx and out.  Each set's
    indices are the batch's shifted by 977 s positions, so the calls gather
    different rows of the shared 256 MiB of caches: 128 sets x 5.24 MB, about
    670 MB, more than four times the L2, so no call finds its rows there."""
    import torch
    N = case.N
    sets = []
    for s in range(SUS_SETS):
        sets.append(dict(q=d["q"].clone(), idx=((d["idx"] + 977 * s) % N).contiguous(),
                         out=torch.empty((case.R, case.H, D), dtype=torch.float32, device=dev)))
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())

    def calls(st):
        for i in range(SUS_CALLS):
            b = sets[i % SUS_SETS]
            dsa.dsa_sparse_attn_decode(b["q"], d["kv"], b["idx"], d["n_sel"], d["sink"], case.scale,
                                       b["out"], st)

    with torch.cuda.stream(side):
        calls(side)                      # scratch and launch attributes exist before capture
        side.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            calls(torch.cuda.current_stream())
        for _ in range(2):
            g.replay()
        side.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        reps = 5
        e0.record(side)
        for _ in range(reps):
            g.replay()
        e1.record(side)
        side.synchronize()
    return e0.elapsed_time(e1) / (reps * SUS_CALLS)


def hold_gpu(stream, ms=4.0):
    """Keep the stream busy for about `ms` milliseconds, so that the host has
    enqueued the timed calls that follow before the GPU reaches them: the
    events then time the calls, not the host's launch latency."""
    import torch
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(ms * 2.0e6))      # cycles at about 2 GHz


def cold_call_ms(fn, flush, stream, reps):
    """Milliseconds of `reps` calls of fn() on `stream` (torch's current
    one), each after an L2-flushing write and bracketed by its own events.
    The stream is held first, so that the host has queued the calls before
    the GPU reaches them."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    hold_gpu(stream)
    for i, (e0, e1) in enumerate(ev):
        flush.fill_(float(i))
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) for e0, e1 in ev]


def topk_timing(dsa, dev, flush, mode, k=K, reps=32):
    """Mean milliseconds of one top-k selection call over the indexer-score
    rows of `mode` (prefill: 2048 causal rows of a 4096 cache; decode: 8
    rows of 32768), the L2 flushed before each call; and the bytes of
    scores it reads."""
    import torch
    scores, n_valid = I.indexer_scores(mode)
    s = torch.from_numpy(scores).to(dev)
    nv = torch.from_numpy(n_valid).to(dev)
    R = scores.shape[0]
    idx = torch.empty((R, k), dtype=torch.int32, device=dev)
    n_sel = torch.empty(R, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        dsa.dsa_topk_select(s, nv, k, idx, n_sel, stream)
    torch.cuda.synchronize()
    ms = cold_call_ms(lambda: dsa.dsa_topk_select(s, nv, k, idx, n_sel, stream), flush, stream, reps)
    assert dsa.dsa_get_device_error() == 0
    return sum(ms) / reps, R, int(n_valid.astype(np.int64).sum()) * 4


def oproj_timing(dsa, dev, flush, d_pre, pre, d_out=OPROJ_D_OUT, reps=32):
    """The prefill rows' attention with a bf16 output, then their output
    projection (out [2048, d_out] fp32 = attn [2048, 64*512] bf16 . w_o) by
    the library's GEMM, and, for comparison, the same product by cuBLAS
    (torch.matmul, bf16 out), each call alone with the L2 flushed before it.
    w_o is seeded N(0, 1/K) on the device (the pages give no projection
    weights or width).  Returns (attention ms, projection ms, cuBLAS ms)."""
    import torch
    K = H * D
    g = torch.Generator(device=dev)
    g.manual_seed(0xD5A0 + 17)
    w_o = (torch.randn((K, d_out), generator=g, device=dev) * K ** -0.5).to(torch.bfloat16)
    attn = torch.empty((PRE_R, H, D), dtype=torch.bfloat16, device=dev)
    out = torch.empty((PRE_R, d_out), dtype=torch.float32, device=dev)
    ref = torch.empty((PRE_R, d_out), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def call_attn():
        dsa.dsa_sparse_attn(d_pre["q"], d_pre["kv"], d_pre["idx"], d_pre["n_sel"], d_pre["sink"], pre.scale,
                            attn, 0, stream)

    def call_proj():
        dsa.dsa_oproj(attn, w_o, out, stream)

    def call_cublas():
        torch.matmul(attn.view(PRE_R, K), w_o, out=ref)

    res = []
    for fn in (call_attn, call_proj, call_cublas):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        res.append(sum(cold_call_ms(fn, flush, stream, reps)) / reps)
    assert dsa.dsa_get_device_error() == 0
    assert torch.isfinite(out).all().item()
    return res[0], res[1], res[2]


def decode_batch_timing(dsa, dev, flush, B=DEC_BIG_B, reps=16, N=DEC_N):
    """Mean milliseconds of one decode call over a batch that fills the GPU
    (B slots of an N-position cache, one row each, k=640), split into
    128-key chunks (dsa_sparse_attn_decode) and with whole rows
    (dsa_sparse_attn_decode_whole_rows), the L2 flushed before each call.
    Inputs are seeded N(0,1) bf16 drawn on the device (20 GB of caches at
    B = 608) and distinct random positions per slot."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(0xD5A0 + 23)
    kv = torch.empty((B, N, D), dtype=torch.bfloat16, device=dev)
    for b0 in range(0, B, 64):
        kv[b0:b0 + 64].normal_(generator=g)
    q = torch.randn((B, H, D), generator=g, device=dev).to(torch.bfloat16)
    sink = torch.randn(H, generator=g, device=dev)
    idx = torch.stack([torch.randperm(N, generator=g, device=dev)[:K] for _ in range(B)]).to(torch.int32)
    n_sel = torch.full((B,), K, dtype=torch.int32, device=dev)
    outs = [torch.empty((B, H, D), dtype=torch.float32, device=dev) for _ in range(2)]
    scale = 1.0 / math.sqrt(D)
    stream = torch.cuda.current_stream()
    calls = (lambda: dsa.dsa_sparse_attn_decode(q, kv, idx, n_sel, sink, scale, outs[0], stream),
             lambda: dsa.dsa_sparse_attn_decode_whole_rows(q, kv, idx, n_sel, sink, scale, outs[1], 1, stream))
    res = []
    for fn in calls:
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        res.append(sum(cold_call_ms(fn, flush, stream, reps)) / reps)
    assert dsa.dsa_get_device_error() == 0
    # the two are the same computation with different rounding orders
    assert torch.isfinite(outs[1]).all().item()
    assert (outs[0] - outs[1]).abs().max().item() <= 1e-3 * outs[0].abs().max().item()
    del kv
    torch.cuda.empty_cache()
    return res[0], res[1]


def decode_rows_timing(dsa, dev, flush, B=DEC_B, T=2, reps=32):
    """Mean milliseconds of one decode call with T query rows a slot (B slots
    of a 32768-position cache, k=640), the L2 flushed before each call."""
    import torch
    c = I.multi_row_decode(B=B, T=T, N=DEC_N)
    t = lambda a, bf: (torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
                       if bf else torch.from_numpy(a).to(dev))
    q, kv, idx, n_sel, sink = t(c.q, True), t(c.kv, True), t(c.idx, False), t(c.n_sel, False), t(c.sink, False)
    out = torch.empty((c.R, H, D), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        dsa.dsa_sparse_attn_decode_rows(q, kv, idx, n_sel, sink, c.scale, out, T, stream)
    torch.cuda.synchronize()
    ms = cold_call_ms(lambda: dsa.dsa_sparse_attn_decode_rows(q, kv, idx, n_sel, sink, c.scale, out, T, stream),
                      flush, stream, reps)
    assert dsa.dsa_get_device_error() == 0
    return sum(ms) / reps, c.R


def single_decode_timing(dsa, dev, flush, reps=32):
    """Median and mean milliseconds of one single-row decode call (64 heads,
    a 4096-position cache, 640 sorted keys), the L2 flushed before each: the
    latency case."""
    import torch
    c = I.single_decode()
    t = lambda a, bf: (torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
                       if bf else torch.from_numpy(a).to(dev))
    q, kv, idx, n_sel, sink = t(c.q, True), t(c.kv, True), t(c.idx, False), t(c.n_sel, False), t(c.sink, False)
    out = torch.empty((1, H, D), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        dsa.dsa_sparse_attn_decode(q, kv, idx, n_sel, sink, c.scale, out, stream)
    torch.cuda.synchronize()
    ms = cold_call_ms(lambda: dsa.dsa_sparse_attn_decode(q, kv, idx, n_sel, sink, c.scale, out, stream),
                      flush, stream, reps)
    assert dsa.dsa_get_device_error() == 0
    return statistics.median(ms), sum(ms) / reps


def bench_decode_rows(args, world, rank, local):
    """Decode with T = --rows-per-slot rows a slot alone (for profiling): one
    JSON line with its time and the KV bytes it selects, in total and as
    distinct rows of each slot (the rows of a slot share most of their picks)."""
    import torch
    from deepseek_v4_top_gb300 import dsa
    import __graft_entry__
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    __graft_entry__.build()
    dsa.load()
    T = max(1, args.rows_per_slot)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    t_ms, rows = decode_rows_timing(dsa, dev, flush, T=T, reps=max(1, args.steps))
    c = I.multi_row_decode(B=DEC_B, T=T, N=DEC_N)
    distinct = 0
    for b in range(DEC_B):
        picks = set()
        for r in range(b * T, (b + 1) * T):
            picks.update(c.idx[r][:c.n_sel[r]].tolist())
        distinct += len(picks)
    if rank == 0:
        print(json.dumps({"metric": "decode with %d rows a slot, ms per call" % T, "ms": t_ms, "rows": rows,
                          "selected_kv_bytes": int(c.n_sel.astype(np.int64).sum()) * D * 2,
                          "distinct_kv_bytes": distinct * D * 2}), flush=True)


def bench_decode_batch(args, world, rank, local):
    """A decode batch that fills the GPU alone (for profiling): --slots slots
    of --slot-positions positions, split and whole-row calls, --steps timed
    calls of each; one JSON line with both times and their HBM fractions."""
    import torch
    from deepseek_v4_top_gb300 import dsa
    import __graft_entry__
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    __graft_entry__.build()
    dsa.load()
    pk, _ = peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    B, N = args.slots, args.slot_positions
    split_ms, whole_ms = decode_batch_timing(dsa, dev, flush, B=B, reps=max(1, args.steps), N=N)
    g = B * K * D * 2
    if rank == 0:
        print(json.dumps({"metric": "decode batch, ms per call (L2 flushed before each)", "slots": B,
                          "positions_per_slot": N, "split_ms": split_ms, "whole_rows_ms": whole_ms,
                          "gathered_bytes": g, "compulsory_bytes": compulsory_bytes(B, g),
                          "whole_rows_gathered_frac_hbm": g / (whole_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                          "split_gathered_frac_hbm": g / (split_ms * 1e-3) / 1e9 / pk["hbm_gbs"]}), flush=True)


def bench_topk(args, world, rank, local):
    """The top-k selection alone (for profiling): prints one JSON line with
    the prefill-row and decode-row timings that the default run reports."""
    import torch
    from deepseek_v4_top_gb300 import dsa
    import __graft_entry__
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    __graft_entry__.build()
    dsa.load()
    pk, _ = peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    out = {}
    for mode in ("prefill", "decode"):
        t_ms, rows, nbytes = topk_timing(dsa, dev, flush, mode, reps=max(1, args.steps))
        out[mode] = {"ms": t_ms, "rows_per_s": rows / (t_ms * 1e-3),
                     "scores_frac_hbm": nbytes / (t_ms * 1e-3) / 1e9 / pk["hbm_gbs"]}
    if rank == 0:
        print(json.dumps({"metric": "top-k selection (k=%d), ms per call" % K, "workloads": out}), flush=True)


def bench_oproj(args, world, rank, local):
    """The output projection alone (for profiling): out [2048, 7168] fp32 =
    attn [2048, K] bf16 . w_o [K, 7168] bf16 (K = 32768 unless --oproj-k),
    through dsa_oproj and, for comparison, cuBLAS (torch.matmul, bf16 out),
    each call alone with the L2 flushed before it."""
    import torch
    from deepseek_v4_top_gb300 import dsa
    import __graft_entry__
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    __graft_entry__.build()
    dsa.load()
    Kp, N = args.oproj_k, OPROJ_D_OUT
    g = torch.Generator(device=dev)
    g.manual_seed(0xD5A0 + 18)
    a = torch.randn((PRE_R, Kp), generator=g, device=dev).to(torch.bfloat16)
    w = (torch.randn((Kp, N), generator=g, device=dev) * Kp ** -0.5).to(torch.bfloat16)
    out = torch.empty((PRE_R, N), dtype=torch.float32, device=dev)
    ref = torch.empty((PRE_R, N), dtype=torch.bfloat16, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    res = {}
    for name, fn in (("dsa_oproj", lambda: dsa.dsa_oproj(a, w, out, stream)),
                     ("cublas", lambda: torch.matmul(a, w, out=ref))):
        for _ in range(args.warmup):
            flush.fill_(0.5)
            fn()
        torch.cuda.synchronize()
        ms_list = cold_call_ms(fn, flush, stream, max(1, args.steps))
        ms = sum(ms_list) / len(ms_list)
        res[name] = {"ms": ms, "tflops": 2.0 * PRE_R * Kp * N / (ms * 1e-3) / 1e12}
    assert dsa.dsa_get_device_error() == 0
    if rank == 0:
        print(json.dumps({"metric": "output projection %dx%dx%d, ms per call" % (PRE_R, Kp, N),
                          "workloads": res}), flush=True)


def bench_ours(args, world, rank, local):
    import torch
    from deepseek_v4_top_gb300 import dsa
    import __graft_entry__
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    # one process a node builds (the others would write the same files), the rest wait for it
    if local == 0:
        __graft_entry__.build()
    barrier(world)
    dsa.load()
    do_dec = args.workload in ("both", "decode")
    do_pre = args.workload in ("both", "prefill")

    dec = I.batched_decode(B=DEC_B, N=DEC_N) if do_dec else None
    pre = I.prefill(rows=PRE_R, N=PRE_N) if do_pre else None

    def up(a, bf16):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if bf16 else a)
        return t.to(dev).view(torch.bfloat16) if bf16 else t.to(dev)

    def upload(c):
        return dict(q=up(c.q, True), kv=up(c.kv, True), idx=up(c.idx, False),
                    n_sel=up(c.n_sel, False), sink=up(c.sink, False))

    d_dec = upload(dec) if do_dec else None
    d_pre = upload(pre) if do_pre else None
    o_dec = torch.empty((DEC_B, H, D), dtype=torch.float32, device=dev) if do_dec else None
    o_pre = torch.empty((PRE_R, H, D), dtype=torch.float32, device=dev) if do_pre else None
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def call_dec(s=stream):
        if do_dec:
            dsa.dsa_sparse_attn_decode(d_dec["q"], d_dec["kv"], d_dec["idx"], d_dec["n_sel"],
                                       d_dec["sink"], dec.scale, o_dec, s)

    def call_pre(s=stream):
        if do_pre:
            dsa.dsa_sparse_attn_prefill(d_pre["q"], d_pre["kv"], d_pre["idx"], d_pre["n_sel"],
                                        d_pre["sink"], pre.scale, o_pre, s)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        call_dec()
        call_pre()
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_error() == 0

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    hold_gpu(stream)
    for i in range(args.steps):
        flush.fill_(float(i))            # evict L2 between steps (outside the events)
        ev[i][0].record(stream)
        call_dec()
        ev[i][1].record(stream)
        call_pre()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t_wall1 = time.time()
    dec_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)]
    pre_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps)]
    dec_avg = reduce_max(sum(dec_ms) / args.steps, world)
    pre_avg = reduce_max(sum(pre_ms) / args.steps, world)
    one_stream_ms = reduce_max(sum(dec_ms) / args.steps + sum(pre_ms) / args.steps, world)
    assert dsa.dsa_get_device_error() == 0

    # The step as a serving engine runs it: the decode batch and the prefill
    # rows are independent calls, so they go on two streams at once, and the
    # decode's CTAs take the SMs that the prefill's last rows leave idle.  The
    # per-call times above (and the roofline) come from the one-stream loop,
    # each call alone.
    side = torch.cuda.Stream(device=dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for i in range(args.warmup):
        flush.fill_(1.0)
        side.wait_stream(stream)
        call_dec(side)
        call_pre(stream)
        stream.wait_stream(side)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t_wall2 = time.time()
    hold_gpu(stream)
    for i in range(args.steps):
        flush.fill_(float(i))            # evict L2 between steps (outside the events)
        evs[i][0].record(stream)
        side.wait_event(evs[i][0])
        call_dec(side)
        ev_dec = torch.cuda.Event()
        ev_dec.record(side)
        call_pre(stream)
        stream.wait_event(ev_dec)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t_wall3 = time.time()
    step_ms = reduce_max(sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps, world)
    assert dsa.dsa_get_device_error() == 0
    dec_sus_ms = reduce_max(decode_sustained(dsa, d_dec, dec, dev), world) if do_dec else None

    # end to end through the public API: host (pinned) inputs in, result out
    pinned = []

    def pin(a):
        t = torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
        pinned.append(t)
        return t

    # Two sets of device inputs and outputs (and of host outputs), used by
    # alternate steps, so that a step's copies can overlap the step before it
    # (a serving loop double-buffers the same way); the KV caches and sinks
    # stay resident.
    e2e_io = []
    if do_dec:
        e2e_io.append((d_dec, pin(dec.q.view(np.int16)), pin(dec.idx), pin(dec.n_sel),
                       [torch.empty(o_dec.shape, dtype=torch.float32).pin_memory() for _ in range(2)],
                       [o_dec, torch.empty_like(o_dec)], False))
    if do_pre:
        e2e_io.append((d_pre, pin(pre.q.view(np.int16)), pin(pre.idx), pin(pre.n_sel),
                       [torch.empty(o_pre.shape, dtype=torch.float32).pin_memory() for _ in range(2)],
                       [o_pre, torch.empty_like(o_pre)], True))
    h2d = sum(t.numel() * t.element_size() for t in pinned)
    d2h = sum(io[4][0].numel() * 4 for io in e2e_io)
    dev_in = [[(d["q"], d["idx"], d["n_sel"]) for d, *_ in e2e_io],
              [(torch.empty_like(d["q"]), torch.empty_like(d["idx"]), torch.empty_like(d["n_sel"]))
               for d, *_ in e2e_io]]

    # The step runs as a user with host-resident tensors would run it: prefill
    # rows in E2E_CHUNKS chunks over three streams (copy in, compute, copy out),
    # so the two copy directions and the kernels overlap; the decode batch goes
    # first on the compute stream.  Rows do not depend on their batch, so the
    # chunked calls give the same bits as one call.
    s_in = torch.cuda.Stream(device=dev)
    s_comp = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)
    comp_done, out_done = {}, {}

    def e2e_step(i, start_ev):
        """Step i on buffer set i % 2; returns the event of its last copy out."""
        k = i % 2
        for st in (s_in, s_comp, s_out):
            st.wait_event(start_ev)
        # the set's inputs were last read by step i - 2's kernels, its outputs
        # last copied out by step i - 2
        if i - 2 in comp_done:
            s_in.wait_event(comp_done.pop(i - 2))
        if i - 2 in out_done:
            s_comp.wait_event(out_done.pop(i - 2))
        for j, (d, hq, hidx, hns, houts, douts, is_pre) in enumerate(e2e_io):
            q, idx, n_sel = dev_in[k][j]
            hout, dout = houts[k], douts[k]
            rows = hq.shape[0]
            chunks = E2E_CHUNKS if is_pre else 1
            bounds = [rows * c // chunks for c in range(chunks + 1)]
            for c in range(chunks):
                a, b = bounds[c], bounds[c + 1]
                with torch.cuda.stream(s_in):
                    q[a:b].view(torch.int16).copy_(hq[a:b], non_blocking=True)
                    idx[a:b].copy_(hidx[a:b], non_blocking=True)
                    n_sel[a:b].copy_(hns[a:b], non_blocking=True)
                    ev_in = torch.cuda.Event()
                    ev_in.record(s_in)
                s_comp.wait_event(ev_in)
                fn = dsa.dsa_sparse_attn_prefill if is_pre else dsa.dsa_sparse_attn_decode
                fn(q[a:b], d["kv"], idx[a:b], n_sel[a:b], d["sink"],
                   pre.scale if is_pre else dec.scale, dout[a:b], s_comp)
                ev_c = torch.cuda.Event()
                ev_c.record(s_comp)
                s_out.wait_event(ev_c)
                with torch.cuda.stream(s_out):
                    hout[a:b].copy_(dout[a:b], non_blocking=True)
        ev_comp = torch.cuda.Event()
        ev_comp.record(s_comp)
        comp_done[i] = ev_comp
        ev_done = torch.cuda.Event()
        ev_done.record(s_out)
        out_done[i] = ev_done
        return ev_done

    e2e_steps = max(3, min(args.steps, 20))
    for i in range(2):
        ev0 = torch.cuda.Event()
        ev0.record(stream)
        stream.wait_event(e2e_step(i, ev0))
    torch.cuda.synchronize()
    comp_done.clear()
    out_done.clear()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    last = None
    for i in range(e2e_steps):
        last = e2e_step(i, e0)
    # every step's copies out are done (each stream runs in order)
    stream.wait_event(last)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1) / e2e_steps, world)
    t_clock1 = time.time()
    clocks.stop()
    assert dsa.dsa_get_device_error() == 0
    for o in (o_dec, o_pre):
        if o is not None:
            assert torch.isfinite(o).all().item()

    pk, pk_note = peaks()
    units = ((DEC_B if do_dec else 0) + (PRE_R if do_pre else 0)) * H
    value = units * world / (step_ms * 1e-3)
    workloads = {}
    if do_dec:
        g = DEC_B * K * D * 2
        workloads["decode_b8"] = {
            "ms": dec_avg, "ms_median": reduce_max(statistics.median(dec_ms), world),
            "row_heads_per_s": DEC_B * H / (dec_avg * 1e-3),
            "gathered_kv_gbs": g / (dec_avg * 1e-3) / 1e9,
            "gathered_frac_hbm": g / (dec_avg * 1e-3) / 1e9 / pk["hbm_gbs"],
            "compulsory_bytes": compulsory_bytes(DEC_B, g),
            "compulsory_gbs": compulsory_bytes(DEC_B, g) / (dec_avg * 1e-3) / 1e9, "launches": 2}
        workloads["decode_b8_sustained"] = {
            "ms": dec_sus_ms, "row_heads_per_s": DEC_B * H / (dec_sus_ms * 1e-3),
            "gathered_kv_gbs": g / (dec_sus_ms * 1e-3) / 1e9,
            "gathered_frac_hbm": g / (dec_sus_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
            "how": "%d calls back to back from one CUDA graph over %d q/idx/out sets; the sets' indices "
                   "are shifted copies, so the calls gather ~670 MB of distinct rows (more than four "
                   "times the L2); no L2 flush" % (SUS_CALLS, SUS_SETS)}
    if args.workload == "both":
        # decode with two query rows a slot, timed on its own (not part of the step)
        t_ms, rows = decode_rows_timing(dsa, dev, flush)
        t_ms = reduce_max(t_ms, world)
        g = rows * K * D * 2
        workloads["decode_b8_t2"] = {
            "ms": t_ms, "row_heads_per_s": rows * H / (t_ms * 1e-3),
            "gathered_kv_gbs": g / (t_ms * 1e-3) / 1e9,
            "gathered_frac_hbm": g / (t_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
            "how": "dsa_sparse_attn_decode_rows, 8 slots x 2 rows (N=32768 per slot), one call a time, "
                   "L2 flushed before each"}
        # one decode row alone: the latency case (not part of the step)
        med, mean = single_decode_timing(dsa, dev, flush)
        med, mean = reduce_max(med, world), reduce_max(mean, world)
        g = K * D * 2
        workloads["decode_b1"] = {
            "ms": mean, "ms_median": med, "row_heads_per_s": H / (mean * 1e-3),
            "gathered_kv_gbs": g / (mean * 1e-3) / 1e9,
            "gathered_frac_hbm": g / (mean * 1e-3) / 1e9 / pk["hbm_gbs"],
            "how": "dsa_sparse_attn_decode, 1 row, 64 heads, N=4096, 640 sorted keys, one call a time, "
                   "L2 flushed before each (split kernel + combine)"}
        # a decode batch that fills the GPU, split and whole-row (not part of the step)
        split_ms, whole_ms = decode_batch_timing(dsa, dev, flush)
        for key, t_ms, how in (
                ("decode_b%d_split" % DEC_BIG_B, split_ms,
                 "dsa_sparse_attn_decode (128-key chunks on separate SMs, then the merge kernel)"),
                ("decode_b%d_whole_rows" % DEC_BIG_B, whole_ms,
                 "dsa_sparse_attn_decode_whole_rows (each row whole in one CTA, no partials)")):
            t_ms = reduce_max(t_ms, world)
            g = DEC_BIG_B * K * D * 2
            cb = compulsory_bytes(DEC_BIG_B, g)
            workloads[key] = {
                "ms": t_ms, "row_heads_per_s": DEC_BIG_B * H / (t_ms * 1e-3),
                "gathered_kv_gbs": g / (t_ms * 1e-3) / 1e9,
                "gathered_frac_hbm": g / (t_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                "compulsory_bytes": cb, "compulsory_gbs": cb / (t_ms * 1e-3) / 1e9,
                "compulsory_frac_hbm": cb / (t_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                "how": how + ", %d slots x 1 row, N=32768 per slot, k=640, one call a time, L2 flushed "
                             "before each; inputs drawn on the device" % DEC_BIG_B}
        # the indexer's top-k selection, timed on its own (not part of the step)
        for mode, key in (("prefill", "topk_prefill_2048"), ("decode", "topk_decode_b8")):
            t_ms, rows, nbytes = topk_timing(dsa, dev, flush, mode)
            t_ms = reduce_max(t_ms, world)
            workloads[key] = {
                "ms": t_ms, "rows_per_s": rows / (t_ms * 1e-3),
                "scores_gbs": nbytes / (t_ms * 1e-3) / 1e9,
                "scores_frac_hbm": nbytes / (t_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                "how": "dsa_topk_select, k=%d, N(0,1) scores, one call a time, L2 flushed before each" % K}
    if do_pre:
        # the prefill rows with a bf16 output, then their output projection
        a_ms, p_ms, c_ms = oproj_timing(dsa, dev, flush, d_pre, pre)
        a_ms, p_ms, c_ms = reduce_max(a_ms, world), reduce_max(p_ms, world), reduce_max(c_ms, world)
        g = PRE_R * K * D * 2
        workloads["prefill_2048_bf16_out"] = {
            "ms": a_ms, "row_heads_per_s": PRE_R * H / (a_ms * 1e-3),
            "gathered_frac_hbm": g / (a_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
            "how": "dsa_sparse_attn, out bf16 [2048, 64, 512] (134 MB instead of 268 MB fp32), one call a time, "
                   "L2 flushed before each"}
        p_flops = 2.0 * PRE_R * H * D * OPROJ_D_OUT
        workloads["oproj_2048x32768x%d" % OPROJ_D_OUT] = {
            "ms": p_ms, "tflops": p_flops / (p_ms * 1e-3) / 1e12,
            "frac_of_measured_matmul": p_flops / (p_ms * 1e-3) / 1e12 / pk["bf16_tflops"],
            "frac_note": "denominator: MEASURED_PEAKS.json bf16_tflops, a best-of-10 torch.matmul "
                         "8192^3 rate on this GPU (not a hardware peak; the nominal dense bf16 peak "
                         "is 2250 TFLOP/s)",
            "cublas_ms": c_ms, "cublas_tflops": p_flops / (c_ms * 1e-3) / 1e12,
            "time_vs_cublas": c_ms / p_ms,
            "how": "dsa_oproj (the library's tcgen05 GEMM, bf16 x bf16 -> fp32): the 2048 rows' bf16 attention "
                   "output times a seeded [32768, %d] bf16 projection, one call a time, L2 flushed before each; "
                   "cublas_ms: torch.matmul of the same operands (cuBLAS, bf16 out), timed the same way, for "
                   "comparison only" % OPROJ_D_OUT}
    roofline = None
    if do_pre:
        g = PRE_R * K * D * 2
        pre_flops = FLOPS_PER_ROW * PRE_R
        pre_tflops = pre_flops / (pre_avg * 1e-3) / 1e12
        workloads["prefill_2048"] = {
            "ms": pre_avg, "ms_median": reduce_max(statistics.median(pre_ms), world),
            "row_heads_per_s": PRE_R * H / (pre_avg * 1e-3),
            "gathered_kv_gbs": g / (pre_avg * 1e-3) / 1e9,
            "gathered_frac_hbm": g / (pre_avg * 1e-3) / 1e9 / pk["hbm_gbs"],
            "compulsory_bytes": compulsory_bytes(PRE_R, PRE_N * D * 2),
            "compulsory_gbs": compulsory_bytes(PRE_R, PRE_N * D * 2) / (pre_avg * 1e-3) / 1e9,
            "tflops": pre_tflops, "launches": 1}
        a = g / (pre_avg * 1e-3) / 1e9
        roofline = {
            "kernel": "dsa_tc_kernel (prefill 2048)",
            "bound": "hbm",
            "achieved": a,
            "peak": pk["hbm_gbs"],
            "unit": "GB/s",
            "frac": a / pk["hbm_gbs"],
            "peak_note": "copy bandwidth " + pk_note,
            "algorithmic_per_launch": "gathered KV: 2048 rows x 640 keys x 1024 B = %d B "
                                      "(logical bytes; the 4 MiB cache stays in L2)" % g,
            "traffic": recorded_traffic(),
            "tensor": {"achieved_tflops": pre_tflops, "peak_tflops": pk["bf16_tflops"],
                       "frac": pre_tflops / pk["bf16_tflops"],
                       "note": "4*H*d*k flops per row x 2048 rows = %.4g FLOP; bf16 burst %s"
                               % (pre_flops, pk_note)},
        }
    else:
        g = DEC_B * K * D * 2
        a = g / (dec_avg * 1e-3) / 1e9
        roofline = {"kernel": "dsa_tc_kernel + dsa_combine_kernel (decode B=8)", "bound": "hbm",
                    "achieved": a, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": a / pk["hbm_gbs"],
                    "peak_note": "copy bandwidth " + pk_note,
                    "algorithmic_per_launch": "8 rows x 640 keys x 1024 B gathered", "traffic": None}
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "row*heads/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_ms,
        "ms_per_step_one_stream": one_stream_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/kv, seeded distinct and causal top-k indices)",
        "config": {
            "workload": WORKLOAD if args.workload == "both" else args.workload + " part of: " + WORKLOAD,
            "decode": {"B": DEC_B, "N": DEC_N}, "prefill": {"rows": PRE_R, "N": PRE_N},
            "heads": H, "d": D, "k": K,
            "parallelism": "dp%d (independent replicas, no collective)" % world,
            "l2": "flushed before every step by writing 2x L2; events bracket the calls only",
            "streams": "the step's decode and prefill calls run on two streams at once (ms_per_step); "
                       "ms_per_step_one_stream and the per-call times run them one after the other "
                       "on one stream",
        },
        "workloads": workloads,
        "roofline": roofline,
        "gpu_launches": (2 * do_dec + do_pre) * args.steps,
        "e2e": {
            "value": units * world / (e2e_ms * 1e-3),
            "unit": "row*heads/s",
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "note": "q, idx, n_sel copied in from pinned host memory and out copied back every "
                    "step; prefill in %d row chunks over three streams (copy in, compute, copy "
                    "out) so that both copy directions overlap the kernels; alternate steps use two "
                    "sets of device buffers, so a step's copies also overlap the step before it; KV "
                    "caches and sinks stay resident" % E2E_CHUNKS,
        },
        "clocks": clocks.summary(t_wall0, t_clock1),
        "wall_s_timed_region": t_wall3 - t_wall2,
        "wall_s_one_stream_loop": t_wall1 - t_wall0,
    }
    # the oracle's rate on the host cores: one GPU only, so that no rank waits
    # on it (at N > 1 each rank's host would share its cores with the others)
    if world == 1 and not args.no_cpu_baseline and do_dec and do_pre:
        cb = oracle_sample(pre, dec, args.cpu_seconds)
        # cores: the threads the timed oracle ran on; the host's own core
        # counts beside it
        line["cpu_baseline"] = {"value": cb["value"], "unit": "row*heads/s", "cores": cb["threads"],
                                "host_cores_online": cb["cores"], "host_cores_usable": cb["cores_usable"],
                                "single_thread_value": cb["single_thread_value"],
                                "kind": "oracle", "sample": cb["sample"]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------ head-sharded (TP)
def bench_tp(args, world, rank, local):
    """The benchmark step with the 64 heads split over the ranks (TensorFold
    PR #1206: 16 heads a rank at world 4): each rank runs the decode and
    prefill calls over its heads, NCCL all-gathers the outputs and the
    library lays them out as [rows, 64, 512].  Total work is fixed, so the
    scaling is strong.  q is cut into the ranks' heads once, before timing
    (a model's sharded q projection would produce it so)."""
    import torch
    from deepseek_v4_top_gb300 import dsa
    import __graft_entry__
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    # one process a node builds (the others would write the same files), the rest wait for it
    if local == 0:
        __graft_entry__.build()
    barrier(world)
    dsa.load()
    plan = dsa.dsa_head_shard(H, world, rank)
    hpr = plan.heads_per_rank
    work = []
    for case, T in ((I.batched_decode(B=DEC_B, N=DEC_N), 1), (I.prefill(rows=PRE_R, N=PRE_N), 0)):
        up = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
        d = dict(q=up(case.q), kv=up(case.kv), idx=torch.from_numpy(case.idx).to(dev),
                 n_sel=torch.from_numpy(case.n_sel).to(dev), sink=torch.from_numpy(case.sink).to(dev))
        ql = torch.empty((case.R, hpr, D), dtype=torch.bfloat16, device=dev)
        sl = torch.empty((hpr,), dtype=torch.float32, device=dev)
        dsa.dsa_shard_heads(d["q"], d["sink"], ql, sl, world, rank)
        work.append(dict(case=case, T=T, d=d, ql=ql, sl=sl,
                         ol=torch.empty((case.R, hpr, D), dtype=torch.float32, device=dev),
                         g=torch.empty((world, case.R, hpr, D), dtype=torch.float32, device=dev),
                         out=torch.empty((case.R, H, D), dtype=torch.float32, device=dev)))
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        for w in work:
            dsa.tp_sparse_attn(w["ql"], w["d"]["kv"], w["d"]["idx"], w["d"]["n_sel"], w["sl"], w["case"].scale,
                               w["ol"], w["g"], w["out"], rows_per_slot=w["T"])

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    assert dsa.dsa_get_device_error() == 0
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    hold_gpu(stream)
    for i in range(args.steps):
        flush.fill_(float(i))
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    clocks.stop()
    step_ms = reduce_max(sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps, world)
    assert dsa.dsa_get_device_error() == 0
    for w in work:
        assert torch.isfinite(w["out"]).all().item()
    units = (DEC_B + PRE_R) * H
    line = {
        "metric": METRIC, "value": units / (step_ms * 1e-3), "unit": "row*heads/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/kv, seeded distinct and causal top-k indices)",
        "config": {"workload": WORKLOAD, "decode": {"B": DEC_B, "N": DEC_N}, "prefill": {"rows": PRE_R, "N": PRE_N},
                   "heads": H, "heads_per_rank": hpr, "d": D, "k": K,
                   "parallelism": "tp%d (heads split over ranks; NCCL all-gather of the outputs)" % world,
                   "l2": "flushed before every step by writing 2x L2; events bracket the calls only"},
        "gpu_launches": 5 * args.steps,      # decode: split + combine + unshard; prefill: attention + unshard
        "clocks": clocks.summary(t0, t1),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------- reference
def bench_reference(args, world, rank):
    """The fp64 CPU oracle, as it stands, on the host cores (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    dec = I.batched_decode(B=DEC_B, N=DEC_N)
    pre = I.prefill(rows=PRE_R, N=PRE_N)
    # each step: one decode row and one prefill row, all 64 heads
    rows = np.repeat(np.arange(1, dtype=np.int32), H)
    heads = np.arange(H, dtype=np.int32)
    threads = 1

    def step(i):
        nonlocal threads
        rp = np.full(H, i % PRE_R, np.int32)
        rd = np.full(H, i % DEC_B, np.int32)
        _, threads = oracle.pairs(pre, rp, heads)
        _, threads = oracle.pairs(dec, rd, heads)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = (time.perf_counter() - t0) / args.steps
    units = 2 * H
    v = units / dt
    desc = ("per step: 1 prefill row + 1 decode row x 64 heads (k=640), fp64 oracle, %d threads"
            % threads)
    del rows
    line = {
        "impl": "reference",
        "metric": METRIC, "value": v, "unit": "row*heads/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same generator and seeds as the GPU arm)",
        "config": {"workload": WORKLOAD, "heads": H, "d": D, "k": K,
                   "parallelism": "host cores of rank 0"},
        "cpu_baseline": {"value": v, "unit": "row*heads/s", "cores": threads,
                         "host_cores_online": host_cores()[1], "host_cores_usable": host_cores()[0],
                         "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": v, "unit": "row*heads/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="approximate CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=("both", "prefill", "decode", "topk", "decode_rows", "oproj",
                                           "decode_batch"),
                    default="both",
                    help="both (the benchmark step), one half of it for profiling, the top-k "
                         "selection alone, decode with --rows-per-slot rows a slot alone, or a decode "
                         "batch of --slots slots alone (split and whole-row calls)")
    ap.add_argument("--slots", type=int, default=DEC_BIG_B, help="slots of the decode_batch workload")
    ap.add_argument("--slot-positions", type=int, default=DEC_N,
                    help="positions a slot of the decode_batch workload (a smaller cache for profiling)")
    ap.add_argument("--rows-per-slot", type=int, default=2,
                    help="rows a slot of the decode_rows workload")
    ap.add_argument("--oproj-k", type=int, default=H * D,
                    help="inner size of the oproj workload (a smaller one for profiling)")
    ap.add_argument("--tp", action="store_true",
                    help="split the 64 heads over the ranks (head-sharded tensor parallelism) instead of "
                         "running independent replicas")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_env()
    if args.impl == "reference":
        bench_reference(args, world, rank)
    elif args.workload == "topk":
        bench_topk(args, world, rank, local)
    elif args.workload == "decode_rows":
        bench_decode_rows(args, world, rank, local)
    elif args.workload == "decode_batch":
        bench_decode_batch(args, world, rank, local)
    elif args.workload == "oproj":
        bench_oproj(args, world, rank, local)
    elif args.tp:
        bench_tp(args, world, rank, local)
    else:
        bench_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
