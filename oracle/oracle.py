"""ctypes loader for the C oracle (test infrastructure only).

``build()`` compiles ``dsa_oracle.c`` with gcc (OpenMP when available) into
``liboracle.so`` beside it.  The wrappers take numpy arrays as produced by
``deepseek_v4_top_gb300.inputs`` and return float64 outputs.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dsa_oracle.c")
LIB_PATH = os.path.join(HERE, "liboracle.so")

_lib = None
_lock = threading.Lock()

_DT = {"f32": 0, "bf16": 1}


def build(force: bool = False) -> str:
    """Compile the oracle.  Plain -O2, IEEE semantics (no fast-math)."""
    if (not force and os.path.exists(LIB_PATH)
            and os.path.getmtime(LIB_PATH) >= os.path.getmtime(SRC)):
        return LIB_PATH
    tmp = LIB_PATH + ".tmp%d" % os.getpid()
    base = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math", SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def load():
    """The oracle library.  DSA_ORACLE_LIB, when set, names another build of
    dsa_oracle.c to load instead (the planted-mistake copies of
    tests/test_oracle_mutants.py, which must fail the pins)."""
    global _lib
    with _lock:
        if _lib is None:
            path = os.environ.get("DSA_ORACLE_LIB") or LIB_PATH
            if path == LIB_PATH:
                build()
            lib = ctypes.CDLL(path)
            P = ctypes.c_void_p
            I = ctypes.c_int
            F = ctypes.c_float
            common = [P, P, P, P, P, F, I, I, I, I, I, I]
            lib.dsa_oracle_rowhead.argtypes = common + [I, I, P]
            lib.dsa_oracle_attn.argtypes = common + [P, I, P]
            lib.dsa_oracle_pairs.argtypes = common + [P, P, I, P, I, P]
            for f in (lib.dsa_oracle_rowhead, lib.dsa_oracle_attn, lib.dsa_oracle_pairs):
                f.restype = I
            lib.dsa_oracle_max_threads.restype = I
            lib.dsa_oracle_topk.argtypes = [P, I, P, I, I, I, P, P, P]
            lib.dsa_oracle_topk.restype = I
            lib.dsa_oracle_oproj.argtypes = [P, P, P, I, I, I, P, P, I]
            lib.dsa_oracle_oproj.restype = I
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _common(case):
    q = np.ascontiguousarray(case.q)
    kv = np.ascontiguousarray(case.kv)
    idx = np.ascontiguousarray(case.idx, dtype=np.int32)
    n_sel = np.ascontiguousarray(case.n_sel, dtype=np.int32)
    sink = np.ascontiguousarray(case.sink, dtype=np.float32)
    keep = (q, kv, idx, n_sel, sink)
    args = [_ptr(q), _ptr(kv), _ptr(idx), _ptr(n_sel), _ptr(sink), ctypes.c_float(case.scale),
            _DT[case.dtype], case.rows_per_slot if case.mode == "decode" else 0, case.R, case.H, case.N,
            case.k_max]
    return keep, args


def attn(case, threads: int = 0):
    """All outputs, float64 [R, H, 512].  Returns (out, threads_used)."""
    lib = load()
    keep, args = _common(case)
    out = np.empty((case.R, case.H, 512), np.float64)
    used = ctypes.c_int(0)
    rc = lib.dsa_oracle_attn(*args, _ptr(out), threads, ctypes.byref(used))
    if rc:
        raise ValueError("oracle rejected its arguments")
    del keep
    return out, used.value


def pairs(case, rows, heads, threads: int = 0):
    """Selected (row, head) outputs, float64 [n, 512].  Returns (out, threads_used)."""
    lib = load()
    keep, args = _common(case)
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    heads = np.ascontiguousarray(heads, dtype=np.int32)
    out = np.empty((len(rows), 512), np.float64)
    used = ctypes.c_int(0)
    rc = lib.dsa_oracle_pairs(*args, _ptr(rows), _ptr(heads), len(rows), _ptr(out), threads,
                              ctypes.byref(used))
    if rc:
        raise ValueError("oracle rejected its arguments")
    del keep
    return out, used.value


def rowhead(case, r: int, h: int):
    lib = load()
    keep, args = _common(case)
    out = np.empty(512, np.float64)
    rc = lib.dsa_oracle_rowhead(*args, r, h, _ptr(out))
    if rc:
        raise ValueError("oracle rejected its arguments")
    del keep
    return out


def max_threads() -> int:
    return int(load().dsa_oracle_max_threads())


def topk(scores, n_valid, k: int, k_max: int = None):
    """Top-k selection of each row of ``scores`` [R, ld] (see dsa_oracle.h).

    Returns (idx int32 [R, k_max], n_sel int32 [R], bad int32 [R])."""
    lib = load()
    scores = np.ascontiguousarray(scores, dtype=np.float32)
    if scores.ndim != 2:
        raise ValueError("scores must be [rows, ld]")
    R, ld = scores.shape
    k_max = k if k_max is None else k_max
    n_valid = np.ascontiguousarray(n_valid, dtype=np.int32)
    idx = np.empty((R, k_max), np.int32)
    n_sel = np.empty(R, np.int32)
    bad = np.empty(R, np.int32)
    rc = lib.dsa_oracle_topk(_ptr(scores), ld, _ptr(n_valid), R, k, k_max, _ptr(idx), _ptr(n_sel), _ptr(bad))
    if rc:
        raise ValueError("oracle rejected its arguments")
    return idx, n_sel, bad


def oproj(a, w_bf16, threads: int = 0):
    """Output projection out = a . w (see dsa_oracle.h): ``a`` [R, K] as float64
    (e.g. attention outputs reshaped to [R, H*512]) or as bf16 bit patterns
    (uint16); ``w_bf16`` [K, d_out] bf16 bit patterns.  Returns (out float64
    [R, d_out], abs float64 [R, d_out] = sum_k |a||w|)."""
    lib = load()
    w = np.ascontiguousarray(w_bf16, dtype=np.uint16)
    if w.ndim != 2:
        raise ValueError("w must be [K, d_out]")
    K, d_out = w.shape
    a = np.ascontiguousarray(a)
    R = a.shape[0]
    if a.size != R * K:
        raise ValueError("a must be [rows, K]")
    out = np.empty((R, d_out), np.float64)
    absv = np.empty((R, d_out), np.float64)
    if a.dtype == np.float64:
        rc = lib.dsa_oracle_oproj(_ptr(a), None, _ptr(w), R, K, d_out, _ptr(out), _ptr(absv), threads)
    elif a.dtype == np.uint16:
        rc = lib.dsa_oracle_oproj(None, _ptr(a), _ptr(w), R, K, d_out, _ptr(out), _ptr(absv), threads)
    else:
        raise TypeError("a must be float64 or bf16 bit patterns (uint16)")
    if rc:
        raise ValueError("oracle rejected its arguments")
    return out, absv
