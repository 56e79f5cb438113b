"""fp64 CPU oracle for the attention forward pass -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never loads it and the
two share no code: the arithmetic lives in ``attn_oracle.c`` (plain C, double
precision, POSIX threads), this module only marshals arrays through ctypes.

What the oracle computes is the plain definition the tiled kernels replace:
the standard attention of the PyTorch decoder layer in section 3 of "OpenAI
Triton: from introduction to model practice" (scores = Q K^T * scale, causal
mask, row softmax, times V), plus the natural-log row log-sum-exp of the
scaled scores that section 5 of that page (Figure 5, Source 2) stores next to
O.  Masked keys are excluded from the softmax (weight exactly zero).

Parity is pinned by the CPU tests in ``tests/test_oracle_pins.py`` (brute force
at extended precision, a library softmax, the online tile-by-tile recurrence,
closed forms and invariances); every function here is pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "rowops_oracle.c"), os.path.join(_HERE, "attn_bwd_oracle.c")]
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into oracle/_build/liboracle.so with gcc."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and all(os.path.getmtime(_LIB_PATH) >= os.path.getmtime(f) for f in _SRCS)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-fPIC", "-shared",
           "-pthread", "-o", tmp, *_SRCS, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _open(path: str):
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    if hasattr(lib, "oracle_attn_fwd_kv"):
        i64 = ctypes.c_int64
        lib.oracle_attn_fwd_kv.restype = ctypes.c_int
        lib.oracle_attn_fwd_kv.argtypes = [dp] * 5 + [i64] * 5 + [
            ctypes.c_double, ctypes.c_int, ctypes.POINTER(i64), i64, ctypes.c_int]
    if hasattr(lib, "oracle_attn_bwd"):
        i64 = ctypes.c_int64
        lib.oracle_attn_bwd.restype = ctypes.c_int
        lib.oracle_attn_bwd.argtypes = [dp] * 7 + [i64] * 4 + [ctypes.c_double, ctypes.c_int,
                                                                ctypes.c_int]
        lib.oracle_attn_bwd_dkv_rows.restype = ctypes.c_int
        lib.oracle_attn_bwd_dkv_rows.argtypes = [dp] * 6 + [i64] * 4 + [
            ctypes.c_double, ctypes.c_int, ctypes.POINTER(i64), i64, ctypes.c_int]
        lib.oracle_attn_bwd_dq_rows.restype = ctypes.c_int
        lib.oracle_attn_bwd_dq_rows.argtypes = [dp] * 5 + [i64] * 4 + [
            ctypes.c_double, ctypes.c_int, ctypes.POINTER(i64), i64, ctypes.c_int]
    if hasattr(lib, "oracle_softmax_rows"):
        for name in ("oracle_softmax_rows", "oracle_row_sum"):
            f = getattr(lib, name)
            f.restype = ctypes.c_int
            f.argtypes = [dp, dp, ctypes.c_int64, ctypes.c_int64]
    lib.oracle_attn_fwd.restype = ctypes.c_int
    lib.oracle_attn_fwd.argtypes = [
        dp, dp, dp, dp, dp, dp,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_double, ctypes.c_int,
        ctypes.POINTER(ctypes.c_int64), ctypes.c_int64, ctypes.c_int]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _open(build())
    return _lib


def _as_f64(x) -> np.ndarray:
    """Exact upcast to a contiguous float64 numpy array (bf16/fp32 -> fp64)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().to("cpu", torch.float64).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
               else (os.cpu_count() or 1))


def attn_fwd(q, k, v, scale: float, causal: bool, rows=None, threads: int | None = None,
             with_probs: bool = False):
    """Exact fp64 attention forward for the selected query rows.

    q, k, v : [B, H, N, d] (torch tensor of any float dtype, or array-like)
    scale   : multiplies Q K^T before masking and softmax (double; pass the
              fp32 value the kernel sees, e.g. float(np.float32(s)))
    causal  : keep keys j <= i only (lower triangle including the diagonal)
    rows    : None for all B*H*N rows in order, else global row ids
              (b*H + h)*N + i
    Returns (o [R, d] float64, lse [R] float64) and, with ``with_probs``, the
    softmax rows p [R, N] as a third element.
    """
    return _run(_load(), q, k, v, scale, causal, rows, threads, with_probs)


def bind(lib_path: str):
    """An ``attn_fwd`` bound to another build of the same C source (the tests
    use it to show that a deliberately broken copy fails the pins)."""
    lib = _open(lib_path)

    def fn(q, k, v, scale, causal, rows=None, threads=None, with_probs=False):
        return _run(lib, q, k, v, scale, causal, rows, threads, with_probs)
    return fn


def _run(lib, q, k, v, scale, causal, rows, threads, with_probs):
    """Marshal arrays into one oracle_attn_fwd call of ``lib``."""
    qd, kd, vd = _as_f64(q), _as_f64(k), _as_f64(v)
    if qd.ndim != 4 or qd.shape != kd.shape or qd.shape != vd.shape:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    B, H, N, d = qd.shape
    if rows is None:
        rows_arr = None
        n_rows = B * H * N
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        n_rows = rows_arr.size
    o = np.zeros((n_rows, d), dtype=np.float64)
    lse = np.zeros((n_rows,), dtype=np.float64)
    probs = np.zeros((n_rows, N), dtype=np.float64) if with_probs else None
    nthreads = int(threads) if threads else default_threads()
    rc = lib.oracle_attn_fwd(
        _ptr(qd), _ptr(kd), _ptr(vd), _ptr(o), _ptr(lse),
        _ptr(probs) if probs is not None else None,
        B, H, N, d, float(scale), 1 if causal else 0,
        rows_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)) if rows_arr is not None else None,
        n_rows, nthreads)
    if rc != 0:
        raise RuntimeError("oracle_attn_fwd failed with code %d" % rc)
    if with_probs:
        return o, lse, probs
    return o, lse


def softmax_rows(x):
    """Exact fp64 softmax over the last axis of a 2-D array (rows).

    Definition of the Triton softmax example in "CS336 lecture 6: kernels and
    Triton": y = exp(x - rowmax) / sum exp(x - rowmax)."""
    xd = _as_f64(x)
    if xd.ndim != 2:
        raise ValueError("x must be [M, N]")
    M, N = xd.shape
    y = np.zeros_like(xd)
    rc = _load().oracle_softmax_rows(_ptr(xd), _ptr(y), M, N)
    if rc != 0:
        raise RuntimeError("oracle_softmax_rows failed")
    return y


def row_sum(x):
    """Exact-as-fp64 sum of every row of a 2-D array (the row-sum example of
    "CS336 lecture 6: kernels and Triton")."""
    xd = _as_f64(x)
    if xd.ndim != 2:
        raise ValueError("x must be [M, N]")
    M, N = xd.shape
    out = np.zeros(M, dtype=np.float64)
    rc = _load().oracle_row_sum(_ptr(xd), _ptr(out), M, N)
    if rc != 0:
        raise RuntimeError("oracle_row_sum failed")
    return out


def attn_bwd(q, k, v, dout, scale: float, causal: bool, threads: int | None = None):
    """Exact fp64 gradients (dq, dk, dv), each [B, H, N, d], of the attention
    forward O = softmax(scale Q K^T [causal]) V for the upstream gradient dout."""
    qd, kd, vd, dd = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    if qd.ndim != 4 or not (qd.shape == kd.shape == vd.shape == dd.shape):
        raise ValueError("q, k, v, dout must share one [B, H, N, d] shape")
    B, H, N, d = qd.shape
    dq, dk, dv = (np.zeros_like(qd) for _ in range(3))
    rc = _load().oracle_attn_bwd(_ptr(qd), _ptr(kd), _ptr(vd), _ptr(dd), _ptr(dq), _ptr(dk),
                                 _ptr(dv), B, H, N, d, float(scale), 1 if causal else 0,
                                 int(threads) if threads else default_threads())
    if rc != 0:
        raise RuntimeError("oracle_attn_bwd failed with code %d" % rc)
    return dq, dk, dv


def attn_bwd_dq_rows(q, k, v, dout, scale: float, causal: bool, rows, threads: int | None = None):
    """Exact fp64 dq for the given global rows (b*H + h)*N + i: [R, d]."""
    qd, kd, vd, dd = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    B, H, N, d = qd.shape
    rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
    out = np.zeros((rows_arr.size, d))
    rc = _load().oracle_attn_bwd_dq_rows(
        _ptr(qd), _ptr(kd), _ptr(vd), _ptr(dd), _ptr(out), B, H, N, d, float(scale),
        1 if causal else 0, rows_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        rows_arr.size, int(threads) if threads else default_threads())
    if rc != 0:
        raise RuntimeError("oracle_attn_bwd_dq_rows failed with code %d" % rc)
    return out


def attn_bwd_dkv_rows(q, k, v, dout, scale: float, causal: bool, rows,
                      threads: int | None = None):
    """Exact fp64 dk and dv for the given global KEY rows (b*H + h)*N + j:
    ([R, d], [R, d]).  Each head holding a selected key costs one pass over
    all of its query rows."""
    qd, kd, vd, dd = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    B, H, N, d = qd.shape
    rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
    dk = np.zeros((rows_arr.size, d))
    dv = np.zeros((rows_arr.size, d))
    rc = _load().oracle_attn_bwd_dkv_rows(
        _ptr(qd), _ptr(kd), _ptr(vd), _ptr(dd), _ptr(dk), _ptr(dv), B, H, N, d, float(scale),
        1 if causal else 0, rows_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        rows_arr.size, int(threads) if threads else default_threads())
    if rc != 0:
        raise RuntimeError("oracle_attn_bwd_dkv_rows failed with code %d" % rc)
    return dk, dv


def attn_fwd_kv(q, k, v, scale: float, causal: bool, rows=None, threads: int | None = None):
    """Exact fp64 forward for queries [B, H, Nq, d] against keys and values
    [B, H, Nk, d].  The queries are the last Nq positions of the key sequence:
    under the causal mask query i sees keys j <= i + (Nk - Nq) (Nq <= Nk).
    rows: None for all B*H*Nq rows, else global ids (b*H + h)*Nq + i.
    Returns (o [R, d], lse [R])."""
    qd, kd, vd = _as_f64(q), _as_f64(k), _as_f64(v)
    if qd.ndim != 4 or kd.shape != vd.shape or qd.shape[:2] != kd.shape[:2] \
            or qd.shape[3] != kd.shape[3]:
        raise ValueError("q [B,H,Nq,d] and k, v [B,H,Nk,d] do not match")
    B, H, Nq, d = qd.shape
    Nk = kd.shape[2]
    if rows is None:
        rows_arr, n_rows = None, B * H * Nq
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        n_rows = rows_arr.size
    o = np.zeros((n_rows, d))
    lse = np.zeros(n_rows)
    rc = _load().oracle_attn_fwd_kv(
        _ptr(qd), _ptr(kd), _ptr(vd), _ptr(o), _ptr(lse), B, H, Nq, Nk, d, float(scale),
        1 if causal else 0,
        rows_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)) if rows_arr is not None else None,
        n_rows, int(threads) if threads else default_threads())
    if rc != 0:
        raise RuntimeError("oracle_attn_fwd_kv failed with code %d" % rc)
    return o, lse
