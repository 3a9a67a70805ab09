"""CPU oracle for exact attention forward — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference
arm may import this package. The CUDA library and its Python binding never do; they share
no code with it. The arithmetic lives in ``attn_oracle.c`` (plain C, double precision); this
file compiles it with gcc on first use (same flags on x86-64 and aarch64, no FMA
contraction, so both machines produce the same bits) and wraps it with ctypes.

Functions:

* ``attn_fwd(q, k, v, causal, rows=None, threads=None)`` — exact attention rows in float64.
  ``q, k, v`` are float32 numpy arrays ``[B, H, N, d]`` holding the exact device values.
  ``rows`` is an optional array of flat row ids ``bh * N + i``; the result is ``[len(rows), d]``
  (or ``[B, H, N, d]`` when ``rows`` is None).
* ``attn_fwd_lse(q, k, v, causal, rows=None, threads=None)`` — the same rows and, per row, the
  base-2 log-sum-exp of its scores, ``log2(sum_j exp(s_j))`` (the running maximum plus the base-2 log of the running total,
  section "Backwards, and training with it"); returns ``(o, lse)``.
* ``attn_weights(q, k, causal, i)`` — the normalised softmax weights of one row of one head.
* ``attn_fwd_kv(q, k, v, causal)`` — ``(o, lse)`` for Nq queries (``q`` ``[B, H, Nq, d]``) against
  Nk >= Nq keys (``k, v`` ``[B, H, Nk, d]``), the queries being the last Nq positions: when causal,
  query i sees keys ``0 .. Nk - Nq + i`` (the key-value cache case).
* ``attn_bwd(q, k, v, dout, causal, threads=None)`` — ``(dq, dk, dv)`` in float64, the
  gradients of exact attention for the output gradient ``dout`` (``attn_bwd_oracle.c``,
  following the steps of the page's section "Backwards, and training with it").

Definitions follow the "Flash attention in PyTorch, then in Triton" page ("Attention's table
of scores", "Attention by hand") and attention.cu's CPU reference ("CPU reference in double").
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BWD_SRC = os.path.join(_HERE, "attn_bwd_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle library with gcc if it is missing or older than its source."""
    os.makedirs(_BUILD, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_BWD_SRC))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, _BWD_SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, dp, fp = ctypes.c_int64, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_float)
            lib.oracle_attn_fwd.argtypes = [fp, fp, fp, i64, i64, i64, i64, ctypes.c_int,
                                            ctypes.POINTER(ctypes.c_int64), i64, dp, ctypes.c_int]
            lib.oracle_attn_fwd.restype = ctypes.c_int
            lib.oracle_attn_fwd_lse.argtypes = [fp, fp, fp, i64, i64, i64, i64, ctypes.c_int,
                                                ctypes.POINTER(ctypes.c_int64), i64, dp, dp, ctypes.c_int]
            lib.oracle_attn_fwd_lse.restype = ctypes.c_int
            lib.oracle_attn_weights.argtypes = [fp, fp, i64, i64, ctypes.c_int, i64, dp]
            lib.oracle_attn_weights.restype = ctypes.c_int
            lib.oracle_attn_bwd.argtypes = [fp, fp, fp, fp, i64, i64, i64, i64, ctypes.c_int, dp, dp, dp,
                                            ctypes.c_int]
            lib.oracle_attn_bwd.restype = ctypes.c_int
            lib.oracle_attn_fwd_kv.argtypes = [fp, fp, fp, i64, i64, i64, i64, i64, ctypes.c_int, dp, dp]
            lib.oracle_attn_fwd_kv.restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _f32(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a


def _run(q, k, v, causal, rows, threads, want_lse):
    lib = _load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    if q.ndim != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    B, H, N, d = q.shape
    threads = threads or default_threads()
    fp = ctypes.POINTER(ctypes.c_float)
    dp = ctypes.POINTER(ctypes.c_double)
    if rows is None:
        out = np.empty((B, H, N, d), dtype=np.float64)
        lse = np.empty((B, H, N), dtype=np.float64) if want_lse else None
        rp, nrows = None, B * H * N
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        out = np.empty((rows.shape[0], d), dtype=np.float64)
        lse = np.empty(rows.shape[0], dtype=np.float64) if want_lse else None
        rp, nrows = rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), rows.shape[0]
    st = lib.oracle_attn_fwd_lse(q.ctypes.data_as(fp), k.ctypes.data_as(fp), v.ctypes.data_as(fp),
                                 B, H, N, d, int(bool(causal)), rp, nrows, out.ctypes.data_as(dp),
                                 lse.ctypes.data_as(dp) if want_lse else None, int(threads))
    if st != 0:
        raise RuntimeError(f"oracle_attn_fwd failed with status {st}")
    return out, lse


def attn_fwd(q, k, v, causal: bool, rows=None, threads: int | None = None) -> np.ndarray:
    return _run(q, k, v, causal, rows, threads, False)[0]


def attn_fwd_lse(q, k, v, causal: bool, rows=None, threads: int | None = None):
    """Rows of the output and their base-2 log-sum-exps ``log2(sum_j exp(s_j))``."""
    return _run(q, k, v, causal, rows, threads, True)


def attn_weights(q, k, causal: bool, i: int) -> np.ndarray:
    """Softmax weights of query row ``i`` for one head (``q, k`` float32 ``[N, d]``)."""
    lib = _load()
    q, k = _f32(q), _f32(k)
    N, d = q.shape
    w = np.empty(N, dtype=np.float64)
    fp = ctypes.POINTER(ctypes.c_float)
    st = lib.oracle_attn_weights(q.ctypes.data_as(fp), k.ctypes.data_as(fp), N, d, int(bool(causal)),
                                 int(i), w.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    if st != 0:
        raise RuntimeError(f"oracle_attn_weights failed with status {st}")
    return w


def attn_bwd(q, k, v, dout, causal: bool, threads: int | None = None):
    """``(dq, dk, dv)`` float64 ``[B, H, N, d]``: gradients of exact attention for ``dout``."""
    lib = _load()
    q, k, v, dout = _f32(q), _f32(k), _f32(v), _f32(dout)
    if q.ndim != 4 or any(t.shape != q.shape for t in (k, v, dout)):
        raise ValueError("q, k, v, dout must share one [B, H, N, d] shape")
    B, H, N, d = q.shape
    outs = [np.empty((B, H, N, d), dtype=np.float64) for _ in range(3)]
    fp = ctypes.POINTER(ctypes.c_float)
    dp = ctypes.POINTER(ctypes.c_double)
    st = lib.oracle_attn_bwd(q.ctypes.data_as(fp), k.ctypes.data_as(fp), v.ctypes.data_as(fp),
                             dout.ctypes.data_as(fp), B, H, N, d, int(bool(causal)),
                             *(x.ctypes.data_as(dp) for x in outs), int(threads or default_threads()))
    if st != 0:
        raise RuntimeError(f"oracle_attn_bwd failed with status {st}")
    return tuple(outs)


def attn_fwd_kv(q, k, v, causal: bool):
    """``(o, lse)`` float64: Nq queries against Nk >= Nq keys, the queries being the last Nq
    positions (causal: query i sees keys ``0 .. Nk - Nq + i``); lse in base 2."""
    lib = _load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    if q.ndim != 4 or k.shape != v.shape or k.ndim != 4 or q.shape[:2] != k.shape[:2] or q.shape[3] != k.shape[3]:
        raise ValueError("q [B, H, Nq, d] and k, v [B, H, Nk, d]")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    o = np.empty((B, H, Nq, d), dtype=np.float64)
    lse = np.empty((B, H, Nq), dtype=np.float64)
    fp = ctypes.POINTER(ctypes.c_float)
    dp = ctypes.POINTER(ctypes.c_double)
    st = lib.oracle_attn_fwd_kv(q.ctypes.data_as(fp), k.ctypes.data_as(fp), v.ctypes.data_as(fp), B, H, Nq, Nk, d,
                                int(bool(causal)), o.ctypes.data_as(dp), lse.ctypes.data_as(dp))
    if st != 0:
        raise RuntimeError(f"oracle_attn_fwd_kv failed with status {st}")
    return o, lse
