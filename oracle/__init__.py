"""fp64 CPU attention oracle -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it, and it shares no code
with that path.

``attn_oracle.c`` holds the arithmetic (the plain definition of attention and
its analytic gradient, in double precision, one head at a time); this module
only compiles it with the host C compiler, marshals numpy arrays and picks the
thread count.  ``tiled.py`` holds a test-only fp64 model of the tiled
algorithm and its memory-traffic counters; ``fp8.py`` the FP8 forward's
quantization (numpy) on top of the fp64 attention here.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into oracle/_build/liboracle.so (plain -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int64)
            i64, cint, cdbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
            lib.oracle_fwd.argtypes = [dp, dp, dp, i64, i64, i64, cint, cdbl, ip, i64, dp, dp, cint]
            lib.oracle_fwd.restype = cint
            lib.oracle_bwd.argtypes = [dp, dp, dp, dp, i64, i64, i64, cint, cdbl, ip, i64, ip, i64,
                                       dp, dp, dp, dp, dp, dp, cint]
            lib.oracle_bwd.restype = cint
            u8p = ctypes.POINTER(ctypes.c_uint8)
            lib.oracle_fwd_masked.argtypes = [dp, dp, dp, i64, i64, i64, i64, i64, u8p, i64, cdbl, ip, i64,
                                              dp, dp, cint]
            lib.oracle_fwd_masked.restype = cint
            lib.oracle_bwd_masked.argtypes = [dp, dp, dp, dp, i64, i64, i64, i64, i64, u8p, i64, cdbl, ip, i64,
                                              ip, i64, dp, dp, dp, dp, dp, dp, cint]
            lib.oracle_bwd_masked.restype = cint
            _lib = lib
    return _lib


def default_threads() -> int:
    return os.cpu_count() or 1


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray, kind=ctypes.c_double):
    return a.ctypes.data_as(ctypes.POINTER(kind))


def _idx(ix, n) -> np.ndarray:
    if ix is None:
        return np.arange(n, dtype=np.int64)
    return np.ascontiguousarray(np.asarray(ix, dtype=np.int64).reshape(-1))


def _mask_args(causal, window, block_mask, block_size, Tq, Tk):
    """(left, right, block pointer, block size, keep-alive array) of the C mask: the window
    (left, right) around the diagonal key r + Tk - Tq replaces `causal` when given (-1 =
    unbounded side); block_mask [ceil(Tq/bs)][ceil(Tk/bs)], nonzero = allowed."""
    if window is None:
        left, right = -1, (0 if causal else -1)
    else:
        assert not causal, "give either causal or a window"
        left, right = int(window[0]), int(window[1])
    if block_mask is None:
        return left, right, ctypes.POINTER(ctypes.c_uint8)(), 1, None
    bm = np.ascontiguousarray(np.asarray(block_mask) != 0, dtype=np.uint8)
    assert bm.shape == (-(-Tq // block_size), -(-Tk // block_size)), bm.shape
    return left, right, bm.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), block_size, bm


def attention_fwd(q, k, v, causal: bool, scale: float, rows=None, nthreads: int | None = None,
                  window=None, block_mask=None, block_size: int = 128):
    """O [len(rows), d] and lse [len(rows)] for one head (q [Tq,d], k/v [Tk,d]).

    rows=None evaluates every query row.  Inputs are converted to float64 first,
    so bf16 inputs enter with exactly their rounded values.  window=(left, right)
    and block_mask select the allowed (row, key) pairs as in attn_oracle.c.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    Tq, d = q.shape
    Tk = k.shape[0]
    assert k.shape == (Tk, d) and v.shape == (Tk, d)
    r = _idx(rows, Tq)
    o = np.zeros((r.size, d), dtype=np.float64)
    lse = np.zeros(r.size, dtype=np.float64)
    nt = nthreads or default_threads()
    if window is None and block_mask is None:
        st = _load().oracle_fwd(_ptr(q), _ptr(k), _ptr(v), Tq, Tk, d, int(bool(causal)), float(scale),
                                _ptr(r, ctypes.c_int64), r.size, _ptr(o), _ptr(lse), nt)
    else:
        left, right, bp, bs, keep = _mask_args(causal, window, block_mask, block_size, Tq, Tk)
        st = _load().oracle_fwd_masked(_ptr(q), _ptr(k), _ptr(v), Tq, Tk, d, left, right, bp, bs, float(scale),
                                       _ptr(r, ctypes.c_int64), r.size, _ptr(o), _ptr(lse), nt)
        del keep
    if st:
        raise RuntimeError(f"oracle_fwd failed with status {st}")
    return o, lse


def attention_bwd(q, k, v, dO, causal: bool, scale: float, rows=None, keys=None,
                  want_o: bool = False, nthreads: int | None = None, window=None, block_mask=None,
                  block_size: int = 128):
    """Analytic gradients of one head.

    Returns a dict with dq [len(rows), d], dk and dv [len(keys), d], and the
    per-row statistics lse [Tq] and D [Tq] (plus o [Tq, d] if want_o).
    rows/keys=None mean every row / every key.
    """
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    Tq, d = q.shape
    Tk = k.shape[0]
    assert dO.shape == (Tq, d) and k.shape == (Tk, d) and v.shape == (Tk, d)
    r = _idx(rows, Tq)
    kk = _idx(keys, Tk)
    dq = np.zeros((r.size, d))
    dk = np.zeros((kk.size, d))
    dv = np.zeros((kk.size, d))
    lse = np.zeros(Tq)
    D = np.zeros(Tq)
    o = np.zeros((Tq, d)) if want_o else None
    nt = nthreads or default_threads()
    o_ptr = _ptr(o) if want_o else ctypes.POINTER(ctypes.c_double)()
    if window is None and block_mask is None:
        st = _load().oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), Tq, Tk, d, int(bool(causal)),
                                float(scale), _ptr(r, ctypes.c_int64), r.size, _ptr(kk, ctypes.c_int64),
                                kk.size, _ptr(dq), _ptr(dk), _ptr(dv), o_ptr, _ptr(lse), _ptr(D), nt)
    else:
        left, right, bp, bs, keep = _mask_args(causal, window, block_mask, block_size, Tq, Tk)
        st = _load().oracle_bwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), Tq, Tk, d, left, right, bp, bs,
                                       float(scale), _ptr(r, ctypes.c_int64), r.size, _ptr(kk, ctypes.c_int64),
                                       kk.size, _ptr(dq), _ptr(dk), _ptr(dv), o_ptr, _ptr(lse), _ptr(D), nt)
        del keep
    if st:
        raise RuntimeError(f"oracle_bwd failed with status {st}")
    out = {"dq": dq, "dk": dk, "dv": dv, "lse": lse, "D": D}
    if want_o:
        out["o"] = o
    return out
