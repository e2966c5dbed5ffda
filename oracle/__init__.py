"""Float64 CPU oracle of the Swin shifted-window attention block.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it to check and to time the GPU library;
the library itself never imports, links or runs anything here, and nothing
here imports the library.  Two independent formulations live in this package:

* ``swin_oracle.c`` (loaded through ctypes): the block written as the pages
  describe it, step by step -- cyclic shift by -s, window partition, QKV
  projection, per-window per-head logits with relative position bias and the
  shift-region mask, softmax, P.V, output projection, window reverse and roll
  back by +s.  Pages: "Boosting Swin Transformer Speed: Profiling, Mixed
  Precision, and Kernel Fusion Secrets" (Introduction, Training
  Optimization) and "Swin Transformer V2" (How It Works).
* ``brute.py``: a window-free NumPy statement for tiny grids that never forms
  a window, a roll or a mask: two tokens attend iff they fall in the same
  shifted window and are adjacent in the original image without wrapping.

Each function states which pin in ``tests/test_oracle.py`` holds it to
something other than itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "swin_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

V1, V2 = 0, 1


def build(force: bool = False) -> str:
    """Compile ``swin_oracle.c`` with gcc (-O2, OpenMP) into liboracle.so."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            dp = ctypes.POINTER(ctypes.c_double)
            i64p = ctypes.POINTER(ctypes.c_int64)
            ci = ctypes.c_int
            lib.oracle_roll.argtypes = [dp, ci, ci, ci, ci, ci, dp]
            lib.oracle_partition.argtypes = [dp, ci, ci, ci, ci, ci, dp]
            lib.oracle_reverse.argtypes = [dp, ci, ci, ci, ci, ci, dp]
            lib.oracle_forward.argtypes = [dp, ci, ci, ci, ci, ci, ci, ci, ci, dp, dp, dp, dp, dp,
                                           dp, dp, i64p, ctypes.c_int64, ci]
            lib.oracle_forward.restype = ci
            lib.oracle_window_attention.argtypes = [dp, ci, ci, ci, ci, ci, ci, ci, ci, dp, dp, dp,
                                                    dp, dp, dp, ctypes.c_int64, dp, dp, dp]
            lib.oracle_window_attention.restype = ci
            lib.oracle_cpb_table.argtypes = [ci, ci, ci, dp, dp, dp, dp]
            lib.oracle_cpb_table.restype = ci
            lib.oracle_max_threads.restype = ci
            _lib = lib
    return _lib


def _d(a):
    """Contiguous float64 copy (or None) and its ctypes pointer."""
    if a is None:
        return None, None
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def roll(x, r):
    """torch.roll of a [B,H,W,C] array by r on both spatial axes."""
    x, px = _d(x)
    y = np.empty_like(x)
    B, H, W, C = x.shape
    _load().oracle_roll(px, B, H, W, C, int(r), y.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return y


def partition(xs, M):
    """[B,H,W,C] -> [B*(H/M)*(W/M), M*M, C], windows and tokens row-major."""
    xs, px = _d(xs)
    B, H, W, C = xs.shape
    xw = np.empty((B * (H // M) * (W // M), M * M, C))
    _load().oracle_partition(px, B, H, W, C, M, xw.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return xw


def reverse(xw, B, H, W, M):
    """Inverse of partition."""
    xw, px = _d(xw)
    C = xw.shape[-1]
    xs = np.empty((B, H, W, C))
    _load().oracle_reverse(px, B, H, W, C, M, xs.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return xs


def forward(x, Wqkv, bqkv, table, tau, Wproj, bproj, *, heads, M, shift, mode,
            windows=None, nthreads=0, out=None):
    """The whole block in float64.  x [B,H,W,C]; Wqkv [3C,C]; bqkv [3C];
    table [(2M-1)^2, heads]; tau [heads] (V2) or None; Wproj [C,C]; bproj [C].
    With ``windows`` (window numbers (b*(H/M)+wi)*(W/M)+wj) only those windows'
    output tokens are computed; the rest of ``out`` is left as given (NaN if
    ``out`` is None)."""
    x, px = _d(x)
    B, H, W, C = x.shape
    Wqkv, pWq = _d(Wqkv)
    bqkv, pbq = _d(bqkv)
    table, pt = _d(table)
    tau, ptau = _d(tau)
    Wproj, pWp = _d(Wproj)
    bproj, pbp = _d(bproj)
    if out is None:
        out = np.full((B, H, W, C), np.nan)
    assert out.dtype == np.float64 and out.flags.c_contiguous and out.shape == x.shape
    if windows is not None:
        wl = np.ascontiguousarray(np.asarray(windows, dtype=np.int64))
        pw, nw = wl.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), len(wl)
    else:
        pw, nw = None, 0
    rc = _load().oracle_forward(px, B, H, W, C, heads, M, shift, mode, pWq, pbq, pt, ptau, pWp, pbp,
                                out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), pw, nw,
                                int(nthreads))
    if rc != 0:
        raise ValueError("oracle_forward rejected the arguments")
    return out


def window_attention(x, Wqkv, bqkv, table, tau, Wproj, bproj, *, heads, M, shift, mode, win):
    """(logits, probs, out) of one window: logits and probs are [heads,N,N]
    (logits -inf where masked); out holds that window's output tokens."""
    x, px = _d(x)
    B, H, W, C = x.shape
    N = M * M
    Wqkv, pWq = _d(Wqkv)
    bqkv, pbq = _d(bqkv)
    table, pt = _d(table)
    tau, ptau = _d(tau)
    Wproj, pWp = _d(Wproj)
    bproj, pbp = _d(bproj)
    logits = np.empty((heads, N, N))
    probs = np.empty((heads, N, N))
    out = np.full((B, H, W, C), np.nan)
    dp = ctypes.POINTER(ctypes.c_double)
    rc = _load().oracle_window_attention(px, B, H, W, C, heads, M, shift, mode, pWq, pbq, pt, ptau,
                                         pWp, pbp, int(win), logits.ctypes.data_as(dp),
                                         probs.ctypes.data_as(dp), out.ctypes.data_as(dp))
    if rc != 0:
        raise ValueError("oracle_window_attention rejected the arguments")
    return logits, probs, out


def cpb_table(W1, b1, W2, *, M, heads):
    """Table of the meta-network G over log-spaced relative coordinates,
    [(2M-1)^2, heads]."""
    W1, p1 = _d(W1)
    b1, pb = _d(b1)
    W2, p2 = _d(W2)
    hidden = W1.shape[0]
    assert W1.shape == (hidden, 2) and W2.shape == (heads, hidden)
    table = np.empty(((2 * M - 1) ** 2, heads))
    rc = _load().oracle_cpb_table(M, heads, hidden, p1, pb, p2,
                                  table.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    if rc != 0:
        raise ValueError("oracle_cpb_table rejected the arguments")
    return table
