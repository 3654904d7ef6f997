"""FP64 CPU oracle for exact masked softmax attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package. It shares no code with the CUDA
library (``online_softmax_02_gb300``) and never imports it; the CUDA library
never imports this package.

Contents
  * ``attn_oracle.c`` (loaded here through ctypes): the plain three-pass
    definition of masked softmax attention plus the per-row log-sum-exp, and
    the plain three-pass row softmax, in double precision. See the header of
    that file for the steps and citations.
  * ``backward.py``: the chain-rule gradients of attention in FP64.
  * ``recurrence.py``: the online (m, l) pair update, its merge, and the
    blockwise query-tile recurrence, written from the pages' equations. They
    are used only to cross-check the direct definition above.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(worked example, closed forms, brute force at 50 digits, library routine,
invariants, and planted mutants that must fail).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_WINDOW = 2
MASK_PADDING = 4

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()


def compile_oracle(src: str = _SRC, out: str = _LIB, force: bool = False) -> str:
    """Compile the C oracle into a shared library with gcc and OpenMP."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


class Oracle:
    """ctypes handle on one build of the C oracle."""

    def __init__(self, lib_path: str | None = None):
        if lib_path is None:
            with _lock:
                lib_path = compile_oracle()
        self.lib_path = lib_path
        self._lib = ctypes.CDLL(lib_path)
        f = self._lib.oracle_attn_rows
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 5 + [
            ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_longlong, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_int]
        self._lib.oracle_max_threads.restype = ctypes.c_int
        g = self._lib.oracle_softmax_rows
        g.restype = ctypes.c_int
        g.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_longlong, ctypes.c_void_p,
                      ctypes.c_void_p, ctypes.c_int]

    def attention(self, q, k, v, scale, mask_kind=MASK_NONE, window=0,
                  seqlens_k=None, rows=None, threads=None):
        """Exact masked attention in FP64.

        q: [B,H,Nq,d], k/v: [B,H,Nk,d] (anything numpy turns into float32
        without rounding: FP32 or BF16 values). ``rows``: optional flat
        row indices (b*H+h)*Nq+i to evaluate; default every row.
        Returns (o, lse): o [B,H,Nq,d] / [len(rows),d], lse [B,H,Nq] /
        [len(rows)], both float64.
        """
        q = np.ascontiguousarray(q, dtype=np.float32)
        k = np.ascontiguousarray(k, dtype=np.float32)
        v = np.ascontiguousarray(v, dtype=np.float32)
        if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
            raise ValueError("q, k, v must be [B,H,N,d]")
        B, H, Nq, d = q.shape
        Nk = k.shape[2]
        if k.shape != (B, H, Nk, d) or v.shape != (B, H, Nk, d):
            raise ValueError("k and v must be [B,H,Nk,d] matching q")
        sl = None
        if mask_kind & MASK_PADDING:
            if seqlens_k is None:
                raise ValueError("padding mask needs seqlens_k")
            sl = np.ascontiguousarray(seqlens_k, dtype=np.int32)
            if sl.shape != (B,):
                raise ValueError("seqlens_k must be [B]")
        if rows is None:
            n = B * H * Nq
            rows_arr = None
        else:
            rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
            n = rows_arr.shape[0]
        o = np.zeros((n, d), dtype=np.float64)
        lse = np.zeros((n,), dtype=np.float64)
        nthreads = threads or default_threads()
        rc = self._lib.oracle_attn_rows(
            q.ctypes.data, k.ctypes.data, v.ctypes.data, B, H, Nq, Nk, d,
            float(scale), int(mask_kind), int(window),
            None if sl is None else sl.ctypes.data,
            None if rows_arr is None else rows_arr.ctypes.data,
            n, o.ctypes.data, lse.ctypes.data, nthreads)
        if rc != 0:
            raise ValueError("oracle_attn_rows failed with code %d" % rc)
        if rows is None:
            return o.reshape(B, H, Nq, d), lse.reshape(B, H, Nq)
        return o, lse

    def softmax_rows(self, x, threads=None):
        """Row softmax of x [rows, n] in FP64 (three-pass safe softmax).
        Returns (y [rows, n], lse [rows]) as float64."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        if x.ndim != 2:
            raise ValueError("x must be [rows, n]")
        rows, n = x.shape
        y = np.zeros((rows, n), dtype=np.float64)
        lse = np.zeros(rows, dtype=np.float64)
        rc = self._lib.oracle_softmax_rows(x.ctypes.data, rows, n, y.ctypes.data,
                                           lse.ctypes.data, threads or default_threads())
        if rc != 0:
            raise ValueError("oracle_softmax_rows failed with code %d" % rc)
        return y, lse

    def max_threads(self) -> int:
        return int(self._lib.oracle_max_threads())


_default: Oracle | None = None


def get() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def attention(*args, **kwargs):
    """Module-level shortcut to ``Oracle().attention`` on the default build."""
    return get().attention(*args, **kwargs)
