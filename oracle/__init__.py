"""CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never imports, links or calls it, and it shares no code with
the product.

Two independent implementations live here:

* ``naive_attention.c`` -- plain fp64 two-pass attention over every allowed
  key of a row (the "standard attention" / "naive full-softmax reference" of
  the pages), and its backward pass by recomputation.  This is THE oracle.
  ``attention()``, ``attention_rows()`` and ``attention_bwd()`` below call
  it through ctypes.
* ``tiled.py`` -- the pages' block-tiled online-softmax loop in fp64 NumPy,
  plus the associative merge of partial softmax states.  It exists to pin the
  oracle (method equivalence at many block sizes) and is never compared with
  the GPU directly.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(library special cases, closed forms, invariants, Decimal brute force, the
tiled mirror, planted mutants).  ``attention_rows()`` has pins of its own for
the steps it adds (turning a flat row index into batch, head and position,
and picking that batch's key length): its rows against torch's fp64 softmax
at the decoded position and, bit for bit, against the same rows of
``attention()``, with slips planted in that decoding caught.  The one item of the pages that cannot be
pinned -- the "hand-computed case" of
"js-flash-attention-tiled-online-softmax-exactness" (Verification), which
prints outputs but no inputs -- is not used anywhere: parity unpinned.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "naive_attention.c")
LIBRARY = os.path.join(_HERE, "_build", "liboracle_attention.so")

_lock = threading.Lock()
_lib = None


def compile_oracle(source: str = SOURCE, output: str = LIBRARY) -> str:
    """Compile the C oracle with gcc (-O2, OpenMP, strict IEEE: no fast-math).

    Rebuilds only when the source is newer than the library.  Portable flags
    only, so the same build line works on x86-64 and aarch64 hosts.
    """
    os.makedirs(os.path.dirname(output), exist_ok=True)
    if os.path.exists(output) and os.path.getmtime(output) >= os.path.getmtime(source):
        return output
    tmp = output + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
           "-fno-fast-math", "-ffp-contract=off", source, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, output)
    return output


class OracleLibrary:
    """ctypes view of one compiled copy of the C oracle."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        i32p = ctypes.POINTER(ctypes.c_int32)
        i64p = ctypes.POINTER(ctypes.c_int64)
        i64 = ctypes.c_int64
        lib.oracle_attention.argtypes = [f32p, f32p, f32p, f64p, f64p, i64, i64, i64, i64,
                                         ctypes.c_int, ctypes.c_double, i32p, ctypes.c_int]
        lib.oracle_attention.restype = ctypes.c_int
        lib.oracle_attention_rows.argtypes = [f32p, f32p, f32p, i64, i64, i64, i64,
                                              ctypes.c_int, ctypes.c_double, i32p,
                                              i64p, i64, f64p, f64p, ctypes.c_int]
        lib.oracle_attention_rows.restype = ctypes.c_int
        lib.oracle_attention_bwd.argtypes = [f32p, f32p, f32p, f32p, f64p, f64p, f64p, i64, i64, i64,
                                             i64, ctypes.c_int, ctypes.c_double, i32p, ctypes.c_int]
        lib.oracle_attention_bwd.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    # -- helpers ---------------------------------------------------------
    @staticmethod
    def _f32(a):
        a = np.ascontiguousarray(a, dtype=np.float32)
        return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))

    @staticmethod
    def _kv(kv_len, B):
        if kv_len is None:
            return None, None
        kv = np.ascontiguousarray(np.asarray(kv_len, dtype=np.int32).reshape(-1))
        if kv.shape[0] != B:
            raise ValueError(f"kv_len has {kv.shape[0]} entries, expected B={B}")
        return kv, kv.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    def attention(self, q, k, v, causal=True, scale=None, kv_len=None, threads=0):
        """All rows: returns (O fp64 [B,H,N,D], LSE fp64 [B,H,N])."""
        q, qp = self._f32(q)
        k, kp = self._f32(k)
        v, vp = self._f32(v)
        B, H, N, D = q.shape
        if k.shape != q.shape or v.shape != q.shape:
            raise ValueError("q, k, v must share the shape [B,H,N,D]")
        scale = default_scale(D) if scale is None else float(scale)
        kv, kvp = self._kv(kv_len, B)
        o = np.empty((B, H, N, D), dtype=np.float64)
        lse = np.empty((B, H, N), dtype=np.float64)
        rc = self.lib.oracle_attention(qp, kp, vp,
                                       o.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                       lse.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                       B, H, N, D, int(bool(causal)), scale, kvp, int(threads))
        if rc != 0:
            raise RuntimeError("oracle_attention failed")
        return o, lse

    def attention_rows(self, q, k, v, rows, causal=True, scale=None, kv_len=None, threads=0):
        """Selected flat rows ((b*H + h)*N + i): returns (O [R,D], LSE [R]) fp64."""
        q, qp = self._f32(q)
        k, kp = self._f32(k)
        v, vp = self._f32(v)
        B, H, N, D = q.shape
        if k.shape != q.shape or v.shape != q.shape:
            raise ValueError("q, k, v must share the shape [B,H,N,D]")
        scale = default_scale(D) if scale is None else float(scale)
        kv, kvp = self._kv(kv_len, B)
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        o = np.empty((rows.shape[0], D), dtype=np.float64)
        lse = np.empty((rows.shape[0],), dtype=np.float64)
        rc = self.lib.oracle_attention_rows(qp, kp, vp, B, H, N, D, int(bool(causal)), scale,
                                            kvp, rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                            rows.shape[0],
                                            o.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                            lse.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                            int(threads))
        if rc != 0:
            raise RuntimeError("oracle_attention_rows failed (bad row index or argument)")
        return o, lse


    def attention_bwd(self, q, k, v, do, causal=True, scale=None, kv_len=None, threads=0):
        """Gradients (dQ, dK, dV), fp64 [B,H,N,D], of sum(O * dO) for O = attention(q,k,v)."""
        q, qp = self._f32(q)
        k, kp = self._f32(k)
        v, vp = self._f32(v)
        do, dop = self._f32(do)
        B, H, N, D = q.shape
        if k.shape != q.shape or v.shape != q.shape or do.shape != q.shape:
            raise ValueError("q, k, v, do must share the shape [B,H,N,D]")
        scale = default_scale(D) if scale is None else float(scale)
        kv, kvp = self._kv(kv_len, B)
        dq, dk, dv = (np.empty((B, H, N, D), dtype=np.float64) for _ in range(3))
        d64 = ctypes.POINTER(ctypes.c_double)
        rc = self.lib.oracle_attention_bwd(qp, kp, vp, dop, dq.ctypes.data_as(d64), dk.ctypes.data_as(d64),
                                           dv.ctypes.data_as(d64), B, H, N, D, int(bool(causal)), scale,
                                           kvp, int(threads))
        if rc != 0:
            raise RuntimeError("oracle_attention_bwd failed")
        return dq, dk, dv


def default_scale(D: int) -> float:
    """softmaxScale default of the pages' constructor: 1/sqrt(d)."""
    return 1.0 / math.sqrt(D)


def library() -> OracleLibrary:
    """The oracle compiled from this directory (built on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = OracleLibrary(compile_oracle())
        return _lib


def attention(q, k, v, causal=True, scale=None, kv_len=None, threads=0):
    return library().attention(q, k, v, causal=causal, scale=scale, kv_len=kv_len, threads=threads)


def attention_bwd(q, k, v, do, causal=True, scale=None, kv_len=None, threads=0):
    return library().attention_bwd(q, k, v, do, causal=causal, scale=scale, kv_len=kv_len,
                                   threads=threads)


def attention_rows(q, k, v, rows, causal=True, scale=None, kv_len=None, threads=0):
    return library().attention_rows(q, k, v, rows, causal=causal, scale=scale,
                                     kv_len=kv_len, threads=threads)
