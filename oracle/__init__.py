"""fp64 CPU oracle for the fused attention forward pass.

TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The oracle shares no code with the CUDA
library (``warp_specialized_attention_gb300``) and neither imports the other;
the only thing both sides consume is the seeded synthetic inputs.

The arithmetic lives in ``attn_oracle.c`` (plain C, double precision, two-pass
softmax, OpenMP over independent rows) and, for the backward pass (the
gradients of that definition), in ``attn_oracle_bwd.c``.  This module compiles it with gcc into
``_attn_oracle.so`` beside the source and marshals numpy float64 arrays into it.
The definition it follows -- attention split into Q K^T, softmax and P V as in
"Tawa: Automatic Warp Specialization for Modern GPUs with Asynchronous
References", Section III-D, Algorithm 1 -- is written out in the C file's header.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_SRC_BWD = os.path.join(_HERE, "attn_oracle_bwd.c")
_LIB = os.path.join(_HERE, "_attn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``_attn_oracle.so`` (gcc, -O2, OpenMP)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= max(os.path.getmtime(_SRC), os.path.getmtime(_SRC_BWD))):
        return _LIB
    tmp = _LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
           "-o", tmp, _SRC, _SRC_BWD, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int64)
            lib.attn_oracle_rows.argtypes = [dp, dp, dp, ctypes.c_int64, ctypes.c_int64,
                                             ip, ctypes.c_int64, ctypes.c_int,
                                             ctypes.c_double, dp, dp]
            lib.attn_oracle_rows.restype = ctypes.c_int
            lib.attn_oracle_full.argtypes = [dp, dp, dp, ctypes.c_int64, ctypes.c_int64,
                                             ctypes.c_int64, ctypes.c_int, ctypes.c_double,
                                             dp, dp]
            lib.attn_oracle_full.restype = ctypes.c_int
            lib.attn_oracle_bwd_slice.argtypes = [dp, dp, dp, dp, ctypes.c_int64,
                                                  ctypes.c_int64, ctypes.c_int,
                                                  ctypes.c_double, dp, dp, dp]
            lib.attn_oracle_bwd_slice.restype = ctypes.c_int
            lib.attn_oracle_threads.argtypes = []
            lib.attn_oracle_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray, ctype=ctypes.c_double):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def threads() -> int:
    """Host threads an oracle call uses (OMP_NUM_THREADS, else all cores)."""
    return int(_load().attn_oracle_threads())


def attention_rows(q_rows, k, v, rows, causal: bool, scale: float):
    """Selected rows of one (batch, head) slice.

    q_rows: (n, D) query rows; rows: (n,) their query indices in [0, S);
    k, v: (S, D).  Returns (o (n, D), lse (n,)) as float64.
    """
    q_rows, k, v = _f64(q_rows), _f64(k), _f64(v)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    n = rows.shape[0]
    S, D = k.shape
    if q_rows.shape != (n, D) or v.shape != (S, D):
        raise ValueError("shape mismatch: q_rows %s rows %s k %s v %s"
                         % (q_rows.shape, rows.shape, k.shape, v.shape))
    o = np.empty((n, D), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    rc = _load().attn_oracle_rows(_ptr(q_rows), _ptr(k), _ptr(v), S, D,
                                  _ptr(rows, ctypes.c_int64), n, int(bool(causal)),
                                  float(scale), _ptr(o), _ptr(lse))
    if rc != 0:
        raise RuntimeError("attn_oracle_rows failed with code %d" % rc)
    return o, lse


def attention(q, k, v, causal: bool, scale: float):
    """Every row of every slice.  q, k, v: (..., S, D).  Returns (o, lse)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    if not (q.shape == k.shape == v.shape) or q.ndim < 2:
        raise ValueError("q, k, v must share one (..., S, D) shape")
    lead = q.shape[:-2]
    S, D = q.shape[-2:]
    BH = int(np.prod(lead)) if lead else 1
    o = np.empty(q.shape, dtype=np.float64)
    lse = np.empty(lead + (S,), dtype=np.float64)
    rc = _load().attn_oracle_full(_ptr(q), _ptr(k), _ptr(v), BH, S, D,
                                  int(bool(causal)), float(scale), _ptr(o), _ptr(lse))
    if rc != 0:
        raise RuntimeError("attn_oracle_full failed with code %d" % rc)
    return o, lse


def attention_bwd(q, k, v, dout, causal: bool, scale: float):
    """Gradients of the forward definition with respect to q, k, v, given dO.

    q, k, v, dout: (..., S, D).  Returns (dq, dk, dv) as float64."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    if not (q.shape == k.shape == v.shape == dout.shape) or q.ndim < 2:
        raise ValueError("q, k, v, dout must share one (..., S, D) shape")
    S, D = q.shape[-2:]
    flat = [t.reshape(-1, S, D) for t in (q, k, v, dout)]
    outs = [np.empty((flat[0].shape[0], S, D), dtype=np.float64) for _ in range(3)]
    lib = _load()
    for bh in range(flat[0].shape[0]):
        sl = [np.ascontiguousarray(t[bh]) for t in flat]
        res = [np.empty((S, D), dtype=np.float64) for _ in range(3)]
        rc = lib.attn_oracle_bwd_slice(*(_ptr(t) for t in sl), S, D, int(bool(causal)),
                                       float(scale), *(_ptr(r) for r in res))
        if rc != 0:
            raise RuntimeError("attn_oracle_bwd_slice failed with code %d" % rc)
        for o, r in zip(outs, res):
            o[bh] = r
    return tuple(o.reshape(q.shape) for o in outs)
