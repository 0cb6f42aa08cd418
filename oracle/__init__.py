"""fp64 CPU oracle for the gated linear attention recurrence (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` leg of
``bench.py`` may import this package.  It shares no code with the CUDA path
in ``chunked_gated_linear_chunk_gb300/csrc`` and that path never imports it.

The work is done by ``oracle.c`` (token-by-token recurrence in double, built
into ``liboracle.so`` with gcc).  This module only converts arrays to
contiguous float64 and calls it.

Parity status per function:
  fwd  -- pinned (closed form for g = 0, Mamba-2 dual form, brute-force
          parallel form, packed documents, special cases; tests/test_oracle.py)
  bwd  -- pinned (central finite differences, adjoint identity, closed form
          for g = 0, two derivations of dg; tests/test_oracle.py)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

GATE_CHANNEL = 0  # GLA: g is [B,T,H,K]
GATE_HEAD = 1  # Mamba-2 SSD: g is [B,T,H]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain C, -O2, pthreads)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm", "-lpthread"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            lib.oracle_count_docs.restype = I64
            lib.oracle_count_docs.argtypes = [I64, I64, P]
            lib.oracle_fwd.restype = ctypes.c_int
            lib.oracle_fwd.argtypes = [I64] * 6 + [ctypes.c_int, ctypes.c_double] + [P] * 5 + [I64] + [P] * 3 + [ctypes.c_int]
            lib.oracle_bwd.restype = ctypes.c_int
            lib.oracle_bwd.argtypes = [I64] * 6 + [ctypes.c_int, ctypes.c_double] + [P] * 5 + [I64] + [P] * 8 + [ctypes.c_int]
            _lib = lib
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor -> exact upcast on the CPU
        x = x.detach().to("cpu")
        import torch

        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _threads(n):
    if n is not None:
        return int(n)
    return max(1, os.cpu_count() or 1)


def count_docs(segment_ids, B: int, T: int) -> int:
    seg = _i32(segment_ids)
    return int(_load().oracle_count_docs(B, T, _ptr(seg)))


def _shapes(q, v, g):
    B, T, Hqk, K = q.shape
    H, V = v.shape[2], v.shape[3]
    gate = GATE_CHANNEL if g.ndim == 4 else GATE_HEAD
    return B, T, H, Hqk, K, V, gate


def fwd(q, k, v, g, scale, segment_ids=None, h0=None, threads=None):
    """Forward: returns (o [B,T,H,V], ht [n_docs,H,K,V]) in float64.

    g of shape [B,T,H,K] selects the per-key-channel (GLA) gate, [B,T,H] the
    per-head (Mamba-2 SSD) gate.  q, k are [B,T,Hqk,K] with Hqk dividing H.
    """
    q, k, v, g, h0 = map(_f64, (q, k, v, g, h0))
    seg = _i32(segment_ids)
    B, T, H, Hqk, K, V, gate = _shapes(q, v, g)
    n = count_docs(seg, B, T)
    o = np.empty((B, T, H, V))
    ht = np.empty((n, H, K, V))
    rc = _load().oracle_fwd(B, T, H, Hqk, K, V, gate, float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                            _ptr(seg), n, _ptr(h0), _ptr(o), _ptr(ht), _threads(threads))
    if rc != 0:
        raise ValueError("oracle_fwd failed with code %d" % rc)
    return o, ht


def bwd(q, k, v, g, do, scale, segment_ids=None, h0=None, dht=None, threads=None):
    """Backward: returns dict dq, dk, dv, dg, dh0 (float64)."""
    q, k, v, g, do, h0, dht = map(_f64, (q, k, v, g, do, h0, dht))
    seg = _i32(segment_ids)
    B, T, H, Hqk, K, V, gate = _shapes(q, v, g)
    n = count_docs(seg, B, T)
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    dg = np.empty_like(g)
    dh0 = np.empty((n, H, K, V))
    rc = _load().oracle_bwd(B, T, H, Hqk, K, V, gate, float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                            _ptr(seg), n, _ptr(h0), _ptr(do), _ptr(dht), _ptr(dq), _ptr(dk), _ptr(dv),
                            _ptr(dg), _ptr(dh0), _threads(threads))
    if rc != 0:
        raise ValueError("oracle_bwd failed with code %d" % rc)
    return {"dq": dq, "dk": dk, "dv": dv, "dg": dg, "dh0": dh0}
