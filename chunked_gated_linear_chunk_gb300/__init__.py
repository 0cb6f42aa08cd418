"""Chunk-parallel gated linear attention (GLA, Mamba-2 SSD) for GB300.

Thin Python binding over the C ABI in ``include/glacore.h`` (library
``libglacore.so``, built from ``csrc/`` by ``_build.py``).  This module only
marshals arguments: PyTorch provides device memory and the current stream;
every step of the computation runs in the library's CUDA kernels.  There is
no CPU or PyTorch fallback: if the library cannot be loaded every call
raises.

Entry points (same names as the C ABI):
    gla_fwd(q, k, v, g, ...)            -> (o, final_state)
    gla_bwd(q, k, v, g, do, ...)        -> (dq, dk, dv, dg, dh0)
    ssd_fwd / ssd_bwd                   (scalar per-head gate, g [B,T,H])
    count_docs(segment_ids)             -> int
    get_device_error()                  -> None or raises GlacoreError

Layouts: q, k [B,T,Hqk,K]; v, o, do [B,T,H,V]; g [B,T,H,K] (GLA) or
[B,T,H] (SSD), fp32; states [n_seqs,H,K,V] fp32; segment_ids [B,T] int32.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "GlacoreError", "load", "gla_fwd", "gla_bwd", "ssd_fwd", "ssd_bwd", "count_docs",
    "get_device_error", "workspace_size", "Problem", "selftest_wait",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libglacore.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE, ERR_DOCS, ERR_RANGE = range(8)
F32, BF16 = 0, 1

EXPORTS = (
    "gla_fwd", "gla_bwd", "ssd_fwd", "ssd_bwd", "gla_fwd_workspace_size", "gla_bwd_workspace_size",
    "ssd_fwd_workspace_size", "ssd_bwd_workspace_size", "glacore_count_docs",
    "glacore_get_device_error", "glacore_status_string", "glacore_version",
    "glacore_set_timing_events", "glacore_timing_count", "glacore_timing_label", "gla_bwd_noalloc",
    "glacore_selftest_wait",
)


class GlacoreError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = _status_string(status)
        super().__init__(f"glacore status {status} ({msg}){': ' + what if what else ''}")


class Problem(ctypes.Structure):
    """Mirror of ``glacore_problem`` in include/glacore.h."""

    _fields_ = [
        ("B", ctypes.c_int64), ("T", ctypes.c_int64), ("H", ctypes.c_int64),
        ("Hqk", ctypes.c_int64), ("K", ctypes.c_int64), ("V", ctypes.c_int64),
        ("dtype", ctypes.c_int32), ("chunk_size", ctypes.c_int32), ("scale", ctypes.c_float),
        ("reserved0", ctypes.c_int32),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("g", ctypes.c_void_p), ("segment_ids", ctypes.c_void_p), ("n_seqs", ctypes.c_int64),
        ("initial_state", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
    ]


_lib = None
_lock = threading.Lock()


def load(path: str | None = None):
    """Loads libglacore.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if path is None:
            from . import _build

            if _build.needs_build():
                _build.build()
        lib = ctypes.CDLL(p)
        P = ctypes.c_void_p
        PP = ctypes.POINTER(Problem)
        for n in ("gla_fwd", "ssd_fwd"):
            f = getattr(lib, n)
            f.restype = ctypes.c_int
            f.argtypes = [PP, P, P, P]
        for n in ("gla_bwd", "ssd_bwd", "gla_bwd_noalloc"):
            f = getattr(lib, n)
            f.restype = ctypes.c_int
            f.argtypes = [PP, P, P, P, P, P, P, P, P]
        for n in ("gla_fwd_workspace_size", "gla_bwd_workspace_size", "ssd_fwd_workspace_size",
                  "ssd_bwd_workspace_size"):
            f = getattr(lib, n)
            f.restype = ctypes.c_size_t
            f.argtypes = [PP]
        lib.glacore_count_docs.restype = ctypes.c_int
        lib.glacore_count_docs.argtypes = [P, ctypes.c_int64, ctypes.c_int64, P, P]
        lib.glacore_get_device_error.restype = ctypes.c_int
        lib.glacore_get_device_error.argtypes = [P]
        lib.glacore_status_string.restype = ctypes.c_char_p
        lib.glacore_status_string.argtypes = [ctypes.c_int]
        lib.glacore_version.restype = ctypes.c_int
        lib.glacore_version.argtypes = []
        lib.glacore_set_timing_events.restype = None
        lib.glacore_set_timing_events.argtypes = [P, ctypes.c_int]
        lib.glacore_timing_count.restype = ctypes.c_int
        lib.glacore_timing_count.argtypes = []
        lib.glacore_timing_label.restype = ctypes.c_char_p
        lib.glacore_timing_label.argtypes = [ctypes.c_int]
        lib.glacore_selftest_wait.restype = ctypes.c_int
        lib.glacore_selftest_wait.argtypes = [ctypes.c_int64, P]
        if path is None:
            _lib = lib
        return lib


def _status_string(s: int) -> str:
    try:
        return load().glacore_status_string(int(s)).decode()
    except OSError:
        return "unknown"


def _check(status: int, what: str):
    if status != OK:
        raise GlacoreError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"q/k/v must be bfloat16 or float32, got {t.dtype}")


def _contig(t, dtype=None):
    if t is None:
        return None
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError("glacore takes CUDA tensors")
    return t if t.is_contiguous() else t.contiguous()


def _new(shape, dtype, device, poison):
    if poison:
        return torch.full(shape, float("nan"), dtype=dtype, device=device)
    return torch.empty(shape, dtype=dtype, device=device)


def count_docs(segment_ids: torch.Tensor) -> int:
    """Number of documents in segment_ids [B,T] (runs a kernel, then syncs)."""
    seg = _contig(segment_ids, torch.int32)
    B, T = seg.shape
    out = torch.empty(1, dtype=torch.int64, device=seg.device)
    _check(load().glacore_count_docs(_ptr(seg), B, T, _ptr(out), _stream(seg.device)), "count_docs")
    return int(out.item())


class LaunchTimer:
    """Per-kernel CUDA-event timing through the library's measurement hook.

    ``with LaunchTimer(n) as t: gla_fwd(...)`` records one event after each
    kernel launch of the call; ``t.labels`` names the kernels and
    ``t.events`` holds the torch events (elapsed times are read after a
    synchronize)."""

    def __init__(self, n: int = 8):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in self.events:  # create the underlying CUDA events
            e.record()
        self._arr = (ctypes.c_void_p * n)(*[e.cuda_event for e in self.events])
        self.labels = []

    def __enter__(self):
        load().glacore_set_timing_events(ctypes.cast(self._arr, ctypes.c_void_p), len(self.events))
        return self

    def __exit__(self, *exc):
        lib = load()
        n = lib.glacore_timing_count()
        self.labels = [lib.glacore_timing_label(i).decode() for i in range(n)]
        lib.glacore_set_timing_events(None, 0)
        return False


def get_device_error():
    """Reads and clears the device error word; raises GlacoreError if set."""
    _check(load().glacore_get_device_error(_stream(torch.cuda.current_device())), "device")


def selftest_wait(cycles: int, device=None):
    """Runs the library's bounded-wait self-test on the current stream: a
    wait that can never complete, with a limit of ``cycles`` SM clocks.  The
    timeout lands in the device error word (read it with get_device_error)."""
    dev = torch.cuda.current_device() if device is None else device
    _check(load().glacore_selftest_wait(int(cycles), _stream(dev)), "selftest_wait")


def _problem(q, k, v, g, scale, segment_ids, initial_state, chunk_size, n_seqs, head_gate):
    q, k, v = _contig(q), _contig(k), _contig(v)
    g = _contig(g, torch.float32)
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    B, T, Hqk, K = q.shape
    H, V = v.shape[2], v.shape[3]
    if tuple(k.shape) != (B, T, Hqk, K) or tuple(v.shape[:2]) != (B, T):
        raise ValueError("shape mismatch between q, k, v")
    if head_gate and tuple(g.shape) != (B, T, H):
        raise ValueError("SSD gate must be [B,T,H]")
    if not head_gate and tuple(g.shape) != (B, T, H, K):
        raise ValueError("GLA gate must be [B,T,H,K]")
    seg = _contig(segment_ids, torch.int32) if segment_ids is not None else None
    if seg is None:
        n = B if T > 0 else 0
    else:
        n = n_seqs if n_seqs is not None else count_docs(seg)
    h0 = _contig(initial_state, torch.float32) if initial_state is not None else None
    if h0 is not None and tuple(h0.shape) != (n, H, K, V):
        raise ValueError(f"initial_state must be [{n},{H},{K},{V}]")
    if scale is None:
        scale = K ** -0.5 if not head_gate else 1.0
    p = Problem(B=B, T=T, H=H, Hqk=Hqk, K=K, V=V, dtype=_dtype_code(q), chunk_size=int(chunk_size),
                scale=float(scale), reserved0=0, q=q.data_ptr(), k=k.data_ptr(), v=v.data_ptr(),
                g=g.data_ptr(), segment_ids=seg.data_ptr() if seg is not None else None, n_seqs=n,
                initial_state=h0.data_ptr() if h0 is not None else None, workspace=None,
                workspace_bytes=0)
    keep = (q, k, v, g, seg, h0)
    return p, keep


def workspace_size(p: Problem, kind: str) -> int:
    return int(getattr(load(), kind + "_workspace_size")(ctypes.byref(p)))


def _workspace(p, kind, device, workspace):
    need = workspace_size(p, kind)
    if need == 0:
        return None
    if workspace is not None and workspace.numel() >= need and workspace.data_ptr() % 256 == 0:
        ws = workspace
    else:
        ws = torch.empty(need, dtype=torch.uint8, device=device)
    p.workspace = ws.data_ptr()
    p.workspace_bytes = ws.numel()
    return ws


def _fwd(kind, q, k, v, g, scale=None, segment_ids=None, initial_state=None,
         output_final_state=False, chunk_size=0, n_seqs=None, out=None, final_out=None,
         workspace=None, poison=False):
    head_gate = kind == "ssd"
    p, keep = _problem(q, k, v, g, scale, segment_ids, initial_state, chunk_size, n_seqs, head_gate)
    dev = keep[0].device
    o = out if out is not None else _new(tuple(keep[2].shape), keep[0].dtype, dev, poison)
    ht = None
    if output_final_state:
        ht = final_out if final_out is not None else _new((p.n_seqs, p.H, p.K, p.V), torch.float32, dev,
                                                          poison)
    ws = _workspace(p, kind + "_fwd", dev, workspace)
    st = getattr(load(), kind + "_fwd")(ctypes.byref(p), _ptr(o), _ptr(ht), _stream(dev))
    _check(st, kind + "_fwd")
    del ws, keep
    return o, ht


def _bwd(kind, q, k, v, g, do, scale=None, segment_ids=None, initial_state=None, dht=None,
         chunk_size=0, n_seqs=None, outs=None, workspace=None, poison=False):
    head_gate = kind == "ssd"
    p, keep = _problem(q, k, v, g, scale, segment_ids, initial_state, chunk_size, n_seqs, head_gate)
    dev = keep[0].device
    do = _contig(do, keep[0].dtype)
    dht = _contig(dht, torch.float32) if dht is not None else None
    if tuple(do.shape) != tuple(keep[2].shape):
        raise ValueError("do must match v")
    if dht is not None and tuple(dht.shape) != (p.n_seqs, p.H, p.K, p.V):
        raise ValueError("dht must be [n_seqs,H,K,V]")
    if outs is not None:
        dq, dk, dv, dg, dh0 = outs
    else:
        dq = _new(tuple(keep[0].shape), keep[0].dtype, dev, poison)
        dk = _new(tuple(keep[1].shape), keep[0].dtype, dev, poison)
        dv = _new(tuple(keep[2].shape), keep[0].dtype, dev, poison)
        dg = _new(tuple(keep[3].shape), torch.float32, dev, poison)
        dh0 = _new((p.n_seqs, p.H, p.K, p.V), torch.float32, dev, poison) if initial_state is not None else None
    ws = _workspace(p, kind + "_bwd", dev, workspace)
    st = getattr(load(), kind + "_bwd")(ctypes.byref(p), _ptr(do), _ptr(dht), _ptr(dq), _ptr(dk), _ptr(dv),
                                        _ptr(dg), _ptr(dh0), _stream(dev))
    _check(st, kind + "_bwd")
    del ws, keep
    return dq, dk, dv, dg, dh0


def gla_fwd(q, k, v, g, scale=None, segment_ids=None, initial_state=None, output_final_state=False,
            chunk_size=0, n_seqs=None, **kw):
    """GLA forward.  Returns (o, final_state or None)."""
    return _fwd("gla", q, k, v, g, scale, segment_ids, initial_state, output_final_state, chunk_size,
                n_seqs, **kw)


def gla_bwd(q, k, v, g, do, scale=None, segment_ids=None, initial_state=None, dht=None, chunk_size=0,
            n_seqs=None, **kw):
    """GLA backward.  Returns (dq, dk, dv, dg, dh0 or None)."""
    return _bwd("gla", q, k, v, g, do, scale, segment_ids, initial_state, dht, chunk_size, n_seqs, **kw)


def ssd_fwd(q, k, v, g, scale=1.0, segment_ids=None, initial_state=None, output_final_state=False,
            chunk_size=0, n_seqs=None, **kw):
    """Mamba-2 SSD forward (g is the per-head log decay [B,T,H])."""
    return _fwd("ssd", q, k, v, g, scale, segment_ids, initial_state, output_final_state, chunk_size,
                n_seqs, **kw)


def ssd_bwd(q, k, v, g, do, scale=1.0, segment_ids=None, initial_state=None, dht=None, chunk_size=0,
            n_seqs=None, **kw):
    """Mamba-2 SSD backward.  Returns (dq, dk, dv, dg, dh0 or None)."""
    return _bwd("ssd", q, k, v, g, do, scale, segment_ids, initial_state, dht, chunk_size, n_seqs, **kw)
