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
    "get_device_error", "workspace_size", "Problem", "selftest_wait", "norm_gate_fwd", "norm_gate_bwd",
    "short_conv_fwd", "short_conv_bwd", "gla_fwd_state", "gla_bwd_state", "state_scan",
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
    "glacore_selftest_wait", "norm_gate_fwd", "norm_gate_bwd", "norm_gate_bwd_workspace_size",
    "short_conv_fwd", "short_conv_bwd", "short_conv_bwd_workspace_size",
    "gla_fwd_state", "gla_bwd_state", "glacore_state_scan", "glacore_last_cuda_error",
)


class GlacoreError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = _status_string(status)
        if status == ERR_CUDA:
            try:
                msg += ": " + load().glacore_last_cuda_error().decode()
            except OSError:
                pass
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
        ("q_stride", ctypes.c_int64), ("k_stride", ctypes.c_int64), ("v_stride", ctypes.c_int64),
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
        lib.glacore_last_cuda_error.restype = ctypes.c_char_p
        lib.glacore_last_cuda_error.argtypes = []
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
        I64, I32, F = ctypes.c_int64, ctypes.c_int32, ctypes.c_float
        lib.norm_gate_fwd.restype = ctypes.c_int
        lib.norm_gate_fwd.argtypes = [P, P, P, I64, I64, I32, F, P, P]
        lib.norm_gate_bwd_workspace_size.restype = ctypes.c_size_t
        lib.norm_gate_bwd_workspace_size.argtypes = [I64, I64]
        lib.norm_gate_bwd.restype = ctypes.c_int
        lib.norm_gate_bwd.argtypes = [P, P, P, P, I64, I64, I32, F, P, P, P, P, ctypes.c_size_t, P]
        lib.short_conv_fwd.restype = ctypes.c_int
        lib.short_conv_fwd.argtypes = [P, P, P, P, I64, I64, I64, I32, I32, I32, P, P]
        lib.short_conv_bwd_workspace_size.restype = ctypes.c_size_t
        lib.short_conv_bwd_workspace_size.argtypes = [I64, I64, I64, I32]
        for n in ("gla_fwd_state",):
            getattr(lib, n).restype = ctypes.c_int
            getattr(lib, n).argtypes = [PP, P, P, P]
        lib.gla_bwd_state.restype = ctypes.c_int
        lib.gla_bwd_state.argtypes = [PP, P, P, P, P]
        lib.glacore_state_scan.restype = ctypes.c_int
        lib.glacore_state_scan.argtypes = [P, P, I64, I64, I64, I64, P, I64, I32, P, P]
        lib.short_conv_bwd.restype = ctypes.c_int
        lib.short_conv_bwd.argtypes = [P, P, P, P, P, I64, I64, I64, I32, I32, I32, P, P, P, P, ctypes.c_size_t, P]
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


def _rows(t):
    """(tensor, token stride): a [B, T, heads, D] tensor whose heads and
    channels are contiguous and whose tokens are evenly spaced (for example
    a slice of one fused projection [B, T, 3 * H * K]) is passed in place
    with its token stride; anything else is made contiguous (stride 0)."""
    if not t.is_cuda:
        raise ValueError("glacore takes CUDA tensors")
    if t.is_contiguous():
        return t, 0
    B, T, Hh, D = t.shape
    st = t.stride()
    if st[3] == 1 and st[2] == D and st[1] >= Hh * D and (B == 1 or st[0] == T * st[1]):
        return t, st[1]
    return t.contiguous(), 0


def _problem(q, k, v, g, scale, segment_ids, initial_state, chunk_size, n_seqs, head_gate):
    (q, qs), (k, ks), (v, vs) = _rows(q), _rows(k), _rows(v)
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
                workspace_bytes=0, q_stride=qs, k_stride=ks, v_stride=vs)
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


# ---- operations around the recurrence ---------------------------------------
def norm_gate_fwd(o, z, w, eps=1e-5, out=None):
    """Per-head RMSNorm times a swish gate over the last axis (V):
    y = o * rsqrt(mean(o^2) + eps) * w * z * sigmoid(z).  o, z [..., V]
    (bf16 or fp32, same dtype), w [V] fp32."""
    o, z = _contig(o), _contig(z)
    w = _contig(w, torch.float32)
    if o.shape != z.shape or o.dtype != z.dtype or tuple(w.shape) != (o.shape[-1],):
        raise ValueError("norm_gate: o and z must match and w must be [V]")
    V = o.shape[-1]
    rows = o.numel() // V if V else 0
    y = out if out is not None else torch.empty_like(o)
    st = load().norm_gate_fwd(_ptr(o), _ptr(z), _ptr(w), rows, V, _dtype_code(o), float(eps), _ptr(y),
                              _stream(o.device))
    _check(st, "norm_gate_fwd")
    return y


def norm_gate_bwd(o, z, w, dy, eps=1e-5, outs=None, workspace=None):
    """Returns (do, dz, dw) of norm_gate_fwd."""
    o, z, dy = _contig(o), _contig(z), _contig(dy)
    w = _contig(w, torch.float32)
    if not (o.shape == z.shape == dy.shape) or not (o.dtype == z.dtype == dy.dtype):
        raise ValueError("norm_gate: o, z and dy must match")
    V = o.shape[-1]
    rows = o.numel() // V if V else 0
    if outs is not None:
        do, dz, dw = outs
    else:
        do, dz = torch.empty_like(o), torch.empty_like(z)
        dw = torch.empty(V, dtype=torch.float32, device=o.device)
    lib = load()
    need = int(lib.norm_gate_bwd_workspace_size(rows, V))
    ws = workspace if workspace is not None and workspace.numel() >= need else torch.empty(
        max(need, 256), dtype=torch.uint8, device=o.device)
    st = lib.norm_gate_bwd(_ptr(o), _ptr(z), _ptr(w), _ptr(dy), rows, V, _dtype_code(o), float(eps), _ptr(do),
                           _ptr(dz), _ptr(dw), _ptr(ws), ws.numel(), _stream(o.device))
    _check(st, "norm_gate_bwd")
    return do, dz, dw


def short_conv_fwd(x, w, b=None, segment_ids=None, activation=True, out=None):
    """Depthwise causal short convolution (+ SiLU) of x [B,T,D]; w [Kc,D]
    fp32 (tap k reads x_{t-(Kc-1-k)}), b [D] fp32 or None, segment_ids
    [B,T] int32 or None."""
    x = _contig(x)
    w = _contig(w, torch.float32)
    b = _contig(b, torch.float32) if b is not None else None
    seg = _contig(segment_ids, torch.int32) if segment_ids is not None else None
    B, T, D = x.shape
    Kc = w.shape[0]
    if tuple(w.shape) != (Kc, D) or (b is not None and tuple(b.shape) != (D,)):
        raise ValueError("short_conv: w must be [Kc, D] and b [D]")
    y = out if out is not None else torch.empty_like(x)
    st = load().short_conv_fwd(_ptr(x), _ptr(w), _ptr(b), _ptr(seg), B, T, D, Kc, _dtype_code(x),
                               1 if activation else 0, _ptr(y), _stream(x.device))
    _check(st, "short_conv_fwd")
    return y


def short_conv_bwd(x, w, b, dy, segment_ids=None, activation=True, outs=None, workspace=None):
    """Returns (dx, dw, db) of short_conv_fwd (db also when b is None)."""
    x, dy = _contig(x), _contig(dy)
    w = _contig(w, torch.float32)
    b = _contig(b, torch.float32) if b is not None else None
    seg = _contig(segment_ids, torch.int32) if segment_ids is not None else None
    B, T, D = x.shape
    Kc = w.shape[0]
    if outs is not None:
        dx, dw, db = outs
    else:
        dx = torch.empty_like(x)
        dw = torch.empty(Kc, D, dtype=torch.float32, device=x.device)
        db = torch.empty(D, dtype=torch.float32, device=x.device)
    lib = load()
    need = int(lib.short_conv_bwd_workspace_size(B, T, D, Kc))
    ws = workspace if workspace is not None and workspace.numel() >= need else torch.empty(
        max(need, 256), dtype=torch.uint8, device=x.device)
    st = lib.short_conv_bwd(_ptr(x), _ptr(w), _ptr(b), _ptr(seg), _ptr(dy), B, T, D, Kc, _dtype_code(x),
                            1 if activation else 0, _ptr(dx), _ptr(dw), _ptr(db), _ptr(ws), ws.numel(),
                            _stream(x.device))
    _check(st, "short_conv_bwd")
    return dx, dw, db


# ---- sequence split across devices ------------------------------------------
def gla_fwd_state(q, k, v, g, scale=None):
    """Local end state (from a zero initial state) and total decay of every
    row: (L [B,H,K,V] fp32, D [B,H,K] fp32).  GLA, no segment_ids."""
    p, keep = _problem(q, k, v, g, scale, None, None, 0, None, False)
    dev = keep[0].device
    L = torch.empty((p.n_seqs, p.H, p.K, p.V), dtype=torch.float32, device=dev)
    D = torch.empty((p.n_seqs, p.H, p.K), dtype=torch.float32, device=dev)
    _check(load().gla_fwd_state(ctypes.byref(p), _ptr(L), _ptr(D), _stream(dev)), "gla_fwd_state")
    del keep
    return L, D


def gla_bwd_state(q, k, v, g, do, scale=None):
    """Local state gradient at the start of every row (from a zero gradient
    at its end) and total decay: (L [B,H,K,V] fp32, D [B,H,K] fp32)."""
    p, keep = _problem(q, k, v, g, scale, None, None, 0, None, False)
    dev = keep[0].device
    do = _contig(do, keep[0].dtype)
    L = torch.empty((p.n_seqs, p.H, p.K, p.V), dtype=torch.float32, device=dev)
    D = torch.empty((p.n_seqs, p.H, p.K), dtype=torch.float32, device=dev)
    _check(load().gla_bwd_state(ctypes.byref(p), _ptr(do), _ptr(L), _ptr(D), _stream(dev)), "gla_bwd_state")
    del keep
    return L, D


def state_scan(L, D, r, seed=None, reverse=False):
    """Fold of the stacked piece states L [R, *mats, K, V] / decays
    D [R, *mats, K] for piece r (forward: pieces before r; reverse: after r),
    starting from seed [*mats, K, V] (or zero)."""
    L = _contig(L, torch.float32)
    D = _contig(D, torch.float32)
    seed = _contig(seed, torch.float32) if seed is not None else None
    R, K, V = L.shape[0], L.shape[-2], L.shape[-1]
    mats = L[0].numel() // (K * V)
    out = torch.empty(L.shape[1:], dtype=torch.float32, device=L.device)
    _check(load().glacore_state_scan(_ptr(L), _ptr(D), R, mats, K, V, _ptr(seed), int(r), 1 if reverse else 0,
                                     _ptr(out), _stream(L.device)), "state_scan")
    return out
