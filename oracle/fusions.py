"""fp64 CPU oracle of the two operations around the recurrence (test
infrastructure: only tests/, __graft_entry__.smoke() and bench.py's CPU
baseline may import it; it shares no code with the CUDA path).

norm_gate -- per-head RMSNorm times a swish output gate (FLAT blog,
    trainstation-project.github.io/blog/flat, "Full Linear Attention Layer":
    the layer's output passes a per-head RMSNorm multiplied by a swish output
    gate; FLA documentation, "Norm Layers with Gating": norm layers combined
    with element-wise swish gating, as used by GLA).  Over each row of V
    values (one token and head):
        n = o / sqrt(mean(o^2) + eps),   y = n * w * z * sigmoid(z).
    The backward is derived by hand below.  Pinned in tests/test_fusions.py
    (closed forms for a constant row and for z = 0, scale invariance, central
    finite differences of every gradient).

short_conv -- depthwise causal short convolution with bias and SiLU (FLAT
    blog, "Depthwise Causal Short Convolution"): with taps W_k (k = 0..Kc-1,
    one weight per channel), tap k reads the input Kc-1-k steps back,
        z_t = b + sum_k W_k * x_{t-(Kc-1-k)},   y_t = SiLU(z_t) = z_t * sigmoid(z_t),
    inputs before the start of the token's document (row start, or a change
    of segment id) read as zero.  Backward as the page states it: dz = dy *
    SiLU'(z) with SiLU'(z) = sigmoid(z) (1 + z (1 - sigmoid(z))); dW_k and db
    are dz times the input that tap reads, reduced over every position; dx is
    the anti-causal correlation of dz with the same taps.  Pinned in
    tests/test_fusions.py (single-tap closed forms, packed documents equal to
    separate runs, central finite differences).
"""
from __future__ import annotations

import numpy as np


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):
        import torch

        a = a.detach().to("cpu", torch.float64).numpy()
    return np.asarray(a, dtype=np.float64)


def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


# ------------------------------------------------------------ norm_gate ----
def norm_gate_fwd(o, z, w, eps):
    """o, z: [..., V]; w: [V].  Returns y [..., V] in float64."""
    o, z, w = _f64(o), _f64(z), _f64(w)
    V = o.shape[-1]
    ms = np.sum(o * o, axis=-1, keepdims=True) / V
    r = 1.0 / np.sqrt(ms + eps)
    n = o * r
    return n * w * (z * _sigmoid(z))


def norm_gate_bwd(o, z, w, dy, eps):
    """Returns (do, dz, dw) in float64 for y = norm_gate_fwd(o, z, w, eps).

    With r = (mean(o^2) + eps)^-1/2, n = o r, u = n w, s = sigmoid(z), g = z s:
      dz = dy u s (1 + z (1 - s))         (derivative of z sigmoid(z))
      dw = sum over rows of dy g n
      dn = dy g w,   do = r dn - r^3 o (dn . o) / V   (derivative of o r)
    """
    o, z, w, dy = _f64(o), _f64(z), _f64(w), _f64(dy)
    V = o.shape[-1]
    ms = np.sum(o * o, axis=-1, keepdims=True) / V
    r = 1.0 / np.sqrt(ms + eps)
    n = o * r
    s = _sigmoid(z)
    g = z * s
    u = n * w
    dz = dy * u * s * (1.0 + z * (1.0 - s))
    dw = np.sum((dy * g * n).reshape(-1, V), axis=0)
    dn = dy * g * w
    dot = np.sum(dn * o, axis=-1, keepdims=True)
    do = r * dn - (r ** 3) * o * dot / V
    return do, dz, dw


# ----------------------------------------------------------- short_conv ----
def _doc_starts(B, T, segment_ids):
    """Boolean [B, T]: True where a document starts (t = 0 or an id change)."""
    start = np.zeros((B, T), dtype=bool)
    if T:
        start[:, 0] = True
    if segment_ids is not None:
        seg = np.asarray(segment_ids)
        start[:, 1:] |= seg[:, 1:] != seg[:, :-1]
    return start


def _shifted(x, start, j):
    """x_{t-j} within the token's document, else 0 ([B, T, D])."""
    B, T, D = x.shape
    out = np.zeros_like(x)
    for b in range(B):
        doc_begin = 0
        for t in range(T):
            if start[b, t]:
                doc_begin = t
            if t - j >= doc_begin:
                out[b, t] = x[b, t - j]
    return out


def short_conv_fwd(x, w, b, segment_ids=None, activation=True):
    """x [B, T, D]; w [Kc, D] (tap k reads x_{t-(Kc-1-k)}); b [D] or None.
    Returns y [B, T, D] in float64 (SiLU applied when activation)."""
    x, w = _f64(x), _f64(w)
    B, T, D = x.shape
    Kc = w.shape[0]
    start = _doc_starts(B, T, None if segment_ids is None else _f64(segment_ids))
    z = np.zeros_like(x) if b is None else np.broadcast_to(_f64(b), x.shape).copy()
    for k in range(Kc):
        z += w[k] * _shifted(x, start, Kc - 1 - k)
    return z * _sigmoid(z) if activation else z


def short_conv_bwd(x, w, b, dy, segment_ids=None, activation=True):
    """Returns (dx, dw, db) in float64."""
    x, w, dy = _f64(x), _f64(w), _f64(dy)
    B, T, D = x.shape
    Kc = w.shape[0]
    start = _doc_starts(B, T, None if segment_ids is None else _f64(segment_ids))
    shifted = [_shifted(x, start, Kc - 1 - k) for k in range(Kc)]
    z = np.zeros_like(x) if b is None else np.broadcast_to(_f64(b), x.shape).copy()
    for k in range(Kc):
        z += w[k] * shifted[k]
    if activation:
        s = _sigmoid(z)
        dz = dy * s * (1.0 + z * (1.0 - s))
    else:
        dz = dy
    dw = np.stack([np.sum((shifted[k] * dz).reshape(-1, D), axis=0) for k in range(Kc)])
    db = np.sum(dz.reshape(-1, D), axis=0)
    # adjoint of the shift inside documents: dx_t += W_k dz_{t+j}, j = Kc-1-k,
    # for t + j in the same document as t
    dx = np.zeros_like(x)
    for bb in range(B):
        doc_end = T
        for t in range(T - 1, -1, -1):
            if t + 1 < T and start[bb, t + 1]:
                doc_end = t + 1
            for k in range(Kc):
                j = Kc - 1 - k
                if t + j < doc_end:
                    dx[bb, t] += w[k] * dz[bb, t + j]
    return dx, dw, db
