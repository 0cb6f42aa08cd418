"""fp64 chunkwise restatement of the recurrence (test infrastructure only).

This is NOT the oracle: the oracle is the token-by-token recurrence in
``oracle.c``.  This module writes out, in double precision and with numpy,
the chunk formulas that a chunk-parallel implementation evaluates, so that
tests can check those formulas against the oracle at several chunk sizes
before any kernel relies on them.  It shares no code with the CUDA path.

Formulas (per document and head, chunk of positions a..e-1, G the inclusive
prefix sum of the log gate inside the chunk, Gam = G at the last position):

  FLAT blog, "Linear Attention / Forward Recurrence" (chunkwise form: causal
  intra-chunk product masked by the lower-triangular M_C with diagonal,
  plus the readout of the carried state) and "Mamba-2" / "Gated Linear
  Attention" (the decay ratios F_t/F_s are exponentiated chunk-local prefix
  sums of log f):

    qt = scale * q * exp(G)            kt = k * exp(-G)
    P  = (qt kt^T) masked to s <= t
    O  = qt S_prev + P V
    S  = diag(exp(Gam)) (S_prev + kt^T V)

  FLAT blog, "Backward Recurrence" and "Backward Kernels" (chunks visited in
  reverse, the state gradient carried across chunks, the gate gradient as a
  within-chunk suffix sum of q*dq - k*dk plus a boundary term from the state
  and state gradient at the chunk boundary):

    dP  = (dO V^T) masked             dHh = diag(exp(Gam)) dH
    dq  = scale * exp(G) * (dO S_prev^T + dP kt)
    dk  = exp(-G) * (dP^T qt + V dHh^T)
    dv  = P^T dO + kt dHh
    dg_t = sum_{r >= t in chunk} (q*dq - k*dk)_r + (S_end * dH) 1_V
    dH <- dHh + qt^T dO
"""
from __future__ import annotations

import numpy as np


def _docs(B, T, seg):
    out = []
    for b in range(B):
        t0 = 0
        for t in range(1, T + 1):
            if t == T or (seg is not None and seg[b, t] != seg[b, t - 1]):
                out.append((b, t0, t))
                t0 = t
    return out


def _gate(g, b, a, e, h, K):
    if g.ndim == 4:
        return g[b, a:e, h, :]
    return np.repeat(g[b, a:e, h][:, None], K, axis=1)


def forward(q, k, v, g, scale, chunk, segment_ids=None, h0=None, keep_states=False):
    B, T, Hqk, K = q.shape
    H, V = v.shape[2], v.shape[3]
    grp = H // Hqk
    docs = _docs(B, T, segment_ids)
    o = np.zeros((B, T, H, V))
    ht = np.zeros((len(docs), H, K, V))
    states = {}
    for d, (b, t0, t1) in enumerate(docs):
        for h in range(H):
            hk = h // grp
            S = np.zeros((K, V)) if h0 is None else h0[d, h].copy()
            for a in range(t0, t1, chunk):
                e = min(a + chunk, t1)
                if keep_states:
                    states[(d, h, a)] = S.copy()
                G = np.cumsum(_gate(g, b, a, e, h, K), axis=0)
                Gam = G[-1]
                qt = scale * q[b, a:e, hk] * np.exp(G)
                kt = k[b, a:e, hk] * np.exp(-G)
                P = np.tril(qt @ kt.T)
                o[b, a:e, h] = qt @ S + P @ v[b, a:e, h]
                S = np.exp(Gam)[:, None] * (S + kt.T @ v[b, a:e, h])
            ht[d, h] = S
    if keep_states:
        return o, ht, states, docs
    return o, ht


def backward(q, k, v, g, do, scale, chunk, segment_ids=None, h0=None, dht=None):
    B, T, Hqk, K = q.shape
    H, V = v.shape[2], v.shape[3]
    grp = H // Hqk
    _, ht, states, docs = forward(q, k, v, g, scale, chunk, segment_ids, h0, keep_states=True)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dgc = np.zeros((B, T, H, K))
    dh0 = np.zeros((len(docs), H, K, V))
    for d, (b, t0, t1) in enumerate(docs):
        for h in range(H):
            hk = h // grp
            dH = np.zeros((K, V)) if dht is None else dht[d, h].copy()
            S_end = ht[d, h]
            starts = list(range(t0, t1, chunk))
            for a in reversed(starts):
                e = min(a + chunk, t1)
                Sp = states[(d, h, a)]
                G = np.cumsum(_gate(g, b, a, e, h, K), axis=0)
                Gam = G[-1]
                qc, kc, vc, oc = q[b, a:e, hk], k[b, a:e, hk], v[b, a:e, h], do[b, a:e, h]
                qt = scale * qc * np.exp(G)
                kt = kc * np.exp(-G)
                P = np.tril(qt @ kt.T)
                dP = np.tril(oc @ vc.T)
                dHh = np.exp(Gam)[:, None] * dH
                dqc = scale * np.exp(G) * (oc @ Sp.T + dP @ kt)
                dkc = np.exp(-G) * (dP.T @ qt + vc @ dHh.T)
                dv[b, a:e, h] = P.T @ oc + kt @ dHh
                dq[b, a:e, hk] += dqc
                dk[b, a:e, hk] += dkc
                acc = qc * dqc - kc * dkc
                suffix = np.cumsum(acc[::-1], axis=0)[::-1]
                dgc[b, a:e, h] = suffix + (S_end * dH).sum(axis=1)[None, :]
                dH = dHh + qt.T @ oc
                S_end = Sp
            dh0[d, h] = dH
    dg = dgc if g.ndim == 4 else dgc.sum(axis=3)
    return {"dq": dq, "dk": dk, "dv": dv, "dg": dg, "dh0": dh0}
