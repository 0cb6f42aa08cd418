"""GPU parity at the workloads' full sizes, in the launch configuration the
bench times.  The oracle is run on sampled (document, head) pairs only: every
(document, head) of GLA is an independent recurrence, so the oracle on a
slice of the inputs gives the exact expected outputs of that slice."""
import numpy as np
import pytest
import torch

import chunked_gated_linear_chunk_gb300 as glc
import oracle
from chunked_gated_linear_chunk_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = dict(o=5e-3, ht=5e-3, dq=2e-2, dk=2e-2, dv=2e-2, dg=2e-2, dh0=2e-2)


def rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


@pytest.fixture(scope="module")
def cfg2():
    d = inputs.make(inputs.WORKLOADS[2])
    x = inputs.to_device(d, "cuda")
    o, _ = glc.gla_fwd(x["q"], x["k"], x["v"], x["g"], d["scale"], poison=True)
    dq, dk, dv, dg, _ = glc.gla_bwd(x["q"], x["k"], x["v"], x["g"], x["do"], d["scale"], poison=True)
    torch.cuda.synchronize()
    glc.get_device_error()
    return d, dict(o=o.cpu(), dq=dq.cpu(), dk=dk.cpu(), dv=dv.cpu(), dg=dg.cpu())


@pytest.mark.parametrize("b,h", [(0, 0), (3, 15), (2, 7)])
def test_gla_bf16_B4_H16_T2048_sampled_heads(cuda_ok, cfg2, b, h):
    d, out = cfg2
    sl = lambda t: t[b:b + 1, :, h:h + 1]
    o, _ = oracle.fwd(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["g"]), d["scale"])
    gr = oracle.bwd(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["g"]), sl(d["do"]), d["scale"])
    errs = dict(o=rel(f64(sl(out["o"])), o))
    for n in ("dq", "dk", "dv", "dg"):
        errs[n] = rel(f64(sl(out[n])), gr[n])
    bad = {n: e for n, e in errs.items() if e > TOL[n]}
    print("rel errors:", {n: f"{e:.2e}" for n, e in errs.items()})
    assert not bad, (bad, errs)


def test_gla_bf16_B4_H16_T2048_all_finite(cuda_ok, cfg2):
    _, out = cfg2
    for n, t in out.items():
        assert torch.isfinite(t.float()).all(), n


def _run_full(w_index, oracle_rows_heads):
    """GPU fwd+bwd at full size; returns inputs and CPU copies of all outputs."""
    d = inputs.make(inputs.WORKLOADS[w_index])
    x = inputs.to_device(d, "cuda")
    w = d["workload"]
    fwd = glc.gla_fwd if w.kind == "gla" else glc.ssd_fwd
    bwd = glc.gla_bwd if w.kind == "gla" else glc.ssd_bwd
    o, ht = fwd(x["q"], x["k"], x["v"], x["g"], d["scale"], x["segment_ids"], x["h0"], True, 64, d["n_seqs"],
                poison=True)
    dq, dk, dv, dg, dh0 = bwd(x["q"], x["k"], x["v"], x["g"], x["do"], d["scale"], x["segment_ids"], x["h0"],
                              x["dht"], 64, d["n_seqs"], poison=True)
    torch.cuda.synchronize()
    glc.get_device_error()
    out = dict(o=o, ht=ht, dq=dq, dk=dk, dv=dv, dg=dg, dh0=dh0)
    return d, {k: (v.cpu() if v is not None else None) for k, v in out.items()}


@pytest.mark.parametrize("h", [0, 11])
def test_long_gla_B1_H16_T65536_sampled_heads(cuda_ok, h):
    """Workload 5 (one row of 65536 tokens: the path splits it into pieces)."""
    d, out = _cached(5)
    sl = lambda t: t[:, :, h:h + 1]
    o, ht = oracle.fwd(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["g"]), d["scale"], None, d["h0"][:, h:h + 1])
    gr = oracle.bwd(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["g"]), sl(d["do"]), d["scale"], None,
                    d["h0"][:, h:h + 1], d["dht"][:, h:h + 1])
    errs = dict(o=rel(f64(sl(out["o"])), o), ht=rel(f64(out["ht"][:, h:h + 1]), ht))
    for n in ("dq", "dk", "dv", "dg"):
        errs[n] = rel(f64(sl(out[n])), gr[n])
    errs["dh0"] = rel(f64(out["dh0"][:, h:h + 1]), gr["dh0"])
    bad = {n: e for n, e in errs.items() if e > TOL[n]}
    print("rel errors:", {n: f"{e:.2e}" for n, e in errs.items()})
    assert not bad, (bad, errs)


@pytest.mark.parametrize("h", [3])
def test_packed_gla_B1_T16384_H16_sampled_head(cuda_ok, h):
    """Workload 4 (packed documents with per-document initial / final states)."""
    d, out = _cached(4)
    sl = lambda t: t[:, :, h:h + 1]
    seg = d["segment_ids"]
    o, ht = oracle.fwd(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["g"]), d["scale"], seg, d["h0"][:, h:h + 1])
    gr = oracle.bwd(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["g"]), sl(d["do"]), d["scale"], seg,
                    d["h0"][:, h:h + 1], d["dht"][:, h:h + 1])
    errs = dict(o=rel(f64(sl(out["o"])), o), ht=rel(f64(out["ht"][:, h:h + 1]), ht))
    for n in ("dq", "dk", "dv", "dg"):
        errs[n] = rel(f64(sl(out[n])), gr[n])
    errs["dh0"] = rel(f64(out["dh0"][:, h:h + 1]), gr["dh0"])
    bad = {n: e for n, e in errs.items() if e > TOL[n]}
    print("rel errors:", {n: f"{e:.2e}" for n, e in errs.items()})
    assert not bad, (bad, errs)


def test_ssd_B4_H32_T4096_sampled_row(cuda_ok):
    """Workload 3 (Mamba-2 SSD, one B/C group shared by 32 heads): batch row 2,
    all heads (dq and dk sum over the heads that share C and B)."""
    d, out = _cached(3)
    b = 2
    sl = lambda t: t[b:b + 1]
    o, _ = oracle.fwd(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["g"]), d["scale"])
    gr = oracle.bwd(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["g"]), sl(d["do"]), d["scale"])
    errs = dict(o=rel(f64(sl(out["o"])), o))
    for n in ("dq", "dk", "dv", "dg"):
        errs[n] = rel(f64(sl(out[n])), gr[n])
    bad = {n: e for n, e in errs.items() if e > TOL[n]}
    print("rel errors:", {n: f"{e:.2e}" for n, e in errs.items()})
    assert not bad, (bad, errs)


_CACHE = {}


def _cached(w_index):
    if w_index not in _CACHE:
        _CACHE.clear()
        _CACHE[w_index] = _run_full(w_index, None)
    return _CACHE[w_index]
