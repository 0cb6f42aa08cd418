"""GPU parity at the workloads' full sizes, in the launch configuration the
bench times, element by element over every output.  The oracle runs the
whole workload (every batch row, document and head) in fp64 on the host
cores."""
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


def _run_full(w_index):
    """GPU fwd+bwd at full size; returns inputs and CPU copies of all outputs."""
    d = inputs.make(inputs.WORKLOADS[w_index])
    x = inputs.to_device(d, "cuda")
    w = d["workload"]
    fwd = glc.gla_fwd if w.kind == "gla" else glc.ssd_fwd
    bwd = glc.gla_bwd if w.kind == "gla" else glc.ssd_bwd
    glc.get_device_error()
    o, ht = fwd(x["q"], x["k"], x["v"], x["g"], d["scale"], x["segment_ids"], x["h0"], w.final_state, w.chunk,
                d["n_seqs"], poison=True)
    dq, dk, dv, dg, dh0 = bwd(x["q"], x["k"], x["v"], x["g"], x["do"], d["scale"], x["segment_ids"], x["h0"],
                              x["dht"], w.chunk, d["n_seqs"], poison=True)
    torch.cuda.synchronize()
    glc.get_device_error()
    out = dict(o=o, ht=ht, dq=dq, dk=dk, dv=dv, dg=dg, dh0=dh0)
    return d, {k: (v.cpu() if v is not None else None) for k, v in out.items()}


def _compare_all(w_index):
    d, out = _run_full(w_index)
    o, ht = oracle.fwd(d["q"], d["k"], d["v"], d["g"], d["scale"], d["segment_ids"], d["h0"])
    gr = oracle.bwd(d["q"], d["k"], d["v"], d["g"], d["do"], d["scale"], d["segment_ids"], d["h0"], d["dht"])
    ref = dict(o=o, dq=gr["dq"], dk=gr["dk"], dv=gr["dv"], dg=gr["dg"])
    if out["ht"] is not None:
        ref["ht"] = ht
    if out["dh0"] is not None:
        ref["dh0"] = gr["dh0"]
    errs = {}
    for n, want in ref.items():
        got = f64(out[n])
        assert got.shape == want.shape, n
        assert np.isfinite(got).all(), f"{n} has non-finite entries"
        errs[n] = rel(got, want)
    bad = {n: e for n, e in errs.items() if e > TOL[n]}
    print("rel errors:", {n: f"{e:.2e}" for n, e in errs.items()})
    assert not bad, (bad, errs)


def test_gla_bf16_B4_H16_T2048_every_head(cuda_ok):
    """Workload 2 (the bench workload): all 64 (row, head) recurrences."""
    _compare_all(2)


def test_ssd_B4_H32_T4096_every_row(cuda_ok):
    """Workload 3 (Mamba-2 SSD, one B/C group shared by 32 heads): all four
    rows and all heads (dq and dk sum over the heads that share C and B)."""
    _compare_all(3)


def test_packed_gla_B1_T16384_H16_every_head(cuda_ok):
    """Workload 4 (packed documents with per-document initial / final states)."""
    _compare_all(4)


def test_long_gla_B1_H16_T65536_every_head(cuda_ok):
    """Workload 5 (one row of 65536 tokens: the path splits it into pieces)."""
    _compare_all(5)


