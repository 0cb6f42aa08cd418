"""gla_bwd_noalloc (the backward that takes no workspace) against gla_bwd.

For callers that cannot allocate device memory at call time: the entry point
uses a fixed device array as scratch.  It is checked through the C ABI
against the ordinary entry point on two calls in a row, each on a different
problem (another seed, length, document split and head count), so the second
call starts from scratch that holds the first call's values and must not
depend on them.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import chunked_gated_linear_chunk_gb300 as glc
from chunked_gated_linear_chunk_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = dict(dq=2e-2, dk=2e-2, dv=2e-2, dg=2e-2, dh0=2e-2)


def rel(a, b):
    a = a.detach().to("cpu", torch.float64).numpy()
    b = b.detach().to("cpu", torch.float64).numpy()
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


def _check_noalloc_against_gla_bwd(lib, d):
    x = inputs.to_device(d, "cuda")
    ref = glc.gla_bwd(x["q"], x["k"], x["v"], x["g"], x["do"], d["scale"], x["segment_ids"], x["h0"],
                      x["dht"], n_seqs=d["n_seqs"])
    torch.cuda.synchronize()
    glc.get_device_error()
    p, keep = glc._problem(x["q"], x["k"], x["v"], x["g"], d["scale"], x["segment_ids"], x["h0"], 0,
                           d["n_seqs"], False)
    assert 0 < glc.workspace_size(p, "gla_bwd") <= (48 << 20)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    outs = [torch.full_like(t, float("nan")) if t is not None else None for t in ref]
    dq, dk, dv, dg, dh0 = outs
    st = lib.gla_bwd_noalloc(ctypes.byref(p), glc._ptr(x["do"]), glc._ptr(x["dht"]), glc._ptr(dq),
                             glc._ptr(dk), glc._ptr(dv), glc._ptr(dg), glc._ptr(dh0), stream)
    assert st == glc.OK, st
    torch.cuda.synchronize()
    glc.get_device_error()
    for name, got, want in zip(("dq", "dk", "dv", "dg", "dh0"), outs, ref):
        if want is None:
            continue
        assert torch.isfinite(got.float()).all(), name
        assert rel(got, want) <= TOL[name], (name, rel(got, want))
    del keep


def test_noalloc_backward_matches_gla_bwd_on_two_calls(cuda_ok):
    lib = glc.load()
    # first call: packed documents, two heads; second call: a different
    # packing, length, seed and head count, started on the first call's scratch
    first = inputs.make(inputs.WORKLOADS[4], seed=30, B=1, T=333, H=3, Hqk=3, doc_mean=90)
    second = inputs.make(inputs.WORKLOADS[4], seed=31, B=2, T=200, H=2, Hqk=2, doc_mean=60)
    _check_noalloc_against_gla_bwd(lib, first)
    _check_noalloc_against_gla_bwd(lib, second)


def test_noalloc_backward_rejects_problems_beyond_its_scratch(cuda_ok):
    lib = glc.load()
    # B4 T4096 H16 K=V=128 bf16 needs ~134 MB of scratch (more than the array)
    p = glc.Problem(B=4, T=4096, H=16, Hqk=16, K=128, V=128, dtype=glc.BF16, chunk_size=64, scale=0.1,
                    reserved0=0, q=256, k=512, v=768, g=1024, segment_ids=None, n_seqs=4, initial_state=None,
                    workspace=None, workspace_bytes=0)
    assert glc.workspace_size(p, "gla_bwd") > (48 << 20)
    o = ctypes.c_void_p(4096)
    st = lib.gla_bwd_noalloc(ctypes.byref(p), o, None, o, o, o, o, None, None)
    assert st == glc.ERR_WORKSPACE
