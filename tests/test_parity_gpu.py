"""GPU parity: the CUDA path against the fp64 oracle, element by element.

Metric (per output tensor): max|gpu - oracle| / max|oracle|.
Tolerances: fp32 inputs 1e-4 on every output; bf16 inputs 5e-3 on o and
final_state and 2e-2 on dq, dk, dv, dg, dh0.  Outputs are NaN-poisoned
before each call, so an element the kernels never write fails the test.
"""
import numpy as np
import pytest
import torch

import chunked_gated_linear_chunk_gb300 as glc
import oracle
from chunked_gated_linear_chunk_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = {
    "fp32": dict(o=1e-4, ht=1e-4, dq=1e-4, dk=1e-4, dv=1e-4, dg=1e-4, dh0=1e-4),
    "bf16": dict(o=5e-3, ht=5e-3, dq=2e-2, dk=2e-2, dv=2e-2, dg=2e-2, dh0=2e-2),
}


def rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30)) if b.size else 0.0


def np64(t):
    return None if t is None else t.detach().to("cpu", torch.float64).numpy()


def run_gpu(d, chunk=0):
    w = d["workload"]
    x = inputs.to_device(d, "cuda")
    fwd = glc.gla_fwd if w.kind == "gla" else glc.ssd_fwd
    bwd = glc.gla_bwd if w.kind == "gla" else glc.ssd_bwd
    o, ht = fwd(x["q"], x["k"], x["v"], x["g"], d["scale"], x["segment_ids"], x["h0"], True, chunk,
                d["n_seqs"], poison=True)
    dq, dk, dv, dg, dh0 = bwd(x["q"], x["k"], x["v"], x["g"], x["do"], d["scale"], x["segment_ids"],
                              x["h0"], x["dht"], chunk, d["n_seqs"], poison=True)
    torch.cuda.synchronize()
    glc.get_device_error()
    return dict(o=np64(o), ht=np64(ht), dq=np64(dq), dk=np64(dk), dv=np64(dv), dg=np64(dg), dh0=np64(dh0))


def run_oracle(d):
    o, ht = oracle.fwd(d["q"], d["k"], d["v"], d["g"], d["scale"], d["segment_ids"], d["h0"])
    gr = oracle.bwd(d["q"], d["k"], d["v"], d["g"], d["do"], d["scale"], d["segment_ids"], d["h0"], d["dht"])
    out = dict(o=o, ht=ht, **gr)
    if d["h0"] is None:
        out["dh0"] = None
    return out


def compare(gpu, ref, dtype, names=("o", "ht", "dq", "dk", "dv", "dg", "dh0")):
    errs = {}
    for n in names:
        if ref.get(n) is None or gpu.get(n) is None:
            continue
        assert gpu[n].shape == ref[n].shape, n
        assert np.isfinite(gpu[n]).all(), f"{n} has non-finite entries"
        errs[n] = rel(gpu[n], ref[n])
    bad = {n: e for n, e in errs.items() if e > TOL[dtype][n]}
    assert not bad, f"over tolerance: {bad} (all: {errs})"
    return errs


def case(base, seed, **over):
    return inputs.make(inputs.WORKLOADS[base], seed=seed, **over)


SMALL = {
    "cfg1_tiny_fp32": lambda: inputs.make(inputs.WORKLOADS[1]),
    "gla_bf16_T200_H2": lambda: case(2, 1, B=2, T=200, H=2, Hqk=2),
    "gla_bf16_T200_h0_dht": lambda: case(5, 2, B=2, T=200, H=2, Hqk=2),
    "gla_bf16_T1": lambda: case(5, 3, B=1, T=1, H=1, Hqk=1),
    "gla_bf16_T63": lambda: case(5, 4, B=1, T=63, H=1, Hqk=1),
    "gla_bf16_T65": lambda: case(5, 5, B=1, T=65, H=1, Hqk=1),
    "gla_bf16_packed": lambda: case(4, 6, B=2, T=300, H=2, Hqk=2, doc_mean=40),
    "ssd_bf16_T200": lambda: case(3, 7, B=1, T=200, H=4),
    "ssd_bf16_packed": lambda: case(3, 8, B=2, T=150, H=4, packed=True, doc_mean=30, initial_state=True,
                                    final_state=True),
    "gla_fp32_K64_V32": lambda: case(1, 9, B=1, T=70, H=2, Hqk=2, K=64, V=32),
    "gla_bf16_K64_V64": lambda: case(2, 10, B=1, T=130, H=2, Hqk=2, K=64, V=64),
    # one (document, head) pair: the tensor-core path splits it into pieces
    "gla_bf16_pieces_T2000": lambda: case(5, 13, B=1, T=2000, H=1, Hqk=1),
    "gla_bf16_pieces_T1000_nostate": lambda: case(2, 14, B=1, T=1000, H=1, Hqk=1),
    "gla_bf16_pieces_packed": lambda: case(4, 15, B=1, T=3000, H=1, Hqk=1, doc_mean=700),
    "gla_bf16_pieces_B2_H2": lambda: case(5, 16, B=2, T=1500, H=2, Hqk=2),
    # SSD (V = 64: its own kernels, one CTA per document and head): a long
    # document on two heads of one B / C group
    "ssd_bf16_T2000": lambda: case(3, 17, B=1, T=2000, H=2),
    # every head its own B / C, both states
    "ssd_bf16_own_bc_h0_dht": lambda: case(3, 20, B=2, T=130, H=4, Hqk=4, initial_state=True,
                                           final_state=True),
    # two B / C groups of two heads, a length past a chunk boundary
    "ssd_bf16_groups2_T257": lambda: case(3, 21, B=1, T=257, H=4, Hqk=2, final_state=True),
    # many short packed documents (most shorter than one 16-token block)
    "ssd_bf16_short_docs": lambda: case(3, 22, B=2, T=200, H=2, packed=True, doc_mean=10, initial_state=True,
                                        final_state=True),
    # SSD with V = 128 (the GLA tensor-core kernels in their per-head-gate
    # mode, both value halves stored) and two B / C groups
    "ssd_bf16_V128_groups2": lambda: case(3, 18, B=1, T=200, H=4, Hqk=2, V=128),
    # SSD with V < 64: the fp32 CUDA-core kernels
    "ssd_bf16_V32": lambda: case(3, 19, B=1, T=130, H=2, V=32),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_cases_against_oracle(cuda_ok, name):
    d = SMALL[name]()
    gpu = run_gpu(d)
    ref = run_oracle(d)
    compare(gpu, ref, d["workload"].dtype)


@pytest.mark.parametrize("chunk", [16, 32, 64])
def test_chunk_size_does_not_change_results_fp32(cuda_ok, chunk):
    """One kernel family (the fp32 CUDA-core kernels) at three chunk lengths,
    each against the oracle at the fp32 tolerance: documents that start
    mid-chunk, a ragged tail and initial / final states."""
    d = case(4, 11, B=2, T=150, H=2, Hqk=2, K=64, V=64, dtype="fp32", doc_mean=40)
    compare(run_gpu(d, chunk=chunk), run_oracle(d), "fp32")


@pytest.mark.parametrize("chunk", [16, 64])
def test_chunk_size_does_not_change_results_bf16(cuda_ok, chunk):
    """The same bf16 problem at chunk 64 (tensor-core kernels) and chunk 16
    (CUDA-core kernels), each against the oracle."""
    d = case(5, 11, B=1, T=300, H=2, Hqk=2)
    compare(run_gpu(d, chunk=chunk), run_oracle(d), "bf16")


def test_empty_sequence(cuda_ok):
    q = torch.zeros(2, 0, 1, 128, dtype=torch.bfloat16, device="cuda")
    g = torch.zeros(2, 0, 1, 128, device="cuda")
    o, ht = glc.gla_fwd(q, q, q, g, output_final_state=True)
    assert o.shape == (2, 0, 1, 128) and ht.shape == (0, 1, 128, 128)


def test_document_count_mismatch_sets_device_error(cuda_ok):
    d = case(4, 12, B=1, T=100, H=1, Hqk=1, doc_mean=20)
    x = inputs.to_device(d, "cuda")
    n = glc.count_docs(x["segment_ids"])
    assert n == d["n_seqs"]
    glc.get_device_error()  # clear
    glc.gla_fwd(x["q"], x["k"], x["v"], x["g"], d["scale"], x["segment_ids"], None, False, 64, n + 1)
    torch.cuda.synchronize()
    with pytest.raises(glc.GlacoreError) as e:
        glc.get_device_error()
    assert e.value.status == glc.ERR_DOCS
    glc.get_device_error()  # cleared
