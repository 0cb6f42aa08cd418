"""Strong decay on the GPU, against the fp64 oracle.

Inside a chunk the GLA kernels factor the decay between tokens t >= s as
exp(G_t) * exp(-G_s), with G the prefix sum of the log-decay from the chunk
start (FLAT blog, "Gated Linear Attention"; "Backward Kernels" names strong
decay as the method's precision edge).  The factors stay in the fp32 / bf16
exponent range while every chunk's summed log-decay in every channel is at
least -80.  The SSD kernels need no such bound: with one decay per head
they apply exp(G_t - G_s) (s <= t) as one factor or as a product of
factors that are each at most 1 (FLAT blog, "Mamba-2"), so Mamba-2 gates
of any strength run forward and backward on the tensor cores.  These tests check the sides of the bound:

- inside it, with decay far stronger than the workloads' (GLA's gate without
  its 1/16 normaliser, per-chunk sums near -52), the tensor-core kernels
  match the oracle;
- past it (a constant log-decay of -3 per token, Mamba-2 gates near -2 per
  token, per-chunk sums of -200 to -300), the tensor-core kernels report
  GLACORE_ERR_RANGE instead of returning wrong numbers, also when the
  sequence is split into pieces and when documents are packed;
- the same inputs run with chunk_size 16 (the CUDA-core kernels, whose
  16-token chunks keep the factors in range down to -80 per 16 tokens)
  match the oracle, plain, packed and with initial / final states.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import chunked_gated_linear_chunk_gb300 as glc
import oracle
from chunked_gated_linear_chunk_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = dict(o=5e-3, ht=5e-3, dq=2e-2, dk=2e-2, dv=2e-2, dg=2e-2, dh0=2e-2)


def rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30)) if b.size else 0.0


def np64(t):
    return None if t is None else t.detach().to("cpu", torch.float64).numpy()


def gate(d, kind, seed):
    """Replaces the workload's gate by a strong one of the same shape."""
    gen = torch.Generator("cpu")
    gen.manual_seed(seed)
    shape = d["g"].shape
    if kind == "logsigmoid":  # GLA gate without the 1/16 normaliser
        g = F.logsigmoid(torch.randn(shape, generator=gen))
    elif kind == "const3":  # -3 per token: -192 per 64-token chunk
        g = torch.full(shape, -3.0)
    elif kind == "sum200_300":  # per-token -3.1 .. -4.7: chunk sums -200 .. -300
        g = -(200.0 + 100.0 * torch.rand(shape, generator=gen)) / 64.0
    elif kind == "ssd2":  # Mamba-2 gate near -2 per token (dt * A with large dt)
        g = -2.0 * (1.0 + 0.25 * torch.randn(shape, generator=gen)).clamp(min=0.25)
    else:
        raise ValueError(kind)
    out = dict(d)
    out["g"] = g.float()
    return out


def run_gpu(d, chunk):
    w = d["workload"]
    x = inputs.to_device(d, "cuda")
    fwd = glc.gla_fwd if w.kind == "gla" else glc.ssd_fwd
    bwd = glc.gla_bwd if w.kind == "gla" else glc.ssd_bwd
    glc.get_device_error()
    o, ht = fwd(x["q"], x["k"], x["v"], x["g"], d["scale"], x["segment_ids"], x["h0"], True, chunk, d["n_seqs"],
                poison=True)
    dq, dk, dv, dg, dh0 = bwd(x["q"], x["k"], x["v"], x["g"], x["do"], d["scale"], x["segment_ids"], x["h0"],
                              x["dht"], chunk, d["n_seqs"], poison=True)
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


def compare(gpu, ref):
    errs = {}
    for n, want in ref.items():
        if want is None or gpu.get(n) is None:
            continue
        assert np.isfinite(gpu[n]).all(), f"{n} has non-finite entries"
        errs[n] = rel(gpu[n], want)
    bad = {n: e for n, e in errs.items() if e > TOL[n]}
    print("rel errors:", {n: f"{e:.2e}" for n, e in errs.items()})
    assert not bad, f"over tolerance: {bad} (all: {errs})"


def case(base, seed, **over):
    return inputs.make(inputs.WORKLOADS[base], seed=seed, **over)


# inside the tensor-core range: GLA without the 1/16 gate normaliser
INSIDE = {
    "gla_T300_H2": lambda: gate(case(5, 41, B=2, T=300, H=2, Hqk=2), "logsigmoid", 1),
    "gla_packed": lambda: gate(case(4, 42, B=2, T=300, H=2, Hqk=2, doc_mean=50), "logsigmoid", 2),
    "gla_pieces_T2000": lambda: gate(case(5, 43, B=1, T=2000, H=1, Hqk=1), "logsigmoid", 3),
    "gla_pieces_packed": lambda: gate(case(4, 44, B=1, T=3000, H=1, Hqk=1, doc_mean=700), "logsigmoid", 4),
}


@pytest.mark.parametrize("name", sorted(INSIDE))
def test_unnormalised_gla_gate_on_tensor_cores(cuda_ok, name):
    d = INSIDE[name]()
    compare(run_gpu(d, 0), run_oracle(d))


# past the tensor-core range
PAST = {
    "gla_const3": lambda: gate(case(5, 51, B=1, T=200, H=2, Hqk=2), "const3", 0),
    "gla_sum200_300": lambda: gate(case(5, 52, B=2, T=150, H=2, Hqk=2), "sum200_300", 5),
    "gla_sum200_300_packed": lambda: gate(case(4, 53, B=2, T=300, H=2, Hqk=2, doc_mean=60), "sum200_300", 6),
    "gla_const3_pieces": lambda: gate(case(5, 54, B=1, T=2000, H=1, Hqk=1), "const3", 0),
    "gla_sum200_300_pieces_packed": lambda: gate(case(4, 55, B=1, T=3000, H=1, Hqk=1, doc_mean=700),
                                                 "sum200_300", 7),
}
# Mamba-2 gates past the GLA kernels' range
SSD_STRONG = {
    "ssd_g2": lambda: gate(case(3, 56, B=1, T=200, H=4), "ssd2", 8),
    "ssd_g2_packed": lambda: gate(case(3, 57, B=2, T=150, H=4, packed=True, doc_mean=40, initial_state=True,
                                       final_state=True), "ssd2", 9),
    "ssd_sum200_300": lambda: gate(case(3, 58, B=1, T=2000, H=2), "sum200_300", 10),
}


@pytest.mark.parametrize("name", sorted(PAST))
def test_decay_past_the_tensor_core_range_is_reported(cuda_ok, name):
    d = PAST[name]()
    w = d["workload"]
    x = inputs.to_device(d, "cuda")
    fwd = glc.gla_fwd if w.kind == "gla" else glc.ssd_fwd
    bwd = glc.gla_bwd if w.kind == "gla" else glc.ssd_bwd
    glc.get_device_error()
    fwd(x["q"], x["k"], x["v"], x["g"], d["scale"], x["segment_ids"], x["h0"], True, 0, d["n_seqs"])
    torch.cuda.synchronize()
    with pytest.raises(glc.GlacoreError) as e:
        glc.get_device_error()
    assert e.value.status == glc.ERR_RANGE
    bwd(x["q"], x["k"], x["v"], x["g"], x["do"], d["scale"], x["segment_ids"], x["h0"], x["dht"], 0, d["n_seqs"])
    torch.cuda.synchronize()
    with pytest.raises(glc.GlacoreError) as e:
        glc.get_device_error()
    assert e.value.status == glc.ERR_RANGE
    glc.get_device_error()  # cleared


@pytest.mark.parametrize("name", sorted(SSD_STRONG))
def test_ssd_strong_decay_on_tensor_cores(cuda_ok, name):
    d = SSD_STRONG[name]()
    compare(run_gpu(d, 0), run_oracle(d))


@pytest.mark.parametrize("name", sorted(PAST) + sorted(SSD_STRONG))
def test_decay_past_the_tensor_core_range_with_chunk_16(cuda_ok, name):
    d = (PAST.get(name) or SSD_STRONG[name])()
    compare(run_gpu(d, 16), run_oracle(d))


def test_chunk_16_reports_decay_past_its_own_range(cuda_ok):
    """-6 per token is -96 per 16-token chunk: past the CUDA-core range too."""
    d = case(5, 59, B=1, T=64, H=1, Hqk=1)
    d["g"] = torch.full_like(d["g"], -6.0)
    x = inputs.to_device(d, "cuda")
    glc.get_device_error()
    glc.gla_fwd(x["q"], x["k"], x["v"], x["g"], d["scale"], None, x["h0"], True, 16)
    torch.cuda.synchronize()
    with pytest.raises(glc.GlacoreError) as e:
        glc.get_device_error()
    assert e.value.status == glc.ERR_RANGE
