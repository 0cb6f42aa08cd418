"""Head sharing and fused-projection inputs on the GPU, against the oracle.

- q, k and v read in place from one fused projection [B, T, 2 Hqk K + H V]
  (token strides in the problem; no copy on the device), on the tensor-core
  and the CUDA-core kernels;
- GLA with shared q / k heads (H / Hqk = 4, a per-value-head gate): dq and
  dk are summed over the heads of a group (FLAT blog, "Gated Linear
  Attention": queries, keys, values and the gate may use different head
  counts)."""
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


def fused_views(d, device):
    """One projection tensor [B, T, Hqk K + Hqk K + H V] holding q, k, v; the
    returned q, k, v are strided views of it."""
    q, k, v = d["q"], d["k"], d["v"]
    B, T, Hqk, K = q.shape
    H, V = v.shape[2], v.shape[3]
    proj = torch.cat([q.reshape(B, T, -1), k.reshape(B, T, -1), v.reshape(B, T, -1)], dim=-1).to(device)
    qv = proj[:, :, :Hqk * K].view(B, T, Hqk, K) if False else proj[:, :, :Hqk * K].unflatten(2, (Hqk, K))
    kv = proj[:, :, Hqk * K:2 * Hqk * K].unflatten(2, (Hqk, K))
    vv = proj[:, :, 2 * Hqk * K:].unflatten(2, (H, V))
    assert not qv.is_contiguous() and qv.stride(1) == proj.shape[2]
    return proj, qv, kv, vv


def run(d, strided, chunk=0):
    x = inputs.to_device(d, "cuda")
    if strided:
        proj, q, k, v = fused_views(d, "cuda")
    else:
        q, k, v = x["q"], x["k"], x["v"]
    w = d["workload"]
    fwd = glc.gla_fwd if w.kind == "gla" else glc.ssd_fwd
    bwd = glc.gla_bwd if w.kind == "gla" else glc.ssd_bwd
    glc.get_device_error()
    o, ht = fwd(q, k, v, x["g"], d["scale"], x["segment_ids"], x["h0"], True, chunk, d["n_seqs"], poison=True)
    dq, dk, dv, dg, dh0 = bwd(q, k, v, x["g"], x["do"], d["scale"], x["segment_ids"], x["h0"], x["dht"], chunk,
                              d["n_seqs"], poison=True)
    torch.cuda.synchronize()
    glc.get_device_error()
    return dict(o=np64(o), ht=np64(ht), dq=np64(dq), dk=np64(dk), dv=np64(dv), dg=np64(dg), dh0=np64(dh0))


def check(d, gpu):
    o, ht = oracle.fwd(d["q"], d["k"], d["v"], d["g"], d["scale"], d["segment_ids"], d["h0"])
    gr = oracle.bwd(d["q"], d["k"], d["v"], d["g"], d["do"], d["scale"], d["segment_ids"], d["h0"], d["dht"])
    ref = dict(o=o, ht=ht, **gr)
    if d["h0"] is None:
        ref["dh0"] = None
    errs = {}
    for n, want in ref.items():
        if want is None or gpu.get(n) is None:
            continue
        assert gpu[n].shape == want.shape, n
        assert np.isfinite(gpu[n]).all(), n
        errs[n] = rel(gpu[n], want)
    tol = TOL[d["workload"].dtype]
    print("rel errors:", {n: f"{e:.2e}" for n, e in errs.items()})
    assert all(e <= tol[n] for n, e in errs.items()), errs


def case(base, seed, **over):
    return inputs.make(inputs.WORKLOADS[base], seed=seed, **over)


CASES = {
    # fused projection, tensor-core kernels
    "fused_qkv_gla_bf16": (lambda: case(2, 61, B=2, T=200, H=2, Hqk=2), True),
    "fused_qkv_gla_bf16_packed_states": (lambda: case(4, 62, B=1, T=400, H=2, Hqk=2, doc_mean=90), True),
    "fused_qkv_gla_bf16_pieces": (lambda: case(5, 63, B=1, T=2000, H=1, Hqk=1), True),
    # fused projection, CUDA-core kernels (fp32)
    "fused_qkv_gla_fp32": (lambda: case(1, 64, B=2, T=90, H=2, Hqk=2, K=64, V=64), True),
    # fused projection, SSD (grouped B / C, V = 64)
    "fused_qkv_ssd_bf16": (lambda: case(3, 65, B=1, T=200, H=4, Hqk=1), True),
    # shared q / k heads, per-channel gate (GQA-style, H / Hqk = 4)
    "gqa4_gla_bf16": (lambda: case(2, 66, B=2, T=300, H=4, Hqk=1), False),
    "gqa4_gla_bf16_packed_states": (lambda: case(4, 67, B=1, T=500, H=8, Hqk=2, doc_mean=120), False),
    "gqa4_gla_bf16_pieces": (lambda: case(5, 68, B=1, T=2000, H=4, Hqk=1), False),
    "gqa4_gla_bf16_fused_qkv": (lambda: case(5, 69, B=2, T=150, H=4, Hqk=1), True),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_layout_against_oracle(cuda_ok, name):
    make, strided = CASES[name]
    d = make()
    check(d, run(d, strided))


def test_fused_projection_is_read_in_place(cuda_ok):
    """The binding passes the strided views themselves: the problem carries
    the projection's token stride and the views' own addresses."""
    d = case(2, 70, B=1, T=64, H=2, Hqk=2)
    proj, q, k, v = fused_views(d, "cuda")
    p, keep = glc._problem(q, k, v, inputs.to_device(d, "cuda")["g"], d["scale"], None, None, 0, None, False)
    assert p.q == q.data_ptr() == proj.data_ptr()
    assert p.k == k.data_ptr() and p.v == v.data_ptr()
    assert p.q_stride == p.k_stride == p.v_stride == proj.shape[2]
    del keep
