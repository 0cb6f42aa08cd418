"""GPU parity of the two fused operations around the recurrence (norm_gate,
short_conv) against their fp64 oracles (oracle/fusions.py), element by
element, through the C ABI.

Tolerance (max|a-b| / max|b|): the kernels compute in fp32 from the exact
input values and round each output once, so bf16 outputs are within half a
bf16 ulp (2^-9 ~ 1.95e-3 of the largest value) plus fp32 arithmetic:
4e-3 for bf16 outputs; 1e-4 for fp32 outputs and for the fp32 weight / bias
gradients (sums over every position)."""
import numpy as np
import pytest
import torch

import chunked_gated_linear_chunk_gb300 as glc
from oracle import fusions as F

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: 4e-3, torch.float32: 1e-4}
TOL_F32 = 1e-4


def rel(a, b):
    a = a.detach().to("cpu", torch.float64).numpy() if hasattr(a, "detach") else a
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30)) if b.size else 0.0


def gen(seed):
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    return g


# ------------------------------------------------------------ norm_gate ----
NG_CASES = [
    # (rows shape prefix, V, dtype, eps)
    ((4, 2048, 16), 128, torch.bfloat16, 1e-5),  # the GLA output of the bench workload
    ((1, 7, 3), 128, torch.bfloat16, 1e-5),
    ((2, 33, 5), 64, torch.bfloat16, 1e-6),
    ((1, 100, 2), 256, torch.bfloat16, 1e-5),
    ((3, 9), 8, torch.bfloat16, 0.0),
    ((2, 61, 4), 128, torch.float32, 1e-5),
    ((1,), 32, torch.float32, 1e-5),
]


@pytest.mark.parametrize("shape,V,dtype,eps", NG_CASES)
def test_norm_gate_against_oracle(cuda_ok, shape, V, dtype, eps):
    g = gen(hash((shape, V)) & 0xFFFF)
    o = torch.randn(*shape, V, generator=g).to(dtype)
    z = (2.0 * torch.randn(*shape, V, generator=g)).to(dtype)
    dy = torch.randn(*shape, V, generator=g).to(dtype)
    w = 1.0 + 0.5 * torch.randn(V, generator=g)
    y = glc.norm_gate_fwd(o.cuda(), z.cuda(), w.cuda(), eps)
    do, dz, dw = glc.norm_gate_bwd(o.cuda(), z.cuda(), w.cuda(), dy.cuda(), eps)
    torch.cuda.synchronize()
    ry = F.norm_gate_fwd(o, z, w, eps)
    rdo, rdz, rdw = F.norm_gate_bwd(o, z, w, dy, eps)
    errs = dict(y=rel(y, ry), do=rel(do, rdo), dz=rel(dz, rdz), dw=rel(dw, rdw))
    print("rel errors:", {k: f"{v:.2e}" for k, v in errs.items()})
    tol = dict(y=TOL[dtype], do=TOL[dtype], dz=TOL[dtype], dw=TOL_F32)
    assert all(np.isfinite(x.float().cpu().numpy()).all() for x in (y, do, dz, dw))
    assert all(errs[k] <= tol[k] for k in errs), errs


def test_norm_gate_empty_rows(cuda_ok):
    o = torch.zeros(0, 128, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(128, device="cuda")
    assert glc.norm_gate_fwd(o, o, w).shape == (0, 128)
    do, dz, dw = glc.norm_gate_bwd(o, o, w, o)
    torch.cuda.synchronize()
    assert torch.all(dw == 0)


# ----------------------------------------------------------- short_conv ----
def conv_case(B, T, D, Kc, dtype, seed, packed=False, bias=True, act=True, doc_mean=20):
    g = gen(seed)
    x = torch.randn(B, T, D, generator=g).to(dtype)
    dy = torch.randn(B, T, D, generator=g).to(dtype)
    w = 0.5 * torch.randn(Kc, D, generator=g)
    b = 0.1 * torch.randn(D, generator=g) if bias else None
    seg = None
    if packed:
        rows = []
        for _ in range(B):
            ids, cur, n = [], 0, 0
            while n < T:
                ln = max(1, int(torch.empty(1).geometric_(1.0 / doc_mean, generator=g).item()))
                ids += [cur] * min(ln, T - n)
                n += ln
                cur += 1
            rows.append(torch.tensor(ids[:T], dtype=torch.int32))
        seg = torch.stack(rows)
    return x, w, b, seg, dy, act


CONV_CASES = {
    "flat_shape_B8_T4096_D2048_K4": lambda: conv_case(8, 4096, 2048, 4, torch.bfloat16, 1),
    "ragged_T37_D24": lambda: conv_case(2, 37, 24, 4, torch.bfloat16, 2),
    "T1": lambda: conv_case(1, 1, 16, 4, torch.bfloat16, 3),
    "T3_K4": lambda: conv_case(3, 3, 8, 4, torch.bfloat16, 4),
    "packed_T300": lambda: conv_case(2, 300, 64, 4, torch.bfloat16, 5, packed=True),
    "packed_short_docs": lambda: conv_case(1, 500, 40, 4, torch.bfloat16, 6, packed=True, doc_mean=3),
    "K3_no_bias": lambda: conv_case(2, 129, 136, 3, torch.bfloat16, 7, bias=False),
    "K2_no_act": lambda: conv_case(2, 100, 48, 2, torch.bfloat16, 8, act=False),
    "K1": lambda: conv_case(1, 70, 16, 1, torch.bfloat16, 9),
    "fp32_packed": lambda: conv_case(2, 257, 72, 4, torch.float32, 10, packed=True),
    "run_edges_T513": lambda: conv_case(1, 513, 1032, 4, torch.bfloat16, 11),
}


@pytest.mark.parametrize("name", sorted(CONV_CASES))
def test_short_conv_against_oracle(cuda_ok, name):
    x, w, b, seg, dy, act = CONV_CASES[name]()
    cu = lambda t: None if t is None else t.cuda()
    y = glc.short_conv_fwd(cu(x), cu(w), cu(b), cu(seg), act)
    dx, dw, db = glc.short_conv_bwd(cu(x), cu(w), cu(b), cu(dy), cu(seg), act)
    torch.cuda.synchronize()
    ry = F.short_conv_fwd(x, w, b, seg, act)
    rdx, rdw, rdb = F.short_conv_bwd(x, w, b, dy, seg, act)
    errs = dict(y=rel(y, ry), dx=rel(dx, rdx), dw=rel(dw, rdw), db=rel(db, rdb))
    print("rel errors:", {k: f"{v:.2e}" for k, v in errs.items()})
    tol = dict(y=TOL[x.dtype], dx=TOL[x.dtype], dw=TOL_F32, db=TOL_F32)
    assert all(errs[k] <= tol[k] for k in errs), errs


def test_short_conv_rejects_bad_shapes(cuda_ok):
    x = torch.zeros(1, 4, 12, dtype=torch.bfloat16, device="cuda")  # D not a multiple of 8
    w = torch.zeros(4, 12, device="cuda")
    with pytest.raises(glc.GlacoreError):
        glc.short_conv_fwd(x, w)
    x = torch.zeros(1, 4, 16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(glc.GlacoreError):
        glc.short_conv_fwd(x, torch.zeros(5, 16, device="cuda"))  # five taps
