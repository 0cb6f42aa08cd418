"""Seeded synthetic inputs for the five workloads (no method arithmetic here).

Shared by the tests, the bench and the smoke check; it imports neither the
oracle nor the CUDA binding.  Everything is drawn on the CPU in fp32 with a
``torch.Generator`` seeded ``1000 + workload index`` (unless a seed is
given), then cast to the workload's dtype, so the GPU and the oracle see
the same bits.

Recipe (stand-ins for the FLAT blog's B8 S4096 N16 K=V=128 shape family;
no public dataset is involved):
  q, v ~ N(0, 1); k ~ N(0, 1) then L2-normalised per token (GLA);
  GLA gate g = logsigmoid(N(0, 1)) / gdiv per key channel (fp32);
  SSD: x, B, C ~ N(0, 1); dt = softplus(N(0, 1) - 4) [B,T,H];
       A_h = -exp(U(0, ln 16)); g = dt * A (fp32); q = C, k = B, v = x;
  do ~ N(0, 1) (dtype); dht ~ N(0, 0.1^2) fp32 where final states are
  returned; initial states ~ N(0, 0.1^2) fp32 where the workload has them;
  packed documents: lengths ~ Geometric(1/1024) (support >= 1), drawn until
  they cover T, the last one truncated.
"""
from __future__ import annotations

import dataclasses
import math

import torch
import torch.nn.functional as F


@dataclasses.dataclass(frozen=True)
class Workload:
    index: int
    name: str
    kind: str  # "gla" | "ssd"
    B: int
    T: int
    H: int
    Hqk: int
    K: int
    V: int
    dtype: str  # "fp32" | "bf16"
    chunk: int = 64
    gdiv: float = 16.0
    initial_state: bool = False
    final_state: bool = False
    packed: bool = False
    doc_mean: int = 1024

    def torch_dtype(self):
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16

    @property
    def tokens(self) -> int:
        return self.B * self.T


WORKLOADS = {
    1: Workload(1, "tiny_gla_fp32_B1_H2_T256_d64", "gla", 1, 256, 2, 2, 64, 64, "fp32",
                final_state=True),
    2: Workload(2, "gla_bf16_B4_H16_T2048_d128", "gla", 4, 2048, 16, 16, 128, 128, "bf16"),
    3: Workload(3, "ssd_bf16_B4_H32_T4096_N128_P64", "ssd", 4, 4096, 32, 1, 128, 64, "bf16"),
    4: Workload(4, "packed_gla_bf16_B1_T16384_H16_d128", "gla", 1, 16384, 16, 16, 128, 128, "bf16",
                initial_state=True, final_state=True, packed=True),
    5: Workload(5, "long_gla_bf16_B1_H16_T65536_d128", "gla", 1, 65536, 16, 16, 128, 128, "bf16",
                gdiv=32.0, initial_state=True, final_state=True),
}


def doc_lengths(T: int, mean: int, gen: torch.Generator):
    lens = []
    total = 0
    p = 1.0 / mean
    while total < T:
        n = int(torch.empty(1).geometric_(p, generator=gen).item())
        n = max(1, n)
        n = min(n, T - total)
        lens.append(n)
        total += n
    return lens


def make(w: Workload, seed: int | None = None, **over) -> dict:
    """Returns a dict of CPU tensors: q, k, v, g, do, segment_ids, h0, dht,
    plus scale, n_seqs and the workload (possibly with fields overridden)."""
    if over:
        w = dataclasses.replace(w, **over)
    gen = torch.Generator("cpu")
    gen.manual_seed(1000 + w.index if seed is None else seed)
    B, T, H, Hqk, K, V = w.B, w.T, w.H, w.Hqk, w.K, w.V
    dt = w.torch_dtype()

    def randn(*shape):
        return torch.randn(*shape, generator=gen, dtype=torch.float32)

    seg = None
    lens = None
    if w.packed:
        lens = []
        rows = []
        did = 0
        for _ in range(B):
            ls = doc_lengths(T, w.doc_mean, gen)
            lens.extend(ls)
            ids = torch.cat([torch.full((n,), did + i, dtype=torch.int32) for i, n in enumerate(ls)])
            did += len(ls)
            rows.append(ids)
        seg = torch.stack(rows, 0)
        n_seqs = len(lens)
    else:
        n_seqs = B if T > 0 else 0
    if w.kind == "gla":
        q = randn(B, T, Hqk, K)
        k = F.normalize(randn(B, T, Hqk, K), dim=-1)
        v = randn(B, T, H, V)
        g = F.logsigmoid(randn(B, T, H, K)) / w.gdiv
        scale = K ** -0.5
    else:
        q = randn(B, T, Hqk, K)  # C
        k = randn(B, T, Hqk, K)  # B
        v = randn(B, T, H, V)  # x
        dtt = F.softplus(randn(B, T, H) - 4.0)
        A = -torch.exp(torch.rand(H, generator=gen) * math.log(16.0))
        g = dtt * A
        scale = 1.0
    do = randn(B, T, H, V)
    h0 = 0.1 * randn(n_seqs, H, K, V) if w.initial_state else None
    dht = 0.1 * randn(n_seqs, H, K, V) if w.final_state else None
    return dict(q=q.to(dt), k=k.to(dt), v=v.to(dt), g=g.float(), do=do.to(dt), segment_ids=seg,
                h0=h0, dht=dht, scale=scale, n_seqs=n_seqs, workload=w, doc_lengths=lens)


def to_device(d: dict, device) -> dict:
    out = dict(d)
    for key in ("q", "k", "v", "g", "do", "segment_ids", "h0", "dht"):
        if out.get(key) is not None:
            out[key] = out[key].to(device)
    return out
