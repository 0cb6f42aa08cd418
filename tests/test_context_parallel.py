"""Context parallelism (the sequence split across ranks) on CPU: two gloo
ranks run cp_gla_fwd / cp_gla_bwd with the fp64 oracle standing in for each
slice's device work (test infrastructure), through real torch.distributed
collectives.  The slices' outputs, put together, must equal the oracle run
over the whole sequence (the split is exact), initial state and dht
included."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleOps:
    """A slice's device work, done by the fp64 oracle on CPU tensors."""

    def fwd_state(self, q, k, v, g, scale):
        import oracle

        _, ht = oracle.fwd(q, k, v, g, scale)
        return torch.from_numpy(ht), torch.exp(g.double().sum(dim=1))

    def bwd_state(self, q, k, v, g, do, scale):
        import oracle

        B, H, K, V = q.shape[0], v.shape[2], q.shape[3], v.shape[3]
        gr = oracle.bwd(q, k, v, g, do, scale, None, np.zeros((B, H, K, V)), None)
        return torch.from_numpy(gr["dh0"]), torch.exp(g.double().sum(dim=1))

    def scan(self, Ls, Ds, r, seed, reverse):
        s = torch.zeros_like(Ls[0]) if seed is None else seed.double().clone()
        order = range(len(Ls) - 1, r, -1) if reverse else range(r)
        for qq in order:
            s = Ds[qq][..., None] * s + Ls[qq]
        return s

    def fwd(self, q, k, v, g, scale, h0):
        import oracle

        o, ht = oracle.fwd(q, k, v, g, scale, None, h0)
        return torch.from_numpy(o), torch.from_numpy(ht)

    def bwd(self, q, k, v, g, do, scale, h0, dht):
        import oracle

        gr = oracle.bwd(q, k, v, g, do, scale, None, h0, dht)
        return tuple(torch.from_numpy(gr[n]) for n in ("dq", "dk", "dv", "dg", "dh0"))


def _inputs(B=2, T=48, H=2, K=8, V=8):
    gen = torch.Generator().manual_seed(5)
    q = torch.randn(B, T, H, K, generator=gen, dtype=torch.float64)
    k = torch.nn.functional.normalize(torch.randn(B, T, H, K, generator=gen, dtype=torch.float64), dim=-1)
    v = torch.randn(B, T, H, V, generator=gen, dtype=torch.float64)
    g = torch.nn.functional.logsigmoid(torch.randn(B, T, H, K, generator=gen, dtype=torch.float64)) / 4
    do = torch.randn(B, T, H, V, generator=gen, dtype=torch.float64)
    h0 = 0.1 * torch.randn(B, H, K, V, generator=gen, dtype=torch.float64)
    dht = 0.1 * torch.randn(B, H, K, V, generator=gen, dtype=torch.float64)
    return q, k, v, g, do, h0, dht


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from chunked_gated_linear_chunk_gb300 import context_parallel as cp

        q, k, v, g, do, h0, dht = _inputs()
        T = q.shape[1]
        sl = slice(rank * T // world, (rank + 1) * T // world)
        part = [t[:, sl].contiguous() for t in (q, k, v, g, do)]
        comm = cp.TorchComm()
        ops = OracleOps()
        o, ht, s_in = cp.cp_gla_fwd(*part[:4], 0.3, h0, comm=comm, ops=ops)
        dq, dk, dv, dg, dh0 = cp.cp_gla_bwd(*part, s_in, 0.3, dht, comm=comm, ops=ops)
        out[rank] = {n: t.numpy() for n, t in dict(o=o, ht=ht, dq=dq, dk=dk, dv=dv, dg=dg, dh0=dh0).items()}
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_equal_the_whole_sequence():
    import oracle

    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
        res = {r: out[r] for r in range(world)}
    q, k, v, g, do, h0, dht = _inputs()
    o, ht = oracle.fwd(q, k, v, g, 0.3, None, h0)
    gr = oracle.bwd(q, k, v, g, do, 0.3, None, h0, dht)
    cat = lambda n: np.concatenate([res[r][n] for r in range(world)], axis=1)
    for n, want in (("o", o), ("dq", gr["dq"]), ("dk", gr["dk"]), ("dv", gr["dv"]), ("dg", gr["dg"])):
        assert np.allclose(cat(n), want, rtol=1e-10, atol=1e-12), n
    for r in range(world):
        assert np.allclose(res[r]["ht"], ht, rtol=1e-10, atol=1e-12)
        assert np.allclose(res[r]["dh0"], gr["dh0"], rtol=1e-10, atol=1e-12)


def test_scan_folds_in_piece_order():
    """state_scan semantics on three pieces, by hand."""
    ops = OracleOps()
    L = [torch.full((1, 2, 2), float(i + 1), dtype=torch.float64) for i in range(3)]
    D = [torch.full((1, 2), 0.5, dtype=torch.float64) for _ in range(3)]
    seed = torch.ones(1, 2, 2, dtype=torch.float64)
    want_fwd = torch.full((1, 2, 2), 0.5 * (0.5 * 1 + 1) + 2, dtype=torch.float64)
    want_rev = torch.full((1, 2, 2), 0.5 * (0.5 * 1 + 3) + 2, dtype=torch.float64)
    assert torch.allclose(ops.scan(L, D, 2, seed, False), want_fwd)
    assert torch.allclose(ops.scan(L, D, 0, seed, True), want_rev)
