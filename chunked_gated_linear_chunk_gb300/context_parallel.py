"""GLA with the sequence split across devices (context parallelism).

Each rank of a process group holds the rank-th consecutive slice of every
batch row (all heads), e.g. q[:, r*T/R:(r+1)*T/R].  The split is exact
(JLA product page: "our split is exact"; FLAT blog, "Future work": sharding
the sequence across chips), because the recurrence is linear in the state:

forward   every rank computes its slice's local end state L_r (from a zero
          state) and total decay D_r (gla_fwd_state); one all-gather; the
          state entering slice r is the fold of the earlier slices
          (state_scan, seeded with the sequence's initial state); gla_fwd
          from that state gives the slice's outputs, and the last rank's
          final state is the sequence's.
backward  every rank computes its slice's local start-state gradient and
          decay (gla_bwd_state); one all-gather; the state gradient leaving
          slice r is the fold of the later slices (seeded with dht);
          gla_bwd from the entering state with that gradient gives the
          slice's dq, dk, dv, dg; rank 0's dh0 is the sequence's.

Every step of the arithmetic runs in the library's kernels; this module
moves the per-slice states between ranks (two all-gathers of B*H*K*(V+1)
fp32 values per direction) and calls the C ABI through the package
binding.  `comm` is any object with rank, world and all_gather(tensor) ->
[tensor per rank] and broadcast(tensor, src) -> tensor; the default wraps
torch.distributed (NCCL on GPUs; gloo in the CPU tests)."""
from __future__ import annotations

import torch


class TorchComm:
    """torch.distributed collectives over `group` (default: the world)."""

    def __init__(self, group=None):
        import torch.distributed as dist

        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)

    def all_gather(self, t):
        out = [torch.empty_like(t) for _ in range(self.world)]
        self.dist.all_gather(out, t.contiguous(), group=self.group)
        return out

    def broadcast(self, t, src):
        t = t.contiguous()
        self.dist.broadcast(t, src, group=self.group)
        return t


class GlacoreOps:
    """The device work of one slice, through the library."""

    def __init__(self):
        import chunked_gated_linear_chunk_gb300 as glc

        self.glc = glc

    def fwd_state(self, q, k, v, g, scale):
        return self.glc.gla_fwd_state(q, k, v, g, scale)

    def bwd_state(self, q, k, v, g, do, scale):
        return self.glc.gla_bwd_state(q, k, v, g, do, scale)

    def scan(self, Ls, Ds, r, seed, reverse):
        return self.glc.state_scan(torch.stack(Ls), torch.stack(Ds), r, seed, reverse)

    def fwd(self, q, k, v, g, scale, h0):
        return self.glc.gla_fwd(q, k, v, g, scale, None, h0, True)

    def bwd(self, q, k, v, g, do, scale, h0, dht):
        return self.glc.gla_bwd(q, k, v, g, do, scale, None, h0, dht)


def cp_gla_fwd(q, k, v, g, scale=None, initial_state=None, comm=None, ops=None):
    """Forward of this rank's slice.  Returns (o, final_state of the whole
    sequence [B,H,K,V] on every rank, the state entering this slice)."""
    comm = comm or TorchComm()
    ops = ops or GlacoreOps()
    L, D = ops.fwd_state(q, k, v, g, scale)
    Ls, Ds = comm.all_gather(L), comm.all_gather(D)
    s_in = ops.scan(Ls, Ds, comm.rank, initial_state, False)
    o, ht = ops.fwd(q, k, v, g, scale, s_in)
    final = comm.broadcast(ht, comm.world - 1)
    return o, final, s_in


def cp_gla_bwd(q, k, v, g, do, s_in, scale=None, dht=None, comm=None, ops=None):
    """Backward of this rank's slice, given the state entering it (from
    cp_gla_fwd).  Returns (dq, dk, dv, dg, dh0 of the whole sequence)."""
    comm = comm or TorchComm()
    ops = ops or GlacoreOps()
    Lr, Dr = ops.bwd_state(q, k, v, g, do, scale)
    Ls, Ds = comm.all_gather(Lr), comm.all_gather(Dr)
    d_out = ops.scan(Ls, Ds, comm.rank, dht, True)
    dq, dk, dv, dg, dh0 = ops.bwd(q, k, v, g, do, scale, s_in, d_out)
    dh0 = comm.broadcast(dh0, 0)
    return dq, dk, dv, dg, dh0
