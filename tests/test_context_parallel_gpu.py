"""Context parallelism through the library's kernels on one GPU: R ranks run
as host threads sharing the GPU (their kernels never wait on one another;
the all-gathers are host-side barriers), each holding one consecutive slice
of every row.  The slices' outputs, put together, must match the oracle run
over the whole sequence at the bf16 tolerances."""
import threading

import numpy as np
import pytest
import torch

import chunked_gated_linear_chunk_gb300 as glc
import oracle
from chunked_gated_linear_chunk_gb300 import context_parallel as cp
from chunked_gated_linear_chunk_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = dict(o=5e-3, ht=5e-3, dq=2e-2, dk=2e-2, dv=2e-2, dg=2e-2, dh0=2e-2)


class ThreadComm:
    def __init__(self, shared, rank, world):
        self.s, self.rank, self.world = shared, rank, world

    def all_gather(self, t):
        self.s["slots"][self.rank] = t
        self.s["bar"].wait()
        out = list(self.s["slots"])
        self.s["bar"].wait()
        return out

    def broadcast(self, t, src):
        if self.rank == src:
            self.s["b"] = t
        self.s["bar"].wait()
        out = self.s["b"]
        self.s["bar"].wait()
        return out


def rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


@pytest.mark.parametrize("R,B,T,H", [(2, 2, 400, 2), (4, 1, 1024, 2)])
def test_threads_as_ranks_match_the_whole_sequence(cuda_ok, R, B, T, H):
    d = inputs.make(inputs.WORKLOADS[5], seed=80 + R, B=B, T=T, H=H, Hqk=H)
    x = inputs.to_device(d, "cuda")
    shared = {"slots": [None] * R, "bar": threading.Barrier(R), "b": None}
    res, errs = {}, []

    def rank_fn(r):
        try:
            sl = slice(r * T // R, (r + 1) * T // R)
            part = [x[n][:, sl].contiguous() for n in ("q", "k", "v", "g", "do")]
            comm = ThreadComm(shared, r, R)
            o, ht, s_in = cp.cp_gla_fwd(*part[:4], d["scale"], x["h0"], comm=comm)
            dq, dk, dv, dg, dh0 = cp.cp_gla_bwd(*part, s_in, d["scale"], x["dht"], comm=comm)
            torch.cuda.synchronize()
            res[r] = dict(o=o, ht=ht, dq=dq, dk=dk, dv=dv, dg=dg, dh0=dh0)
        except Exception as e:  # noqa: BLE001
            errs.append(e)
            shared["bar"].abort()

    ts = [threading.Thread(target=rank_fn, args=(r,)) for r in range(R)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errs, errs
    glc.get_device_error()
    o, ht = oracle.fwd(d["q"], d["k"], d["v"], d["g"], d["scale"], None, d["h0"])
    gr = oracle.bwd(d["q"], d["k"], d["v"], d["g"], d["do"], d["scale"], None, d["h0"], d["dht"])
    f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()
    cat = lambda n: np.concatenate([f64(res[r][n]) for r in range(R)], axis=1)
    e = dict(o=rel(cat("o"), o), dq=rel(cat("dq"), gr["dq"]), dk=rel(cat("dk"), gr["dk"]),
             dv=rel(cat("dv"), gr["dv"]), dg=rel(cat("dg"), gr["dg"]),
             ht=max(rel(f64(res[r]["ht"]), ht) for r in range(R)),
             dh0=max(rel(f64(res[r]["dh0"]), gr["dh0"]) for r in range(R)))
    print("rel errors:", {n: f"{v:.2e}" for n, v in e.items()})
    assert all(e[n] <= TOL[n] for n in e), e


def test_state_entries_match_the_oracle(cuda_ok):
    """gla_fwd_state: the final state from zero and exp(sum g); gla_bwd_state:
    dh0 with dht = 0 and the same decay."""
    d = inputs.make(inputs.WORKLOADS[2], seed=90, B=2, T=300, H=2, Hqk=2)
    x = inputs.to_device(d, "cuda")
    L, D = glc.gla_fwd_state(x["q"], x["k"], x["v"], x["g"], d["scale"])
    Lr, Dr = glc.gla_bwd_state(x["q"], x["k"], x["v"], x["g"], x["do"], d["scale"])
    torch.cuda.synchronize()
    glc.get_device_error()
    _, ht = oracle.fwd(d["q"], d["k"], d["v"], d["g"], d["scale"])
    B, H, K, V = 2, 2, 128, 128
    gr = oracle.bwd(d["q"], d["k"], d["v"], d["g"], d["do"], d["scale"], None, np.zeros((B, H, K, V)), None)
    dec = np.exp(d["g"].double().sum(dim=1).numpy())
    f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()
    assert rel(f64(L), ht) <= 5e-3
    assert rel(f64(Lr), gr["dh0"]) <= 2e-2
    assert rel(f64(D), dec) <= 1e-5 and rel(f64(Dr), dec) <= 1e-5


def test_library_call_from_a_fresh_host_thread(cuda_ok):
    """A host thread that has made no CUDA call yet calls the C ABI directly
    (buffers allocated by the main thread): the library binds the device's
    context itself before it encodes its tensor maps."""
    import ctypes

    d = inputs.make(inputs.WORKLOADS[2], seed=91, B=1, T=256, H=2, Hqk=2)
    x = inputs.to_device(d, "cuda")
    p, keep = glc._problem(x["q"], x["k"], x["v"], x["g"], d["scale"], None, None, 0, None, False)
    o = torch.full_like(x["v"], float("nan"))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    status = []
    t = threading.Thread(target=lambda: status.append(glc.load().gla_fwd(ctypes.byref(p), glc._ptr(o), None, stream)))
    t.start()
    t.join()
    torch.cuda.synchronize()
    assert status == [glc.OK], status
    glc.get_device_error()
    ro, _ = oracle.fwd(d["q"], d["k"], d["v"], d["g"], d["scale"])
    assert rel(o.double().cpu().numpy(), ro) <= 5e-3
    del keep
