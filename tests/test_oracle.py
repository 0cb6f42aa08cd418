"""Pins for the fp64 oracle (CPU only).

Each test checks the oracle against something other than itself: central
finite differences, textbook closed forms, an independently written
parallel (quadratic) form, the Mamba-2 dual form, packing invariants and a
chunkwise restatement evaluated at many chunk sizes.  A dropped term, a
wrong sign, a transposed operand or an off-by-one in the causal mask breaks
at least one of them.
"""
import numpy as np
import pytest

import oracle
from oracle import chunkwise

RNG = np.random.default_rng(42)


def rand_case(B=1, T=12, H=1, Hqk=None, K=3, V=3, gate="channel", seg=None, h0=True, dht=True,
              gscale=0.5, rng=RNG):
    Hqk = H if Hqk is None else Hqk
    q = rng.standard_normal((B, T, Hqk, K))
    k = rng.standard_normal((B, T, Hqk, K))
    v = rng.standard_normal((B, T, H, V))
    if gate == "channel":
        g = -gscale * rng.random((B, T, H, K)) - 0.01
    else:
        g = -gscale * rng.random((B, T, H)) - 0.01
    do = rng.standard_normal((B, T, H, V))
    n = oracle.count_docs(seg, B, T)
    h0a = rng.standard_normal((n, H, K, V)) if h0 else None
    dhta = rng.standard_normal((n, H, K, V)) if dht else None
    return dict(q=q, k=k, v=v, g=g, do=do, seg=seg, h0=h0a, dht=dhta, scale=0.7)


def loss(c, **over):
    d = dict(c)
    d.update(over)
    o, ht = oracle.fwd(d["q"], d["k"], d["v"], d["g"], d["scale"], d["seg"], d["h0"])
    val = float((o * d["do"]).sum())
    if d["dht"] is not None:
        val += float((ht * d["dht"]).sum())
    return val


def grads(c):
    return oracle.bwd(c["q"], c["k"], c["v"], c["g"], c["do"], c["scale"], c["seg"], c["h0"], c["dht"])


def rel(a, b):
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)


# ---------------------------------------------------------------- P1 ----
@pytest.mark.parametrize("gate,H,Hqk", [("channel", 1, 1), ("head", 2, 1), ("channel", 2, 2)])
def test_finite_differences_every_gradient(gate, H, Hqk):
    """Central differences (h = 1e-6) of <do,o> + <dht,ht> for every input entry."""
    seg = np.array([[0] * 5 + [1] * 7], dtype=np.int32)  # 2 documents, B1 T12
    c = rand_case(B=1, T=12, H=H, Hqk=Hqk, K=3, V=3, gate=gate, seg=seg)
    gr = grads(c)
    eps = 1e-6
    for name, gname in [("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("h0", "dh0")]:
        x = c[name]
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = x.copy()
            xm = x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            num[idx] = (loss(c, **{name: xp}) - loss(c, **{name: xm})) / (2 * eps)
        assert rel(gr[gname], num) < 1e-7, (name, rel(gr[gname], num))


def test_adjoint_identity_random_directions():
    """<grad L, dx> equals the directional derivative for random dx (all inputs at once)."""
    rng = np.random.default_rng(7)
    seg = np.array([[3] * 9 + [1] * 20 + [3] * 11, [5] * 40], dtype=np.int32)
    c = rand_case(B=2, T=40, H=2, K=4, V=5, seg=seg, rng=rng)
    gr = grads(c)
    names = [("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("h0", "dh0")]
    for _ in range(3):
        dirs = {n: rng.standard_normal(c[n].shape) for n, _ in names}
        eps = 1e-6
        plus = {n: c[n] + eps * dirs[n] for n, _ in names}
        minus = {n: c[n] - eps * dirs[n] for n, _ in names}
        num = (loss(c, **plus) - loss(c, **minus)) / (2 * eps)
        ana = sum(float((gr[gn] * dirs[n]).sum()) for n, gn in names)
        assert abs(num - ana) <= 1e-7 * max(1.0, abs(ana))


# ---------------------------------------------------------------- P2 ----
def test_closed_form_no_gate():
    """g = 0, h0 = 0: textbook causal linear attention and its gradients."""
    rng = np.random.default_rng(1)
    B, T, H, K, V = 2, 37, 3, 5, 4
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    v = rng.standard_normal((B, T, H, V))
    do = rng.standard_normal((B, T, H, V))
    g = np.zeros((B, T, H, K))
    s = 0.3
    o, ht = oracle.fwd(q, k, v, g, s)
    gr = oracle.bwd(q, k, v, g, do, s)
    for b in range(B):
        for h in range(H):
            Q, Kt, Vv, dO = q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h]
            A = np.tril(Q @ Kt.T)
            assert rel(o[b, :, h], s * A @ Vv) < 1e-12
            assert rel(ht[b, h], Kt.T @ Vv) < 1e-12
            dA = np.tril(dO @ Vv.T)
            assert rel(gr["dq"][b, :, h], s * dA @ Kt) < 1e-12
            assert rel(gr["dk"][b, :, h], s * dA.T @ Q) < 1e-12
            assert rel(gr["dv"][b, :, h], s * A.T @ dO) < 1e-12
            # dh0 with g = 0 is scale * sum_t q_t do_t^T (no dht here)
            assert rel(gr["dh0"][b, h], s * Q.T @ dO) < 1e-12


# ---------------------------------------------------------------- P3 ----
def test_mamba2_dual_form_and_gla_equivalence():
    """Scalar gate: o = (scale Q K^T (.) L) V with L_ts = exp(G_t - G_s); and GLA with
    every channel equal to the head gate gives the same o, dq, dk, dv, and its dg
    summed over K equals the head-gate dg."""
    rng = np.random.default_rng(3)
    B, T, H, Hqk, K, V = 2, 29, 4, 2, 6, 3
    q = rng.standard_normal((B, T, Hqk, K))
    k = rng.standard_normal((B, T, Hqk, K))
    v = rng.standard_normal((B, T, H, V))
    do = rng.standard_normal((B, T, H, V))
    gh = -rng.random((B, T, H)) * 0.8
    s = 1.0
    o, _ = oracle.fwd(q, k, v, gh, s)
    for b in range(B):
        for h in range(H):
            hk = h // (H // Hqk)
            G = np.cumsum(gh[b, :, h])
            L = np.tril(np.exp(G[:, None] - G[None, :]))
            ref = (s * (q[b, :, hk] @ k[b, :, hk].T) * L) @ v[b, :, h]
            assert rel(o[b, :, h], ref) < 1e-12
    gc = np.repeat(gh[..., None], K, axis=3)
    # GLA needs per-head q/k: expand the shared group explicitly
    qe = np.repeat(q, H // Hqk, axis=2)
    ke = np.repeat(k, H // Hqk, axis=2)
    o2, _ = oracle.fwd(qe, ke, v, gc, s)
    assert rel(o2, o) < 1e-12
    g1 = oracle.bwd(q, k, v, gh, do, s)
    g2 = oracle.bwd(qe, ke, v, gc, do, s)
    assert rel(g2["dv"], g1["dv"]) < 1e-12
    assert rel(g2["dq"].reshape(B, T, Hqk, H // Hqk, K).sum(3), g1["dq"]) < 1e-12
    assert rel(g2["dk"].reshape(B, T, Hqk, H // Hqk, K).sum(3), g1["dk"]) < 1e-12
    assert rel(g2["dg"].sum(3), g1["dg"]) < 1e-12


# ---------------------------------------------------------------- P4 ----
def test_gla_bruteforce_parallel_form():
    """o_t = scale sum_{s<=t} (q_t e^{G_t-G_s}) . k_s v_s + scale (q_t e^{G_t})^T h0."""
    rng = np.random.default_rng(4)
    B, T, H, K, V = 1, 23, 2, 5, 4
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    v = rng.standard_normal((B, T, H, V))
    g = -rng.random((B, T, H, K)) * 0.6
    h0 = rng.standard_normal((1, H, K, V))
    s = 0.5
    o, _ = oracle.fwd(q, k, v, g, s, h0=h0)
    ref = np.zeros_like(o)
    for h in range(H):
        G = np.cumsum(g[0, :, h], axis=0)
        for t in range(T):
            acc = (q[0, t, h] * np.exp(G[t])) @ h0[0, h]
            for s_ in range(t + 1):
                w = np.sum(q[0, t, h] * np.exp(G[t] - G[s_]) * k[0, s_, h])
                acc = acc + w * v[0, s_, h]
            ref[0, t, h] = s * acc
    assert rel(o, ref) < 1e-12


# ---------------------------------------------------------------- P5 ----
@pytest.mark.parametrize("gate", ["channel", "head"])
def test_dg_two_derivations(gate):
    """Recurrence form (oracle) == suffix sum of q*dq - k*dk plus (S_end (.) dht) 1_V."""
    rng = np.random.default_rng(5)
    seg = np.array([[0] * 10 + [1] * 15 + [2] * 6], dtype=np.int32)
    c = rand_case(B=1, T=31, H=2, K=4, V=3, gate=gate, seg=seg, rng=rng)
    gr = grads(c)
    _, ht = oracle.fwd(c["q"], c["k"], c["v"], c["g"], c["scale"], seg, c["h0"])
    docs = [(0, 10), (10, 25), (25, 31)]
    for d, (t0, t1) in enumerate(docs):
        for h in range(2):
            a = c["q"][0, t0:t1, h] * gr["dq"][0, t0:t1, h] - c["k"][0, t0:t1, h] * gr["dk"][0, t0:t1, h]
            suf = np.cumsum(a[::-1], axis=0)[::-1] + (ht[d, h] * c["dht"][d, h]).sum(1)[None, :]
            ref = suf if gate == "channel" else suf.sum(1)
            assert rel(gr["dg"][0, t0:t1, h], ref) < 1e-12


# ---------------------------------------------------------------- P6 ----
@pytest.mark.parametrize("chunk", [1, 3, 16, 64, 256])
@pytest.mark.parametrize("T", [1, 63, 65, 200])
def test_chunkwise_restatement_matches(chunk, T):
    rng = np.random.default_rng(100 + T + chunk)
    B, H, K, V = 2, 2, 8, 6
    # documents that start mid-chunk, one of length 1
    seg = np.zeros((B, T), dtype=np.int32)
    if T > 5:
        seg[0, T // 3:] = 1
        seg[0, T // 3 + 1:] = 2
        seg[1, T // 2:] = 7
    c = rand_case(B=B, T=T, H=H, K=K, V=V, seg=seg, rng=rng, gscale=0.3)
    o, ht = oracle.fwd(c["q"], c["k"], c["v"], c["g"], c["scale"], seg, c["h0"])
    o2, ht2 = chunkwise.forward(c["q"], c["k"], c["v"], c["g"], c["scale"], chunk, seg, c["h0"])
    assert rel(o2, o) < 1e-12 and rel(ht2, ht) < 1e-12
    gr = grads(c)
    gr2 = chunkwise.backward(c["q"], c["k"], c["v"], c["g"], c["do"], c["scale"], chunk, seg, c["h0"], c["dht"])
    for n in ("dq", "dk", "dv", "dg", "dh0"):
        assert rel(gr2[n], gr[n]) < 1e-11, n


def test_chunkwise_head_gate_shared_qk():
    rng = np.random.default_rng(11)
    c = rand_case(B=1, T=70, H=4, Hqk=1, K=8, V=4, gate="head", rng=rng)
    gr = grads(c)
    gr2 = chunkwise.backward(c["q"], c["k"], c["v"], c["g"], c["do"], c["scale"], 16, None, c["h0"], c["dht"])
    for n in ("dq", "dk", "dv", "dg", "dh0"):
        assert rel(gr2[n], gr[n]) < 1e-11, n


# ---------------------------------------------------------------- P7 ----
def test_packed_documents_equal_separate_runs():
    rng = np.random.default_rng(6)
    lens = [1, 17, 64, 3, 40]
    T = sum(lens)
    seg = np.concatenate([np.full(n, i * 3 % 5, dtype=np.int32) for i, n in enumerate(lens)])[None, :]
    c = rand_case(B=1, T=T, H=2, K=4, V=5, seg=seg, rng=rng)
    o, ht = oracle.fwd(c["q"], c["k"], c["v"], c["g"], c["scale"], seg, c["h0"])
    gr = grads(c)
    t0 = 0
    for d, n in enumerate(lens):
        sl = slice(t0, t0 + n)
        od, htd = oracle.fwd(c["q"][:, sl], c["k"][:, sl], c["v"][:, sl], c["g"][:, sl], c["scale"],
                             None, c["h0"][d:d + 1])
        gd = oracle.bwd(c["q"][:, sl], c["k"][:, sl], c["v"][:, sl], c["g"][:, sl], c["do"][:, sl],
                        c["scale"], None, c["h0"][d:d + 1], c["dht"][d:d + 1])
        assert np.array_equal(o[:, sl], od) and np.array_equal(ht[d], htd[0])
        for n_ in ("dq", "dk", "dv", "dg"):
            assert np.array_equal(gr[n_][:, sl], gd[n_])
        assert np.array_equal(gr["dh0"][d], gd["dh0"][0])
        t0 += n


def test_each_batch_row_is_a_document():
    rng = np.random.default_rng(8)
    c = rand_case(B=3, T=9, H=1, K=2, V=2, rng=rng)
    seg = np.zeros((3, 9), dtype=np.int32)  # same id in every row: still 3 documents
    assert oracle.count_docs(seg, 3, 9) == 3
    o1, h1 = oracle.fwd(c["q"], c["k"], c["v"], c["g"], 1.0, seg, c["h0"])
    o2, h2 = oracle.fwd(c["q"], c["k"], c["v"], c["g"], 1.0, None, c["h0"])
    assert np.array_equal(o1, o2) and np.array_equal(h1, h2)


# ---------------------------------------------------------------- P8 ----
def test_full_forgetting_gate():
    """g = -inf (exp(g) = 0): only the current token survives, o_t = scale (q_t.k_t) v_t."""
    rng = np.random.default_rng(9)
    B, T, H, K, V = 1, 10, 2, 3, 4
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    v = rng.standard_normal((B, T, H, V))
    g = np.full((B, T, H, K), -np.inf)
    o, ht = oracle.fwd(q, k, v, g, 0.9, h0=rng.standard_normal((1, H, K, V)))
    ref = 0.9 * np.einsum("bthk,bthk->bth", q, k)[..., None] * v
    assert rel(o, ref) < 1e-14
    assert rel(ht[0], np.einsum("hk,hv->hkv", k[0, -1], v[0, -1])) < 1e-14


def test_linearity_in_v_and_h0():
    rng = np.random.default_rng(10)
    c = rand_case(B=1, T=15, H=2, K=3, V=3, rng=rng)
    v2 = rng.standard_normal(c["v"].shape)
    o1, _ = oracle.fwd(c["q"], c["k"], c["v"], c["g"], 0.5)
    o2, _ = oracle.fwd(c["q"], c["k"], v2, c["g"], 0.5)
    o3, _ = oracle.fwd(c["q"], c["k"], 2.0 * c["v"] - 3.0 * v2, c["g"], 0.5)
    assert rel(o3, 2.0 * o1 - 3.0 * o2) < 1e-12
    z = np.zeros_like(c["v"])
    oh, _ = oracle.fwd(c["q"], c["k"], z, c["g"], 0.5, h0=c["h0"])
    oh2, _ = oracle.fwd(c["q"], c["k"], z, c["g"], 0.5, h0=-2.5 * c["h0"])
    o4, _ = oracle.fwd(c["q"], c["k"], c["v"], c["g"], 0.5, h0=c["h0"])
    assert rel(oh2, -2.5 * oh) < 1e-12
    assert rel(o4, o1 + oh) < 1e-12


def test_dh0_without_gate():
    rng = np.random.default_rng(12)
    c = rand_case(B=1, T=14, H=1, K=3, V=2, rng=rng)
    g = np.zeros_like(c["g"])
    gr = oracle.bwd(c["q"], c["k"], c["v"], g, c["do"], 0.8, None, c["h0"], c["dht"])
    ref = 0.8 * c["q"][0, :, 0].T @ c["do"][0, :, 0] + c["dht"][0, 0]
    assert rel(gr["dh0"][0, 0], ref) < 1e-12


# ---------------------------------------------------------------- P9 ----
def test_piece_split_handoff():
    """Running a document in pieces with the exact state hand-off
    S_in[p] = diag(D_{p-1}) S_in[p-1] + L_{p-1} (L = piece end state from zero,
    D = exp of the piece's summed log gate) equals the unsplit run."""
    rng = np.random.default_rng(13)
    c = rand_case(B=1, T=90, H=2, K=4, V=3, rng=rng)
    o, ht = oracle.fwd(c["q"], c["k"], c["v"], c["g"], 0.6, None, c["h0"])
    cuts = [0, 25, 26, 64, 90]
    S_in = c["h0"].copy()
    for p in range(len(cuts) - 1):
        sl = slice(cuts[p], cuts[p + 1])
        op, _ = oracle.fwd(c["q"][:, sl], c["k"][:, sl], c["v"][:, sl], c["g"][:, sl], 0.6, None, S_in)
        assert rel(op, o[:, sl]) < 1e-12
        _, L = oracle.fwd(c["q"][:, sl], c["k"][:, sl], c["v"][:, sl], c["g"][:, sl], 0.6, None, None)
        D = np.exp(c["g"][0, sl].sum(axis=0))  # [H, K]
        S_in = D[None, :, :, None] * S_in + L
    assert rel(S_in, ht) < 1e-12


def test_empty_sequence():
    q = np.zeros((1, 0, 1, 2))
    v = np.zeros((1, 0, 1, 2))
    g = np.zeros((1, 0, 1, 2))
    o, ht = oracle.fwd(q, q, v, g, 1.0)
    assert o.shape == (1, 0, 1, 2) and ht.shape == (0, 1, 2, 2)
