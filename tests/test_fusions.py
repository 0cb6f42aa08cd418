"""Pins of the fp64 oracles of the two fused operations around the recurrence
(oracle/fusions.py): closed forms, invariances, packed documents and central
finite differences.  CPU only."""
import math

import numpy as np
import pytest

from oracle import fusions as F

RNG = np.random.default_rng(1234)


# ------------------------------------------------------------ norm_gate ----
def test_norm_gate_constant_row_closed_form():
    """A constant row c * 1 has mean square c^2, so with eps = 0 the norm is
    sign(c) * 1 and y = sign(c) * w * swish(z).  z = ln 3 gives sigmoid = 3/4,
    so swish(ln 3) = 0.75 ln 3 (a wrong mean, a missing root or a sigmoid in
    place of swish all fail)."""
    V = 8
    w = np.linspace(0.5, 2.0, V)
    z = np.full((1, V), math.log(3.0))
    for c in (2.5, -0.25):
        y = F.norm_gate_fwd(np.full((1, V), c), z, w, 0.0)
        want = math.copysign(1.0, c) * w * 0.75 * math.log(3.0)
        assert np.allclose(y[0], want, rtol=1e-13, atol=0)


def test_norm_gate_zero_gate_and_scale_invariance():
    o = RNG.normal(size=(4, 16))
    w = RNG.normal(size=16)
    assert np.all(F.norm_gate_fwd(o, np.zeros_like(o), w, 1e-5) == 0.0)
    z = RNG.normal(size=(4, 16))
    assert np.allclose(F.norm_gate_fwd(3.7 * o, z, w, 0.0), F.norm_gate_fwd(o, z, w, 0.0), rtol=1e-13, atol=1e-15)


def test_norm_gate_eps_enters_the_mean_square():
    """mean(o^2) + eps: a row of zeros but one entry a, eps = a^2 (V - 1) / V
    doubles the mean square, so the norm of that entry is 1/sqrt(2) * sqrt(V)."""
    V, a = 4, 0.8
    o = np.zeros((1, V))
    o[0, 1] = a
    eps = a * a / V
    y = F.norm_gate_fwd(o, np.full((1, V), 50.0), np.ones(V), eps)  # swish(50) = 50 to 1e-20
    assert y[0, 1] == pytest.approx(a / math.sqrt(2 * a * a / V) * 50.0, rel=1e-12)


def _fd(f, x, idx, h=1e-6):
    e = np.zeros_like(x)
    e[idx] = h
    return (f(x + e) - f(x - e)) / (2 * h)


def test_norm_gate_gradients_by_finite_differences():
    o, z, dy = (RNG.normal(size=(3, 5, 16)) for _ in range(3))
    w = RNG.normal(size=16)
    eps = 1e-5
    do, dz, dw = F.norm_gate_bwd(o, z, w, dy, eps)
    loss = lambda o_, z_, w_: float(np.sum(F.norm_gate_fwd(o_, z_, w_, eps) * dy))
    for idx in [(0, 0, 0), (1, 2, 3), (2, 4, 15)]:
        assert _fd(lambda t: loss(t, z, w), o, idx) == pytest.approx(do[idx], rel=1e-7, abs=1e-9)
        assert _fd(lambda t: loss(o, t, w), z, idx) == pytest.approx(dz[idx], rel=1e-7, abs=1e-9)
    for i in (0, 7, 15):
        assert _fd(lambda t: loss(o, z, t), w, (i,)) == pytest.approx(dw[i], rel=1e-7, abs=1e-9)


# ----------------------------------------------------------- short_conv ----
def test_short_conv_last_tap_is_identity_and_silu():
    """Only the last tap (which reads x_t) set to 1, no bias: z = x; with
    SiLU, x = ln 3 gives 0.75 ln 3."""
    B, T, D, Kc = 2, 7, 3, 4
    x = RNG.normal(size=(B, T, D))
    w = np.zeros((Kc, D))
    w[Kc - 1] = 1.0
    assert np.array_equal(F.short_conv_fwd(x, w, None, activation=False), x)
    x2 = np.full((1, 1, 1), math.log(3.0))
    assert F.short_conv_fwd(x2, np.ones((1, 1)), None)[0, 0, 0] == pytest.approx(0.75 * math.log(3.0), rel=1e-14)


def test_short_conv_first_tap_is_a_causal_shift_reset_per_document():
    """Only tap 0 set: y_t = x_{t-(Kc-1)}, zero for the first Kc-1 tokens of
    every document (row start or segment id change)."""
    B, T, D, Kc = 1, 10, 2, 4
    x = RNG.normal(size=(B, T, D))
    w = np.zeros((Kc, D))
    w[0] = 1.0
    seg = np.array([[0, 0, 0, 0, 0, 1, 1, 1, 1, 1]])
    y = F.short_conv_fwd(x, w, None, seg, activation=False)
    want = np.zeros_like(x)
    want[0, 3:5] = x[0, 0:2]
    want[0, 8:10] = x[0, 5:7]
    assert np.array_equal(y, want)


def test_short_conv_packed_documents_equal_separate_runs():
    D, Kc = 4, 4
    lens = [1, 5, 3, 8]
    x = RNG.normal(size=(1, sum(lens), D))
    dy = RNG.normal(size=x.shape)
    w, b = RNG.normal(size=(Kc, D)), RNG.normal(size=D)
    seg = np.concatenate([np.full(n, i) for i, n in enumerate(lens)])[None]
    y = F.short_conv_fwd(x, w, b, seg)
    dx, dw, db = F.short_conv_bwd(x, w, b, dy, seg)
    o = 0
    dws, dbs = np.zeros_like(dw), np.zeros_like(db)
    for n in lens:
        sl = slice(o, o + n)
        assert np.array_equal(y[:, sl], F.short_conv_fwd(x[:, sl], w, b))
        dxi, dwi, dbi = F.short_conv_bwd(x[:, sl], w, b, dy[:, sl])
        assert np.allclose(dx[:, sl], dxi, rtol=0, atol=1e-14)
        dws += dwi
        dbs += dbi
        o += n
    assert np.allclose(dw, dws, atol=1e-12) and np.allclose(db, dbs, atol=1e-12)


def test_short_conv_input_gradient_is_the_adjoint():
    """Without the activation the convolution is linear in x:
    <dy, conv(dx_probe)> = <conv^T dy, dx_probe> for any probe."""
    B, T, D, Kc = 2, 11, 3, 4
    w = RNG.normal(size=(Kc, D))
    seg = np.array([[0] * 4 + [1] * 7, [2] * 11])
    dy = RNG.normal(size=(B, T, D))
    probe = RNG.normal(size=(B, T, D))
    dx, _, _ = F.short_conv_bwd(probe, w, None, dy, seg, activation=False)
    lhs = np.sum(dy * F.short_conv_fwd(probe, w, None, seg, activation=False))
    assert lhs == pytest.approx(np.sum(dx * probe), rel=1e-12)


def test_short_conv_gradients_by_finite_differences():
    B, T, D, Kc = 2, 9, 5, 4
    x, dy = RNG.normal(size=(B, T, D)), RNG.normal(size=(B, T, D))
    w, b = RNG.normal(size=(Kc, D)), RNG.normal(size=D)
    seg = np.array([[0, 0, 0, 1, 1, 1, 1, 2, 2], [5] * 9])
    dx, dw, db = F.short_conv_bwd(x, w, b, dy, seg)
    loss = lambda x_, w_, b_: float(np.sum(F.short_conv_fwd(x_, w_, b_, seg) * dy))
    for idx in [(0, 0, 0), (0, 2, 1), (0, 6, 4), (1, 8, 2)]:
        assert _fd(lambda t: loss(t, w, b), x, idx) == pytest.approx(dx[idx], rel=1e-7, abs=1e-9)
    for idx in [(0, 0), (1, 3), (3, 4)]:
        assert _fd(lambda t: loss(x, t, b), w, idx) == pytest.approx(dw[idx], rel=1e-7, abs=1e-9)
    assert _fd(lambda t: loss(x, w, t), b, (2,)) == pytest.approx(db[2], rel=1e-7, abs=1e-9)
