"""Pins of the SwiGLU gate/up oracle to facts outside itself (CPU only).

The oracle (oracle/swiglu.py) follows ch05 "Acceleration principles: Triton
kernels and fused LoRA", §5.6 (SwiGLU(x) = (W_g x * sigma(W_g x)) * W_u x) with
each projection a LoRA layer of §5.3.  Pins:
  silu_values : sigma(0) = 1/2, sigma(+-ln 3) = 3/4, 1/4 give closed forms of
                silu and silu'; silu(z) - silu(-z) = z; silu(z) -> z and -> 0
  silu_fd     : silu' equals central differences of silu
  plain_gates : A = 0 reduces both projections to X W^T (numpy matmuls)
  up_zero     : Wu = Bu = 0 => H = 0, dX = 0, dAg = dBg = dAu = 0 exactly,
                dBu = s (dH * silu(X Wg^T + s X Ag^T Bg^T))^T X Au^T
  brute       : scalar pure-Python loops with math.exp on a tiny problem
  fd          : central differences of L = <dH, H> in X, Ag, Bg, Au, Bu
  sampled     : the sampled rows equal the full results
Each mutant planted below (a dropped term, swapped operands) fails at least
one pin.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import swiglu


def _problem(seed, M=4, d_in=6, d_ff=5, r=2):
    rng = np.random.default_rng(seed)
    f = lambda *s: rng.standard_normal(s) * 0.7
    return dict(X=f(M, d_in), Wg=f(d_ff, d_in), Ag=f(r, d_in), Bg=f(d_ff, r),
                Wu=f(d_ff, d_in), Au=f(r, d_in), Bu=f(d_ff, r), dH=f(M, d_ff))


def _args(p):
    return p["X"], p["Wg"], p["Ag"], p["Bg"], p["Wu"], p["Au"], p["Bu"]


def pin_silu_values():
    ln3 = math.log(3.0)
    z = np.array([0.0, ln3, -ln3])
    assert np.allclose(swiglu.silu(z), [0.0, 0.75 * ln3, -0.25 * ln3], rtol=0, atol=1e-15)
    assert np.allclose(swiglu.silu_grad(z), [0.5, 0.75 * (1 + 0.25 * ln3),
                                             0.25 * (1 - 0.75 * ln3)], rtol=0, atol=1e-15)
    rng = np.random.default_rng(0)
    w = rng.standard_normal(50) * 5
    assert np.allclose(swiglu.silu(w) - swiglu.silu(-w), w, rtol=0, atol=1e-12)
    assert swiglu.silu(np.array([40.0]))[0] == 40.0
    assert abs(swiglu.silu(np.array([-40.0]))[0]) < 1e-15


def pin_silu_fd():
    z = np.linspace(-6, 6, 41)
    h = 1e-5
    fd = (swiglu.silu(z + h) - swiglu.silu(z - h)) / (2 * h)
    assert np.allclose(swiglu.silu_grad(z), fd, rtol=0, atol=1e-8)


def pin_plain_gates(seed=1, alpha=8.0):
    p = _problem(seed)
    p["Ag"] = np.zeros_like(p["Ag"])
    p["Au"] = np.zeros_like(p["Au"])
    gate, up, H = swiglu.forward(*_args(p), alpha)
    g_ref = p["X"] @ p["Wg"].T
    u_ref = p["X"] @ p["Wu"].T
    assert np.allclose(gate, g_ref, rtol=1e-13, atol=1e-13)
    assert np.allclose(up, u_ref, rtol=1e-13, atol=1e-13)
    assert np.allclose(H, g_ref / (1 + np.exp(-g_ref)) * u_ref, rtol=1e-12, atol=1e-13)


def pin_up_zero(seed=2, alpha=6.0):
    p = _problem(seed)
    p["Wu"] = np.zeros_like(p["Wu"])
    p["Bu"] = np.zeros_like(p["Bu"])
    r = p["Ag"].shape[0]
    s = alpha / r
    _, _, H = swiglu.forward(*_args(p), alpha)
    dX, dAg, dBg, dAu, dBu = swiglu.backward(p["dH"], *_args(p), alpha)
    assert np.array_equal(H, np.zeros_like(H))
    for z in (dX, dAg, dBg, dAu):
        assert np.array_equal(z, np.zeros_like(z))
    gate = p["X"] @ p["Wg"].T + s * (p["X"] @ p["Ag"].T) @ p["Bg"].T
    d_up = p["dH"] * gate / (1 + np.exp(-gate))
    assert np.allclose(dBu, s * d_up.T @ (p["X"] @ p["Au"].T), rtol=1e-12, atol=1e-13)


def _brute(p, alpha):
    """Scalar loops straight from the definitions, no numpy arithmetic."""
    X, Wg, Ag, Bg, Wu, Au, Bu, dH = (p[k].tolist() for k in
                                     ("X", "Wg", "Ag", "Bg", "Wu", "Au", "Bu", "dH"))
    M, d_in, d_ff, r = len(X), len(X[0]), len(Wg), len(Ag)
    s = alpha / r
    sig = lambda z: 1.0 / (1.0 + math.exp(-z))

    def proj(W, A, B):
        Hl = [[sum(X[m][k] * A[i][k] for k in range(d_in)) for i in range(r)] for m in range(M)]
        return Hl, [[sum(X[m][k] * W[o][k] for k in range(d_in)) +
                     s * sum(Hl[m][i] * B[o][i] for i in range(r))
                     for o in range(d_ff)] for m in range(M)]

    Hg, G = proj(Wg, Ag, Bg)
    Hu, U = proj(Wu, Au, Bu)
    H = [[G[m][o] * sig(G[m][o]) * U[m][o] for o in range(d_ff)] for m in range(M)]
    dG = [[dH[m][o] * U[m][o] * (sig(G[m][o]) + G[m][o] * sig(G[m][o]) * (1 - sig(G[m][o])))
           for o in range(d_ff)] for m in range(M)]
    dU = [[dH[m][o] * G[m][o] * sig(G[m][o]) for o in range(d_ff)] for m in range(M)]

    def back(D, W, A, B, Hl):
        Gl = [[sum(D[m][o] * B[o][i] for o in range(d_ff)) for i in range(r)] for m in range(M)]
        dX = [[sum(D[m][o] * W[o][k] for o in range(d_ff)) +
               s * sum(Gl[m][i] * A[i][k] for i in range(r)) for k in range(d_in)] for m in range(M)]
        dA = [[s * sum(Gl[m][i] * X[m][k] for m in range(M)) for k in range(d_in)] for i in range(r)]
        dB = [[s * sum(D[m][o] * Hl[m][i] for m in range(M)) for i in range(r)] for o in range(d_ff)]
        return dX, dA, dB

    dXg, dAg, dBg = back(dG, Wg, Ag, Bg, Hg)
    dXu, dAu, dBu = back(dU, Wu, Au, Bu, Hu)
    dX = [[dXg[m][k] + dXu[m][k] for k in range(d_in)] for m in range(M)]
    return [np.array(v) for v in (G, U, H, dX, dAg, dBg, dAu, dBu)]


def pin_brute(seed=3, alpha=4.0):
    p = _problem(seed)
    ref = _brute(p, alpha)
    got = list(swiglu.forward(*_args(p), alpha)) + list(swiglu.backward(p["dH"], *_args(p), alpha))
    for g, e in zip(got, ref):
        assert np.allclose(g, e, rtol=1e-12, atol=1e-12)


def pin_fd(seed=4, alpha=6.0, h=1e-6):
    p = _problem(seed)
    dX, dAg, dBg, dAu, dBu = swiglu.backward(p["dH"], *_args(p), alpha)
    grads = dict(X=dX, Ag=dAg, Bg=dBg, Au=dAu, Bu=dBu)
    L = lambda q: swiglu.loss(q["dH"], *_args(q), alpha)
    for name, g in grads.items():
        for idx in np.ndindex(*g.shape):
            q = {k: v.copy() for k, v in p.items()}
            q[name][idx] += h
            lp = L(q)
            q[name][idx] -= 2 * h
            lm = L(q)
            assert abs((lp - lm) / (2 * h) - g[idx]) < 1e-6 * (1 + abs(g[idx])), (name, idx)


ALL_PINS = [pin_silu_values, pin_silu_fd, pin_plain_gates, pin_up_zero, pin_brute, pin_fd]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_adapter_grads_mm_agree_with_backward(seed=6, alpha=8.0):
    """The matmul route to the four adapter gradients agrees with the plain
    backward to float64 rounding."""
    rng = np.random.default_rng(seed)
    M, d_in, d_ff, r = 40, 24, 36, 5
    X = rng.standard_normal((M, d_in))
    Wg, Wu = rng.standard_normal((2, d_ff, d_in)) / 5
    Ag, Au = rng.standard_normal((2, r, d_in)) / 5
    Bg, Bu = rng.standard_normal((2, d_ff, r)) / 5
    dH = rng.standard_normal((M, d_ff))
    ref = swiglu.backward(dH, X, Wg, Ag, Bg, Wu, Au, Bu, alpha)[1:]
    got = swiglu.adapter_grads_mm(dH, X, Wg, Ag, Bg, Wu, Au, Bu, alpha)
    for g, e in zip(got, ref):
        np.testing.assert_allclose(g, e, rtol=0, atol=1e-12 * np.abs(e).max())


def test_sampled_rows_equal_full(seed=5, alpha=8.0):
    p = _problem(seed, M=9, d_in=10, d_ff=7, r=3)
    _, _, H = swiglu.forward(*_args(p), alpha)
    dX = swiglu.backward(p["dH"], *_args(p), alpha)[0]
    smp = swiglu.SampledRows(*_args(p), p["dH"], alpha)
    rows = np.array([0, 4, 8, 3])
    assert np.allclose(smp.h_rows(rows), H[rows], rtol=0, atol=1e-14)
    assert np.allclose(smp.dx_rows(rows), dX[rows], rtol=0, atol=1e-13)


# ---- mutants: each plausible slip must fail at least one pin -----------------

def _mut_dropped_term(z):
    return swiglu.sigmoid(z)  # silu' without the z sigma (1 - sigma) term


def _mut_d_up_uses_gate(dH, gate, up):
    d_gate = oracle._f64(dH) * up * swiglu.silu_grad(gate)
    return d_gate, oracle._f64(dH) * gate  # gate instead of silu(gate)


def _mut_swapped_projections(dH, X, Wg, Ag, Bg, Wu, Au, Bu, alpha, lib=None):
    gate, up, _ = swiglu.forward(X, Wg, Ag, Bg, Wu, Au, Bu, alpha, lib=lib)
    d_gate, d_up = swiglu.elementwise_backward(dH, gate, up)
    dXg, dAg, dBg = oracle.backward(d_up, X, Wg, Ag, Bg, alpha, lib=lib)  # swapped
    dXu, dAu, dBu = oracle.backward(d_gate, X, Wu, Au, Bu, alpha, lib=lib)
    return dXg + dXu, dAg, dBg, dAu, dBu


def _mut_sigmoid_on_up(X, Wg, Ag, Bg, Wu, Au, Bu, alpha, lib=None):
    _, gate = oracle.forward(X, Wg, Ag, Bg, alpha, lib=lib)
    _, up = oracle.forward(X, Wu, Au, Bu, alpha, lib=lib)
    return gate, up, gate * swiglu.sigmoid(up) * up


MUTANTS = [("silu_grad", _mut_dropped_term), ("elementwise_backward", _mut_d_up_uses_gate),
           ("backward", _mut_swapped_projections), ("forward", _mut_sigmoid_on_up)]


@pytest.mark.parametrize("name,fn", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(monkeypatch, name, fn):
    monkeypatch.setattr(swiglu, name, fn)
    failed = []
    for pin in ALL_PINS:
        try:
            pin()
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin catches the mutant of {name}"
