"""Pins of the fp64 oracle to facts outside itself (CPU only).

Every pin is a function of the loaded oracle library so that
`test_oracle_mutants.py` can run the same pins against copies of the oracle
with a planted mistake and check that each mistake is caught.

Pins (equation of ch05 "Acceleration principles: Triton kernels and fused
LoRA", §5.3, and of ch01 "Project background", §1.2; gradient list of ch05
§5.3):
  hand     : a hand-worked integer example (tests/golden/hand_worked_r2.json)
  fd       : central finite differences of L = <dY, Y> using only the forward;
             L is linear in X, in A and in B, so the difference quotient
             equals the gradient up to fp64 rounding for any step
  merged   : Y = X (W + s B A)^T and dX = dY (W + s B A), by numpy
  b_zero   : B = 0  =>  Y = X W^T, dA = 0 exactly, dB = s dY^T X A^T
  w_zero   : W = 0  =>  Y = s X A^T B^T, dX = s dY B A
  identity : r = d_in = d_out, A = B = I  =>  Y = X W^T + s X
  integers : small-integer inputs, exact equality with int64 numpy matmuls
  brute    : numpy fp64 matmuls on random tiny inputs, every output
  transpose: dX(dY; W, A, B) == Y(X:=dY; W:=W^T, A:=B^T, B:=A^T) bit for bit
  sampled  : the sampled routines equal the full ones bit for bit
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_r2.json")


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _problem(seed, M=5, d_in=7, d_out=6, r=3):
    rng = np.random.default_rng(seed)
    return dict(X=_rand(rng, M, d_in), W=_rand(rng, d_out, d_in),
                A=_rand(rng, r, d_in), B=_rand(rng, d_out, r),
                dY=_rand(rng, M, d_out))


# ---- pins as functions of the library --------------------------------------

def pin_hand(lib):
    g = json.load(open(GOLDEN))
    X, W, A, B, dY = (np.array(g[k], dtype=np.float64) for k in ("X", "W", "A", "B", "dY"))
    e = g["expected"]
    H, Y = oracle.forward(X, W, A, B, g["alpha"], lib=lib)
    dX, dA, dB = oracle.backward(dY, X, W, A, B, g["alpha"], lib=lib)
    assert np.array_equal(H, np.array(e["H"], dtype=np.float64))
    assert np.array_equal(Y, np.array(e["Y"], dtype=np.float64))
    assert np.array_equal(dX, np.array(e["dX"], dtype=np.float64))
    assert np.array_equal(dA, np.array(e["dA"], dtype=np.float64))
    assert np.array_equal(dB, np.array(e["dB"], dtype=np.float64))
    assert oracle.loss(dY, X, W, A, B, g["alpha"], lib=lib) == e["L"]


def pin_fd(lib, seed=1, alpha=6.0):
    p = _problem(seed)
    X, W, A, B, dY = p["X"], p["W"], p["A"], p["B"], p["dY"]
    dX, dA, dB = oracle.backward(dY, X, W, A, B, alpha, lib=lib)
    h = 0.5

    def L(**kw):
        q = dict(X=X, W=W, A=A, B=B)
        q.update(kw)
        return oracle.loss(dY, q["X"], q["W"], q["A"], q["B"], alpha, lib=lib)

    for name, T, grad in (("X", X, dX), ("A", A, dA), ("B", B, dB)):
        fd = np.empty_like(T)
        for idx in np.ndindex(T.shape):
            Tp = T.copy(); Tp[idx] += h
            Tm = T.copy(); Tm[idx] -= h
            fd[idx] = (L(**{name: Tp}) - L(**{name: Tm})) / (2 * h)
        scale = max(1.0, np.abs(grad).max())
        assert np.abs(fd - grad).max() <= 1e-10 * scale, name


def pin_merged(lib, seed=2, alpha=12.0):
    p = _problem(seed, M=9, d_in=11, d_out=10, r=4)
    X, W, A, B, dY = p["X"], p["W"], p["A"], p["B"], p["dY"]
    s = alpha / 4
    Wm = W + s * (B @ A)
    _, Y = oracle.forward(X, W, A, B, alpha, lib=lib)
    dX, _, _ = oracle.backward(dY, X, W, A, B, alpha, lib=lib)
    np.testing.assert_allclose(Y, X @ Wm.T, rtol=0, atol=1e-12 * np.abs(Y).max())
    np.testing.assert_allclose(dX, dY @ Wm, rtol=0, atol=1e-12 * np.abs(dX).max())


def pin_b_zero(lib, seed=3, alpha=8.0):
    p = _problem(seed, M=6, d_in=9, d_out=7, r=2)
    X, W, A, dY = p["X"], p["W"], p["A"], p["dY"]
    B = np.zeros((7, 2))
    s = alpha / 2
    _, Y = oracle.forward(X, W, A, B, alpha, lib=lib)
    dX, dA, dB = oracle.backward(dY, X, W, A, B, alpha, lib=lib)
    np.testing.assert_allclose(Y, X @ W.T, rtol=0, atol=1e-12 * np.abs(Y).max())
    np.testing.assert_allclose(dX, dY @ W, rtol=0, atol=1e-12 * np.abs(dX).max())
    assert np.all(dA == 0.0)
    ref = s * dY.T @ (X @ A.T)
    np.testing.assert_allclose(dB, ref, rtol=0, atol=1e-12 * np.abs(ref).max())


def pin_w_zero(lib, seed=4, alpha=3.0):
    p = _problem(seed, M=4, d_in=8, d_out=5, r=3)
    X, A, B, dY = p["X"], p["A"], p["B"], p["dY"]
    W = np.zeros((5, 8))
    s = alpha / 3
    _, Y = oracle.forward(X, W, A, B, alpha, lib=lib)
    dX, _, _ = oracle.backward(dY, X, W, A, B, alpha, lib=lib)
    refY = s * (X @ A.T) @ B.T
    refX = s * (dY @ B) @ A
    np.testing.assert_allclose(Y, refY, rtol=0, atol=1e-12 * np.abs(refY).max())
    np.testing.assert_allclose(dX, refX, rtol=0, atol=1e-12 * np.abs(refX).max())


def pin_identity(lib, seed=5, alpha=10.0):
    d = 6
    p = _problem(seed, M=4, d_in=d, d_out=d, r=d)
    X, W = p["X"], p["W"]
    I = np.eye(d)
    s = alpha / d
    _, Y = oracle.forward(X, W, I, I, alpha, lib=lib)
    ref = X @ W.T + s * X
    np.testing.assert_allclose(Y, ref, rtol=0, atol=1e-12 * np.abs(ref).max())


def pin_integers(lib, seed=6):
    rng = np.random.default_rng(seed)
    M, d_in, d_out, r = 7, 12, 9, 4
    Xi = rng.integers(-3, 4, (M, d_in))
    Wi = rng.integers(-3, 4, (d_out, d_in))
    Ai = rng.integers(-3, 4, (r, d_in))
    Bi = rng.integers(-3, 4, (d_out, r))
    dYi = rng.integers(-3, 4, (M, d_out))
    alpha = 8.0  # s = 2
    H, Y = oracle.forward(Xi, Wi, Ai, Bi, alpha, lib=lib)
    dX, dA, dB = oracle.backward(dYi, Xi, Wi, Ai, Bi, alpha, lib=lib)
    Hi = Xi @ Ai.T
    Gi = dYi @ Bi
    assert np.array_equal(H, Hi.astype(np.float64))
    assert np.array_equal(Y, (Xi @ Wi.T + 2 * Hi @ Bi.T).astype(np.float64))
    assert np.array_equal(dX, (dYi @ Wi + 2 * Gi @ Ai).astype(np.float64))
    assert np.array_equal(dA, (2 * Gi.T @ Xi).astype(np.float64))
    assert np.array_equal(dB, (2 * dYi.T @ Hi).astype(np.float64))


def pin_brute(lib, seed=7, alpha=5.0):
    p = _problem(seed, M=13, d_in=17, d_out=11, r=5)
    X, W, A, B, dY = p["X"], p["W"], p["A"], p["B"], p["dY"]
    s = alpha / 5
    H, Y = oracle.forward(X, W, A, B, alpha, lib=lib)
    dX, dA, dB = oracle.backward(dY, X, W, A, B, alpha, lib=lib)
    Hn = X @ A.T
    Gn = dY @ B
    for got, ref in ((H, Hn), (Y, X @ W.T + s * Hn @ B.T), (dX, dY @ W + s * Gn @ A),
                     (dA, s * Gn.T @ X), (dB, s * dY.T @ Hn)):
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12 * np.abs(ref).max())


def pin_transpose(lib, seed=8, alpha=7.0):
    p = _problem(seed, M=6, d_in=9, d_out=8, r=3)
    X, W, A, B, dY = p["X"], p["W"], p["A"], p["B"], p["dY"]
    dX, _, _ = oracle.backward(dY, X, W, A, B, alpha, lib=lib)
    _, Yt = oracle.forward(dY, np.ascontiguousarray(W.T), np.ascontiguousarray(B.T),
                           np.ascontiguousarray(A.T), alpha, lib=lib)
    assert np.array_equal(dX, Yt)


ALL_PINS = [pin_hand, pin_fd, pin_merged, pin_b_zero, pin_w_zero, pin_identity,
            pin_integers, pin_brute, pin_transpose]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.load())


def test_sampled_equals_full():
    p = _problem(9, M=37, d_in=24, d_out=40, r=8)
    X, W, A, B, dY = p["X"], p["W"], p["A"], p["B"], p["dY"]
    alpha = 16.0
    _, Y = oracle.forward(X, W, A, B, alpha)
    dX, dA, dB = oracle.backward(dY, X, W, A, B, alpha)
    S = oracle.Sampled(X, W, A, B, dY, alpha)
    rows = [0, 5, 36, 17]
    assert np.array_equal(S.y_rows(rows), Y[rows])
    assert np.array_equal(S.dx_rows(rows), dX[rows])
    ii, kk = [0, 7, 3, 3], [0, 23, 11, 2]
    assert np.array_equal(S.da_entries(ii, kk), dA[ii, kk])
    oo, jj = [0, 39, 20, 20], [7, 0, 4, 5]
    assert np.array_equal(S.db_entries(oo, jj), dB[oo, jj])
    assert np.array_equal(S.dA(), dA) and np.array_equal(S.dB(), dB)
    # columns computed on demand (no full H/G) give the same bits
    S2 = oracle.Sampled(X, W, A, B, dY, alpha)
    assert np.array_equal(S2.da_entries(ii, kk), dA[ii, kk])
    assert np.array_equal(S2.db_entries(oo, jj), dB[oo, jj])


def test_full_skinny_routines_equal_the_full_backward():
    """Sampled.G/dA/dB read transposed copies through the H routine: every
    element is the same sum in the same order, so the bits match the
    backward's own G, dA and dB routines."""
    p = _problem(11, M=45, d_in=33, d_out=50, r=7)
    X, W, A, B, dY = p["X"], p["W"], p["A"], p["B"], p["dY"]
    alpha = 12.0
    dX, dA, dB = oracle.backward(dY, X, W, A, B, alpha)
    S = oracle.Sampled(X, W, A, B, dY, alpha)
    lib = oracle.load()
    G = np.empty((45, 7))
    lib.lora_oracle_g(oracle._p(np.ascontiguousarray(dY)), oracle._p(np.ascontiguousarray(B)),
                      45, 50, 7, oracle._p(G))
    assert np.array_equal(S.G(), G)
    assert np.array_equal(S.dA(), dA)
    assert np.array_equal(S.dB(), dB)


def test_matmul_rows_agree_with_the_loops():
    """The frozen-W products taken by numpy's matmul agree with the plain
    loops to float64 rounding (they differ only in summation order)."""
    p = _problem(12, M=70, d_in=300, d_out=260, r=9)
    X, W, A, B, dY = p["X"], p["W"], p["A"], p["B"], p["dY"]
    alpha = 18.0
    _, Y = oracle.forward(X, W, A, B, alpha)
    dX, _, _ = oracle.backward(dY, X, W, A, B, alpha)
    for all_rows in (False, True):
        S = oracle.Sampled(X, W, A, B, dY, alpha)
        if all_rows:  # full H and G cached first
            S.H(), S.G()
        rows = np.arange(70) if all_rows else np.array([0, 3, 69, 40])
        np.testing.assert_allclose(S.y_rows_mm(rows), Y[rows], rtol=0,
                                   atol=1e-13 * np.abs(Y).max())
        np.testing.assert_allclose(S.dx_rows_mm(rows), dX[rows], rtol=0,
                                   atol=1e-13 * np.abs(dX).max())


def test_empty_batch():
    """M = 0: no tokens; Y and dX are empty and dA = dB = 0 (empty sums)."""
    p = _problem(10, M=1, d_in=8, d_out=8, r=2)
    X = np.zeros((0, 8)); dY = np.zeros((0, 8))
    H, Y = oracle.forward(X, p["W"], p["A"], p["B"], 4.0)
    dX, dA, dB = oracle.backward(dY, X, p["W"], p["A"], p["B"], 4.0)
    assert Y.shape == (0, 8) and dX.shape == (0, 8)
    assert np.all(dA == 0) and np.all(dB == 0)
