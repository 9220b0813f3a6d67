"""Pins of the fp8 frozen-W oracle (oracle/fp8.py) to facts outside itself
(CPU only).

  decode    : the value of each of the 256 e4m3 codes equals PyTorch's
              float8_e4m3fn reading of the same byte
  encode    : rounding random in-range values agrees with PyTorch's
              float32 -> float8_e4m3fn conversion, byte for byte
  roundtrip : every finite value encodes back to its own code
  ties      : the midpoint of two neighbouring values goes to the even code
  saturate  : values above 448 give the largest finite code
  scale     : the exponent is the smallest e with amax <= 448 * 2^e, on
              hand-picked boundary values
  lossless  : small-integer X, W, dY are quantised without loss, so the fp8
              layer equals the plain LoRA oracle (itself pinned)
  hand      : a 2-token example worked out by hand
              (tests/golden/fp8_hand_worked.json) whose X, W and dY round in
              e4m3 (ties included) and whose small entries fall into the
              subnormal range under a per-tensor scale but not under a
              per-row one: it fixes that W is quantised with one tensor scale,
              X and dY with one scale per row, and that the low-rank terms and
              the adapter gradients use the unquantised inputs
Each planted mutant below fails at least one pin.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8


def pin_decode():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = fp8.e4m3_decode(np.arange(256))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def pin_encode(seed=0):
    rng = np.random.default_rng(seed)
    x = np.concatenate([rng.uniform(-448, 448, 4000),
                        rng.standard_normal(4000) * 0.05,
                        rng.standard_normal(2000) * 2.0 ** -8]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.e4m3_encode(x.astype(np.float64)), ref)


def pin_roundtrip():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    assert np.array_equal(fp8.e4m3_encode(fp8.e4m3_decode(codes)), codes.astype(np.uint8))


def pin_ties():
    v = fp8.e4m3_decode(np.arange(0x7F))
    mid = (v[:-1] + v[1:]) / 2
    codes = fp8.e4m3_encode(mid)
    lo = np.arange(0x7E)
    expect = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(codes, expect.astype(np.uint8))


def pin_saturate():
    assert list(fp8.e4m3_encode(np.array([448.0, 464.0, 1000.0, -1e6]))) == [0x7E, 0x7E, 0x7E, 0xFE]


def pin_scale():
    a = np.array([448.0, 448.5, 224.0, 224.1, 1.0, 0.0, 896.0, 3.5])
    # 448*2^0 >= 448; 448.5 needs 2^1; 224 = 448*2^-1; 224.1 needs 2^0;
    # 1 <= 448*2^-8 = 1.75 but not 0.875; 0 -> 0; 896 = 448*2; 3.5 = 448*2^-7
    assert list(fp8.pow2_scale_exponent(a)) == [0, 1, -1, 0, -8, 0, 1, -7]


def pin_lossless(seed=1, alpha=8.0):
    rng = np.random.default_rng(seed)
    M, d_in, d_out, r = 6, 9, 5, 3
    X = rng.integers(-15, 16, (M, d_in)).astype(np.float64)
    W = rng.integers(-15, 16, (d_out, d_in)).astype(np.float64)
    A = rng.standard_normal((r, d_in))
    B = rng.standard_normal((d_out, r))
    dY = rng.integers(-15, 16, (M, d_out)).astype(np.float64)
    H, Y = fp8.forward(X, W, A, B, alpha)
    H0, Y0 = oracle.forward(X, W, A, B, alpha)
    assert np.allclose(H, H0, rtol=1e-14, atol=1e-12)
    assert np.allclose(Y, Y0, rtol=1e-13, atol=1e-11)
    for g, e in zip(fp8.backward(dY, X, W, A, B, alpha), oracle.backward(dY, X, W, A, B, alpha)):
        assert np.allclose(g, e, rtol=1e-13, atol=1e-11)


GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fp8_hand_worked.json")


def _exact(values, shape=None):
    a = np.array([float(Fraction(v)) for v in values], dtype=np.float64)
    return a.reshape(shape) if shape is not None else a


def pin_hand():
    g = json.load(open(GOLDEN))
    sh = g["shapes"]
    X, W, A, B, dY = (_exact(g[k], sh[k]) for k in ("X", "W", "A", "B", "dY"))
    e = g["expected"]
    alpha = g["alpha"]
    wq, ws = fp8.quantize_tensor(W)
    assert list(wq.reshape(-1)) == e["W_codes"]
    assert np.array_equal(np.asarray(ws), np.float64(Fraction(e["W_scale"])))
    for x, codes, scales in ((X, "X_codes", "X_scales"), (dY, "dY_codes", "dY_scales")):
        q, sc = fp8.quantize_rows(x)
        assert list(q.reshape(-1)) == e[codes]
        assert np.array_equal(sc, _exact(e[scales]))
    H, Y = fp8.forward(X, W, A, B, alpha)
    assert np.array_equal(H.reshape(-1), _exact(e["H"]))
    assert np.array_equal(Y, _exact(e["Y"], (2, 2)))
    dX, dA, dB = fp8.backward(dY, X, W, A, B, alpha)
    assert np.array_equal(dX, _exact(e["dX"], (2, 2)))
    assert np.array_equal(dA, _exact(e["dA"], (1, 2)))
    assert np.array_equal(dB, _exact(e["dB"], (2, 1)))


ALL_PINS = [pin_decode, pin_encode, pin_roundtrip, pin_ties, pin_saturate, pin_scale,
            pin_lossless, pin_hand]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_quantize_rows_bounds(seed=2):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((50, 300)) * np.exp(rng.uniform(-8, 8, (50, 1)))
    codes, scale = fp8.quantize_rows(x)
    amax = np.abs(x).max(axis=1)
    assert np.all(amax <= 448 * scale) and np.all(amax > 224 * scale)
    err = np.abs(fp8.dequant_rows(codes, scale) - x)
    assert np.all(err <= (2.0 ** -4) * np.abs(x) + 2.0 ** -10 * scale[:, None])


# ---- mutants ----------------------------------------------------------------

def _mut_ties_away(x):
    x = np.asarray(x, dtype=np.float64)
    flat = x.reshape(-1)
    v = fp8._POS_VALUES
    a = np.minimum(np.abs(flat), 448.0)
    dist = np.abs(v[None, :] - a[:, None])
    best = np.argmin(dist[:, ::-1], axis=1)  # ties go to the larger value
    code = len(v) - 1 - best
    return (code | np.where(np.signbit(flat), 0x80, 0)).astype(np.uint8).reshape(x.shape)


def _mut_scale_off_by_one(amax):
    amax = np.asarray(amax, dtype=np.float64)
    m, k = np.frexp(amax)
    return np.where(amax > 0, k - 8, 0).astype(np.int64)


def _mut_bias8_decode(codes):
    c = np.asarray(codes, dtype=np.int64)
    e, m = (c >> 3) & 0xF, c & 7
    v = np.where(e == 0, m / 8 * 2.0 ** -7, (1 + m / 8) * 2.0 ** (e - 8))
    return np.where(c & 0x80, -v, v)


def _mut_forward_no_w_quant(X, W, A, B, alpha, lib=None):
    X, W, A, B = map(oracle._f64, (X, W, A, B))
    Xq, xs = fp8.quantize_rows(X)
    s = alpha / B.shape[1]
    return X @ A.T, fp8.dequant_rows(Xq, xs) @ W.T + s * (X @ A.T) @ B.T


def _mut_rows_one_scale(x):
    """X and dY quantised with one scale for the whole tensor."""
    x = oracle._f64(x)
    codes, scale = fp8.quantize_tensor(x)
    return codes, np.full(x.shape[0], scale)


def _mut_w_row_scales(w):
    """W quantised with one scale per row (a scale that the dX product,
    summed over d_out, could not factor out)."""
    codes, scales = fp8.quantize_rows(w)
    return codes, scales[:, None]


def _mut_backward_no_dy_quant(dY, X, W, A, B, alpha, lib=None):
    dY, X, W, A, B = map(oracle._f64, (dY, X, W, A, B))
    Wq, ws = fp8.quantize_tensor(W)
    s = alpha / B.shape[1]
    G, H = dY @ B, X @ A.T
    return dY @ (fp8.e4m3_decode(Wq) * ws) + s * G @ A, s * G.T @ X, s * dY.T @ H


def _mut_backward_quantised_grads(dY, X, W, A, B, alpha, lib=None):
    """dA and dB taken from the quantised X and dY."""
    dX, _, _ = _ORIG_BACKWARD(dY, X, W, A, B, alpha)
    dY, X, A, B = map(oracle._f64, (dY, X, A, B))
    Xd = fp8.dequant_rows(*fp8.quantize_rows(X))
    dYd = fp8.dequant_rows(*fp8.quantize_rows(dY))
    s = alpha / B.shape[1]
    G, H = dYd @ B, Xd @ A.T
    return dX, s * G.T @ Xd, s * dYd.T @ H


_ORIG_BACKWARD = fp8.backward

MUTANTS = [("e4m3_encode", _mut_ties_away), ("pow2_scale_exponent", _mut_scale_off_by_one),
           ("e4m3_decode", _mut_bias8_decode), ("forward", _mut_forward_no_w_quant),
           ("quantize_rows", _mut_rows_one_scale), ("quantize_tensor", _mut_w_row_scales),
           ("backward", _mut_backward_no_dy_quant),
           ("backward", _mut_backward_quantised_grads)]


@pytest.mark.parametrize("name,fn", MUTANTS, ids=[m[1].__name__ for m in MUTANTS])
def test_mutant_is_caught(monkeypatch, name, fn):
    monkeypatch.setattr(fp8, name, fn)
    failed = []
    for pin in ALL_PINS:
        try:
            pin()
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin catches the mutant of {name}"
