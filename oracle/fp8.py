"""fp64 CPU oracle of the LoRA layer with an fp8 frozen-W GEMM -- TEST INFRASTRUCTURE.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of
`bench.py` may import this module.  The CUDA path never does.

ch05 "Acceleration principles: Triton kernels and fused LoRA", §5.9 (fp8
mixed-precision training on fp8 tensor cores) applied to the frozen-weight
product of the LoRA layer of §5.3, with the low-rank extension kept in bf16.
The pages fix no format or scaling recipe; the reading taken here:

  * fp8 is OCP e4m3 (1 sign bit, 4 exponent bits with bias 7, 3 mantissa
    bits; largest finite value 448, subnormals m/8 * 2^-6, no infinities),
    rounding to nearest with ties to even, saturating to +-448.
  * Scales are powers of two, so dividing by a scale is exact and the only
    rounding is the one to e4m3: a block with absolute maximum a > 0 gets
    2^e with e the smallest integer such that a <= 448 * 2^e (a = 0: 2^0).
  * W has one scale for the whole tensor (its product is summed over d_in in
    the forward and over d_out in the backward, so only a tensor scale factors
    out of both); X (forward) and dY (backward) have one scale per row.

Equations (s = alpha / r; Q(.) = the quantised value, codes times scale):

    Y  = Q(X) Q(W)^T + s (X A^T) B^T
    dX = Q(dY) Q(W)  + s (dY B) A
    dA = s (dY B)^T X,   dB = s dY^T (X A^T)          (the bf16 inputs, unquantised)
"""
from __future__ import annotations

import numpy as np

from . import _f64, Sampled, load

E4M3_MAX = 448.0


def e4m3_values() -> np.ndarray:
    """Value of every code 0..255 (NaN for the two NaN codes), from the format."""
    out = np.empty(256)
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        e = (c >> 3) & 0xF
        m = c & 0x7
        if e == 0xF and m == 0x7:
            out[c] = np.nan
        elif e == 0:
            out[c] = sign * (m / 8.0) * 2.0 ** -6
        else:
            out[c] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


_VALUES = e4m3_values()
# the 127 non-negative finite values in increasing order, with their codes
_POS_CODES = np.array([c for c in range(0x7F)], dtype=np.int64)   # 0x00..0x7E
_POS_VALUES = _VALUES[_POS_CODES]


def e4m3_encode(x) -> np.ndarray:
    """Codes (uint8) of x rounded to nearest e4m3, ties to the even code,
    saturating to +-448, the sign bit kept.  x must be finite."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.searchsorted(_POS_VALUES, a, side="left")          # first value >= a
    hi = np.minimum(hi, len(_POS_VALUES) - 1)
    lo = np.maximum(hi - 1, 0)
    vhi, vlo = _POS_VALUES[hi], _POS_VALUES[lo]
    exact = vhi == a
    d_lo, d_hi = a - vlo, vhi - a
    pick_hi = exact | (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    code = _POS_CODES[idx]
    # rounding keeps the sign bit (negative values that round to zero give -0)
    return (code | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


def e4m3_decode(codes) -> np.ndarray:
    return _VALUES[np.asarray(codes, dtype=np.int64)]


def pow2_scale_exponent(amax) -> np.ndarray:
    """Smallest integer e with amax <= 448 * 2^e (0 where amax == 0)."""
    amax = np.asarray(amax, dtype=np.float64)
    m, k = np.frexp(amax)                  # amax = m 2^k, m in [0.5, 1)
    e = np.where(m <= 0.875, k - 9, k - 8)  # 448 = 0.875 * 2^9
    return np.where(amax > 0, e, 0).astype(np.int64)


def quantize_rows(x):
    """(codes [rows, cols] uint8, scales [rows] float64 powers of two)."""
    x = _f64(x)
    e = pow2_scale_exponent(np.abs(x).max(axis=1) if x.shape[1] else np.zeros(x.shape[0]))
    scale = np.ldexp(1.0, e)
    return e4m3_encode(x / scale[:, None]), scale


def quantize_tensor(w):
    """(codes uint8, scale float64 power of two) with one scale for all of w."""
    w = _f64(w)
    e = int(pow2_scale_exponent(np.abs(w).max() if w.size else 0.0))
    scale = float(np.ldexp(1.0, e))
    return e4m3_encode(w / scale), scale


def dequant_rows(codes, scale):
    return e4m3_decode(codes) * np.asarray(scale)[:, None]


def forward(X, W, A, B, alpha: float, lib=None):
    """Returns (H, Y): H = X A^T in fp64, Y = Q(X) Q(W)^T + s H B^T."""
    lib = lib or load()
    X, W, A, B = map(_f64, (X, W, A, B))
    r = B.shape[1]
    s = float(alpha) / r
    Wq, w_scale = quantize_tensor(W)
    Xq, x_scale = quantize_rows(X)
    Wd = e4m3_decode(Wq) * w_scale
    Xd = dequant_rows(Xq, x_scale)
    smp = Sampled(X, W, A, B, None, alpha, lib=lib)
    H = smp.H()
    return H, Xd @ Wd.T + s * (H @ B.T)


def backward(dY, X, W, A, B, alpha: float, lib=None):
    """Returns (dX, dA, dB)."""
    lib = lib or load()
    dY, X, W, A, B = map(_f64, (dY, X, W, A, B))
    r = B.shape[1]
    s = float(alpha) / r
    Wq, w_scale = quantize_tensor(W)
    dYq, dy_scale = quantize_rows(dY)
    Wd = e4m3_decode(Wq) * w_scale
    dYd = dequant_rows(dYq, dy_scale)
    smp = Sampled(X, W, A, B, dY, alpha, lib=lib)
    G, H = smp.G(), smp.H()
    dX = dYd @ Wd + s * (G @ A)
    return dX, s * (G.T @ X), s * (dY.T @ H)


class SampledRows:
    """Rows of Y and dX, and all of dA and dB, of a large problem: the same
    definitions as forward() and backward() (per-row scales of X and dY are
    those of the sampled rows alone; W's tensor scale needs all of W)."""

    def __init__(self, X, W, A, B, dY, alpha: float, lib=None):
        self.lib = lib or load()
        self.smp = Sampled(X, W, A, B, dY, alpha, lib=self.lib)
        self.s = self.smp.s
        Wq, w_scale = quantize_tensor(self.smp.W)
        self.Wd = e4m3_decode(Wq) * w_scale

    def y_rows(self, rows) -> np.ndarray:
        rows = np.asarray(rows, dtype=np.int64)
        Xd = dequant_rows(*quantize_rows(self.smp.X[rows]))
        return Xd @ self.Wd.T + self.s * (self.smp.H()[rows] @ self.smp.B.T)

    def dx_rows(self, rows) -> np.ndarray:
        rows = np.asarray(rows, dtype=np.int64)
        dYd = dequant_rows(*quantize_rows(self.smp.dY[rows]))
        return dYd @ self.Wd + self.s * (self.smp.G()[rows] @ self.smp.A)

    def dA(self) -> np.ndarray:
        return self.smp.dA()

    def dB(self) -> np.ndarray:
        return self.smp.dB()
