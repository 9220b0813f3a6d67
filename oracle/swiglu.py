"""fp64 CPU oracle of the SwiGLU gate/up pair of LoRA layers -- TEST INFRASTRUCTURE.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of
`bench.py` may import this module.  The CUDA path never does.

What it computes (ch05 "Acceleration principles: Triton kernels and fused
LoRA", §5.6 fused SwiGLU: SwiGLU(x) = (W_g x * sigma(W_g x)) * W_u x, three
matrix products with a SiLU and an elementwise product in between, the SiLU
and the product fused into the matmul epilogue), with each of the gate and up
projections a LoRA layer of §5.3 with the same rank r and scale s = alpha / r,
rows of X being tokens:

    gate = X Wg^T + s (X Ag^T) Bg^T          up = X Wu^T + s (X Au^T) Bu^T
    H    = silu(gate) * up,  silu(z) = z sigma(z),  sigma(z) = 1 / (1 + e^-z)

Backward for the loss L = <dH, H> (dH the upstream gradient), by the chain
rule through the elementwise step, then each projection's LoRA backward:

    d_gate = dH * up * silu'(gate),   silu'(z) = sigma(z) (1 + z (1 - sigma(z)))
    d_up   = dH * silu(gate)
    dX     = d_gate Wg + s (d_gate Bg) Ag + d_up Wu + s (d_up Bu) Au
    dAg    = s (d_gate Bg)^T X            dBg = s d_gate^T (X Ag^T)
    dAu    = s (d_up Bu)^T X              dBu = s d_up^T (X Au^T)

The LoRA pieces are the pinned plain-loop routines of this package; the
elementwise steps are written out below in numpy float64.
"""
from __future__ import annotations

import numpy as np

from . import _f64, backward as lora_backward, forward as lora_forward, load, Sampled


def sigmoid(z):
    """sigma(z) = 1 / (1 + exp(-z)), written so that exp never overflows."""
    z = np.asarray(z, dtype=np.float64)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-z[pos]))
    ez = np.exp(z[~pos])
    out[~pos] = ez / (1.0 + ez)
    return out


def silu(z):
    """silu(z) = z sigma(z) (the SiLU of ch05 §5.6)."""
    z = np.asarray(z, dtype=np.float64)
    return z * sigmoid(z)


def silu_grad(z):
    """d silu / dz = sigma(z) + z sigma(z) (1 - sigma(z))."""
    z = np.asarray(z, dtype=np.float64)
    sg = sigmoid(z)
    return sg * (1.0 + z * (1.0 - sg))


def forward(X, Wg, Ag, Bg, Wu, Au, Bu, alpha: float, lib=None):
    """Returns (gate, up, H) as float64 arrays."""
    lib = lib or load()
    _, gate = lora_forward(X, Wg, Ag, Bg, alpha, lib=lib)
    _, up = lora_forward(X, Wu, Au, Bu, alpha, lib=lib)
    return gate, up, silu(gate) * up


def elementwise_backward(dH, gate, up):
    """(d_gate, d_up) from the upstream dH and the two pre-activations."""
    dH = _f64(dH)
    return dH * up * silu_grad(gate), dH * silu(gate)


def backward(dH, X, Wg, Ag, Bg, Wu, Au, Bu, alpha: float, lib=None):
    """Returns (dX, dAg, dBg, dAu, dBu) as float64 arrays for L = <dH, H>."""
    lib = lib or load()
    gate, up, _ = forward(X, Wg, Ag, Bg, Wu, Au, Bu, alpha, lib=lib)
    d_gate, d_up = elementwise_backward(dH, gate, up)
    dXg, dAg, dBg = lora_backward(d_gate, X, Wg, Ag, Bg, alpha, lib=lib)
    dXu, dAu, dBu = lora_backward(d_up, X, Wu, Au, Bu, alpha, lib=lib)
    return dXg + dXu, dAg, dBg, dAu, dBu


def adapter_grads_mm(dH, X, Wg, Ag, Bg, Wu, Au, Bu, alpha: float, lib=None):
    """(dAg, dBg, dAu, dBu) as backward() defines them, for shapes where the
    plain loops would take minutes: gate and up take their frozen-weight
    products X Wg^T and X Wu^T from numpy's float64 matmul (a library GEMM as
    one step, summing in its own order); the low-rank terms, the elementwise
    step and the adapter gradients are the plain routines."""
    lib = lib or load()
    X = _f64(X)
    out = []
    pre = []
    for W, A, B in ((Wg, Ag, Bg), (Wu, Au, Bu)):
        smp = Sampled(X, W, A, B, None, alpha, lib=lib)
        pre.append(X @ smp.W.T + smp.s * (smp.H() @ smp.B.T))
    d_gate, d_up = elementwise_backward(dH, pre[0], pre[1])
    for d, W, A, B in ((d_gate, Wg, Ag, Bg), (d_up, Wu, Au, Bu)):
        smp = Sampled(X, W, A, B, d, alpha, lib=lib)
        out += [smp.dA(), smp.dB()]
    return tuple(out)


def loss(dH, X, Wg, Ag, Bg, Wu, Au, Bu, alpha: float, lib=None) -> float:
    """L = <dH, H> from the oracle's forward (sum in fp64)."""
    _, _, H = forward(X, Wg, Ag, Bg, Wu, Au, Bu, alpha, lib=lib)
    return float(np.sum(_f64(dH) * H))


class SampledRows:
    """H and dX of chosen token rows of a large problem (the same per-row sums
    as the full routines).  dA and dB depend on every row and are not offered."""

    def __init__(self, X, Wg, Ag, Bg, Wu, Au, Bu, dH, alpha: float, lib=None):
        self.lib = lib or load()
        self.alpha = alpha
        self.g = Sampled(X, Wg, Ag, Bg, None, alpha, lib=self.lib)
        self.u = Sampled(X, Wu, Au, Bu, None, alpha, lib=self.lib)
        self.dH = _f64(dH) if dH is not None else None
        self.X = self.g.X
        self.W = (self.g.W, self.u.W)
        self.A = (self.g.A, self.u.A)
        self.B = (self.g.B, self.u.B)

    def gate_up_rows(self, rows):
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        return self.g.y_rows(rows), self.u.y_rows(rows)

    def h_rows(self, rows):
        gate, up = self.gate_up_rows(rows)
        return silu(gate) * up

    def h_rows_mm(self, rows):
        """h_rows with the frozen-W products from numpy's matmul."""
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        return silu(self.g.y_rows_mm(rows)) * self.u.y_rows_mm(rows)

    def dx_rows_mm(self, rows):
        """dx_rows with the frozen-W products from numpy's matmul."""
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        gate, up = self.g.y_rows_mm(rows), self.u.y_rows_mm(rows)
        d_gate, d_up = elementwise_backward(self.dH[rows], gate, up)
        Xs = np.ascontiguousarray(self.X[rows])
        local = np.arange(len(rows), dtype=np.int64)
        out = np.zeros((len(rows), self.X.shape[1]))
        for d, W, A, B in ((d_gate, self.W[0], self.A[0], self.B[0]),
                           (d_up, self.W[1], self.A[1], self.B[1])):
            out += Sampled(Xs, W, A, B, d, self.alpha, lib=self.lib).dx_rows_mm(local)
        return out

    def dx_rows(self, rows):
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        gate, up = self.gate_up_rows(rows)
        d_gate, d_up = elementwise_backward(self.dH[rows], gate, up)
        # dX of a row needs only that row of d_gate / d_up: run the LoRA dX
        # routine on the sampled rows alone
        Xs = np.ascontiguousarray(self.X[rows])
        local = np.arange(len(rows), dtype=np.int64)
        out = np.zeros((len(rows), self.X.shape[1]))
        for d, W, A, B in ((d_gate, self.W[0], self.A[0], self.B[0]),
                           (d_up, self.W[1], self.A[1], self.B[1])):
            out += Sampled(Xs, W, A, B, d, self.alpha, lib=self.lib).dx_rows(local)
        return out
