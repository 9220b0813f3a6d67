"""fp64 CPU oracle of the LoRA layer over a 4-bit frozen W -- TEST INFRASTRUCTURE.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of
`bench.py` may import this module.  The CUDA path never does.

The Unsloth inference notes ("4-bit quantisation with in-register
dequantisation": weights fetched from HBM in a compact INT4 / FP4 format,
turned back into FP16 / BF16 on chip with their scaling factors, then fed
to the tensor cores) applied to the frozen W of the LoRA layer of ch05
"Acceleration principles: Triton kernels and fused LoRA", §5.3 (QLoRA's
frozen 4-bit base weight).  The pages fix no layout; the reading taken here:

  * symmetric INT4: q in [-8, 7], stored as the code q + 8 in a nibble, two
    per byte, the even column in the low nibble;
  * one bf16 scale per group of 64 consecutive weights of a row of W
    (along d_in), scale = bf16(absmax / 7) (1 for an all-zero group), both
    divisions in fp32, bf16 rounding to nearest even;
  * q = clamp(rint(w / scale), -8, 7) in fp32, ties to even;
  * the dequantised weight is bf16((code - 8) * scale): the exact product
    rounded once to bf16, nearest even.

The layer is then the plain LoRA layer (the pinned oracle of this package)
on the dequantised W:
    Y  = X Wd^T + s (X A^T) B^T
    dX = dY Wd + s (dY B) A,   dA = s (dY B)^T X,   dB = s dY^T (X A^T)
"""
from __future__ import annotations

import numpy as np

from . import _f64, backward as lora_backward, forward as lora_forward, load, Sampled

GROUP = 64


def bf16_round(x) -> np.ndarray:
    """float32 values rounded to bf16 (nearest, ties to even), as float32."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).reshape(f.shape)


def quantize_w(W):
    """(codes [d_out, d_in] uint8 in 0..15, scales [d_out, d_in / 64] float32
    holding bf16 values)."""
    W = np.asarray(_f64(W), dtype=np.float32)  # bf16 inputs: exact in float32
    d_out, d_in = W.shape
    g = W.reshape(d_out, d_in // GROUP, GROUP)
    amax = np.abs(g).max(axis=2)
    scale = bf16_round(amax / np.float32(7.0))
    scale = np.where(scale == 0, np.float32(1.0), scale).astype(np.float32)
    q = np.rint(g / scale[:, :, None]).astype(np.float32)
    q = np.clip(q, -8, 7)
    return (q + 8).astype(np.uint8).reshape(d_out, d_in), scale


def pack(codes) -> np.ndarray:
    """[d_out, d_in] codes -> [d_out, d_in / 2] bytes, even column low."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def unpack(packed) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty((p.shape[0], p.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = p & 0xF
    out[:, 1::2] = p >> 4
    return out


def dequantize(codes, scales) -> np.ndarray:
    """bf16((code - 8) * scale) as float64 [d_out, d_in]."""
    c = np.asarray(codes, dtype=np.float32) - np.float32(8)
    s = np.repeat(np.asarray(scales, dtype=np.float32), GROUP, axis=1)
    return bf16_round(c * s).astype(np.float64)  # the product is exact in float32


def forward(X, codes, scales, A, B, alpha: float, lib=None):
    """Returns (H, Y) of the layer over the dequantised W."""
    return lora_forward(X, dequantize(codes, scales), A, B, alpha, lib=lib or load())


def backward(dY, X, codes, scales, A, B, alpha: float, lib=None):
    """Returns (dX, dA, dB) of the layer over the dequantised W."""
    return lora_backward(dY, X, dequantize(codes, scales), A, B, alpha, lib=lib or load())


def sampled(X, codes, scales, A, B, dY, alpha: float, lib=None) -> Sampled:
    """The plain oracle's sampled routines (rows of Y and dX, all of dA and
    dB) for the layer over the dequantised W."""
    return Sampled(X, dequantize(codes, scales), A, B, dY, alpha, lib=lib or load())
