"""Pins of the 4-bit frozen-W oracle (oracle/q4.py) to facts outside itself
(CPU only).

  bf16     : bf16 rounding equals PyTorch's float32 -> bfloat16 conversion
  dequant  : the dequantised weight equals PyTorch's bfloat16 of the float32
             product (code - 8) * scale
  pack     : pack and unpack are inverse; byte = even code | odd code << 4
  lossless : W built from codes on power-of-two scales (each group holding a
             +-7 * scale entry) quantises back to itself, and the layer then
             equals the plain LoRA oracle (itself pinned) on that W
  bounds   : every group's absmax entry gets |q| = 7 and every entry is within
             half a scale step of its dequantised value (plus bf16 rounding)
Each planted mutant below fails at least one pin.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import q4


def pin_bf16(seed=0):
    rng = np.random.default_rng(seed)
    x = np.concatenate([rng.standard_normal(5000).astype(np.float32),
                        (rng.integers(0, 1 << 16, 2000) * 2.0 ** -8).astype(np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(q4.bf16_round(x), ref)


def pin_dequant(seed=1):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, (8, 128)).astype(np.uint8)
    scales = torch.from_numpy(rng.uniform(1e-3, 2.0, (8, 2)).astype(np.float32)).to(
        torch.bfloat16).float().numpy()
    prod = (codes.astype(np.float32) - 8) * np.repeat(scales, 64, axis=1)
    ref = torch.from_numpy(prod).to(torch.bfloat16).double().numpy()
    assert np.array_equal(q4.dequantize(codes, scales), ref)


def pin_pack(seed=2):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, (5, 64)).astype(np.uint8)
    packed = q4.pack(codes)
    assert packed.shape == (5, 32)
    assert int(packed[0, 0]) == int(codes[0, 0]) | (int(codes[0, 1]) << 4)
    assert np.array_equal(q4.unpack(packed), codes)


def pin_lossless(seed=3, alpha=8.0):
    rng = np.random.default_rng(seed)
    d_out, d_in, M, r = 6, 128, 5, 3
    q = rng.integers(-7, 8, (d_out, d_in)).astype(np.float64)
    q[:, ::64] = 7 * rng.choice([-1.0, 1.0], (d_out, d_in // 64))  # each group's absmax is 7
    e = rng.integers(-8, 3, (d_out, d_in // 64))
    W = q * np.repeat(np.ldexp(1.0, e), 64, axis=1)
    codes, scales = q4.quantize_w(W)
    assert np.array_equal(q4.dequantize(codes, scales), W)
    X = rng.standard_normal((M, d_in))
    A = rng.standard_normal((r, d_in))
    B = rng.standard_normal((d_out, r))
    dY = rng.standard_normal((M, d_out))
    _, Y = q4.forward(X, codes, scales, A, B, alpha)
    _, Y0 = oracle.forward(X, W, A, B, alpha)
    assert np.array_equal(Y, Y0)
    for g, e0 in zip(q4.backward(dY, X, codes, scales, A, B, alpha),
                     oracle.backward(dY, X, W, A, B, alpha)):
        assert np.array_equal(g, e0)


def pin_bounds(seed=4):
    rng = np.random.default_rng(seed)
    W = torch.from_numpy(rng.standard_normal((16, 256)) * np.exp(rng.uniform(-4, 4, (16, 1)))
                         ).to(torch.bfloat16).double().numpy()
    codes, scales = q4.quantize_w(W)
    qs = codes.astype(np.int64) - 8
    g = qs.reshape(16, 4, 64)
    wg = np.abs(W).reshape(16, 4, 64)
    top = np.take_along_axis(np.abs(g), wg.argmax(axis=2)[:, :, None], axis=2)
    assert np.all(top == 7)
    step = np.repeat(scales, 64, axis=1).astype(np.float64)
    err = np.abs(q4.dequantize(codes, scales) - W)
    assert np.all(err <= 0.5 * step * (1 + 2.0 ** -6) + np.abs(W) * 2.0 ** -8)


ALL_PINS = [pin_bf16, pin_dequant, pin_pack, pin_lossless, pin_bounds]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


# ---- mutants ----------------------------------------------------------------

def _mut_pack_swapped(codes):
    c = np.asarray(codes, dtype=np.uint8)
    return (c[:, 1::2] | (c[:, 0::2] << 4)).astype(np.uint8)


def _mut_dequant_unrounded(codes, scales):
    c = np.asarray(codes, dtype=np.float64) - 8
    return c * np.repeat(np.asarray(scales, dtype=np.float64), 64, axis=1) * (1 + 2.0 ** -12)


def _mut_scale_over_8(W):
    W = np.asarray(oracle._f64(W), dtype=np.float32)
    d_out, d_in = W.shape
    g = W.reshape(d_out, d_in // 64, 64)
    scale = q4.bf16_round(np.abs(g).max(axis=2) / np.float32(8.0))
    scale = np.where(scale == 0, np.float32(1.0), scale).astype(np.float32)
    q = np.clip(np.rint(g / scale[:, :, None]), -8, 7)
    return (q + 8).astype(np.uint8).reshape(d_out, d_in), scale


def _mut_bf16_truncates(x):
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    return (f.view(np.uint32) & 0xFFFF0000).view(np.float32)


MUTANTS = [("pack", _mut_pack_swapped), ("dequantize", _mut_dequant_unrounded),
           ("quantize_w", _mut_scale_over_8), ("bf16_round", _mut_bf16_truncates)]


@pytest.mark.parametrize("name,fn", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(monkeypatch, name, fn):
    monkeypatch.setattr(q4, name, fn)
    failed = []
    for pin in ALL_PINS:
        try:
            pin()
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin catches the mutant of {name}"
