"""The LoRA layer over a 4-bit frozen W, on the GPU vs the oracle (needs a GB300).

Quantisation is byte work: the packed codes and the bf16 scales must equal
the oracle's exactly, and so must the dequantised W (one rounding of an
exact product on both sides).  The layer's outputs are compared with
max|T_gpu - T_ref| / max|T_ref| <= 1e-2 against the oracle on the
dequantised W; small ragged shapes element by element, the 4096^2 q_proj
shape on one row of Y and dX in every 128-row m-tile and on all of dA and
dB.  The
dequantising GEMM must also give, bit for bit, what the bf16 layer gives on
the dequantised W: both run the same tiles in the same order, so any
difference is a wrong element of the expanded tile.
"""
import numpy as np
import pytest
import torch

from oracle import q4 as oq4
import rank_linear_gb300 as rl
from rank_linear_gb300.synth import make_inputs

pytestmark = pytest.mark.gpu

TOL = 1e-2
DEV = "cuda:0"


def rel_err(got, ref) -> float:
    if isinstance(got, torch.Tensor):
        got = got.detach().double().cpu().numpy()
    den = np.abs(ref).max()
    return float(np.abs(got - ref).max() / (den if den > 0 else 1.0))


def inputs(M, d_in, d_out, r, seed):
    t = make_inputs(M, d_in, d_out, r, "bf16", seed=seed)
    t["B"] = (t["B"].float() * 10).bfloat16()  # a low-rank term that matters
    return t


def run_gpu(t, alpha, need_dX=True, keep_saved=True):
    g = {k: v.to(DEV) for k, v in t.items()}
    qw = rl.quantize_w_q4(g["W"])
    Y, saved = rl.q4_forward(g["X"], qw, g["A"], g["B"], alpha)
    dX, dA, dB = rl.q4_backward(g["dY"], g["X"], qw, g["A"], g["B"], alpha,
                                saved if keep_saved else None, need_dX=need_dX)
    torch.cuda.synchronize()
    rl.device_status()
    return Y, dX, dA, dB


def test_quantisation_is_byte_exact():
    t = make_inputs(16, 1024, 1040, 16, "bf16", seed=3)
    W = (t["W"].float() * torch.linspace(0.01, 3.0, 1040)[:, None]).bfloat16()
    W[7, 64:128] = 0.0          # an all-zero group gets scale 1
    W[9, :64] = 1e-30           # a tiny group
    W[11, 5] = 7.0              # an exact multiple of the scale
    qw = rl.quantize_w_q4(W.to(DEV))
    torch.cuda.synchronize()
    codes, scales = oq4.quantize_w(W)
    assert np.array_equal(qw.codes.cpu().numpy(), oq4.pack(codes))
    got_scales = qw.scales.float().cpu().numpy()
    assert np.array_equal(got_scales, scales.T)


def test_dequantisation_is_byte_exact():
    t = make_inputs(16, 512, 264, 16, "bf16", seed=4)
    qw = rl.quantize_w_q4(t["W"].to(DEV))
    Wd = rl.dequantize_w_q4(qw)
    torch.cuda.synchronize()
    codes, scales = oq4.quantize_w(t["W"])
    assert np.array_equal(Wd.double().cpu().numpy(), oq4.dequantize(codes, scales))


# M, d_in, d_out, r, alpha (d_in a multiple of 64, d_out of 8)
SMALL = [
    (300, 384, 272, 16, 32.0),     # ragged M and N
    (129, 192, 264, 12, 24.0),     # d_out not a multiple of 16, r not of 8
    (1, 64, 64, 1, 2.0),           # one token, rank one, one K block
    (256, 512, 384, 256, 512.0),   # maximum rank
    (1000, 1024, 776, 64, 128.0),  # backward K (d_out) with a ragged last block
    (2048, 1536, 2560, 128, 256.0),
    (1024, 4096, 5120, 16, 32.0),  # both GEMMs' last waves split two ways
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s[:4])))
def test_small_against_oracle(shape):
    M, d_in, d_out, r, alpha = shape
    t = inputs(M, d_in, d_out, r, seed=sum(shape[:4]))
    got = run_gpu(t, alpha)
    codes, scales = oq4.quantize_w(t["W"])
    _, Yr = oq4.forward(t["X"], codes, scales, t["A"], t["B"], alpha)
    ref = (Yr,) + tuple(oq4.backward(t["dY"], t["X"], codes, scales, t["A"], t["B"], alpha))
    errs = {n: rel_err(g, e) for n, g, e in zip(("Y", "dX", "dA", "dB"), got, ref)}
    for n, e in errs.items():
        assert e <= TOL, f"{n}: {e:.3e} ({errs})"


@pytest.mark.parametrize("shape", [SMALL[0], SMALL[4], SMALL[6]],
                         ids=lambda s: "x".join(map(str, s[:4])))
def test_same_bits_as_the_bf16_layer_on_dequantised_w(shape):
    """The bf16 layer runs with 256 x 256 tiles here, the only width of the
    dequantising GEMM, so both run the same tiles and splits in the same
    order."""
    from rank_linear_gb300 import _lib
    M, d_in, d_out, r, alpha = shape
    t = inputs(M, d_in, d_out, r, seed=7 + sum(shape[:4]))
    g = {k: v.to(DEV) for k, v in t.items()}
    qw = rl.quantize_w_q4(g["W"])
    Wd = rl.dequantize_w_q4(qw)
    L = _lib.lib()
    _lib.check(L.lora_debug_gemm_width(256), "gemm width")
    try:
        Y4, s4 = rl.q4_forward(g["X"], qw, g["A"], g["B"], alpha)
        Y16, s16 = rl.forward(g["X"], Wd, g["A"], g["B"], alpha)
        dX4, _, _ = rl.q4_backward(g["dY"], g["X"], qw, g["A"], g["B"], alpha, s4)
        dX16, _, _ = rl.backward(g["dY"], g["X"], Wd, g["A"], g["B"], alpha, s16)
        torch.cuda.synchronize()
    finally:
        L.lora_debug_gemm_width(0)
    rl.device_status()
    assert torch.equal(Y4, Y16)
    assert torch.equal(dX4, dX16)


def test_q_proj_shape_full_size():
    """4096^2 q_proj shape: Y and dX on one row of every 128-row m-tile, all
    of dA and dB, against the oracle's sampled routines over its own
    quantisation of W."""
    M = d_in = d_out = 4096
    r, alpha = 16, 16.0
    t = inputs(M, d_in, d_out, r, seed=0)
    Y, dX, dA, dB = run_gpu(t, alpha)
    codes, scales = oq4.quantize_w(t["W"])
    S = oq4.sampled(t["X"], codes, scales, t["A"], t["B"], t["dY"], alpha)
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([[0, M - 1],
                                     np.arange(0, M, 128) + rng.integers(0, 128, M // 128)]))
    errs = {"Y": rel_err(Y[rows], S.y_rows_mm(rows)), "dX": rel_err(dX[rows], S.dx_rows_mm(rows)),
            "dA": rel_err(dA, S.dA()), "dB": rel_err(dB, S.dB())}
    for k, e in errs.items():
        assert e <= TOL, f"{k}: {e:.3e} ({errs})"


def test_recompute_without_saved_and_without_dX():
    t = inputs(500, 512, 384, 24, seed=11)
    a = run_gpu(t, 48.0)
    b = run_gpu(t, 48.0, need_dX=False, keep_saved=False)
    assert b[1] is None
    for x, y in zip((a[0], a[2], a[3]), (b[0], b[2], b[3])):
        assert torch.equal(x, y)


def test_deterministic():
    t = inputs(1000, 1024, 768, 64, seed=5)
    a = run_gpu(t, 128.0)
    b = run_gpu(t, 128.0)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_no_tokens():
    t = inputs(0, 256, 128, 8, seed=6)
    Y, dX, dA, dB = run_gpu(t, 16.0)
    assert Y.shape == (0, 128) and dX.shape == (0, 256)
    assert not dA.abs().any() and not dB.abs().any()


def test_rejects_d_in_not_a_multiple_of_64():
    W = torch.zeros(64, 96, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(RuntimeError, match="multiple of 64"):
        rl.quantize_w_q4(W)


def test_autograd_matches_the_explicit_calls():
    t = inputs(300, 256, 192, 16, seed=12)
    g = {k: v.to(DEV) for k, v in t.items()}
    qw = rl.quantize_w_q4(g["W"])
    X = g["X"].reshape(2, 150, 256).clone().requires_grad_(True)
    A = g["A"].clone().requires_grad_(True)
    B = g["B"].clone().requires_grad_(True)
    Y = rl.lora_linear_q4(X, qw, A, B, 32.0)
    Y.backward(g["dY"].reshape(2, 150, 192))
    Y2, saved = rl.q4_forward(g["X"], qw, g["A"], g["B"], 32.0)
    dX2, dA2, dB2 = rl.q4_backward(g["dY"], g["X"], qw, g["A"], g["B"], 32.0, saved)
    torch.cuda.synchronize()
    assert Y.shape == (2, 150, 192)
    assert torch.equal(Y.reshape(300, 192), Y2)
    assert torch.equal(X.grad.reshape(300, 256), dX2)
    assert torch.equal(A.grad, dA2) and torch.equal(B.grad, dB2)
