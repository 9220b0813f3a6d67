"""The LoRA layer with an fp8 (e4m3) frozen-W product, on the GPU vs the
oracle (needs a GB300).

Quantisation is byte work: the codes and scales of W and of X's rows must
equal the oracle's exactly (both sides take every rounding decision in exact
arithmetic, the scales being powers of two).  The layer's outputs are
compared with max|T_gpu - T_ref| / max|T_ref| <= 1e-2, the oracle applying
the same quantisation; small ragged shapes element by element, the 4096^2
q_proj shape on one row of Y and dX in every 128-row m-tile and on all of dA
and dB.
"""
import numpy as np
import pytest
import torch

from oracle import fp8 as ofp8
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


def run_gpu(t, alpha, need_dX=True):
    g = {k: v.to(DEV) for k, v in t.items()}
    qw = rl.quantize_w_fp8(g["W"])
    Y, saved = rl.fp8_forward(g["X"], qw, g["A"], g["B"], alpha)
    dX, dA, dB = rl.fp8_backward(g["dY"], g["X"], qw, g["A"], g["B"], alpha, saved,
                                 need_dX=need_dX)
    torch.cuda.synchronize()
    rl.device_status()
    return Y, dX, dA, dB


def test_w_quantisation_is_byte_exact():
    t = make_inputs(64, 4096, 1040, 16, "bf16", seed=3)
    W = (t["W"].float() * torch.linspace(0.01, 3.0, 4096)).bfloat16()  # a wide range
    qw = rl.quantize_w_fp8(W.to(DEV))
    torch.cuda.synchronize()
    codes, scale = ofp8.quantize_tensor(W)
    assert np.array_equal(qw.Wq.cpu().numpy(), codes)
    assert np.array_equal(qw.WqT.cpu().numpy(), codes.T)
    assert float(qw.w_scale.item()) == scale


def test_row_quantisation_is_byte_exact():
    x = make_inputs(777, 1024, 16, 16, "bf16", seed=4)["X"]
    x = (x.float() * torch.exp(torch.linspace(-20, 20, 777))[:, None]).bfloat16()
    x[5] = 0.0  # an all-zero row gets scale 1
    q, scale = rl.quantize_rows_fp8(x.to(DEV))
    torch.cuda.synchronize()
    codes, ref_scale = ofp8.quantize_rows(x)
    assert np.array_equal(scale.cpu().numpy().astype(np.float64), ref_scale)
    assert np.array_equal(q.cpu().numpy(), codes)


# M, d_in, d_out, r, alpha (d_in, d_out multiples of 16)
SMALL = [
    (300, 384, 272, 16, 32.0),     # ragged M and N, K not a multiple of 128
    (129, 144, 272, 12, 24.0),     # r not a multiple of 8
    (1, 64, 64, 1, 2.0),           # one token, rank one
    (256, 512, 384, 256, 512.0),   # maximum rank
    (1000, 1024, 768, 64, 128.0),
    (2048, 1536, 2560, 128, 256.0),
    (1024, 4096, 5120, 16, 32.0),  # both GEMMs' last waves split two ways
]


@pytest.fixture
def gemm_width():
    """Forces the main GEMMs' tile width for one test, then restores the
    cost model's choice."""
    from rank_linear_gb300 import _lib
    L = _lib.lib()
    yield lambda w: _lib.check(L.lora_debug_gemm_width(w), "gemm width")
    L.lora_debug_gemm_width(0)


@pytest.mark.parametrize("width", [256, 512])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s[:4])))
def test_small_against_oracle(shape, width, gemm_width):
    """Both GEMMs with 256 x 256 pair tiles (tail split where it applies) and
    with 256 x 512 pair tiles."""
    gemm_width(width)
    M, d_in, d_out, r, alpha = shape
    t = inputs(M, d_in, d_out, r, seed=sum(shape[:4]))
    got = run_gpu(t, alpha)
    _, Yr = ofp8.forward(t["X"], t["W"], t["A"], t["B"], alpha)
    ref = (Yr,) + tuple(ofp8.backward(t["dY"], t["X"], t["W"], t["A"], t["B"], alpha))
    errs = {n: rel_err(g, e) for n, g, e in zip(("Y", "dX", "dA", "dB"), got, ref)}
    for n, e in errs.items():
        assert e <= TOL, f"{n}: {e:.3e} ({errs})"


def test_wide_tail_split_path(gemm_width):
    """M = 2000, d_in = 5888, d_out = 6000 with 256 x 512 tiles: each GEMM has
    8 x 12 = 96 tiles, so on 76 CTA pairs the last wave's 20 are split in two
    K ranges (e4m3 main segment, bf16 extension in the same accumulator, the
    row scale applied after the two partials are added).  Given the full
    workspace the results are bitwise repeatable and differ from the unsplit
    ones (minimal workspace); both agree with the oracle on every element."""
    gemm_width(512)
    M, d_in, d_out, r, alpha = 2000, 5888, 6000, 24, 48.0
    t = inputs(M, d_in, d_out, r, seed=23)
    g = {k: v.to(DEV) for k, v in t.items()}
    qw = rl.quantize_w_fp8(g["W"])
    rup = lambda n: (n + 255) // 256 * 256
    r_pad = 32
    fwd_min = rup(M * d_in) + rup(M * 4) + rup(d_out * r_pad * 2)
    bwd_min = (rup(M * d_out) + rup(M * 4) + rup(M * r_pad * 2) + rup(r_pad * M * 2)
               + rup(d_in * r_pad * 2))
    full = torch.empty(rl.fp8_workspace_bytes(M, d_in, d_out, r), dtype=torch.uint8, device=DEV)
    minimal = torch.empty(max(fwd_min, bwd_min), dtype=torch.uint8, device=DEV)
    assert full.numel() > minimal.numel()

    def run(ws):
        Y, saved = rl.fp8_forward(g["X"], qw, g["A"], g["B"], alpha, workspace=ws)
        dX, dA, dB = rl.fp8_backward(g["dY"], g["X"], qw, g["A"], g["B"], alpha, saved,
                                     workspace=ws)
        torch.cuda.synchronize()
        rl.device_status()
        return Y, dX, dA, dB

    s1, s2, u = run(full), run(full), run(minimal)
    for a, b in zip(s1, s2):
        assert torch.equal(a, b)
    assert not torch.equal(s1[0], u[0]) and not torch.equal(s1[1], u[1])  # the split ran
    _, Yr = ofp8.forward(t["X"], t["W"], t["A"], t["B"], alpha)
    ref = (Yr,) + tuple(ofp8.backward(t["dY"], t["X"], t["W"], t["A"], t["B"], alpha))
    for got in (s1, u):
        errs = {n: rel_err(x, e) for n, x, e in zip(("Y", "dX", "dA", "dB"), got, ref)}
        for n, e in errs.items():
            assert e <= TOL, f"{n}: {e:.3e} ({errs})"


def test_q_proj_shape_full_size():
    """4096^2 q_proj shape: Y and dX on one row of every 128-row m-tile, all
    of dA and dB, against the oracle's sampled routines."""
    M = d_in = d_out = 4096
    r, alpha = 16, 16.0
    t = inputs(M, d_in, d_out, r, seed=0)
    Y, dX, dA, dB = run_gpu(t, alpha)
    S = ofp8.SampledRows(t["X"], t["W"], t["A"], t["B"], t["dY"], alpha)
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([[0, M - 1],
                                     np.arange(0, M, 128) + rng.integers(0, 128, M // 128)]))
    errs = {"Y": rel_err(Y[rows], S.y_rows(rows)), "dX": rel_err(dX[rows], S.dx_rows(rows)),
            "dA": rel_err(dA, S.dA()), "dB": rel_err(dB, S.dB())}
    for k, e in errs.items():
        assert e <= TOL, f"{k}: {e:.3e} ({errs})"


def test_deterministic():
    t = inputs(1000, 1024, 768, 64, seed=5)
    a = run_gpu(t, 128.0)
    b = run_gpu(t, 128.0)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("width", [256, 512])
def test_skip_dx_leaves_da_db_unchanged(width, gemm_width):
    """Without dX the backward runs the same skinny launches (their grouping
    follows the tile width, not whether dX is asked for), so dA and dB carry
    the same bits."""
    gemm_width(width)
    t = inputs(1000, 1024, 768, 64, seed=9)
    full = run_gpu(t, 128.0)
    part = run_gpu(t, 128.0, need_dX=False)
    assert part[1] is None
    for i in (0, 2, 3):
        assert torch.equal(full[i], part[i])


def test_close_to_the_bf16_layer():
    """fp8 quantisation of X, W, dY is the only difference from the bf16 layer."""
    t = inputs(512, 1024, 1024, 16, seed=6)
    g = {k: v.to(DEV) for k, v in t.items()}
    Y8 = run_gpu(t, 32.0)[0]
    Y16, _ = rl.forward(g["X"], g["W"], g["A"], g["B"], 32.0)
    torch.cuda.synchronize()
    assert rel_err(Y8, Y16.double().cpu().numpy()) < 0.1


def test_autograd_matches_the_explicit_calls():
    t = inputs(300, 256, 192, 16, seed=12)
    g = {k: v.to(DEV) for k, v in t.items()}
    qw = rl.quantize_w_fp8(g["W"])
    X = g["X"].reshape(2, 150, 256).clone().requires_grad_(True)
    A = g["A"].clone().requires_grad_(True)
    B = g["B"].clone().requires_grad_(True)
    Y = rl.lora_linear_fp8(X, qw, A, B, 32.0)
    Y.backward(g["dY"].reshape(2, 150, 192))
    Y2, saved = rl.fp8_forward(g["X"], qw, g["A"], g["B"], 32.0)
    dX2, dA2, dB2 = rl.fp8_backward(g["dY"], g["X"], qw, g["A"], g["B"], 32.0, saved)
    torch.cuda.synchronize()
    assert Y.shape == (2, 150, 192)
    assert torch.equal(Y.reshape(300, 192), Y2)
    assert torch.equal(X.grad.reshape(300, 256), dX2)
    assert torch.equal(A.grad, dA2) and torch.equal(B.grad, dB2)


def test_back_to_back_backward_calls():
    """Backward calls with different upstream gradients, enqueued back to back
    on one workspace (the dA pass starts in the dX GEMM's last wave), each
    give what they give when run alone."""
    M, d_in, d_out, r, alpha = 2048, 2048, 2048, 16, 32.0
    g = {k: v.to(DEV) for k, v in inputs(M, d_in, d_out, r, seed=41).items()}
    qw = rl.quantize_w_fp8(g["W"])
    ws = torch.empty(rl.fp8_workspace_bytes(M, d_in, d_out, r), dtype=torch.uint8, device=DEV)
    _, saved = rl.fp8_forward(g["X"], qw, g["A"], g["B"], alpha, workspace=ws)
    gen = torch.Generator(device=DEV).manual_seed(7)
    dYs = [torch.randn(M, d_out, device=DEV, generator=gen).bfloat16() for _ in range(4)]
    alone = []
    for dY in dYs:
        alone.append(rl.fp8_backward(dY, g["X"], qw, g["A"], g["B"], alpha, saved, workspace=ws))
        torch.cuda.synchronize()
    chained = [rl.fp8_backward(dY, g["X"], qw, g["A"], g["B"], alpha, saved, workspace=ws)
               for dY in dYs]
    torch.cuda.synchronize()
    rl.device_status()
    for a, b in zip(alone, chained):
        for x, y in zip(a, b):
            assert torch.equal(x, y)
    assert not torch.equal(alone[0][1], alone[1][1])
