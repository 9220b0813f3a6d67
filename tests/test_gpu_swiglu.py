"""The SwiGLU gate/up pair of LoRA layers on the GPU vs the fp64 oracle
(needs a GB300).

Metric per output tensor T: max|T_gpu - T_ref| / max|T_ref| <= 1e-2 (bf16).
The gradients carry one rounding more than the plain layer's: d_gate and
d_up are bf16 intermediates (from bf16-saved gate and up), and each gradient
is a dot product over them.  On the one shape where that product cancels
(one token, rank one: dAg is a single 64-term sum that cancels to 1.85e-2 of
max|ref|), its gradients may instead meet the forward error bound of such a
product, max|T_gpu - T_ref| <= 2^-7 max|T_abs|, T_abs being the same formula
on absolute values (relative error <= 4 u per term, u = 2^-9); every other
shape meets 1e-2 of max|ref|.  Small and ragged shapes are compared element by
element; the full gate/up workload (Llama-3-8B MLP shape) on one token row of
H and dX in every 128-row m-tile and on all four adapter gradients.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import swiglu as osw
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


def make_pair(M, d_in, d_ff, r, seed):
    """Gate and up projections drawn like the LoRA layer's inputs (two seeds)."""
    g = make_inputs(M, d_in, d_ff, r, "bf16", seed=seed)
    u = make_inputs(M, d_in, d_ff, r, "bf16", seed=seed + 1000)
    # larger adapters than the init-like B ~ N(0, 0.02) so the low-rank term matters
    return dict(X=g["X"], Wg=g["W"], Ag=g["A"], Bg=(g["B"].float() * 10).bfloat16(),
                Wu=u["W"], Au=u["A"], Bu=(u["B"].float() * 10).bfloat16(), dH=g["dY"])


def run_gpu(t, alpha, need_dX=True):
    g = {k: v.to(DEV) for k, v in t.items()}
    args = [g[k] for k in ("Wg", "Ag", "Bg", "Wu", "Au", "Bu")]
    H, saved = rl.swiglu_forward(g["X"], *args, alpha)
    grads = rl.swiglu_backward(g["dH"], g["X"], *args, alpha, saved, need_dX=need_dX)
    torch.cuda.synchronize()
    rl.device_status()
    return (H,) + tuple(grads)


def oracle_all(t, alpha):
    args = [t[k] for k in ("X", "Wg", "Ag", "Bg", "Wu", "Au", "Bu")]
    _, _, H = osw.forward(*args, alpha)
    return (H,) + tuple(osw.backward(t["dH"], *args, alpha))


def oracle_abs(t, alpha):
    """dX, dAg, dBg, dAu, dBu computed on absolute values (error-bound scale)."""
    args = [t[k] for k in ("X", "Wg", "Ag", "Bg", "Wu", "Au", "Bu")]
    gate, up, _ = osw.forward(*args, alpha)
    dH = np.abs(oracle._f64(t["dH"]))
    d_gate = dH * np.abs(up) * np.abs(osw.silu_grad(gate))
    d_up = dH * np.abs(osw.silu(gate))
    a = {k: np.abs(oracle._f64(t[k])) for k in ("X", "Wg", "Ag", "Bg", "Wu", "Au", "Bu")}
    dXg, dAg, dBg = oracle.backward(d_gate, a["X"], a["Wg"], a["Ag"], a["Bg"], alpha)
    dXu, dAu, dBu = oracle.backward(d_up, a["X"], a["Wu"], a["Au"], a["Bu"], alpha)
    return dXg + dXu, dAg, dBg, dAu, dBu


def meets_bar(got, ref, ref_abs=None):
    """1e-2 of max|ref|; or, where ref_abs is given (the cancelling shape
    only), the dot-product error bound 2^-7 max|T_abs|."""
    if isinstance(got, torch.Tensor):
        got = got.detach().double().cpu().numpy()
    err = float(np.abs(got - ref).max())
    if err <= TOL * float(np.abs(ref).max()):
        return True
    return ref_abs is not None and err <= 2.0 ** -7 * float(np.abs(ref_abs).max())


# the single shape whose gradients are one cancelling dot product
CANCELLING = (1, 64, 64, 1, 2.0)


NAMES = ("H", "dX", "dAg", "dBg", "dAu", "dBu")

# M, d_in, d_ff, r, alpha
SMALL = [
    (300, 392, 264, 16, 32.0),     # M, K and the gated columns ragged
    (520, 520, 1000, 24, 48.0),    # r not a multiple of 16 (padded to 32)
    (129, 136, 264, 12, 24.0),     # r not a multiple of 8 (B padded / transposed)
    (1, 64, 64, 1, 2.0),           # one token, rank one
    (256, 512, 384, 256, 512.0),   # maximum rank: extension K = 512
    (64, 8, 8, 8, 16.0),           # K smaller than one block
    (2048, 1536, 2560, 128, 256.0),  # gated GEMM's last wave split two ways
    (1024, 5120, 1024, 16, 32.0),  # dX GEMM's last wave split two ways
]


@pytest.fixture
def gemm_width():
    """Forces the tile width of the GEMMs that may take 256 x 512 tiles (here
    the dX GEMM) for one test, then restores the cost model's choice."""
    from rank_linear_gb300 import _lib
    L = _lib.lib()
    yield lambda w: _lib.check(L.lora_debug_gemm_width(w), "gemm width")
    L.lora_debug_gemm_width(0)


@pytest.mark.parametrize("width", [256, 512])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s[:4])))
def test_small_against_oracle(shape, width, gemm_width):
    gemm_width(width)
    M, d_in, d_ff, r, alpha = shape
    t = make_pair(M, d_in, d_ff, r, seed=sum(shape[:4]))
    got = run_gpu(t, alpha)
    ref = oracle_all(t, alpha)
    bound = (None,) + oracle_abs(t, alpha) if tuple(shape) == CANCELLING else (None,) * 6
    errs = {n: rel_err(g, e) for n, g, e in zip(NAMES, got, ref)}
    for n, g, e, b in zip(NAMES, got, ref, bound):
        assert meets_bar(g, e, b), f"{n}: {errs[n]:.3e} ({errs})"


def test_wide_dx_tail_split(gemm_width):
    """M = 2000, d_in = 6000, d_ff = 1024: the dX GEMM over [d_gate | d_up]
    (its B map switching from Wg to Wu mid-K) with 256 x 512 tiles has 8 x 12
    = 96 tiles, so on 76 CTA pairs the last wave's 20 are split in two K
    ranges.  Given the full workspace the results are bitwise repeatable and
    dX differs from the unsplit one (minimal workspace); both agree with the
    oracle on every element."""
    gemm_width(512)
    M, d_in, d_ff, r, alpha = 2000, 6000, 1024, 24, 48.0
    t = make_pair(M, d_in, d_ff, r, seed=71)
    g = {k: v.to(DEV) for k, v in t.items()}
    args = [g[k] for k in ("Wg", "Ag", "Bg", "Wu", "Au", "Bu")]
    rup = lambda n: (n + 255) // 256 * 256
    half, r_pad = 1024, 32
    bwd_min = (rup(M * 2 * half * 2) + rup(M * 2 * r_pad * 2) + 2 * rup(r_pad * M * 2)
               + rup(2 * r_pad * d_in * 2))
    full = torch.empty(rl.swiglu_workspace_bytes(M, d_in, d_ff, r), dtype=torch.uint8, device=DEV)
    minimal = torch.empty(bwd_min, dtype=torch.uint8, device=DEV)
    assert full.numel() > minimal.numel()
    H, saved = rl.swiglu_forward(g["X"], *args, alpha, workspace=full)

    def run(ws):
        grads = rl.swiglu_backward(g["dH"], g["X"], *args, alpha, saved, workspace=ws)
        torch.cuda.synchronize()
        rl.device_status()
        return grads

    s1, s2, u = run(full), run(full), run(minimal)
    for a, b in zip(s1, s2):
        assert torch.equal(a, b)
    assert not torch.equal(s1[0], u[0])  # the split ran
    hargs = [t[k] for k in ("X", "Wg", "Ag", "Bg", "Wu", "Au", "Bu")]
    smp = osw.SampledRows(*hargs, t["dH"], alpha)
    rows = np.arange(M)
    ref_h = smp.h_rows_mm(rows)
    ref = (smp.dx_rows_mm(rows),) + tuple(osw.adapter_grads_mm(t["dH"], *hargs, alpha))
    assert rel_err(H, ref_h) <= TOL
    for got in (s1, u):
        errs = {n: rel_err(x, e) for n, x, e in zip(NAMES[1:], got, ref)}
        for n, e in errs.items():
            assert e <= TOL, f"{n}: {e:.3e} ({errs})"


def test_wide_gated_tail_split(gemm_width):
    """M = 2000, d_in = 1024, d_ff = 3000: the gated GEMM with 256 x 512 tiles
    (256 outputs of both projections each, the last tile column ragged) has
    8 x 12 = 96 tiles, so on 76 CTA pairs the last wave's 20 are split in two
    K ranges, each range's partial holding gate and up of both halves.  Given
    the full workspace H (and the saved gate and up) are bitwise repeatable and
    differ from the unsplit ones (minimal workspace); both agree with the
    oracle on every element."""
    gemm_width(512)
    M, d_in, d_ff, r, alpha = 2000, 1024, 3000, 24, 48.0
    t = make_pair(M, d_in, d_ff, r, seed=72)
    g = {k: v.to(DEV) for k, v in t.items()}
    args = [g[k] for k in ("Wg", "Ag", "Bg", "Wu", "Au", "Bu")]
    rup = lambda n: (n + 255) // 256 * 256
    full = torch.empty(rl.swiglu_workspace_bytes(M, d_in, d_ff, r), dtype=torch.uint8, device=DEV)
    minimal = torch.empty(rup(M * 2 * 32 * 2), dtype=torch.uint8, device=DEV)  # [sH_g | sH_u]
    assert full.numel() > minimal.numel()

    def run(ws):
        H, saved = rl.swiglu_forward(g["X"], *args, alpha, workspace=ws)
        torch.cuda.synchronize()
        rl.device_status()
        return H, saved

    (h1, s1), (h2, s2), (hu, su) = run(full), run(full), run(minimal)
    assert torch.equal(h1, h2) and torch.equal(s1, s2)
    assert not torch.equal(h1, hu)  # the split ran
    hargs = [t[k] for k in ("X", "Wg", "Ag", "Bg", "Wu", "Au", "Bu")]
    ref = osw.SampledRows(*hargs, t["dH"], alpha).h_rows_mm(np.arange(M))
    for H in (h1, hu):
        assert rel_err(H, ref) <= TOL, f"H: {rel_err(H, ref):.3e}"


def test_full_gate_up():
    """Llama-3-8B MLP gate/up shape (M = 8192 tokens, d_in = 4096,
    d_ff = 14336, r = 16): H and dX on one row of every 128-row m-tile, and
    all of dAg, dBg, dAu, dBu."""
    M, d_in, d_ff, r, alpha = 8192, 4096, 14336, 16, 32.0
    t = make_pair(M, d_in, d_ff, r, seed=0)
    H, dX, dAg, dBg, dAu, dBu = run_gpu(t, alpha)
    args = [t[k] for k in ("X", "Wg", "Ag", "Bg", "Wu", "Au", "Bu")]
    smp = osw.SampledRows(*args, t["dH"], alpha)
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([[0, M - 1],
                                     np.arange(0, M, 128) + rng.integers(0, 128, M // 128)]))
    errs = {"H": rel_err(H[rows], smp.h_rows_mm(rows)),
            "dX": rel_err(dX[rows], smp.dx_rows_mm(rows))}
    for name, got, ref in zip(("dAg", "dBg", "dAu", "dBu"), (dAg, dBg, dAu, dBu),
                              osw.adapter_grads_mm(t["dH"], *args, alpha)):
        errs[name] = rel_err(got, ref)
    for k, e in errs.items():
        assert e <= TOL, f"{k}: {e:.3e} ({errs})"


def test_inference_forward_keeps_nothing_and_agrees():
    t = make_pair(300, 392, 264, 16, seed=9)
    g = {k: v.to(DEV) for k, v in t.items()}
    args = [g[k] for k in ("Wg", "Ag", "Bg", "Wu", "Au", "Bu")]
    H1, saved = rl.swiglu_forward(g["X"], *args, 32.0)
    H2, none = rl.swiglu_forward(g["X"], *args, 32.0, keep=False)
    torch.cuda.synchronize()
    rl.device_status()
    assert none is None and saved is not None
    assert torch.equal(H1, H2)


def test_deterministic():
    t = make_pair(520, 520, 1000, 24, seed=5)
    a = run_gpu(t, 48.0)
    b = run_gpu(t, 48.0)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_skip_dx_leaves_the_rest_unchanged():
    t = make_pair(300, 392, 264, 16, seed=6)
    full = run_gpu(t, 32.0)
    part = run_gpu(t, 32.0, need_dX=False)
    assert part[1] is None
    for i in (0, 2, 3, 4, 5):
        assert torch.equal(full[i], part[i])


def test_autograd():
    M, d_in, d_ff, r, alpha = 130, 128, 256, 8, 16.0
    t = make_pair(M, d_in, d_ff, r, seed=7)
    g = {k: v.to(DEV) for k, v in t.items()}
    X = g["X"].clone().reshape(2, 65, d_in).requires_grad_(True)
    params = {k: g[k].clone().requires_grad_(k in ("Ag", "Bg", "Au", "Bu"))
              for k in ("Wg", "Ag", "Bg", "Wu", "Au", "Bu")}
    H = rl.lora_swiglu(X, *(params[k] for k in ("Wg", "Ag", "Bg", "Wu", "Au", "Bu")), alpha)
    H.backward(g["dH"].reshape(2, 65, d_ff))
    ref = oracle_all(t, alpha)
    assert rel_err(H.reshape(M, d_ff), ref[0]) <= TOL
    assert rel_err(X.grad.reshape(M, d_in), ref[1]) <= TOL
    for name, e in zip(("Ag", "Bg", "Au", "Bu"), ref[2:]):
        assert rel_err(params[name].grad, e) <= TOL, name
    assert params["Wg"].grad is None and params["Wu"].grad is None


def test_empty_batch():
    t = make_pair(0, 64, 64, 8, seed=8)
    g = {k: v.to(DEV) for k, v in t.items()}
    args = [g[k] for k in ("Wg", "Ag", "Bg", "Wu", "Au", "Bu")]
    H, saved = rl.swiglu_forward(g["X"], *args, 16.0)
    dX, dAg, dBg, dAu, dBu = rl.swiglu_backward(g["dH"], g["X"], *args, 16.0, saved)
    torch.cuda.synchronize()
    assert H.shape == (0, 64) and dX.shape == (0, 64)
    for z in (dAg, dBg, dAu, dBu):
        assert torch.count_nonzero(z) == 0


def test_back_to_back_backward_calls():
    """Backward calls with different upstream gradients, enqueued back to back
    on one workspace (the dA passes start in the dX GEMM's last wave), each
    give what they give when run alone."""
    M, d_in, d_ff, r, alpha = 2048, 1024, 2816, 16, 32.0
    g = {k: v.to(DEV) for k, v in make_pair(M, d_in, d_ff, r, seed=31).items()}
    args = [g[k] for k in ("Wg", "Ag", "Bg", "Wu", "Au", "Bu")]
    ws = torch.empty(rl.swiglu_workspace_bytes(M, d_in, d_ff, r), dtype=torch.uint8, device=DEV)
    _, saved = rl.swiglu_forward(g["X"], *args, alpha, workspace=ws)
    gen = torch.Generator(device=DEV).manual_seed(6)
    dHs = [torch.randn(M, d_ff, device=DEV, generator=gen).bfloat16() for _ in range(4)]
    alone = []
    for dH in dHs:
        alone.append(rl.swiglu_backward(dH, g["X"], *args, alpha, saved, workspace=ws))
        torch.cuda.synchronize()
    chained = [rl.swiglu_backward(dH, g["X"], *args, alpha, saved, workspace=ws) for dH in dHs]
    torch.cuda.synchronize()
    rl.device_status()
    for a, b in zip(alone, chained):
        for x, y in zip(a, b):
            assert torch.equal(x, y)
    assert not torch.equal(alone[0][1], alone[1][1])
