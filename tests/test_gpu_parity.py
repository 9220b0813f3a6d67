"""CUDA path vs the fp64 oracle, through the C ABI (needs a GB300).

Metric for every output tensor T: max|T_gpu - T_ref| / max|T_ref|, which
must be <= 1e-2 for bf16 and <= 1e-5 for the fp32 debug dtype.  Small and
ragged shapes are compared element by element; the full-size workloads, in
the launch configuration the benchmark times, on all of dA and dB and on one
row of Y and dX in every 128-row m-tile (all rows of the 4096^2 workload).
"""
import numpy as np
import pytest
import torch

import oracle
import rank_linear_gb300 as rl
from rank_linear_gb300.synth import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "fp32": 1e-5}
DEV = "cuda:0"


def rel_err(got, ref) -> float:
    if isinstance(got, torch.Tensor):
        got = got.detach().double().cpu().numpy()
    den = np.abs(ref).max()
    return float(np.abs(got - ref).max() / (den if den > 0 else 1.0))


def run_gpu(t, alpha, saved_none=False, need_dX=True):
    g = {k: v.to(DEV) for k, v in t.items()}
    Y, saved = rl.forward(g["X"], g["W"], g["A"], g["B"], alpha)
    dX, dA, dB = rl.backward(g["dY"], g["X"], g["W"], g["A"], g["B"], alpha,
                             None if saved_none else saved, need_dX=need_dX)
    torch.cuda.synchronize()
    rl.device_status()
    return Y, dX, dA, dB


def check_full(t, alpha, dt):
    Y, dX, dA, dB = run_gpu(t, alpha)
    _, Yr = oracle.forward(t["X"], t["W"], t["A"], t["B"], alpha)
    dXr, dAr, dBr = oracle.backward(t["dY"], t["X"], t["W"], t["A"], t["B"], alpha)
    errs = {"Y": rel_err(Y, Yr), "dX": rel_err(dX, dXr), "dA": rel_err(dA, dAr),
            "dB": rel_err(dB, dBr)}
    for k, e in errs.items():
        assert e <= TOL[dt], f"{k}: {e:.3e} > {TOL[dt]} ({errs})"
    return errs


def check_full_mm(t, alpha):
    """Every element, the frozen-W products of the oracle taken by its
    matmul step (the plain loops would stream W once per row)."""
    Y, dX, dA, dB = run_gpu(t, alpha)
    S = oracle.Sampled(t["X"], t["W"], t["A"], t["B"], t["dY"], alpha)
    rows = np.arange(t["X"].shape[0])
    errs = {"Y": rel_err(Y, S.y_rows_mm(rows)), "dX": rel_err(dX, S.dx_rows_mm(rows)),
            "dA": rel_err(dA, S.dA()), "dB": rel_err(dB, S.dB())}
    for k, e in errs.items():
        assert e <= TOL["bf16"], f"{k}: {e:.3e} ({errs})"
    return Y, dX, dA, dB


@pytest.fixture
def gemm_width():
    """Forces the main GEMMs' tile width for one test, then restores the
    cost model's choice."""
    from rank_linear_gb300 import _lib
    L = _lib.lib()
    yield lambda w: _lib.check(L.lora_debug_gemm_width(w), "gemm width")
    L.lora_debug_gemm_width(0)


# M, d_in, d_out, r, alpha: several tiles in every dimension plus ragged tails
SMALL_BF16 = [
    (300, 392, 264, 16, 32.0),     # M, K and N all ragged
    (520, 520, 1000, 24, 48.0),    # r not a multiple of 16 (padded to 32)
    (129, 136, 264, 12, 24.0),     # r not a multiple of 8 (B padded in the forward)
    (1, 64, 64, 1, 2.0),           # one token, rank one
    (256, 512, 384, 256, 512.0),   # maximum rank
    (1000, 1024, 768, 64, 128.0),
    (2048, 1536, 2560, 128, 256.0),
    (64, 8, 8, 8, 16.0),           # K smaller than one block
    (777, 4104, 520, 16, 16.0),    # long ragged K (dX GEMM has a ragged N)
]


@pytest.mark.parametrize("M,d_in,d_out,r,alpha", SMALL_BF16)
def test_bf16_elementwise(M, d_in, d_out, r, alpha):
    t = make_inputs(M, d_in, d_out, r, "bf16", seed=M + r)
    check_full(t, alpha, "bf16")


@pytest.mark.parametrize("width", [256, 512])
@pytest.mark.parametrize("M,d_in,d_out,r,alpha", SMALL_BF16)
def test_bf16_each_tile_width(M, d_in, d_out, r, alpha, width, gemm_width):
    """Both GEMMs with 256 x 256 pair tiles (tail split where it applies) and
    with 256 x 512 pair tiles (half of the last tile's columns, or all of
    its second half, past N), element by element."""
    gemm_width(width)
    t = make_inputs(M, d_in, d_out, r, "bf16", seed=M + r + width)
    check_full(t, alpha, "bf16")


@pytest.mark.parametrize("M,d_in,d_out,r,alpha", [
    (2000, 1000, 5000, 24, 48.0),   # forward: 80 wide tiles (pairs take two); ragged M, K, N
    (2000, 5000, 1000, 40, 80.0),   # dX GEMM: 80 wide tiles, MN-major B; ragged everything
])
def test_wide_tiles_several_per_pair(M, d_in, d_out, r, alpha, gemm_width):
    """256 x 512 tiles with more tiles than CTA pairs, so a pair starts its
    next tile's half-0 MMAs while its epilogue still drains half 1 of the
    last: every element against the oracle, and bitwise repeatable."""
    gemm_width(512)
    t = make_inputs(M, d_in, d_out, r, "bf16", seed=M + d_in + r)
    a = check_full_mm(t, alpha)
    b = run_gpu(t, alpha)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("M,d_in,d_out,r,alpha", [
    (64, 256, 256, 8, 16.0),       # the tiny fp32 workload
    (130, 200, 72, 5, 10.0),       # ragged, odd widths allowed in fp32
])
def test_fp32_elementwise(M, d_in, d_out, r, alpha):
    t = make_inputs(M, d_in, d_out, r, "fp32", seed=3)
    check_full(t, alpha, "fp32")


def test_tiny_workload_fp32():
    w = WORKLOADS["tiny_fp32"]
    t = make_inputs(w.M, w.d_in, w.d_out, w.r, w.dtype, seed=0)
    check_full(t, w.alpha, "fp32")


def rows_per_m_tile(M, seed, tile=128):
    """One random row inside every 128-row m-tile, plus the first and last
    rows: every CTA's rows of every pair tile of every raster group (and so,
    comparing whole rows, every output tile) is checked."""
    rng = np.random.default_rng(seed)
    starts = np.arange(0, M, tile)
    picks = starts + rng.integers(0, tile, len(starts))
    return np.unique(np.concatenate([[0, M - 1], np.minimum(picks, M - 1)]))


@pytest.mark.parametrize("name", ["llama3_8b_q_proj", "llama3_8b_gate_up",
                                  "llama3_8b_down_proj", "qwen_wide_ffn"])
def test_full_size(name):
    """The full-size workloads in the launch configuration the benchmark
    times (full workspace: tail splits on): all of dA and dB, and Y and dX on
    one row of every 128-row m-tile -- every row on the 4096^2 workload."""
    w = WORKLOADS[name]
    t = make_inputs(w.M, w.d_in, w.d_out, w.r, w.dtype, seed=0, device=DEV)
    Y, dX, dA, dB = run_gpu(t, w.alpha)
    host = {k: v.cpu() for k, v in t.items()}
    del t
    S = oracle.Sampled(host["X"], host["W"], host["A"], host["B"], host["dY"], w.alpha)
    rows = np.arange(w.M) if name == "llama3_8b_q_proj" else rows_per_m_tile(w.M, seed=1)
    errs = {"Y": rel_err(Y[rows], S.y_rows_mm(rows)),
            "dX": rel_err(dX[rows], S.dx_rows_mm(rows)),
            "dA": rel_err(dA, S.dA()), "dB": rel_err(dB, S.dB())}
    for k, e in errs.items():
        assert e <= TOL["bf16"], f"{name} {k}: {e:.3e} ({errs})"
    for T in (Y, dX, dA, dB):
        assert torch.isfinite(T).all()


def test_bitwise_deterministic():
    t = make_inputs(1000, 1024, 768, 64, "bf16", seed=11)
    a = run_gpu(t, 128.0)
    b = run_gpu(t, 128.0)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("width", [256, 512])
def test_recompute_when_saved_is_null(width, gemm_width):
    gemm_width(width)
    t = make_inputs(300, 392, 264, 16, "bf16", seed=5)
    a = run_gpu(t, 32.0)
    b = run_gpu(t, 32.0, saved_none=True)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("width", [256, 512])
def test_skip_dx(width, gemm_width):
    """dA and dB do not depend on whether dX is computed (each tile width
    has its own launch grouping, the same with and without dX)."""
    gemm_width(width)
    t = make_inputs(300, 392, 264, 16, "bf16", seed=5)
    a = run_gpu(t, 32.0)
    b = run_gpu(t, 32.0, need_dX=False)
    assert b[1] is None
    assert torch.equal(a[2], b[2]) and torch.equal(a[3], b[3])


def test_skip_dx_beside_short_last_wave():
    """At 4096 x 4096 x 4096 the dX GEMM's 128 wide tiles leave a short last
    wave on 76 CTA pairs, and the dA + dB pass after it splits K at most in
    two. That choice follows from the shape alone, so dA and dB carry the
    same bits when dX is not computed (and no GEMM runs before the pass)."""
    t = make_inputs(4096, 4096, 4096, 16, "bf16", seed=8)
    a = run_gpu(t, 16.0)
    b = run_gpu(t, 16.0, need_dX=False)
    assert b[1] is None
    assert torch.equal(a[2], b[2]) and torch.equal(a[3], b[3])


def test_b_zero_gives_exact_zero_dA():
    """B = 0 (a fresh LoRA adapter): dA = 0 exactly and Y = X W^T."""
    t = make_inputs(300, 392, 264, 16, "bf16", seed=6)
    t["B"] = torch.zeros_like(t["B"])
    Y, dX, dA, dB = run_gpu(t, 32.0)
    assert torch.count_nonzero(dA) == 0
    ref = t["X"].double() @ t["W"].double().T
    assert rel_err(Y, ref.numpy()) <= TOL["bf16"]


def test_transposition_identity():
    """dX(dY; W, A, B) equals Y(X := dY; W := W^T, A := B^T, B := A^T)."""
    M, d_in, d_out, r, alpha = 300, 392, 264, 16, 32.0
    t = make_inputs(M, d_in, d_out, r, "bf16", seed=7)
    _, dX, _, _ = run_gpu(t, alpha)
    g = {k: v.to(DEV) for k, v in t.items()}
    Yt, _ = rl.forward(g["dY"], g["W"].T.contiguous(), g["B"].T.contiguous(),
                       g["A"].T.contiguous(), alpha)
    torch.cuda.synchronize()
    ref = dX.double().cpu().numpy()
    assert rel_err(Yt, ref) <= 4e-3


def test_empty_batch():
    t = make_inputs(1, 64, 64, 16, "bf16", seed=8)
    g = {k: v.to(DEV) for k, v in t.items()}
    X0 = g["X"][:0]
    dY0 = g["dY"][:0]
    Y, saved = rl.forward(X0, g["W"], g["A"], g["B"], 32.0)
    dX, dA, dB = rl.backward(dY0, X0, g["W"], g["A"], g["B"], 32.0, saved)
    torch.cuda.synchronize()
    assert Y.shape == (0, 64) and dX.shape == (0, 64)
    assert torch.count_nonzero(dA) == 0 and torch.count_nonzero(dB) == 0


def test_autograd_function():
    M, d_in, d_out, r, alpha = 2 * 150, 256, 320, 16, 32.0
    t = make_inputs(M, d_in, d_out, r, "bf16", seed=9)
    X = t["X"].to(DEV).reshape(2, 150, d_in).requires_grad_(True)
    W = t["W"].to(DEV)
    A = t["A"].to(DEV).requires_grad_(True)
    B = t["B"].to(DEV).requires_grad_(True)
    Y = rl.lora_linear(X, W, A, B, alpha)
    Y.backward(t["dY"].to(DEV).reshape(2, 150, d_out))
    torch.cuda.synchronize()
    _, Yr = oracle.forward(t["X"], t["W"], t["A"], t["B"], alpha)
    dXr, dAr, dBr = oracle.backward(t["dY"], t["X"], t["W"], t["A"], t["B"], alpha)
    assert rel_err(Y.reshape(M, d_out), Yr) <= 1e-2
    assert rel_err(X.grad.reshape(M, d_in), dXr) <= 1e-2
    assert rel_err(A.grad, dAr) <= 1e-2
    assert rel_err(B.grad, dBr) <= 1e-2


@pytest.mark.parametrize("width,kinds", [
    (512, ["down_fwd", "main_fwd", "down_bwd", "main_bwd", "grad_a_b"]),
    (256, ["down_fwd", "main_fwd", "down_bwd_grad_b", "main_bwd", "grad_a"]),
])
def test_timing_hook_records_every_launch(width, kinds, gemm_width):
    """Five launches a step; with 256 x 512 tiles dB runs after the dX GEMM
    beside dA, with 256 x 256 tiles beside s dY B before it."""
    from rank_linear_gb300 import _lib
    gemm_width(width)
    t = make_inputs(300, 392, 264, 16, "bf16", seed=5)
    g = {k: v.to(DEV) for k, v in t.items()}
    evs, arr, kinds_out = rl.timing_events(8)
    L = _lib.lib()
    n0 = rl.launch_count()
    assert L.lora_set_timing_events(arr, kinds_out, 8) == 0
    Y, saved = rl.forward(g["X"], g["W"], g["A"], g["B"], 32.0)
    rl.backward(g["dY"], g["X"], g["W"], g["A"], g["B"], 32.0, saved)
    used = L.lora_timing_used()
    L.lora_set_timing_events(None, None, 0)
    torch.cuda.synchronize()
    assert used == rl.launch_count() - n0 == 5
    assert [_lib.KERNEL_KINDS[k] for k in kinds_out[:used]] == kinds
    for j in range(used):
        assert evs[2 * j].elapsed_time(evs[2 * j + 1]) > 0


def test_timing_hook_rejects_uncreated_events():
    import ctypes
    from rank_linear_gb300 import _lib
    arr = (ctypes.c_void_p * 2)(None, None)
    assert _lib.lib().lora_set_timing_events(arr, None, 1) == _lib.LORA_ERR_INVALID_ARG


def test_tail_split_path(gemm_width):
    """M = 4096, d_in = d_out = 2816 with 256 x 256 tiles (the width of the
    SwiGLU, fp8 and 4-bit GEMMs, forced here for the plain layer): the last
    wave (24 of 76 pairs' tiles) is split across CTA pairs given the full
    workspace.  The split results are bitwise repeatable, agree with the
    unsplit ones (minimal workspace) and with the oracle on sampled rows."""
    gemm_width(256)
    M, d = 4096, 2816
    r, alpha = 16, 16.0
    t = make_inputs(M, d, d, r, "bf16", seed=12, device=DEV)
    X, W, A, B, dY = t["X"], t["W"], t["A"], t["B"], t["dY"]
    full = torch.empty(rl.workspace_bytes(M, d, d, r, torch.bfloat16), dtype=torch.uint8,
                       device=DEV)
    minimal = torch.empty(16 * d * 2 + 2 * 16 * M * 2, dtype=torch.uint8, device=DEV)  # B^T, sG, sG^T
    assert full.numel() > minimal.numel()

    def run(ws):
        Y, saved = rl.forward(X, W, A, B, alpha, workspace=ws)
        dX, dA, dB = rl.backward(dY, X, W, A, B, alpha, saved, workspace=ws)
        torch.cuda.synchronize()
        rl.device_status()
        return Y, dX, dA, dB

    s1, s2, u = run(full), run(full), run(minimal)
    for a, b in zip(s1, s2):
        assert torch.equal(a, b)
    for a, b in zip(s1, u):
        assert rel_err(a, b.double().cpu().numpy()) <= 4e-3
    assert not torch.equal(s1[0], u[0]) and not torch.equal(s1[1], u[1])  # the split ran
    host = {k: v.cpu() for k, v in t.items()}
    S = oracle.Sampled(host["X"], host["W"], host["A"], host["B"], host["dY"], alpha)
    rows = np.array([0, 2047, 3071, 3584, 4095])  # include rows of the split tiles
    assert rel_err(s1[0][rows], S.y_rows(rows)) <= TOL["bf16"]
    assert rel_err(s1[1][rows], S.dx_rows(rows)) <= TOL["bf16"]


def test_wide_tail_split_path(gemm_width):
    """M = 2000, d_in = 5896, d_out = 6000 with 256 x 512 tiles: each GEMM
    has 8 x 12 = 96 tiles, so on 76 CTA pairs the last wave's 20 are split
    two ways, each range's partial holding both accumulator halves (the last
    tile column ends past N, the last m-tile past M).  Given the full
    workspace the split results are bitwise repeatable and differ from the
    unsplit ones (minimal workspace); both agree with the oracle on every
    element."""
    gemm_width(512)
    M, d_in, d_out, r, alpha = 2000, 5896, 6000, 24, 48.0
    t = make_inputs(M, d_in, d_out, r, "bf16", seed=17, device=DEV)
    X, W, A, B, dY = t["X"], t["W"], t["A"], t["B"], t["dY"]
    full = torch.empty(rl.workspace_bytes(M, d_in, d_out, r, torch.bfloat16),
                       dtype=torch.uint8, device=DEV)
    rup = lambda n: (n + 255) // 256 * 256
    r_pad = 32  # the rank padded to a multiple of 16
    minimal = torch.empty(rup(r_pad * d_out * 2) + 2 * rup(r_pad * M * 2), dtype=torch.uint8,
                          device=DEV)  # B^T, sG, sG^T
    assert full.numel() > minimal.numel()

    def run(ws):
        Y, saved = rl.forward(X, W, A, B, alpha, workspace=ws)
        dX, dA, dB = rl.backward(dY, X, W, A, B, alpha, saved, workspace=ws)
        torch.cuda.synchronize()
        rl.device_status()
        return Y, dX, dA, dB

    s1, s2, u = run(full), run(full), run(minimal)
    for a, b in zip(s1, s2):
        assert torch.equal(a, b)
    assert not torch.equal(s1[0], u[0]) and not torch.equal(s1[1], u[1])  # the split ran
    host = {k: v.cpu() for k, v in t.items()}
    S = oracle.Sampled(host["X"], host["W"], host["A"], host["B"], host["dY"], alpha)
    rows = np.arange(M)
    ref = {"Y": S.y_rows_mm(rows), "dX": S.dx_rows_mm(rows), "dA": S.dA(), "dB": S.dB()}
    for got in (s1, u):
        errs = {k: rel_err(g, ref[k]) for k, g in zip(("Y", "dX", "dA", "dB"), got)}
        for k, e in errs.items():
            assert e <= TOL["bf16"], f"{k}: {e:.3e} ({errs})"


@pytest.mark.parametrize("M,d", [(2048, 2048), (4096, 4096)])
def test_back_to_back_backward_calls(M, d):
    """The dA pass starts in the dX GEMM's last wave without waiting for the
    GEMM: it relies on the GEMM letting it start only once every kernel
    before the GEMM -- among them the pass that writes sG -- has finished.
    Backward calls with different upstream gradients, enqueued back to back
    on one workspace (each overwrites the previous call's sG), must each
    give what they give when run alone."""
    r, alpha = 16, 16.0
    t = make_inputs(M, d, d, r, "bf16", seed=21, device=DEV)
    X, W, A, B = t["X"], t["W"], t["A"], t["B"]
    ws = torch.empty(rl.workspace_bytes(M, d, d, r, torch.bfloat16), dtype=torch.uint8,
                     device=DEV)
    _, saved = rl.forward(X, W, A, B, alpha, workspace=ws)
    gen = torch.Generator(device=DEV).manual_seed(5)
    dYs = [torch.randn(M, d, device=DEV, generator=gen).bfloat16() for _ in range(4)]
    alone = []
    for dY in dYs:
        alone.append(rl.backward(dY, X, W, A, B, alpha, saved, workspace=ws))
        torch.cuda.synchronize()
    chained = [rl.backward(dY, X, W, A, B, alpha, saved, workspace=ws) for dY in dYs]
    torch.cuda.synchronize()
    rl.device_status()
    for a, b in zip(alone, chained):
        for x, y in zip(a, b):
            assert torch.equal(x, y)
    assert not torch.equal(alone[0][1], alone[1][1])  # the calls' dA really differ


def test_back_to_back_alternating_dx():
    """Backward calls that alternate between computing dX (the dA pass then
    overlaps the dX GEMM) and skipping it (the dA pass follows the s dY B
    pass and waits for it), enqueued back to back on one workspace, each give
    what they give when run alone."""
    M = d = 2048
    r, alpha = 16, 16.0
    t = make_inputs(M, d, d, r, "bf16", seed=23, device=DEV)
    X, W, A, B = t["X"], t["W"], t["A"], t["B"]
    ws = torch.empty(rl.workspace_bytes(M, d, d, r, torch.bfloat16), dtype=torch.uint8,
                     device=DEV)
    _, saved = rl.forward(X, W, A, B, alpha, workspace=ws)
    gen = torch.Generator(device=DEV).manual_seed(9)
    dYs = [torch.randn(M, d, device=DEV, generator=gen).bfloat16() for _ in range(6)]
    flags = [True, False, True, False, False, True]
    alone = []
    for dY, f in zip(dYs, flags):
        alone.append(rl.backward(dY, X, W, A, B, alpha, saved, need_dX=f, workspace=ws))
        torch.cuda.synchronize()
    chained = [rl.backward(dY, X, W, A, B, alpha, saved, need_dX=f, workspace=ws)
               for dY, f in zip(dYs, flags)]
    torch.cuda.synchronize()
    rl.device_status()
    for a, b, f in zip(alone, chained, flags):
        assert (a[0] is None) == (not f) and (b[0] is None) == (not f)
        for x, y in zip(a, b):
            if x is not None:
                assert torch.equal(x, y)
