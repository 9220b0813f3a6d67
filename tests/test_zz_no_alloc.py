"""lora_linear_bwd_noalloc against lora_linear_bwd, through the C ABI (GPU).

Some callers cannot allocate device memory at the moment they run the
backward: a plugin inside a host application that owns all device memory and
offers it no allocator, or a latency-critical loop that must not call
cudaMalloc (which may synchronise the device) once it is running.  For them
the library has lora_linear_bwd_noalloc, which takes its scratch from an
array built into the library instead of a caller workspace.

The tests make two calls in a row -- so the second call finds the first
call's leftovers in the shared scratch -- and compare each result with
lora_linear_bwd given its own workspace, within the parity tolerance of the
other tests (bit for bit where both take the same path), and with the fp64
oracle.  One pair of calls is on a shape whose dX GEMM takes the tail-split
path inside the array, which keeps per-tile arrival counters there.  A shape
needing more than the built-in scratch is refused.  The file name makes
pytest collect it last.
"""
import numpy as np
import pytest
import torch

import rank_linear_gb300 as rl
from rank_linear_gb300 import _lib
from rank_linear_gb300.synth import make_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TOL = {"bf16": 1e-2, "fp32": 1e-5}
CODE = {"bf16": _lib.LORA_BF16, "fp32": _lib.LORA_FP32}
SCRATCH_BYTES = 16 << 20  # LORA_NOALLOC_SCRATCH_BYTES


def _p(t):
    return None if t is None else (t.data_ptr() or None)


def _noalloc_bwd(g, alpha, saved, dt, with_dx=True):
    M, d_in = g["X"].shape
    d_out, r = g["B"].shape
    dX = torch.empty_like(g["X"]) if with_dx else None
    dA = torch.empty(r, d_in, dtype=g["X"].dtype, device=DEV)
    dB = torch.empty(d_out, r, dtype=g["X"].dtype, device=DEV)
    st = _lib.lib().lora_linear_bwd_noalloc(
        _p(g["dY"]), _p(g["X"]), _p(g["W"]), _p(g["A"]), _p(g["B"]), _p(saved), float(alpha),
        r, M, d_in, d_out, CODE[dt], _p(dX), _p(dA), _p(dB),
        torch.cuda.current_stream().cuda_stream or None)
    _lib.check(st, "lora_linear_bwd_noalloc")
    return dX, dA, dB


def _rel(got, ref):
    got = got.double().cpu().numpy()
    ref = ref.double().cpu().numpy()
    den = np.abs(ref).max()
    return float(np.abs(got - ref).max() / (den if den > 0 else 1.0))


# M = 4096, d_in = 2816, d_out = 4096, r = 16: on a GB300 (76 CTA pairs),
# with 256 x 256 tiles (forced through the library's test hook; the width
# of the SwiGLU, fp8 and 4-bit GEMMs), the dX GEMM's last wave is split two
# ways, and its split region fits in the array
SPLIT_PROBLEM = (4096, 2816, 4096, 16, 16.0)


def _rows_per_m_tile(M, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, M - 1], np.arange(0, M, 128) +
                                     rng.integers(0, 128, (M + 127) // 128)]).clip(0, M - 1))


def test_split_problem_twice_in_a_row():
    """Two calls in a row on the problem whose dX GEMM takes the tail-split
    path (its fp32 partials and arrival counters live in the shared array;
    the second call finds the first call's counters there).  Each call gives
    the same bits as lora_linear_bwd with a full workspace -- so the split
    path ran -- which differ from the unsplit (minimal-workspace) bits, and
    agrees with the oracle on all of dA and dB and one row of dX per 128-row
    m-tile."""
    L = _lib.lib()
    _lib.check(L.lora_debug_gemm_width(256), "gemm width")
    try:
        _split_problem_twice_in_a_row()
    finally:
        L.lora_debug_gemm_width(0)


def _split_problem_twice_in_a_row():
    import oracle
    M, d_in, d_out, r, alpha = SPLIT_PROBLEM
    bf = torch.bfloat16
    need_split = rl.workspace_bytes(M, d_in, d_out, r, bf)
    saved_room = (rl.saved_bytes(M, r, bf) + 255) // 256 * 256
    no_split = 3 * ((16 * 4096 * 2 + 255) // 256 * 256)  # B^T, sG, sG^T
    assert no_split < need_split - saved_room <= SCRATCH_BYTES
    t = make_inputs(M, d_in, d_out, r, "bf16", seed=41, device=DEV)
    g = dict(t)
    full = torch.empty(need_split, dtype=torch.uint8, device=DEV)
    minimal = torch.empty(no_split, dtype=torch.uint8, device=DEV)
    _, saved = rl.forward(g["X"], g["W"], g["A"], g["B"], alpha, workspace=full)
    gen = torch.Generator(device=DEV).manual_seed(42)
    dYs = [g["dY"], torch.randn(M, d_out, device=DEV, generator=gen).bfloat16()]
    got = []
    for dY in dYs:  # back to back, nothing in between
        got.append(_noalloc_bwd(dict(g, dY=dY), alpha, saved, "bf16"))
    torch.cuda.synchronize()
    rl.device_status()
    host = {k: t[k].cpu() for k in ("X", "W", "A", "B")}
    for dY, (dX, dA, dB) in zip(dYs, got):
        ref = rl.backward(dY, g["X"], g["W"], g["A"], g["B"], alpha, saved, workspace=full)
        unsplit = rl.backward(dY, g["X"], g["W"], g["A"], g["B"], alpha, saved,
                              workspace=minimal)
        torch.cuda.synchronize()
        for a, b in zip((dX, dA, dB), ref):
            assert torch.equal(a, b)
            assert _rel(a, b) <= TOL["bf16"]
        assert not torch.equal(ref[0], unsplit[0])  # the split path gives other bits
        S = oracle.Sampled(host["X"], host["W"], host["A"], host["B"], dY.cpu(), alpha)
        rows = _rows_per_m_tile(M, seed=43)
        for name, a, e in (("dX", dX[rows], S.dx_rows_mm(rows)), ("dA", dA, S.dA()),
                           ("dB", dB, S.dB())):
            err = _rel(a, torch.from_numpy(e))
            assert err <= TOL["bf16"], f"{name}: {err:.3e}"
    assert not torch.equal(got[0][1], got[1][1])  # the two calls' dA really differ


# two different problems, run back to back through the shared scratch
PROBLEMS = [
    (1000, 1024, 768, 64, 128.0, "bf16", True),
    (300, 392, 264, 16, 32.0, "bf16", False),   # smaller: leftovers of the first call remain
]


def test_two_calls_in_a_row_match_the_workspace_backward():
    results = []
    for M, d_in, d_out, r, alpha, dt, use_saved in PROBLEMS:
        t = make_inputs(M, d_in, d_out, r, dt, seed=M)
        g = {k: v.to(DEV) for k, v in t.items()}
        _, saved = rl.forward(g["X"], g["W"], g["A"], g["B"], alpha)
        ref = rl.backward(g["dY"], g["X"], g["W"], g["A"], g["B"], alpha, saved)
        got = _noalloc_bwd(g, alpha, saved if use_saved else None, dt)
        results.append((dt, ref, got))
    torch.cuda.synchronize()
    rl.device_status()
    for dt, ref, got in results:
        for name, a, b in zip(("dX", "dA", "dB"), got, ref):
            e = _rel(a, b)
            assert e <= TOL[dt], f"{name}: {e:.3e}"


def test_fp32_and_skipped_dx():
    t = make_inputs(64, 256, 256, 8, "fp32", seed=0)
    g = {k: v.to(DEV) for k, v in t.items()}
    _, saved = rl.forward(g["X"], g["W"], g["A"], g["B"], 16.0)
    ref = rl.backward(g["dY"], g["X"], g["W"], g["A"], g["B"], 16.0, saved)
    got = _noalloc_bwd(g, 16.0, saved, "fp32", with_dx=False)
    torch.cuda.synchronize()
    assert got[0] is None
    assert _rel(got[1], ref[1]) <= TOL["fp32"] and _rel(got[2], ref[2]) <= TOL["fp32"]


def test_shape_beyond_the_scratch_is_refused():
    # B^T, sG and sG^T need 2*256*(16384 + 2*8200) bytes > 16 MiB.  Real
    # buffers of the stated sizes are passed, but nothing may run.
    M, d_in, d_out, r = 8200, 64, 16384, 256
    bf = torch.bfloat16
    g = {"dY": torch.empty(M, d_out, dtype=bf, device=DEV),
         "X": torch.empty(M, d_in, dtype=bf, device=DEV),
         "W": torch.empty(d_out, d_in, dtype=bf, device=DEV),
         "A": torch.empty(r, d_in, dtype=bf, device=DEV),
         "B": torch.empty(d_out, r, dtype=bf, device=DEV)}
    saved = torch.empty(rl.saved_bytes(M, r, bf), dtype=torch.uint8, device=DEV)
    assert rl.workspace_bytes(M, d_in, d_out, r, bf) - rl.saved_bytes(M, r, bf) > SCRATCH_BYTES
    n0 = rl.launch_count()
    with pytest.raises(_lib.LoraError) as ei:
        _noalloc_bwd(g, 512.0, saved, "bf16")
    assert ei.value.status == _lib.LORA_ERR_UNSUPPORTED
    assert "built-in scratch" in str(ei.value)
    assert rl.launch_count() == n0
