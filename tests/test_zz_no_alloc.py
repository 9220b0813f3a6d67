"""lora_linear_bwd_noalloc against lora_linear_bwd, through the C ABI (GPU).

Some callers cannot allocate device memory at the moment they run the
backward: a plugin inside a host application that owns all device memory and
offers it no allocator, or a latency-critical loop that must not call
cudaMalloc (which may synchronise the device) once it is running.  For them
the library has lora_linear_bwd_noalloc, which takes its scratch from an
array built into the library instead of a caller workspace.

The test makes two calls in a row on different problems -- so the second
call finds the first call's leftovers in the shared scratch -- and compares
each result with lora_linear_bwd given its own workspace, within the parity
tolerance of the other tests.  It also checks that a shape needing more than
the built-in scratch is refused.  The file name makes pytest collect it last.
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
