"""Bounded device-side waits (needs a GB300).

The library's test hooks leave one pipeline stage of the backward's dA pass,
or of its dX GEMM, unfilled.  The wait for it must run out after its limit (about 2 s) instead
of spinning forever; the kernel then leaves through its abort path, the
device status word reports LORA_ERR_TIMEOUT, and the CUDA context stays
usable: the next call is correct.  No GPU fault, trap or hang is involved.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import rank_linear_gb300 as rl
from rank_linear_gb300 import _lib
from rank_linear_gb300.synth import make_inputs

pytestmark = pytest.mark.gpu


def rel_err(got, ref) -> float:
    got = got.detach().double().cpu().numpy()
    return float(np.abs(got - ref).max() / np.abs(ref).max())


def test_withheld_arrival_times_out_and_the_context_survives():
    L = _lib.lib()
    M, d_in, d_out, r, alpha = 256, 512, 384, 16, 32.0
    t = make_inputs(M, d_in, d_out, r, "bf16", seed=11)
    g = {k: v.to("cuda:0") for k, v in t.items()}
    dXr, dAr, dBr = oracle.backward(t["dY"], t["X"], t["W"], t["A"], t["B"], alpha)
    rl.device_status()  # nothing pending from earlier tests

    Y, saved = rl.forward(g["X"], g["W"], g["A"], g["B"], alpha)
    assert L.lora_debug_withhold_arrive(1) == _lib.LORA_OK
    t0 = time.time()
    dX, dA, dB = rl.backward(g["dY"], g["X"], g["W"], g["A"], g["B"], alpha, saved)
    status = L.lora_device_status(1)  # synchronises, reads and clears the word
    waited = time.time() - t0
    assert status == _lib.LORA_ERR_TIMEOUT, L.lora_last_error()
    assert waited > 1.0, f"the wait gave up after {waited:.2f} s, before its limit"
    assert waited < 30.0
    assert L.lora_device_status(1) == _lib.LORA_OK  # cleared
    # the launches before the stalled one finished normally
    assert rel_err(dX, dXr) <= 1e-2
    assert rel_err(dB, dBr) <= 1e-2

    # the hook was used up: the next call is correct
    dX, dA, dB = rl.backward(g["dY"], g["X"], g["W"], g["A"], g["B"], alpha, saved)
    torch.cuda.synchronize()
    rl.device_status()
    _, Yr = oracle.forward(t["X"], t["W"], t["A"], t["B"], alpha)
    for got, ref in ((Y, Yr), (dX, dXr), (dA, dAr), (dB, dBr)):
        assert rel_err(got, ref) <= 1e-2


@pytest.mark.parametrize("width", [256, 512])
def test_withheld_gemm_stage_times_out_and_the_context_survives(width):
    """The dX GEMM's odd CTA of the first pair never loads its first stage:
    the even CTA's MMA wait runs out, both CTAs of every pair leave through
    the abort path (the even CTA settles each stage's outstanding phase
    before either CTA exits), the status word reports LORA_ERR_TIMEOUT, and
    the next call is correct -- for both tile widths."""
    L = _lib.lib()
    M, d_in, d_out, r, alpha = 512, 1024, 768, 16, 32.0
    t = make_inputs(M, d_in, d_out, r, "bf16", seed=13)
    g = {k: v.to("cuda:0") for k, v in t.items()}
    _, Yr = oracle.forward(t["X"], t["W"], t["A"], t["B"], alpha)
    dXr, dAr, dBr = oracle.backward(t["dY"], t["X"], t["W"], t["A"], t["B"], alpha)
    assert L.lora_debug_gemm_width(width) == _lib.LORA_OK
    try:
        rl.device_status()
        Y, saved = rl.forward(g["X"], g["W"], g["A"], g["B"], alpha)
        assert L.lora_debug_withhold_gemm_stage(1) == _lib.LORA_OK
        t0 = time.time()
        dX, dA, dB = rl.backward(g["dY"], g["X"], g["W"], g["A"], g["B"], alpha, saved)
        status = L.lora_device_status(1)
        waited = time.time() - t0
        assert status == _lib.LORA_ERR_TIMEOUT, L.lora_last_error()
        assert waited > 1.0, f"the wait gave up after {waited:.2f} s, before its limit"
        assert waited < 60.0
        assert L.lora_device_status(1) == _lib.LORA_OK
        # the launches that do not depend on dX completed normally
        assert rel_err(dA, dAr) <= 1e-2 and rel_err(dB, dBr) <= 1e-2
        # the hook was used up: the next call is correct
        dX, dA, dB = rl.backward(g["dY"], g["X"], g["W"], g["A"], g["B"], alpha, saved)
        torch.cuda.synchronize()
        rl.device_status()
        for got, ref in ((Y, Yr), (dX, dXr), (dA, dAr), (dB, dBr)):
            assert rel_err(got, ref) <= 1e-2
    finally:
        L.lora_debug_withhold_gemm_stage(0)
        L.lora_debug_gemm_width(0)
