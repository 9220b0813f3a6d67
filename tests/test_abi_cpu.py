"""The C ABI library loads, exports every declared entry point, and rejects
bad arguments with a status before touching CUDA (CPU only: no launches)."""
import ctypes
import os
import re

import pytest

from rank_linear_gb300 import _lib, build

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include")
HEADERS = sorted(os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h"))
L = None


def setup_module():
    global L
    build.build()
    L = _lib.lib()


def declared_functions():
    src = "".join(open(h).read() for h in HEADERS)
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lora_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(_lib.SIGNATURES), "binding and header disagree"


def test_status_strings():
    for code, name in enumerate(["LORA_OK", "LORA_ERR_INVALID_ARG", "LORA_ERR_UNSUPPORTED",
                                 "LORA_ERR_WORKSPACE", "LORA_ERR_CUDA", "LORA_ERR_TIMEOUT"]):
        assert L.lora_status_string(code).decode() == name


def test_sizes():
    # bf16: sH [M, r_pad] + transposed copy [r_pad, roundup(M, 8)], 256-B aligned
    assert L.lora_linear_saved_bytes(4096, 16, _lib.LORA_BF16) == 4096 * 16 * 2 * 2
    assert L.lora_linear_saved_bytes(100, 8, _lib.LORA_BF16) == 3328 + 16 * 104 * 2
    assert L.lora_linear_saved_bytes(0, 16, _lib.LORA_BF16) == 0
    assert L.lora_linear_saved_bytes(64, 8, _lib.LORA_FP32) == 64 * 8 * 4
    assert L.lora_linear_saved_bytes(64, 0, _lib.LORA_BF16) == 0
    ws = L.lora_linear_workspace_bytes(4096, 4096, 4096, 16, _lib.LORA_BF16)
    # B^T [16, 4096] + sG [4096, 16] + sG^T [16, 4096] + the dX GEMM's tail split
    # (no GPU here: sized for 76 CTA pairs; 256 pair tiles leave 28 in the last
    # wave, split 2 ways: 28 x 2 ranges x 2 CTAs x 128 x 256 fp32, and 2 x 28
    # counters) + room for a recomputed saved buffer
    split = 28 * 2 * 2 * 128 * 256 * 4 + 256
    assert ws == 3 * 4096 * 16 * 2 + split + 4096 * 16 * 2 * 2
    base = 16 * 14336 * 2 + 2 * 8192 * 16 * 2 + 8192 * 16 * 2 * 2
    # gate/up: the dX GEMM (N = 4096, K = 14336 + 64) takes 256 x 512 tiles,
    # 256 of them, 28 in the last wave, split 2 ways: 28 x 2 ranges x 2 CTAs x
    # 128 x 512 fp32 + the counters
    ws2 = L.lora_linear_workspace_bytes(8192, 4096, 14336, 16, _lib.LORA_BF16)
    assert ws2 == base + 28 * 2 * 2 * 128 * 512 * 4 + 256
    # shapes whose last wave is more than half full at either tile width
    # (1792 or 896 tiles: 44 or 60 in the last wave) are not split
    ws3 = L.lora_linear_workspace_bytes(8192, 14336, 14336, 16, _lib.LORA_BF16)
    assert ws3 == base
    assert L.lora_linear_workspace_bytes(0, 64, 64, 16, _lib.LORA_BF16) == 0


FAKE = 0x100000  # aligned non-null "device" address; never dereferenced here


def fwd(**kw):
    a = dict(X=FAKE, W=FAKE, A=FAKE, B=FAKE, alpha=16.0, r=16, M=128, d_in=256, d_out=256,
             dt=_lib.LORA_BF16, Y=FAKE, saved=FAKE, ws=FAKE, ws_bytes=1 << 30)
    a.update(kw)
    return L.lora_linear_fwd(a["X"], a["W"], a["A"], a["B"], a["alpha"], a["r"], a["M"],
                             a["d_in"], a["d_out"], a["dt"], a["Y"], a["saved"], a["ws"],
                             a["ws_bytes"], None)


def bwd(**kw):
    a = dict(dY=FAKE, X=FAKE, W=FAKE, A=FAKE, B=FAKE, saved=FAKE, alpha=16.0, r=16, M=128,
             d_in=256, d_out=256, dt=_lib.LORA_BF16, dX=FAKE, dA=FAKE, dB=FAKE, ws=FAKE,
             ws_bytes=1 << 30)
    a.update(kw)
    return L.lora_linear_bwd(a["dY"], a["X"], a["W"], a["A"], a["B"], a["saved"], a["alpha"],
                             a["r"], a["M"], a["d_in"], a["d_out"], a["dt"], a["dX"], a["dA"],
                             a["dB"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(r=0), _lib.LORA_ERR_INVALID_ARG),
    (dict(r=257), _lib.LORA_ERR_INVALID_ARG),
    (dict(M=-1), _lib.LORA_ERR_INVALID_ARG),
    (dict(d_in=0), _lib.LORA_ERR_INVALID_ARG),
    (dict(dt=7), _lib.LORA_ERR_INVALID_ARG),
    (dict(alpha=float("nan")), _lib.LORA_ERR_INVALID_ARG),
    (dict(X=None), _lib.LORA_ERR_INVALID_ARG),
    (dict(W=None), _lib.LORA_ERR_INVALID_ARG),
    (dict(Y=None), _lib.LORA_ERR_INVALID_ARG),
    (dict(saved=None), _lib.LORA_ERR_INVALID_ARG),
    (dict(A=FAKE + 8), _lib.LORA_ERR_INVALID_ARG),
    (dict(d_in=260), _lib.LORA_ERR_UNSUPPORTED),
    (dict(d_out=100), _lib.LORA_ERR_UNSUPPORTED),
    (dict(M=1 << 29), _lib.LORA_ERR_UNSUPPORTED),
    (dict(r=12, ws=None, ws_bytes=0), _lib.LORA_ERR_WORKSPACE),   # r % 8 != 0 pads B
    (dict(r=12, ws_bytes=16), _lib.LORA_ERR_WORKSPACE),
])
def test_fwd_rejects(kw, code):
    assert fwd(**kw) == code
    assert L.lora_last_error().decode() != ""


@pytest.mark.parametrize("kw,code", [
    (dict(dY=None), _lib.LORA_ERR_INVALID_ARG),
    (dict(dA=None), _lib.LORA_ERR_INVALID_ARG),
    (dict(dB=None), _lib.LORA_ERR_INVALID_ARG),
    (dict(dB=FAKE + 2), _lib.LORA_ERR_INVALID_ARG),
    (dict(ws=None, ws_bytes=0), _lib.LORA_ERR_WORKSPACE),
    (dict(ws_bytes=1024), _lib.LORA_ERR_WORKSPACE),
    (dict(saved=None, ws_bytes=3 * 128 * 16 * 2 + 256), _lib.LORA_ERR_WORKSPACE),
    (dict(dt=_lib.LORA_FP32, ws_bytes=4), _lib.LORA_ERR_WORKSPACE),
    (dict(d_out=12), _lib.LORA_ERR_UNSUPPORTED),
    (dict(r=300), _lib.LORA_ERR_INVALID_ARG),
])
def test_bwd_rejects(kw, code):
    assert bwd(**kw) == code


def bwd_noalloc(**kw):
    a = dict(dY=FAKE, X=FAKE, W=FAKE, A=FAKE, B=FAKE, saved=FAKE, alpha=16.0, r=16, M=128,
             d_in=256, d_out=256, dt=_lib.LORA_BF16, dX=FAKE, dA=FAKE, dB=FAKE)
    a.update(kw)
    return L.lora_linear_bwd_noalloc(a["dY"], a["X"], a["W"], a["A"], a["B"], a["saved"],
                                     a["alpha"], a["r"], a["M"], a["d_in"], a["d_out"], a["dt"],
                                     a["dX"], a["dA"], a["dB"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(dY=None), _lib.LORA_ERR_INVALID_ARG),
    (dict(dB=FAKE + 2), _lib.LORA_ERR_INVALID_ARG),
    (dict(r=300), _lib.LORA_ERR_INVALID_ARG),
    (dict(d_out=12), _lib.LORA_ERR_UNSUPPORTED),
    # more scratch than the built-in array holds
    (dict(M=8200, d_in=64, d_out=16384, r=256), _lib.LORA_ERR_UNSUPPORTED),
])
def test_bwd_noalloc_rejects(kw, code):
    n0 = L.lora_launch_count()
    assert bwd_noalloc(**kw) == code
    assert L.lora_launch_count() == n0


def _no_device() -> bool:
    import torch
    return not torch.cuda.is_available()


@pytest.mark.skipif(not _no_device(),
                    reason="valid arguments with fake pointers: only where no device can run them")
def test_bwd_noalloc_device_status_is_that_of_bwd():
    """Valid arguments (fake pointers, so only where no device is usable):
    the allocation-free backward checks the device the way lora_linear_bwd
    does, before it looks up its array, so both return the same status and
    launch nothing."""
    n0 = L.lora_launch_count()
    a = bwd()
    b = bwd_noalloc()
    assert a == b
    assert a in (_lib.LORA_ERR_CUDA, _lib.LORA_ERR_UNSUPPORTED)
    assert L.lora_launch_count() == n0


def test_timing_hook_set_and_clear():
    assert L.lora_set_timing_events(None, None, 0) == _lib.LORA_OK
    assert L.lora_timing_used() == 0


def test_swiglu_sizes_and_rejects():
    M, d_in, d_ff, r = 300, 64, 200, 16
    # gate, up [M, d_ff] + [sH_g | sH_u] [M, 32] + two transposes [16, 304], 256-byte granules
    rup = lambda x: (x + 255) // 256 * 256
    assert L.lora_swiglu_saved_bytes(M, d_ff, r) == (2 * rup(M * d_ff * 2) + rup(M * 32 * 2)
                                                     + 2 * rup(16 * 304 * 2))
    assert L.lora_swiglu_saved_bytes(0, d_ff, r) == 0
    assert L.lora_swiglu_saved_bytes(M, d_ff, 0) == 0
    assert L.lora_swiglu_workspace_bytes(M, d_in, d_ff, 300) == 0
    fake = ctypes.c_void_p(4096)
    args = lambda dt=_lib.LORA_BF16, r=16, d_ff=200: (fake,) * 7 + (
        32.0, r, M, d_in, d_ff, dt, fake, fake, None, 0, None)
    assert L.lora_swiglu_fwd(*args(dt=_lib.LORA_FP32)) == _lib.LORA_ERR_UNSUPPORTED
    assert L.lora_swiglu_fwd(*args(r=0)) == _lib.LORA_ERR_INVALID_ARG
    assert L.lora_swiglu_fwd(*args(d_ff=204)) == _lib.LORA_ERR_UNSUPPORTED
    bad = list(args())
    bad[1] = None  # Wg
    assert L.lora_swiglu_fwd(*bad) == _lib.LORA_ERR_INVALID_ARG
    # the backward needs the saved buffer and a workspace
    bwd = (fake,) * 8 + (None, 32.0, 16, M, d_in, 200, _lib.LORA_BF16) + (fake,) * 5 + (
        fake, 1 << 40, None)
    assert L.lora_swiglu_bwd(*bwd) == _lib.LORA_ERR_INVALID_ARG
    bwd = (fake,) * 9 + (32.0, 16, M, d_in, 200, _lib.LORA_BF16) + (fake,) * 5 + (None, 0, None)
    assert L.lora_swiglu_bwd(*bwd) == _lib.LORA_ERR_WORKSPACE


def test_q4_rejects():
    fake = ctypes.c_void_p(4096)
    M = 300
    fwd = lambda d_in=256, d_out=128, r=16, codes=fake, ws=(fake, 1 << 40): (
        fake, codes, fake, fake, fake, 32.0, r, M, d_in, d_out, fake, fake) + ws + (None,)
    assert L.lora_q4_fwd(*fwd(d_in=96)) == _lib.LORA_ERR_UNSUPPORTED
    assert L.lora_q4_fwd(*fwd(d_out=12)) == _lib.LORA_ERR_UNSUPPORTED
    assert L.lora_q4_fwd(*fwd(r=0)) == _lib.LORA_ERR_INVALID_ARG
    assert L.lora_q4_fwd(*fwd(codes=None)) == _lib.LORA_ERR_INVALID_ARG
    assert L.lora_q4_fwd(*fwd(r=12, ws=(None, 0))) == _lib.LORA_ERR_WORKSPACE  # pad of B
    bwd = lambda d_in=256, saved=fake, ws=(fake, 1 << 40): (
        fake, fake, fake, fake, fake, fake, saved, 32.0, 16, M, d_in, 128, fake, fake,
        fake) + ws + (None,)
    assert L.lora_q4_bwd(*bwd(d_in=100)) == _lib.LORA_ERR_UNSUPPORTED
    assert L.lora_q4_bwd(*bwd(ws=(None, 0))) == _lib.LORA_ERR_WORKSPACE
    assert L.lora_q4_quantize_w(fake, 128, 96, fake, fake, None) == _lib.LORA_ERR_UNSUPPORTED
    assert L.lora_q4_quantize_w(fake, 128, 128, None, fake, None) == _lib.LORA_ERR_INVALID_ARG
    assert L.lora_q4_dequantize_w(fake, fake, 128, 32, fake, None) == _lib.LORA_ERR_UNSUPPORTED


def test_withhold_hook_arguments():
    assert L.lora_debug_withhold_arrive(-1) == _lib.LORA_ERR_INVALID_ARG
    assert L.lora_debug_withhold_arrive(0) == _lib.LORA_OK


def test_product_path_needs_the_library(monkeypatch, tmp_path):
    """Without the built library the Python layer raises; it has no fallback."""
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU or PyTorch fallback"):
        _lib.lib()
