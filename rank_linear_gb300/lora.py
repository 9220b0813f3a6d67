"""Python face of the fused LoRA linear layer.

    Y  = X W^T + s (X A^T) B^T,   s = alpha / r
(ch05 "Acceleration principles: Triton kernels and fused LoRA", §5.3, LoRA
equation), with the backward's dX, dA and dB (W frozen; the gradient list of
ch05 §5.3).  Every step runs in the CUDA library through the C ABI; PyTorch
only allocates device memory and supplies the current stream.  The autograd
wrapper mirrors the custom autograd function with a hand-derived backward
that the Unsloth essay describes for LoRA.
"""
from __future__ import annotations

import torch

from . import _lib

_DT = {torch.bfloat16: _lib.LORA_BF16, torch.float32: _lib.LORA_FP32}


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise TypeError(f"unsupported dtype {t.dtype}; use bfloat16 or float32")
    return _DT[t.dtype]


def _ptr(t):
    return None if t is None else t.data_ptr() or None


def _check_dev(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def saved_bytes(M: int, r: int, dtype: torch.dtype) -> int:
    return int(_lib.lib().lora_linear_saved_bytes(M, r, _DT[dtype]))


def workspace_bytes(M: int, d_in: int, d_out: int, r: int, dtype: torch.dtype) -> int:
    return int(_lib.lib().lora_linear_workspace_bytes(M, d_in, d_out, r, _DT[dtype]))


def _buffer(nbytes: int, device) -> torch.Tensor:
    # 256-byte granules keep every sub-buffer 16-byte aligned
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)


def _stream_ptr(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream or None


def forward(X, W, A, B, alpha: float, *, Y=None, saved=None, workspace=None, stream=None):
    """Y = X W^T + (alpha/r) X A^T B^T.  Returns (Y, saved)."""
    _check_dev(X, W, A, B)
    M, d_in = X.shape
    d_out, r = B.shape
    dt = _dtype_code(X)
    L = _lib.lib()
    if Y is None:
        Y = torch.empty(M, d_out, dtype=X.dtype, device=X.device)
    if saved is None:
        saved = _buffer(L.lora_linear_saved_bytes(M, r, dt), X.device)
    ws_need = L.lora_linear_workspace_bytes(M, d_in, d_out, r, dt)
    if workspace is None:
        workspace = _buffer(ws_need, X.device)
    st = L.lora_linear_fwd(_ptr(X), _ptr(W), _ptr(A), _ptr(B), float(alpha), r, M, d_in, d_out,
                           dt, _ptr(Y), _ptr(saved), _ptr(workspace), workspace.numel(),
                           _stream_ptr(stream))
    _lib.check(st, "lora_linear_fwd")
    return Y, saved


def backward(dY, X, W, A, B, alpha: float, saved=None, *, need_dX=True, dX=None, dA=None,
             dB=None, workspace=None, stream=None):
    """Returns (dX or None, dA, dB) for the upstream gradient dY."""
    _check_dev(dY, X, W, A, B)
    M, d_in = X.shape
    d_out, r = B.shape
    dt = _dtype_code(X)
    L = _lib.lib()
    if need_dX and dX is None:
        dX = torch.empty(M, d_in, dtype=X.dtype, device=X.device)
    if dA is None:
        dA = torch.empty(r, d_in, dtype=X.dtype, device=X.device)
    if dB is None:
        dB = torch.empty(d_out, r, dtype=X.dtype, device=X.device)
    if workspace is None:
        workspace = _buffer(L.lora_linear_workspace_bytes(M, d_in, d_out, r, dt), X.device)
    st = L.lora_linear_bwd(_ptr(dY), _ptr(X), _ptr(W), _ptr(A), _ptr(B), _ptr(saved),
                           float(alpha), r, M, d_in, d_out, dt, _ptr(dX) if need_dX else None,
                           _ptr(dA), _ptr(dB), _ptr(workspace), workspace.numel(),
                           _stream_ptr(stream))
    _lib.check(st, "lora_linear_bwd")
    return (dX if need_dX else None), dA, dB


class LoRALinearFunction(torch.autograd.Function):
    """Autograd function: saves the low-rank activation for the backward."""

    @staticmethod
    def forward(ctx, X, W, A, B, alpha):
        shape = X.shape
        X2 = X.reshape(-1, shape[-1]).contiguous()
        Y, saved = forward(X2, W.contiguous(), A.contiguous(), B.contiguous(), alpha)
        ctx.save_for_backward(X2, W, A, B, saved)
        ctx.alpha = alpha
        ctx.x_shape = shape
        return Y.reshape(*shape[:-1], W.shape[0])

    @staticmethod
    def backward(ctx, dY):
        X2, W, A, B, saved = ctx.saved_tensors
        dY2 = dY.reshape(-1, dY.shape[-1]).contiguous()
        dX, dA, dB = backward(dY2, X2, W.contiguous(), A.contiguous(), B.contiguous(), ctx.alpha,
                              saved, need_dX=ctx.needs_input_grad[0])
        if dX is not None:
            dX = dX.reshape(ctx.x_shape)
        return dX, None, dA, dB, None


def lora_linear(X, W, A, B, alpha: float):
    """Y = X W^T + (alpha/r) (X A^T) B^T with gradients for X, A and B."""
    return LoRALinearFunction.apply(X, W, A, B, alpha)


def device_status(clear: bool = True) -> None:
    """Raise if a bounded device-side wait ran out since the last check."""
    _lib.check(_lib.lib().lora_device_status(1 if clear else 0), "device status")


def timing_events(n_pairs: int, stream=None):
    """Create 2*n_pairs timing events (recorded once so that the CUDA event
    objects exist) and the ctypes arrays the library's timing hook takes."""
    import ctypes
    st = stream if stream is not None else torch.cuda.current_stream()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n_pairs)]
    for e in evs:
        e.record(st)
    st.synchronize()
    arr = (ctypes.c_void_p * (2 * n_pairs))(*[e.cuda_event for e in evs])
    kinds = (ctypes.c_int * max(1, n_pairs))()
    return evs, arr, kinds


def launch_count() -> int:
    return int(_lib.lib().lora_launch_count())


# ---------------------------------------------------------------- SwiGLU pair
# H = silu(gate) * up with gate and up each a LoRA layer (ch05 "Acceleration
# principles: Triton kernels and fused LoRA", §5.6 fused SwiGLU, over the
# LoRA layer of §5.3); bf16 only.

def swiglu_saved_bytes(M: int, d_ff: int, r: int) -> int:
    return int(_lib.lib().lora_swiglu_saved_bytes(M, d_ff, r))


def swiglu_workspace_bytes(M: int, d_in: int, d_ff: int, r: int) -> int:
    return int(_lib.lib().lora_swiglu_workspace_bytes(M, d_in, d_ff, r))


def swiglu_forward(X, Wg, Ag, Bg, Wu, Au, Bu, alpha: float, *, H=None, saved=None,
                   workspace=None, stream=None, keep=True):
    """H = silu(gate) * up.  Returns (H, saved); saved holds gate and up for the
    backward, or is None with keep=False (inference: nothing is kept)."""
    _check_dev(X, Wg, Ag, Bg, Wu, Au, Bu)
    M, d_in = X.shape
    d_ff, r = Bg.shape
    dt = _dtype_code(X)
    L = _lib.lib()
    if H is None:
        H = torch.empty(M, d_ff, dtype=X.dtype, device=X.device)
    if saved is None and keep:
        saved = _buffer(L.lora_swiglu_saved_bytes(M, d_ff, r), X.device)
    if workspace is None:
        workspace = _buffer(L.lora_swiglu_workspace_bytes(M, d_in, d_ff, r), X.device)
    st = L.lora_swiglu_fwd(_ptr(X), _ptr(Wg), _ptr(Ag), _ptr(Bg), _ptr(Wu), _ptr(Au), _ptr(Bu),
                           float(alpha), r, M, d_in, d_ff, dt, _ptr(H), _ptr(saved),
                           _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _lib.check(st, "lora_swiglu_fwd")
    return H, saved


def swiglu_backward(dH, X, Wg, Ag, Bg, Wu, Au, Bu, alpha: float, saved, *, need_dX=True,
                    dX=None, dAg=None, dBg=None, dAu=None, dBu=None, workspace=None,
                    stream=None):
    """Returns (dX or None, dAg, dBg, dAu, dBu) for the upstream gradient dH."""
    _check_dev(dH, X, Wg, Ag, Bg, Wu, Au, Bu)
    M, d_in = X.shape
    d_ff, r = Bg.shape
    dt = _dtype_code(X)
    L = _lib.lib()
    new = lambda *s: torch.empty(*s, dtype=X.dtype, device=X.device)
    if need_dX and dX is None:
        dX = new(M, d_in)
    dAg = new(r, d_in) if dAg is None else dAg
    dAu = new(r, d_in) if dAu is None else dAu
    dBg = new(d_ff, r) if dBg is None else dBg
    dBu = new(d_ff, r) if dBu is None else dBu
    if workspace is None:
        workspace = _buffer(L.lora_swiglu_workspace_bytes(M, d_in, d_ff, r), X.device)
    st = L.lora_swiglu_bwd(_ptr(dH), _ptr(X), _ptr(Wg), _ptr(Ag), _ptr(Bg), _ptr(Wu), _ptr(Au),
                           _ptr(Bu), _ptr(saved), float(alpha), r, M, d_in, d_ff, dt,
                           _ptr(dX) if need_dX else None, _ptr(dAg), _ptr(dBg), _ptr(dAu),
                           _ptr(dBu), _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    _lib.check(st, "lora_swiglu_bwd")
    return (dX if need_dX else None), dAg, dBg, dAu, dBu


class LoRASwiGLUFunction(torch.autograd.Function):
    """Autograd function of the gated pair: saves gate, up and the low-rank
    activations for the backward."""

    @staticmethod
    def forward(ctx, X, Wg, Ag, Bg, Wu, Au, Bu, alpha):
        shape = X.shape
        X2 = X.reshape(-1, shape[-1]).contiguous()
        ws = [t.contiguous() for t in (Wg, Ag, Bg, Wu, Au, Bu)]
        H, saved = swiglu_forward(X2, *ws, alpha)
        ctx.save_for_backward(X2, *ws, saved)
        ctx.alpha = alpha
        ctx.x_shape = shape
        return H.reshape(*shape[:-1], Wg.shape[0])

    @staticmethod
    def backward(ctx, dH):
        X2, Wg, Ag, Bg, Wu, Au, Bu, saved = ctx.saved_tensors
        dH2 = dH.reshape(-1, dH.shape[-1]).contiguous()
        dX, dAg, dBg, dAu, dBu = swiglu_backward(dH2, X2, Wg, Ag, Bg, Wu, Au, Bu, ctx.alpha, saved,
                                                 need_dX=ctx.needs_input_grad[0])
        if dX is not None:
            dX = dX.reshape(ctx.x_shape)
        return dX, None, dAg, dBg, None, dAu, dBu, None


def lora_swiglu(X, Wg, Ag, Bg, Wu, Au, Bu, alpha: float):
    """silu(X Wg^T + s X Ag^T Bg^T) * (X Wu^T + s X Au^T Bu^T) with gradients for
    X and the four adapter matrices (Wg, Wu frozen)."""
    return LoRASwiGLUFunction.apply(X, Wg, Ag, Bg, Wu, Au, Bu, alpha)


# ---------------------------------------------------------------- fp8 frozen W
# The LoRA layer with its frozen-weight product on e4m3 values (ch05
# "Acceleration principles: Triton kernels and fused LoRA", §5.9 fp8 over the
# LoRA layer of §5.3): W quantised once with one power-of-two scale, X and dY
# per row on every call; the low-rank extension and dA, dB stay bf16.

class FP8Weight(tuple):
    """(Wq [d_out, d_in], WqT [d_in, d_out]) e4m3 bytes and w_scale (1 float)."""
    __slots__ = ()

    def __new__(cls, Wq, WqT, w_scale):
        return super().__new__(cls, (Wq, WqT, w_scale))

    Wq = property(lambda self: self[0])
    WqT = property(lambda self: self[1])
    w_scale = property(lambda self: self[2])


def quantize_w_fp8(W, stream=None) -> FP8Weight:
    """Quantise a frozen bf16 W once for the fp8 layer."""
    _check_dev(W)
    d_out, d_in = W.shape
    L = _lib.lib()
    Wq = torch.empty(d_out, d_in, dtype=torch.uint8, device=W.device)
    WqT = torch.empty(d_in, d_out, dtype=torch.uint8, device=W.device)
    scale = torch.empty(1, dtype=torch.float32, device=W.device)
    ws = _buffer(L.lora_fp8_quantize_w_workspace_bytes(), W.device)
    _lib.check(L.lora_fp8_quantize_w(_ptr(W), d_out, d_in, _ptr(Wq), _ptr(WqT), _ptr(scale),
                                     _ptr(ws), ws.numel(), _stream_ptr(stream)),
               "lora_fp8_quantize_w")
    return FP8Weight(Wq, WqT, scale)


def quantize_rows_fp8(x, stream=None):
    """(codes [rows, cols] uint8, scale [rows] float32) of a bf16 matrix."""
    _check_dev(x)
    rows, cols = x.shape
    q = torch.empty(rows, cols, dtype=torch.uint8, device=x.device)
    scale = torch.empty(max(rows, 1), dtype=torch.float32, device=x.device)
    _lib.check(_lib.lib().lora_fp8_quantize_rows(_ptr(x), rows, cols, _ptr(q), _ptr(scale),
                                                  _stream_ptr(stream)), "lora_fp8_quantize_rows")
    return q, scale[:rows]


def fp8_workspace_bytes(M: int, d_in: int, d_out: int, r: int) -> int:
    return int(_lib.lib().lora_fp8_workspace_bytes(M, d_in, d_out, r))


def fp8_forward(X, qw: FP8Weight, A, B, alpha: float, *, Y=None, saved=None, workspace=None,
                stream=None):
    """Y = Q(X) Q(W)^T + (alpha/r) X A^T B^T.  Returns (Y, saved)."""
    _check_dev(X, A, B)
    M, d_in = X.shape
    d_out, r = B.shape
    L = _lib.lib()
    if Y is None:
        Y = torch.empty(M, d_out, dtype=X.dtype, device=X.device)
    if saved is None:
        saved = _buffer(L.lora_linear_saved_bytes(M, r, _lib.LORA_BF16), X.device)
    if workspace is None:
        workspace = _buffer(L.lora_fp8_workspace_bytes(M, d_in, d_out, r), X.device)
    st = L.lora_fp8_fwd(_ptr(X), _ptr(qw.Wq), _ptr(qw.w_scale), _ptr(A), _ptr(B), float(alpha),
                        r, M, d_in, d_out, _ptr(Y), _ptr(saved), _ptr(workspace),
                        workspace.numel(), _stream_ptr(stream))
    _lib.check(st, "lora_fp8_fwd")
    return Y, saved


def fp8_backward(dY, X, qw: FP8Weight, A, B, alpha: float, saved, *, need_dX=True, dX=None,
                 dA=None, dB=None, workspace=None, stream=None):
    """Returns (dX or None, dA, dB) for the upstream gradient dY."""
    _check_dev(dY, X, A, B)
    M, d_in = X.shape
    d_out, r = B.shape
    L = _lib.lib()
    if need_dX and dX is None:
        dX = torch.empty(M, d_in, dtype=X.dtype, device=X.device)
    dA = torch.empty(r, d_in, dtype=X.dtype, device=X.device) if dA is None else dA
    dB = torch.empty(d_out, r, dtype=X.dtype, device=X.device) if dB is None else dB
    if workspace is None:
        workspace = _buffer(L.lora_fp8_workspace_bytes(M, d_in, d_out, r), X.device)
    st = L.lora_fp8_bwd(_ptr(dY), _ptr(X), _ptr(qw.WqT), _ptr(qw.w_scale), _ptr(A), _ptr(B),
                        _ptr(saved), float(alpha), r, M, d_in, d_out,
                        _ptr(dX) if need_dX else None, _ptr(dA), _ptr(dB), _ptr(workspace),
                        workspace.numel(), _stream_ptr(stream))
    _lib.check(st, "lora_fp8_bwd")
    return (dX if need_dX else None), dA, dB


# The LoRA layer over a 4-bit frozen W (ch05 "Acceleration principles: Triton
# kernels and fused LoRA", §5.3's layer with QLoRA's 4-bit base weight, and
# the Unsloth inference notes' on-chip dequantisation): symmetric INT4 codes
# with one bf16 scale per 64 weights along d_in, expanded to bf16 in shared
# memory inside the GEMMs.

class Q4Weight(tuple):
    """(codes [d_out, d_in / 2] uint8, scales [d_in / 64, d_out] bf16)."""
    __slots__ = ()

    def __new__(cls, codes, scales):
        return super().__new__(cls, (codes, scales))

    codes = property(lambda self: self[0])
    scales = property(lambda self: self[1])


def quantize_w_q4(W, stream=None) -> Q4Weight:
    """Quantise a frozen bf16 W [d_out, d_in] (d_in % 64 == 0) to 4 bits once."""
    _check_dev(W)
    d_out, d_in = W.shape
    codes = torch.empty(d_out, d_in // 2, dtype=torch.uint8, device=W.device)
    scales = torch.empty(max(d_in // 64, 1), d_out, dtype=torch.bfloat16, device=W.device)
    _lib.check(_lib.lib().lora_q4_quantize_w(_ptr(W), d_out, d_in, _ptr(codes), _ptr(scales),
                                             _stream_ptr(stream)), "lora_q4_quantize_w")
    return Q4Weight(codes, scales)


def dequantize_w_q4(qw: Q4Weight, stream=None):
    """The bf16 W [d_out, d_in] the 4-bit layer computes with."""
    d_out, half = qw.codes.shape
    Wd = torch.empty(d_out, 2 * half, dtype=torch.bfloat16, device=qw.codes.device)
    _lib.check(_lib.lib().lora_q4_dequantize_w(_ptr(qw.codes), _ptr(qw.scales), d_out, 2 * half,
                                               _ptr(Wd), _stream_ptr(stream)),
               "lora_q4_dequantize_w")
    return Wd


def q4_forward(X, qw: Q4Weight, A, B, alpha: float, *, Y=None, saved=None, workspace=None,
               stream=None):
    """Y = X Wd^T + (alpha/r) X A^T B^T.  Returns (Y, saved)."""
    _check_dev(X, A, B, qw.codes, qw.scales)
    M, d_in = X.shape
    d_out, r = B.shape
    L = _lib.lib()
    if Y is None:
        Y = torch.empty(M, d_out, dtype=X.dtype, device=X.device)
    if saved is None:
        saved = _buffer(L.lora_linear_saved_bytes(M, r, _lib.LORA_BF16), X.device)
    if workspace is None:
        workspace = _buffer(L.lora_linear_workspace_bytes(M, d_in, d_out, r, _lib.LORA_BF16),
                            X.device)
    st = L.lora_q4_fwd(_ptr(X), _ptr(qw.codes), _ptr(qw.scales), _ptr(A), _ptr(B), float(alpha),
                       r, M, d_in, d_out, _ptr(Y), _ptr(saved), _ptr(workspace),
                       workspace.numel(), _stream_ptr(stream))
    _lib.check(st, "lora_q4_fwd")
    return Y, saved


def q4_backward(dY, X, qw: Q4Weight, A, B, alpha: float, saved=None, *, need_dX=True, dX=None,
                dA=None, dB=None, workspace=None, stream=None):
    """Returns (dX or None, dA, dB) for the upstream gradient dY."""
    _check_dev(dY, X, A, B, qw.codes, qw.scales)
    M, d_in = X.shape
    d_out, r = B.shape
    L = _lib.lib()
    if need_dX and dX is None:
        dX = torch.empty(M, d_in, dtype=X.dtype, device=X.device)
    dA = torch.empty(r, d_in, dtype=X.dtype, device=X.device) if dA is None else dA
    dB = torch.empty(d_out, r, dtype=X.dtype, device=X.device) if dB is None else dB
    if workspace is None:
        workspace = _buffer(L.lora_linear_workspace_bytes(M, d_in, d_out, r, _lib.LORA_BF16),
                            X.device)
    st = L.lora_q4_bwd(_ptr(dY), _ptr(X), _ptr(qw.codes), _ptr(qw.scales), _ptr(A), _ptr(B),
                       _ptr(saved), float(alpha), r, M, d_in, d_out,
                       _ptr(dX) if need_dX else None, _ptr(dA), _ptr(dB), _ptr(workspace),
                       workspace.numel(), _stream_ptr(stream))
    _lib.check(st, "lora_q4_bwd")
    return (dX if need_dX else None), dA, dB


# ---------------------------------------------------------------- autograd: quantised W

class LoRAFP8Function(torch.autograd.Function):
    """Autograd function of the layer with an fp8 frozen-W product."""

    @staticmethod
    def forward(ctx, X, Wq, WqT, w_scale, A, B, alpha):
        shape = X.shape
        X2 = X.reshape(-1, shape[-1]).contiguous()
        A, B = A.contiguous(), B.contiguous()
        qw = FP8Weight(Wq, WqT, w_scale)
        Y, saved = fp8_forward(X2, qw, A, B, alpha)
        ctx.save_for_backward(X2, Wq, WqT, w_scale, A, B, saved)
        ctx.alpha = alpha
        ctx.x_shape = shape
        return Y.reshape(*shape[:-1], B.shape[0])

    @staticmethod
    def backward(ctx, dY):
        X2, Wq, WqT, w_scale, A, B, saved = ctx.saved_tensors
        dY2 = dY.reshape(-1, dY.shape[-1]).contiguous()
        dX, dA, dB = fp8_backward(dY2, X2, FP8Weight(Wq, WqT, w_scale), A, B, ctx.alpha, saved,
                                  need_dX=ctx.needs_input_grad[0])
        if dX is not None:
            dX = dX.reshape(ctx.x_shape)
        return dX, None, None, None, dA, dB, None


def lora_linear_fp8(X, qw: FP8Weight, A, B, alpha: float):
    """Q(X) Q(W)^T + (alpha/r) (X A^T) B^T with gradients for X, A and B."""
    return LoRAFP8Function.apply(X, qw.Wq, qw.WqT, qw.w_scale, A, B, alpha)


class LoRAQ4Function(torch.autograd.Function):
    """Autograd function of the layer over a 4-bit frozen W."""

    @staticmethod
    def forward(ctx, X, codes, scales, A, B, alpha):
        shape = X.shape
        X2 = X.reshape(-1, shape[-1]).contiguous()
        A, B = A.contiguous(), B.contiguous()
        Y, saved = q4_forward(X2, Q4Weight(codes, scales), A, B, alpha)
        ctx.save_for_backward(X2, codes, scales, A, B, saved)
        ctx.alpha = alpha
        ctx.x_shape = shape
        return Y.reshape(*shape[:-1], B.shape[0])

    @staticmethod
    def backward(ctx, dY):
        X2, codes, scales, A, B, saved = ctx.saved_tensors
        dY2 = dY.reshape(-1, dY.shape[-1]).contiguous()
        dX, dA, dB = q4_backward(dY2, X2, Q4Weight(codes, scales), A, B, ctx.alpha, saved,
                                 need_dX=ctx.needs_input_grad[0])
        if dX is not None:
            dX = dX.reshape(ctx.x_shape)
        return dX, None, None, dA, dB, None


def lora_linear_q4(X, qw: Q4Weight, A, B, alpha: float):
    """X Wd^T + (alpha/r) (X A^T) B^T over the 4-bit W, with gradients for X, A and B."""
    return LoRAQ4Function.apply(X, qw.codes, qw.scales, A, B, alpha)
