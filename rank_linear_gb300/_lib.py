"""ctypes binding of the C ABI in include/lora_linear.h (marshalling only).

The library is required: loading fails loudly if `liblora_linear.so` has not
been built; there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liblora_linear.so")

LORA_OK, LORA_ERR_INVALID_ARG, LORA_ERR_UNSUPPORTED, LORA_ERR_WORKSPACE, \
    LORA_ERR_CUDA, LORA_ERR_TIMEOUT = range(6)
LORA_BF16, LORA_FP32 = 0, 1
KERNEL_KINDS = ["prep", "down_fwd", "main_fwd", "down_bwd", "main_bwd", "grad_a", "grad_b",
                "down_bwd_grad_b", "swiglu_grad", "quant", "grad_a_b"]

_vp, _i64, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
_int, _f32 = ctypes.c_int, ctypes.c_float

SIGNATURES = {
    "lora_linear_saved_bytes": ([_i64, _int, _int], _sz),
    "lora_linear_workspace_bytes": ([_i64, _i64, _i64, _int, _int], _sz),
    "lora_linear_fwd": ([_vp, _vp, _vp, _vp, _f32, _int, _i64, _i64, _i64, _int,
                         _vp, _vp, _vp, _sz, _vp], _int),
    "lora_linear_bwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _f32, _int, _i64, _i64, _i64, _int,
                         _vp, _vp, _vp, _vp, _sz, _vp], _int),
    "lora_linear_bwd_noalloc": ([_vp, _vp, _vp, _vp, _vp, _vp, _f32, _int, _i64, _i64, _i64,
                                 _int, _vp, _vp, _vp, _vp], _int),
    "lora_status_string": ([_int], ctypes.c_char_p),
    "lora_last_error": ([], ctypes.c_char_p),
    "lora_device_status": ([_int], _int),
    "lora_launch_count": ([], ctypes.c_uint64),
    "lora_set_timing_events": ([ctypes.POINTER(_vp), ctypes.POINTER(_int), _int], _int),
    "lora_debug_withhold_arrive": ([_int], _int),
    "lora_debug_gemm_width": ([_int], _int),
    "lora_debug_withhold_gemm_stage": ([_int], _int),
    "lora_timing_used": ([], _int),
    "lora_fp8_quantize_w_workspace_bytes": ([], _sz),
    "lora_fp8_quantize_w": ([_vp, _i64, _i64, _vp, _vp, _vp, _vp, _sz, _vp], _int),
    "lora_fp8_quantize_rows": ([_vp, _i64, _i64, _vp, _vp, _vp], _int),
    "lora_fp8_workspace_bytes": ([_i64, _i64, _i64, _int], _sz),
    "lora_fp8_fwd": ([_vp, _vp, _vp, _vp, _vp, _f32, _int, _i64, _i64, _i64, _vp, _vp, _vp,
                      _sz, _vp], _int),
    "lora_fp8_bwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _f32, _int, _i64, _i64, _i64, _vp,
                      _vp, _vp, _vp, _sz, _vp], _int),
    "lora_q4_quantize_w": ([_vp, _i64, _i64, _vp, _vp, _vp], _int),
    "lora_q4_dequantize_w": ([_vp, _vp, _i64, _i64, _vp, _vp], _int),
    "lora_q4_fwd": ([_vp, _vp, _vp, _vp, _vp, _f32, _int, _i64, _i64, _i64, _vp, _vp, _vp, _sz,
                     _vp], _int),
    "lora_q4_bwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _f32, _int, _i64, _i64, _i64, _vp, _vp,
                     _vp, _vp, _sz, _vp], _int),
    "lora_swiglu_saved_bytes": ([_i64, _i64, _int], _sz),
    "lora_swiglu_workspace_bytes": ([_i64, _i64, _i64, _int], _sz),
    "lora_swiglu_fwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _f32, _int, _i64, _i64, _i64, _int,
                         _vp, _vp, _vp, _sz, _vp], _int),
    "lora_swiglu_bwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _f32, _int, _i64, _i64,
                         _i64, _int, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _int),
}

_lib = None
_lock = threading.Lock()


class LoraError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


def lib():
    """The loaded library (built on first use if sources are present)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -m rank_linear_gb300.build` "
                    "(nvcc, sm_103a); there is no CPU or PyTorch fallback")
            L = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in SIGNATURES.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = res
            _lib = L
        return _lib


def check(status: int, what: str = "lora call") -> None:
    if status != LORA_OK:
        L = lib()
        name = L.lora_status_string(status).decode()
        detail = L.lora_last_error().decode()
        raise LoraError(status, f"{what}: {name}: {detail}")
