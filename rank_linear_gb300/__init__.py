"""Fused LoRA linear layer (forward + backward, frozen base weight) for one
GB300 (sm_103a), as hand-written CUDA behind a C ABI.

Importing this package does not load the CUDA library; the first call does,
and fails loudly if it has not been built.
"""
from .lora import (FP8Weight, Q4Weight, dequantize_w_q4, q4_backward, q4_forward,
                   quantize_w_q4, LoRAFP8Function, LoRAQ4Function, lora_linear_fp8,
                   lora_linear_q4, LoRALinearFunction, LoRASwiGLUFunction, backward, device_status,
                   forward, fp8_backward, fp8_forward, fp8_workspace_bytes, launch_count,
                   lora_linear, lora_swiglu, quantize_rows_fp8, quantize_w_fp8, saved_bytes,
                   swiglu_backward,
                   swiglu_forward, swiglu_saved_bytes, swiglu_workspace_bytes, timing_events,
                   workspace_bytes)

__all__ = ["FP8Weight", "Q4Weight", "dequantize_w_q4", "q4_backward", "q4_forward",
           "quantize_w_q4", "LoRAFP8Function", "LoRAQ4Function", "lora_linear_fp8",
           "lora_linear_q4", "LoRALinearFunction", "LoRASwiGLUFunction", "backward", "device_status",
           "forward", "fp8_backward", "fp8_forward", "fp8_workspace_bytes", "quantize_rows_fp8", "quantize_w_fp8",
           "launch_count", "lora_linear", "lora_swiglu", "saved_bytes", "swiglu_backward",
           "swiglu_forward", "swiglu_saved_bytes", "swiglu_workspace_bytes", "timing_events",
           "workspace_bytes"]
