"""Fused LoRA linear layer (forward + backward, frozen base weight) for one
GB300 (sm_103a), as hand-written CUDA behind a C ABI.

Importing this package does not load the CUDA library; the first call does,
and fails loudly if it has not been built.
"""
from .lora import (LoRALinearFunction, LoRASwiGLUFunction, backward, device_status, forward,
                   launch_count, lora_linear, lora_swiglu, saved_bytes, swiglu_backward,
                   swiglu_forward, swiglu_saved_bytes, swiglu_workspace_bytes, timing_events,
                   workspace_bytes)

__all__ = ["LoRALinearFunction", "LoRASwiGLUFunction", "backward", "device_status", "forward",
           "launch_count", "lora_linear", "lora_swiglu", "saved_bytes", "swiglu_backward",
           "swiglu_forward", "swiglu_saved_bytes", "swiglu_workspace_bytes", "timing_events",
           "workspace_bytes"]
