"""Fused LoRA linear layer (forward + backward, frozen base weight) for one
GB300 (sm_103a), as hand-written CUDA behind a C ABI.

Importing this package does not load the CUDA library; the first call does,
and fails loudly if it has not been built.
"""
from .lora import (LoRALinearFunction, backward, device_status, forward, launch_count,
                   timing_events,
                   lora_linear, saved_bytes, workspace_bytes)

__all__ = ["LoRALinearFunction", "backward", "device_status", "forward", "launch_count",
           "lora_linear", "saved_bytes", "timing_events", "workspace_bytes"]
