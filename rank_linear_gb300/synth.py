"""Seeded synthetic inputs for the LoRA linear layer.

This module only draws random tensors and names workloads; it holds none of
the layer's arithmetic.  Both the CUDA path (tests, bench) and the CPU oracle
take their inputs from here, so the two always see the same stored values.

Workloads follow the layer shapes the pages use: a Llama-3-8B q_proj
(4096 x 4096 with rank-16 adapters, ch01 "Project background", §1.2), the
Llama-3-8B MLP projections, and a Qwen-class wide FFN (FFN width 27,648 from
the Qwen inference post's table).  LoRA rank and alpha follow the usual
r / alpha = 2r conventions of the Unsloth essay's VLM recipe table.

Distributions (0.02 is a standard deviation):
    X  ~ N(0, 1)               [M, d_in]
    W  ~ N(0, 1/d_in)          [d_out, d_in]   (frozen base weight)
    A  ~ U(-1/sqrt(d_in), +1/sqrt(d_in))   [r, d_in]
    B  ~ N(0, 0.02^2)          [d_out, r]
    dY ~ N(0, 1)               [M, d_out]     (upstream gradient)
drawn in the order X, W, A, B, dY from one torch.Generator, in fp32, then
cast to the workload dtype.
"""
from __future__ import annotations

from dataclasses import dataclass, asdict

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    M: int        # tokens (batch x sequence)
    d_in: int
    d_out: int
    r: int
    alpha: float
    dtype: str    # "bf16" or "fp32"
    # "linear": one LoRA layer; "swiglu": the gate/up pair, d_out = FFN width
    # (the up projection's W, A, B are drawn with seed + 1000); "fp8": one
    # LoRA layer whose frozen-W product runs on e4m3 values; "q4": one LoRA
    # layer over a 4-bit frozen W (codes + bf16 scales per 64 weights)
    layer: str = "linear"

    def as_dict(self) -> dict:
        return asdict(self)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_fp32", 64, 256, 256, 8, 16.0, "fp32"),
        Workload("llama3_8b_q_proj", 4096, 4096, 4096, 16, 16.0, "bf16"),
        Workload("llama3_8b_gate_up", 8192, 4096, 14336, 16, 32.0, "bf16"),
        Workload("llama3_8b_down_proj", 8192, 14336, 4096, 64, 128.0, "bf16"),
        Workload("qwen_wide_ffn", 16384, 5120, 27648, 128, 256.0, "bf16"),
        Workload("llama3_8b_swiglu_gate_up", 8192, 4096, 14336, 16, 32.0, "bf16", "swiglu"),
        Workload("llama3_8b_q_proj_fp8", 4096, 4096, 4096, 16, 16.0, "bf16", "fp8"),
        Workload("llama3_8b_gate_up_fp8", 8192, 4096, 14336, 16, 32.0, "bf16", "fp8"),
        Workload("llama3_8b_q_proj_q4", 4096, 4096, 4096, 16, 16.0, "bf16", "q4"),
        Workload("llama3_8b_gate_up_q4", 8192, 4096, 14336, 16, 32.0, "bf16", "q4"),
    ]
}

TORCH_DTYPES = {"bf16": torch.bfloat16, "fp32": torch.float32}


def make_inputs(M: int, d_in: int, d_out: int, r: int, dtype: str = "bf16",
                seed: int = 0, device: str | torch.device = "cpu",
                which: str = "X,W,A,B,dY") -> dict:
    """Draw X, W, A, B, dY (in that order) from one seeded generator.

    `which` selects the tensors returned; all five are always drawn so the
    values of each tensor do not depend on the selection.
    """
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    f32 = dict(dtype=torch.float32, device=dev, generator=g)
    out = {}
    out["X"] = torch.randn(M, d_in, **f32)
    out["W"] = torch.randn(d_out, d_in, **f32).mul_(d_in ** -0.5)
    out["A"] = torch.rand(r, d_in, **f32).mul_(2.0).sub_(1.0).mul_(d_in ** -0.5)
    out["B"] = torch.randn(d_out, r, **f32).mul_(0.02)
    out["dY"] = torch.randn(M, d_out, **f32)
    td = TORCH_DTYPES[dtype]
    keep = [k.strip() for k in which.split(",")]
    return {k: out[k].to(td).contiguous() for k in keep}


def workload_inputs(name: str, seed: int = 0, device="cpu") -> dict:
    w = WORKLOADS[name]
    return make_inputs(w.M, w.d_in, w.d_out, w.r, w.dtype, seed, device)
