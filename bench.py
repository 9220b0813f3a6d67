"""Benchmark of the fused LoRA linear layer, forward + backward, on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

One step = one forward and one backward of the layer (every kernel of the
hot path) over one synthetic batch of the named workload, inputs resident in
HBM.  The metric is algorithmic TFLOP/s,
    4 M d_in d_out + 6 M r (d_in + d_out)   FLOPs per step (no dW: W frozen),
divided by the device time of the step (CUDA events on the launching stream;
L2 is flushed by a 256 MiB write before every step, outside the events).

Beside the contract keys the line carries the median step beside the mean;
on the default workload (the Llama-3-8B q_proj shape) the other two Llama-3-8B
shapes of the metric (gate/up, down_proj), each from its own timed region with
its own clocks and roofline; an end-to-end figure that also copies Y and dX
out ("e2e_all_outputs"); and, informationally, the step rated against
NVIDIA's datasheet BF16 figures and (plain layer, one GPU) the same step run
as separate PyTorch ops with autograd ("torch_unfused": as many steps, the
same flush, its own record of the SM clock, which decides the comparison on
power-capped shapes).

Rank 0 prints one JSON line.  Under torchrun each rank runs an independent
replica on its own GPU (the layer needs no exchange), the timed region is
bracketed by barriers, and the slowest rank's time is used.

--impl reference times the fp64 CPU oracle on the host cores instead, on a
bounded token sample of the same workload (the pages ship no runnable
reference implementation).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("fused LoRA fwd+bwd TFLOP/s on 1 GB300 (Llama-3-8B shapes); "
          "% of BF16 tensor peak")
DEFAULT_WORKLOAD = "llama3_8b_q_proj"
FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# NVIDIA's datasheet BF16 tensor figures, turned into dense (no 2:4 sparsity)
# figures per GPU, reported beside the measured peak.  The GB300 NVL72
# datasheet gives 360 PFLOPS FP16/BF16 with sparsity for its 72 GPUs
# (180 dense / 72 = 2.5 PF each); the HGX B300 datasheet 36 PFLOPS with
# sparsity for 8 GPUs (18 dense / 8 = 2.25 PF each).  This part is the
# NVL72's GB300, so its figure is the one the percentage uses.
DATASHEET_BF16_TFLOPS = {"gb300_nvl72_per_gpu": 2500.0, "hgx_b300_per_gpu": 2250.0}
DATASHEET_SOURCE = ("NVIDIA GB300 NVL72 datasheet: 360 PFLOPS FP16/BF16 tensor with sparsity "
                    "for 72 GPUs -> 2.5 PF dense per GPU; NVIDIA HGX B300 datasheet: 36 PFLOPS "
                    "with sparsity for 8 GPUs -> 2.25 PF dense per GPU")
# the Llama-3-8B shapes the metric is quoted on, besides the default q_proj one
OTHER_LLAMA_SHAPES = ("llama3_8b_gate_up", "llama3_8b_down_proj")


def step_flops(M, d_in, d_out, r):
    return 4 * M * d_in * d_out + 6 * M * r * (d_in + d_out)


def kernel_work(kind, M, d_in, d_out, r, w_bytes=None):
    """Algorithmic (flops, bytes) of one launch of each kernel kind (bf16).
    w_bytes: bytes of the frozen W as stored (default bf16; the 4-bit layer
    passes its codes plus scales)."""
    e = 2
    wb = e * d_out * d_in if w_bytes is None else w_bytes
    return {
        "prep": (0, e * 2 * d_out * r),
        "down_fwd": (2 * M * d_in * r, e * (M * d_in + r * d_in + M * r)),
        "main_fwd": (2 * M * d_out * (d_in + r),
                     e * (M * d_in + M * r + d_out * r + M * d_out) + wb),
        "down_bwd": (2 * M * d_out * r, e * (M * d_out + r * d_out + M * r)),
        "main_bwd": (2 * M * d_in * (d_out + r),
                     e * (M * d_out + M * r + r * d_in + M * d_in) + wb),
        "grad_a": (2 * M * d_in * r, e * (M * d_in + M * r + r * d_in)),
        "grad_b": (2 * M * d_out * r, e * (M * d_out + M * r + d_out * r)),
        # e4m3 quantisation of X's rows (bf16 in, bytes and scales out)
        "quant": (0, e * M * d_in + M * d_in + 4 * M),
        # s dY B and dY^T sH in one launch; dY counted once
        "down_bwd_grad_b": (4 * M * d_out * r,
                            e * (M * d_out + r * d_out + 2 * M * r + d_out * r)),
        # dA and dB in one launch after the dX GEMM (X and dY each read once)
        "grad_a_b": (2 * M * r * (d_in + d_out),
                     e * (M * d_in + M * d_out + 2 * M * r + r * d_in + d_out * r)),
    }[kind]


def kernel_work_swiglu(kind, M, d_in, d_ff, r):
    """Algorithmic (flops, bytes) of one launch of the gated pair's kernels."""
    e = 2
    return {
        "prep": (0, e * 4 * r * d_in),
        "down_fwd": (4 * M * d_in * r, e * (M * d_in + 2 * r * d_in + 2 * M * r)),
        "main_fwd": (4 * M * d_ff * (d_in + r),
                     e * (M * d_in + 2 * d_ff * d_in + 2 * M * r + 2 * d_ff * r + 3 * M * d_ff)),
        "swiglu_grad": (0, e * 5 * M * d_ff),
        "down_bwd_grad_b": (4 * M * d_ff * r, e * (M * d_ff + r * d_ff + 2 * M * r + d_ff * r)),
        "main_bwd": (4 * M * d_in * (d_ff + r),
                     e * (2 * M * d_ff + 2 * d_ff * d_in + 2 * M * r + 2 * r * d_in + M * d_in)),
        "grad_a": (4 * M * d_in * r, e * (M * d_in + 2 * M * r + 2 * r * d_in)),
    }[kind]


BOUND = {"prep": "hbm", "swiglu_grad": "hbm", "quant": "hbm", "down_fwd": "hbm", "down_bwd": "hbm", "grad_a": "hbm",
         "grad_b": "hbm", "down_bwd_grad_b": "hbm", "grad_a_b": "hbm", "main_fwd": "tensor",
         "main_bwd": "tensor"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained",
                                                     d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return dict(FALLBACK_PEAKS, source="fallback")


def _strip_comments(src: str) -> str:
    """C/C++ source without its // and /* */ comments (string literals kept)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == '"':  # string literal, escapes kept
            j = i + 1
            while j < n and src[j] != '"':
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "".join(out)


# the sources each kernel kind is compiled from (kinds not listed: all)
KERNEL_FILES = {"main_fwd": ("tc_main.cu", "ptx.cuh", "internal.h"),
                "main_bwd": ("tc_main.cu", "ptx.cuh", "internal.h")}


def kernel_source_hash(files=None):
    """Hash of kernel sources (`files` of csrc/, default all) with comments
    removed and whitespace runs collapsed: a committed ncu traffic figure
    stays valid across comment and layout edits, and across edits of other
    kernels' files, not across its own kernel's code."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "rank_linear_gb300", "csrc")
    for f in sorted(files if files is not None else os.listdir(csrc)):
        code = _strip_comments(open(os.path.join(csrc, f), encoding="utf-8").read())
        h.update(" ".join(code.split()).encode())
    return h.hexdigest()[:16]


def load_traffic(workload, kind):
    """DRAM bytes per launch from a committed ncu capture, if it matches the
    current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(p))
    except Exception:
        return None
    ent = d.get(workload, {}).get(kind)
    if not ent or ent.get("source_hash") != kernel_source_hash(KERNEL_FILES.get(kind)):
        return None
    return ent.get("bytes_per_launch")


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        inside = [p for t, p in self.samples if t0 <= t <= t1]
        window = "timed"
        if not inside:  # timed region shorter than the sampling period
            near = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            inside = [p for _, p in near]
            window = "nearest"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        mx = [num(p[2]) for p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for p in inside for n, v in zip(names, p[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "window": window}


# ---------------------------------------------------------------- dist
def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of x over all ranks (x itself when world == 1)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- CPU oracle
def layer_flops(w, tokens):
    """Algorithmic fwd+bwd FLOPs of the workload's layer on `tokens` tokens
    (the gated pair is two LoRA layers; its SiLU is not counted)."""
    return step_flops(tokens, w.d_in, w.d_out, w.r) * (2 if w.layer == "swiglu" else 1)


def oracle_run(t, alpha, layer="linear"):
    import oracle
    if layer == "fp8":
        from oracle import fp8
        fp8.forward(t["X"], t["W"], t["A"], t["B"], alpha)
        fp8.backward(t["dY"], t["X"], t["W"], t["A"], t["B"], alpha)
        return
    if layer == "q4":
        from oracle import q4
        codes, scales = q4.quantize_w(t["W"])
        q4.forward(t["X"], codes, scales, t["A"], t["B"], alpha)
        q4.backward(t["dY"], t["X"], codes, scales, t["A"], t["B"], alpha)
        return
    if "Wu" in t:
        from oracle import swiglu
        args = [t[k] for k in ("X", "W", "A", "B", "Wu", "Au", "Bu")]
        swiglu.forward(*args, alpha)
        swiglu.backward(t["dY"], *args, alpha)
        return
    oracle.forward(t["X"], t["W"], t["A"], t["B"], alpha)
    oracle.backward(t["dY"], t["X"], t["W"], t["A"], t["B"], alpha)


def oracle_inputs(w, tokens):
    from rank_linear_gb300.synth import make_inputs
    t = make_inputs(tokens, w.d_in, w.d_out, w.r, w.dtype, seed=0)
    if w.layer == "swiglu":
        u = make_inputs(tokens, w.d_in, w.d_out, w.r, w.dtype, seed=1000, which="W,A,B")
        t.update(Wu=u["W"], Au=u["A"], Bu=u["B"])
    import numpy as np
    return {k: np.ascontiguousarray(v.double().numpy()) for k, v in t.items()}


def oracle_sample_tokens(w, budget_s):
    """Largest token count (power of two, <= M) whose oracle fwd+bwd fits
    budget_s seconds, from one calibration run on 8 tokens."""
    t = oracle_inputs(w, 8)
    t0 = time.perf_counter()
    oracle_run(t, w.alpha, w.layer)
    per_token = (time.perf_counter() - t0) / 8
    tokens = 8
    while tokens * 2 <= w.M and tokens * 2 * per_token <= budget_s:
        tokens *= 2
    return tokens


def cpu_baseline(w, budget_s=15.0):
    import oracle
    tokens = oracle_sample_tokens(w, budget_s)
    t = oracle_inputs(w, tokens)
    t0 = time.perf_counter()
    oracle_run(t, w.alpha, w.layer)
    dt = time.perf_counter() - t0
    return {"value": layer_flops(w, tokens) / dt / 1e12, "unit": "TFLOP/s",
            "cores": oracle.threads(), "kind": "oracle",
            "sample": f"one fp64 fwd+bwd ({w.layer} layer) of {tokens} of the {w.M} tokens "
                      f"({w.d_in}x{w.d_out}, r={w.r}); {dt:.2f} s"}


def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    total_budget = 90.0
    per_step = max(0.05, total_budget / max(1, args.steps + args.warmup))
    tokens = oracle_sample_tokens(w, per_step)
    t = oracle_inputs(w, tokens)
    for _ in range(args.warmup):
        oracle_run(t, w.alpha, w.layer)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_run(t, w.alpha, w.layer)
        times.append(time.perf_counter() - t0)
    sec = sum(times)
    value = layer_flops(w, tokens) * args.steps / sec / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sec / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "layer": w.layer, "M": w.M, "d_in": w.d_in, "d_out": w.d_out, "r": w.r,
                   "alpha": w.alpha, "sample_tokens": tokens},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.threads(),
                         "kind": "oracle",
                         "sample": f"each step: fp64 fwd+bwd of {tokens} of the {w.M} tokens"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU
def run_torch_unfused(w, t, dev, stream, steps, flush, gpu_index):
    """The unfused layer as separate PyTorch ops with autograd (W frozen), in the
    workload's dtype on the same GPU: the baseline the fused kernels replace.
    Same step (forward + backward), same number of steps, same L2 flush, same
    FLOP count; its own clock record, since on power-capped shapes the SM
    clock decides the comparison."""
    import torch
    X = t["X"].detach().clone().requires_grad_(True)
    W = t["W"].detach()
    A = t["A"].detach().clone().requires_grad_(True)
    B = t["B"].detach().clone().requires_grad_(True)
    dY = t["dY"]
    s = w.alpha / w.r

    def step():
        X.grad = A.grad = B.grad = None
        Y = X @ W.t() + ((X @ A.t()) @ B.t()) * s
        Y.backward(dY)

    for _ in range(3):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    clocks = ClockSampler(gpu_index)
    clocks.start()
    time.sleep(0.3)
    wall0 = time.time()
    for e0, e1 in ev:
        flush.zero_()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    time.sleep(0.2)
    clocks.stop()
    sec = sum(e0.elapsed_time(e1) for e0, e1 in ev) / 1e3
    return {"value": step_flops(w.M, w.d_in, w.d_out, w.r) * steps / sec / 1e12,
            "unit": "TFLOP/s", "ms_per_step": 1e3 * sec / steps, "steps": steps,
            "clocks": clocks.summary(wall0, wall1),
            "what": "X W^T + s (X A^T) B^T as separate torch ops (cuBLAS) with autograd, "
                    "same dtype, same steps, L2 flushed before every step; informational"}


def measure(args, w, dev, stream, rank, world, local, steps):
    """Warm-up, K timed steps (clocks sampled meanwhile) and a second pass of
    K steps with events around every library launch, for one workload.
    Returns the step's figures, the per-kernel breakdown and the dominant
    kernel's roofline; "inputs" holds the drawn tensors."""
    import torch
    import rank_linear_gb300 as rl
    from rank_linear_gb300 import _lib
    from rank_linear_gb300.synth import make_inputs
    L = _lib.lib()
    swiglu = w.layer == "swiglu"
    fp8 = w.layer == "fp8"
    q4 = w.layer == "q4"
    M, d_in, d_out, r, alpha = w.M, w.d_in, w.d_out, w.r, w.alpha
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    t = make_inputs(M, d_in, d_out, r, w.dtype, seed=rank, device=dev)
    X, W, A, B, dY = t["X"], t["W"], t["A"], t["B"], t["dY"]
    Y = torch.empty(M, d_out, dtype=tdt, device=dev)
    dX = torch.empty(M, d_in, dtype=tdt, device=dev)
    dA = torch.empty(r, d_in, dtype=tdt, device=dev)
    dB = torch.empty(d_out, r, dtype=tdt, device=dev)
    saved = torch.empty(max(1, rl.saved_bytes(M, r, tdt)), dtype=torch.uint8, device=dev)
    ws = torch.empty(max(1, rl.workspace_bytes(M, d_in, d_out, r, tdt)), dtype=torch.uint8,
                     device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step():
        rl.forward(X, W, A, B, alpha, Y=Y, saved=saved, workspace=ws, stream=stream)
        rl.backward(dY, X, W, A, B, alpha, saved, dX=dX, dA=dA, dB=dB, workspace=ws,
                    stream=stream)

    if fp8:  # the frozen W quantised once (outside the timed steps), X and dY per call
        qw = rl.quantize_w_fp8(W)
        ws = torch.empty(max(1, rl.fp8_workspace_bytes(M, d_in, d_out, r)), dtype=torch.uint8,
                         device=dev)

        def step():
            rl.fp8_forward(X, qw, A, B, alpha, Y=Y, saved=saved, workspace=ws, stream=stream)
            rl.fp8_backward(dY, X, qw, A, B, alpha, saved, dX=dX, dA=dA, dB=dB, workspace=ws,
                            stream=stream)

    if q4:  # the frozen W quantised to 4 bits once (outside the timed steps)
        qw4 = rl.quantize_w_q4(W)

        def step():
            rl.q4_forward(X, qw4, A, B, alpha, Y=Y, saved=saved, workspace=ws, stream=stream)
            rl.q4_backward(dY, X, qw4, A, B, alpha, saved, dX=dX, dA=dA, dB=dB, workspace=ws,
                           stream=stream)

    if swiglu:  # the gate/up pair: H = silu(gate) * up, d_out = FFN width
        tu = make_inputs(M, d_in, d_out, r, w.dtype, seed=rank + 1000, device=dev,
                         which="W,A,B")
        Wu, Au, Bu = tu["W"], tu["A"], tu["B"]
        dAu = torch.empty(r, d_in, dtype=tdt, device=dev)
        dBu = torch.empty(d_out, r, dtype=tdt, device=dev)
        saved = torch.empty(max(1, rl.swiglu_saved_bytes(M, d_out, r)), dtype=torch.uint8,
                            device=dev)
        ws = torch.empty(max(1, rl.swiglu_workspace_bytes(M, d_in, d_out, r)),
                         dtype=torch.uint8, device=dev)

        def step():
            rl.swiglu_forward(X, W, A, B, Wu, Au, Bu, alpha, H=Y, saved=saved, workspace=ws,
                              stream=stream)
            rl.swiglu_backward(dY, X, W, A, B, Wu, Au, Bu, alpha, saved, dX=dX, dAg=dA,
                               dBg=dB, dAu=dAu, dBu=dBu, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    rl.device_status()

    n0 = rl.launch_count()
    step()
    torch.cuda.synchronize()
    launches_per_step = rl.launch_count() - n0
    s_ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    e_ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]

    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)

    # Timed region: K steps, nothing between the library's launches (events
    # between them would break the programmatic-dependent-launch overlap).
    barrier(world)
    torch.cuda.synchronize()
    c0 = rl.launch_count()
    wall0 = time.time()
    for i in range(steps):
        flush.zero_()
        s_ev[i].record(stream)
        step()
        e_ev[i].record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    launched = rl.launch_count() - c0
    barrier(world)
    rl.device_status()

    # Second pass of K steps with an event pair around every launch of the
    # library (per-kernel durations for the breakdown and the roofline).
    n_pairs = launches_per_step * steps
    kev, karr, kinds = rl.timing_events(n_pairs, stream)
    torch.cuda.synchronize()
    _lib.check(L.lora_set_timing_events(karr, kinds, n_pairs), "timing hook")
    for i in range(steps):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    used = L.lora_timing_used()
    L.lora_set_timing_events(None, None, 0)
    rl.device_status()
    if clocks:
        time.sleep(0.2)
        clocks.stop()

    step_ms = [a.elapsed_time(b) for a, b in zip(s_ev, e_ev)]
    sec = max_over_ranks(sum(step_ms) / 1e3, world, dev)
    med_s = max_over_ranks(statistics.median(step_ms) / 1e3, world, dev)
    flops = step_flops(M, d_in, d_out, r) * (2 if swiglu else 1)

    per_kind = {}
    for j in range(used):
        k = _lib.KERNEL_KINDS[kinds[j]]
        per_kind.setdefault(k, []).append(kev[2 * j].elapsed_time(kev[2 * j + 1]))
    total_k = sum(sum(v) for v in per_kind.values())
    kern = {k: {"launches": len(v), "avg_us": 1e3 * sum(v) / len(v),
                "share": sum(v) / total_k} for k, v in per_kind.items()}
    dom = max(per_kind, key=lambda k: sum(per_kind[k]))

    peaks = load_peaks()
    if swiglu:
        fl, by = kernel_work_swiglu(dom, M, d_in, d_out, r)
    else:  # 4-bit W: codes (half a byte each) and a bf16 scale per 64 weights
        fl, by = kernel_work(dom, M, d_in, d_out, r,
                             w_bytes=d_out * d_in // 2 + d_out * d_in // 32 if q4 else None)
    avg_s = sum(per_kind[dom]) / len(per_kind[dom]) / 1e3
    clk = clocks.summary(wall0, wall1) if clocks else None
    # A tensor-bound kernel is rated against the burst figure unless the GPU
    # sat at its power cap during the timed steps: then the kernel ran as
    # part of sustained work, and the sustained figure is its peak.
    capped = bool(clk) and "sw_power_cap" in clk.get("reasons", [])
    bf16_peak = peaks["bf16_tflops_sustained"] if capped else peaks["bf16_tflops"]
    kind = "sustained (sw_power_cap active)" if capped else "burst"
    peak_note = f" ({kind})"
    if BOUND[dom] == "tensor" and fp8:  # e4m3 products: 2 x the bf16 rate (nominal ratio)
        ach, peak, unit = fl / avg_s / 1e12, 2 * bf16_peak, "TFLOP/s"
        peak_note = f" bf16 {kind} x 2 (nominal e4m3 / bf16 ratio)"
    elif BOUND[dom] == "tensor":
        ach, peak, unit = fl / avg_s / 1e12, bf16_peak, "TFLOP/s"
    else:
        ach, peak, unit = by / avg_s / 1e9, peaks["hbm_gbs"], "GB/s"
    roofline = {"kernel": dom, "bound": BOUND[dom], "achieved": ach, "peak": peak,
                "unit": unit, "frac": ach / peak, "peak_source": peaks["source"] + peak_note,
                "traffic": load_traffic(w.name, dom)}
    return {"value": world * flops * steps / sec / 1e12,
            "value_median": world * flops / med_s / 1e12,
            "ms_per_step": 1e3 * sec / steps, "ms_per_step_median": 1e3 * med_s,
            "launched": launched, "kernels": kern, "roofline": roofline, "clocks": clk,
            "peaks": peaks, "inputs": t, "dtype": tdt, "flush": flush}


def run_ours(args, w):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from rank_linear_gb300 import _lib
    _lib.lib()

    swiglu = w.layer == "swiglu"
    fp8 = w.layer == "fp8"
    q4 = w.layer == "q4"
    # CPU baseline first (rank 0, N = 1 only), before the GPU is busy
    cpu = cpu_baseline(w) if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None
    stream = torch.cuda.current_stream()

    res = measure(args, w, dev, stream, rank, world, local, args.steps)
    t, tdt = res["inputs"], res["dtype"]

    e2e = e2e_all = None
    if not (args.no_e2e or swiglu or fp8 or q4):
        e2e = run_e2e(args, w, t, tdt, dev, stream, world)
        e2e_all = run_e2e(args, w, t, tdt, dev, stream, world, all_outputs=True)
    unfused = None
    if rank == 0 and world == 1 and not (swiglu or fp8 or q4 or args.no_unfused):
        unfused = run_torch_unfused(w, t, dev, stream, args.steps, res["flush"], local)

    # The other Llama-3-8B shapes of the metric, each in its own timed region
    others = None
    if w.name == DEFAULT_WORKLOAD and not args.no_other_shapes:
        from rank_linear_gb300.synth import WORKLOADS
        del t, res["inputs"], res["flush"]
        torch.cuda.empty_cache()
        others = {}
        for name in OTHER_LLAMA_SHAPES:
            wo = WORKLOADS[name]
            ro = measure(args, wo, dev, stream, rank, world, local, args.steps)
            others[name] = {
                "value": ro["value"], "unit": "TFLOP/s", "ms_per_step": ro["ms_per_step"],
                "value_median": ro["value_median"],
                "ms_per_step_median": ro["ms_per_step_median"],
                "pct_of_bf16_peak": 100.0 * ro["value"] / world / ro["peaks"]["bf16_tflops"],
                "config": {"M": wo.M, "d_in": wo.d_in, "d_out": wo.d_out, "r": wo.r,
                           "alpha": wo.alpha},
                "roofline": ro["roofline"], "kernels": ro["kernels"], "clocks": ro["clocks"],
                "gpu_launches": ro["launched"], "steps": args.steps}
            del ro
            torch.cuda.empty_cache()

    if rank == 0:
        value = res["value"]
        peaks = res["peaks"]
        ds = DATASHEET_BF16_TFLOPS["gb300_nvl72_per_gpu"]
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": res["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": ("e4m3 W product, bf16 elsewhere" if fp8 else
                      "4-bit W codes expanded to bf16, bf16 elsewhere" if q4 else w.dtype),
            "data": "synthetic",
            "config": {"workload": w.name, "layer": w.layer, "M": w.M, "d_in": w.d_in,
                       "d_out": w.d_out, "r": w.r,
                       "alpha": w.alpha, "l2": "flushed before every step (256 MiB write)",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "ms_per_step_median": res["ms_per_step_median"],
            "value_median": res["value_median"],
            "pct_of_bf16_peak": 100.0 * value / world / peaks["bf16_tflops"],
            "pct_of_datasheet_bf16_peak": 100.0 * value / world / ds,
            "pct_of_datasheet_bf16_peak_hgx_b300": (
                100.0 * value / world / DATASHEET_BF16_TFLOPS["hgx_b300_per_gpu"]),
            "datasheet_bf16_tflops": ds, "datasheet_source": DATASHEET_SOURCE,
            "roofline": res["roofline"], "kernels": res["kernels"],
            "kernel_timing": "second pass of the same K steps with CUDA events around "
                             "every library launch (on the launching stream)",
            "other_llama3_8b_shapes": others,
            "cpu_baseline": cpu, "e2e": e2e, "e2e_all_outputs": e2e_all,
            "torch_unfused": unfused,
            "gpu_launches": res["launched"],
            "clocks": res["clocks"],
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(args, w, t, tdt, dev, stream, world, all_outputs=False):
    """Same metric through the public API with pinned host buffers.  Every
    step copies its inputs -- the batch's activations X and the upstream
    gradient dY -- in, and its result -- the gradients dA and dB the
    optimizer takes -- out, inside the timed region.  The frozen W and the
    adapters A, B are model state: uploaded once, before, and kept on the
    GPU; Y and dX stay on the GPU for the neighbouring layers, unless
    all_outputs, when they are copied out every step as well.  Steps are
    pipelined the way a training loop would be: two device buffer sets,
    uploads on one stream, the layer on the launching stream, downloads on a
    third, so that step i+1's upload and step i-1's download overlap step
    i's kernels."""
    import torch
    import rank_linear_gb300 as rl
    M, d_in, d_out, r, alpha = w.M, w.d_in, w.d_out, w.r, w.alpha
    per_step = ("X", "dY")
    h_in = {k: t[k].cpu().pin_memory() for k in per_step}
    state = {k: t[k] for k in ("W", "A", "B")}  # model state, resident on the GPU
    outs = {"dA": (r, d_in), "dB": (d_out, r)}
    if all_outputs:
        outs.update(Y=(M, d_out), dX=(M, d_in))
    nbuf = 2
    d_in_t = [{k: torch.empty_like(t[k]) for k in per_step} for _ in range(nbuf)]
    d_out_t = [{k: torch.empty(s, dtype=tdt, device=dev) for k, s in outs.items()}
               for _ in range(nbuf)]
    # Y and dX: among the outputs copied out, or device-only activations
    d_act = [{k: (d_out_t[b][k] if k in outs else
                  torch.empty(shape, dtype=tdt, device=dev))
              for k, shape in (("Y", (M, d_out)), ("dX", (M, d_in)))} for b in range(nbuf)]
    h_out = [{k: torch.empty(s, dtype=tdt).pin_memory() for k, s in outs.items()}
             for _ in range(nbuf)]
    saved = torch.empty(max(1, rl.saved_bytes(M, r, tdt)), dtype=torch.uint8, device=dev)
    ws = torch.empty(max(1, rl.workspace_bytes(M, d_in, d_out, r, tdt)), dtype=torch.uint8,
                     device=dev)
    s_up = torch.cuda.Stream(device=dev)
    s_down = torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()
    up_done = [ev() for _ in range(nbuf)]
    comp_done = [ev() for _ in range(nbuf)]
    down_done = [ev() for _ in range(nbuf)]
    for b in range(nbuf):  # every buffer starts free
        comp_done[b].record(stream)
        down_done[b].record(stream)

    def step(i):
        b = i % nbuf
        din, dout, hout = d_in_t[b], d_out_t[b], h_out[b]
        s_up.wait_event(comp_done[b])  # step i-2 has finished reading din
        with torch.cuda.stream(s_up):
            for k in h_in:
                din[k].copy_(h_in[k], non_blocking=True)
        up_done[b].record(s_up)
        stream.wait_event(up_done[b])
        stream.wait_event(down_done[b])  # step i-2's results have left dout
        W, A, B = state["W"], state["A"], state["B"]
        rl.forward(din["X"], W, A, B, alpha, Y=d_act[b]["Y"], saved=saved, workspace=ws,
                   stream=stream)
        rl.backward(din["dY"], din["X"], W, A, B, alpha, saved, dX=d_act[b]["dX"],
                    dA=dout["dA"], dB=dout["dB"], workspace=ws, stream=stream)
        comp_done[b].record(stream)
        s_down.wait_event(comp_done[b])
        with torch.cuda.stream(s_down):
            for k in hout:
                hout[k].copy_(dout[k], non_blocking=True)
        down_done[b].record(s_down)

    for i in range(max(nbuf, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    n = max(3, min(args.steps, 50))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(stream)  # before the first upload; everything after depends on it
    s_up.wait_event(e0)
    s_down.wait_event(e0)
    for i in range(n):
        step(i)
    stream.wait_stream(s_down)  # e1 follows the last download
    e1.record(stream)
    torch.cuda.synchronize()
    sec = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev)
    bi = sum(v.numel() * v.element_size() for v in h_in.values())
    bo = sum(v.numel() * v.element_size() for v in h_out[0].values())
    return {"value": world * step_flops(M, d_in, d_out, r) * n / sec / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": n,
            "inputs": ("every step: X and dY copied in, Y, dX, dA and dB copied out "
                       "(pinned host); " if all_outputs else
                       "every step: X and dY copied in, dA and dB copied out (pinned host); ")
                      + "W, A, B resident (uploaded once, before); "
                      + ("" if all_outputs else "Y and dX stay on the GPU; ")
                      + "uploads, kernels and downloads on three streams with two device "
                        "buffer sets (step i+1's upload and step i-1's download overlap step "
                        "i's kernels)"}


def main(argv=None):
    from rank_linear_gb300.synth import WORKLOADS
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-unfused", action="store_true",
                    help="skip the informational unfused PyTorch timing")
    ap.add_argument("--no-other-shapes", action="store_true",
                    help="default workload only: skip timing the gate/up and down_proj shapes")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)  # at least three untimed warm-up steps
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
