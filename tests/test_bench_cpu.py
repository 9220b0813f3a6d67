"""bench.py's contract pieces that need no GPU: the reference arm's JSON line,
the algorithmic FLOP / byte counts behind the roofline, and the rule that a
committed ncu traffic figure is used only for the kernel sources it was taken
from."""
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

REQUIRED = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
            "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"}


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
         "--workload", "tiny_fp32", "--steps", "2", "--warmup", "1"],
        capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert REQUIRED <= set(d)
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] >= 3
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny_fp32" and d["config"]["layer"] == "linear"
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_step_flops_closed_form():
    # 4 M d_in d_out (two W products) + 6 M r (d_in + d_out) (six skinny products)
    M, d_in, d_out, r = 8192, 4096, 14336, 16
    assert bench.step_flops(M, d_in, d_out, r) == 4 * M * d_in * d_out + 6 * M * r * (d_in + d_out)


def test_kernel_work_counts_w_as_stored():
    M = d_in = d_out = 4096
    r = 16
    fl16, by16 = bench.kernel_work("main_fwd", M, d_in, d_out, r)
    q4_bytes = d_out * d_in // 2 + d_out * d_in // 32  # codes + one bf16 scale per 64
    fl4, by4 = bench.kernel_work("main_fwd", M, d_in, d_out, r, w_bytes=q4_bytes)
    assert fl16 == fl4 == 2 * M * d_out * (d_in + r)
    assert by16 - by4 == 2 * d_out * d_in - q4_bytes
    # the forward GEMM reads X, W, sH, B once and writes Y once
    assert by16 == 2 * (M * d_in + d_out * d_in + M * r + d_out * r + M * d_out)
    # the gated pair is two layers
    from rank_linear_gb300.synth import WORKLOADS
    w = WORKLOADS["llama3_8b_swiglu_gate_up"]
    assert bench.layer_flops(w, 100) == 2 * bench.step_flops(100, w.d_in, w.d_out, w.r)


def test_traffic_only_for_matching_sources(tmp_path, monkeypatch):
    h = bench.kernel_source_hash()
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps({
        "wl_a": {"main_fwd": {"bytes_per_launch": 123, "source_hash": h}},
        "wl_b": {"main_fwd": {"bytes_per_launch": 456, "source_hash": "0" * 16}}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # kernel_source_hash reads the real sources; only traffic.json moves
    monkeypatch.setattr(bench, "kernel_source_hash", lambda files=None: h)
    assert bench.load_traffic("wl_a", "main_fwd") == 123
    assert bench.load_traffic("wl_b", "main_fwd") is None
    assert bench.load_traffic("wl_a", "main_bwd") is None



def test_kernel_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    csrc = tmp_path / "rank_linear_gb300" / "csrc"
    csrc.mkdir(parents=True)
    f = csrc / "k.cu"
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    f.write_text('// header\nint a = 1; /* note */\nconst char *s = "x // y";\n')
    h0 = bench.kernel_source_hash()
    f.write_text('// a longer header\n// over two lines\nint a = 1;\n\nconst char *s = "x // y";\n')
    assert bench.kernel_source_hash() == h0          # comments and layout only
    f.write_text('int a = 2;\nconst char *s = "x // y";\n')
    assert bench.kernel_source_hash() != h0          # code
    f.write_text('int a = 1;\nconst char *s = "x / y";\n')
    assert bench.kernel_source_hash() != h0          # a string literal is code


def test_reference_arm_under_torchrun_prints_once():
    """Launched as the driver launches N > 1 (torchrun, one process per rank):
    rank 0 alone times the oracle and prints the line; the other rank exits 0
    without work."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    out = subprocess.run(
        [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
         "--master-addr", "127.0.0.1", "--master-port", str(port),
         os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
         "--workload", "tiny_fp32", "--steps", "2", "--warmup", "1"],
        capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
