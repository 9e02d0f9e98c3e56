"""Host-side logic of bench.py (no GPU): the algorithmic work it divides by, the ncu traffic
lookup guarded by the kernel source hash, and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import numpy as np

import bench
import moe_inputs as mi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NV = 9 / 16  # NVFP4 bytes per element: half a code byte + one E4M3 scale per 16 values


def test_kernel_work_hand_example():
    # 3 tokens, top-2 over 4 experts, local experts 1..2 (two local): slots routed to
    # experts 1 and 2 count, the others are masked
    cfg = mi.MoEConfig("hand", M=3, H=256, I=128, E=4, top_k=2, local_offset=1, num_local=2)
    ids = np.array([[1, 0], [2, 1], [3, 0]], dtype=np.int32)
    w, step, R, active = bench.kernel_work(cfg, ids)
    assert R == 3 and active == 2
    H, I, N1, M, k = 256, 128, 256, 3, 2  # SwiGLU: N1 = 2 I
    # the scope table's count: active experts' weights and alphas (no intermediates)
    assert w["gemm1"]["bytes"] == active * N1 * H * NV + 2 * 4
    assert w["gemm2"]["bytes"] == active * H * I * NV + 2 * 4
    # this implementation's own round trips on top: permuted rows, intermediate, expert rows
    assert w["gemm1"]["bytes_incl_intermediates"] == active * N1 * H * NV + R * H * NV + R * I * NV + 2 * 4
    assert w["gemm2"]["bytes_incl_intermediates"] == active * H * I * NV + R * I * NV + R * H * 2 + 2 * 4
    assert w["gemm1"]["flops"] == 2.0 * R * H * N1
    assert w["gemm2"]["flops"] == 2.0 * R * I * H
    # the kernels' algorithmic bytes add up to the whole step's: weights, alphas, BF16 in and
    # out, routing ids and weights
    assert sum(v["bytes"] for v in w.values()) == step["bytes"]
    assert step["bytes"] == active * (N1 * H + H * I) * NV + 8 * 2 + 2 * M * H * 2 + M * k * 8
    assert step["flops"] == w["gemm1"]["flops"] + w["gemm2"]["flops"]


def test_roofline_bound_and_fraction():
    peaks = {"hbm_gbs": 8000.0, "bf16_tflops": 2000.0, "source": "test"}
    # 8 GB in 2 ms at 8 TB/s peak: HBM-bound, achieved 4 TB/s = half the peak
    r = bench.roofline(8e9, 1e12, 2e-3, peaks)
    assert r["bound"] == "hbm" and abs(r["frac"] - 0.5) < 1e-12 and r["unit"] == "GB/s"
    # 1 GB and 12 PFLOP in 2 ms: tensor-bound at 2000 x 6 = 12 PF/s, so frac = (1 ms) / (2 ms)
    r = bench.roofline(1e9, 12e12, 2e-3, peaks)
    assert r["bound"] == "tensor" and abs(r["frac"] - 0.5) < 1e-12 and r["unit"] == "TFLOP/s"


def test_warmup_below_three_is_rejected():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                          "--steps", "1", "--warmup", "2"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode != 0 and "--warmup" in out.stderr


def test_traffic_lookup_follows_the_kernel_hash(monkeypatch):
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    with open(path) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert rows, "no traffic rows"
    h = bench.kernel_source_hash()
    for workload, kernel, nbytes, _, row_hash in rows:
        name = {"gemm_chained": "gemm1+gemm2 (chained)", "gemm_decode": "gemm1+gemm2 (decode)"}.get(kernel, kernel)
        got = bench.traffic_from_profiles(name, workload)
        assert got == (int(nbytes) if row_hash == h else None)
    # a changed kernel source makes every committed figure stale
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert all(bench.traffic_from_profiles(k, w) is None for w, k, *_ in rows)


def test_workload_names_state_the_sizes():
    for name, cfg in mi.CONFIGS.items():
        s = bench.workload_name(cfg)
        assert s.startswith(name) and f"H={cfg.H}" in s and f"top_k={cfg.top_k}" in s


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                          "--steps", "2", "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
