"""The benchmark's host-side contract on CPU: the reference arm's JSON line and the algorithmic
work it credits (the roofline's numerator)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "impl",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1
    assert d["unit"] == "tokens/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"].startswith("tiny:")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_layer_work_counts_the_defined_flops_and_bytes():
    sys.path.insert(0, ROOT)
    import bench
    from moe_inputs import CONFIGS
    cfg = CONFIGS["v3_prefill"]
    T, H, N, I, S, K = cfg.T, cfg.hidden, cfg.n_routed, cfg.inter, cfg.n_shared, cfg.top_k
    counts = [0] * N
    for e in range(0, N, 2):           # 128 touched experts
        counts[e] = 2 * T * K // N
    kept = T * K
    w = bench.layer_work(cfg, counts, kept)
    # gate 2·T·H·N, SwiGLU 6·H·I per routed row and per token·shared expert
    assert w["flops"] == 2 * T * H * N + 6 * H * I * (kept + T * S)
    assert w["up_flops"] + w["down_flops"] == 6 * H * I * (kept + T * S)
    # bytes: x in + out, W_g, W13 + W2 of touched + shared experts, logits, (idx, w)
    assert w["touched"] == 128
    assert w["weight_bytes"] == (128 + S) * 3 * H * I * 2
    assert w["bytes"] == 2 * T * H * 2 + N * H * 2 + w["weight_bytes"] + T * N * 4 + T * K * 8
    assert bench.job_tokens_per_s(10.0, 4, 512, 5) == pytest.approx(4 * 512 * 5 / 0.010)


def test_traffic_capture_keyed_by_code_not_comments(tmp_path):
    """A committed DRAM-traffic capture stays valid across comment edits of the kernel sources
    (// and /* */) and is dropped by any change to the code of any of them."""
    sys.path.insert(0, ROOT)
    import bench
    src, hdr = tmp_path / "k.cu", tmp_path / "h.cuh"
    src.write_text("// header\nint f(int a) {  // add one\n  return a + 1;\n}\n")
    hdr.write_text("/* helper */\nint g(int b) { return b * 2; }\n")
    d0 = bench.code_digest(str(src), str(hdr))
    src.write_text("// another header\n\nint f(int a) {\n  return a + 1;  // still one\n}\n")
    hdr.write_text("/* a helper,\n   over two lines */\nint g(int b) { return b * 2; }\n")
    assert bench.code_digest(str(src), str(hdr)) == d0
    hdr.write_text("int g(int b) { return /* doubled */ b * 3; }\n")
    assert bench.code_digest(str(src), str(hdr)) != d0
    hdr.write_text("/* helper */\nint g(int b) { return b * 2; }\n")
    src.write_text("int f(int a) {\n  return a + 2;\n}\n")
    assert bench.code_digest(str(src), str(hdr)) != d0
    # the GEMM digest covers the kernel file, its PTX helpers and the shared argument layout
    assert set(bench.GEMM_SOURCES) == {"gemm_tc.cu", "common.cuh", "internal.h"}
    assert len(bench.gemm_digest()) == 64
