"""bench.py end to end on a small workload: one JSON line that keeps the contract (the
keys, their types and the relations between them), from the CUDA library."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout=600):
    env = dict(os.environ, PYTHONUNBUFFERED="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       env=env, capture_output=True, text=True, timeout=timeout)
    assert p.returncode == 0, p.stderr[-3000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout[-2000:]
    return json.loads(lines[0])


@pytest.mark.gpu
@pytest.mark.parametrize("workload,tokens", [("tiny_fp32", None), ("qwen3_foe", 2048)])
def test_bench_line_keeps_the_contract(workload, tokens):
    args = ["--workload", workload, "--steps", "3", "--warmup", "3", "--cpu-seconds", "1",
            "--no-placement"]
    if tokens:
        args += ["--tokens", str(tokens)]
    j = _run(args)
    assert j["metric"] and j["unit"] == "tokens/s" and j["higher_is_better"] is True
    assert j["n_gpus"] == 1 and j["steps"] == 3 and j["warmup"] == 3
    assert j["value"] > 0 and j["ms_per_step"] > 0
    T = tokens or {"tiny_fp32": 64, "qwen3_foe": 16384}[workload]
    # value = tokens of the timed steps / their time
    assert abs(j["value"] - T / (j["ms_per_step"] / 1e3)) <= 1e-3 * j["value"]
    assert j["scaling"] == "weak" and j["data"].startswith("synthetic")
    assert j["dtype"] == ("f32" if workload == "tiny_fp32" else "bf16")
    assert j["config"]["workload"].startswith(f"{workload}: T={T},")
    e = j["e2e"]
    assert e["value"] > 0 and e["unit"] == "tokens/s"
    b = 4 if workload == "tiny_fp32" else 2
    d = {"tiny_fp32": 128, "qwen3_foe": 2048}[workload]
    assert e["d2h_bytes_per_step"] == T * d * b                  # the layer output y
    assert e["h2d_bytes_per_step"] >= T * d * b                  # x (and the token ids)
    assert isinstance(j["gpu_launches"], int) and j["gpu_launches"] > 0
    r = j["roofline"]
    assert r["bound"] in ("hbm", "tensor") and r["unit"] in ("GB/s", "TFLOP/s")
    assert r["achieved"] > 0 and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    assert "traffic" in r
    c = j["cpu_baseline"]
    assert c["kind"] == "oracle" and c["value"] > 0 and c["cores"] >= 1 and c["sample"]
    k = j["clocks"]
    assert k["sm_max_mhz"] > 0 and isinstance(k["reasons"], list)
    assert set(j["stages"]) >= {"route", "predict_shuffle", "lar", "dispatch", "expert_ffn",
                                "combine"}
