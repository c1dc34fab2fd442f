"""bench.py's reference arm (the CPU oracle on the host's cores) keeps the JSON-line
contract and runs on rank 0 only. It needs no GPU, so it is checked here on the CPU
with the smallest workload. It is a pure host process: it never imports the package's
binding, never maps libsmoe.so and never creates a CUDA context."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ARGS = ["--impl", "reference", "--workload", "tiny_fp32", "--steps", "2", "--warmup", "3",
        "--cpu-seconds", "1"]


def _run(env_extra):
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    env.update(env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *ARGS], cwd=ROOT,
                          env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_contract_line():
    r = _run({})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    out = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in out, key
    assert out["impl"] == "reference"
    assert out["steps"] == 2 and out["warmup"] == 3 and out["n_gpus"] == 1
    assert out["unit"] == "tokens/s" and out["higher_is_better"] is True
    assert out["value"] > 0
    assert out["config"]["workload"].startswith("tiny_fp32: T=64")
    cb = out["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == out["value"] and cb["cores"] >= 1
    assert out["e2e"] == {"value": out["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    r = _run({"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{")]


def test_reference_arm_never_touches_the_library():
    code = ("import sys, runpy\n"
            f"sys.argv = ['bench.py'] + {ARGS!r}\n"
            "runpy.run_path('bench.py', run_name='__main__')\n"
            "mods = [m for m in sys.modules if m.endswith('binding')]\n"
            "assert not mods, mods\n"
            "maps = open('/proc/self/maps').read()\n"
            "assert 'libsmoe' not in maps\n"
            "import torch\n"
            "assert not torch.cuda.is_initialized()\n"
            "print('clean')\n")
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "clean" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]


def test_cpu_oracle_rate_sample_reaches_most_of_the_target(monkeypatch):
    """The CPU baseline's sample grows until one oracle call takes at least 0.7 of the
    target seconds (or the whole batch), also when the oracle's cost per token falls as
    the sample grows (as numpy's matrix products do) and when its first call carries a
    one-time cost: a fake clock and a fake oracle stand in for both."""
    import types

    import numpy as np

    sys.path.insert(0, ROOT)
    import bench
    import oracle as O
    from routing_token_shuffle_gb300 import synth
    clock = [0.0]
    calls = []
    cost = {}

    def fake_layer_forward(x, *args, **kw):
        n = len(x)
        calls.append(n)
        clock[0] += cost["a"] + cost["c"] * n ** cost["p"] + (cost["first"] if len(calls) == 1 else 0)

    monkeypatch.setattr(bench, "time", types.SimpleNamespace(perf_counter=lambda: clock[0]))
    monkeypatch.setattr(O, "layer_forward", fake_layer_forward)
    cfg = synth.CONFIGS["dsv2_prefill"]
    z = np.zeros((cfg.T, 1), np.float32)
    h = bench.HostLayer(cfg, z, np.zeros(cfg.T, np.int32), None, None, None, None, None, None)
    for a_, c_, p_, first in ((0.3, 0.01, 0.8, 0.0), (1.0, 0.05, 0.6, 3.0), (0.2, 0.02, 0.7, 6.0),
                              (2.5, 0.002, 1.0, 0.0), (0.5, 0.08, 0.5, 1.0)):
        cost.update(a=a_, c=c_, p=p_, first=first)
        for target in (4.0, 10.0, 15.0):
            calls.clear()
            rate, n, secs, cores = bench.cpu_oracle_rate(h, target)
            assert (secs >= 0.7 * target or n == cfg.T) and len(calls) <= 9, (cost, target, n, secs, calls)
            assert rate == n / secs and cores >= 1
