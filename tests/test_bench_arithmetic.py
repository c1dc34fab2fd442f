"""bench.py's roofline arithmetic: the algorithmic bytes and flops per stage equal the
figures worked out by hand from each workload's shapes (each input read once, each output
written once; b = 2 bytes for bf16). The reported fractions divide these by measured
durations, so they are pinned here on the CPU."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from routing_token_shuffle_gb300 import synth  # noqa: E402

MB, GB, TF = 1e6, 1e9, 1e12


def rel(a, b):
    return abs(a - b) / b


@pytest.mark.parametrize("name,flops", [
    ("mixtral", 2.886 * TF),        # 6 d F T K = 6 * 4096 * 14336 * 8192
    ("dsv2_prefill", 3.092 * TF),   # 6 d F (T K + S T) = 6 * 5120 * 1536 * 65536
    ("dsv2_decode", 0.02416 * TF),  # 6 * 5120 * 1536 * (64 * 6 + 2 * 64)
    ("qwen3_foe", 1.237 * TF),      # 6 * 2048 * 768 * 131072
])
def test_ffn_flops(name, flops):
    assert rel(bench.ffn_flops(synth.CONFIGS[name]), flops) < 1e-3


def test_ffn_bytes_are_the_touched_weights_plus_activations():
    mix = synth.CONFIGS["mixtral"]
    # 8 experts x 3 matrices x 14336 x 4096 x 2 B = 2.818 GB of weights
    w = bench.ffn_bytes(mix, 8) - bench.ffn_bytes(mix, 0)
    assert rel(w, 2.818 * GB) < 1e-3
    dsv2 = synth.CONFIGS["dsv2_prefill"]
    # 160 routed + 2 shared experts x 3 x 1536 x 5120 x 2 B = 7.644 GB
    assert rel(bench.ffn_bytes(dsv2, 160) - bench.ffn_bytes(dsv2, 0) + 2 * 3 * 1536 * 5120 * 2,
               7.644 * GB) < 1e-3
    # activations: X_disp read, H written and read, Y_disp written: rows (d + 2F + d) b
    rows = mix.T * mix.K
    assert bench.ffn_bytes(mix, 0) == rows * (4096 + 2 * 14336 + 4096) * 2


def test_stage_bytes_mixtral():
    cfg = synth.CONFIGS["mixtral"]
    s = bench.stage_bytes(cfg)
    assert rel(s["route"], 33.79 * MB) < 1e-3      # x + W_g + fp32 logits + idx/w
    # the shuffle stage computes the permutation alone: ids, C_p rows, pred/perm/offsets
    assert s["predict_shuffle"] == 4096 * (4 + 8 * 4 + 3 * 4)
    # the dispatch stage sorts, then reads x once and writes x_shuf and the T K rows
    assert rel(s["dispatch"], 134.3 * MB) < 1e-3
    assert rel(s["combine"], 100.7 * MB) < 1e-3    # T K rows + y written
    assert s["lar"] == 4096 * 2 * 4 + 4096 * 4
    # where the FFN copies the rows itself, the shuffle stage moves x and x_shuf
    assert rel(bench.stage_bytes(cfg, rows_in_ffn=True)["predict_shuffle"], 67.30 * MB) < 1e-3


def test_stage_bytes_dsv2_and_the_in_gemm_copy():
    cfg = synth.CONFIGS["dsv2_prefill"]
    s = bench.stage_bytes(cfg)
    # x read once, x_shuf written (2 T d b) and the T K dispatched rows written
    assert rel(s["dispatch"], 671.7 * MB) < 1e-3
    assert rel(s["combine"], 755.4 * MB) < 1e-3    # (T K + S T + T) d b + 8 T K
    # with the row copy inside the up GEMM the dispatch only moves indices
    q = synth.CONFIGS["qwen3_foe"]
    assert bench.stage_bytes(q, rows_in_ffn=True)["dispatch"] == q.T * q.K * 16


def test_whole_job_rate_counts_every_rank():
    assert bench.whole_job_rate(4096 * 10, 1, 0.02) == pytest.approx(2048000.0)
    assert bench.whole_job_rate(4096 * 10, 4, 0.02) == pytest.approx(4 * 2048000.0)
