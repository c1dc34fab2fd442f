"""The C-ABI library loads without a GPU, exports every declared entry point and
rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

from routing_token_shuffle_gb300 import binding as B
from routing_token_shuffle_gb300 import build as build_mod
from routing_token_shuffle_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.lib()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names.update(re.findall(r"SMOE_API\s+[\w\s\*]+?\b(smoe_\w+)\s*\(", src))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(B.SIGNATURES), "binding is missing a declared entry point"


def test_no_stray_exports(lib):
    """Only smoe_* symbols are visible (the static CUDA runtime stays local)."""
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True,
                         text=True).stdout
    syms = [l.split()[-1] for l in out.splitlines() if l.strip() and " T " in l]
    assert syms and all(s.startswith("smoe_") for s in syms), syms


def test_status_strings(lib):
    for code in range(-8, 1):
        assert lib.smoe_status_string(code)
    assert lib.smoe_status_string(123) == b"unknown status"


@pytest.mark.parametrize("name", list(synth.CONFIGS))
def test_workspace_size_valid_configs(lib, name):
    d = B.desc_from_config(synth.CONFIGS[name])
    assert B.workspace_size(d) > 0


def base_desc(**kw):
    d = dict(T=64, d=128, E=8, K=2, H=1, F=256, n_shared=0, P=2, vocab=512, dtype="bf16")
    d.update(kw)
    return B.make_desc(**d)


@pytest.mark.parametrize("kw,code", [
    (dict(K=9), -2), (dict(H=3), -2), (dict(K=3, H=2), -2), (dict(E=1024), -2),
    (dict(K=33, E=64), -2), (dict(P=33), -2), (dict(d=100), -2), (dict(F=12), -2),
    (dict(T=-1), -2), (dict(n_shared=9), -2), (dict(vocab=0), -2),
])
def test_bad_shapes_rejected(lib, kw, code):
    d = base_desc(**kw)
    assert lib.smoe_workspace_size(ctypes.byref(d)) == 0
    rc = lib.smoe_route(ctypes.byref(d), 16, 16, None, 16, 16, 16, None, 0, None)
    assert rc == code
    assert lib.smoe_last_error()


def test_bad_enum_and_null(lib):
    d = base_desc()
    d.dtype = 7
    assert lib.smoe_route(ctypes.byref(d), 16, 16, None, 16, 16, 16, None, 0, None) == -1
    d = base_desc()
    assert lib.smoe_route(ctypes.byref(d), 16, 16, None, 16, None, 16, None, 0, None) == -1
    assert lib.smoe_route(None, 16, 16, None, 16, 16, 16, None, 0, None) == -1


def test_misaligned_pointer_rejected(lib):
    d = base_desc()
    assert lib.smoe_route(ctypes.byref(d), 16 + 4, 16, None, 16, 16, 16, None, 0, None) == -3


def test_workspace_checks(lib):
    d = base_desc()
    n = B.workspace_size(d)
    args = [ctypes.byref(d), 16, 16, 16, 16, 16, 16, 16, None]
    assert lib.smoe_predict_shuffle(*args, None, n, None) == -4
    assert lib.smoe_predict_shuffle(*args, 256 + 16, n, None) == -3
    assert lib.smoe_predict_shuffle(*args, 256, n - 1, None) == -4


def test_grouped_source_rule_needs_divisibility(lib):
    d = base_desc(E=12, K=3, H=3, P=4)
    n = B.workspace_size(d)
    assert lib.smoe_lar(ctypes.byref(d), 16, None, 16, 16, 256, n, None) == -2


def test_newer_entry_points_validate_on_the_host(lib):
    """Missing or misaligned required pointers are rejected before any CUDA call by the
    inter-layer, routed-forward, prefetch and combine entry points."""
    d = base_desc()
    n = B.workspace_size(d)
    D = ctypes.byref(d)
    # smoe_token_cluster(desc, topk_idx, expert_part, cluster, ws, ws_bytes, stream)
    assert lib.smoe_token_cluster(D, None, 16, 16, 256, n, None) == -1
    assert lib.smoe_token_cluster(D, 16 + 8, 16, 16, 256, n, None) == -3
    # smoe_predict_shuffle_inter(desc, ids, conf, map, prev, table_a, x, pred, perm, off,
    #                            x_shuf, ws, ws_bytes, stream)
    assert lib.smoe_predict_shuffle_inter(D, 16, 16, 16, None, 16, None, 16, 16, 16, None, 256,
                                          n, None) == -1
    assert lib.smoe_predict_shuffle_inter(D, 16, 16, 16, 16, 16 + 4, None, 16, 16, 16, None, 256,
                                          n, None) == -3
    # smoe_moe_forward_routed(desc, x, idx, w, w1, w3, w2, y, ws, ws_bytes, stream)
    assert lib.smoe_moe_forward_routed(D, 16, 16, 16, 16, 16, None, 16, 256, n, None) == -1
    assert lib.smoe_moe_forward_routed(D, 16, 16, 16, 16, 16, 16, 16, None, n, None) == -4
    # smoe_prefetch_predict(desc, r, d_l, y, gamma, beta, w_gate_next, logits_q, logits_s,
    #                       pred_idx, true_idx, hits, qs_out, ws, ws_bytes, stream)
    assert lib.smoe_prefetch_predict(D, None, 16, 16, 16, 16, 16, None, None, 16, 16, 16, None,
                                     256, n, None) == -1
    # smoe_combine(desc, y_disp, pair_row, topk_w, y_shared, y_out, ws, ws_bytes, stream)
    assert lib.smoe_combine(D, 16, 16 + 4, 16, None, 16, 256, n, None) == -3
    assert lib.smoe_combine(D, 16, 16, 16, None, None, 256, n, None) == -1


def test_ffn_gather_validates_on_the_host(lib):
    """smoe_expert_ffn_gather rejects missing or misaligned pointers before any CUDA call."""
    d = base_desc()
    n = B.workspace_size(d)
    D = ctypes.byref(d)
    # smoe_expert_ffn_gather(desc, x_src, row_slot, x, x_disp, expert_off, w1, w3, w2, y_disp,
    #                        y_shared, ws, ws_bytes, stream)
    assert lib.smoe_expert_ffn_gather(D, 16, None, None, 16, 16, 16, 16, 16, 16, None, 256, n,
                                      None) == -1
    assert lib.smoe_expert_ffn_gather(D, 16, 16 + 4, None, 16, 16, 16, 16, 16, 16, None, 256, n,
                                      None) == -3
    assert lib.smoe_expert_ffn_gather(D, 16, 16, None, 16, 16, 16, 16, 16, 16, None, 256, 16,
                                      None) == -4


def test_shuffle_dispatch_rows_validates_on_the_host(lib):
    d = base_desc()
    n = B.workspace_size(d)
    D = ctypes.byref(d)
    # smoe_shuffle_dispatch_rows(desc, x, shuf_perm, pair_row, x_shuf, x_disp, ws, ws_bytes,
    #                            stream)
    f = lib.smoe_shuffle_dispatch_rows
    assert f(D, None, 16, 16, 16, 16, 256, n, None) == -1        # x missing
    assert f(D, 16, 16, None, 16, 16, 256, n, None) == -1        # pair_row missing
    assert f(D, 16, 16, 16, 16, None, 256, n, None) == -1        # x_disp missing
    assert f(D, 16, None, 16, 16, 16, 256, n, None) == -1        # x_shuf without shuf_perm
    assert f(D, 16, 16 + 4, 16, 16, 16, 256, n, None) == -3      # misaligned
    assert f(D, 16, 16, 16, 16, 16, 256, 16, None) == -4         # workspace too small


def test_ffn_gather_fused_query(lib):
    """The row copy runs inside the up GEMM only on bf16 two-SM tiles with F <= 1024: of
    the workloads, the Qwen3-shaped layer (F = 768, 1024 rows per expert)."""
    fused = {name: B.smoe_expert_ffn_gather_fused(B.desc_from_config(cfg))
             for name, cfg in synth.CONFIGS.items()}
    assert fused == {name: name == "qwen3_foe" for name in synth.CONFIGS}, fused
    assert B.smoe_expert_ffn_gather_fused(base_desc(T=1024, E=8, K=2, F=1024))
    assert not B.smoe_expert_ffn_gather_fused(base_desc(T=1024, E=8, K=2, F=1088))
    assert not B.smoe_expert_ffn_gather_fused(base_desc(T=1023, E=8, K=2, F=256))  # < 256 rows
    assert not B.smoe_expert_ffn_gather_fused(base_desc(T=1024, E=8, K=2, F=256, dtype="f32"))
    assert not B.smoe_expert_ffn_gather_fused(base_desc(K=9))                     # invalid


def test_prefetch_rejects_d_above_8192(lib):
    d = base_desc(d=8200)
    n = B.workspace_size(d)
    rc = lib.smoe_prefetch_predict(ctypes.byref(d), 16, 16, 16, 16, 16, 16, None, None, 16, 16,
                                   16, None, 256, n, None)
    assert rc == -2 and b"8192" in lib.smoe_last_error()


def test_binding_refuses_strided_views(lib):
    """The ABI takes dense row-major buffers: a transposed or column-sliced tensor is refused
    by the binding before the C call, instead of being read as if it were dense."""
    import torch
    d = base_desc(T=16, d=64, E=8, K=2)
    y_disp = torch.zeros(64, 32)                     # [d, T*K] storage, viewed transposed
    pair_row = torch.zeros(16, 2, dtype=torch.int32)
    topk_w = torch.zeros(16, 4)[:, :2]               # column slice
    y_out = torch.zeros(16, 64)
    ws = torch.zeros(256, dtype=torch.uint8)
    with pytest.raises(ValueError, match="not contiguous"):
        B.smoe_combine(d, y_disp.t(), pair_row, topk_w.contiguous(), y_out, ws, stream=0)
    with pytest.raises(ValueError, match="not contiguous"):
        B.smoe_combine(d, y_disp.t().contiguous(), pair_row, topk_w, y_out, ws, stream=0)
    assert B._ptr(y_out[3:7]) == y_out.data_ptr() + 3 * 64 * 4   # a row range stays dense


def test_exchange_srs_sag_validate_on_the_host(lib):
    """The expert-parallel exchange, SRS and SAG reject missing, misaligned or badly sized
    arguments before any CUDA call."""
    d = base_desc()
    n = B.workspace_size(d)
    D = ctypes.byref(d)
    # smoe_ep_exchange(desc, idx, src_part, map, x, send_counts, recv_off, pair_recv,
    #                  recv_token, x_recv, ws, ws_bytes, stream)
    assert lib.smoe_ep_exchange(D, None, None, 16, None, 16, 16, 16, 16, None, 256, n, None) == -1
    assert lib.smoe_ep_exchange(D, 16, 16 + 4, 16, None, 16, 16, 16, 16, None, 256, n,
                                None) == -3
    assert lib.smoe_ep_exchange(D, 16, None, 16, None, 16, 16, 16, 16, 16, 256, n, None) == -1
    assert lib.smoe_ep_exchange(D, 16, None, 16, None, 16, 16, 16, 16, None, 256, n - 1,
                                None) == -4
    # smoe_srs(desc, R, x_parts, perm, x_shuf, ws, ws_bytes, stream)
    assert lib.smoe_srs(D, 0, 16, 16, 16, 256, n, None) == -2
    assert lib.smoe_srs(D, 65, 16, 16, 16, 256, n, None) == -2
    assert lib.smoe_srs(D, 2, 16, None, 16, 256, n, None) == -1
    assert lib.smoe_srs(D, 2, 16, 16, 16 + 8, 256, n, None) == -3
    # smoe_sag(desc, y_shuf, perm, y, ws, ws_bytes, stream)
    assert lib.smoe_sag(D, 16, 16, None, 256, n, None) == -1
    assert lib.smoe_sag(D, 16, 16, 16, None, n, None) == -4
