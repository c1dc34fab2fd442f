"""GPU parity: every entry point of the C ABI against the CPU oracle.

Indices, permutations, offsets and counts are compared bit for bit, given the fp32
logits the GPU exported; values are compared within 2e-2 (max over rows of the
row's max-abs error over its max-abs reference value). Each workload runs at a
ragged size the oracle checks in full and at its full size, where values are
checked on a seeded sample of tokens that includes the last (ragged-tail) token.
"""
import numpy as np
import pytest
import torch

import oracle as O
import routing_token_shuffle_gb300 as smoe
from routing_token_shuffle_gb300 import synth

from _cases import Case, block_edge_rows, rel_err_rows, sample_tokens, to_np

pytestmark = pytest.mark.gpu

VALUE_TOL = 2e-2
MARGIN = 1e-3

CASES = [("tiny_fp32", None), ("tiny_fp32", 37), ("mixtral", 1001), ("dsv2_prefill", 1537),
         ("dsv2_decode", None), ("qwen3_foe", 3001),
         ("mixtral", None), ("dsv2_prefill", None), ("qwen3_foe", None)]
IDS = [f"{n}-T{t or 'full'}" for n, t in CASES]

_cache = {}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()
    yield
    _cache.clear()


def get_case(name, T):
    key = (name, T)
    if key not in _cache:
        if len(_cache) > 2:
            _cache.clear()
            torch.cuda.empty_cache()
        _cache[key] = Case(name, "cuda", T=T)
    return _cache[key]


def i32(*shape):
    return torch.empty(*shape, dtype=torch.int32, device="cuda")


def f32(*shape):
    return torch.empty(*shape, dtype=torch.float32, device="cuda")


def run_route(c, desc, ws):
    cfg = c.cfg
    logits, idx, w = f32(cfg.T, cfg.E), i32(cfg.T, cfg.K), f32(cfg.T, cfg.K)
    smoe.smoe_route(desc, c.x, c.w_gate, idx, w, logits_out=logits, ws=ws)
    return logits, idx, w


@pytest.mark.parametrize("name,T", CASES, ids=IDS)
def test_route(name, T):
    c = get_case(name, T)
    cfg = c.cfg
    desc = smoe.desc_from_config(cfg)
    ws = smoe.workspace(desc)
    logits, idx, w = run_route(c, desc, ws)
    torch.cuda.synchronize()
    L = to_np(logits)
    ref_idx = O.topk_select(L, cfg.K, cfg.H)
    assert np.array_equal(to_np(idx), ref_idx)
    np.testing.assert_allclose(to_np(w), O.gate_weights(L, ref_idx), rtol=2e-6, atol=1e-7)
    rows = sample_tokens(cfg.T, 64)
    ref_l = O.gate_logits(c.x_np[rows], to_np(c.w_gate))
    err = np.abs(L[rows] - ref_l).max(axis=1) / np.abs(ref_l).max(axis=1)
    assert err.max() < 1e-4, err.max()
    # routing the oracle's logits through logits_in gives the oracle's routes
    full_ref = O.gate_logits(c.x_np, to_np(c.w_gate)) if cfg.T <= 4096 else None
    if full_ref is not None:
        lin = torch.as_tensor(full_ref, device="cuda")
        idx2, w2 = i32(cfg.T, cfg.K), f32(cfg.T, cfg.K)
        smoe.smoe_route(desc, None, None, idx2, w2, logits_in=lin, ws=ws)
        torch.cuda.synchronize()
        assert np.array_equal(to_np(idx2), O.topk_select(full_ref, cfg.K, cfg.H))


@pytest.mark.parametrize("E,K,H", [(8, 2, 1), (160, 6, 1), (128, 8, 8), (64, 8, 2), (512, 32, 1),
                                   (16, 16, 16), (33 * 3, 3, 3), (8, 8, 1), (32, 8, 1),
                                   (33, 3, 1), (65, 5, 1), (129, 9, 1), (256, 16, 2),
                                   (257, 4, 1), (300, 20, 5), (64, 8, 8), (256, 8, 8)])
@pytest.mark.parametrize("renorm", [0, 1])
def test_route_selection_ties(E, K, H, renorm):
    """Many exact ties (small-integer logits, +0 and -0): lower index wins. The shapes
    cover every selection kernel: 8 lanes per token (E <= 32, 64, 128), 16 lanes
    (E <= 256 or 8 < K <= 16), one warp per token (E > 256 or K > 16) and grouped top-1
    over 8 groups (E = 64, 128, 256)."""
    T = 777
    rng = np.random.default_rng(E + K + H)
    vals = np.array([-2.0, -1.0, -0.0, 0.0, 1.0, 3.0], np.float32)
    L = vals[rng.integers(0, len(vals), size=(T, E))]
    L[:50] = rng.standard_normal((50, E)).astype(np.float32)
    desc = smoe.make_desc(T, 64, E, K, H, 64, 0, 2, 100, "bf16", renorm)
    idx, w = i32(T, K), f32(T, K)
    smoe.smoe_route(desc, None, None, idx, w, logits_in=torch.as_tensor(L, device="cuda"))
    torch.cuda.synchronize()
    ref = O.topk_select(L, K, H)
    assert np.array_equal(to_np(idx), ref)
    np.testing.assert_allclose(to_np(w), O.gate_weights(L, ref, renorm=bool(renorm)), rtol=2e-6,
                               atol=1e-7)



@pytest.mark.parametrize("T,d,E,K,H", [(1001, 256, 8, 2, 1), (777, 512, 160, 6, 1),
                                       (5000, 256, 128, 8, 8), (19000, 128, 64, 8, 2),
                                       (300, 192, 16, 8, 8), (300, 192, 16, 16, 16),
                                       (650, 320, 99, 3, 3),
                                       (64, 1024, 8, 8, 1), (2000, 256, 256, 16, 2),
                                       (129, 512, 256, 8, 8), (700, 256, 64, 8, 8),
                                       (64, 5120, 160, 6, 1), (1, 64, 1, 1, 1),
                                       (5, 64, 256, 16, 16), (130, 64, 129, 16, 1),
                                       (33, 4096, 40, 8, 4), (20000, 128, 64, 8, 2),
                                       (40000, 64, 128, 8, 8)])
@pytest.mark.parametrize("renorm", [0, 1])
def test_route_fused_gemm_ties(T, d, E, K, H, renorm):
    """The bf16 gate GEMM with the selection in its epilogue (E <= 256, K <= 8 lanes per
    token for E <= 128, else 16), split over clusters of 1, 2, 4 or 8 CTAs, and with more
    128-row tiles than SMs in its compact form (256 threads, two CTAs per SM); E = 16 with
    K = 16 takes the two-launch path. x and W_g in {-1, 0, 1} make every logit an exact
    small integer, so the exported logits must equal the exact products and many of them
    tie (the lower index must win); picks and weights are then checked against the
    oracle's selection on those logits."""
    rng = np.random.default_rng(T + d + E + K + H)
    xn = rng.integers(-1, 2, size=(T, d)).astype(np.float32)
    wn = rng.integers(-1, 2, size=(E, d)).astype(np.float32)
    x = torch.as_tensor(xn, device="cuda").to(torch.bfloat16)
    wg = torch.as_tensor(wn, device="cuda").to(torch.bfloat16)
    desc = smoe.make_desc(T, d, E, K, H, 64, 0, 2, 100, "bf16", renorm)
    ws = smoe.workspace(desc)
    logits, idx, w = f32(T, E), i32(T, K), f32(T, K)
    smoe.smoe_route(desc, x, wg, idx, w, logits_out=logits, ws=ws)
    smoe.smoe_get_status(ws)
    torch.cuda.synchronize()
    L = to_np(logits)
    exact = (xn.astype(np.float64) @ wn.astype(np.float64).T).astype(np.float32)
    assert np.array_equal(L, exact)
    ref = O.topk_select(L, K, H)
    assert np.array_equal(to_np(idx), ref)
    np.testing.assert_allclose(to_np(w), O.gate_weights(L, ref, renorm=bool(renorm)), rtol=2e-6,
                               atol=1e-7)

def run_shuffle(c, desc, ws, with_x=True):
    cfg = c.cfg
    pred, perm, off = i32(cfg.T), i32(cfg.T), i32(cfg.P + 1)
    xs = torch.empty_like(c.x) if with_x else None
    smoe.smoe_predict_shuffle(desc, c.ids_d, c.conf_d, c.emap_d, pred, perm, off, ws,
                              x=c.x if with_x else None, x_shuf=xs)
    return pred, perm, off, xs


@pytest.mark.parametrize("name,T", CASES, ids=IDS)
def test_predict_shuffle(name, T):
    c = get_case(name, T)
    cfg = c.cfg
    desc = smoe.desc_from_config(cfg)
    ws = smoe.workspace(desc)
    pred, perm, off, xs = run_shuffle(c, desc, ws)
    smoe.smoe_get_status(ws)
    ref_pred = O.predict_partition(c.ids, c.conf, c.emap, cfg.P)
    ref_perm, ref_off = O.token_shuffle(ref_pred, cfg.P)
    assert np.array_equal(to_np(pred), ref_pred)
    assert np.array_equal(to_np(perm), ref_perm)
    assert np.array_equal(to_np(off), ref_off)
    assert torch.equal(xs, c.x[torch.as_tensor(ref_perm, device="cuda").long()])


def test_predict_ties_and_empty_partitions():
    """Rows with exactly tied partition scores and partitions without experts."""
    V, E, P, T = 64, 12, 5, 3000
    rng = np.random.default_rng(5)
    conf = np.full((V, E), 0.25, np.float32)
    conf[: V // 2] = (rng.integers(0, 9, size=(V // 2, E)) / 8).astype(np.float32)
    emap = np.array([0, 1, 3, 0, 1, 3, 0, 1, 3, 0, 1, 3], np.int32)   # partitions 2, 4 empty
    ids = rng.integers(0, V, size=T).astype(np.int32)
    desc = smoe.make_desc(T, 64, E, 2, 1, 64, 0, P, V, "bf16")
    ws = smoe.workspace(desc)
    pred, perm, off = i32(T), i32(T), i32(P + 1)
    smoe.smoe_predict_shuffle(desc, torch.as_tensor(ids, device="cuda"),
                              torch.as_tensor(conf, device="cuda"),
                              torch.as_tensor(emap, device="cuda"), pred, perm, off, ws)
    smoe.smoe_get_status(ws)
    ref = O.predict_partition(ids, conf, emap, P)
    assert np.array_equal(to_np(pred), ref)
    rp, ro = O.token_shuffle(ref, P)
    assert np.array_equal(to_np(perm), rp) and np.array_equal(to_np(off), ro)


@pytest.mark.parametrize("name,T", CASES, ids=IDS)
def test_lar(name, T):
    c = get_case(name, T)
    cfg = c.cfg
    desc = smoe.desc_from_config(cfg)
    ws = smoe.workspace(desc)
    logits, idx, w = run_route(c, desc, ws)
    pred, perm, off, _ = run_shuffle(c, desc, ws, with_x=False)
    counts = torch.empty(4, dtype=torch.int64, device="cuda")
    smoe.smoe_lar(desc, idx, c.emap_d, counts, ws, src_part=pred)
    got = to_np(counts).astype(np.uint64)
    ref = O.lar_counts(to_np(idx), c.emap, cfg.P, cfg.H, src_part=to_np(pred))
    assert np.array_equal(got, ref)
    if cfg.P % cfg.H == 0 or cfg.H >= cfg.P:
        foe_map = synth.placement_foe(cfg.E, cfg.H, cfg.P)
        smoe.smoe_lar(desc, idx, torch.as_tensor(foe_map, device="cuda"), counts, ws)
        ref2 = O.lar_counts(to_np(idx), foe_map, cfg.P, cfg.H)
        assert np.array_equal(to_np(counts).astype(np.uint64), ref2)
        if cfg.H >= cfg.P:
            assert ref2[0] == ref2[1]           # rho_foe = min(H/G, 1) = 1
    smoe.smoe_get_status(ws)


@pytest.mark.parametrize("name,T", CASES, ids=IDS)
def test_dispatch(name, T):
    c = get_case(name, T)
    cfg = c.cfg
    desc = smoe.desc_from_config(cfg)
    ws = smoe.workspace(desc)
    logits, idx, w = run_route(c, desc, ws)
    pred, perm, off, xs = run_shuffle(c, desc, ws)
    TK = cfg.T * cfg.K
    eo, pr, rt, rs = i32(cfg.E + 1), i32(cfg.T, cfg.K), i32(TK), i32(TK)
    xd = torch.empty(TK, cfg.d, dtype=c.x.dtype, device="cuda")
    smoe.smoe_dispatch(desc, idx, eo, pr, rt, ws, shuf_perm=perm, x_src=xs, x_disp=xd, row_slot=rs)
    smoe.smoe_get_status(ws)
    r_eo, r_pr, r_rt = O.expert_dispatch(to_np(idx), cfg.E, to_np(perm))
    assert np.array_equal(to_np(eo), r_eo)
    assert np.array_equal(to_np(pr), r_pr)
    assert np.array_equal(to_np(rt), r_rt)
    slot_of = np.empty(cfg.T, np.int64)
    slot_of[to_np(perm)] = np.arange(cfg.T)
    assert np.array_equal(to_np(rs), slot_of[r_rt])          # row -> slot of its token
    assert torch.equal(xd, c.x[torch.as_tensor(r_rt, device="cuda").long()])
    # without the shuffle: token order, source rows straight from x
    smoe.smoe_dispatch(desc, idx, eo, pr, rt, ws, x_src=c.x, x_disp=xd)
    smoe.smoe_get_status(ws)
    r_eo, r_pr, r_rt = O.expert_dispatch(to_np(idx), cfg.E, None)
    assert np.array_equal(to_np(pr), r_pr) and np.array_equal(to_np(rt), r_rt)
    assert torch.equal(xd, c.x[torch.as_tensor(r_rt, device="cuda").long()])


@pytest.mark.parametrize("name,T", CASES, ids=IDS)
def test_shuffle_dispatch_rows(name, T):
    """x_shuf and the dispatched rows written from one read of x: bit for bit the
    oracle's shuffle (x[perm]) and dispatch (x[row_token]) on the oracle's own
    permutations, with the shuffle and without it (rows in token order, no x_shuf); a
    slot with an out-of-range token gives a zero x_shuf row and a pair_row entry out of
    range is skipped, both reported."""
    c = get_case(name, T)
    cfg = c.cfg
    desc = smoe.desc_from_config(cfg)
    ws = smoe.workspace(desc)
    logits, idx, w = run_route(c, desc, ws)
    pred, perm, off, _ = run_shuffle(c, desc, ws, with_x=False)
    smoe.smoe_get_status(ws)
    ref_pred = O.predict_partition(c.ids, c.conf, c.emap, cfg.P)
    ref_perm, _ = O.token_shuffle(ref_pred, cfg.P)
    assert np.array_equal(to_np(perm), ref_perm)
    TK = cfg.T * cfg.K
    eo, pr, rt = i32(cfg.E + 1), i32(cfg.T, cfg.K), i32(TK)
    smoe.smoe_dispatch(desc, idx, eo, pr, rt, ws, shuf_perm=perm)
    r_eo, r_pr, r_rt = O.expert_dispatch(to_np(idx), cfg.E, ref_perm)
    assert np.array_equal(to_np(pr), r_pr)
    xsh = torch.full_like(c.x, 5.0)
    xd = torch.full((TK, cfg.d), 7.0, dtype=c.x.dtype, device="cuda")
    smoe.smoe_shuffle_dispatch_rows(desc, c.x, pr, xd, ws, shuf_perm=perm, x_shuf=xsh)
    smoe.smoe_get_status(ws)
    assert torch.equal(xsh, c.x[torch.as_tensor(ref_perm, device="cuda").long()])
    assert torch.equal(xd, c.x[torch.as_tensor(r_rt, device="cuda").long()])
    # without the shuffle: the pairs in token order, no x_shuf
    smoe.smoe_dispatch(desc, idx, eo, pr, rt, ws)
    _, r_pr0, r_rt0 = O.expert_dispatch(to_np(idx), cfg.E, None)
    xd0 = torch.full_like(xd, 3.0)
    smoe.smoe_shuffle_dispatch_rows(desc, c.x, pr, xd0, ws)
    smoe.smoe_get_status(ws)
    assert torch.equal(xd0, c.x[torch.as_tensor(r_rt0, device="cuda").long()])
    # planted bad entries: a slot's token and one pair's row
    s_bad, t_bad = cfg.T // 3, int(ref_perm[cfg.T // 2])
    bad_perm = perm.clone()
    bad_perm[s_bad] = cfg.T + 7
    bad_pr = torch.as_tensor(r_pr, device="cuda").clone()
    r_lost = int(bad_pr[t_bad, 0])
    bad_pr[t_bad, 0] = -3
    xsh2, xd2 = torch.full_like(c.x, 5.0), torch.full_like(xd, 7.0)
    smoe.smoe_shuffle_dispatch_rows(desc, c.x, bad_pr, xd2, ws, shuf_perm=bad_perm, x_shuf=xsh2)
    with pytest.raises(smoe.SmoeError):
        smoe.smoe_get_status(ws)
    assert (xsh2[s_bad] == 0).all()
    keep_s = torch.ones(cfg.T, dtype=torch.bool, device="cuda")
    keep_s[s_bad] = False
    assert torch.equal(xsh2[keep_s], xsh[keep_s])
    assert (xd2[r_lost] == 7.0).all()                      # the skipped row is untouched
    t_skip = int(ref_perm[s_bad])                          # that slot's rows were not written
    lost = {r_lost} | {int(r) for r in r_pr[t_skip]}
    keep_r = torch.ones(TK, dtype=torch.bool, device="cuda")
    keep_r[sorted(lost)] = False
    assert torch.equal(xd2[keep_r], xd[keep_r])


@pytest.mark.parametrize("T,d,K,dtype", [(300, 64, 32, "bf16"), (37, 8, 3, "bf16"),
                                         (129, 200, 5, "bf16"), (64, 256, 1, "f32"),
                                         (1000, 2056, 7, "bf16")],
                         ids=["d64-K32", "d8-K3", "d200-K5", "d256f32-K1", "d2056-K7"])
def test_shuffle_dispatch_rows_row_lengths(T, d, K, dtype):
    """One read of x for x_shuf and the dispatched rows, at row lengths of 1 to 257
    16-byte vectors (fewer than a warp's lanes, a ragged last chunk, several chunks) and
    K up to 32: every x_shuf row is x[perm[s]] and every dispatched row x[t] of its pair,
    for random permutations of the slots and of the T K rows."""
    E = 32
    desc = smoe.make_desc(T, d, E, K, 1, 64, 0, 2, 100, dtype)
    ws = smoe.workspace(desc)
    g = torch.Generator(device="cuda").manual_seed(T + d + K)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    x = torch.randn(T, d, generator=g, device="cuda").to(tdt)
    perm = torch.randperm(T, generator=g, device="cuda").to(torch.int32)
    pair_row = torch.randperm(T * K, generator=g, device="cuda").to(torch.int32).view(T, K)
    xsh = torch.full_like(x, 5.0)
    xd = torch.full((T * K, d), 7.0, dtype=tdt, device="cuda")
    smoe.smoe_shuffle_dispatch_rows(desc, x, pair_row, xd, ws, shuf_perm=perm, x_shuf=xsh)
    smoe.smoe_get_status(ws)
    assert torch.equal(xsh, x[perm.long()])
    ref = torch.empty_like(xd)
    ref[pair_row.long().view(-1)] = x.repeat_interleave(K, dim=0)
    assert torch.equal(xd, ref)


GATHER_CASES = [("tiny_fp32", 37), ("mixtral", 1001), ("dsv2_prefill", 1537), ("dsv2_decode", None),
                ("qwen3_foe", 3001), ("mixtral", None), ("qwen3_foe", None)]


@pytest.mark.parametrize("name,T", GATHER_CASES, ids=[f"{n}-T{t or 'full'}" for n, t in GATHER_CASES])
def test_expert_ffn_gather(name, T):
    """smoe_expert_ffn_gather (the dispatch's row copy inside the up GEMM on two-SM tiles,
    a copy launch before the FFN otherwise) writes the same X_disp rows and, bit for bit,
    the same expert outputs as smoe_dispatch's rows followed by smoe_expert_ffn, also in
    place (X_disp and Y_disp one buffer); a bad row index gives a zero row and a data
    error."""
    c = get_case(name, T)
    cfg = c.cfg
    desc = smoe.desc_from_config(cfg)
    ws = smoe.workspace(desc)
    logits, idx, w = run_route(c, desc, ws)
    pred, perm, off, xs = run_shuffle(c, desc, ws)
    TK = cfg.T * cfg.K
    eo, pr, rt, rs = i32(cfg.E + 1), i32(cfg.T, cfg.K), i32(TK), i32(TK)
    xd = torch.empty(TK, cfg.d, dtype=c.x.dtype, device="cuda")
    smoe.smoe_dispatch(desc, idx, eo, pr, rt, ws, shuf_perm=perm, x_src=xs, x_disp=xd, row_slot=rs)
    yd = torch.empty_like(xd)

    def shared():
        return (torch.empty(cfg.n_shared, cfg.T, cfg.d, dtype=c.x.dtype, device="cuda")
                if cfg.n_shared else None)

    ysh = shared()
    smoe.smoe_expert_ffn(desc, xd, eo, c.w1, c.w3, c.w2, yd, ws, x=c.x, y_shared=ysh)
    xd2, yd2, ysh2 = torch.full_like(xd, 3.0), torch.full_like(xd, 5.0), shared()
    smoe.smoe_expert_ffn_gather(desc, xs, rs, xd2, eo, c.w1, c.w3, c.w2, yd2, ws, x=c.x,
                                y_shared=ysh2)
    smoe.smoe_get_status(ws)
    assert torch.equal(xd2, xd)
    assert torch.equal(yd2, yd)
    if ysh is not None:
        assert torch.equal(ysh2, ysh)
    buf = torch.full_like(xd, 7.0)
    smoe.smoe_expert_ffn_gather(desc, xs, rs, buf, eo, c.w1, c.w3, c.w2, buf, ws, x=c.x,
                                y_shared=ysh2)
    smoe.smoe_get_status(ws)
    assert torch.equal(buf, yd)
    bad = rs.clone()
    bad[TK // 2] = cfg.T + 5
    xd3 = torch.full_like(xd, 3.0)
    smoe.smoe_expert_ffn_gather(desc, xs, bad, xd3, eo, c.w1, c.w3, c.w2, yd2, ws, x=c.x,
                                y_shared=ysh2)
    with pytest.raises(smoe.SmoeError):
        smoe.smoe_get_status(ws)
    assert (xd3[TK // 2] == 0).all()
    keep = torch.ones(TK, dtype=torch.bool, device="cuda")
    keep[TK // 2] = False
    assert torch.equal(xd3[keep], xd[keep])


@pytest.mark.parametrize("d,F,counts,S", [
    (2048, 768, [700, 1300, 0, 1024, 97, 3001, 256, 1], 0),
    (5120, 512, [300, 0, 513, 129, 1100], 1),
    (256, 256, [64, 300, 450, 0, 129, 128, 513, 500], 1),
    (384, 704, [1, 2000, 255, 700], 0)],
    ids=["d2048-chunk4", "d5120-chunk1", "d256-chunk32", "d384-chunk16"])
def test_expert_ffn_gather_in_gemm(d, F, counts, S):
    """The in-GEMM row copy (bf16 two-SM tiles, F <= 1024) with chunks of 1 to 32 rows,
    ragged and empty expert segments and shared experts: X_disp and the expert outputs
    equal a torch row gather followed by smoe_expert_ffn, bit for bit."""
    E, K = len(counts), 2
    TK = sum(counts)
    T = (TK + K - 1) // K
    desc = smoe.make_desc(T, d, E, K, 1, F, S, 2, 100, "bf16")
    assert smoe.smoe_expert_ffn_gather_fused(desc)
    g = torch.Generator(device="cuda").manual_seed(d + F)
    x = torch.randn(T, d, generator=g, device="cuda").to(torch.bfloat16)
    w1 = (torch.randn(E + S, F, d, generator=g, device="cuda") / d ** 0.5).to(torch.bfloat16)
    w3 = (torch.randn(E + S, F, d, generator=g, device="cuda") / d ** 0.5).to(torch.bfloat16)
    w2 = (torch.randn(E + S, d, F, generator=g, device="cuda") / F ** 0.5).to(torch.bfloat16)
    slots = torch.randint(0, T, (T * K,), generator=g, device="cuda", dtype=torch.int32)
    slots[TK:] = 0
    eo = torch.as_tensor(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32), device="cuda")
    ws = smoe.workspace(desc)
    xd_ref = x[slots.long()]
    xd_ref[TK:] = 0
    y_ref = torch.empty_like(xd_ref)
    ysh_ref = torch.empty(S, T, d, dtype=torch.bfloat16, device="cuda") if S else None
    smoe.smoe_expert_ffn(desc, xd_ref, eo, w1, w3, w2, y_ref, ws, x=x, y_shared=ysh_ref)
    xd, y = torch.zeros_like(xd_ref), torch.full_like(xd_ref, 9.0)
    ysh = torch.empty_like(ysh_ref) if S else None
    smoe.smoe_expert_ffn_gather(desc, x, slots, xd, eo, w1, w3, w2, y, ws, x=x, y_shared=ysh)
    smoe.smoe_get_status(ws)
    assert torch.equal(xd[:TK], xd_ref[:TK])
    assert torch.equal(y[:TK], y_ref[:TK])
    if S:
        assert torch.equal(ysh, ysh_ref)


@pytest.mark.parametrize("name,T", CASES, ids=IDS)
def test_expert_ffn_and_combine(name, T):
    c = get_case(name, T)
    cfg = c.cfg
    desc = smoe.desc_from_config(cfg)
    ws = smoe.workspace(desc)
    logits, idx, w = run_route(c, desc, ws)
    TK = cfg.T * cfg.K
    eo, pr, rt = i32(cfg.E + 1), i32(cfg.T, cfg.K), i32(TK)
    xd = torch.empty(TK, cfg.d, dtype=c.x.dtype, device="cuda")
    smoe.smoe_dispatch(desc, idx, eo, pr, rt, ws, x_src=c.x, x_disp=xd)
    yd = torch.empty_like(xd)
    ysh = (torch.empty(cfg.n_shared, cfg.T, cfg.d, dtype=c.x.dtype, device="cuda")
           if cfg.n_shared else None)
    smoe.smoe_expert_ffn(desc, xd, eo, c.w1, c.w3, c.w2, yd, ws, x=c.x, y_shared=ysh)
    y = torch.empty_like(c.x)
    smoe.smoe_combine(desc, yd, pr, w, y, ws, y_shared=ysh)
    smoe.smoe_get_status(ws)
    torch.cuda.synchronize()
    # expert outputs on sampled rows plus the first and last row of every 64-row block of
    # every expert segment: both CTAs of every tile, every wave of the persistent schedule
    eo_n, rt_n, idx_n = to_np(eo), to_np(rt), to_np(idx)
    rows = set(sample_tokens(TK, 48, seed=1).tolist())
    rows.update(block_edge_rows(eo_n).tolist())
    rows = np.array(sorted(rows))
    row_exp = np.searchsorted(eo_n, rows, side="right") - 1
    ref = np.zeros((len(rows), cfg.d))
    for e in np.unique(row_exp):
        sel = row_exp == e
        ref[sel] = O.swiglu_ffn(c.x_np[rt_n[rows[sel]]], *c.expert_weights_np(int(e)))
    assert rel_err_rows(to_np(yd)[rows], ref).max() <= VALUE_TOL
    if cfg.n_shared:
        toks = np.union1d(sample_tokens(cfg.T, 16, seed=2), block_edge_rows([0, cfg.T]))
        for j in range(cfg.n_shared):
            rj = O.swiglu_ffn(c.x_np[toks], *c.expert_weights_np(cfg.E + j))
            assert rel_err_rows(to_np(ysh[j])[toks], rj).max() <= VALUE_TOL
    # combine against the oracle's combine of the GPU's own expert outputs
    toks = sample_tokens(cfg.T, 256, seed=3)
    y_rows = to_np(yd)
    ysh_n = to_np(ysh)[:, toks] if cfg.n_shared else None
    ref_y = O.combine(y_rows, to_np(pr)[toks], to_np(w)[toks], ysh_n)
    tol = 1e-5 if cfg.dtype == "f32" else 8e-3
    assert rel_err_rows(to_np(y)[toks], ref_y).max() <= tol


@pytest.mark.parametrize("name,T", CASES, ids=IDS)
def test_layer_forward(name, T):
    c = get_case(name, T)
    cfg = c.cfg
    desc = smoe.desc_from_config(cfg)
    ws = smoe.workspace(desc)
    TK = cfg.T * cfg.K
    outs = dict(logits=f32(cfg.T, cfg.E), topk_idx=i32(cfg.T, cfg.K), topk_w=f32(cfg.T, cfg.K),
                pred_part=i32(cfg.T), shuf_perm=i32(cfg.T), part_off=i32(cfg.P + 1),
                expert_off=i32(cfg.E + 1), pair_row=i32(cfg.T, cfg.K), row_token=i32(TK),
                lar=torch.empty(4, dtype=torch.int64, device="cuda"))
    y = torch.empty_like(c.x)
    W = smoe.layer_weights(c.w_gate, c.w1, c.w3, c.w2, c.conf_d, c.emap_d)
    smoe.smoe_layer_forward(desc, W, smoe.layer_io(c.x, c.ids_d, y, **outs), ws)
    smoe.smoe_get_status(ws)
    torch.cuda.synchronize()
    L = to_np(outs["logits"])
    idx = O.topk_select(L, cfg.K, cfg.H)
    assert np.array_equal(to_np(outs["topk_idx"]), idx)
    pred = O.predict_partition(c.ids, c.conf, c.emap, cfg.P)
    perm, off = O.token_shuffle(pred, cfg.P)
    eo, pr, rt = O.expert_dispatch(idx, cfg.E, perm)
    for k, ref in (("pred_part", pred), ("shuf_perm", perm), ("part_off", off),
                   ("expert_off", eo), ("pair_row", pr), ("row_token", rt)):
        assert np.array_equal(to_np(outs[k]), ref), k
    assert np.array_equal(to_np(outs["lar"]).astype(np.uint64),
                          O.lar_counts(idx, c.emap, cfg.P, cfg.H, src_part=pred))
    # values against the oracle's own routing, tokens near a routing tie excluded; at large
    # T a sample plus the tokens of the first and last row of every 64-row block of every
    # expert segment and of the shared experts' rows (every tile of both GEMMs)
    if cfg.T <= 1024:
        toks = np.arange(cfg.T)
    else:
        toks = np.union1d(sample_tokens(cfg.T, 40, seed=4), rt[block_edge_rows(eo)])
        if cfg.n_shared:
            toks = np.union1d(toks, block_edge_rows([0, cfg.T]))
    own_logits = O.gate_logits(c.x_np[toks], to_np(c.w_gate))
    margin = O.selection_margin(own_logits, cfg.K, cfg.H)
    keep = margin >= MARGIN
    assert keep.mean() > 0.8
    own_idx = np.zeros((cfg.T, cfg.K), np.int64)
    own_w = np.zeros((cfg.T, cfg.K))
    own_idx[toks] = O.topk_select(own_logits, cfg.K, cfg.H)
    own_w[toks] = O.gate_weights(own_logits, own_idx[toks])
    ref = c.oracle_tokens(toks[keep], own_idx, own_w)
    got = to_np(y)[toks[keep]].astype(np.float64)
    err = rel_err_rows(got, ref)
    fro = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    print(f"\nlayer_forward {name} T={cfg.T}: checked {int(keep.sum())} of {len(toks)} sampled "
          f"tokens ({int((~keep).sum())} excluded, margin < {MARGIN}); max row rel "
          f"{err.max():.2e}, global Frobenius rel {fro:.2e}")
    assert err.max() <= VALUE_TOL, err.max()
    assert fro <= VALUE_TOL, fro


def test_layer_forward_host_buffers():
    c = get_case("tiny_fp32", None)
    cfg = c.cfg
    desc = smoe.desc_from_config(cfg)
    ws = smoe.workspace(desc)
    W = smoe.layer_weights(c.w_gate, c.w1, c.w3, c.w2, c.conf_d, c.emap_d)
    y_dev = torch.empty_like(c.x)
    smoe.smoe_layer_forward(desc, W, smoe.layer_io(c.x, c.ids_d, y_dev), ws)
    xh = c.x.cpu().pin_memory()
    ih = torch.as_tensor(c.ids).pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    smoe.smoe_layer_forward_host(desc, W, xh, ih, yh, ws)
    torch.cuda.synchronize()
    assert torch.equal(yh, y_dev.cpu())


@pytest.mark.parametrize("name,T", [("qwen3_foe", 3001), ("dsv2_prefill", 1537), ("mixtral", 1001),
                                    ("qwen3_foe", None)],
                         ids=["qwen3-T3001", "dsv2-T1537-shared", "mixtral-T1001", "qwen3-full-two-sm"])
def test_skip_shuffle_is_lossless(name, T):
    """Dispatching without the shuffle gives the same output, bit for bit (the shuffle only
    moves data: the pages call s-MoE lossless): through the one-read row pass for x_shuf
    and the dispatched rows (the first three), and through the up GEMM's own row copy
    on two-SM tiles (the full Qwen3-shaped layer)."""
    c = get_case(name, T)
    cfg = c.cfg
    desc = smoe.desc_from_config(cfg)
    ws = smoe.workspace(desc)
    W = smoe.layer_weights(c.w_gate, c.w1, c.w3, c.w2, c.conf_d, c.emap_d)
    y1, y2 = torch.empty_like(c.x), torch.empty_like(c.x)
    smoe.smoe_layer_forward(desc, W, smoe.layer_io(c.x, c.ids_d, y1), ws)
    smoe.smoe_layer_forward(desc, W, smoe.layer_io(c.x, c.ids_d, y2, skip_shuffle=1), ws)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("T", [3001, None])
def test_prefetch_predict(T):
    c = get_case("qwen3_foe", T)
    cfg = c.cfg
    desc = smoe.desc_from_config(cfg)
    ws = smoe.workspace(desc)
    r, wgn, gamma, beta = synth.predictor_inputs(cfg, "cuda")
    wgn_l = wgn.to(cfg.torch_dtype)
    d_l = synth.round_bf16(torch.randn(cfg.d, device="cuda", generator=torch.Generator(
        device="cuda").manual_seed(11)) * 0.3)
    W = smoe.layer_weights(c.w_gate, c.w1, c.w3, c.w2, c.conf_d, c.emap_d)
    y = torch.empty_like(c.x)
    smoe.smoe_layer_forward(desc, W, smoe.layer_io(c.x, c.ids_d, y), ws)
    lq, ls = f32(cfg.T, cfg.E), f32(cfg.T, cfg.E)
    pi, ti = i32(cfg.T, cfg.K), i32(cfg.T, cfg.K)
    hits = torch.empty(1, dtype=torch.int64, device="cuda")
    smoe.smoe_prefetch_predict(desc, r, d_l, y, gamma, beta, wgn_l, pi, ti, hits, ws,
                               logits_q=lq, logits_s=ls)
    smoe.smoe_get_status(ws)
    torch.cuda.synchronize()
    Lq, Ls = to_np(lq), to_np(ls)
    rp, rtru = O.topk_select(Lq, cfg.K, cfg.H), O.topk_select(Ls, cfg.K, cfg.H)
    assert np.array_equal(to_np(pi), rp) and np.array_equal(to_np(ti), rtru)
    assert int(to_np(hits)[0]) == O.hit_count(rp, rtru)
    toks = sample_tokens(cfg.T, 64, seed=5)
    ref = O.prefetch_predict(to_np(r)[toks], to_np(d_l), to_np(y)[toks], to_np(gamma),
                             to_np(beta), to_np(wgn_l), cfg.K, cfg.H)
    assert rel_err_rows(Lq[toks], ref["logits_q"]).max() <= VALUE_TOL
    assert rel_err_rows(Ls[toks], ref["logits_s"]).max() <= VALUE_TOL
    # y rows equal to the default vector: every prediction is a hit
    y_eq = d_l.to(cfg.torch_dtype).expand(cfg.T, cfg.d).contiguous()
    smoe.smoe_prefetch_predict(desc, r, d_l, y_eq, gamma, beta, wgn_l, pi, ti, hits, ws)
    torch.cuda.synchronize()
    assert int(to_np(hits)[0]) == cfg.T * cfg.K


def test_out_of_range_data_is_reported_and_skipped():
    c = get_case("tiny_fp32", None)
    cfg = c.cfg
    desc = smoe.desc_from_config(cfg)
    ws = smoe.workspace(desc)
    bad = c.ids_d.clone()
    bad[5] = cfg.vocab + 3
    pred, perm, off = i32(cfg.T), i32(cfg.T), i32(cfg.P + 1)
    smoe.smoe_predict_shuffle(desc, bad, c.conf_d, c.emap_d, pred, perm, off, ws)
    with pytest.raises(smoe.SmoeError) as ei:
        smoe.smoe_get_status(ws)
    assert ei.value.code == -6
    ref = O.predict_partition(c.ids, c.conf, c.emap, cfg.P)
    got = to_np(pred)
    assert got[5] == 0 and np.array_equal(np.delete(got, 5), np.delete(ref, 5))
    smoe.smoe_get_status(ws)          # cleared
    idx = i32(cfg.T, cfg.K)
    idx.fill_(1)
    idx[3, 1] = cfg.E + 10
    eo, pr, rt = i32(cfg.E + 1), i32(cfg.T, cfg.K), i32(cfg.T * cfg.K)
    smoe.smoe_dispatch(desc, idx, eo, pr, rt, ws)
    with pytest.raises(smoe.SmoeError):
        smoe.smoe_get_status(ws)


def test_empty_batch():
    desc = smoe.make_desc(0, 128, 8, 2, 1, 256, 0, 2, 512, "f32")
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    ws_n = smoe.workspace_size(desc)
    ws = torch.zeros(max(ws_n, 256), dtype=torch.uint8, device="cuda")
    off = torch.full((3,), 7, dtype=torch.int32, device="cuda")
    e = torch.empty(0, dtype=torch.int32, device="cuda")
    conf = torch.zeros(512, 8, device="cuda")
    emap = torch.zeros(8, dtype=torch.int32, device="cuda")
    smoe.smoe_predict_shuffle(desc, conf, conf, emap, conf, conf, off, ws)
    torch.cuda.synchronize()
    assert to_np(off).tolist() == [0, 0, 0]
    del e


@pytest.mark.parametrize("T,E,K,S,d,F", [(2500, 8, 2, 0, 256, 384), (1537, 4, 2, 1, 512, 256),
                                         (4099, 16, 2, 0, 128, 640)])
def test_expert_ffn_two_sm_tiles_ragged(T, E, K, S, d, F):
    """Shapes with at least 256 rows per expert take the two-SM tiles; ragged expert
    segments, a partial last n-tile (F = 640, 384) and a shared expert."""
    assert T * K >= 256 * E
    g = torch.Generator(device="cuda").manual_seed(T + E)
    x = (torch.randn(T, d, generator=g, device="cuda")).to(torch.bfloat16)
    w1 = (torch.randn(E + S, F, d, generator=g, device="cuda") / d ** 0.5).to(torch.bfloat16)
    w3 = (torch.randn(E + S, F, d, generator=g, device="cuda") / d ** 0.5).to(torch.bfloat16)
    w2 = (torch.randn(E + S, d, F, generator=g, device="cuda") / F ** 0.5).to(torch.bfloat16)
    logits = torch.randn(T, E, generator=g, device="cuda") * 2
    desc = smoe.make_desc(T, d, E, K, 1, F, S, 2, 100, "bf16")
    ws = smoe.workspace(desc)
    idx, w = i32(T, K), f32(T, K)
    smoe.smoe_route(desc, None, None, idx, w, logits_in=logits, ws=ws)
    eo, pr, rt = i32(E + 1), i32(T, K), i32(T * K)
    xd = torch.empty(T * K, d, dtype=torch.bfloat16, device="cuda")
    smoe.smoe_dispatch(desc, idx, eo, pr, rt, ws, x_src=x, x_disp=xd)
    yd = torch.empty_like(xd)
    ysh = torch.empty(S, T, d, dtype=torch.bfloat16, device="cuda") if S else None
    smoe.smoe_expert_ffn(desc, xd, eo, w1, w3, w2, yd, ws, x=x, y_shared=ysh)
    smoe.smoe_get_status(ws)
    torch.cuda.synchronize()
    eo_n, rt_n = to_np(eo), to_np(rt)
    xn = to_np(x).astype(np.float64)
    W = [tuple(to_np(m[e]).astype(np.float64) for m in (w1, w3, w2)) for e in range(E + S)]
    ref = np.zeros((T * K, d))
    for e in range(E):
        lo, hi = eo_n[e], eo_n[e + 1]
        ref[lo:hi] = O.swiglu_ffn(xn[rt_n[lo:hi]], *W[e])
    assert rel_err_rows(to_np(yd), ref).max() <= VALUE_TOL
    for j in range(S):
        assert rel_err_rows(to_np(ysh[j]), O.swiglu_ffn(xn, *W[E + j])).max() <= VALUE_TOL


@pytest.mark.parametrize("d,F", [(384, 704), (256, 256)])
def test_expert_ffn_two_sm_tail_tiles(d, F):
    """Two-SM tiles end a group with a swapped tile (weight rows as the MMA's 256 rows, the
    group's last tokens as its N = 32 .. 192 columns) when its last rows fit in 192 and
    with a full 256-row tile otherwise. Expert segments of 64, 300, 450, 0, 129, 128, 513
    and 257 rows hit every case (a group that is only a swapped tile, swapped tails of 44,
    1 and 1 rows, a 128-row swapped group, a 129-row group whose N = 160 tokens come
    through the 128-row box, a 194-row M = 256 tail, an empty group), and the shared
    expert's 1100 rows end in a 76-row swapped tail; F = 704 and d = 384 leave half-valid
    last n-tiles in the up and the down GEMM."""
    counts = [64, 300, 450, 0, 129, 128, 513, 257]
    E, K, S, T = len(counts), 2, 1, 1100
    assert T * K >= 256 * E and sum(counts) <= T * K
    g = torch.Generator(device="cuda").manual_seed(d + F)
    x = torch.randn(T, d, generator=g, device="cuda").to(torch.bfloat16)
    xd = torch.randn(T * K, d, generator=g, device="cuda").to(torch.bfloat16)
    w1 = (torch.randn(E + S, F, d, generator=g, device="cuda") / d ** 0.5).to(torch.bfloat16)
    w3 = (torch.randn(E + S, F, d, generator=g, device="cuda") / d ** 0.5).to(torch.bfloat16)
    w2 = (torch.randn(E + S, d, F, generator=g, device="cuda") / F ** 0.5).to(torch.bfloat16)
    eo_n = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    eo = torch.as_tensor(eo_n, device="cuda")
    desc = smoe.make_desc(T, d, E, K, 1, F, S, 2, 100, "bf16")
    ws = smoe.workspace(desc)
    yd = torch.full_like(xd, 7.0)
    ysh = torch.empty(S, T, d, dtype=torch.bfloat16, device="cuda")
    smoe.smoe_expert_ffn(desc, xd, eo, w1, w3, w2, yd, ws, x=x, y_shared=ysh)
    smoe.smoe_get_status(ws)
    torch.cuda.synchronize()
    xdn, xn = to_np(xd).astype(np.float64), to_np(x).astype(np.float64)
    W = [tuple(to_np(m[e]).astype(np.float64) for m in (w1, w3, w2)) for e in range(E + S)]
    y = to_np(yd)
    for e in range(E):
        lo, hi = eo_n[e], eo_n[e + 1]
        if hi > lo:
            assert rel_err_rows(y[lo:hi], O.swiglu_ffn(xdn[lo:hi], *W[e])).max() <= VALUE_TOL, e
    assert (y[eo_n[-1]:] == 7.0).all()   # rows past the last group are not written
    assert rel_err_rows(to_np(ysh[0]), O.swiglu_ffn(xn, *W[E])).max() <= VALUE_TOL


@pytest.mark.parametrize("counts,S,T", [
    ([300] * 32, 0, 4800),                       # every group ends in a 44-row tail
    ([512] * 8, 0, 2048),                        # no tail: two-SM tiles move to the other kernel
    ([1, 700, 0, 256, 255, 1000, 129, 3, 2000, 44] * 3, 1, 13000)],
    ids=["all-tails", "no-tails", "ragged-shared"])
def test_expert_ffn_two_sm_tail_mixes(counts, S, T):
    """Two-SM tiles on row mixes at the extremes: every group ending in a 44-row swapped
    tail, no tail at all (whole 256-row tiles only), and ragged groups (1, 3 and 44 rows,
    129 and 188-row swapped remainders, 255-, 232- and 208-row M = 256 ones, empty groups,
    multiples of 256) with a shared expert. Every row equals the oracle's expert FFN; rows
    past the last group are not written."""
    d, F, K = 256, 256, 2
    E = len(counts)
    assert T * K >= 256 * E and sum(counts) <= T * K
    g = torch.Generator(device="cuda").manual_seed(E + S)
    x = torch.randn(T, d, generator=g, device="cuda").to(torch.bfloat16)
    xd = torch.randn(T * K, d, generator=g, device="cuda").to(torch.bfloat16)
    w1 = (torch.randn(E + S, F, d, generator=g, device="cuda") / d ** 0.5).to(torch.bfloat16)
    w3 = (torch.randn(E + S, F, d, generator=g, device="cuda") / d ** 0.5).to(torch.bfloat16)
    w2 = (torch.randn(E + S, d, F, generator=g, device="cuda") / F ** 0.5).to(torch.bfloat16)
    eo_n = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    eo = torch.as_tensor(eo_n, device="cuda")
    desc = smoe.make_desc(T, d, E, K, 1, F, S, 2, 100, "bf16")
    ws = smoe.workspace(desc)
    yd = torch.full_like(xd, 7.0)
    ysh = torch.empty(S, T, d, dtype=torch.bfloat16, device="cuda") if S else None
    smoe.smoe_expert_ffn(desc, xd, eo, w1, w3, w2, yd, ws, x=x, y_shared=ysh)
    smoe.smoe_get_status(ws)
    torch.cuda.synchronize()
    xdn, xn = to_np(xd).astype(np.float64), to_np(x).astype(np.float64)
    W = [tuple(to_np(m[e]).astype(np.float64) for m in (w1, w3, w2)) for e in range(E + S)]
    y = to_np(yd)
    ref = np.zeros_like(xdn)
    for e in range(E):
        lo, hi = eo_n[e], eo_n[e + 1]
        ref[lo:hi] = O.swiglu_ffn(xdn[lo:hi], *W[e])
    n = eo_n[-1]
    assert rel_err_rows(y[:n], ref[:n]).max() <= VALUE_TOL
    assert (y[n:] == 7.0).all()
    for j in range(S):
        assert rel_err_rows(to_np(ysh[j]), O.swiglu_ffn(xn, *W[E + j])).max() <= VALUE_TOL


@pytest.mark.parametrize("seed", range(6))
def test_expert_ffn_random_row_mixes(seed):
    """Two-SM expert FFN on seeded random row counts (a skewed draw with empty and 1-row
    groups, remainders on both sides of 128 and 192, a shared expert on odd seeds),
    against the oracle's expert FFN row by row."""
    rng = np.random.default_rng(1000 + seed)
    E, K, d, F = 16, 2, 256, 320
    counts = rng.choice([0, 1, 37, 129, 160, 192, 193, 255, 256, 300, 449, 520, 700],
                        size=E).astype(np.int64)
    S = seed % 2
    T = max(int(counts.sum()) // K + 1, 256 * E // K)   # two-SM tiles: T K >= 256 E
    assert T * K >= 256 * E and counts.sum() <= T * K
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = torch.randn(T, d, generator=g, device="cuda").to(torch.bfloat16)
    xd = torch.randn(T * K, d, generator=g, device="cuda").to(torch.bfloat16)
    w1 = (torch.randn(E + S, F, d, generator=g, device="cuda") / d ** 0.5).to(torch.bfloat16)
    w3 = (torch.randn(E + S, F, d, generator=g, device="cuda") / d ** 0.5).to(torch.bfloat16)
    w2 = (torch.randn(E + S, d, F, generator=g, device="cuda") / F ** 0.5).to(torch.bfloat16)
    eo_n = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    desc = smoe.make_desc(T, d, E, K, 1, F, S, 2, 100, "bf16")
    ws = smoe.workspace(desc)
    yd = torch.full_like(xd, 7.0)
    ysh = torch.empty(S, T, d, dtype=torch.bfloat16, device="cuda") if S else None
    smoe.smoe_expert_ffn(desc, xd, torch.as_tensor(eo_n, device="cuda"), w1, w3, w2, yd, ws,
                         x=x, y_shared=ysh)
    smoe.smoe_get_status(ws)
    torch.cuda.synchronize()
    xdn, xn = to_np(xd).astype(np.float64), to_np(x).astype(np.float64)
    W = [tuple(to_np(m[e]).astype(np.float64) for m in (w1, w3, w2)) for e in range(E + S)]
    y = to_np(yd)
    n = eo_n[-1]
    ref = np.zeros((n, d))
    for e in range(E):
        lo, hi = eo_n[e], eo_n[e + 1]
        if hi > lo:
            ref[lo:hi] = O.swiglu_ffn(xdn[lo:hi], *W[e])
    if n:
        assert rel_err_rows(y[:n], ref).max() <= VALUE_TOL
    assert (y[n:] == 7.0).all()
    for j in range(S):
        assert rel_err_rows(to_np(ysh[j]), O.swiglu_ffn(xn, *W[E + j])).max() <= VALUE_TOL


@pytest.mark.parametrize("name,T", [("tiny_fp32", None), ("dsv2_prefill", 1537), ("qwen3_foe", 3001),
                                    ("dsv2_prefill", None)],
                         ids=["tiny", "dsv2-T1537", "qwen3-T3001", "dsv2-full"])
def test_inter_layer_predictor(name, T):
    """Token clusters from a previous layer's routes and the more-confident-of-C_p-and-A
    prediction, bit-exact against the oracle, with table A profiled by the oracle."""
    c = get_case(name, T)
    cfg = c.cfg
    desc = smoe.desc_from_config(cfg)
    ws = smoe.workspace(desc)
    wprev = synth.previous_layer_gate(cfg, "cuda")
    # previous layer's routes of the measured batch (GPU) and cluster per token
    lg, idx, w = f32(cfg.T, cfg.E), i32(cfg.T, cfg.K), f32(cfg.T, cfg.K)
    smoe.smoe_route(desc, c.x, wprev, idx, w, logits_out=lg, ws=ws)
    clus = i32(cfg.T)
    smoe.smoe_token_cluster(desc, idx, c.emap_d, clus, ws)
    smoe.smoe_get_status(ws)
    prev = O.token_cluster(O.topk_select(to_np(lg), cfg.K, cfg.H), c.emap, cfg.P)
    assert np.array_equal(to_np(clus), prev)
    # table A from the profile batch, both layers routed by the oracle
    _, px = synth.token_batch(cfg, c.emb, "profile", min(cfg.profile_tokens, 8192), "cuda")
    pxn = to_np(px.to(cfg.torch_dtype))
    _, pidx_prev, _ = O.route(pxn, to_np(wprev), cfg.K, cfg.H)
    table = O.markov_table(O.token_cluster(pidx_prev, c.emap, cfg.P),
                           O.token_cluster(c.profile_idx, c.emap, cfg.P), cfg.P)
    for tab in (table, np.full((cfg.P, cfg.P), 0.9, np.float32) * np.eye(cfg.P, dtype=np.float32)):
        pred, perm, off = i32(cfg.T), i32(cfg.T), i32(cfg.P + 1)
        xs = torch.empty_like(c.x)
        smoe.smoe_predict_shuffle_inter(desc, c.ids_d, c.conf_d, c.emap_d, clus,
                                        torch.as_tensor(tab, device="cuda"), pred, perm, off, ws,
                                        x=c.x, x_shuf=xs)
        smoe.smoe_get_status(ws)
        ref = O.predict_partition_inter(c.ids, c.conf, c.emap, cfg.P, cfg.K, prev, tab)
        assert np.array_equal(to_np(pred), ref)
        rp, ro = O.token_shuffle(ref, cfg.P)
        assert np.array_equal(to_np(perm), rp) and np.array_equal(to_np(off), ro)
        assert torch.equal(xs, c.x[torch.as_tensor(rp, device="cuda").long()])


@pytest.mark.parametrize("name,T", [("dsv2_prefill", 1537), ("mixtral", 1001)], ids=["dsv2", "mixtral"])
def test_moe_forward_routed(name, T):
    """The MoE body with caller-supplied routes, against the oracle's defining sum."""
    c = get_case(name, T)
    cfg = c.cfg
    desc = smoe.desc_from_config(cfg)
    ws = smoe.workspace(desc)
    rng = np.random.default_rng(41)
    L = (rng.standard_normal((cfg.T, cfg.E)) * 2).astype(np.float32)
    idx = O.topk_select(L, cfg.K, cfg.H)
    w = O.gate_weights(L, idx).astype(np.float32)
    y = torch.empty_like(c.x)
    smoe.smoe_moe_forward_routed(desc, c.x, torch.as_tensor(idx, device="cuda"),
                                 torch.as_tensor(w, device="cuda"), c.w1, c.w3, c.w2, y, ws)
    smoe.smoe_get_status(ws)
    toks = sample_tokens(cfg.T, 24, seed=6)
    ref = c.oracle_tokens(toks, idx, w.astype(np.float64))
    assert rel_err_rows(to_np(y)[toks], ref).max() <= VALUE_TOL


def test_speculative_execution_qwen3():
    """Prefetch predictor -> speculative execution of the predicted experts on the next
    layer's input s, against the oracle on the same s rows and logits."""
    c = get_case("qwen3_foe", 3001)
    cfg = c.cfg
    desc = smoe.desc_from_config(cfg)
    ws = smoe.workspace(desc)
    r, wgn, gamma, beta = synth.predictor_inputs(cfg, "cuda")
    wgn_l = wgn.to(cfg.torch_dtype)
    d_l = synth.round_bf16(torch.randn(cfg.d, device="cuda", generator=torch.Generator(
        device="cuda").manual_seed(12)) * 0.3)
    W = smoe.layer_weights(c.w_gate, c.w1, c.w3, c.w2, c.conf_d, c.emap_d)
    y = torch.empty_like(c.x)
    smoe.smoe_layer_forward(desc, W, smoe.layer_io(c.x, c.ids_d, y), ws)
    lq, ls = f32(cfg.T, cfg.E), f32(cfg.T, cfg.E)
    pi, ti = i32(cfg.T, cfg.K), i32(cfg.T, cfg.K)
    hits = torch.empty(1, dtype=torch.int64, device="cuda")
    qs = torch.empty(2, cfg.T, cfg.d, dtype=cfg.torch_dtype, device="cuda")
    smoe.smoe_prefetch_predict(desc, r, d_l, y, gamma, beta, wgn_l, pi, ti, hits, ws,
                               logits_q=lq, logits_s=ls, qs_out=qs)
    pidx, pw, tidx, tw = i32(cfg.T, cfg.K), f32(cfg.T, cfg.K), i32(cfg.T, cfg.K), f32(cfg.T, cfg.K)
    smoe.smoe_route(desc, None, None, pidx, pw, logits_in=lq)
    smoe.smoe_route(desc, None, None, tidx, tw, logits_in=ls)
    assert torch.equal(pidx, pi) and torch.equal(tidx, ti)
    s_rows = qs[1].contiguous()
    y_spec, y_true = torch.empty_like(c.x), torch.empty_like(c.x)
    smoe.smoe_moe_forward_routed(desc, s_rows, pidx, pw, c.w1, c.w3, c.w2, y_spec, ws)
    smoe.smoe_moe_forward_routed(desc, s_rows, tidx, tw, c.w1, c.w3, c.w2, y_true, ws)
    smoe.smoe_get_status(ws)
    torch.cuda.synchronize()
    toks = sample_tokens(cfg.T, 24, seed=7)
    Lq, Ls = to_np(lq), to_np(ls)
    p_idx, t_idx = O.topk_select(Lq, cfg.K, cfg.H), O.topk_select(Ls, cfg.K, cfg.H)
    p_w, t_w = O.gate_weights(Lq, p_idx), O.gate_weights(Ls, t_idx)
    sn = to_np(s_rows).astype(np.float64)
    w1n = [to_np(c.w1[e]).astype(np.float64) for e in range(cfg.E)]
    w3n = [to_np(c.w3[e]).astype(np.float64) for e in range(cfg.E)]
    w2n = [to_np(c.w2[e]).astype(np.float64) for e in range(cfg.E)]
    ref_spec, ref_true, ref_dev = O.speculative_execution(
        sn[toks], p_idx[toks], p_w[toks], t_idx[toks], t_w[toks], np.stack(w1n), np.stack(w3n),
        np.stack(w2n))
    assert rel_err_rows(to_np(y_spec)[toks], ref_spec).max() <= VALUE_TOL
    assert rel_err_rows(to_np(y_true)[toks], ref_true).max() <= VALUE_TOL
    ys, yt = to_np(y_spec)[toks].astype(np.float64), to_np(y_true)[toks].astype(np.float64)
    gpu_dev = np.linalg.norm(ys - yt) / np.linalg.norm(yt)
    assert abs(gpu_dev - ref_dev) <= 0.02 + 0.02 * ref_dev


LIMIT_SHAPES = [
    # T, d, E, K, H, F, S, P, vocab, dtype
    (300, 64, 512, 32, 1, 64, 8, 32, 1000, "bf16"),   # every size limit at once
    (129, 8, 16, 16, 16, 8, 1, 3, 50, "f32"),         # d = F = 8: one partial k-block
    (1, 128, 8, 2, 1, 256, 0, 2, 10, "bf16"),          # a single token
    (2048, 256, 64, 8, 8, 128, 2, 8, 700, "bf16"),     # grouped routing with shared experts
    (4096, 128, 8, 2, 2, 384, 1, 4, 300, "bf16"),      # two-SM tiles with a shared expert
]


@pytest.mark.parametrize("T,d,E,K,H,F,S,P,V,dt", LIMIT_SHAPES,
                         ids=[f"T{s[0]}-d{s[1]}-E{s[2]}-K{s[3]}-H{s[4]}-S{s[6]}-P{s[7]}-{s[9]}"
                              for s in LIMIT_SHAPES])
def test_layer_forward_at_limits(T, d, E, K, H, F, S, P, V, dt):
    """The whole layer at the ABI's limits (E = 512, K = 32, P = 32, 8 shared experts),
    at the smallest d and F, at T = 1 and with grouped routing: indices bit-exact given the
    GPU's logits, values against the oracle's own routing."""
    rng = np.random.default_rng(T + E + K)
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    def t(a):
        return torch.as_tensor(np.asarray(a, np.float32)).to(tdt).cuda().contiguous()
    x = t(rng.standard_normal((T, d)))
    wg = t(rng.standard_normal((E, d)) / np.sqrt(d))
    w1 = t(rng.standard_normal((E + S, F, d)) / np.sqrt(d))
    w3 = t(rng.standard_normal((E + S, F, d)) / np.sqrt(d))
    w2 = t(rng.standard_normal((E + S, d, F)) / np.sqrt(F))
    conf = rng.random((V, E)).astype(np.float32)
    conf = (conf / conf.sum(1, keepdims=True) * K).astype(np.float32)
    emap = rng.integers(0, P, size=E).astype(np.int32)
    ids = rng.integers(0, V, size=T).astype(np.int32)
    desc = smoe.make_desc(T, d, E, K, H, F, S, P, V, dt)
    ws = smoe.workspace(desc)
    outs = dict(logits=f32(T, E), topk_idx=i32(T, K), topk_w=f32(T, K), pred_part=i32(T),
                shuf_perm=i32(T), part_off=i32(P + 1), expert_off=i32(E + 1),
                pair_row=i32(T, K), row_token=i32(T * K),
                lar=torch.empty(4, dtype=torch.int64, device="cuda"))
    y = torch.empty_like(x)
    conf_d = torch.as_tensor(conf, device="cuda")
    emap_d = torch.as_tensor(emap, device="cuda")
    ids_d = torch.as_tensor(ids, device="cuda")
    W = smoe.layer_weights(wg, w1, w3, w2, conf_d, emap_d)
    smoe.smoe_layer_forward(desc, W, smoe.layer_io(x, ids_d, y, **outs), ws)
    smoe.smoe_get_status(ws)
    torch.cuda.synchronize()
    xn, wgn = to_np(x).astype(np.float64), to_np(wg).astype(np.float64)
    w1n, w3n, w2n = (to_np(m).astype(np.float64) for m in (w1, w3, w2))
    ref = O.layer_forward(xn, ids, wgn, w1n, w3n, w2n, conf, emap, K=K, H=H, P=P, n_shared=S,
                          logits=to_np(outs["logits"]))
    for k, name in (("topk_idx", "idx"), ("pred_part", "pred"), ("shuf_perm", "shuf_perm"),
                    ("part_off", "part_off"), ("expert_off", "expert_off"),
                    ("pair_row", "pair_row"), ("row_token", "row_token")):
        assert np.array_equal(to_np(outs[k]), ref[name]), k
    assert np.array_equal(to_np(outs["lar"]).astype(np.uint64), ref["lar"])
    own = O.layer_forward(xn, ids, wgn, w1n, w3n, w2n, conf, emap, K=K, H=H, P=P, n_shared=S)
    keep = O.selection_margin(own["logits"], K, H) >= MARGIN
    assert keep.mean() > 0.5
    err = rel_err_rows(to_np(y)[keep], own["y"][keep])
    assert err.max() <= VALUE_TOL, err.max()


@pytest.mark.parametrize("T,E,K,S,d,F,skew", [(3000, 8, 2, 0, 200, 328, True),
                                               (2600, 8, 2, 1, 200, 328, False),
                                               (700, 16, 4, 2, 136, 72, True)])
def test_expert_ffn_skewed_and_odd_sizes(T, E, K, S, d, F, skew):
    """Expert FFN + combine with d and F not multiples of 64 (partial k-blocks and a
    partial last n-tile, two-SM and single-SM tiles) and with every token routed to the
    same K experts (the other experts get no rows)."""
    g = torch.Generator(device="cuda").manual_seed(T + d)
    x = torch.randn(T, d, generator=g, device="cuda").to(torch.bfloat16)
    w1 = (torch.randn(E + S, F, d, generator=g, device="cuda") / d ** 0.5).to(torch.bfloat16)
    w3 = (torch.randn(E + S, F, d, generator=g, device="cuda") / d ** 0.5).to(torch.bfloat16)
    w2 = (torch.randn(E + S, d, F, generator=g, device="cuda") / F ** 0.5).to(torch.bfloat16)
    logits = torch.randn(T, E, generator=g, device="cuda")
    if skew:
        logits[:, :K] += 100.0        # experts 0..K-1 win for every token
    desc = smoe.make_desc(T, d, E, K, 1, F, S, 2, 100, "bf16")
    ws = smoe.workspace(desc)
    idx, w = i32(T, K), f32(T, K)
    smoe.smoe_route(desc, None, None, idx, w, logits_in=logits, ws=ws)
    eo, pr, rt = i32(E + 1), i32(T, K), i32(T * K)
    xd = torch.empty(T * K, d, dtype=torch.bfloat16, device="cuda")
    smoe.smoe_dispatch(desc, idx, eo, pr, rt, ws, x_src=x, x_disp=xd)
    yd = torch.empty_like(xd)
    ysh = torch.empty(S, T, d, dtype=torch.bfloat16, device="cuda") if S else None
    smoe.smoe_expert_ffn(desc, xd, eo, w1, w3, w2, yd, ws, x=x, y_shared=ysh)
    y = torch.empty_like(x)
    smoe.smoe_combine(desc, yd, pr, w, y, ws, y_shared=ysh)
    smoe.smoe_get_status(ws)
    torch.cuda.synchronize()
    if skew:
        assert (np.diff(to_np(eo))[K:] == 0).all()
    xn = to_np(x).astype(np.float64)
    W = [tuple(to_np(m[e]).astype(np.float64) for m in (w1, w3, w2)) for e in range(E + S)]
    ref = O.moe_output(xn, to_np(idx), to_np(w).astype(np.float64),
                       np.stack([a for a, _, _ in W]), np.stack([b for _, b, _ in W]),
                       np.stack([c for _, _, c in W]), S)
    assert rel_err_rows(to_np(y), ref).max() <= VALUE_TOL


@pytest.mark.parametrize("T,d,E,K,H,dt", [(200, 64, 512, 32, 1, "bf16"), (300, 8, 16, 16, 16, "f32"),
                                          (64, 8192, 8, 2, 1, "bf16"), (1, 128, 8, 2, 1, "bf16")])
def test_prefetch_predict_at_limits(T, d, E, K, H, dt):
    """The prefetch predictor at E = 512 / K = 32, at d = 8 and d = 8192 (its largest
    row), and for a single token: routes and hits bit-exact given the GPU's logits,
    logits against the oracle's LayerNorm + gate."""
    rng = np.random.default_rng(d + E)
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    r = torch.as_tensor(rng.standard_normal((T, d)).astype(np.float32), device="cuda")
    d_l = torch.as_tensor((0.3 * rng.standard_normal(d)).astype(np.float32), device="cuda")
    y = torch.as_tensor(rng.standard_normal((T, d)).astype(np.float32)).to(tdt).cuda()
    gamma = torch.as_tensor((1 + 0.1 * rng.standard_normal(d)).astype(np.float32), device="cuda")
    beta = torch.as_tensor((0.1 * rng.standard_normal(d)).astype(np.float32), device="cuda")
    wgn = torch.as_tensor((rng.standard_normal((E, d)) / np.sqrt(d)).astype(np.float32)).to(tdt).cuda()
    desc = smoe.make_desc(T, d, E, K, H, 64, 0, 2, 16, dt)
    ws = smoe.workspace(desc)
    lq, ls = f32(T, E), f32(T, E)
    pi, ti = i32(T, K), i32(T, K)
    hits = torch.empty(1, dtype=torch.int64, device="cuda")
    smoe.smoe_prefetch_predict(desc, r, d_l, y, gamma, beta, wgn, pi, ti, hits, ws,
                               logits_q=lq, logits_s=ls)
    smoe.smoe_get_status(ws)
    torch.cuda.synchronize()
    Lq, Ls = to_np(lq), to_np(ls)
    rp, rtru = O.topk_select(Lq, K, H), O.topk_select(Ls, K, H)
    assert np.array_equal(to_np(pi), rp) and np.array_equal(to_np(ti), rtru)
    assert int(to_np(hits)[0]) == O.hit_count(rp, rtru)
    ref = O.prefetch_predict(to_np(r), to_np(d_l), to_np(y).astype(np.float64), to_np(gamma),
                             to_np(beta), to_np(wgn).astype(np.float64), K, H)
    assert rel_err_rows(Lq, ref["logits_q"]).max() <= VALUE_TOL
    assert rel_err_rows(Ls, ref["logits_s"]).max() <= VALUE_TOL


def test_moe_forward_routed_at_limits():
    """Caller-given routes at E = 512, K = 32 with 8 shared experts."""
    T, d, E, K, S, F = 300, 64, 512, 32, 8, 64
    rng = np.random.default_rng(9)
    def t(a):
        return torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16).cuda().contiguous()
    x = t(rng.standard_normal((T, d)))
    w1 = t(rng.standard_normal((E + S, F, d)) / np.sqrt(d))
    w3 = t(rng.standard_normal((E + S, F, d)) / np.sqrt(d))
    w2 = t(rng.standard_normal((E + S, d, F)) / np.sqrt(F))
    idx_n = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    w_n = rng.random((T, K)).astype(np.float32)
    desc = smoe.make_desc(T, d, E, K, 1, F, S, 2, 16, "bf16")
    ws = smoe.workspace(desc)
    y = torch.empty_like(x)
    smoe.smoe_moe_forward_routed(desc, x, torch.as_tensor(idx_n, device="cuda"),
                                 torch.as_tensor(w_n, device="cuda"), w1, w3, w2, y, ws)
    smoe.smoe_get_status(ws)
    torch.cuda.synchronize()
    ref = O.moe_output(to_np(x).astype(np.float64), idx_n, w_n.astype(np.float64),
                       to_np(w1).astype(np.float64), to_np(w3).astype(np.float64),
                       to_np(w2).astype(np.float64), S)
    assert rel_err_rows(to_np(y), ref).max() <= VALUE_TOL


def test_device_timeout_is_reported_and_the_context_survives():
    """A bounded device wait that can never complete gives up after its limit, the
    status word reports SMOE_ERR_DEVICE_TIMEOUT, and the next launches run normally."""
    c = get_case("tiny_fp32", None)
    cfg = c.cfg
    desc = smoe.desc_from_config(cfg)
    ws = smoe.workspace(desc)
    smoe.smoe_selftest_device_timeout(ws)
    with pytest.raises(smoe.SmoeError) as ei:
        smoe.smoe_get_status(ws)
    assert ei.value.code == -7
    smoe.smoe_get_status(ws)                       # cleared
    logits, idx, w = run_route(c, desc, ws)
    smoe.smoe_get_status(ws)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(idx), O.topk_select(to_np(logits), cfg.K, cfg.H))


@pytest.mark.parametrize("name,T", [("tiny_fp32", 37), ("dsv2_prefill", 1537), ("qwen3_foe", 3001)],
                         ids=["tiny-T37", "dsv2-T1537", "qwen3-T3001"])
def test_no_write_past_any_buffer(name, T):
    """Canary words after every output buffer and after the workspace: a layer forward
    (and the prefetch predictor on the Qwen3 shape) writes nothing past the sizes the
    header documents."""
    c = get_case(name, T)
    cfg = c.cfg
    desc = smoe.desc_from_config(cfg)
    CAN = 4096                                   # bytes of canary after each buffer
    MAGIC = 0x5A

    def guarded(nbytes):
        buf = torch.full((nbytes + CAN,), MAGIC, dtype=torch.uint8, device="cuda")
        return buf

    def view(buf, shape, dtype):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        return buf[:n].view(dtype).view(*shape)

    ws_n = smoe.workspace_size(desc)
    ws_buf = guarded(ws_n)
    ws_buf[:256].zero_()
    ws = ws_buf[:ws_n]
    TK = cfg.T * cfg.K
    i4, f4 = torch.int32, torch.float32
    shapes = dict(logits=((cfg.T, cfg.E), f4), topk_idx=((cfg.T, cfg.K), i4),
                  topk_w=((cfg.T, cfg.K), f4), pred_part=((cfg.T,), i4), shuf_perm=((cfg.T,), i4),
                  part_off=((cfg.P + 1,), i4), expert_off=((cfg.E + 1,), i4),
                  pair_row=((cfg.T, cfg.K), i4), row_token=((TK,), i4), lar=((4,), torch.int64))
    bufs, outs = {}, {}
    for k, (shape, dt) in shapes.items():
        nbytes = int(np.prod(shape)) * torch.empty((), dtype=dt).element_size()
        bufs[k] = guarded(nbytes)
        outs[k] = view(bufs[k], shape, dt)
    ybytes = cfg.T * cfg.d * c.x.element_size()
    bufs["y"] = guarded(ybytes)
    y = view(bufs["y"], (cfg.T, cfg.d), c.x.dtype)
    W = smoe.layer_weights(c.w_gate, c.w1, c.w3, c.w2, c.conf_d, c.emap_d)
    smoe.smoe_layer_forward(desc, W, smoe.layer_io(c.x, c.ids_d, y, **outs), ws)
    if cfg.prefetch:
        r, wgn, gamma, beta = synth.predictor_inputs(cfg, "cuda")
        d_l = torch.zeros(cfg.d, device="cuda")
        for k, shape in (("pi", (cfg.T, cfg.K)), ("ti", (cfg.T, cfg.K))):
            bufs[k] = guarded(int(np.prod(shape)) * 4)
            outs[k] = view(bufs[k], shape, i4)
        bufs["hits"] = guarded(8)
        hits = view(bufs["hits"], (1,), torch.int64)
        smoe.smoe_prefetch_predict(desc, r, d_l, y, gamma, beta, wgn.to(cfg.torch_dtype),
                                   outs["pi"], outs["ti"], hits, ws)
    smoe.smoe_get_status(ws)
    torch.cuda.synchronize()
    for k, buf in bufs.items():
        tail = buf[buf.numel() - CAN:]
        assert bool((tail == MAGIC).all()), f"write past the end of {k}"
    assert bool((ws_buf[ws_n:] == MAGIC).all()), "write past the end of the workspace"
