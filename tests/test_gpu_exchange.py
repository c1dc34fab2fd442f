"""GPU parity of the expert-parallel exchange between simulated devices ("Speculative
MoE" §1 EP dispatch/combine) and of SRS / SAG (§3.1), against the CPU oracle.

The exchange plan (send counts, receive offsets, receive row of every pair, token of
every receive row) is compared bit for bit; receive rows are pure copies and must be
identical; SRS sums R partials in fp32 and is compared within the rounding of one
store to the layer dtype; SAG is a pure permutation of rows."""
import json
import os

import numpy as np
import pytest
import torch

import oracle as O
import routing_token_shuffle_gb300 as smoe

from _cases import Case, rel_err_rows, to_np

pytestmark = pytest.mark.gpu

GOLD = os.path.join(os.path.dirname(__file__), "golden")
CASES = [("tiny_fp32", 37), ("mixtral", 1001), ("dsv2_prefill", 1537), ("dsv2_decode", None),
         ("qwen3_foe", 3001), ("dsv2_prefill", None), ("qwen3_foe", None)]
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
        _cache.clear()
        torch.cuda.empty_cache()
        _cache[key] = Case(name, "cuda", T=T)
    return _cache[key]


def i32(*shape):
    return torch.empty(*shape, dtype=torch.int32, device="cuda")


def exchange(desc, idx, emap, ws, src=None, x=None, with_rows=False):
    T, K, P = desc.T, desc.K, desc.P
    out = dict(send_counts=i32(P, P), recv_off=i32(P * P + 1), pair_recv=i32(T, K),
               recv_token=i32(T * K))
    xr = torch.empty(T * K, desc.d, dtype=x.dtype, device="cuda") if with_rows else None
    smoe.smoe_ep_exchange(desc, idx, emap, out["send_counts"], out["recv_off"],
                          out["pair_recv"], out["recv_token"], ws, src_part=src, x=x, x_recv=xr)
    smoe.smoe_get_status(ws)
    return out, xr


def check_plan(out, ref):
    names = ("send_counts", "recv_off", "pair_recv", "recv_token")
    for n, r in zip(names, ref):
        assert np.array_equal(to_np(out[n]), r), n


def test_exchange_fig2_golden():
    """The hand-worked Fig. 2-shaped exchange through the C ABI."""
    with open(os.path.join(GOLD, "ep_exchange_fig2_hand.json")) as f:
        g = json.load(f)
    desc = smoe.make_desc(8, 64, 4, 2, 1, 64, 0, 2, 16, "bf16")
    ws = smoe.workspace(desc)
    idx = torch.tensor(g["routes"], dtype=torch.int32, device="cuda")
    emap = torch.tensor(g["expert_part"], dtype=torch.int32, device="cuda")
    pred = torch.tensor(g["pred"], dtype=torch.int32, device="cuda")
    for case, src in (("sts", pred), ("contiguous", None)):
        out, _ = exchange(desc, idx, emap, ws, src=src)
        for n in ("send_counts", "recv_off", "recv_token", "pair_recv"):
            assert to_np(out[n]).tolist() == g[case][n], (case, n)


@pytest.mark.parametrize("name,T", CASES, ids=IDS)
def test_ep_exchange(name, T):
    c = get_case(name, T)
    cfg = c.cfg
    desc = smoe.desc_from_config(cfg)
    ws = smoe.workspace(desc)
    idx, w = i32(cfg.T, cfg.K), torch.empty(cfg.T, cfg.K, device="cuda")
    smoe.smoe_route(desc, c.x, c.w_gate, idx, w, ws=ws)
    pred, perm, off = i32(cfg.T), i32(cfg.T), i32(cfg.P + 1)
    smoe.smoe_predict_shuffle(desc, c.ids_d, c.conf_d, c.emap_d, pred, perm, off, ws)
    idx_np, pred_np = to_np(idx), to_np(pred)
    # s-TS sources, with the receive rows
    out, xr = exchange(desc, idx, c.emap_d, ws, src=pred, x=c.x, with_rows=True)
    ref = O.ep_exchange(idx_np, c.emap, cfg.P, pred_np)
    check_plan(out, ref)
    assert torch.equal(xr, c.x[out["recv_token"].long()])
    # the diagonal is the local-activation count of the same sources
    lar = torch.zeros(4, dtype=torch.int64, device="cuda")
    smoe.smoe_lar(desc, idx, c.emap_d, lar, ws, src_part=pred)
    assert int(np.trace(to_np(out["send_counts"]))) == int(lar[0].item())
    # contiguous split
    out, _ = exchange(desc, idx, c.emap_d, ws)
    check_plan(out, O.ep_exchange(idx_np, c.emap, cfg.P, None))
    # the return trip: combining the receive rows through pair_recv gives sum_k w_k x_t
    out, xr = exchange(desc, idx, c.emap_d, ws, src=pred, x=c.x, with_rows=True)
    y = torch.empty_like(c.x)
    smoe.smoe_combine(desc, xr, out["pair_recv"], w, y, ws)
    smoe.smoe_get_status(ws)
    want = O.combine(c.x_np[to_np(out["recv_token"])], to_np(out["pair_recv"]), to_np(w))
    tol = 1e-5 if cfg.dtype == "f32" else 8e-3
    assert rel_err_rows(to_np(y), want).max() <= tol


@pytest.mark.parametrize("T,E,K,P", [(1, 8, 2, 1), (4096, 64, 4, 32), (3001, 160, 6, 8),
                                     (257, 16, 16, 16)])
def test_ep_exchange_limits(T, E, K, P):
    """One device; 32 devices (1024 (dst, src) buckets); K = E; a ragged T."""
    g = torch.Generator(device="cuda").manual_seed(T + P)
    idx = torch.argsort(torch.rand(T, E, generator=g, device="cuda"), dim=1)[:, :K]
    idx = idx.to(torch.int32).contiguous()
    emap = torch.randint(0, P, (E,), generator=g, device="cuda", dtype=torch.int32)
    src = torch.randint(0, P, (T,), generator=g, device="cuda", dtype=torch.int32)
    desc = smoe.make_desc(T, 64, E, K, 1, 64, 0, P, 100, "bf16")
    ws = smoe.workspace(desc)
    x = torch.randn(T, 64, generator=g, device="cuda").to(torch.bfloat16)
    for s in (src, None):
        out, xr = exchange(desc, idx, emap, ws, src=s, x=x, with_rows=True)
        check_plan(out, O.ep_exchange(to_np(idx), to_np(emap), P,
                                      None if s is None else to_np(s)))
        assert torch.equal(xr, x[out["recv_token"].long()])


def test_ep_exchange_empty_and_bad_source():
    desc0 = smoe.make_desc(0, 64, 8, 2, 1, 64, 0, 4, 100, "bf16")
    ws0 = smoe.workspace(desc0)
    t = torch.zeros(16, dtype=torch.int32, device="cuda")
    sc, ro = torch.full((16,), 5, dtype=torch.int32, device="cuda"), torch.full(
        (17,), 5, dtype=torch.int32, device="cuda")
    smoe.smoe_ep_exchange(desc0, t, t, sc, ro, t, t, ws0)
    torch.cuda.synchronize()
    assert sc.cpu().tolist() == [0] * 16 and ro.cpu().tolist() == [0] * 17
    # a source device out of range is counted as device 0 and reported
    T, E, K, P = 64, 8, 2, 4
    desc = smoe.make_desc(T, 64, E, K, 1, 64, 0, P, 100, "bf16")
    ws = smoe.workspace(desc)
    idx = torch.stack([torch.arange(K, dtype=torch.int32)] * T).cuda()
    emap = torch.arange(E, dtype=torch.int32, device="cuda") % P
    src = torch.zeros(T, dtype=torch.int32, device="cuda")
    src[5] = P
    out = dict(send_counts=i32(P, P), recv_off=i32(P * P + 1), pair_recv=i32(T, K),
               recv_token=i32(T * K))
    smoe.smoe_ep_exchange(desc, idx, emap, out["send_counts"], out["recv_off"], out["pair_recv"],
                          out["recv_token"], ws, src_part=src)
    with pytest.raises(smoe.SmoeError):
        smoe.smoe_get_status(ws)
    src[5] = 0
    check_plan(out, O.ep_exchange(to_np(idx), to_np(emap), P, to_np(src)))


@pytest.mark.parametrize("dtype,T,d,R", [("bf16", 1537, 5120, 2), ("bf16", 64, 2048, 8),
                                         ("bf16", 1, 64, 1), ("f32", 1001, 128, 3),
                                         ("bf16", 4096, 4096, 4), ("f32", 37, 8, 5)])
def test_srs_and_sag(dtype, T, d, R):
    """SRS: the R partials of every token added in fp32 and written in slot order; SAG:
    slot order back to token order. Partials are seeded values of the layer dtype."""
    g = torch.Generator(device="cuda").manual_seed(T * R + d)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    parts = torch.randn(R, T, d, generator=g, device="cuda").to(tdt)
    perm = torch.randperm(T, generator=g, device="cuda").to(torch.int32)
    desc = smoe.make_desc(T, d, 8, 2, 1, 64, 0, 2, 100, dtype)
    ws = smoe.workspace(desc)
    xs = torch.empty(T, d, dtype=tdt, device="cuda")
    smoe.smoe_srs(desc, parts, perm, xs, ws)
    y = torch.empty_like(xs)
    smoe.smoe_sag(desc, xs, perm, y, ws)
    smoe.smoe_get_status(ws)
    p64 = to_np(parts).astype(np.float64)
    want = O.shuffled_reduce_scatter(p64, to_np(perm))
    # error bound per element: R fp32 additions (R 2^-24 sum_r |x_r|) and one rounding
    # of the sum to the layer dtype (unit roundoff 2^-8 for bf16, 2^-24 for fp32)
    u_store = 2.0 ** -24 if dtype == "f32" else 2.0 ** -8
    mag = np.abs(p64).sum(axis=0)[to_np(perm)]
    bound = u_store * np.abs(want) + R * 2.0 ** -24 * mag
    assert (np.abs(to_np(xs) - want) <= bound * (1 + 1e-6) + 1e-30).all()
    if R == 1:
        assert torch.equal(xs, parts[0][perm.long()])
    # SAG is the inverse permutation, bit for bit
    assert torch.equal(y[perm.long()], xs)
    back = O.shuffled_allgather(to_np(xs), to_np(perm))
    assert np.array_equal(to_np(y), back)
