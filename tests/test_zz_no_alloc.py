"""The workspace-free shuffle entry point, for callers that cannot allocate device
memory (runtimes that reserve all their device memory at start-up and forbid
allocation afterwards, hosts whose memory pool belongs to another framework). It must
return exactly what the workspace entry point returns, call after call, although all
calls share one library-held scratch array, and what the oracle's definition gives.

Kept in its own file, collected last, so a run that stops at the first failure has
already run every other test; it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def smoe():
    import __graft_entry__
    __graft_entry__.build()
    import routing_token_shuffle_gb300 as m
    assert torch.cuda.is_available()
    return m


def make_inputs(seed, T, d, E, P, V):
    g = torch.Generator(device="cuda").manual_seed(seed)
    ids = torch.randint(0, V, (T,), generator=g, device="cuda", dtype=torch.int32)
    conf = torch.rand(V, E, generator=g, device="cuda")
    conf[: V // 3] = torch.round(conf[: V // 3] * 4) / 4          # exact partition-score ties
    emap = torch.randint(0, P, (E,), generator=g, device="cuda", dtype=torch.int32)
    x = torch.randn(T, d, generator=g, device="cuda").to(torch.bfloat16)
    return ids, conf, emap, x


def run_both(smoe, desc, ids, conf, emap, x, ws):
    T, P = desc.T, desc.P
    i32 = dict(dtype=torch.int32, device="cuda")
    ref = [torch.empty(T, **i32), torch.empty(T, **i32), torch.empty(P + 1, **i32),
           torch.empty_like(x)]
    smoe.smoe_predict_shuffle(desc, ids, conf, emap, ref[0], ref[1], ref[2], ws, x=x,
                              x_shuf=ref[3])
    got = [torch.full((T,), -7, **i32), torch.full((T,), -7, **i32),
           torch.full((P + 1,), -7, **i32), torch.zeros_like(x)]
    # straight through the C ABI, no workspace argument
    rc = smoe.lib().smoe_predict_shuffle_noalloc(
        ctypes.byref(desc), ids.data_ptr(), conf.data_ptr(), emap.data_ptr(), x.data_ptr(),
        got[0].data_ptr(), got[1].data_ptr(), got[2].data_ptr(), got[3].data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert rc == 0, smoe.lib().smoe_last_error()
    torch.cuda.synchronize()
    return ref, got


def test_noalloc_matches_workspace_entry_point_twice(smoe):
    # two calls in a row with different shapes and data: nothing may leak from the first
    shapes = [(5000, 256, 64, 8, 3000), (1537, 128, 160, 5, 700)]
    for call, (T, d, E, P, V) in enumerate(shapes):
        desc = smoe.make_desc(T, d, E, 2, 1, 64, 0, P, V, "bf16")
        ws = smoe.workspace(desc)
        ids, conf, emap, x = make_inputs(100 + call, T, d, E, P, V)
        ref, got = run_both(smoe, desc, ids, conf, emap, x, ws)
        for r, g in zip(ref, got):
            assert torch.equal(r, g), f"call {call} differs from smoe_predict_shuffle"


def test_noalloc_rejects_too_many_tokens(smoe):
    desc = smoe.make_desc(1024 * 1024 + 1, 128, 8, 2, 1, 64, 0, 2, 100, "bf16")
    t = torch.zeros(16, dtype=torch.int32, device="cuda")
    rc = smoe.lib().smoe_predict_shuffle_noalloc(ctypes.byref(desc), t.data_ptr(), t.data_ptr(),
                                                 t.data_ptr(), None, t.data_ptr(), t.data_ptr(),
                                                 t.data_ptr(), None, None)
    assert rc == -2
    assert b"1048576" in smoe.lib().smoe_last_error()


def test_noalloc_at_the_token_limit(smoe):
    # T = 1048576 fills every one of the scratch's 4096 tiles, with P = 32 partitions
    T, d, E, P, V = 1024 * 1024, 8, 64, 32, 5000
    desc = smoe.make_desc(T, d, E, 2, 1, 64, 0, P, V, "bf16")
    ws = smoe.workspace(desc)
    ids, conf, emap, x = make_inputs(7, T, d, E, P, V)
    ref, got = run_both(smoe, desc, ids, conf, emap, x, ws)
    for r, g in zip(ref, got):
        assert torch.equal(r, g)
    off = ref[2].cpu().numpy()
    assert off[0] == 0 and off[-1] == T and (np.diff(off) >= 0).all()


def test_noalloc_matches_the_oracle(smoe):
    # the predicted partitions and the stable shuffle straight from their definitions
    import oracle as O
    T, d, E, P, V = 3001, 64, 160, 8, 2000
    desc = smoe.make_desc(T, d, E, 6, 1, 64, 0, P, V, "bf16")
    ids, conf, emap, x = make_inputs(11, T, d, E, P, V)
    i32 = dict(dtype=torch.int32, device="cuda")
    pred, perm, off = torch.empty(T, **i32), torch.empty(T, **i32), torch.empty(P + 1, **i32)
    xs = torch.empty_like(x)
    for _ in range(2):
        smoe.smoe_predict_shuffle_noalloc(desc, ids, conf, emap, pred, perm, off, x=x, x_shuf=xs)
        torch.cuda.synchronize()
        want_pred = O.predict_partition(ids.cpu().numpy(), conf.cpu().numpy(),
                                        emap.cpu().numpy(), P)
        want_perm, want_off = O.token_shuffle(want_pred, P)
        assert np.array_equal(pred.cpu().numpy(), want_pred)
        assert np.array_equal(perm.cpu().numpy(), want_perm)
        assert np.array_equal(off.cpu().numpy(), want_off)
        assert torch.equal(xs, x[perm.long()])


def test_noalloc_without_rows_and_with_no_tokens(smoe):
    # x_shuf = None through the Python wrapper: indices only
    T, d, E, P, V = 777, 64, 8, 2, 300
    desc = smoe.make_desc(T, d, E, 2, 1, 64, 0, P, V, "bf16")
    ws = smoe.workspace(desc)
    ids, conf, emap, x = make_inputs(5, T, d, E, P, V)
    ref, _ = run_both(smoe, desc, ids, conf, emap, x, ws)
    i32 = dict(dtype=torch.int32, device="cuda")
    pred, perm, off = (torch.full((T,), -3, **i32), torch.full((T,), -3, **i32),
                       torch.full((P + 1,), -3, **i32))
    smoe.smoe_predict_shuffle_noalloc(desc, ids, conf, emap, pred, perm, off)
    torch.cuda.synchronize()
    assert torch.equal(pred, ref[0]) and torch.equal(perm, ref[1]) and torch.equal(off, ref[2])
    # T = 0: nothing to predict, every partition offset is zero
    desc0 = smoe.make_desc(0, d, E, 2, 1, 64, 0, P, V, "bf16")
    off0 = torch.full((P + 1,), -3, **i32)
    smoe.smoe_predict_shuffle_noalloc(desc0, ids, conf, emap, pred, perm, off0)
    torch.cuda.synchronize()
    assert off0.cpu().tolist() == [0] * (P + 1)
