"""The host side of a real expert-parallel exchange across processes, with two gloo
ranks on the CPU (one rank per simulated device, P = 2): each rank sends its own rows in
(dst, t, k) order and must receive exactly its segment of the single-device receive
layout; the return trip brings every expert output back to its token's rank, where the
combine gives sum_k w_k f(x_t). The plan comes from the oracle (no GPU here); on GPUs
the same calls run over NCCL."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import oracle as O
    from routing_token_shuffle_gb300 import ep
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        dist.init_process_group("gloo", rank=rank, world_size=world)
        P, T, E, K, d = world, 40, 8, 3, 16
        rng = np.random.default_rng(5)
        idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
        emap = (np.arange(E) % P).astype(np.int32)
        src = rng.integers(0, P, T).astype(np.int32)
        w = rng.random((T, K))
        x = torch.as_tensor(rng.standard_normal((T, d)))
        send_counts, recv_off, pair_recv, recv_token = O.ep_exchange(idx, emap, P, src)
        recv_token_t = torch.as_tensor(recv_token, dtype=torch.int64)
        tokens, counts = ep.send_order(recv_token_t, torch.as_tensor(recv_off), P, rank)
        assert counts == send_counts[rank].tolist()
        x_recv, rcounts = ep.dispatch(x[tokens], counts)
        assert rcounts == send_counts[:, rank].tolist()
        lo, hi = recv_off[rank * P], recv_off[rank * P + P]
        assert torch.equal(x_recv, x[recv_token_t[lo:hi]])
        # "experts": device q scales its rows by q + 2; the outputs go back to the sources
        y_back = ep.combine_back(x_recv * (rank + 2), counts, rcounts)
        mine = np.nonzero(src == rank)[0]
        rows = ep.send_rows_of_pairs(pair_recv[mine], recv_off, P, rank)
        y = (torch.as_tensor(w[mine])[:, :, None] * y_back[rows]).sum(1)
        scale = torch.as_tensor(emap[idx[mine]] + 2.0)
        want = (torch.as_tensor(w[mine]) * scale)[:, :, None] * x[mine][:, None, :]
        assert torch.allclose(y, want.sum(1), rtol=1e-12, atol=1e-12)
        dist.destroy_process_group()
        q.put((rank, "ok"))
    except Exception as e:  # report to the parent instead of hanging it
        q.put((rank, repr(e)))


def test_two_rank_exchange_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert res == {0: "ok", 1: "ok"}, res
