"""Host side of a real expert-parallel exchange across processes ("Speculative MoE" §1:
under expert parallelism each token is sent from its device to the devices of its K
experts, and the expert outputs are sent back the same way).

On one GPU, ``smoe_ep_exchange`` lays out what P devices would exchange: the send
counts [P, P] and the receive rows sorted by (dst, src, t, k). With one process per
device, each rank sends its own rows in (dst, t, k) order; the rows arriving at rank q
are then exactly segment q of that layout. These helpers turn a rank's part of the plan
into the two all-to-all calls of ``torch.distributed`` (NCCL between GPUs, gloo on the
host): first the per-destination counts, then the rows (all2allv). Nothing here does
any of the layer's arithmetic.
"""
from __future__ import annotations

import torch


def send_order(recv_token, recv_off, P: int, rank: int):
    """Token of each row this rank sends, in (dst, t, k) order: the concatenation over
    destinations q of receive segment (dst q, src rank) of the single-device layout.
    Returns (tokens, counts): an index tensor and the P per-destination row counts."""
    off = [int(v) for v in recv_off.tolist()]
    segs = [(off[q * P + rank], off[q * P + rank + 1]) for q in range(P)]
    parts = [recv_token[a:b] for a, b in segs]
    tokens = torch.cat(parts) if parts else recv_token[:0]
    return tokens, [b - a for a, b in segs]


def exchange_counts(send_counts: list[int], group=None) -> list[int]:
    """All-to-all of the per-destination row counts: returns how many rows this rank
    receives from every source."""
    import torch.distributed as dist
    inp = torch.tensor(send_counts, dtype=torch.int64)
    if dist.get_backend(group) == "nccl":
        inp = inp.cuda()
    out = torch.empty_like(inp)
    dist.all_to_all_single(out, inp, group=group)
    return [int(v) for v in out.cpu().tolist()]


def dispatch(x_send, send_counts: list[int], recv_counts: list[int] | None = None, group=None):
    """Rows x_send [sum(send_counts), d], grouped by destination, to their destinations.
    Returns (x_recv, recv_counts): the rows this rank receives, grouped by source in
    source order, each source's rows in the order it sent them."""
    import torch.distributed as dist
    if recv_counts is None:
        recv_counts = exchange_counts(send_counts, group)
    x_recv = x_send.new_empty((sum(recv_counts),) + tuple(x_send.shape[1:]))
    dist.all_to_all_single(x_recv, x_send.contiguous(), recv_counts, send_counts, group=group)
    return x_recv, recv_counts


def combine_back(y_recv, send_counts: list[int], recv_counts: list[int], group=None):
    """The return trip: expert outputs y_recv (in receive order) back to the ranks that
    sent the rows; the result is in this rank's send order."""
    import torch.distributed as dist
    y_back = y_recv.new_empty((sum(send_counts),) + tuple(y_recv.shape[1:]))
    dist.all_to_all_single(y_back, y_recv.contiguous(), send_counts, recv_counts, group=group)
    return y_back


def send_rows_of_pairs(pair_recv, recv_off, P: int, rank: int):
    """For pairs whose token sits on this rank: their row in this rank's send buffer
    (and so in the buffer combine_back returns), from their row in the single-device
    receive layout. pair_recv [n, K] of this rank's tokens; returns the same shape."""
    off = torch.as_tensor(recv_off, dtype=torch.int64)
    r = torch.as_tensor(pair_recv, dtype=torch.int64)
    seg = torch.searchsorted(off, r, right=True) - 1           # segment (dst q, src rank)
    q = seg // P
    counts = torch.stack([off[qq * P + rank + 1] - off[qq * P + rank] for qq in range(P)])
    base = torch.cumsum(counts, 0) - counts
    return r - off[seg] + base[q]
