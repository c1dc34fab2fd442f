"""Offline tables for the speculative shuffle (not timed, not on the layer's hot path).

"Speculative MoE" §4.1 and Fig. 3: token activations are profiled offline into a
token-expert confidence table C_p = Pr(E_k | token); an id that never appeared takes
the row of its cosine-nearest profiled id in embedding space. §3.2 (s-EG): experts
that fire together are placed on the same device. The routes these tools count come
from the library's own routing kernel (smoe_route) on a profiling batch.
"""
from __future__ import annotations

import numpy as np


def confidence_table(profile_ids, profile_idx, vocab: int, E: int, K: int, emb_rows=None,
                     rows_needed=None) -> np.ndarray:
    """C_p [vocab, E] float32: share of each id's profile occurrences routed to expert e.

    Unseen ids take the row of the cosine-nearest seen id (the lower id on ties), or
    K/E when nothing was seen or no embedding is given. ``rows_needed`` restricts the
    nearest-neighbour fill to the ids that will be looked up."""
    ids = np.asarray(profile_ids, dtype=np.int64)
    idx = np.asarray(profile_idx, dtype=np.int64)
    occ = np.bincount(ids, minlength=vocab)
    pair = np.bincount((ids[:, None] * E + idx).ravel(), minlength=vocab * E).reshape(vocab, E)
    table = np.full((vocab, E), K / E, dtype=np.float64)
    seen = np.flatnonzero(occ)
    table[seen] = pair[seen] / occ[seen, None]
    if len(seen) and emb_rows is not None:
        want = np.arange(vocab) if rows_needed is None else np.unique(np.asarray(rows_needed))
        unseen = want[occ[want] == 0]
        if len(unseen):
            es = np.asarray(emb_rows(seen), dtype=np.float32)
            es /= np.linalg.norm(es, axis=1, keepdims=True)
            for lo in range(0, len(unseen), 2048):
                blk = unseen[lo:lo + 2048]
                eu = np.asarray(emb_rows(blk), dtype=np.float32)
                eu /= np.linalg.norm(eu, axis=1, keepdims=True)
                table[blk] = table[seen[np.argmax(eu @ es.T, axis=1)]]
    return table.astype(np.float32)


def coclustered_placement(profile_idx, E: int, P: int, order) -> np.ndarray:
    """Greedy s-EG-style placement: experts, in the given (seeded) order, join the
    partition whose current members they co-fire with most often, among partitions
    with room left (E/P experts each); ties go to the lower partition."""
    idx = np.asarray(profile_idx, dtype=np.int64)
    n, K = idx.shape
    onehot = np.zeros((n, E), dtype=np.float32)
    np.put_along_axis(onehot, idx, 1.0, axis=1)
    co = (onehot.T @ onehot).astype(np.int64)
    np.fill_diagonal(co, 0)
    cap = E // P
    place = np.full(E, -1, dtype=np.int32)
    members = [[] for _ in range(P)]
    for e in np.asarray(order, dtype=np.int64):
        best, best_aff = -1, -1
        for p in range(P):
            if len(members[p]) >= cap:
                continue
            aff = int(co[e, members[p]].sum()) if members[p] else 0
            if aff > best_aff:
                best, best_aff = p, aff
        place[e] = best
        members[best].append(int(e))
    return place


def cluster_of(routes, expert_part, P: int) -> np.ndarray:
    """Each token's cluster: the partition holding most of its routed experts (lower
    partition on ties)."""
    part = np.asarray(expert_part, dtype=np.int64)[np.asarray(routes, dtype=np.int64)]
    hist = np.zeros((part.shape[0], P), dtype=np.int64)
    for k in range(part.shape[1]):
        np.add.at(hist, (np.arange(part.shape[0]), part[:, k]), 1)
    return hist.argmax(axis=1).astype(np.int32)


def transition_table(prev_cluster, cur_cluster, P: int) -> np.ndarray:
    """Table A [P, P] float32 of "Speculative MoE" §4.1's 2-gram model: the share of the
    profile tokens of previous cluster c that land in cluster p (uniform if c is unseen)."""
    idx = np.asarray(prev_cluster, dtype=np.int64) * P + np.asarray(cur_cluster, dtype=np.int64)
    counts = np.bincount(idx, minlength=P * P).reshape(P, P).astype(np.float64)
    tot = counts.sum(axis=1, keepdims=True)
    table = np.full((P, P), 1.0 / P)
    seen = tot[:, 0] > 0
    table[seen] = counts[seen] / tot[seen]
    return table.astype(np.float32)
