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


def activation_counts(profile_ids, profile_idx, vocab: int, E: int) -> np.ndarray:
    """act[v, e] = number of profile occurrences of token id v routed to expert e."""
    ids = np.asarray(profile_ids, dtype=np.int64)
    idx = np.asarray(profile_idx, dtype=np.int64)
    return np.bincount((ids[:, None] * E + idx).ravel(),
                       minlength=vocab * E).reshape(vocab, E).astype(np.float64)


def balanced_token_map(act, expert_part, P: int, slack: float = 0.1) -> np.ndarray:
    """Stage two of the co-clustering: each token id goes to the cluster holding most of its
    activations under the expert map, taken in order of decreasing frequency, into clusters
    whose load stays within (1 + slack) times the mean (else the least loaded one). slack < 0
    drops the load cap (pure argmax, the map the route predictor itself follows)."""
    act = np.asarray(act, dtype=np.float64)
    m = np.asarray(expert_part, dtype=np.int64)
    local = act @ np.eye(P)[m]
    if slack < 0:
        return local.argmax(axis=1).astype(np.int32)
    freq = act.sum(axis=1)
    cap = (1.0 + slack) * freq.sum() / P
    load = np.zeros(P)
    tau = np.zeros(act.shape[0], np.int32)
    for v in np.argsort(-freq, kind="stable"):
        order = np.argsort(-local[v], kind="stable")
        fits = [p for p in order if load[p] + freq[v] <= cap]
        choice = int(fits[0]) if fits else int(np.argmin(load))
        tau[v] = choice
        load[choice] += freq[v]
    return tau


def ceo_placement(act, P: int, theta: float = 0.1, iters: int = 40, samples: int = 64,
                  elite: float = 0.125, smoothing: float = 0.7, slack: float = 0.1,
                  seed: int = 0):
    """Balanced token-expert co-clustering ("Speculative MoE" §4.2), two stages.

    Stage one searches balanced expert maps (E/P experts per cluster) by cross-entropy
    optimisation: a per-expert categorical distribution over clusters is sampled into maps
    (experts in a random order, each drawn among the clusters with room left); a map is
    scored by the objective with every token in the cluster holding most of its activations
    (theta times the load imbalance of that token map plus (1 - theta) times the remote
    share); the distribution moves toward the elite maps. Stage two places the tokens of
    the best map under a load cap (balanced_token_map). Returns (expert_part, token_part,
    cost), cost of the final pair under the same objective; token ids with no activation
    sit in cluster 0 and weigh nothing."""
    act = np.asarray(act, dtype=np.float64)
    V, E = act.shape
    if E % P:
        raise ValueError("E must be a multiple of P")
    keep = act.sum(axis=1) > 0
    a = act[keep]
    freq = a.sum(axis=1)
    total = a.sum()
    rng = np.random.default_rng(seed)
    prob = np.full((E, P), 1.0 / P)
    n_elite = max(1, int(round(elite * samples)))
    eye = np.eye(P)
    best_m, best_c = None, np.inf
    for _ in range(iters):
        order = np.argsort(rng.random((samples, E)), axis=1)
        room = np.full((samples, P), E // P)
        maps = np.empty((samples, E), np.int64)
        u = rng.random((samples, E))
        rows = np.arange(samples)
        for j in range(E):
            e = order[:, j]
            w = prob[e] * (room > 0)
            cdf = np.cumsum(w, axis=1)
            pick = (cdf < (u[:, j] * cdf[:, -1])[:, None]).sum(axis=1)
            pick = np.minimum(pick, P - 1)
            while True:       # a zero-probability cluster with room can not be picked
                bad = room[rows, pick] <= 0
                if not bad.any():
                    break
                pick[bad] = np.argmax(room[bad], axis=1)
            maps[rows, e] = pick
            room[rows, pick] -= 1
        onehot = eye[maps].transpose(1, 0, 2).reshape(E, samples * P)
        local = (a @ onehot).reshape(-1, samples, P).transpose(1, 0, 2)   # [samples, V, P]
        tau = local.argmax(axis=2)
        remote = total - np.take_along_axis(local, tau[..., None], axis=2).sum(axis=(1, 2))
        loads = np.stack([np.bincount(tau[i], weights=freq, minlength=P)
                          for i in range(samples)])
        mean = loads.mean(axis=1)
        imb = np.where(mean > 0, (loads.max(axis=1) - mean) / np.maximum(mean, 1e-300), 0.0)
        cost = theta * imb + (1.0 - theta) * (remote / total if total > 0 else 0.0)
        top = np.argsort(cost, kind="stable")[:n_elite]
        if cost[top[0]] < best_c:
            best_c, best_m = float(cost[top[0]]), maps[top[0]].copy()
        freq_e = eye[maps[top]].mean(axis=0)                # [E, P]
        prob = smoothing * freq_e + (1.0 - smoothing) * prob
    tau_k = balanced_token_map(a, best_m, P, slack)
    load = np.bincount(tau_k, weights=freq, minlength=P)
    mean = load.mean()
    local = a @ eye[best_m]
    remote = total - local[np.arange(len(tau_k)), tau_k].sum()
    cost = (theta * ((load.max() - mean) / mean if mean > 0 else 0.0)
            + (1.0 - theta) * (remote / total if total > 0 else 0.0))
    tau_full = np.zeros(V, np.int32)
    tau_full[keep] = tau_k
    return best_m.astype(np.int32), tau_full, float(cost)
