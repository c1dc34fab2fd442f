"""Offline table tools of the package (not timed, not on the layer path): the confidence
table, the cluster transition table and the co-clustering placement, against the oracle's
definitions."""
import numpy as np
import pytest

import oracle as O
from routing_token_shuffle_gb300 import profiling


def test_confidence_table_matches_oracle():
    rng = np.random.default_rng(1)
    V, E, K, n, d = 60, 8, 2, 500, 16
    ids = rng.integers(0, V // 2, size=n)
    idx = O.topk_select(rng.standard_normal((n, E)).astype(np.float32), K)
    emb = rng.standard_normal((V, d))
    a = profiling.confidence_table(ids, idx, V, E, K, emb_rows=lambda v: emb[np.asarray(v)])
    b = O.profile_confidence(ids, idx, V, E, K, emb_rows=lambda v: emb[np.asarray(v)])
    np.testing.assert_allclose(a, b, rtol=1e-6)


def test_transition_table_and_cluster_match_oracle():
    rng = np.random.default_rng(2)
    T, E, K, P = 400, 12, 3, 4
    emap = (np.arange(E) % P).astype(np.int32)
    i1 = O.topk_select(rng.standard_normal((T, E)).astype(np.float32), K)
    i2 = O.topk_select(rng.standard_normal((T, E)).astype(np.float32), K)
    c1, c2 = profiling.cluster_of(i1, emap, P), profiling.cluster_of(i2, emap, P)
    assert np.array_equal(c1, O.token_cluster(i1, emap, P))
    np.testing.assert_array_equal(profiling.transition_table(c1, c2, P), O.markov_table(c1, c2, P))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_ceo_finds_brute_force_optimum_remote_only(seed):
    """theta = 0 without a load cap: every token sits in its best cluster, so the search
    reduces to balanced expert maps; on a tiny instance it must reach the exhaustive
    optimum."""
    rng = np.random.default_rng(seed)
    act = rng.integers(0, 4, size=(5, 6)).astype(float)
    opt, _, _ = O.coclustering_bruteforce(act, 2, 0.0)
    m, tau, cost = profiling.ceo_placement(act, 2, theta=0.0, iters=20, samples=32,
                                            slack=-1.0, seed=seed)
    assert np.bincount(m, minlength=2).tolist() == [3, 3]
    assert abs(cost - O.coclustering_cost(act, m, tau, 2, 0.0)) < 1e-12
    assert abs(cost - opt) < 1e-12


def test_ceo_balanced_cost_consistent_and_better_than_identity():
    rng = np.random.default_rng(5)
    V, E, P = 40, 16, 4
    # tokens in 4 groups, each group firing a scattered set of 4 experts
    groups = rng.permutation(E).reshape(P, E // P)
    act = np.zeros((V, E))
    for v in range(V):
        g = groups[v % P]
        act[v, g] = rng.integers(1, 5, size=len(g))
    m, tau, cost = profiling.ceo_placement(act, P, theta=0.1, iters=40, samples=64, seed=3)
    assert np.bincount(m, minlength=P).tolist() == [E // P] * P
    assert abs(cost - O.coclustering_cost(act, m, tau, P, 0.1)) < 1e-12
    ident = (np.arange(E) * P // E).astype(np.int32)
    tau_id = np.argmax(np.stack([act[:, ident == p].sum(1) for p in range(P)], 1), 1)
    assert cost < O.coclustering_cost(act, ident, tau_id, P, 0.1)
    assert cost < 0.05       # the planted grouping is recovered almost exactly


def test_balanced_token_map_respects_cap():
    rng = np.random.default_rng(7)
    act = rng.integers(0, 6, size=(200, 16)).astype(float)
    m = (np.arange(16) % 4).astype(np.int32)
    tau = profiling.balanced_token_map(act, m, 4, slack=0.05)
    load = np.bincount(tau, weights=act.sum(1), minlength=4)
    assert load.max() <= 1.05 * load.mean() + act.sum(1).max()
    free = profiling.balanced_token_map(act, m, 4, slack=-1.0)
    local = np.stack([act[:, m == p].sum(1) for p in range(4)], 1)
    assert np.array_equal(free, local.argmax(1))


def test_activation_counts():
    ids = np.array([3, 3, 0])
    idx = np.array([[1, 2], [1, 0], [2, 1]])
    act = profiling.activation_counts(ids, idx, 5, 4)
    assert act.shape == (5, 4) and act.sum() == 6
    assert act[3].tolist() == [1, 2, 1, 0] and act[0].tolist() == [0, 1, 1, 0]
