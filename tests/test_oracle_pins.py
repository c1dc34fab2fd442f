"""Pins for the CPU oracle: brute force, closed forms, invariants and hand-worked
fixtures (tests/golden), none of which reuses the oracle's own code path."""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- top-K ------


def brute_topk(row, K):
    """All C(E,K) subsets: the chosen set is the one whose every member precedes every
    non-member in the order (logit descending, index ascending)."""
    E = len(row)

    def before(a, b):
        return row[a] > row[b] or (row[a] == row[b] and a < b)

    winners = []
    for S in itertools.combinations(range(E), K):
        rest = [j for j in range(E) if j not in S]
        if all(before(a, b) for a in S for b in rest):
            winners.append(S)
    assert len(winners) == 1
    S = list(winners[0])
    # order inside the set: repeatedly the member that precedes all others
    out = []
    while S:
        best = [a for a in S if all(a == b or before(a, b) for b in S)]
        assert len(best) == 1
        out.append(best[0])
        S.remove(best[0])
    return out


@pytest.mark.parametrize("E,K", [(4, 1), (4, 2), (6, 3), (8, 2), (8, 5), (8, 8)])
def test_topk_brute_force(E, K):
    rng = np.random.default_rng(E * 10 + K)
    # values from a small set so exact ties are common; include +0 and -0
    vals = np.array([-1.0, -0.0, 0.0, 0.5, 1.0, 2.0], dtype=np.float32)
    logits = vals[rng.integers(0, len(vals), size=(64, E))]
    logits[:8] = rng.standard_normal((8, E)).astype(np.float32)
    idx = O.topk_select(logits, K)
    for t in range(logits.shape[0]):
        assert list(idx[t]) == brute_topk(logits[t].tolist(), K), t


def test_topk_signed_zero_ties():
    logits = np.array([[-0.0, 0.0, -1.0, 0.0]], dtype=np.float32)
    assert O.topk_select(logits, 2).tolist() == [[0, 1]]
    logits = np.array([[0.0, -0.0, -0.0, -2.0]], dtype=np.float32)
    assert O.topk_select(logits, 3).tolist() == [[0, 1, 2]]


def test_grouped_H1_is_plain_topk():
    rng = np.random.default_rng(1)
    logits = rng.standard_normal((50, 16)).astype(np.float32)
    for t in range(50):
        assert list(O.topk_select(logits, 4, H=1)[t]) == brute_topk(logits[t].tolist(), 4)


def test_grouped_one_pick_per_group_direct_loop():
    rng = np.random.default_rng(2)
    E, H = 32, 8
    logits = rng.integers(-2, 3, size=(40, E)).astype(np.float32)
    idx = O.topk_select(logits, H, H=H)
    per = E // H
    for t in range(40):
        for h in range(H):
            best = h * per
            for e in range(h * per, (h + 1) * per):
                if logits[t, e] > logits[t, best]:
                    best = e
            assert idx[t, h] == best


def test_grouped_brute_force_two_per_group():
    rng = np.random.default_rng(3)
    E, H, K = 8, 2, 4
    logits = rng.integers(-1, 2, size=(30, E)).astype(np.float32)
    idx = O.topk_select(logits, K, H=H)
    for t in range(30):
        exp = brute_topk(logits[t, :4].tolist(), 2) + [4 + j for j in brute_topk(logits[t, 4:].tolist(), 2)]
        assert list(idx[t]) == exp


def test_grouped_H_equals_E_identity():
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((10, 8)).astype(np.float32)
    assert (O.topk_select(logits, 8, H=8) == np.arange(8)).all()


def test_softmax_topk_golden():
    g = load("softmax_topk_hand.json")
    logits = np.array(g["logits"], dtype=np.float32)
    idx = O.topk_select(logits, 2)
    assert idx.tolist() == g["top2_idx"]
    np.testing.assert_allclose(O.gate_weights(logits, idx), g["top2_w"], atol=g["tolerance"])
    np.testing.assert_allclose(O.gate_weights(logits, idx, renorm=True), g["top2_w_renorm"],
                               atol=g["tolerance"])
    gi = O.topk_select(logits, 2, H=2)
    assert gi.tolist() == g["grouped_H2_K2_idx"]
    np.testing.assert_allclose(O.gate_weights(logits, gi), g["grouped_H2_K2_w"], atol=g["tolerance"])


def test_softmax_properties():
    rng = np.random.default_rng(5)
    logits = (rng.standard_normal((20, 12)) * 3).astype(np.float32)
    allidx = np.tile(np.arange(12), (20, 1))
    w = O.gate_weights(logits, allidx)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, atol=1e-12)
    # shift invariance and the exp ratio
    w2 = O.gate_weights(logits + np.float32(10.0), allidx)
    np.testing.assert_allclose(w, w2, rtol=1e-5)
    l64 = logits.astype(np.float64)
    np.testing.assert_allclose(w[:, 1] / w[:, 0], np.exp(l64[:, 1] - l64[:, 0]), rtol=1e-12)


def test_selection_margin():
    logits = np.array([[3.0, 1.0, 2.0, 0.5], [1.0, 1.0, 1.0, 1.0]], dtype=np.float32)
    np.testing.assert_allclose(O.selection_margin(logits, 2), [1.0, 0.0])
    np.testing.assert_allclose(O.selection_margin(logits, 2, H=2), [1.5, 0.0])


def test_gate_logits_exact_small_integers():
    rng = np.random.default_rng(6)
    x = rng.integers(-3, 4, size=(7, 5)).astype(np.float32)
    wg = rng.integers(-3, 4, size=(4, 5)).astype(np.float32)
    exp = [[sum(int(x[t, j]) * int(wg[e, j]) for j in range(5)) for e in range(4)] for t in range(7)]
    assert O.gate_logits(x, wg).tolist() == exp


def test_gate_logits_rounded_once_to_float32():
    """Logits are float32 (one rounding of the exact dot product): 1 + 2^-30 is 1.0."""
    x = np.array([[1.0, 2.0 ** -30]])
    wg = np.array([[1.0, 1.0], [1.0, -1.0]])
    out = O.gate_logits(x, wg)
    assert out.dtype == np.float32
    assert out.tolist() == [[1.0, 1.0]]


def test_topk_compares_float32_logits():
    """Selection compares float32 values: logits that differ only below float32 resolution
    are a tie, which the lower index wins."""
    logits = np.array([[1.0, 1.0 + 1e-12, 0.0, -1.0],
                       [-1.0, 0.5 + 1e-13, 0.5, 0.25]])
    assert O.topk_select(logits, 1).tolist() == [[0], [1]]
    assert O.topk_select(logits, 2).tolist() == [[0, 1], [1, 2]]


# ------------------------------------------------ predicted partition --------


def test_predict_exact_rationals():
    """C_p values are multiples of 1/64, so float32 sums are exact and the argmax can be
    checked with exact rational arithmetic."""
    rng = np.random.default_rng(7)
    V, E, P = 40, 12, 3
    conf = (rng.integers(0, 65, size=(V, E)) / 64.0).astype(np.float32)
    emap = rng.integers(0, P, size=E).astype(np.int32)
    ids = rng.integers(0, V, size=200).astype(np.int32)
    pred = O.predict_partition(ids, conf, emap, P)
    for t, v in enumerate(ids):
        sc = [sum((Fraction(float(conf[v, e])) for e in range(E) if emap[e] == p), Fraction(0))
              for p in range(P)]
        best = max(sc)
        assert pred[t] == sc.index(best)


def test_predict_scores_are_float32_sums_in_ascending_expert_order():
    """Partition scores add the C_p entries of the partition's experts one float32 add at a
    time, in ascending expert order; equal scores go to the lower partition.
    Row 0: partition 1 sums 1 + 2^-24, which rounds to 1.0 (half an ulp, to even), so it
    ties partition 0's 1.0 and partition 0 wins (a float64 sum would pick 1).
    Row 1: partition 1's entries 2^-24, 2^-24, 1 sum to 1 + 2^-23 in ascending order and
    beat partition 0's 1.0 (in descending order they would round back to 1.0 and tie)."""
    tiny = np.float32(2.0 ** -24)
    conf = np.array([[1.0, 1.0, tiny, 0.0],
                     [1.0, tiny, tiny, 1.0]], dtype=np.float32)
    emap = np.array([0, 1, 1, 1], np.int32)
    assert O.predict_partition(np.array([0, 1]), conf, emap, 2).tolist() == [0, 1]


def test_predict_single_partition():
    conf = np.random.default_rng(8).random((10, 6)).astype(np.float32)
    assert (O.predict_partition(np.arange(10), conf, np.zeros(6, np.int32), 1) == 0).all()


# ---------------------------------------------------- shuffle / LAR ----------


def test_fig2_golden_shuffle_lar_dispatch():
    g = load("shuffle_lar_fig2_hand.json")
    conf = np.array(g["conf_rows"], dtype=np.float32)
    emap = np.array(g["expert_part"], dtype=np.int32)
    routes = np.array(g["routes"], dtype=np.int32)
    pred = O.predict_partition(np.array(g["token_ids"]), conf, emap, g["P"])
    assert pred.tolist() == g["pred"]
    perm, off = O.token_shuffle(pred, g["P"])
    assert perm.tolist() == g["shuf_perm"] and off.tolist() == g["part_off"]
    lar = O.lar_counts(routes, emap, g["P"], 1, src_part=pred)
    L = g["lar"]
    assert lar.tolist() == [L["local"], L["total"], L["base_local"], L["max_local"]]
    eo, pr, rt = O.expert_dispatch(routes, 4, perm)
    assert eo.tolist() == g["expert_off"]
    assert rt.tolist() == g["row_token"]
    assert pr.tolist() == g["pair_row"]


@pytest.mark.parametrize("T,P", [(1, 1), (37, 3), (500, 8), (64, 2)])
def test_shuffle_invariants(T, P):
    rng = np.random.default_rng(T + P)
    pred = rng.integers(0, P, size=T).astype(np.int32)
    perm, off = O.token_shuffle(pred, P)
    assert sorted(perm.tolist()) == list(range(T))                  # bijection
    hist = [sum(1 for v in pred if v == p) for p in range(P)]
    assert off.tolist() == [sum(hist[:p]) for p in range(P + 1)]    # scan of histogram
    keys = pred[perm]
    assert all(keys[i] <= keys[i + 1] for i in range(T - 1))        # sorted
    for p in range(P):                                                # stable
        seg = perm[off[p]:off[p + 1]]
        assert all(seg[i] < seg[i + 1] for i in range(len(seg) - 1))
        assert (pred[seg] == p).all()


def direct_lar(idx, emap, P, H, src):
    T, K = idx.shape
    local = base = mx = 0
    for t in range(T):
        cnt = [0] * P
        for k in range(K):
            dst = int(emap[idx[t, k]])
            cnt[dst] += 1
            s = src(t, k)
            if dst == s:
                local += 1
            if dst == (t * P) // T:
                base += 1
        mx += max(cnt)
    return [local, T * K, base, mx]


@pytest.mark.parametrize("T,E,K,P", [(50, 8, 2, 2), (33, 16, 4, 4), (20, 12, 3, 3)])
def test_lar_direct_count(T, E, K, P):
    rng = np.random.default_rng(T * E)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx = O.topk_select(logits, K)
    emap = rng.integers(0, P, size=E).astype(np.int32)
    pred = rng.integers(0, P, size=T).astype(np.int32)
    got = O.lar_counts(idx, emap, P, 1, src_part=pred).tolist()
    assert got == direct_lar(idx, emap, P, 1, lambda t, k: int(pred[t]))
    assert got[0] <= got[3]        # alpha_sTS <= alpha_max


@pytest.mark.parametrize("K", [2, 4])
def test_lar_foe_rule_direct_count(K):
    """H < G: copy (t, h) sits on h (G/H) + (t mod G/H); with K/H > 1 the group of slot
    k is k // (K/H), not k mod H."""
    rng = np.random.default_rng(11 + K)
    T, E, H, G = 40, 16, 2, 8
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx = O.topk_select(logits, K, H=H)
    # group h spans partitions 4h..4h+3; its j-th expert is on 4h + (j mod 4)
    emap = np.array([(e // 8) * 4 + (e % 8) % 4 for e in range(E)], np.int32)
    got = O.lar_counts(idx, emap, G, H).tolist()
    exp = direct_lar(idx, emap, G, H, lambda t, k: (k // (K // H)) * (G // H) + t % (G // H))
    assert got == exp


@pytest.mark.parametrize("H,G,K", [(4, 2, 8), (4, 4, 8), (8, 2, 8)])
def test_lar_foe_rule_direct_count_H_ge_G(H, G, K):
    """H >= G: every copy for group h sits on floor(h G / H), checked on a random map."""
    rng = np.random.default_rng(100 * H + G)
    T, E = 30, 16
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx = O.topk_select(logits, K, H=H)
    emap = rng.integers(0, G, size=E).astype(np.int32)
    got = O.lar_counts(idx, emap, G, H).tolist()
    exp = direct_lar(idx, emap, G, H, lambda t, k: ((k // (K // H)) * G) // H)
    assert got == exp


@pytest.mark.parametrize("H", [1, 2])
def test_layer_alpha_counts_from_predicted_partition(H):
    """The layer's alpha counts a routed pair as local when its expert sits on the
    partition the token was shuffled to (its predicted partition)."""
    x, ids, wg, w1, w3, w2, conf, emap = tiny_layer(seed=40 + H, T=60, E=8, K=4, H=H, P=4)
    out = O.layer_forward(x, ids, wg, w1, w3, w2, conf, emap, K=4, H=H, P=4)
    pred = out["pred"]
    assert len(set(pred.tolist())) > 1
    assert out["lar"].tolist() == direct_lar(out["idx"], emap, 4, H, lambda t, k: int(pred[t]))


def test_lar_max_equals_sts_when_table_is_exact():
    """alpha_sTS = alpha_max when every id is unique and C_p is profiled on that batch."""
    rng = np.random.default_rng(12)
    T, E, K, P = 300, 16, 4, 4
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx = O.topk_select(logits, K)
    ids = np.arange(T, dtype=np.int32)
    conf = O.profile_confidence(ids, idx, T, E, K)
    emap = (np.arange(E) % P).astype(np.int32)
    pred = O.predict_partition(ids, conf, emap, P)
    lar = O.lar_counts(idx, emap, P, 1, src_part=pred)
    assert lar[0] == lar[3]


# ------------------------------------------------------ closed forms ---------


def test_closed_forms_golden():
    g = load("foe_closed_forms.json")
    for G, v in zip(g["rho_moe"]["G"], g["rho_moe"]["value"]):
        assert O.rho_moe(G) == v
    for c in g["rho_foe"]:
        assert O.rho_foe(c["H"], c["G"]) == c["value"]
    for c in g["a2a_intra"]:
        assert O.a2a_volume_intra(c["k"], c["G"], c["H"]) == c["value"]
    a = g["asymptote"]
    assert abs(O.foe_asymptote(a["k"], a["H"], a["r"]) - a["value_exact"]) < 1e-12
    assert round(O.foe_asymptote(a["k"], a["H"], a["r"]), 1) == a["value_printed"]


@pytest.mark.parametrize("G", [2, 4, 8])
def test_rho_moe_uniform_routing(G):
    """Uniform routing puts a pair on its token's (contiguous-split) partition with
    probability 1/G."""
    T, E, K = 65536, 32, 2
    rng = np.random.default_rng(100 + G)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx = O.topk_select(logits, K)
    emap = (np.arange(E) * G // E).astype(np.int32)
    lar = O.lar_counts(idx, emap, G, 1, src_part=np.zeros(T, np.int32))
    alpha_base = lar[2] / lar[1]
    assert abs(alpha_base - O.rho_moe(G)) <= 4 * 0.5 / math.sqrt(T)


@pytest.mark.parametrize("G", [2, 4, 8])
def test_rho_foe_exact_when_H_ge_G(G):
    T, E, H = 4096, 64, 8
    rng = np.random.default_rng(200 + G)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx = O.topk_select(logits, H, H=H)
    per = E // H
    emap = np.array([((e // per) * G) // H for e in range(E)], np.int32)
    lar = O.lar_counts(idx, emap, G, H)
    assert lar[0] == lar[1]                        # alpha_FoE = min(H/G, 1) = 1
    # remote traffic identity: remote pairs = T K - local = T * k (G - H)/G ... = 0 here
    assert lar[1] - lar[0] == 0


def test_rho_foe_H2_G8():
    T, E, H, G = 65536, 32, 2, 8
    K = 2
    rng = np.random.default_rng(300)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx = O.topk_select(logits, K, H=H)
    per = E // H
    emap = np.array([(e // per) * (G // H) + (e % per) % (G // H) for e in range(E)], np.int32)
    lar = O.lar_counts(idx, emap, G, H)
    alpha = lar[0] / lar[1]
    assert abs(alpha - O.rho_foe(H, G)) <= 4 * 0.5 / math.sqrt(T)
    # remote pairs per token, both ways, against 2k(G-H)/G
    remote_both = 2 * (lar[1] - lar[0]) / T
    assert abs(remote_both - O.a2a_volume_intra(K, G, H)) <= 2 * K * 4 * 0.5 / math.sqrt(T)


# ----------------------------------------------------------- dispatch --------


@pytest.mark.parametrize("T,E,K", [(1, 4, 1), (45, 8, 2), (100, 16, 6), (64, 8, 8)])
def test_dispatch_invariants(T, E, K):
    rng = np.random.default_rng(T + E + K)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx = O.topk_select(logits, K)
    perm = rng.permutation(T).astype(np.int32)
    eo, pr, rt = O.expert_dispatch(idx, E, perm)
    assert sorted(pr.ravel().tolist()) == list(range(T * K))       # bijection
    hist = [int((idx == e).sum()) for e in range(E)]
    assert eo.tolist() == [sum(hist[:e]) for e in range(E + 1)]
    slot = np.empty(T, np.int64)
    slot[perm] = np.arange(T)
    key = {}
    for t in range(T):
        for k in range(K):
            r = int(pr[t, k])
            assert rt[r] == t
            assert eo[idx[t, k]] <= r < eo[idx[t, k] + 1]
            key[r] = (int(idx[t, k]), int(slot[t]), k)
    ks = [key[r] for r in range(T * K)]
    assert ks == sorted(ks)                                          # key (expert, s, k)


def test_dispatch_without_shuffle_is_token_order():
    rng = np.random.default_rng(9)
    idx = O.topk_select(rng.standard_normal((30, 6)).astype(np.float32), 2)
    a = O.expert_dispatch(idx, 6, None)
    b = O.expert_dispatch(idx, 6, np.arange(30))
    for u, v in zip(a, b):
        assert (u == v).all()


# -------------------------------------------------------- FFN / combine ------


def test_swiglu_golden():
    g = load("swiglu_hand.json")
    x, w1, w3, w2 = (np.array(g[k]) for k in ("x", "w1", "w3", "w2"))
    np.testing.assert_allclose(O.swiglu_hidden(x, w1, w3), g["hidden"], rtol=1e-15)
    np.testing.assert_allclose(O.swiglu_ffn(x, w1, w3, w2), g["y"], rtol=1e-15)


def test_swiglu_structure():
    rng = np.random.default_rng(10)
    x = rng.standard_normal((5, 6))
    w1, w3 = rng.standard_normal((2, 4, 6))
    w2 = rng.standard_normal((6, 4))
    y = O.swiglu_ffn(x, w1, w3, w2)
    assert np.all(O.swiglu_ffn(x, np.zeros_like(w1), w3, w2) == 0)   # silu(0) = 0
    np.testing.assert_allclose(O.swiglu_ffn(x, w1, 2 * w3, w2), 2 * y, rtol=1e-13)
    np.testing.assert_allclose(O.swiglu_ffn(x, w1, w3, -3 * w2), -3 * y, rtol=1e-13)
    # large positive gate pre-activations: silu(z) -> z, so y -> ((x W1^T)(x W3^T)) W2^T
    big = 1e3 * np.abs(w1)
    xp = np.abs(x)
    lin = ((xp @ big.T) * (xp @ w3.T)) @ w2.T
    np.testing.assert_allclose(O.swiglu_ffn(xp, big, w3, w2), lin, rtol=1e-12)


def test_silu_values():
    assert O.silu(0.0) == 0.0
    assert abs(O.silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert abs(O.silu(-40.0)) < 1e-15


def test_combine_identity_experts():
    """With each expert the identity, combine returns sum_k w_k x."""
    rng = np.random.default_rng(13)
    T, E, K, d = 40, 8, 3, 5
    x = rng.standard_normal((T, d))
    idx = O.topk_select(rng.standard_normal((T, E)).astype(np.float32), K)
    w = rng.random((T, K))
    eo, pr, rt = O.expert_dispatch(idx, E, rng.permutation(T))
    y = O.combine(x[rt], pr, w)
    for t in range(T):
        exp = np.zeros(d)
        for k in range(K):
            exp += w[t, k] * x[t]
        np.testing.assert_allclose(y[t], exp, rtol=1e-14, atol=1e-14)
    ysh = rng.standard_normal((2, T, d))
    np.testing.assert_allclose(O.combine(x[rt], pr, w, ysh) - y, ysh[0] + ysh[1], atol=1e-13)


def tiny_layer(seed=0, T=48, d=16, E=8, K=2, H=1, F=24, S=0, P=2, V=50):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d))
    ids = rng.integers(0, V, size=T).astype(np.int32)
    wg = rng.standard_normal((E, d)) / math.sqrt(d)
    w1 = rng.standard_normal((E + S, F, d)) / math.sqrt(d)
    w3 = rng.standard_normal((E + S, F, d)) / math.sqrt(d)
    w2 = rng.standard_normal((E + S, d, F)) / math.sqrt(F)
    conf = rng.random((V, E)).astype(np.float32)
    emap = (np.arange(E) % P).astype(np.int32)
    return x, ids, wg, w1, w3, w2, conf, emap


def test_one_expert_K1_is_weighted_ffn():
    x, ids, wg, w1, w3, w2, conf, emap = tiny_layer(E=1, K=1, P=1)
    out = O.layer_forward(x, ids, wg, w1, w3, w2, conf, emap, K=1, P=1)
    np.testing.assert_allclose(out["w"], 1.0)
    np.testing.assert_allclose(out["y"], O.swiglu_ffn(x, w1[0], w3[0], w2[0]), rtol=1e-13)


@pytest.mark.parametrize("S,H,K,E", [(0, 1, 2, 8), (2, 1, 3, 8), (0, 4, 4, 8)])
def test_dispatched_path_equals_definition(S, H, K, E):
    x, ids, wg, w1, w3, w2, conf, emap = tiny_layer(seed=S + H, E=E, K=K, H=H, S=S)
    out = O.layer_forward(x, ids, wg, w1, w3, w2, conf, emap, K=K, H=H, P=2, n_shared=S)
    y2 = O.layer_forward_dispatched(x, out["idx"], out["w"], w1, w3, w2, out["shuf_perm"], S)
    np.testing.assert_allclose(out["y"], y2, rtol=1e-12, atol=1e-12)
    # definition, token by token, with explicit loops
    E_ = w1.shape[0] - S
    for t in range(0, x.shape[0], 7):
        exp = sum(out["w"][t, k] * O.swiglu_ffn(x[t:t + 1], w1[out["idx"][t, k]],
                                                 w3[out["idx"][t, k]], w2[out["idx"][t, k]])[0]
                  for k in range(K))
        for j in range(S):
            exp = exp + O.swiglu_ffn(x[t:t + 1], w1[E_ + j], w3[E_ + j], w2[E_ + j])[0]
        np.testing.assert_allclose(out["y"][t], exp, rtol=1e-12, atol=1e-12)


def test_layer_dispatch_follows_the_shuffle():
    """Inside each expert's segment the layer's dispatch orders pairs by (shuffled slot of
    the token, k), and every row maps back to its pair: checked against the layer's own
    predicted partitions, which differ from token order here."""
    x, ids, wg, w1, w3, w2, conf, emap = tiny_layer(seed=52, T=40, E=8, K=3, P=4)
    out = O.layer_forward(x, ids, wg, w1, w3, w2, conf, emap, K=3, P=4)
    perm, idx, pr, rt, eo = (out[k] for k in ("shuf_perm", "idx", "pair_row", "row_token",
                                              "expert_off"))
    assert not np.array_equal(perm, np.arange(40))
    slot = np.empty(40, np.int64)
    slot[perm] = np.arange(40)
    for e in range(8):
        keys = []
        for r in range(eo[e], eo[e + 1]):
            t = int(rt[r])
            k = [kk for kk in range(3) if pr[t, kk] == r]
            assert len(k) == 1 and idx[t, k[0]] == e
            keys.append((int(slot[t]), k[0]))
        assert keys == sorted(keys)


def _group_picks_ok(logits, idx, K, H):
    """Slots [h K/H, (h+1) K/H) hold group h's K/H best experts (brute force per group)."""
    T, E = logits.shape
    per, kh = E // H, K // H
    for t in range(T):
        for h in range(H):
            got = [int(e) - h * per for e in idx[t, h * kh:(h + 1) * kh]]
            if got != brute_topk(logits[t, h * per:(h + 1) * per].tolist(), kh):
                return False
    return True


@pytest.mark.parametrize("H,K", [(2, 2), (4, 4), (2, 4)])
def test_route_and_layer_pick_within_groups(H, K):
    """The router and the layer both select per group: slot block h holds the K/H best
    experts of group h, by brute force on the float32 logits."""
    x, ids, wg, w1, w3, w2, conf, emap = tiny_layer(seed=60 + H + K, T=40, E=8, K=K, H=H)
    logits, idx, _ = O.route(x, wg, K, H)
    assert _group_picks_ok(logits, idx, K, H)
    out = O.layer_forward(x, ids, wg, w1, w3, w2, conf, emap, K=K, H=H, P=2)
    assert _group_picks_ok(out["logits"], out["idx"], K, H)
    # the plain top-K differs from the grouped picks on this batch
    assert not _group_picks_ok(logits, O.topk_select(logits, K), K, H)


def test_layer_renormalised_weights():
    """With renorm the layer's K weights per token sum to 1 and are the plain weights
    scaled by their sum; the output is the weighted sum with those weights."""
    x, ids, wg, w1, w3, w2, conf, emap = tiny_layer(seed=53, T=30, E=8, K=2)
    plain = O.layer_forward(x, ids, wg, w1, w3, w2, conf, emap, K=2, P=2)
    ren = O.layer_forward(x, ids, wg, w1, w3, w2, conf, emap, K=2, P=2, renorm=True)
    np.testing.assert_allclose(ren["w"].sum(axis=1), 1.0, rtol=1e-13)
    np.testing.assert_allclose(ren["w"], plain["w"] / plain["w"].sum(axis=1, keepdims=True),
                               rtol=1e-13)
    y = np.zeros_like(ren["y"])
    for t in range(30):
        for k in range(2):
            e = ren["idx"][t, k]
            y[t] += ren["w"][t, k] * O.swiglu_ffn(x[t:t + 1], w1[e], w3[e], w2[e])[0]
    np.testing.assert_allclose(ren["y"], y, rtol=1e-12, atol=1e-12)


def test_lossless_invariant():
    """The shuffle and the prediction do not change the layer output (Speculative MoE
    summary: lossless), and permuting tokens permutes the output."""
    x, ids, wg, w1, w3, w2, conf, emap = tiny_layer(seed=3, S=1)
    a = O.layer_forward(x, ids, wg, w1, w3, w2, conf, emap, K=2, P=2, n_shared=1)
    conf2 = np.random.default_rng(99).random(conf.shape).astype(np.float32)
    emap2 = np.array([1, 1, 0, 0, 1, 0, 1, 0], np.int32)
    b = O.layer_forward(x, ids, wg, w1, w3, w2, conf2, emap2, K=2, P=2, n_shared=1)
    assert (a["y"] == b["y"]).all()
    y_disp_b = O.layer_forward_dispatched(x, b["idx"], b["w"], w1, w3, w2, b["shuf_perm"], 1)
    np.testing.assert_allclose(a["y"], y_disp_b, rtol=1e-12, atol=1e-12)
    perm = np.random.default_rng(5).permutation(x.shape[0])
    c = O.layer_forward(x[perm], ids[perm], wg, w1, w3, w2, conf, emap, K=2, P=2, n_shared=1)
    np.testing.assert_allclose(c["y"], a["y"][perm], rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------- prefetch --------


def test_layernorm_golden_and_moments():
    g = load("layernorm_hand.json")
    q = O.layer_norm(np.array(g["d"])[None, :] + np.array(g["r"]), np.ones(4), np.zeros(4))
    np.testing.assert_allclose(q, g["q"], rtol=1e-14)
    v = np.random.default_rng(14).standard_normal((10, 64)) * 3 + 1
    q = O.layer_norm(v, np.ones(64), np.zeros(64))
    np.testing.assert_allclose(q.mean(axis=1), 0, atol=1e-12)
    var = v.var(axis=1)
    np.testing.assert_allclose(q.var(axis=1), var / (var + 1e-5), rtol=1e-12)
    q2 = O.layer_norm(v, 2 * np.ones(64), np.full(64, 0.5))
    np.testing.assert_allclose(q2, 2 * q + 0.5, rtol=1e-12)


def test_hit_count_brute():
    a = np.array([[0, 1, 2], [3, 4, 5]])
    b = np.array([[2, 9, 0], [6, 7, 8]])
    assert O.hit_count(a, b) == 2
    assert O.hit_count(a, a) == 6


def test_prefetch_hit_rate_one_when_default_vector_is_exact():
    rng = np.random.default_rng(15)
    T, d, E, K = 64, 32, 16, 4
    r = rng.standard_normal((T, d))
    d_l = rng.standard_normal(d)
    y = np.tile(d_l, (T, 1))
    wgn = rng.standard_normal((E, d)) / math.sqrt(d)
    out = O.prefetch_predict(r, d_l, y, np.ones(d), np.zeros(d), wgn, K)
    assert out["hits"] == T * K
    out2 = O.prefetch_predict(r, d_l, y, np.ones(d), np.zeros(d), wgn, 8, H=4)
    assert out2["hits"] == T * 8


# ------------------------------------------------------- offline tables ------


def test_profile_confidence_counts_and_oov():
    ids = np.array([0, 0, 1, 3, 3, 3], np.int32)
    idx = np.array([[0, 1], [0, 2], [1, 2], [3, 0], [3, 1], [0, 3]], np.int32)
    emb = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 0.1], [0.0, 2.0], [0.9, 0.0]])
    conf = O.profile_confidence(ids, idx, 5, 4, 2, emb_rows=lambda v: emb[np.asarray(v)])
    np.testing.assert_allclose(conf[0], [1.0, 0.5, 0.5, 0.0])
    np.testing.assert_allclose(conf[1], [0.0, 1.0, 1.0, 0.0])
    np.testing.assert_allclose(conf[3], [2 / 3, 1 / 3, 0.0, 1.0])
    # id 2 is nearest (cosine) to id 0; id 4 points the same way as id 0 exactly
    np.testing.assert_array_equal(conf[2], conf[0])
    np.testing.assert_array_equal(conf[4], conf[0])
    np.testing.assert_allclose(conf[[0, 1, 3]].sum(axis=1), 2.0)      # K per seen row
    empty = O.profile_confidence(np.zeros(0, np.int32), np.zeros((0, 2), np.int32), 3, 4, 2)
    np.testing.assert_allclose(empty, 0.5)


def test_profile_confidence_oov_is_cosine_not_dot_product():
    """An unseen id takes the row of the seen id at the smallest angle, not the largest dot
    product: id 4 = (0.3, 1) is at the same angle to ids 1 = (0, 1) and 3 = (0, 2), so the
    lower id (1) wins, although id 3's dot product is twice id 1's."""
    ids = np.array([0, 1, 3, 3], np.int32)
    idx = np.array([[0, 1], [1, 2], [3, 0], [0, 3]], np.int32)
    emb = np.array([[1.0, 0.0], [0.0, 1.0], [5.0, 5.0], [0.0, 2.0], [0.3, 1.0]])
    conf = O.profile_confidence(ids, idx, 5, 4, 2, emb_rows=lambda v: emb[np.asarray(v)],
                                rows_needed=np.array([4]))
    np.testing.assert_array_equal(conf[4], conf[1])
    assert not np.array_equal(conf[1], conf[3])
    np.testing.assert_allclose(conf[2], 0.5)          # unseen and not needed: K/E


# ------------------------------------------------- inter-layer predictor -----


def test_inter_layer_golden():
    g = load("inter_layer_hand.json")
    emap = np.array(g["expert_part"], np.int32)
    assert O.token_cluster(np.array(g["prev_idx"]), emap, g["P"]).tolist() == g["prev_cluster"]
    assert O.token_cluster(np.array(g["cur_idx"]), emap, g["P"]).tolist() == g["cur_cluster"]
    a = O.markov_table(g["prev_cluster"], g["cur_cluster"], g["P"])
    np.testing.assert_array_equal(a, np.array(g["table_a"], np.float32))
    conf = np.array(g["conf_rows"], np.float32)
    ids = np.array(g["token_ids"])
    assert O.predict_partition(ids, conf, emap, g["P"]).tolist() == g["pred_intra"]
    for case in g["cases"]:
        got = O.predict_partition_inter(ids, conf, emap, g["P"], g["K"],
                                        g["query_prev_cluster"], np.array(case["table_a"]))
        assert got.tolist() == case["pred"], case["why"]


def test_token_cluster_brute_force():
    rng = np.random.default_rng(21)
    P, E, K, T = 5, 20, 6, 200
    idx = O.topk_select(rng.standard_normal((T, E)).astype(np.float32), K)
    emap = rng.integers(0, P, size=E).astype(np.int32)
    got = O.token_cluster(idx, emap, P)
    for t in range(T):
        cnt = [0] * P
        for k in range(K):
            cnt[emap[idx[t, k]]] += 1
        assert got[t] == cnt.index(max(cnt))


def test_markov_table_rows_and_counts():
    rng = np.random.default_rng(22)
    P = 4
    prev = rng.integers(0, P - 1, size=500)           # cluster P-1 never seen before
    cur = rng.integers(0, P, size=500)
    a = O.markov_table(prev, cur, P)
    np.testing.assert_allclose(a.sum(axis=1), 1.0, rtol=1e-6)
    np.testing.assert_allclose(a[P - 1], 1.0 / P)
    for c in range(P - 1):
        n = sum(1 for i in range(500) if prev[i] == c)
        for p in range(P):
            m = sum(1 for i in range(500) if prev[i] == c and cur[i] == p)
            assert abs(a[c, p] - m / n) < 1e-6


def test_inter_never_confident_reduces_to_intra():
    """An all-uniform table A (confidence 1/P) never beats the intra-layer confidence
    max_p score/K >= 1/P (C_p rows of profiled ids sum to K)."""
    rng = np.random.default_rng(23)
    V, E, K, P, T = 30, 12, 3, 4, 300
    idx = O.topk_select(rng.standard_normal((V, E)).astype(np.float32), K)
    conf = O.profile_confidence(np.arange(V), idx, V, E, K)
    emap = (np.arange(E) % P).astype(np.int32)
    ids = rng.integers(0, V, size=T)
    uni = np.full((P, P), 1.0 / P, np.float32)
    prev = rng.integers(0, P, size=T)
    assert np.array_equal(O.predict_partition_inter(ids, conf, emap, P, K, prev, uni),
                          O.predict_partition(ids, conf, emap, P))


def test_inter_prediction_ties_go_to_the_lower_partition():
    """When table A is the more confident source and its row has two largest entries, the
    inter-layer prediction is the lower partition. Intra confidence here: each C_p row is
    spread evenly (score K/P per partition -> 1/P = 1/3 < 0.5)."""
    V, E, K, P = 4, 6, 3, 3
    conf = np.full((V, E), K / E, np.float32)
    emap = (np.arange(E) % P).astype(np.int32)
    a = np.array([[0.0, 0.5, 0.5], [0.5, 0.0, 0.5], [0.5, 0.5, 0.0]], np.float32)
    prev = np.array([0, 1, 2, 0])
    got = O.predict_partition_inter(np.arange(V), conf, emap, P, K, prev, a)
    assert got.tolist() == [1, 0, 0, 1]


def test_speculative_execution_pins():
    """Identical predicted and true routes give zero deviation; changing one token's one
    route changes that token's output by exactly the weighted difference of the two
    experts' outputs (and no other token)."""
    x, ids, wg, w1, w3, w2, conf, emap = tiny_layer(seed=31, E=8, K=2, S=1)
    logits = O.gate_logits(x, wg)
    idx = O.topk_select(logits, 2)
    w = O.gate_weights(logits, idx)
    y_spec, y_true, dev = O.speculative_execution(x, idx, w, idx, w, w1, w3, w2, n_shared=1)
    assert dev == 0.0 and (y_spec == y_true).all()
    idx2 = idx.copy()
    old = int(idx2[5, 1])
    new = (old + 1) % 8 if (old + 1) % 8 != idx2[5, 0] else (old + 2) % 8
    idx2[5, 1] = new
    y2, _, dev2 = O.speculative_execution(x, idx2, w, idx, w, w1, w3, w2, n_shared=1)
    diff = y2 - y_true
    assert np.abs(np.delete(diff, 5, axis=0)).max() < 1e-12
    exp = w[5, 1] * (O.swiglu_ffn(x[5:6], w1[new], w3[new], w2[new])[0]
                     - O.swiglu_ffn(x[5:6], w1[old], w3[old], w2[old])[0])
    np.testing.assert_allclose(diff[5], exp, rtol=1e-10, atol=1e-12)
    assert dev2 > 0


def test_speculative_execution_uses_the_predicted_weights():
    """Same routes, predicted weights twice the true ones, no shared expert: the routed
    output is linear in the weights, so y_spec = 2 y_true exactly and the deviation is 1."""
    x, ids, wg, w1, w3, w2, conf, emap = tiny_layer(seed=32, E=8, K=2, S=0)
    logits = O.gate_logits(x, wg)
    idx = O.topk_select(logits, 2)
    w = O.gate_weights(logits, idx)
    y_spec, y_true, dev = O.speculative_execution(x, idx, 2.0 * w, idx, w, w1, w3, w2)
    np.testing.assert_allclose(y_spec, 2.0 * y_true, rtol=1e-13, atol=0)
    assert abs(dev - 1.0) < 1e-12


# ------------------------------------------------- co-clustering (s-EG) ------


def test_coclustering_cost_hand():
    """Two tokens, four experts, two clusters. act: token 0 fires experts 0,1 (3 and 1
    times), token 1 fires experts 2,3 (2 and 2). Expert map (0,0,1,1) with tokens (0,1):
    nothing remote, loads 4 and 4 -> cost 0. Tokens (0,0): token 1's 4 activations remote
    (of 8 = 0.5), loads 8 and 0 -> imbalance (8 - 4)/4 = 1; theta 0.25 -> 0.25 + 0.375."""
    act = np.array([[3, 1, 0, 0], [0, 0, 2, 2]], float)
    assert O.coclustering_cost(act, [0, 0, 1, 1], [0, 1], 2, 0.25) == 0.0
    assert abs(O.coclustering_cost(act, [0, 0, 1, 1], [0, 0], 2, 0.25) - 0.625) < 1e-15
    # expert map (0,1,0,1): token 0 loses expert 1 (1), token 1 loses expert 2 (2) -> 3/8
    assert abs(O.coclustering_cost(act, [0, 1, 0, 1], [0, 1], 2, 0.0) - 0.375) < 1e-15


def test_coclustering_bruteforce_hand_enumerated():
    """The exhaustive co-clustering search returns the first optimum of a hand-enumerated
    instance (golden/coclustering_hand.json): the cost, the balanced expert map and the
    token map. Each balanced map's best token map and cost, worked by hand, are checked
    through the cost function too."""
    g = load("coclustering_hand.json")
    act = np.array(g["act"], float)
    P, theta = g["P"], g["theta"]
    for row in g["per_map_best"]:
        c = O.coclustering_cost(act, row["expert_part"], row["token_part"], P, theta)
        assert abs(c - row["cost"]) < 1e-12, row
    cost, m, tau = O.coclustering_bruteforce(act, P, theta)
    opt = g["optimum"]
    assert abs(cost - opt["cost"]) < 1e-12
    assert m.tolist() == opt["expert_part"]
    assert tau.tolist() == opt["token_part"]
    assert all(int(np.sum(m == p)) == act.shape[1] // P for p in range(P))


# ------------------------------------------ expert-parallel exchange (EP) ------


@pytest.mark.parametrize("case", ["sts", "contiguous"])
def test_ep_exchange_fig2_golden(case):
    g = load("ep_exchange_fig2_hand.json")
    src = g["pred"] if case == "sts" else None
    sc, ro, pr, rt = O.ep_exchange(np.array(g["routes"]), g["expert_part"], g["P"], src)
    want = g[case]
    assert sc.tolist() == want["send_counts"]
    assert ro.tolist() == want["recv_off"]
    assert rt.tolist() == want["recv_token"]
    assert pr.tolist() == want["pair_recv"]


@pytest.mark.parametrize("T,E,K,P,shuffled", [(1, 4, 2, 2, True), (37, 8, 2, 2, True),
                                               (64, 16, 4, 4, False), (200, 160, 6, 8, True),
                                               (50, 12, 3, 3, False)])
def test_ep_exchange_invariants(T, E, K, P, shuffled):
    """Counts by a direct double loop; the receive layout is a bijection whose segment
    offsets are the scan of those counts read destination-major; the key (dst, src) never
    decreases along it and (t, k) increases inside a segment; the local pairs are the
    alpha count of the same sources."""
    rng = np.random.default_rng(T * 7 + E)
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    emap = rng.integers(0, P, E).astype(np.int32)
    src = rng.integers(0, P, T).astype(np.int32) if shuffled else None
    sc, ro, pr, rt = O.ep_exchange(idx, emap, P, src)
    srcv = src if shuffled else np.array([t * P // T for t in range(T)])
    direct = np.zeros((P, P), int)
    for t in range(T):
        for k in range(K):
            direct[srcv[t], emap[idx[t, k]]] += 1
    assert sc.tolist() == direct.tolist()
    run = [0]
    for q in range(P):
        for p in range(P):
            run.append(run[-1] + direct[p, q])
    assert ro.tolist() == run
    assert sorted(pr.ravel().tolist()) == list(range(T * K))
    keys = []
    for r in range(T * K):
        t, k = divmod(int(np.nonzero(pr.ravel() == r)[0][0]), K)
        assert rt[r] == t
        keys.append((emap[idx[t, k]], srcv[t], t, k))
    assert keys == sorted(keys)
    lar = O.lar_counts(idx, emap, P, src_part=srcv)
    assert int(np.trace(sc)) == int(lar[0])
    assert int(sc.sum()) == T * K


def test_srs_sag_golden_and_round_trip():
    g = load("ep_exchange_fig2_hand.json")["srs"]
    red = O.shuffled_reduce_scatter(np.array(g["x_parts"]), g["shuf_perm"])
    assert red.tolist() == g["reduced_in_slot_order"]
    back = O.shuffled_allgather(red, g["shuf_perm"])
    assert back.ravel().tolist() == [11.0, 22.0, 33.0]
    rng = np.random.default_rng(3)
    xp = rng.standard_normal((3, 40, 5))
    perm = rng.permutation(40)
    # one partial is the plain shuffle gather; the round trip restores token order
    assert np.array_equal(O.shuffled_reduce_scatter(xp[:1], perm), xp[0][perm])
    np.testing.assert_allclose(O.shuffled_allgather(O.shuffled_reduce_scatter(xp, perm), perm),
                               xp[0] + xp[1] + xp[2], rtol=0, atol=1e-15)
