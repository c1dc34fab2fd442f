"""CPU oracle for the single-device MoE-layer forward pass.

TEST INFRASTRUCTURE. This is the slow, plain definition that the CUDA path is
checked against. Only the test suite, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` may import or run it; the product
library never does, and it shares no code, header, table or helper with the
CUDA path (both are fed by the seeded generator, which holds no layer math).

Precision. Values are computed in float64 (numpy; matmul is the only library
primitive used for arithmetic). Where floating point decides an integer, the
decision is taken in float32, the precision the kernels take it in:
  * top-K selection compares float32 logits;
  * predicted-partition scores are float32 sums in ascending expert order.

Sources (page title, section):
  [sMoE]  "Speculative MoE" (research-notes page): §1 background (top-K gating,
          EP dispatch/combine), §2 local activation rate, §3.1 s-TS, Fig. 2,
          §4.1 route prediction (confidence table C_p, OOV fill), §7 glossary (LAR).
  [FoE]   "Federation of Experts (FoE)" (aitrends article): the grouped MoE block
          (E_h, TopK per group on r_full), rho_moe = 1/G, rho_foe = min(H/G, 1),
          A2A volume 2k(G-H)/G and the asymptote kHr/(kH + r(H-1)).
  [SpecE] "Speculating Experts Accelerates Inference for Mixture-of-Experts"
          (gist.science summary): §2.A default vector d_l, quasi-hidden state
          q_l = LN_{l+1}(d_l + r_l), hit rate (§4).

Readings where the pages are silent (each is also listed in the design notes):
  R1 ties in top-K: lower expert index wins; selection on float32 logits;
     output group-major, descending logit within a group.
  R2 weights: softmax over all E experts, w = g[idx], no renormalisation unless
     asked (``renorm``); the same global softmax under grouped routing.
  R3 predicted partition: argmax over partitions of the summed C_p row, lower
     partition wins ties.
  R4 shuffle and dispatch orders are stable (counting sorts).
  R5 FoE source partition of token copy (t, h): see ``foe_source``.
  R6 shared experts: weight 1, excluded from alpha.
  R7 LayerNorm: biased variance, eps = 1e-5.
  R8b a token's cluster at a layer is the partition holding most of its experts
     (lower partition on ties); table A counts cluster transitions between layers.

Parity pins: every function here is checked by tests/test_oracle_pins.py
against brute force, closed forms or hand-computed fixtures.
"""
from __future__ import annotations

import numpy as np
import scipy.special

# ----------------------------------------------------------------------------
# a1/a2: gate GEMM, softmax and (grouped) top-K          [sMoE §1, FoE block]
# ----------------------------------------------------------------------------


def gate_logits(x, w_gate):
    """logits[t, e] = sum_j x[t, j] w_gate[e, j], accumulated in float64, rounded once
    to float32 (the router reads r_full[i]: [FoE]; top-K gating: [sMoE §1])."""
    x64 = np.asarray(x, dtype=np.float64)
    w64 = np.asarray(w_gate, dtype=np.float64)
    return (x64 @ w64.T).astype(np.float32)


def topk_select(logits, K, H=1):
    """Grouped top-K: group h owns experts [h E/H, (h+1) E/H) and picks its K/H best
    experts on its own [FoE grouped block: I_h[i] = TopK over E_h, k/H each].
    H = 1 is ordinary top-K. Repeated argmax; np.argmax returns the first maximum,
    so the lower index wins ties (R1). Output [T, K] int32, group-major."""
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    assert E % H == 0 and K % H == 0 and K // H <= E // H
    assert np.all(np.isfinite(logits)), "logits must be finite"
    per, kh = E // H, K // H
    idx = np.empty((T, K), dtype=np.int32)
    rows = np.arange(T)
    for h in range(H):
        sub = logits[:, h * per:(h + 1) * per]
        taken = np.zeros(sub.shape, dtype=bool)
        for j in range(kh):
            cand = np.where(taken, -np.inf, sub)
            a = np.argmax(cand, axis=1)
            taken[rows, a] = True
            idx[:, h * kh + j] = h * per + a
    return idx


def gate_weights(logits, idx, renorm=False):
    """g = softmax(logits) over all E (float64, max-subtracted); w[t, k] = g[t, idx[t, k]]
    (R2). With renorm the K selected weights are divided by their sum."""
    l64 = np.asarray(logits, dtype=np.float64)
    m = l64.max(axis=1, keepdims=True)
    ex = np.exp(l64 - m)
    g = ex / ex.sum(axis=1, keepdims=True)
    w = np.take_along_axis(g, np.asarray(idx, dtype=np.int64), axis=1)
    if renorm:
        w = w / w.sum(axis=1, keepdims=True)
    return w


def route(x, w_gate, K, H=1, renorm=False):
    """(logits float32 [T,E], idx int32 [T,K], w float64 [T,K])."""
    logits = gate_logits(x, w_gate)
    idx = topk_select(logits, K, H)
    return logits, idx, gate_weights(logits, idx, renorm)


def selection_margin(logits, K, H=1):
    """Per token: the K-th minus the (K+1)-th largest logit (per group, K/H-th minus
    (K/H+1)-th; minimum over groups; +inf where a group is fully selected). Tokens with
    a small margin can flip their route under rounding; end-to-end value checks skip
    them."""
    l64 = np.asarray(logits, dtype=np.float64)
    T, E = l64.shape
    per, kh = E // H, K // H
    margin = np.full(T, np.inf)
    for h in range(H):
        sub = -np.sort(-l64[:, h * per:(h + 1) * per], axis=1)
        if kh < per:
            margin = np.minimum(margin, sub[:, kh - 1] - sub[:, kh])
    return margin


# ----------------------------------------------------------------------------
# a3: predicted partition from the confidence table C_p       [sMoE §4.1, §3.1]
# ----------------------------------------------------------------------------


def predict_partition(token_ids, conf, expert_part, P):
    """pred[t] = argmax_p sum_{e : map[e] = p} C_p[id_t, e] (R3).

    C_p[v, e] = Pr(E_e | token v) is looked up by token id; the scores are float32
    sums over e in ascending order (one float32 add per expert), and np.argmax takes
    the lower partition on ties."""
    ids = np.asarray(token_ids, dtype=np.int64)
    conf = np.asarray(conf, dtype=np.float32)
    emap = np.asarray(expert_part, dtype=np.int64)
    rows = conf[ids]                              # [T, E] float32
    score = np.zeros((len(ids), P), dtype=np.float32)
    for e in range(conf.shape[1]):
        score[:, emap[e]] = score[:, emap[e]] + rows[:, e]   # float32 + float32 -> float32
    return np.argmax(score, axis=1).astype(np.int32)


def token_cluster(idx, expert_part, P):
    """A token's cluster (EP partition) at one layer: the partition holding the most of
    its routed experts, the lower partition on ties (R8b)."""
    dst = np.asarray(expert_part, dtype=np.int64)[np.asarray(idx, dtype=np.int64)]
    counts = np.stack([np.sum(dst == p, axis=1) for p in range(P)], axis=1)
    return np.argmax(counts, axis=1).astype(np.int32)


def markov_table(prev_cluster, cur_cluster, P):
    """Table A of the 2-gram model over a token's cluster sequence [sMoE §4.1
    inter-layer]: A[c, p] = #(tokens in cluster c at the previous layer and p at this
    layer) / #(tokens in cluster c at the previous layer), float32; a row with no tokens
    is uniform 1/P."""
    prev = np.asarray(prev_cluster, dtype=np.int64)
    cur = np.asarray(cur_cluster, dtype=np.int64)
    counts = np.zeros((P, P), dtype=np.float64)
    np.add.at(counts, (prev, cur), 1.0)
    rows = counts.sum(axis=1, keepdims=True)
    a = np.where(rows > 0, counts / np.maximum(rows, 1.0), 1.0 / P)
    return a.astype(np.float32)


def predict_partition_inter(token_ids, conf, expert_part, P, K, prev_cluster, table_a):
    """Intra-layer prediction (predict_partition) and inter-layer prediction (row
    prev_cluster[t] of table A), adopting the more confident one [sMoE §4.1: whichever
    of the two is more confident]. Intra confidence = best partition score / K in float32
    (the C_p row sums to K); inter confidence = the largest entry of the A row; the inter
    prediction (its first largest entry) is adopted only when strictly more confident."""
    ids = np.asarray(token_ids, dtype=np.int64)
    conf = np.asarray(conf, dtype=np.float32)
    emap = np.asarray(expert_part, dtype=np.int64)
    rows = conf[ids]
    score = np.zeros((len(ids), P), dtype=np.float32)
    for e in range(conf.shape[1]):
        score[:, emap[e]] = score[:, emap[e]] + rows[:, e]
    pred_intra = np.argmax(score, axis=1)
    conf_intra = score[np.arange(len(ids)), pred_intra] / np.float32(K)   # float32 division
    a_rows = np.asarray(table_a, dtype=np.float32)[np.asarray(prev_cluster, dtype=np.int64)]
    pred_inter = np.argmax(a_rows, axis=1)
    conf_inter = a_rows[np.arange(len(ids)), pred_inter]
    return np.where(conf_inter > conf_intra, pred_inter, pred_intra).astype(np.int32)


# ----------------------------------------------------------------------------
# a4: speculative token shuffle                           [sMoE §3.1, Fig. 2]
# ----------------------------------------------------------------------------


def token_shuffle(pred, P):
    """Group tokens by predicted partition, keeping token order inside a partition.

    Returns shuf_perm [T] (slot s -> token t) and part_off [P+1], the exclusive prefix
    sum of the partition histogram: partition p owns slots part_off[p]..part_off[p+1]-1."""
    pred = np.asarray(pred, dtype=np.int64)
    counts = np.bincount(pred, minlength=P)
    part_off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    shuf_perm = np.argsort(pred, kind="stable").astype(np.int32)
    return shuf_perm, part_off


# ----------------------------------------------------------------------------
# a5: local activation rate alpha                  [sMoE §2, §7; FoE rho]
# ----------------------------------------------------------------------------


def foe_source(t, h, G, H):
    """Partition holding token copy (t, h) under FoE's grouped layout (R5).

    H >= G: group h, and every token's copy for it, lives on floor(h G / H).
    H <  G: group h spans G/H partitions and its copies are spread round-robin over
    them by token: h (G/H) + (t mod G/H)."""
    if H >= G:
        return (h * G) // H
    return h * (G // H) + (t % (G // H))


def lar_counts(idx, expert_part, P, H=1, src_part=None):
    """[local, total, base_local, max_local] as uint64.

    local      #(t, k) with map[idx[t,k]] == src(t, k): src = src_part[t] when given
               (the token's shuffled partition), else FoE's foe_source(t, k // (K/H)).
    total      T K routed pairs (shared experts excluded, R6).
    base_local the same count with the unshuffled contiguous split src = floor(t P / T).
    max_local  sum over t of max_p #{k : map[idx[t,k]] = p}: the best any single
               source partition per token could do."""
    idx = np.asarray(idx, dtype=np.int64)
    emap = np.asarray(expert_part, dtype=np.int64)
    T, K = idx.shape
    kh = K // H
    dst = emap[idx]                                    # [T, K]
    t = np.arange(T)
    if src_part is not None:
        src = np.repeat(np.asarray(src_part, dtype=np.int64)[:, None], K, axis=1)
    else:
        src = np.empty((T, K), dtype=np.int64)
        for k in range(K):
            src[:, k] = [foe_source(int(tt), k // kh, P, H) for tt in t]
    local = int(np.sum(dst == src))
    base = (t * P) // T
    base_local = int(np.sum(dst == base[:, None]))
    per_part = np.stack([np.sum(dst == p, axis=1) for p in range(P)], axis=1)
    max_local = int(per_part.max(axis=1).sum())
    return np.array([local, T * K, base_local, max_local], dtype=np.uint64)


# ----------------------------------------------------------------------------
# a6: expert permutation / dispatch into per-expert buffers      [sMoE §1 EP]
# ----------------------------------------------------------------------------


def expert_dispatch(idx, E, shuf_perm=None):
    """Sort the T K (token, k) pairs by expert, stably in (shuffled slot s, k) order.

    Returns expert_off [E+1] (exclusive scan of the per-expert pair counts),
    pair_row [T, K] (row of pair (t, k) in the expert-contiguous buffer) and
    row_token [T K] (token of each row). Without a shuffle, s = t."""
    idx = np.asarray(idx, dtype=np.int64)
    T, K = idx.shape
    perm = np.arange(T) if shuf_perm is None else np.asarray(shuf_perm, dtype=np.int64)
    # pairs enumerated in (s, k) order
    tok_of_q = np.repeat(perm, K)
    k_of_q = np.tile(np.arange(K), T)
    exp_of_q = idx[tok_of_q, k_of_q]
    order = np.argsort(exp_of_q, kind="stable")        # row r -> pair q
    counts = np.bincount(exp_of_q, minlength=E)
    expert_off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    pair_row = np.empty((T, K), dtype=np.int32)
    pair_row[tok_of_q[order], k_of_q[order]] = np.arange(T * K, dtype=np.int32)
    row_token = tok_of_q[order].astype(np.int32)
    return expert_off, pair_row, row_token


# ----------------------------------------------------------------------------
# a7/a8: SwiGLU expert FFN
# ----------------------------------------------------------------------------


def silu(z):
    """silu(z) = z * sigmoid(z); sigmoid from scipy's expit (a library primitive)."""
    z = np.asarray(z, dtype=np.float64)
    return z * scipy.special.expit(z)


def swiglu_ffn(x_rows, w1_e, w3_e, w2_e):
    """y = (silu(x W1^T) * (x W3^T)) W2^T in float64, W1/W3 [F, d], W2 [d, F]."""
    x64 = np.asarray(x_rows, dtype=np.float64)
    a = x64 @ np.asarray(w1_e, dtype=np.float64).T
    b = x64 @ np.asarray(w3_e, dtype=np.float64).T
    h = silu(a) * b
    return h @ np.asarray(w2_e, dtype=np.float64).T


def swiglu_hidden(x_rows, w1_e, w3_e):
    """The SwiGLU hidden activation silu(x W1^T) * (x W3^T), float64."""
    x64 = np.asarray(x_rows, dtype=np.float64)
    a = x64 @ np.asarray(w1_e, dtype=np.float64).T
    b = x64 @ np.asarray(w3_e, dtype=np.float64).T
    return silu(a) * b


# ----------------------------------------------------------------------------
# a9: combine back into token order                  [sMoE §1 EP combine; FoE sum]
# ----------------------------------------------------------------------------


def combine(y_rows, pair_row, w, y_shared=None):
    """y[t] = sum_{k=0}^{K-1} w[t,k] y_rows[pair_row[t,k]] + sum_j y_shared[j, t], float64,
    in original token order. y_rows is the expert-contiguous output buffer."""
    y_rows = np.asarray(y_rows, dtype=np.float64)
    pair_row = np.asarray(pair_row, dtype=np.int64)
    w = np.asarray(w, dtype=np.float64)
    T, K = pair_row.shape
    y = np.zeros((T, y_rows.shape[1]), dtype=np.float64)
    for k in range(K):
        y += w[:, k:k + 1] * y_rows[pair_row[:, k]]
    if y_shared is not None:
        for j in range(y_shared.shape[0]):
            y += np.asarray(y_shared[j], dtype=np.float64)
    return y


# ----------------------------------------------------------------------------
# Whole layer
# ----------------------------------------------------------------------------


def moe_output(x, idx, w, w1, w3, w2, n_shared=0):
    """The layer's defining sum, token by token through its own experts:
    y[t] = sum_k w[t,k] FFN_{idx[t,k]}(x[t]) + sum_j FFN_{E+j}(x[t]).
    Rows routed to one expert are evaluated together (one matmul per expert)."""
    x64 = np.asarray(x, dtype=np.float64)
    idx = np.asarray(idx, dtype=np.int64)
    T, K = idx.shape
    E = w1.shape[0] - n_shared
    y = np.zeros_like(x64)
    for e in range(E):
        tt, kk = np.nonzero(idx == e)
        if len(tt) == 0:
            continue
        ye = swiglu_ffn(x64[tt], w1[e], w3[e], w2[e])
        np.add.at(y, tt, w[tt, kk][:, None] * ye)
    for j in range(n_shared):
        y += swiglu_ffn(x64, w1[E + j], w3[E + j], w2[E + j])
    return y


def layer_forward(x, token_ids, w_gate, w1, w3, w2, conf, expert_part, *, K, H=1, P,
                  n_shared=0, renorm=False, logits=None):
    """Every step of the layer, in order, as plain definitions. Returns a dict with
    logits, idx, w, pred, shuf_perm, part_off, lar, expert_off, pair_row, row_token and y.
    If ``logits`` is given the gate GEMM is skipped and those float32 logits are routed."""
    if logits is None:
        logits = gate_logits(x, w_gate)
    idx = topk_select(logits, K, H)
    w = gate_weights(logits, idx, renorm)
    E = np.asarray(w_gate).shape[0]
    pred = predict_partition(token_ids, conf, expert_part, P)
    shuf_perm, part_off = token_shuffle(pred, P)
    lar = lar_counts(idx, expert_part, P, H, src_part=pred)
    expert_off, pair_row, row_token = expert_dispatch(idx, E, shuf_perm)
    y = moe_output(x, idx, w, w1, w3, w2, n_shared)
    return dict(logits=logits, idx=idx, w=w, pred=pred, shuf_perm=shuf_perm,
                part_off=part_off, lar=lar, expert_off=expert_off, pair_row=pair_row,
                row_token=row_token, y=y)


def layer_forward_dispatched(x, idx, w, w1, w3, w2, shuf_perm, n_shared=0):
    """The same output computed the way an expert-parallel layer moves data: shuffle
    rows by shuf_perm, gather pairs into expert-contiguous rows, run each expert on its
    segment, then combine through pair_row. Equal to moe_output (losslessness)."""
    x64 = np.asarray(x, dtype=np.float64)
    E = w1.shape[0] - n_shared
    expert_off, pair_row, row_token = expert_dispatch(idx, E, shuf_perm)
    x_disp = x64[row_token]
    y_rows = np.zeros_like(x_disp)
    for e in range(E):
        lo, hi = expert_off[e], expert_off[e + 1]
        if hi > lo:
            y_rows[lo:hi] = swiglu_ffn(x_disp[lo:hi], w1[e], w3[e], w2[e])
    y_sh = None
    if n_shared:
        y_sh = np.stack([swiglu_ffn(x64, w1[E + j], w3[E + j], w2[E + j])
                         for j in range(n_shared)])
    return combine(y_rows, pair_row, w, y_sh)


# ----------------------------------------------------------------------------
# Expert-parallel exchange between P simulated devices   [sMoE §1 EP; §3.1 SRS/SAG]
# ----------------------------------------------------------------------------


def ep_exchange(idx, expert_part, P, src_part=None):
    """The expert-parallel all-to-all dispatch that P devices would run [sMoE §1: each
    token is sent from its device to the devices of its K experts, and the results come
    back the same way]. Token t sits on device src(t): src_part[t] (the s-TS predicted
    partition, §3.1), or the contiguous split floor(t P / T) when src_part is None.
    Pair (t, k) goes to device dst = map[idx[t, k]]; a pair with dst == src stays local.

    Device q's receive buffer holds its pairs from source 0, then source 1, ...; inside
    one (dst, src) segment the pairs keep the source's token order, then k (what an
    all2allv delivers from send buffers laid out that way). All P receive buffers are
    concatenated, device 0 first, so the pairs are sorted by the key (dst, src, t, k).

    Returns send_counts [P, P] int32 (pairs from device p to device q), recv_off
    [P*P + 1] int32 (segment (dst q, src p) is rows recv_off[q P + p] .. recv_off[q P +
    p + 1]), pair_recv [T, K] int32 (row of pair (t, k)) and recv_token [T K] int32
    (token of each row)."""
    idx = np.asarray(idx, dtype=np.int64)
    emap = np.asarray(expert_part, dtype=np.int64)
    T, K = idx.shape
    t = np.arange(T)
    src = (t * P) // max(T, 1) if src_part is None else np.asarray(src_part, dtype=np.int64)
    tok = np.repeat(t, K)                      # pairs enumerated in (t, k) order
    kk = np.tile(np.arange(K), T)
    dst = emap[idx[tok, kk]]
    key = dst * P + src[tok]
    order = np.argsort(key, kind="stable")     # receive row r -> pair
    counts = np.bincount(key, minlength=P * P)
    recv_off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    send_counts = counts.reshape(P, P).T.astype(np.int32)   # [src, dst]
    pair_recv = np.empty((T, K), dtype=np.int32)
    pair_recv[tok[order], kk[order]] = np.arange(T * K, dtype=np.int32)
    return send_counts, recv_off, pair_recv, tok[order].astype(np.int32)


def shuffled_reduce_scatter(x_parts, shuf_perm):
    """SRS [sMoE §3.1]: the R tensor-parallel partial sums of the activations are added
    and each token lands in the slot the speculative shuffle gave it, so partition p
    receives the reduced rows of the tokens predicted for it (slots part_off[p] ..).
    x_parts [R, T, d]; returns float64 [T, d] in slot order."""
    x = np.asarray(x_parts, dtype=np.float64)
    return x.sum(axis=0)[np.asarray(shuf_perm, dtype=np.int64)]


def shuffled_allgather(y_shuf, shuf_perm):
    """SAG [sMoE §3.1]: rows held in slot order are returned to token order,
    y[shuf_perm[s]] = y_shuf[s]."""
    y_shuf = np.asarray(y_shuf)
    y = np.empty_like(y_shuf)
    y[np.asarray(shuf_perm, dtype=np.int64)] = y_shuf
    return y


# ----------------------------------------------------------------------------
# a10: next-layer prefetch predictor                                 [SpecE §2.A]
# ----------------------------------------------------------------------------


def layer_norm(v, gamma, beta, eps=1e-5):
    """LN over the last axis, biased variance (R7), float64."""
    v = np.asarray(v, dtype=np.float64)
    mu = v.mean(axis=-1, keepdims=True)
    var = ((v - mu) ** 2).mean(axis=-1, keepdims=True)
    return (v - mu) / np.sqrt(var + eps) * np.asarray(gamma, np.float64) + np.asarray(beta, np.float64)


def hit_count(pred_idx, true_idx):
    """sum_t |pred_t intersect true_t| over the routed expert sets."""
    pred_idx = np.asarray(pred_idx)
    true_idx = np.asarray(true_idx)
    return int(sum(len(set(p.tolist()) & set(q.tolist())) for p, q in zip(pred_idx, true_idx)))


def prefetch_predict(r, d_l, y, gamma, beta, w_gate_next, K, H=1, eps=1e-5,
                     logits_q=None, logits_s=None):
    """q = LN(d_l + r) predicts the next router input s = LN(r + y); both are routed by
    the next layer's gate with the layer's routing rule. Returns q, s, the float32
    logits of both, the predicted and true routes and the hit count.
    If logits_q / logits_s are given, the routes are selected from them instead."""
    q = layer_norm(np.asarray(d_l, np.float64)[None, :] + np.asarray(r, np.float64), gamma, beta, eps)
    s = layer_norm(np.asarray(r, np.float64) + np.asarray(y, np.float64), gamma, beta, eps)
    if logits_q is None:
        logits_q = gate_logits(q, w_gate_next)
    if logits_s is None:
        logits_s = gate_logits(s, w_gate_next)
    pred_idx = topk_select(logits_q, K, H)
    true_idx = topk_select(logits_s, K, H)
    return dict(q=q, s=s, logits_q=logits_q, logits_s=logits_s, pred_idx=pred_idx,
                true_idx=true_idx, hits=hit_count(pred_idx, true_idx))


def speculative_execution(s_rows, pred_idx, pred_w, true_idx, true_w, w1, w3, w2, n_shared=0):
    """[SpecE §2.B] Run the experts predicted from q (weights from q's logits) instead of
    the router's true ones on the same next-layer input s. Returns the speculative output,
    the true output and the relative Frobenius deviation between them."""
    y_spec = moe_output(s_rows, pred_idx, pred_w, w1, w3, w2, n_shared)
    y_true = moe_output(s_rows, true_idx, true_w, w1, w3, w2, n_shared)
    dev = float(np.linalg.norm(y_spec - y_true) / max(np.linalg.norm(y_true), 1e-300))
    return y_spec, y_true, dev


# ----------------------------------------------------------------------------
# Offline tables                                             [sMoE §4.1, Fig. 3]
# ----------------------------------------------------------------------------


def profile_confidence(profile_ids, profile_idx, vocab, E, K, emb_rows=None, rows_needed=None):
    """Token-expert confidence table C_p [vocab, E] float32.

    C_p[v, e] = #(profile occurrences of v whose route includes e) / #(occurrences of v).
    An id never seen in the profile takes the row of the seen id whose embedding is
    cosine-nearest (lower id wins ties); with no seen ids every row is K/E.
    ``emb_rows(ids) -> array [len(ids), d]`` supplies embeddings; ``rows_needed``
    limits the nearest-neighbour fill to those ids (other unseen rows stay K/E)."""
    ids = np.asarray(profile_ids, dtype=np.int64)
    idx = np.asarray(profile_idx, dtype=np.int64)
    occ = np.bincount(ids, minlength=vocab).astype(np.float64)
    hits = np.zeros((vocab, E), dtype=np.float64)
    for k in range(idx.shape[1]):
        np.add.at(hits, (ids, idx[:, k]), 1.0)
    conf = np.full((vocab, E), K / E, dtype=np.float64)
    seen = np.nonzero(occ > 0)[0]
    conf[seen] = hits[seen] / occ[seen, None]
    if len(seen) and emb_rows is not None:
        targets = np.arange(vocab) if rows_needed is None else np.unique(np.asarray(rows_needed))
        unseen = targets[occ[targets] == 0]
        if len(unseen):
            es = np.asarray(emb_rows(seen), dtype=np.float64)
            es = es / np.linalg.norm(es, axis=1, keepdims=True)
            for lo in range(0, len(unseen), 1024):
                blk = unseen[lo:lo + 1024]
                eu = np.asarray(emb_rows(blk), dtype=np.float64)
                eu = eu / np.linalg.norm(eu, axis=1, keepdims=True)
                nn = np.argmax(eu @ es.T, axis=1)     # first maximum: lower seen id
                conf[blk] = conf[seen[nn]]
    return conf.astype(np.float32)


def coclustering_cost(act, expert_part, token_part, P, theta):
    """Objective of balanced token-expert co-clustering [sMoE §4.2]: theta times the load
    imbalance (token frequency per cluster: (max - mean) / mean) plus (1 - theta) times the
    remote activations (share of token-expert activations whose token and expert sit in
    different clusters). act [V, E]: activation counts of each token id and expert."""
    act = np.asarray(act, dtype=np.float64)
    m = np.asarray(expert_part, dtype=np.int64)
    tau = np.asarray(token_part, dtype=np.int64)
    freq = act.sum(axis=1)
    load = np.array([freq[tau == p].sum() for p in range(P)])
    mean = load.mean()
    imbalance = (load.max() - mean) / mean if mean > 0 else 0.0
    remote = sum(act[v, e] for v in range(act.shape[0]) for e in range(act.shape[1])
                 if m[e] != tau[v])
    total = act.sum()
    return theta * imbalance + (1.0 - theta) * (remote / total if total > 0 else 0.0)


def coclustering_bruteforce(act, P, theta):
    """Exact optimum of coclustering_cost over every balanced expert map (E/P experts per
    cluster) and every token map, for tiny instances. Returns (cost, expert_part, token_part)."""
    import itertools
    act = np.asarray(act, dtype=np.float64)
    V, E = act.shape
    best = (np.inf, None, None)
    for m in itertools.product(range(P), repeat=E):
        if any(m.count(p) != E // P for p in range(P)):
            continue
        for tau in itertools.product(range(P), repeat=V):
            c = coclustering_cost(act, m, tau, P, theta)
            if c < best[0] - 1e-15:
                best = (c, np.array(m, np.int32), np.array(tau, np.int32))
    return best


# ----------------------------------------------------------------------------
# Closed forms printed on the pages                                       [FoE]
# ----------------------------------------------------------------------------


def rho_moe(G):
    """Fraction of a token's routes resolved locally under uniform routing: 1/G."""
    return 1.0 / G


def rho_foe(H, G):
    """FoE's locally resolved fraction: min(H/G, 1)."""
    return min(H / G, 1.0)


def a2a_volume_intra(k, G, H):
    """Intra-node all-to-all volume per token under FoE, both ways: 2k(G-H)/G."""
    return 2.0 * k * (G - H) / G


def foe_asymptote(k, H, r):
    """T_moe / T_foe -> kHr / (kH + r(H-1)) with bandwidth ratio r = B_intra / B_inter."""
    return k * H * r / (k * H + r * (H - 1))
