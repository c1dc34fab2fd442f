"""The pins must be able to fail: each case below plants one plausible mistake (a dropped
term, a wrong sign, index or axis, a transposed operand, a broken tie rule) in a copy of
the CPU oracle and runs tests/test_oracle_pins.py against that copy, which must fail.

The copy lives in a temporary directory; the oracle itself is never modified. A control
run of the unmodified copy must pass, so a failure can only come from the planted change.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE_SRC = os.path.join(ROOT, "oracle", "smoe_oracle.py")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# (name, text in the oracle, replacement). Each text occurs exactly once.
MUTATIONS = [
    # gate GEMM and selection
    ("gate_logits: experts in reverse order",
     "w64 = np.asarray(w_gate, dtype=np.float64)",
     "w64 = np.asarray(w_gate, dtype=np.float64)[::-1]"),
    ("gate_logits: dot product over a shifted feature",
     "return (x64 @ w64.T).astype(np.float32)",
     "return (x64 @ np.roll(w64, 1, axis=1).T).astype(np.float32)"),
    ("topk_select: higher index wins ties",
     "a = np.argmax(cand, axis=1)",
     "a = cand.shape[1] - 1 - np.argmax(cand[:, ::-1], axis=1)"),
    ("topk_select: group offset dropped",
     "idx[:, h * kh + j] = h * per + a",
     "idx[:, h * kh + j] = a"),
    ("topk_select: taken experts not masked",
     "cand = np.where(taken, -np.inf, sub)",
     "cand = np.where(taken, np.float32(-1e30), sub) if j == 0 else sub"),
    ("topk_select: slot order within a group reversed",
     "idx[:, h * kh + j] = h * per + a",
     "idx[:, h * kh + (kh - 1 - j)] = h * per + a"),
    ("topk_select: selection on float64 instead of float32 logits",
     "    logits = np.asarray(logits, dtype=np.float32)\n    T, E = logits.shape\n    assert E % H",
     "    logits = np.asarray(logits, dtype=np.float64)\n    T, E = logits.shape\n    assert E % H"),
    ("gate_logits: not rounded to float32",
     "return (x64 @ w64.T).astype(np.float32)",
     "return (x64 @ w64.T)"),
    ("selection_margin: maximum over groups instead of minimum",
     "margin = np.minimum(margin, sub[:, kh - 1] - sub[:, kh])",
     "margin = np.where(np.isinf(margin), sub[:, kh - 1] - sub[:, kh],"
     " np.maximum(margin, sub[:, kh - 1] - sub[:, kh]))"),
    ("gate_weights: softmax over tokens instead of experts",
     "g = ex / ex.sum(axis=1, keepdims=True)",
     "g = ex / ex.sum(axis=0, keepdims=True)"),
    ("gate_weights: renormalisation dropped",
     "w = w / w.sum(axis=1, keepdims=True)",
     "w = w"),
    ("gate_weights: sign of the logits flipped",
     "ex = np.exp(l64 - m)",
     "ex = np.exp(m - l64)"),
    ("selection_margin: off by one rank",
     "margin = np.minimum(margin, sub[:, kh - 1] - sub[:, kh])",
     "margin = np.minimum(margin, sub[:, kh - 1] - sub[:, -1])"),
    # predicted partition, clusters, table A
    ("predict_partition: higher partition wins ties",
     "    return np.argmax(score, axis=1).astype(np.int32)\n\n\ndef token_cluster",
     "    return (P - 1 - np.argmax(score[:, ::-1], axis=1)).astype(np.int32)\n\n\n"
     "def token_cluster"),
    ("predict_partition: scores overwritten, not summed",
     "        score[:, emap[e]] = score[:, emap[e]] + rows[:, e]   # float32",
     "        score[:, emap[e]] = rows[:, e]   # float32"),
    ("predict_partition: scores summed in float64",
     "    score = np.zeros((len(ids), P), dtype=np.float32)\n    for e in range(conf.shape[1]):\n"
     "        score[:, emap[e]] = score[:, emap[e]] + rows[:, e]   # float32",
     "    score = np.zeros((len(ids), P), dtype=np.float64)\n    for e in range(conf.shape[1]):\n"
     "        score[:, emap[e]] = score[:, emap[e]] + rows[:, e]   # float32"),
    ("predict_partition: experts summed in descending order",
     "    for e in range(conf.shape[1]):\n        score[:, emap[e]] = score[:, emap[e]] + rows[:, e]   # float32",
     "    for e in reversed(range(conf.shape[1])):\n        score[:, emap[e]] = score[:, emap[e]] + rows[:, e]   # float32"),
    ("predict_partition: expert map ignored",
     "        score[:, emap[e]] = score[:, emap[e]] + rows[:, e]   # float32",
     "        score[:, e % P] = score[:, e % P] + rows[:, e]   # float32"),
    ("token_cluster: higher partition wins ties",
     "    return np.argmax(counts, axis=1).astype(np.int32)",
     "    return (P - 1 - np.argmax(counts[:, ::-1], axis=1)).astype(np.int32)"),
    ("markov_table: transposed counts",
     "np.add.at(counts, (prev, cur), 1.0)",
     "np.add.at(counts, (cur, prev), 1.0)"),
    ("markov_table: empty row left at zero",
     "a = np.where(rows > 0, counts / np.maximum(rows, 1.0), 1.0 / P)",
     "a = np.where(rows > 0, counts / np.maximum(rows, 1.0), 0.0)"),
    ("predict_partition_inter: inter wins ties",
     "np.where(conf_inter > conf_intra, pred_inter, pred_intra)",
     "np.where(conf_inter >= conf_intra, pred_inter, pred_intra)"),
    ("predict_partition_inter: intra confidence not divided by K",
     "conf_intra = score[np.arange(len(ids)), pred_intra] / np.float32(K)",
     "conf_intra = score[np.arange(len(ids)), pred_intra]"),
    # shuffle, alpha, dispatch
    ("token_shuffle: unstable within a partition",
     'shuf_perm = np.argsort(pred, kind="stable").astype(np.int32)',
     'shuf_perm = (len(pred) - 1 - np.argsort(pred[::-1], kind="stable")).astype(np.int32)'),
    ("token_shuffle: offsets of the reversed histogram",
     "part_off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)\n    shuf_perm",
     "part_off = np.concatenate([[0], np.cumsum(counts[::-1])]).astype(np.int32)\n"
     "    shuf_perm"),
    ("foe_source: wrong group stride",
     "return h * (G // H) + (t % (G // H))",
     "return h * H + (t % (G // H))"),
    ("foe_source: H >= G branch off by one group",
     "return (h * G) // H",
     "return ((h + 1) * G) // H % G"),
    ("lar_counts: base split round-robin instead of contiguous",
     "base = (t * P) // T",
     "base = t % P"),
    ("lar_counts: max over tokens instead of partitions",
     "max_local = int(per_part.max(axis=1).sum())",
     "max_local = int(per_part.max(axis=0).sum())"),
    ("lar_counts: FoE group index from k mod K/H",
     "src[:, k] = [foe_source(int(tt), k // kh, P, H) for tt in t]",
     "src[:, k] = [foe_source(int(tt), k % H, P, H) for tt in t]"),
    ("expert_dispatch: pairs in (k, s) order",
     "tok_of_q = np.repeat(perm, K)\n    k_of_q = np.tile(np.arange(K), T)",
     "tok_of_q = np.tile(perm, K)\n    k_of_q = np.repeat(np.arange(K), T)"),
    ("expert_dispatch: unstable sort by expert",
     'order = np.argsort(exp_of_q, kind="stable")',
     'order = np.argsort(exp_of_q, kind="quicksort")'),
    ("lar_counts: total counts a shared expert per token",
     "return np.array([local, T * K, base_local, max_local], dtype=np.uint64)",
     "return np.array([local, T * (K + 1), base_local, max_local], dtype=np.uint64)"),
    ("foe_source: H >= G groups spread round-robin",
     "return (h * G) // H",
     "return h % G"),
    ("expert_dispatch: shuffle ignored",
     "perm = np.arange(T) if shuf_perm is None else np.asarray(shuf_perm, dtype=np.int64)",
     "perm = np.arange(T)"),
    ("expert_dispatch: offsets shifted by one expert",
     "expert_off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)",
     "expert_off = np.concatenate([[0], np.cumsum(np.roll(counts, 1))]).astype(np.int32)"),
    # FFN, combine, layer
    ("silu: z factor dropped",
     "return z * scipy.special.expit(z)",
     "return scipy.special.expit(z)"),
    ("silu: sign of the sigmoid argument",
     "return z * scipy.special.expit(z)",
     "return z * scipy.special.expit(-z)"),
    ("swiglu_ffn: W1 and W3 swapped",
     "    h = silu(a) * b\n    return h @",
     "    h = a * silu(b)\n    return h @"),
    ("swiglu_hidden: W1 and W3 swapped",
     "    return silu(a) * b\n",
     "    return a * silu(b)\n"),
    ("combine: routing weight dropped",
     "y += w[:, k:k + 1] * y_rows[pair_row[:, k]]",
     "y += y_rows[pair_row[:, k]]"),
    ("combine: shared experts dropped",
     "            y += np.asarray(y_shared[j], dtype=np.float64)",
     "            pass"),
    ("moe_output: weight of the first slot for every slot",
     "np.add.at(y, tt, w[tt, kk][:, None] * ye)",
     "np.add.at(y, tt, w[tt, 0][:, None] * ye)"),
    ("moe_output: shared expert takes a routed expert's weights",
     "        y += swiglu_ffn(x64, w1[E + j], w3[E + j], w2[E + j])\n    return y",
     "        y += swiglu_ffn(x64, w1[j], w3[j], w2[j])\n    return y"),
    ("layer_forward: alpha from the unshuffled rule",
     "lar = lar_counts(idx, expert_part, P, H, src_part=pred)",
     "lar = lar_counts(idx, expert_part, P, H)"),
    # prefetch predictor
    ("layer_norm: eps dropped",
     "return (v - mu) / np.sqrt(var + eps)",
     "return (v - mu) / np.sqrt(var)"),
    ("route: groups dropped",
     "    idx = topk_select(logits, K, H)\n    return logits, idx, gate_weights(logits, idx, renorm)",
     "    idx = topk_select(logits, K)\n    return logits, idx, gate_weights(logits, idx, renorm)"),
    ("layer_forward: groups dropped",
     "    idx = topk_select(logits, K, H)\n    w = gate_weights(logits, idx, renorm)\n    E =",
     "    idx = topk_select(logits, K)\n    w = gate_weights(logits, idx, renorm)\n    E ="),
    ("prefetch_predict: true routes without groups",
     "true_idx = topk_select(logits_s, K, H)",
     "true_idx = topk_select(logits_s, K)"),
    ("predict_partition_inter: last largest entry of the A row",
     "pred_inter = np.argmax(a_rows, axis=1)",
     "pred_inter = P - 1 - np.argmax(a_rows[:, ::-1], axis=1)"),
    ("layer_forward: dispatch ignores the shuffle",
     "expert_off, pair_row, row_token = expert_dispatch(idx, E, shuf_perm)\n    y = moe_output",
     "expert_off, pair_row, row_token = expert_dispatch(idx, E)\n    y = moe_output"),
    ("layer_forward: renormalisation not passed on",
     "    w = gate_weights(logits, idx, renorm)\n    E = np.asarray(w_gate).shape[0]",
     "    w = gate_weights(logits, idx)\n    E = np.asarray(w_gate).shape[0]"),
    ("coclustering_cost: imbalance from max - min",
     "imbalance = (load.max() - mean) / mean if mean > 0 else 0.0",
     "imbalance = (load.max() - load.min()) / mean if mean > 0 else 0.0"),
    ("coclustering_cost: local activations counted as remote",
     "if m[e] != tau[v])",
     "if m[e] == tau[v])"),
    ("markov_table: rows normalised by column sums",
     "rows = counts.sum(axis=1, keepdims=True)",
     "rows = counts.sum(axis=0, keepdims=True)"),
    ("layer_norm: eps added outside the square root",
     "return (v - mu) / np.sqrt(var + eps)",
     "return (v - mu) / (np.sqrt(var) + eps)"),
    ("prefetch_predict: residual dropped from the true next input",
     "s = layer_norm(np.asarray(r, np.float64) + np.asarray(y, np.float64), gamma, beta, eps)",
     "s = layer_norm(np.asarray(y, np.float64), gamma, beta, eps)"),
    ("speculative_execution: deviation relative to the speculative output",
     "dev = float(np.linalg.norm(y_spec - y_true) / max(np.linalg.norm(y_true), 1e-300))",
     "dev = float(np.linalg.norm(y_spec - y_true) / max(np.linalg.norm(y_spec), 1e-300))"),
    ("layer_norm: unbiased variance",
     "var = ((v - mu) ** 2).mean(axis=-1, keepdims=True)",
     "var = ((v - mu) ** 2).sum(axis=-1, keepdims=True) / (v.shape[-1] - 1)"),
    ("layer_norm: gamma and beta swapped",
     "* np.asarray(gamma, np.float64) + np.asarray(beta, np.float64)",
     "* np.asarray(beta, np.float64) + np.asarray(gamma, np.float64)"),
    ("prefetch_predict: default vector dropped",
     "q = layer_norm(np.asarray(d_l, np.float64)[None, :] + np.asarray(r, np.float64)",
     "q = layer_norm(np.asarray(r, np.float64)"),
    ("hit_count: union instead of intersection",
     "len(set(p.tolist()) & set(q.tolist()))",
     "len(set(p.tolist()) | set(q.tolist()))"),
    ("speculative_execution: true weights on the predicted routes",
     "y_spec = moe_output(s_rows, pred_idx, pred_w, w1, w3, w2, n_shared)",
     "y_spec = moe_output(s_rows, pred_idx, true_w, w1, w3, w2, n_shared)"),
    # offline tables and closed forms
    ("profile_confidence: divided by all occurrences",
     "conf[seen] = hits[seen] / occ[seen, None]",
     "conf[seen] = hits[seen] / occ.sum()"),
    ("profile_confidence: farthest id fills unseen rows",
     "nn = np.argmax(eu @ es.T, axis=1)",
     "nn = np.argmin(eu @ es.T, axis=1)"),
    ("profile_confidence: nearest by dot product instead of cosine",
     "            es = es / np.linalg.norm(es, axis=1, keepdims=True)\n",
     "            es = es\n"),
    ("profile_confidence: fill 1/E instead of K/E",
     "conf = np.full((vocab, E), K / E, dtype=np.float64)",
     "conf = np.full((vocab, E), 1.0 / E, dtype=np.float64)"),
    ("coclustering_cost: theta on the wrong term",
     "return theta * imbalance + (1.0 - theta) * (remote / total",
     "return (1.0 - theta) * imbalance + theta * (remote / total"),
    ("coclustering_bruteforce: balance constraint dropped",
     "if any(m.count(p) != E // P for p in range(P)):",
     "if False:"),
    ("coclustering_bruteforce: the last of equal-cost optima kept",
     "if c < best[0] - 1e-15:",
     "if c <= best[0] + 1e-15:"),
    ("coclustering_bruteforce: the last token never tried outside cluster 0",
     "for tau in itertools.product(range(P), repeat=V):",
     "for tau in itertools.product(*([range(P)] * (V - 1) + [range(1)])):"),
    ("ep_exchange: receive layout source-major",
     "key = dst * P + src[tok]",
     "key = src[tok] * P + dst"),
    ("ep_exchange: send counts not transposed to [src, dst]",
     "send_counts = counts.reshape(P, P).T.astype(np.int32)",
     "send_counts = counts.reshape(P, P).astype(np.int32)"),
    ("ep_exchange: contiguous split off by one",
     "src = (t * P) // max(T, 1) if src_part is None",
     "src = (t * P) // (T + 1) if src_part is None"),
    ("ep_exchange: pairs enumerated k-major",
     "    tok = np.repeat(t, K)                      # pairs enumerated in (t, k) order\n"
     "    kk = np.tile(np.arange(K), T)",
     "    tok = np.tile(t, K)                      # pairs enumerated in (t, k) order\n"
     "    kk = np.repeat(np.arange(K), T)"),
    ("shuffled_reduce_scatter: summed over tokens instead of ranks",
     "return x.sum(axis=0)[np.asarray(shuf_perm, dtype=np.int64)]",
     "return x.sum(axis=1, keepdims=True).repeat(x.shape[1], 1)[0][np.asarray(shuf_perm, dtype=np.int64)]"),
    ("shuffled_allgather: gathers instead of scattering",
     "y[np.asarray(shuf_perm, dtype=np.int64)] = y_shuf",
     "y[:] = y_shuf[np.asarray(shuf_perm, dtype=np.int64)]"),
    ("rho_foe: max instead of min",
     "return min(H / G, 1.0)",
     "return max(H / G, 1.0)"),
    ("a2a_volume_intra: sign of H",
     "return 2.0 * k * (G - H) / G",
     "return 2.0 * k * (G + H) / G"),
    ("foe_asymptote: (H - 1) term dropped",
     "return k * H * r / (k * H + r * (H - 1))",
     "return k * H * r / (k * H + r * H)"),
]

_RUNNER = (
    "import os, sys\n"
    "copy = sys.argv[1]\n"
    "sys.path.insert(0, copy)\n"
    "import oracle\n"
    "assert os.path.dirname(oracle.smoe_oracle.__file__) == os.path.join(copy, 'oracle')\n"
    "import pytest\n"
    "sys.exit(pytest.main(['-x', '-q', '-p', 'no:cacheprovider', sys.argv[2]]))\n"
)


def _run_pins(tmp_root, name, source):
    """Write `source` as the oracle module of a fresh copy and run the pins on it."""
    copy = os.path.join(tmp_root, name)
    pkg = os.path.join(copy, "oracle")
    os.makedirs(pkg)
    shutil.copy(os.path.join(ROOT, "oracle", "__init__.py"), pkg)
    with open(os.path.join(pkg, "smoe_oracle.py"), "w") as f:
        f.write(source)
    env = dict(os.environ, PYTHONDONTWRITEBYTECODE="1")
    r = subprocess.run([sys.executable, "-c", _RUNNER, copy, PINS], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:] + r.stderr[-2000:]


def test_every_planted_mistake_fails_a_pin(tmp_path):
    with open(ORACLE_SRC) as f:
        src = f.read()
    sources = {"control": src}
    for i, (name, old, new) in enumerate(MUTATIONS):
        assert src.count(old) == 1, f"{name}: the text to change must occur exactly once"
        sources[f"m{i:02d}"] = src.replace(old, new)
    workers = max(1, min(8, (os.cpu_count() or 2)))
    with ThreadPoolExecutor(workers) as ex:
        results = dict(zip(sources, ex.map(lambda kv: _run_pins(str(tmp_path), *kv),
                                           sources.items())))
    rc, out = results.pop("control")
    assert rc == 0, "the unmodified copy must pass the pins:\n" + out
    survived = [MUTATIONS[int(k[1:])][0] for k, (rc, _) in results.items() if rc == 0]
    assert not survived, "planted mistakes no pin caught: " + "; ".join(survived)
    # a failure must be a failing test (1), not a crash of the runner or of collection
    crashed = [MUTATIONS[int(k[1:])][0] + ": " + out[-400:]
               for k, (rc, out) in results.items() if rc not in (0, 1)]
    assert not crashed, "\n".join(crashed)
