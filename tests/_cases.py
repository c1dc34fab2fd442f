"""Seeded test cases shared by the GPU parity tests: inputs from the generator,
expected values from the oracle only."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
from routing_token_shuffle_gb300 import synth


def to_np(t):
    return t.detach().float().cpu().numpy() if t.is_floating_point() else t.detach().cpu().numpy()


class Case:
    """Device inputs of one workload plus the oracle-profiled confidence table."""

    def __init__(self, name, device, T=None, profile_tokens=None, placement="identity"):
        cfg = synth.CONFIGS[name]
        if T is not None:
            cfg = cfg.with_tokens(T)
        self.cfg = cfg
        self.dev = torch.device(device)
        self.emb = synth.Embedding(cfg, self.dev)
        self.ids, x32 = synth.token_batch(cfg, self.emb, "ids", cfg.T, self.dev)
        self.x = x32.to(cfg.torch_dtype).contiguous()
        self.w_gate, self.w1, self.w3, self.w2 = synth.layer_weights_lowp(cfg, self.dev)
        self.emap = synth.placement_identity(cfg)
        if placement == "foe":
            self.emap = synth.placement_foe(cfg.E, cfg.H, cfg.P)
        n_prof = profile_tokens or min(cfg.profile_tokens, 8192)
        pids, px = synth.token_batch(cfg, self.emb, "profile", n_prof, self.dev)
        _, pidx, _ = O.route(to_np(px), to_np(self.w_gate), cfg.K, cfg.H)
        self.profile_ids, self.profile_idx = pids, pidx
        self.conf = O.profile_confidence(pids, pidx, cfg.vocab, cfg.E, cfg.K,
                                         emb_rows=lambda v: to_np(self.emb.rows(v)),
                                         rows_needed=self.ids)
        self.conf_d = torch.as_tensor(self.conf, device=self.dev)
        self.emap_d = torch.as_tensor(self.emap, device=self.dev)
        self.ids_d = torch.as_tensor(self.ids, device=self.dev)
        self._x_np = None

    @property
    def x_np(self):
        if self._x_np is None:
            self._x_np = to_np(self.x).astype(np.float64)
        return self._x_np

    def expert_weights_np(self, e):
        return (to_np(self.w1[e]).astype(np.float64), to_np(self.w3[e]).astype(np.float64),
                to_np(self.w2[e]).astype(np.float64))

    def oracle_tokens(self, tokens, idx, w):
        """Oracle layer output for the given tokens, each through its own experts.
        Experts are visited one at a time so only one expert's float64 weights are
        held on the host."""
        cfg = self.cfg
        tokens = np.asarray(tokens)
        out = np.zeros((len(tokens), cfg.d))
        sel = np.asarray(idx)[tokens]
        for e in range(cfg.E + cfg.n_shared):
            if e < cfg.E:
                rows, ks = np.nonzero(sel == e)
            else:
                rows, ks = np.arange(len(tokens)), None
            if len(rows) == 0:
                continue
            ye = O.swiglu_ffn(self.x_np[tokens[rows]], *self.expert_weights_np(e))
            wk = np.ones(len(rows)) if ks is None else np.asarray(w)[tokens[rows], ks]
            np.add.at(out, rows, wk[:, None] * ye)
        return out


def rel_err_rows(got, ref):
    """Per row: max-abs error over the row's max-abs reference value."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return np.abs(got - ref).max(axis=1) / np.maximum(np.abs(ref).max(axis=1), 1e-30)


def sample_tokens(T, n=48, seed=0):
    """A seeded sample of token indices that always includes the first and the last
    (ragged tail) tokens."""
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(T, size=min(n, T), replace=False).tolist())
    pick.update({0, T - 1})
    return np.array(sorted(pick))


def block_edge_rows(offsets, block=64):
    """First and last row of every `block`-row block of every segment [offsets[e],
    offsets[e+1]): one row per CTA half of every GEMM tile, whatever the tile shape (256-row
    pair tiles, 128-row tiles, 64-row halves of a 128-row pair tail), in every wave of a
    persistent schedule."""
    rows = set()
    for lo, hi in zip(offsets[:-1], offsets[1:]):
        for b in range(int(lo), int(hi), block):
            rows.add(b)
            rows.add(min(b + block - 1, int(hi) - 1))
    return np.array(sorted(rows), dtype=np.int64)
