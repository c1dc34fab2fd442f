"""Seeded synthetic inputs for the MoE-layer hot path.

This module only draws random numbers and lays them out: token ids, token
activations, weights, residuals and simple placement maps. It holds none of the
layer's arithmetic (no gate, no top-K, no prediction, no FFN), so both the
CUDA path and the CPU oracle can be fed from it without sharing any method code.

Workloads (stand-ins for the pages' evaluation models, whose trained weights and
datasets are not available):

* ``tiny_fp32``   -- a tiny fp32 layer for exhaustive parity.
* ``mixtral``     -- Mixtral-8x7B-shaped prefill layer (Speculative MoE, §5
  experiments: DeepSeek-V2 and Mixtral-8x7B).
* ``dsv2_prefill``/``dsv2_decode`` -- DeepSeek-V2-shaped layer, 160 routed + 2
  shared experts, prefill and a 64-token decode step.
* ``qwen3_foe``   -- Qwen3-30B-A3B-shaped layer routed with Federation of
  Experts' grouped top-k/H (8 groups of 16 experts, one pick per group), plus the
  next-layer prefetch predictor of "Speculating Experts Accelerates Inference
  for MoE" (§2.A, quasi-hidden state).

Token ids are truncated Zipf(1.1) draws (a heavy-headed vocabulary as in the
pages' LongBench/GSM8K/HumanEval text workloads, which are not reproduced).
Activations are ``emb[id] + N(0, 0.1^2)``; for the bf16 workloads the embedding
table is clustered (64 centroids, ``emb = centroid + 0.5 N(0,1)``) so that
semantically close ids share routes, the token-expert conjugacy that Speculative
MoE §2 builds on.

Large tensors are drawn by torch's seeded generator on the target device
(Philox on CUDA, MT19937 on CPU); small integer draws (ids, cluster labels,
seeded orders) come from numpy PCG64 streams spawned from
``SeedSequence(workload index)``.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

# Stream names spawned from SeedSequence(workload index), in this fixed order.
STREAMS = ("ids", "emb", "noise", "weights", "profile", "placement", "predictor", "prev_layer")


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    index: int          # seed of the workload (SeedSequence entropy)
    T: int              # tokens in the measured batch
    d: int              # model dimension
    E: int              # routed experts
    K: int              # routed experts per token
    H: int              # expert groups (Federation of Experts); 1 = plain top-K
    F: int              # expert hidden size (SwiGLU)
    n_shared: int       # always-on shared experts
    P: int              # simulated expert-parallel partitions (G on the FoE page)
    vocab: int
    dtype: str          # "f32" or "bf16": activations, weights and output
    placement: str      # identity expert->partition placement: "mod" or "contiguous"
    emb_kind: str       # "gaussian" or "clustered"
    profile_tokens: int  # tokens in the offline C_p profiling batch
    w2_std_from_d: bool = False  # tiny_fp32 draws every weight from N(0, 1/d)
    prefetch: bool = False       # run the next-layer prefetch predictor
    weight_index: int | None = None  # share weights/tables with another workload

    @property
    def seed_index(self) -> int:
        return self.index if self.weight_index is None else self.weight_index

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def with_tokens(self, T: int) -> "LayerConfig":
        return dataclasses.replace(self, T=T)


CONFIGS = {
    c.name: c
    for c in [
        LayerConfig("tiny_fp32", 0, T=64, d=128, E=8, K=2, H=1, F=256, n_shared=0, P=2,
                    vocab=512, dtype="f32", placement="mod", emb_kind="gaussian",
                    profile_tokens=4096, w2_std_from_d=True),
        LayerConfig("mixtral", 1, T=4096, d=4096, E=8, K=2, H=1, F=14336, n_shared=0, P=2,
                    vocab=32000, dtype="bf16", placement="contiguous", emb_kind="clustered",
                    profile_tokens=65536),
        LayerConfig("dsv2_prefill", 2, T=8192, d=5120, E=160, K=6, H=1, F=1536, n_shared=2,
                    P=8, vocab=102400, dtype="bf16", placement="contiguous",
                    emb_kind="clustered", profile_tokens=65536),
        LayerConfig("dsv2_decode", 3, T=64, d=5120, E=160, K=6, H=1, F=1536, n_shared=2,
                    P=8, vocab=102400, dtype="bf16", placement="contiguous",
                    emb_kind="clustered", profile_tokens=65536, weight_index=2),
        LayerConfig("qwen3_foe", 4, T=16384, d=2048, E=128, K=8, H=8, F=768, n_shared=0,
                    P=8, vocab=32000, dtype="bf16", placement="contiguous",
                    emb_kind="clustered", profile_tokens=65536, prefetch=True),
    ]
}

N_CENTROIDS = 64
ZIPF_S = 1.1
NOISE_STD = 0.1


def _streams(index: int) -> dict[str, np.random.SeedSequence]:
    return dict(zip(STREAMS, np.random.SeedSequence(index).spawn(len(STREAMS))))


def _torch_gen(ss: np.random.SeedSequence, salt: int, device) -> torch.Generator:
    seed = int(np.random.SeedSequence(ss.generate_state(2).tolist() + [salt]).generate_state(1,
               dtype=np.uint64)[0] & ((1 << 63) - 1))
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def zipf_ids(rng: np.random.Generator, vocab: int, n: int, s: float = ZIPF_S) -> np.ndarray:
    """Truncated Zipf draws: p(r) ~ r^-s for rank r = 1..vocab, id = r - 1 (inverse CDF)."""
    ranks = np.arange(1, vocab + 1, dtype=np.float64)
    cdf = np.cumsum(ranks ** (-s))
    cdf /= cdf[-1]
    u = rng.random(n)
    ids = np.searchsorted(cdf, u, side="right")
    return np.minimum(ids, vocab - 1).astype(np.int32)


def round_bf16(t: torch.Tensor) -> torch.Tensor:
    """Round to bf16 (round-to-nearest-even) and back to fp32."""
    return t.to(torch.bfloat16).to(torch.float32)


class Embedding:
    """Embedding rows, materialised lazily so a 102400 x 5120 table never has to exist.

    Row v is drawn from a generator keyed by (workload seed, v), so any subset of
    rows can be produced on any device in any order with the same values (for a
    given device kind)."""

    def __init__(self, cfg: LayerConfig, device):
        self.cfg = cfg
        self.device = torch.device(device)
        ss = _streams(cfg.seed_index)["emb"]
        rng = np.random.Generator(np.random.PCG64(ss))
        self.cluster = rng.integers(0, N_CENTROIDS, size=cfg.vocab).astype(np.int64)
        self._ss = ss
        if cfg.emb_kind == "clustered":
            g = _torch_gen(ss, 0, self.device)
            self.centroids = torch.randn(N_CENTROIDS, cfg.d, generator=g, device=self.device)
        else:
            self.centroids = None

    def rows(self, ids) -> torch.Tensor:
        """fp32 [len(ids), d] embedding rows (duplicates allowed)."""
        ids = np.asarray(ids, dtype=np.int64)
        uniq, inv = np.unique(ids, return_inverse=True)
        out = torch.empty(len(uniq), self.cfg.d, device=self.device)
        # Draw noise in blocks of 4096 ids: block b uses its own generator, row v
        # takes row (v mod 4096) of block (v // 4096)'s draw.
        blk = 4096
        for b in np.unique(uniq // blk):
            sel = np.nonzero(uniq // blk == b)[0]
            g = _torch_gen(self._ss, 1 + int(b), self.device)
            n = min(blk, self.cfg.vocab - int(b) * blk)
            block = torch.randn(n, self.cfg.d, generator=g, device=self.device)
            local = torch.as_tensor(uniq[sel] - int(b) * blk, device=self.device)
            out[torch.as_tensor(sel, device=self.device)] = block[local]
        if self.centroids is not None:
            cl = torch.as_tensor(self.cluster[uniq], device=self.device)
            out = self.centroids[cl] + 0.5 * out
        return out[torch.as_tensor(inv, device=self.device)]


def token_batch(cfg: LayerConfig, emb: Embedding, stream: str, n: int, device, salt: int = 0):
    """(ids int32 numpy [n], x fp32 tensor [n, d]) with x = emb[id] + N(0, 0.1^2), rounded to
    the workload dtype's precision."""
    st = _streams(cfg.index)[stream]
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(
        st.generate_state(2).tolist() + [salt])))
    ids = zipf_ids(rng, cfg.vocab, n)
    g = _torch_gen(st, 100 + salt, device)
    x = emb.rows(ids) + NOISE_STD * torch.randn(n, cfg.d, generator=g, device=device)
    if cfg.dtype == "bf16":
        x = round_bf16(x)
    return ids, x


def layer_weights(cfg: LayerConfig, device, experts=None):
    """Gate and expert weights, fp32 tensors already rounded to the workload dtype.

    w_gate [E, d] ~ N(0, 1/d); w1, w3 [E+S, F, d] ~ N(0, 1/d); w2 [E+S, d, F] ~ N(0, 1/F)
    (N(0, 1/d) for tiny_fp32, whose description draws every weight from N(0, 1/d)).
    Each expert is drawn from its own generator, so ``experts`` may select a subset.
    """
    ss = _streams(cfg.seed_index)["weights"]
    n_all = cfg.E + cfg.n_shared
    experts = list(range(n_all)) if experts is None else list(experts)
    rnd = (lambda t: t) if cfg.dtype == "f32" else round_bf16
    g = _torch_gen(ss, 0, device)
    w_gate = rnd(torch.randn(cfg.E, cfg.d, generator=g, device=device) / math.sqrt(cfg.d))
    w2_std = 1.0 / math.sqrt(cfg.d if cfg.w2_std_from_d else cfg.F)
    w1 = torch.empty(len(experts), cfg.F, cfg.d, device=device)
    w3 = torch.empty_like(w1)
    w2 = torch.empty(len(experts), cfg.d, cfg.F, device=device)
    for i, e in enumerate(experts):
        ge = _torch_gen(ss, 1 + e, device)
        w1[i] = rnd(torch.randn(cfg.F, cfg.d, generator=ge, device=device) / math.sqrt(cfg.d))
        w3[i] = rnd(torch.randn(cfg.F, cfg.d, generator=ge, device=device) / math.sqrt(cfg.d))
        w2[i] = rnd(torch.randn(cfg.d, cfg.F, generator=ge, device=device) * w2_std)
    return w_gate, w1, w3, w2


def layer_weights_lowp(cfg: LayerConfig, device):
    """The same weights as ``layer_weights`` stored directly in the workload dtype,
    drawn expert by expert so no full fp32 copy is ever held (DeepSeek-V2-shaped
    weights are 7.6 GB in bf16)."""
    ss = _streams(cfg.seed_index)["weights"]
    n_all = cfg.E + cfg.n_shared
    dt = cfg.torch_dtype
    g = _torch_gen(ss, 0, device)
    w_gate = (torch.randn(cfg.E, cfg.d, generator=g, device=device) / math.sqrt(cfg.d)).to(dt)
    w2_std = 1.0 / math.sqrt(cfg.d if cfg.w2_std_from_d else cfg.F)
    w1 = torch.empty(n_all, cfg.F, cfg.d, device=device, dtype=dt)
    w3 = torch.empty_like(w1)
    w2 = torch.empty(n_all, cfg.d, cfg.F, device=device, dtype=dt)
    for e in range(n_all):
        ge = _torch_gen(ss, 1 + e, device)
        w1[e] = (torch.randn(cfg.F, cfg.d, generator=ge, device=device) / math.sqrt(cfg.d)).to(dt)
        w3[e] = (torch.randn(cfg.F, cfg.d, generator=ge, device=device) / math.sqrt(cfg.d)).to(dt)
        w2[e] = (torch.randn(cfg.d, cfg.F, generator=ge, device=device) * w2_std).to(dt)
    return w_gate, w1, w3, w2


def placement_identity(cfg: LayerConfig) -> np.ndarray:
    """Identity expert->partition map: e mod P ("mod") or e // (E/P) ("contiguous")."""
    e = np.arange(cfg.E)
    if cfg.placement == "mod":
        return (e % cfg.P).astype(np.int32)
    return (e * cfg.P // cfg.E).astype(np.int32)


def placement_foe(E: int, H: int, G: int) -> np.ndarray:
    """Federation of Experts placement: group h = experts [h E/H, (h+1) E/H).

    H >= G: group h lives on partition floor(h G / H).
    H <  G: group h spans partitions h (G/H) .. h (G/H) + G/H - 1 and its j-th
    expert sits on partition h (G/H) + (j mod G/H)."""
    out = np.empty(E, np.int32)
    per = E // H
    for e in range(E):
        h, j = divmod(e, per)
        if H >= G:
            out[e] = h * G // H
        else:
            out[e] = h * (G // H) + (j % (G // H))
    return out


def seeded_order(cfg: LayerConfig, n: int) -> np.ndarray:
    """A seeded permutation of range(n) from the placement stream."""
    rng = np.random.Generator(np.random.PCG64(_streams(cfg.seed_index)["placement"]))
    return rng.permutation(n).astype(np.int64)


def predictor_inputs(cfg: LayerConfig, device):
    """Residual r_l [T, d] ~ N(0,1) (fp32), next-layer gate W_g' [E, d] ~ N(0, 1/d) in the
    workload dtype (as fp32 values), LayerNorm gamma = 1 and beta = 0."""
    ss = _streams(cfg.index)["predictor"]
    g = _torch_gen(ss, 0, device)
    r = torch.randn(cfg.T, cfg.d, generator=g, device=device)
    g2 = _torch_gen(ss, 1, device)
    wg_next = torch.randn(cfg.E, cfg.d, generator=g2, device=device) / math.sqrt(cfg.d)
    if cfg.dtype == "bf16":
        wg_next = round_bf16(wg_next)
    gamma = torch.ones(cfg.d, device=device)
    beta = torch.zeros(cfg.d, device=device)
    return r, wg_next, gamma, beta


def profile_batch_for_default_vector(cfg: LayerConfig, emb: Embedding, device, n: int = 1024):
    """The separate seeded token batch whose mean layer output is the default vector d_l."""
    return token_batch(cfg, emb, "predictor", n, device, salt=7)


def previous_layer_gate(cfg: LayerConfig, device):
    """Router weight of a stand-in previous MoE layer [E, d] ~ N(0, 1/d) in the workload
    dtype: routing the same token representations through it gives each token a
    previous-layer cluster for the inter-layer predictor."""
    g = _torch_gen(_streams(cfg.seed_index)["prev_layer"], 0, device)
    w = torch.randn(cfg.E, cfg.d, generator=g, device=device) / math.sqrt(cfg.d)
    return w.to(cfg.torch_dtype)
