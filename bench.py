#!/usr/bin/env python
"""MoE-layer forward throughput on GB300: tokens/s of the whole hot path.

One step = one pass of the layer over one batch held in HBM: gate GEMM + softmax +
(grouped) top-K -> C_p prediction + token shuffle -> local-activation counts ->
expert dispatch -> grouped SwiGLU FFN -> combine (-> next-layer prefetch predictor on
the Qwen3-shaped FoE workload). Every stage is one C-ABI call of libsmoe.so; CUDA
events between the calls give per-stage times inside the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line (rank 0). Under torchrun every rank runs the same layer on its
own seeded batch (replicas, weak scaling, no data-path collective); the timing is the
maximum over ranks. ``--impl reference`` times the CPU oracle on this host instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "dsv2_prefill"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------- helpers

METRIC = ("MoE-layer tokens/s (gate+top-K, s-TS predict+shuffle, LAR, dispatch, grouped SwiGLU "
          "FFN, combine) on GB300")


def workload_label(cfg) -> str:
    return (f"{cfg.name}: T={cfg.T}, d={cfg.d}, E={cfg.E}, K={cfg.K}, H={cfg.H}, F={cfg.F}, "
            f"shared={cfg.n_shared}, P={cfg.P}, vocab={cfg.vocab}")


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--impl", default="native", choices=["native", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-placement", action="store_true",
                   help="skip the (untimed) co-clustered placement report")
    p.add_argument("--tokens", type=int, default=None,
                   help="override the workload's batch size T (the default is its own T)")
    p.add_argument("--seed", type=int, default=0,
                   help="draw another seeded token batch (weights and tables unchanged)")
    p.add_argument("--cpu-seconds", type=float, default=15.0,
                   help="target CPU time of the oracle baseline sample")
    return p.parse_args(argv)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init_dist(world: int, backend: str, timeout_s: float | None = None):
    """Join the process group (world > 1). With timeout_s, a collective that a rank never
    joins (it failed or exited) raises on the others after that many seconds instead of
    blocking: the host-side failure detection of the multi-rank bench."""
    import datetime

    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        kw = {} if timeout_s is None else {"timeout": datetime.timedelta(seconds=timeout_s)}
        dist.init_process_group(backend=backend, **kw)
    return world > 1


def barrier(active: bool):
    if active:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, active: bool, device="cpu") -> float:
    """Maximum of a per-rank float over all ranks (identity on one rank)."""
    if not active:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, seconds_max: float) -> float:
    """Throughput of the whole job: units of all ranks over the slowest rank's time."""
    return units_per_rank * world / seconds_max


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_hash(*names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "routing_token_shuffle_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def stage_bytes(cfg, rows_in_ffn: bool = False) -> dict:
    """Algorithmic bytes per stage (each input read once, each output written once). With
    rows_in_ffn the shuffle copies x to x_shuf, the dispatch stage only sorts (indices in,
    pair_row / row_token / row_slot out) and its row copy runs inside the expert FFN's up
    GEMM; otherwise the shuffle stage computes the permutation alone and the dispatch
    stage sorts, then writes x_shuf and X_disp from one read of x."""
    T, d, E, K, S, b = cfg.T, cfg.d, cfg.E, cfg.K, cfg.n_shared, cfg.elem_bytes
    rows = 2 * T * d * b                       # x read, x_shuf written
    return {
        "route": T * d * b + E * d * b + T * E * 4 + T * K * 8,
        "predict_shuffle": T * 4 + T * E * 4 + 3 * T * 4 + (rows if rows_in_ffn else 0),
        "lar": T * K * 4 + T * 4,
        "dispatch": (T * K * 16 if rows_in_ffn else T * K * 12 + T * 4 + rows + T * K * d * b),
        "combine": T * K * d * b + S * T * d * b + T * K * 8 + T * d * b,
    }


def ffn_flops(cfg) -> float:
    return 6.0 * cfg.d * cfg.F * (cfg.T * cfg.K + cfg.n_shared * cfg.T)


def ffn_bytes(cfg, touched_experts: int) -> int:
    """Algorithmic bytes of the grouped FFN: the weights of every expert that received at
    least one row (plus the shared experts) read once, X_disp and x read once, H written
    and read once, the expert outputs written once."""
    T, d, F, K, S, b = cfg.T, cfg.d, cfg.F, cfg.K, cfg.n_shared, cfg.elem_bytes
    weights = (touched_experts + S) * 3 * F * d * b
    acts = (T * K + S * T) * d * b + 2 * (T * K + S * T) * F * b + (T * K + S * T) * d * b
    return weights + acts


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while the timed region runs."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.proc = None
        self.path = None
        self.gpu_id = gpu_id

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "50"]
            if self.gpu_id:
                cmd += ["-i", self.gpu_id]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self, window=None) -> dict | None:
        """Summarise the samples; with window = (t0, t1) in time.time() seconds keep only
        the samples taken inside it (all samples if none fall inside)."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == 9:
                    rows.append(parts)
        os.unlink(self.path)
        if window is not None:
            import datetime
            inside = []
            for r in rows:
                try:
                    ts = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    continue
                if window[0] <= ts <= window[1]:
                    inside.append(r)
            rows = inside or rows
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------- workload

class Workload:
    """Device-resident inputs of one workload and the per-stage C-ABI calls of a step."""

    def __init__(self, name: str, device, rank: int = 0, tokens: int | None = None,
                 seed: int = 0):
        import numpy as np
        import torch

        import routing_token_shuffle_gb300 as smoe
        from routing_token_shuffle_gb300 import profiling, synth

        self.smoe = smoe
        cfg = synth.CONFIGS[name]
        if tokens is not None:
            import dataclasses
            cfg = dataclasses.replace(cfg, T=tokens)
        self.cfg = cfg
        dev = torch.device(device)
        self.dev = dev
        self.emb = synth.Embedding(cfg, dev)
        self.ids, x32 = synth.token_batch(cfg, self.emb, "ids", cfg.T, dev,
                                          salt=rank + 1000 * seed)
        self.x = x32.to(cfg.torch_dtype).contiguous()
        del x32
        self.w_gate, self.w1, self.w3, self.w2 = synth.layer_weights_lowp(cfg, dev)
        self.emap = synth.placement_identity(cfg)
        self.desc = smoe.desc_from_config(cfg)
        self.ws = smoe.workspace(self.desc, dev)
        # offline C_p: route a seeded profiling batch with the library, count on the host
        n_prof = cfg.profile_tokens
        pids, px = synth.token_batch(cfg, self.emb, "profile", n_prof, dev)
        px = px.to(cfg.torch_dtype)
        chunk = min(n_prof, 8192)
        pdesc = smoe.desc_from_config(cfg, T=chunk)
        pws = smoe.workspace(pdesc, dev)
        pidx = torch.empty(n_prof, cfg.K, dtype=torch.int32, device=dev)
        pw = torch.empty(chunk, cfg.K, device=dev)
        for lo in range(0, n_prof, chunk):
            smoe.smoe_route(pdesc, px[lo:lo + chunk], self.w_gate, pidx[lo:lo + chunk], pw,
                            ws=pws)
        self.profile_idx = pidx.cpu().numpy()
        del pw, pws
        del px
        self.profile_ids = pids
        self.conf = profiling.confidence_table(
            pids, self.profile_idx, cfg.vocab, cfg.E, cfg.K,
            emb_rows=lambda v: self.emb.rows(v).cpu().numpy(), rows_needed=self.ids)
        self.conf_d = torch.as_tensor(self.conf, device=dev)
        self.emap_d = torch.as_tensor(self.emap, device=dev)
        self.ids_d = torch.as_tensor(self.ids, device=dev)
        T, K, E, P = cfg.T, cfg.K, cfg.E, cfg.P
        i32 = dict(dtype=torch.int32, device=dev)
        self.logits = torch.empty(T, E, device=dev)
        self.idx = torch.empty(T, K, **i32)
        self.w = torch.empty(T, K, device=dev)
        self.pred = torch.empty(T, **i32)
        self.perm = torch.empty(T, **i32)
        self.part_off = torch.empty(P + 1, **i32)
        self.lar = torch.zeros(4, dtype=torch.int64, device=dev)
        self.expert_off = torch.empty(E + 1, **i32)
        self.pair_row = torch.empty(T, K, **i32)
        self.row_token = torch.empty(T * K, **i32)
        self.x_shuf = torch.empty_like(self.x)
        self.x_disp = torch.empty(T * K, cfg.d, dtype=self.x.dtype, device=dev)
        self.row_slot = torch.empty(T * K, **i32)
        # the library copies the dispatched rows inside the up GEMM for this layer shape
        self.rows_in_ffn = smoe.smoe_expert_ffn_gather_fused(self.desc)
        self.y_sh = (torch.empty(cfg.n_shared, T, cfg.d, dtype=self.x.dtype, device=dev)
                     if cfg.n_shared else None)
        self.y = torch.empty_like(self.x)
        self.weights = smoe.layer_weights(self.w_gate, self.w1, self.w3, self.w2, self.conf_d,
                                          self.emap_d)
        # inter-layer predictor inputs: a stand-in previous layer routes the profile batch and
        # the measured batch; table A counts cluster transitions on the profile batch
        wprev = synth.previous_layer_gate(cfg, dev)
        _, px2 = synth.token_batch(cfg, self.emb, "profile", n_prof, dev)
        px2 = px2.to(cfg.torch_dtype)
        pprev = torch.empty(n_prof, cfg.K, dtype=torch.int32, device=dev)
        pws2 = smoe.workspace(pdesc, dev)
        pw2 = torch.empty(chunk, cfg.K, device=dev)
        for lo in range(0, n_prof, chunk):
            smoe.smoe_route(pdesc, px2[lo:lo + chunk], wprev, pprev[lo:lo + chunk], pw2,
                            ws=pws2)
        table = profiling.transition_table(
            profiling.cluster_of(pprev.cpu().numpy(), self.emap, cfg.P),
            profiling.cluster_of(self.profile_idx, self.emap, cfg.P), cfg.P)
        del px2, pws2, pw2, pprev
        bidx = torch.empty(cfg.T, cfg.K, dtype=torch.int32, device=dev)
        bw = torch.empty(cfg.T, cfg.K, device=dev)
        smoe.smoe_route(self.desc, self.x, wprev, bidx, bw, ws=self.ws)
        prev_cluster = torch.empty(cfg.T, dtype=torch.int32, device=dev)
        smoe.smoe_token_cluster(self.desc, bidx, self.emap_d, prev_cluster, self.ws)
        self.inter = dict(prev=prev_cluster, table=torch.as_tensor(table, device=dev))
        self.prefetch = None
        if cfg.prefetch:
            r, wgn, gamma, beta = synth.predictor_inputs(cfg, dev)
            # default vector d_l: mean layer output over a separate 1024-token batch
            _, xp = synth.profile_batch_for_default_vector(cfg, self.emb, dev)
            xp = xp.to(cfg.torch_dtype)
            dd = smoe.desc_from_config(cfg, T=xp.shape[0])
            wsd = smoe.workspace(dd, dev)
            yp = torch.empty_like(xp)
            ids_p = torch.zeros(xp.shape[0], dtype=torch.int32, device=dev)
            smoe.smoe_layer_forward(dd, self.weights, smoe.layer_io(xp, ids_p, yp), wsd)
            d_l = yp.float().mean(dim=0).contiguous()
            del wsd, xp, yp
            self.prefetch = dict(r=r, d_l=d_l, wgn=wgn.to(cfg.torch_dtype), gamma=gamma, beta=beta,
                                 pi=torch.empty(T, K, **i32), ti=torch.empty(T, K, **i32),
                                 hits=torch.zeros(1, dtype=torch.int64, device=dev))
        if dev.type == "cuda":
            torch.cuda.synchronize()

    STAGES = ("route", "predict_shuffle", "lar", "dispatch", "expert_ffn", "combine", "prefetch")

    def step(self, events=None):
        """One forward of the layer; records an event after each stage when given. Each
        stage is also an NVTX range (named as in STAGES) for timeline profilers."""
        import torch
        s, c = self.smoe, self
        nvtx = torch.cuda.nvtx

        def rec(i):
            nvtx.range_pop()
            if events is not None:
                events[i].record()
            if i + 1 < len(Workload.STAGES):
                nvtx.range_push(Workload.STAGES[i + 1])

        nvtx.range_push(Workload.STAGES[0])
        s.smoe_route(c.desc, c.x, c.w_gate, c.idx, c.w, logits_out=c.logits, ws=c.ws)
        rec(0)
        # the rows of x_shuf are written here when the FFN copies the dispatched rows
        # itself, else with the dispatched rows after the dispatch's sort
        s.smoe_predict_shuffle(c.desc, c.ids_d, c.conf_d, c.emap_d, c.pred, c.perm, c.part_off,
                               c.ws, x=c.x, x_shuf=c.x_shuf if c.rows_in_ffn else None)
        rec(1)
        s.smoe_lar(c.desc, c.idx, c.emap_d, c.lar, c.ws, src_part=c.pred)
        rec(2)
        if c.rows_in_ffn:
            # the dispatch sorts; the FFN copies the rows inside its up GEMM
            s.smoe_dispatch(c.desc, c.idx, c.expert_off, c.pair_row, c.row_token, c.ws,
                            shuf_perm=c.perm, row_slot=c.row_slot)
            rec(3)
            s.smoe_expert_ffn_gather(c.desc, c.x_shuf, c.row_slot, c.x_disp, c.expert_off, c.w1,
                                     c.w3, c.w2, c.x_disp, c.ws, x=c.x, y_shared=c.y_sh)
        else:
            # the dispatch sorts; then one pass over x writes x_shuf and the dispatched rows
            s.smoe_dispatch(c.desc, c.idx, c.expert_off, c.pair_row, c.row_token, c.ws,
                            shuf_perm=c.perm)
            s.smoe_shuffle_dispatch_rows(c.desc, c.x, c.pair_row, c.x_disp, c.ws,
                                         shuf_perm=c.perm, x_shuf=c.x_shuf)
            rec(3)
            s.smoe_expert_ffn(c.desc, c.x_disp, c.expert_off, c.w1, c.w3, c.w2, c.x_disp, c.ws,
                              x=c.x, y_shared=c.y_sh)
        rec(4)
        s.smoe_combine(c.desc, c.x_disp, c.pair_row, c.w, c.y, c.ws, y_shared=c.y_sh)
        rec(5)
        if c.prefetch is not None:
            p = c.prefetch
            s.smoe_prefetch_predict(c.desc, p["r"], p["d_l"], c.y, p["gamma"], p["beta"], p["wgn"],
                                    p["pi"], p["ti"], p["hits"], c.ws)
        rec(6)


def plain_topk_hit_rate(wl):
    """Hit rate of the prefetch predictor when the next router takes a plain top-K over all
    experts instead of the layer's grouped rule."""
    import torch
    s, c, p = wl.smoe, wl.cfg, wl.prefetch
    desc = s.make_desc(c.T, c.d, c.E, c.K, 1, c.F, c.n_shared, c.P, c.vocab, c.dtype)
    i32 = dict(dtype=torch.int32, device=wl.dev)
    pi, ti = torch.empty(c.T, c.K, **i32), torch.empty(c.T, c.K, **i32)
    hits = torch.zeros(1, dtype=torch.int64, device=wl.dev)
    s.smoe_prefetch_predict(desc, p["r"], p["d_l"], wl.y, p["gamma"], p["beta"], p["wgn"], pi, ti,
                            hits, wl.ws)
    torch.cuda.synchronize()
    return float(hits.item() / (c.T * c.K))


def speculative_execution_report(wl):
    """Run the next layer's stand-in (this layer's experts) on s = LN(r + y) with the
    routes predicted from q and with the true routes; report the hit rate, the relative
    deviation of the speculative output and the time of one routed forward."""
    import torch
    s, c, p = wl.smoe, wl.cfg, wl.prefetch
    dev = wl.dev
    lq = torch.empty(c.T, c.E, device=dev)
    ls = torch.empty(c.T, c.E, device=dev)
    qs = torch.empty(2, c.T, c.d, dtype=c.torch_dtype, device=dev)
    s.smoe_prefetch_predict(wl.desc, p["r"], p["d_l"], wl.y, p["gamma"], p["beta"], p["wgn"],
                            p["pi"], p["ti"], p["hits"], wl.ws, logits_q=lq, logits_s=ls,
                            qs_out=qs)
    i32 = dict(dtype=torch.int32, device=dev)
    pidx, tidx = torch.empty(c.T, c.K, **i32), torch.empty(c.T, c.K, **i32)
    pw, tw = torch.empty(c.T, c.K, device=dev), torch.empty(c.T, c.K, device=dev)
    s.smoe_route(wl.desc, None, None, pidx, pw, logits_in=lq)
    s.smoe_route(wl.desc, None, None, tidx, tw, logits_in=ls)
    s_rows = qs[1].contiguous()
    y_spec, y_true = torch.empty_like(wl.x), torch.empty_like(wl.x)
    s.smoe_moe_forward_routed(wl.desc, s_rows, tidx, tw, wl.w1, wl.w3, wl.w2, y_true, wl.ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(5):
        s.smoe_moe_forward_routed(wl.desc, s_rows, pidx, pw, wl.w1, wl.w3, wl.w2, y_spec, wl.ws)
    e1.record()
    torch.cuda.synchronize()
    d = (y_spec.float() - y_true.float()).norm() / y_true.float().norm()
    return {"hit_rate": float(p["hits"].item() / (c.T * c.K)),
            "rel_deviation_fro": round(float(d), 4),
            "routed_forward_ms": round(e0.elapsed_time(e1) / 5, 4)}


def ep_exchange_report(wl):
    """The expert-parallel exchange P devices would run for this batch (outside the timed
    step): the plan and the receive rows built on this GPU with the s-TS sources, its time
    and achieved bandwidth, and the bytes that would cross links each way. Then SRS and
    SAG with two tensor-parallel partials (x and a copy)."""
    import torch
    s, c = wl.smoe, wl.cfg
    dev = wl.dev
    T, K, P, b = c.T, c.K, c.P, c.elem_bytes
    i32 = dict(dtype=torch.int32, device=dev)
    sc, ro = torch.empty(P, P, **i32), torch.empty(P * P + 1, **i32)
    pr, rt = torch.empty(T, K, **i32), torch.empty(T * K, **i32)
    xr = wl.x_disp  # T K rows: reused as the receive buffer

    def once():
        s.smoe_ep_exchange(wl.desc, wl.idx, wl.emap_d, sc, ro, pr, rt, wl.ws, src_part=wl.pred,
                           x=wl.x, x_recv=xr)

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    once()
    ev[0].record()
    for _ in range(10):
        once()
    ev[1].record()
    torch.cuda.synchronize()
    ms = ev[0].elapsed_time(ev[1]) / 10
    counts = sc.cpu().numpy()
    local = int(counts.trace())
    moved = 2 * T * K * c.d * b + T * K * 12 + T * K * 4
    parts = torch.stack([wl.x, wl.x])
    xs, yb = torch.empty_like(wl.x), torch.empty_like(wl.x)
    s.smoe_srs(wl.desc, parts, wl.perm, xs, wl.ws)
    s.smoe_sag(wl.desc, xs, wl.perm, yb, wl.ws)
    ev2 = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    ev2[0].record()
    for _ in range(10):
        s.smoe_srs(wl.desc, parts, wl.perm, xs, wl.ws)
    ev2[1].record()
    for _ in range(10):
        s.smoe_sag(wl.desc, xs, wl.perm, yb, wl.ws)
    ev2[2].record()
    torch.cuda.synchronize()
    srs_ms, sag_ms = ev2[0].elapsed_time(ev2[1]) / 10, ev2[1].elapsed_time(ev2[2]) / 10
    return {"ms": round(ms, 4), "GB/s": round(moved / (ms / 1e3) / 1e9, 1),
            "local_pairs": local, "remote_pairs": int(T * K - local),
            "link_bytes_each_way": int((T * K - local) * c.d * b),
            "srs_R2_ms": round(srs_ms, 4), "sag_ms": round(sag_ms, 4)}


def placement_report(wl):
    """Offline s-EG placement: co-cluster the profile batch's token-expert activations
    (cross-entropy optimisation, seeded) and measure, on this batch, α and the imbalance
    of the predicted partitions (largest / mean) under the workload's map and under the
    co-clustered map. Not timed; the layer step keeps the workload's map."""
    import time

    import numpy as np
    import torch
    from routing_token_shuffle_gb300 import profiling
    s, c = wl.smoe, wl.cfg
    t0 = time.perf_counter()
    act = profiling.activation_counts(wl.profile_ids, wl.profile_idx, c.vocab, c.E)
    m, _, cost = profiling.ceo_placement(act, c.P, theta=0.1, seed=0)
    secs = time.perf_counter() - t0
    out = {"tool_s": round(secs, 2), "objective_theta_0.1": round(cost, 4)}
    for name, emap in (("workload_map", wl.emap), ("coclustered_map", m)):
        em = torch.as_tensor(np.ascontiguousarray(emap, dtype=np.int32), device=wl.dev)
        pred, perm = torch.empty_like(wl.pred), torch.empty_like(wl.perm)
        off = torch.empty_like(wl.part_off)
        lar = torch.zeros(4, dtype=torch.int64, device=wl.dev)
        s.smoe_predict_shuffle(wl.desc, wl.ids_d, wl.conf_d, em, pred, perm, off, wl.ws)
        s.smoe_lar(wl.desc, wl.idx, em, lar, wl.ws, src_part=pred)
        torch.cuda.synchronize()
        li, sizes = lar.cpu().numpy(), np.diff(off.cpu().numpy())
        out[name] = {"alpha_sTS": round(float(li[0] / li[1]), 4),
                     "alpha_base": round(float(li[2] / li[1]), 4),
                     "partition_imbalance": round(float(sizes.max() / sizes.mean()), 3)}
    return out


# ----------------------------------------------------------------- CPU oracle

class HostLayer:
    """One workload's inputs as host float32 / int32 arrays, the form the CPU oracle takes."""

    def __init__(self, cfg, x, ids, w_gate, w1, w3, w2, conf, emap):
        self.cfg, self.x, self.ids, self.w_gate = cfg, x, ids, w_gate
        self.w1, self.w3, self.w2, self.conf, self.emap = w1, w3, w2, conf, emap


def host_layer_from_workload(wl) -> HostLayer:
    """The native arm's device-resident inputs copied to the host (for the CPU baseline)."""
    f = (lambda t: t.float().cpu().numpy())
    return HostLayer(wl.cfg, f(wl.x), wl.ids, f(wl.w_gate), f(wl.w1), f(wl.w3), f(wl.w2),
                     wl.conf, wl.emap)


def cpu_oracle_rate(h: HostLayer, target_s: float, max_tokens: int | None = None):
    """Tokens/s of the CPU oracle on the first n tokens of the workload's batch, n sized
    so one timed pass takes about target_s seconds. Returns (rate, n, seconds, cores)."""
    import oracle as O
    cfg = h.cfg
    cap = cfg.T if max_tokens is None else min(cfg.T, max_tokens)

    def run(n):
        t0 = time.perf_counter()
        O.layer_forward(h.x[:n], h.ids[:n], h.w_gate, h.w1, h.w3, h.w2, h.conf, h.emap, K=cfg.K,
                        H=cfg.H, P=cfg.P, n_shared=cfg.n_shared)
        return time.perf_counter() - t0

    # time = a + b n: a fixed part per call (the oracle converts every expert's weights to
    # float64 on each call) plus a part per token; two sizes fix both (after one untimed
    # call that takes the one-time costs), then n is chosen so that one call takes about
    # target_s
    n0, n1 = min(cap, 16), min(cap, 128)
    run(n0)
    t0 = run(n0)
    n, t = n0, t0
    if n1 > n0:
        t1 = run(n1)
        b = max((t1 - t0) / (n1 - n0), 1e-9)
        a = max(t0 - b * n0, 0.0)
        n = int(max(n0, min(cap, (target_s - a) / b)))
        t = t1 if n == n1 else run(n)
    # the per-token cost falls as n grows (larger matrix products per expert) and the two
    # small calls fix it poorly, so the fit can undershoot: grow n by the measured rate,
    # at least doubling it, until one call takes 0.7 of target_s (at most four calls)
    for _ in range(4):
        if t >= 0.7 * target_s or n >= cap:
            break
        n = int(min(cap, max(2 * n, n * 0.9 * target_s / max(t, 1e-3))))
        t = run(n)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return n / t, n, t, cores


def reference_inputs(name: str, tokens: int | None = None, seed: int = 0) -> HostLayer:
    """The workload built on the host alone, for the reference arm: the seeded generator on
    the CPU (same shapes and distributions; torch's CPU generator draws other values than
    its CUDA one) and C_p profiled from the oracle's own routes. Neither the CUDA library
    nor a GPU is touched."""
    import dataclasses

    import numpy as np

    import oracle as O
    from routing_token_shuffle_gb300 import synth
    cfg = synth.CONFIGS[name]
    if tokens is not None:
        cfg = dataclasses.replace(cfg, T=tokens)
    emb = synth.Embedding(cfg, "cpu")
    ids, x = synth.token_batch(cfg, emb, "ids", cfg.T, "cpu", salt=1000 * seed)
    w_gate, w1, w3, w2 = synth.layer_weights(cfg, "cpu")
    wg = w_gate.numpy()
    pids, px = synth.token_batch(cfg, emb, "profile", cfg.profile_tokens, "cpu")
    pidx = np.empty((len(pids), cfg.K), np.int32)
    for lo in range(0, len(pids), 8192):
        _, pidx[lo:lo + 8192], _ = O.route(px[lo:lo + 8192].numpy(), wg, cfg.K, cfg.H)
    del px
    conf = O.profile_confidence(pids, pidx, cfg.vocab, cfg.E, cfg.K,
                                emb_rows=lambda v: emb.rows(v).numpy(), rows_needed=ids)
    return HostLayer(cfg, x.numpy(), ids, wg, w1.numpy(), w3.numpy(), w2.numpy(), conf,
                     synth.placement_identity(cfg))


# ----------------------------------------------------------------- arms

def run_native(args):
    import torch

    import routing_token_shuffle_gb300 as smoe
    from routing_token_shuffle_gb300 import build as build_mod

    rank, world, local_rank = dist_env()
    world = max(world, 1)
    if world != args.gpus and world > 1:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE {world}")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0:
        build_mod.build()
    active = init_dist(world, "nccl")
    barrier(active)
    build_mod.build()
    wl = Workload(args.workload, dev, rank=rank, tokens=args.tokens, seed=args.seed)
    cfg = wl.cfg
    peaks, peaks_kind = load_peaks()

    for _ in range(max(args.warmup, 3)):
        wl.step()
    smoe.smoe_get_status(wl.ws)
    torch.cuda.synchronize()

    nst = len(Workload.STAGES)
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    sampler = ClockSampler(uuid)
    barrier(active)
    torch.cuda.synchronize()
    sampler.start()
    t_pre = time.time()
    t_s = time.perf_counter()
    while time.perf_counter() - t_s < 0.4:   # keep the GPU busy while nvidia-smi starts
        wl.step()
        torch.cuda.synchronize()
    barrier(active)
    # the timed region: K steps back to back on one stream, one event on each side
    launches0 = smoe.kernel_launches()
    t_wall0 = time.time()
    wall0 = time.perf_counter()
    start.record()
    for i in range(args.steps):
        wl.step()
    stop.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    launches = smoe.kernel_launches() - launches0
    t_wall1 = time.time()
    barrier(active)
    total_ms = start.elapsed_time(stop)
    total_ms_max = max_over_ranks(total_ms, active, device=dev)
    ms_per_step = total_ms_max / args.steps
    value = whole_job_rate(cfg.T * args.steps, world, total_ms_max / 1e3)

    # per-stage breakdown: another K steps with an event after every stage (not part of
    # the value above; the events cost a little, reported as stage_pass_ms_per_step)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst)] for _ in range(args.steps)]
    start2 = torch.cuda.Event(enable_timing=True)
    start2.record()
    for i in range(args.steps):
        wl.step(evs[i])
    torch.cuda.synchronize()
    t_wall2 = time.time()
    # clocks: samples taken while the layer ran, from the untimed pre-roll through the
    # timed region and the stage pass (all the same back-to-back steps)
    clocks = sampler.stop(window=(t_pre, t_wall2))
    if clocks is not None:
        clocks["window_s"] = round(t_wall2 - t_pre, 3)
        clocks["timed_region_s"] = round(t_wall1 - t_wall0, 3)
    stage_ms = {s: 0.0 for s in Workload.STAGES}
    for i in range(args.steps):
        prev = start2 if i == 0 else evs[i - 1][-1]
        for j, sname in enumerate(Workload.STAGES):
            stage_ms[sname] += prev.elapsed_time(evs[i][j])
            prev = evs[i][j]
    stage_ms = {k: v / args.steps for k, v in stage_ms.items()}
    stage_pass_ms = start2.elapsed_time(evs[-1][-1]) / args.steps
    smoe.smoe_get_status(wl.ws)

    # end to end through the host-buffer entry point (H2D of x and ids, the layer, D2H of
    # y every step). Two schedules: serial (one stream, each step's copies and kernels in
    # turn) and pipelined the way a serving loop runs (two streams and two workspaces in
    # turn, so one step's copies overlap the other step's kernels). The pipelined one is
    # the reported value.
    xh = [wl.x.cpu().pin_memory() for _ in range(2)]
    ih = [torch.as_tensor(wl.ids).pin_memory() for _ in range(2)]
    yh = [torch.empty_like(xh[0]).pin_memory() for _ in range(2)]
    streams = [torch.cuda.current_stream(), torch.cuda.Stream()]
    wss = [wl.ws, smoe.workspace(wl.desc, dev)]

    def e2e_step(i, nstreams):
        j = i % nstreams
        smoe.smoe_layer_forward_host(wl.desc, wl.weights, xh[j], ih[j], yh[j], wss[j],
                                     stream=streams[j])

    def e2e_run(nstreams):
        for i in range(4):
            e2e_step(i, nstreams)
        torch.cuda.synchronize()
        barrier(active)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(streams[0])
        streams[1].wait_event(e0)
        for i in range(args.steps):
            e2e_step(i, nstreams)
        streams[0].wait_stream(streams[1])
        e1.record(streams[0])
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1), active, device=dev)

    e2e_serial_ms = e2e_run(1)
    e2e_ms = e2e_run(2)
    del wss
    e2e_value = whole_job_rate(cfg.T * args.steps, world, e2e_ms / 1e3)
    e2e_serial_value = whole_job_rate(cfg.T * args.steps, world, e2e_serial_ms / 1e3)
    h2d = xh[0].numel() * xh[0].element_size() + ih[0].numel() * ih[0].element_size()
    d2h = yh[0].numel() * yh[0].element_size()

    # roofline of the dominant kernel: the grouped expert FFN GEMMs. Its bound follows
    # from its arithmetic intensity against the measured ridge point (decode-sized
    # batches touch every expert's weights for a few rows: HBM-bound).
    ffn_ms = stage_ms["expert_ffn"]
    # the burst peak for a timed region under a second, the sustained (power-capped) one
    # for a region of seconds
    long_region = total_ms / 1e3 >= 1.0
    peak_key = "bf16_tflops_sustained" if long_region else "bf16_tflops"
    peak_tf = peaks.get(peak_key, FALLBACK_PEAKS[peak_key])
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    eo = wl.expert_off.cpu().numpy()
    touched = int((eo[1:] > eo[:-1]).sum())
    fbytes = ffn_bytes(cfg, touched)
    achieved_tf = ffn_flops(cfg) / (ffn_ms / 1e3) / 1e12
    traffic = None
    tfile = os.path.join(ROOT, "profiles", "expert_ffn_traffic.json")
    if os.path.exists(tfile):
        with open(tfile) as f:
            tj = json.load(f)
        if tj.get("source_hash") == source_hash("ffn.cu"):
            traffic = tj.get("workloads", {}).get(cfg.name, {}).get("bytes_per_step")
    kernel_name = "expert_ffn (grouped SwiGLU up + down GEMMs)"
    if wl.rows_in_ffn:
        kernel_name = ("expert_ffn (grouped SwiGLU up + down GEMMs, the dispatch's row copy "
                       "inside the up GEMM)")
    if ffn_flops(cfg) / fbytes >= peak_tf * 1e12 / (hbm * 1e9):
        roofline = {"bound": "tensor", "achieved": round(achieved_tf, 2), "peak": peak_tf,
                    "unit": "TFLOP/s", "frac": round(achieved_tf / peak_tf, 4),
                    "traffic": traffic, "kernel": kernel_name,
                    "peak_kind": f"{peaks_kind} bf16 {'sustained' if long_region else 'burst'}"
                                 f" (timed region {total_ms / 1e3:.3f} s)"}
    else:
        achieved_gbs = fbytes / (ffn_ms / 1e3) / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": hbm,
                    "unit": "GB/s", "frac": round(achieved_gbs / hbm, 4), "traffic": traffic,
                    "kernel": kernel_name, "peak_kind": f"{peaks_kind} HBM copy",
                    "algorithmic_bytes": fbytes, "experts_touched": touched}
    sb = stage_bytes(cfg, wl.rows_in_ffn)
    stages = {}
    for k, ms in stage_ms.items():
        ent = {"ms": round(ms, 4)}
        if k in sb and ms > 0:
            gbs = sb[k] / (ms / 1e3) / 1e9
            ent.update({"GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4)})
        stages[k] = ent
    stages["expert_ffn"]["TFLOP/s"] = round(achieved_tf, 2)
    if wl.rows_in_ffn:
        stages["dispatch"]["rows"] = "sort only; the row copy runs inside the expert_ffn up GEMM"
    else:
        stages["dispatch"]["rows"] = ("sort, then one read of x writes x_shuf and the T K "
                                      "dispatched rows (predict_shuffle computes the "
                                      "permutation only)")

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, n, secs, cores = cpu_oracle_rate(host_layer_from_workload(wl), args.cpu_seconds)
        cpu = {"value": round(rate, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"first {n} of the {cfg.T} tokens of this workload's batch, the whole "
                         f"layer in float64 numpy ({secs:.1f} s)"}
    lar = wl.lar.cpu().numpy()
    inter_info = None
    if wl.inter is not None:
        pred_i = torch.empty_like(wl.pred)
        perm_i = torch.empty_like(wl.perm)
        off_i = torch.empty_like(wl.part_off)
        lar_i = torch.zeros(4, dtype=torch.int64, device=dev)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        for rep in range(11):
            if rep == 1:
                ev[0].record()
            smoe.smoe_predict_shuffle_inter(wl.desc, wl.ids_d, wl.conf_d, wl.emap_d,
                                            wl.inter["prev"], wl.inter["table"], pred_i, perm_i,
                                            off_i, wl.ws, x=wl.x, x_shuf=wl.x_shuf)
        ev[1].record()
        smoe.smoe_lar(wl.desc, wl.idx, wl.emap_d, lar_i, wl.ws, src_part=pred_i)
        torch.cuda.synchronize()
        li = lar_i.cpu().numpy()
        inter_info = {"alpha_sTS_inter": float(li[0] / li[1]),
                      "predict_shuffle_inter_ms": round(ev[0].elapsed_time(ev[1]) / 10, 4)}
    result = {
        "metric": METRIC,
        "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype,
        "data": "synthetic (seeded; random-init weights of the workload's shape)",
        "config": {"workload": workload_label(cfg),
                   "global_batch": cfg.T * world, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (expert weights "
                         f"{3 * (cfg.E + cfg.n_shared) * cfg.F * cfg.d * cfg.elem_bytes / 1e9:.2f}"
                         " GB streamed every step)"},
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "schedule": "two streams and two workspaces in turn",
                "serial_value": round(e2e_serial_value, 1)},
        "gpu_launches": int(launches),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "clocks": clocks,
        "stages": stages,
        "alpha": {"sTS": float(lar[0] / lar[1]), "base": float(lar[2] / lar[1]),
                  "max": float(lar[3] / lar[1])},
        "wall_s_timed": round(wall, 3),
        "stage_pass_ms_per_step": round(stage_pass_ms, 4),
    }
    if inter_info is not None:
        result["alpha"]["sTS_with_table_A"] = inter_info["alpha_sTS_inter"]
        result["stages"]["predict_shuffle_inter (outside the step)"] = {
            "ms": inter_info["predict_shuffle_inter_ms"]}
    result["ep_exchange"] = ep_exchange_report(wl)
    if not args.no_placement:
        result["placement"] = placement_report(wl)
    if cfg.H > 1:
        # FoE layout: each token's group copies sit on their groups' partitions
        lar_f = torch.zeros(4, dtype=torch.int64, device=dev)
        smoe.smoe_lar(wl.desc, wl.idx, wl.emap_d, lar_f, wl.ws)
        torch.cuda.synchronize()
        lf = lar_f.cpu().numpy()
        result["alpha"]["FoE"] = float(lf[0] / lf[1])
    if wl.prefetch is not None:
        result["prefetch_hit_rate"] = float(wl.prefetch["hits"].item() / (cfg.T * cfg.K))
        result["prefetch_hit_rate_plain_topk"] = plain_topk_hit_rate(wl)
        result["speculative_execution"] = speculative_execution_report(wl)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if active:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args):
    """The CPU oracle as it stands, on this host's cores, same workload and metric. A pure
    host process: inputs come from the seeded generator on the CPU, C_p from the oracle's
    own routes; the CUDA library is never loaded and no CUDA context is created."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    h = reference_inputs(args.workload, tokens=args.tokens, seed=args.seed)
    cfg = h.cfg
    per_step = max(1.0, min(args.cpu_seconds, 100.0 / max(args.steps + args.warmup, 1)))
    rate, n, secs, cores = cpu_oracle_rate(h, per_step)
    import oracle as O
    x, ids = h.x[:n], h.ids[:n]
    for _ in range(args.warmup):
        O.layer_forward(x, ids, h.w_gate, h.w1, h.w3, h.w2, h.conf, h.emap, K=cfg.K, H=cfg.H,
                        P=cfg.P, n_shared=cfg.n_shared)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        O.layer_forward(x, ids, h.w_gate, h.w1, h.w3, h.w2, h.conf, h.emap, K=cfg.K, H=cfg.H,
                        P=cfg.P, n_shared=cfg.n_shared)
    secs = time.perf_counter() - t0
    value = n * args.steps / secs
    sample = (f"first {n} of the {cfg.T} tokens of the batch per step, whole layer in float64 "
              f"numpy")
    print(json.dumps({
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 3), "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, drawn on the host)",
        "config": {"workload": workload_label(cfg), "global_batch": n},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
