"""Benchmark one Medusa decoding step on synthetic Vicuna-7B/13B-shaped inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one pass of the whole hot path on one batch of input:
    medusa_heads -> medusa_build_tree -> medusa_tree_attention -> medusa_evaluate_posterior
The headline workload is the 7B shape at batch 1 (d=4096, V=32000, K=5 heads,
s=(4,3,2,2,1) cut to 64 nodes, 32 x 128 attention heads, prefix 1024, typical
acceptance eps=0.09, delta=0.3).  The same step is also timed on the 13B shape
(d=5120, 40 attention heads, prefix 4096) and on a ragged batch of 8 sequences
at the 7B shape (prefixes 256..4096), each reported per call beside the
headline.  Inputs are seeded random values of those shapes.

The metric is the step's achieved HBM bandwidth: algorithmic bytes of the step
(every weight, cache and logits byte the method must read once, plus its
outputs) divided by the device time of the step; the step time in microseconds
is reported beside it.  One JSON line goes to stdout.

Multi-GPU: the step does not shard (one sequence batch, one GPU); with N > 1
every rank runs an independent replica and rank 0 reports the aggregate.

--impl reference times the float64 CPU oracle (the only other implementation
of this method here) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import datetime
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

L2_BYTES = 129 * 1024 * 1024  # GB300 L2

METRIC = "Medusa step µs and achieved HBM GB/s (heads+tree attn+posterior), 7B shape, bs1"
UNIT = "GB/s"
CLOCK_WINDOW_S = 0.6  # the headline's timed steps continue this long for the clock record


# ------------------------------------------------------------ accounting ---

def step_bytes(cfg: synth.StepConfig, heads_frac: float = 1.0, attn_heads=None) -> dict:
    """Algorithmic bytes per step, by stage (every byte the method must move
    once).  heads_frac / attn_heads describe a sample of the workload."""
    e = 2 if cfg.dtype == "bf16" else 4
    B, K, d, V, S = cfg.B, cfg.K, cfg.d, cfg.V, cfg.top_s
    R, n = cfg.R, cfg.n
    W = (R + 63) // 64
    H = cfg.H if attn_heads is None else attn_heads
    heads = (K * (d * d + d + V * d) * e) * heads_frac + B * d * e + B * K * S * 8
    tree = B * K * S * 8 + B * 4 + B * 4 + B * R * (4 * 4 + 8 * W) + B * n * (K + 1) * 4 + B * 4
    prefix_kv = sum(2 * p * H * cfg.dh * e for p in cfg.prefix)
    attn = prefix_kv + B * R * H * cfg.dh * e * 4 + B * R * W * 8 + B * 4
    post = B * R * V * e + B * R * 12 + B * (2 + 2 * (K + 1)) * 4
    return dict(heads=heads, tree=tree, attention=attn, posterior=post,
                total=heads + tree + attn + post)


def heads_flops(cfg: synth.StepConfig) -> float:
    """Multiply-adds of the heads' two GEMVs (x2 flops each)."""
    return 2.0 * cfg.B * cfg.K * (cfg.d * cfg.d + cfg.V * cfg.d)


def measured_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            return json.load(open(p)), "measured"
        except Exception:
            pass
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ---------------------------------------------------------------- clocks ---

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running.

    Samples carry nvidia-smi's timestamp; `begin()` / `end()` mark the timed
    region on the host clock (called with the device synchronised, so they
    bracket the GPU work), and the summary keeps the samples taken inside
    it.  A region shorter than the sampling interval may hold none: the
    summary then falls back to every sample and says so."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 10

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="medusa_clocks_", suffix=".csv")
        self.f = os.fdopen(fd, "w")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
            self.f.close()
            os.unlink(self.path)
            self.path = None
        return self

    def begin(self):
        self.t0 = datetime.datetime.now()

    def end(self):
        self.t1 = datetime.datetime.now()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(2 * self.INTERVAL_MS / 1000)  # the sample after the region
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        with open(self.path) as f:
            lines = f.readlines()
        os.unlink(self.path)
        self.path = None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        samples = []  # (time, sm MHz, max MHz, active reasons)
        for line in lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                sm, mx = float(parts[2]), float(parts[3])
            except ValueError:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
            except ValueError:
                ts = None  # counted only when no sample can be placed in the region
            act = {nm for nm, v in zip(names, parts[6:10]) if v.lower().startswith("active")}
            samples.append((ts, sm, mx, act))
        if not samples:
            return None
        inside = [x for x in samples if x[0] is not None and self.t0 is not None
                  and self.t1 is not None and self.t0 <= x[0] <= self.t1]
        use = inside or samples
        return {"sm_mhz": float(np.median([x[1] for x in use])),
                "sm_max_mhz": float(max(x[2] for x in use)),
                "reasons": sorted(set().union(*(x[3] for x in use))),
                "samples": len(use), "in_timed_region": bool(inside),
                "interval_ms": self.INTERVAL_MS}


# ------------------------------------------------------------ CPU oracle ---

def oracle_step(cfg, inp, heads_sample=None, attn_heads=None):
    """One oracle pass over (a sample of) the step; returns seconds."""
    import oracle
    hi = inp["heads"]
    t0 = time.perf_counter()
    if heads_sample is None:
        ids, logp, _, _ = oracle.heads(hi.h, hi.W1, hi.b1, hi.W2, cfg.top_s)
    else:
        k = heads_sample
        ids1, logp1, _, _ = oracle.heads(hi.h, hi.W1[k:k + 1], hi.b1[k:k + 1], hi.W2[k:k + 1],
                                         cfg.top_s)
        ids = np.repeat(ids1, cfg.K, axis=1)
        logp = np.repeat(logp1, cfg.K, axis=1)
    t = oracle.build_tree(inp["root"], ids, logp, cfg.s, cfg.n, prefix_len=np.asarray(cfg.prefix))
    ai = inp["attn"]
    if attn_heads is None:
        oracle.tree_attention(ai.q, ai.k_cache, ai.v_cache, ai.prefix_len, t["anc_mask"],
                              1.0 / math.sqrt(cfg.dh))
    else:
        sl = lambda x: np.ascontiguousarray(x[..., :attn_heads, :])
        oracle.tree_attention(sl(ai.q), [sl(k) for k in ai.k_cache], [sl(v) for v in ai.v_cache],
                              ai.prefix_len, t["anc_mask"], 1.0 / math.sqrt(cfg.dh))
    oracle.posterior(inp["logits"], t["tokens"], t["parent"], t["depth"], cfg.K, oracle.TYPICAL,
                     cfg.eps, cfg.delta, cfg.temperature)
    return time.perf_counter() - t0


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(cfg, inp, nb_total: float, budget_s: float = 10.0) -> dict:
    """The oracle on the full step: single-threaded (the parity build, as it
    stands) and on every host core (its OpenMP build, same bits).  Each leg
    runs whole steps until about budget_s / 2 of host time has passed."""
    import oracle
    oracle.build()

    def leg():
        secs = []
        tb = time.perf_counter()
        while True:
            secs.append(oracle_step(cfg, inp))
            if time.perf_counter() - tb > budget_s / 2 or len(secs) >= 5:
                return secs

    oracle.set_parallel(False)
    one = leg()
    out = {"value": round(nb_total / float(np.mean(one)) / 1e9, 4), "unit": UNIT, "cores": 1,
           "kind": "oracle",
           "sample": f"{len(one)} full oracle steps of the same workload (single-threaded "
                     f"float64 C), mean {float(np.mean(one)):.2f} s per step"}
    cores = host_cores()
    if oracle.parallel_available() and cores > 1:
        oracle.set_parallel(True)
        try:
            cores = oracle.threads()
            allc = leg()
        finally:
            oracle.set_parallel(False)
        out["all_cores"] = {
            "value": round(nb_total / float(np.mean(allc)) / 1e9, 4), "unit": UNIT,
            "cores": cores, "kind": "oracle (OpenMP build, same bits)",
            "sample": f"{len(allc)} full oracle steps on {cores} threads, mean "
                      f"{float(np.mean(allc)):.2f} s per step"}
    return out


def make_inputs(cfg):
    hi = synth.heads_inputs(cfg)
    root = synth.root_tokens(cfg)
    ai = synth.attention_inputs(cfg)
    logits = synth.base_logits(cfg)
    return dict(heads=hi, root=root, attn=ai, logits_f32=logits)


def plant_on(inp, cfg, tree_np):
    lg = inp["logits_f32"].copy()
    synth.plant_chain(lg, tree_np["tokens"], tree_np["parent"], tree_np["depth"], 3,
                      synth.rng_for(cfg, "plant"))
    inp["logits"] = synth.cast(lg, cfg.dtype)


# ------------------------------------------------------------------ step ---

CALLS = ("heads", "tree", "attention", "posterior")


class StepRunner:
    """Device-resident inputs, outputs and workspace of one decoding step on
    one workload, and the step itself: the four public calls on one stream.

    The verification logits carry one planted accepted chain (length 3) on
    the tree this step's heads produce."""

    def __init__(self, m, cfg, dev, T):
        import torch
        self.m, self.cfg, self.dev = m, cfg, dev
        self.inp = inp = make_inputs(cfg)
        hi = inp["heads"]
        self.W1, self.b1, self.W2 = T(hi.W1), T(hi.b1), T(hi.W2)
        B, K, S, R, n, d = cfg.B, cfg.K, cfg.top_s, cfg.R, cfg.n, cfg.d
        # h and the root share one device buffer, so that a step's first
        # inputs arrive in one copy
        h_bytes = B * d * 2
        self.start = torch.empty(h_bytes + 16 * ((B * 4 + 15) // 16), dtype=torch.uint8,
                                 device=dev)
        self.h = self.start[:h_bytes].view(torch.bfloat16).view(B, d)
        self.root = self.start[h_bytes:h_bytes + B * 4].view(torch.int32)
        self.h.copy_(T(hi.h))
        self.root.copy_(T(inp["root"]))
        ai = inp["attn"]
        self.q = T(ai.q)
        self.kc = [T(x) for x in ai.k_cache]
        self.vc = [T(x) for x in ai.v_cache]
        self.kptr, self.vptr = m.cache_pointers(self.kc, dev), m.cache_pointers(self.vc, dev)
        self.prefix = T(ai.prefix_len)
        ws_bytes = max(m.heads_workspace_size(B, K, d, cfg.V, S),
                       m.build_tree_workspace_size(B, K, S, n),
                       m.tree_attention_workspace_size(m.BF16, B, R, cfg.H, cfg.dh, cfg.P_max),
                       m.posterior_workspace_size(B, R))
        self.ws = m.new_workspace(ws_bytes, dev)
        self.ids = torch.empty((B, K, S), dtype=torch.int32, device=dev)
        self.logp = torch.empty((B, K, S), dtype=torch.float32, device=dev)
        self.tree = m.Tree.empty(B, n, K, dev)
        self.out = torch.empty_like(self.q)
        # the posterior's results share one device buffer (one copy back per step)
        quad = lambda x: (x + 3) // 4 * 4  # int32 slots, 16-byte aligned pieces
        res_sizes = (B, B * (K + 1), B * (K + 1), B)
        self.results = torch.zeros(sum(quad(x) for x in res_sizes), dtype=torch.int32,
                                   device=dev)
        views, o = [], 0
        for x in res_sizes:
            views.append(self.results[o:o + x])
            o += quad(x)
        self.post = m.Posterior(views[0], views[1].view(B, K + 1), views[2].view(B, K + 1),
                                views[3], None)
        self.stream = torch.cuda.current_stream(dev)
        m.heads(self.h, self.W1, self.b1, self.W2, S, ws=self.ws, out=(self.ids, self.logp))
        m.build_tree(self.root, self.ids, self.logp, cfg.s, n, prefix_len=self.prefix,
                     ws=self.ws, out=self.tree)
        tnp = {k: getattr(self.tree, k).cpu().numpy() for k in ("tokens", "parent", "depth")}
        plant_on(inp, cfg, tnp)
        self.logits = T(inp["logits"])
        self.mode = m.TYPICAL if cfg.mode == "typical" else m.GREEDY
        self.nb = step_bytes(cfg)

    def step(self, record=None, before_attention=None, post=None):
        """One step; `post` replaces the device result buffers (e.g. pinned
        host ones that the posterior writes directly)."""
        m, cfg = self.m, self.cfg
        if record is not None:
            record[0].record(self.stream)
        m.heads(self.h, self.W1, self.b1, self.W2, cfg.top_s, ws=self.ws,
                out=(self.ids, self.logp))
        if record is not None:
            record[1].record(self.stream)
        m.build_tree(self.root, self.ids, self.logp, cfg.s, cfg.n, prefix_len=self.prefix,
                     ws=self.ws, out=self.tree)
        if record is not None:
            record[2].record(self.stream)
        if before_attention is not None:
            before_attention()
        m.tree_attention(self.q, self.kptr, self.vptr, self.prefix, cfg.P_max,
                         self.tree.anc_mask, out=self.out, ws=self.ws)
        if record is not None:
            record[3].record(self.stream)
        m.evaluate_posterior(self.logits, self.tree.tokens, self.tree.parent, self.tree.depth,
                             cfg.K, self.mode, cfg.eps, cfg.delta, cfg.temperature, ws=self.ws,
                             out=self.post if post is None else post)
        if record is not None:
            record[4].record(self.stream)

    def check_status(self, where: str):
        if self.m.read_device_status(self.ws) != 0:
            raise RuntimeError(f"device status set {where} ({self.cfg.name})")

    def warm(self, steps: int) -> float:
        """Untimed warm-up steps; returns a rough device time per step (s)."""
        import torch
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(self.stream)
        for _ in range(steps):
            self.step()
        z.record(self.stream)
        torch.cuda.synchronize(self.dev)
        self.check_status("during warm-up")
        return a.elapsed_time(z) * 1e-3 / max(steps, 1)

    def per_call(self, steps: int) -> dict:
        """Region 2: the same steps with an event around every call (an event
        between calls cuts the programmatic-dependent-launch overlap of
        consecutive kernels, so the calls' sum exceeds the step)."""
        import torch
        recs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
        for i in range(steps):
            self.step(recs[i])
        torch.cuda.synchronize(self.dev)
        return {c: [r[j].elapsed_time(r[j + 1]) for r in recs] for j, c in enumerate(CALLS)}

    def stages(self, per_call: dict, peak_gbs: float) -> dict:
        out = {}
        for k, v in per_call.items():
            ms = float(np.mean(v))
            gbs = self.nb[k] / (ms * 1e-3) / 1e9
            out[k] = {"us": round(ms * 1e3, 2), "us_median": round(float(np.median(v)) * 1e3, 2),
                      "us_p10": round(float(np.percentile(v, 10)) * 1e3, 2),
                      "us_p90": round(float(np.percentile(v, 90)) * 1e3, 2),
                      "bytes": int(self.nb[k]), "GB/s": round(gbs, 1),
                      "frac_hbm": round(gbs / peak_gbs, 4)}
        hms = float(np.mean(per_call["heads"]))
        out["heads"]["TFLOP/s"] = round(heads_flops(self.cfg) / (hms * 1e-3) / 1e12, 2)
        return out


def time_heads_modes(m, r, dev, T, reps: int, peak_gbs: float) -> dict:
    """The LM head joining the heads' pass and the sampled drafts, on the
    runner's workload, each timed over a loop of `reps` calls (events at the
    two ends; the weights exceed L2, so no call finds them there)."""
    import torch
    cfg = r.cfg
    B, K, S, d, V = cfg.B, cfg.K, cfg.top_s, cfg.d, cfg.V
    w_lm = T(synth.lm_head_weight(cfg))
    ws_lm = m.new_workspace(m.heads_lm_workspace_size(B, K, d, V, S), dev)
    lm_out = (torch.empty((B,), dtype=torch.int32, device=dev),
              torch.empty((B,), dtype=torch.float32, device=dev),
              torch.empty((B, K, S), dtype=torch.int32, device=dev),
              torch.empty((B, K, S), dtype=torch.float32, device=dev))
    ws_smp = m.new_workspace(m.heads_workspace_size(B, K, d, V, 1), dev)
    smp_out = (torch.empty((B, K), dtype=torch.int32, device=dev),
               torch.empty((B, K, V), dtype=torch.float32, device=dev))
    calls = {
        "heads_lm": (lambda: m.heads_lm(r.h, w_lm, r.W1, r.b1, r.W2, S, ws=ws_lm, out=lm_out),
                     r.nb["heads"] + V * d * 2 + B * 8),
        "heads_sample": (lambda: m.heads_sample(r.h, r.W1, r.b1, r.W2, 1.0, 11, 0, ws=ws_smp,
                                                out=smp_out),
                         r.nb["heads"] + B * K * V * 4),
    }
    out = {}
    for name, (fn, nbytes) in calls.items():
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(r.stream)
        for _ in range(reps):
            fn()
        z.record(r.stream)
        torch.cuda.synchronize(dev)
        us = a.elapsed_time(z) / reps * 1e3
        gbs = nbytes / (us * 1e-6) / 1e9
        out[name] = {"us": round(us, 2), "bytes": int(nbytes), "GB/s": round(gbs, 1),
                     "frac_hbm": round(gbs / peak_gbs, 4)}
    if m.read_device_status(ws_lm) != 0 or m.read_device_status(ws_smp) != 0:
        raise RuntimeError(f"device status set by the heads modes ({cfg.name})")
    del w_lm
    return out


def executor_e2e(m, r, cfg, steps: int, peak_gbs: float) -> dict:
    """The workload's step end to end through the step executor in graph
    mode: every step copies its inputs from pinned host memory (h and the
    root first; q, every sequence's tree K/V rows and the logits on the side
    stream) and the posterior writes its results into pinned host memory;
    one native call issues the step and waits for the results."""
    import torch
    B, K, R = cfg.B, cfg.K, cfg.R
    ai = r.inp["attn"]
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    host_start = torch.empty(r.start.numel(), dtype=torch.uint8).pin_memory()
    host_start.copy_(r.start.cpu())
    late = [(r.q, bf(ai.q).pin_memory()), (r.logits, bf(r.inp["logits"]).pin_memory())]
    for b in range(B):
        P = cfg.prefix[b]
        late.append((r.kc[b][P:P + R], bf(ai.k_cache[b][P:P + R]).pin_memory()))
        late.append((r.vc[b][P:P + R], bf(ai.v_cache[b][P:P + R]).pin_memory()))
    post = m.Posterior.pinned(B, R, K, with_accept=False)
    ex = m.StepExecutor(
        h=r.h, W1=r.W1, b1=r.b1, W2=r.W2, top_s=cfg.top_s, topk=(r.ids, r.logp), root=r.root,
        s=cfg.s, n=cfg.n, prefix_len=r.prefix, tree=r.tree, q=r.q, k_ptrs=r.kptr,
        v_ptrs=r.vptr, P_max=cfg.P_max, attn_out=r.out, logits=r.logits, post=post, K=K,
        mode=r.mode, eps=cfg.eps, delta=cfg.delta, temperature=cfg.temperature, ws=r.ws,
        early=[(r.start, host_start)], late=late, graph=True)
    for _ in range(3):
        ex.run()
    t0 = time.perf_counter()
    for _ in range(steps):
        ex.run()
    sec = (time.perf_counter() - t0) / steps
    ex.close()
    r.check_status("in the end-to-end steps")
    gbs = r.nb["total"] / sec / 1e9
    h2d = host_start.numel() + sum(h.numel() * h.element_size() for _, h in late)
    d2h = sum(t.numel() * t.element_size()
              for t in (post.accept_len, post.path, post.path_tokens, post.next_token))
    return {"us_per_step": round(sec * 1e6, 2), "GB/s": round(gbs, 1),
            "frac_hbm": round(gbs / peak_gbs, 4), "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": steps,
            "api": "StepExecutor(graph=True).run"}


def time_side_step(m, cfg, dev, T, steps: int, warmup: int, peak_gbs: float,
                   heads_modes: bool = False) -> dict:
    """The whole step on another workload (13B shape, batch of 8), timed like
    the headline: events at the two ends of `steps` steps, then per call."""
    import torch
    r = StepRunner(m, cfg, dev, T)
    r.warm(warmup)
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(r.stream)
    for _ in range(steps):
        r.step()
    z.record(r.stream)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(z) / steps
    pc = r.per_call(steps)
    r.check_status("in the timed steps")
    gbs = r.nb["total"] / (ms * 1e-3) / 1e9
    out = {"workload": cfg.name, "B": cfg.B, "d": cfg.d, "V": cfg.V, "K": cfg.K,
           "attn_heads": cfg.H, "head_dim": cfg.dh, "prefix": list(cfg.prefix),
           "tree_nodes": cfg.n, "accept": cfg.mode, "steps": steps,
           "us_per_step": round(ms * 1e3, 2), "bytes_per_step": int(r.nb["total"]),
           "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peak_gbs, 4),
           "stages": r.stages(pc, peak_gbs),
           "e2e": executor_e2e(m, r, cfg, steps, peak_gbs)}
    if heads_modes:
        out["heads_modes"] = time_heads_modes(m, r, dev, T, max(steps, 20), peak_gbs)
    del r
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------- size scan ---

def scan_sizes(m, dev, T, timed_loop, peak_gbs: float) -> dict:
    """Tree attention and the posterior alone over the tree-size x context
    sweep (n in {16,32,64,128} x prefix in {512,2048,8192}, greedy and
    typical) and on the ragged batch of 8, where their bytes, not the launch
    latency, set the time.  Trees come from seeded random top-s tables.
    Consecutive calls rotate through enough input copies that none finds its
    inputs in L2."""
    import torch
    out = {"attention": [], "posterior": []}
    cfgs = [synth.batch8()] + [synth.sweep(n, P) for n in synth.SWEEP_N for P in synth.SWEEP_P]
    post_done = set()
    for cfg in cfgs:
        rng = np.random.default_rng(cfg.seed)
        B, K, S = cfg.B, cfg.K, cfg.top_s
        ids = np.stack([np.stack([rng.choice(cfg.V, size=S, replace=False) for _ in range(K)])
                        for _ in range(B)]).astype(np.int32)
        p = rng.dirichlet(np.ones(S + 1), size=(B, K))[..., :S]
        logp = np.log(-np.sort(-p, axis=-1)).astype(np.float32)
        prefix = T(np.asarray(cfg.prefix, np.int32))
        tree = m.build_tree(T(np.arange(B, dtype=np.int32)), T(ids), T(logp), cfg.s, cfg.n,
                            prefix_len=prefix)
        nb = step_bytes(cfg)
        copies = max(2, int(np.ceil(2 * L2_BYTES / nb["attention"])))
        a0 = synth.attention_inputs(cfg)
        q = T(a0.q)
        k0 = [T(x) for x in a0.k_cache]
        v0 = [T(x) for x in a0.v_cache]
        # the other copies are rotations of the first (still N(0,1) values)
        kc = [k0] + [[x.roll(r, dims=0).contiguous() for x in k0] for r in range(1, copies)]
        vc = [v0] + [[x.roll(r, dims=0).contiguous() for x in v0] for r in range(1, copies)]
        ptrs = [(m.cache_pointers(k, dev), m.cache_pointers(v, dev)) for k, v in zip(kc, vc)]
        ws = m.new_workspace(max(
            m.tree_attention_workspace_size(m.BF16, B, cfg.R, cfg.H, cfg.dh, cfg.P_max),
            m.posterior_workspace_size(B, cfg.R)), dev)
        o = torch.empty_like(q)
        it = [0]

        def attn():
            kp, vp = ptrs[it[0] % copies]
            it[0] += 1
            m.tree_attention(q, kp, vp, prefix, cfg.P_max, tree.anc_mask, out=o, ws=ws)

        us = timed_loop(attn)
        # algorithmic MMA work: q.k and p.v over every prefix slot and over
        # the ancestors-or-self of each node
        depth = tree.depth.cpu().numpy()
        flops = 4.0 * cfg.H * cfg.dh * (cfg.R * sum(cfg.prefix) + float((depth + 1).sum()))
        gbs = nb["attention"] / (us * 1e-6) / 1e9
        out["attention"].append({"config": cfg.name.replace("_greedy", ""), "B": B,
                                 "prefix": list(cfg.prefix), "tree_rows": cfg.R,
                                 "us": round(us, 2), "bytes": int(nb["attention"]),
                                 "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peak_gbs, 4),
                                 "TFLOP/s": round(flops / (us * 1e-6) / 1e12, 1),
                                 "input_copies": copies})
        del kc, vc, ptrs, k0, v0
        # the posterior depends on the tree (R, B) only, not on the prefix
        if (B, cfg.R) not in post_done:
            post_done.add((B, cfg.R))
            lcopies = max(2, int(np.ceil(2 * L2_BYTES / nb["posterior"])))
            lg0 = T(synth.cast(synth.base_logits(cfg), "bf16"))
            logits = [lg0] + [lg0.roll(r, dims=-1).contiguous() for r in range(1, lcopies)]
            post = m.Posterior.empty(B, cfg.R, K, dev, with_accept=False)
            for mode, mname in ((m.GREEDY, "greedy"), (m.TYPICAL, "typical")):
                def posterior():
                    lg = logits[it[0] % lcopies]
                    it[0] += 1
                    m.evaluate_posterior(lg, tree.tokens, tree.parent, tree.depth, K, mode,
                                         ws=ws, out=post)

                us = timed_loop(posterior)
                gbs = nb["posterior"] / (us * 1e-6) / 1e9
                out["posterior"].append({"config": ("batch8" if B > 1 else f"sweep_n{cfg.n}"),
                                         "mode": mname, "B": B, "tree_rows": cfg.R,
                                         "us": round(us, 2), "bytes": int(nb["posterior"]),
                                         "GB/s": round(gbs, 1),
                                         "frac_hbm": round(gbs / peak_gbs, 4),
                                         "input_copies": lcopies})
            del logits
        if m.read_device_status(ws) != 0:
            raise RuntimeError(f"device status set in the size scan ({cfg.name})")
        del q, o
        torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------ distributed ---

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of x over all ranks (x itself without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(seconds_per_step: float, bytes_per_step: float, device=None):
    """Replicas: every rank runs the same step on its own GPU.  The job's time
    per step is the slowest rank's; the job's throughput counts every rank's
    bytes.  Returns (slowest seconds per step, aggregate GB/s)."""
    import torch.distributed as dist
    world = dist.get_world_size() if dist.is_available() and dist.is_initialized() else 1
    slowest = max_over_ranks(seconds_per_step, device)
    return slowest, world * bytes_per_step / slowest / 1e9


# -------------------------------------------------------------- reference ---

def run_reference(args, cfg):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    inp = make_inputs(cfg)
    ids, logp, _, _ = oracle.heads(inp["heads"].h, inp["heads"].W1[:1], inp["heads"].b1[:1],
                                   inp["heads"].W2[:1], cfg.top_s)
    t = oracle.build_tree(inp["root"], np.repeat(ids, cfg.K, 1), np.repeat(logp, cfg.K, 1), cfg.s,
                          cfg.n, prefix_len=np.asarray(cfg.prefix))
    plant_on(inp, cfg, t)
    attn_heads = 4
    sample_bytes = step_bytes(cfg, heads_frac=1.0 / cfg.K, attn_heads=attn_heads)["total"]
    for _ in range(args.warmup):
        oracle_step(cfg, inp, heads_sample=0, attn_heads=attn_heads)
    secs = [oracle_step(cfg, inp, heads_sample=0, attn_heads=attn_heads) for _ in range(args.steps)]
    per = float(np.mean(secs))
    value = sample_bytes / per / 1e9
    sample = (f"per step: 1 of {cfg.K} heads (W1+W2 of head 0), the full tree, {attn_heads} of "
              f"{cfg.H} attention heads, the full posterior; {sample_bytes / 1e6:.1f} MB of the "
              f"step's {step_bytes(cfg)['total'] / 1e6:.1f} MB")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(per * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, Vicuna-7B shapes)",
        "config": workload_config(cfg, args.gpus),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(cfg, world: int) -> dict:
    """The `config` object of both arms' JSON lines."""
    return {"workload": "v7b_bs1_step", "d": cfg.d, "V": cfg.V, "K": cfg.K, "s": list(cfg.s),
            "tree_nodes": cfg.n, "attn_heads": cfg.H, "head_dim": cfg.dh, "prefix": cfg.P_max,
            "batch": cfg.B, "accept": cfg.mode, "bytes_per_step": int(step_bytes(cfg)["total"]),
            "parallelism": f"replicas{world}",
            "l2": "inputs larger than L2: 1.50 GB of weights, KV and logits per step"}


# -------------------------------------------------------------------- ours ---

def run_ours(args, cfg):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    import medusa_speculative_decoding_02_gb300 as m
    m.lib()
    peaks, peak_src = measured_peaks()
    peak_gbs = peaks["hbm_gbs"]

    def T(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    run = StepRunner(m, cfg, dev, T)
    B, K, R = cfg.B, cfg.K, cfg.R
    stream = run.stream
    est = run.warm(args.warmup)
    window_steps = max(0, int(math.ceil(args.clock_window_s / max(est, 1e-6))) - args.steps)

    # Region 1: exactly `steps` steps as a user runs them, events only at the
    # two ends; `value` and `ms_per_step` come from these.  The same loop then
    # continues, without a break, for the clock window, so that the clock
    # samples cover the timed steps; its own rate is reported beside them.
    # Region 2: the same steps with an event around every call.
    t_start, t_end, t_win = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    launches0 = m.launch_count()
    with ClockSampler(dev.index) as clk:
        barrier()
        torch.cuda.synchronize(dev)
        clk.begin()
        t_start.record(stream)
        for _ in range(args.steps):
            run.step()
        t_end.record(stream)
        launches = m.launch_count() - launches0
        for _ in range(window_steps):
            run.step()
        t_win.record(stream)
        torch.cuda.synchronize(dev)
        clk.end()
        barrier()
        per_call = run.per_call(args.steps)
        run.check_status("in the timed steps")
        # the same step on the 13B shape and on the ragged batch of 8
        side = {"v13b_step": time_side_step(m, synth.v13b(), dev, T, args.steps, args.warmup,
                                            peak_gbs),
                "batch8_step": time_side_step(m, synth.batch8(), dev, T, args.steps,
                                              args.warmup, peak_gbs, heads_modes=True)}
    total_ms = t_start.elapsed_time(t_end)
    win_ms = t_start.elapsed_time(t_win)
    nb = run.nb
    s_step, value = replica_throughput(total_ms / args.steps * 1e-3, nb["total"], dev)
    ms_step = s_step * 1e3

    # ---- Region 3: rows past the step proper and the size scan, each timed
    # over a loop with events at the two ends.
    h, W1, b1, W2, S = run.h, run.W1, run.b1, run.W2, cfg.top_s
    ws, post, logits, tree = run.ws, run.post, run.logits, run.tree
    kptr, vptr, prefix, mode = run.kptr, run.vptr, run.prefix, run.mode
    # The KV-cache commit moves the accepted path's rows inside the tree
    # slots; new_prefix_len goes to its own buffer, so every repetition sees
    # the same prefix.
    new_prefix = torch.empty_like(prefix)
    row_bytes = cfg.H * cfg.dh * 2
    path_np = post.path.cpu().numpy()
    moved = int(sum(1 for b in range(B) for qq in range(int(post.accept_len[b]) + 1)
                    if path_np[b, qq] != qq))
    commit_bytes = 2 * 2 * moved * row_bytes  # K and V, each row read once and written once
    reps = max(args.steps, 20)
    host_us = {}  # wall time per call of each timed loop (host enqueue included)

    def timed_loop(fn):
        """GPU microseconds per call.  A short call can take longer to enqueue
        on the host than to run, so a sleep kernel first holds the stream
        while the host queues every call; the events then bracket GPU
        execution alone."""
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(int(2.5e9 * (2 * wall + 2e-4)))  # > the enqueue time, at <= 2.5 GHz
        a.record(stream)
        for _ in range(reps):
            fn()
        z.record(stream)
        torch.cuda.synchronize(dev)
        host_us[fn.__name__] = round(wall / reps * 1e6, 2)
        return a.elapsed_time(z) / reps * 1e3  # microseconds

    def post_only():
        m.evaluate_posterior(logits, tree.tokens, tree.parent, tree.depth, K, mode, cfg.eps,
                             cfg.delta, cfg.temperature, ws=ws, out=post)

    def post_commit():
        m.evaluate_posterior_commit(logits, tree.tokens, tree.parent, tree.depth, K, kptr, vptr,
                                    prefix, cfg.H, cfg.dh, new_prefix_len=new_prefix, mode=mode,
                                    eps=cfg.eps, delta=cfg.delta, temperature=cfg.temperature,
                                    ws=ws, out=post)

    def commit_only():
        m.commit_kv(m.BF16, kptr, vptr, prefix, post.path, post.accept_len, R, cfg.H, cfg.dh,
                    new_prefix_len=new_prefix, ws=ws)

    # the LM head joining the heads' weight pass (the root is produced, not given)
    w_lm = T(synth.lm_head_weight(cfg))
    ws_lm = m.new_workspace(m.heads_lm_workspace_size(B, K, cfg.d, cfg.V, S), dev)
    lm_out = (torch.empty((B,), dtype=torch.int32, device=dev),
              torch.empty((B,), dtype=torch.float32, device=dev),
              torch.empty((B, K, S), dtype=torch.int32, device=dev),
              torch.empty((B, K, S), dtype=torch.float32, device=dev))

    def heads_lm():
        m.heads_lm(h, w_lm, W1, b1, W2, S, ws=ws_lm, out=lm_out)

    def heads_only():
        m.heads(h, W1, b1, W2, S, ws=ws, out=(run.ids, run.logp))

    us_heads_lm = timed_loop(heads_lm)
    us_heads = timed_loop(heads_only)
    lm_bytes = nb["heads"] + cfg.V * cfg.d * 2 + B * 8
    del w_lm

    # exact speculative sampling: drafts sampled in the heads pass, then the
    # p/q posterior on a chain (verification rows: this step's first K+1 rows)
    ws_smp = m.new_workspace(max(m.heads_workspace_size(B, K, cfg.d, cfg.V, 1),
                                 m.speculative_workspace_size(B, K)), dev)
    smp_out = (torch.empty((B, K), dtype=torch.int32, device=dev),
               torch.empty((B, K, cfg.V), dtype=torch.float32, device=dev))
    chain = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    chain_logits = logits[:, :K + 1].contiguous()
    spec_out = m.Speculative(*[torch.empty(sh, dtype=torch.int32, device=dev)
                               for sh in ((B,), (B, K + 1), (B,), (B, K))])

    def heads_sample():
        m.heads_sample(h, W1, b1, W2, 1.0, 11, 0, ws=ws_smp, out=smp_out)

    def spec_post():
        m.speculative_posterior(chain_logits, chain, smp_out[1], 1.0, 11, 0, ws=ws_smp,
                                out=spec_out)

    heads_sample()
    chain[:, 0] = run.root
    chain[:, 1:] = smp_out[0]
    us_heads_sample = timed_loop(heads_sample)
    us_spec = timed_loop(spec_post)
    smp_bytes = nb["heads"] + B * K * cfg.V * 4                       # + the drafts' logits
    spec_bytes = B * (K + 1) * cfg.V * 2 + 2 * B * K * cfg.V * 4     # p rows; q rows twice
    us_post = timed_loop(post_only)
    us_post_commit = timed_loop(post_commit)
    us_commit = timed_loop(commit_only)
    if m.read_device_status(ws) != 0:
        raise RuntimeError("device status set by the commit")
    size_scan = scan_sizes(m, dev, T, timed_loop, peak_gbs)
    next_rows = {"commit_kv": {
        "us": round(us_commit, 2), "rows_moved": moved, "bytes": commit_bytes,
        "GB/s": round(commit_bytes / (us_commit * 1e-6) / 1e9, 1),
        "fused_posterior_commit_us": round(us_post_commit, 2),
        "posterior_alone_us": round(us_post, 2),
        "note": "launch-latency bound: a few hundred KB per step",
        "host_loop_us": {k: v for k, v in host_us.items()}},
        "speculative_sampling": {
            "heads_sample_us": round(us_heads_sample, 2), "heads_sample_bytes": int(smp_bytes),
            "heads_sample_GB/s": round(smp_bytes / (us_heads_sample * 1e-6) / 1e9, 1),
            "posterior_us": round(us_spec, 2), "posterior_bytes": int(spec_bytes),
            "note": "drafts by Gumbel-max in the weight pass; posterior on a chain of K drafts"},
        "heads_lm": {
            "us": round(us_heads_lm, 2), "bytes": int(lm_bytes),
            "GB/s": round(lm_bytes / (us_heads_lm * 1e-6) / 1e9, 1),
            "frac_hbm": round(lm_bytes / (us_heads_lm * 1e-6) / 1e9 / peak_gbs, 4),
            "heads_alone_us": round(us_heads, 2),
            "note": "LM head (32000 x 4096) + 5 Medusa heads in one weight pass"}}

    # ---- end to end through the public API with pinned host buffers
    ai = run.inp["attn"]
    host_start = torch.empty(run.start.numel(), dtype=torch.uint8).pin_memory()
    host_start.copy_(run.start.cpu())
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    host_in = {
        "start": host_start,  # h and the root
        "q": bf(ai.q).pin_memory(),
        "k_tree": bf(ai.k_cache[0][cfg.prefix[0]:]).pin_memory(),
        "v_tree": bf(ai.v_cache[0][cfg.prefix[0]:]).pin_memory(),
        "logits": bf(run.inp["logits"]).pin_memory(),
    }
    # the step's results (accept_len, path, path_tokens, next_token) land in
    # pinned host memory: the posterior kernel writes them there directly
    host_post = m.Posterior.pinned(B, cfg.R, K, with_accept=False)
    result_tensors = (host_post.accept_len, host_post.path, host_post.path_tokens,
                      host_post.next_token)
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in result_tensors)
    P0 = cfg.prefix[0]
    copy_stream = torch.cuda.Stream(dev)

    def e2e_issue():
        # h and the root start the step; q, the tree's K/V rows and the
        # verification logits are first read by the attention and the
        # posterior, so they travel on a second stream during the heads pass
        main = torch.cuda.current_stream(dev)
        copy_stream.wait_stream(main)
        run.start.copy_(host_in["start"], non_blocking=True)
        with torch.cuda.stream(copy_stream):
            run.q.copy_(host_in["q"], non_blocking=True)
            run.kc[0][P0:].copy_(host_in["k_tree"], non_blocking=True)
            run.vc[0][P0:].copy_(host_in["v_tree"], non_blocking=True)
            run.logits.copy_(host_in["logits"], non_blocking=True)
        run.step(before_attention=lambda: main.wait_stream(copy_stream), post=host_post)

    def e2e_eager():
        e2e_issue()
        torch.cuda.current_stream(dev).synchronize()

    # the public step API: the whole step (input copies, calls, result
    # copies) captured once as a CUDA graph, replayed every step
    graph = m.StepGraph(e2e_issue)

    def e2e_graph():
        graph.replay()
        torch.cuda.current_stream(dev).synchronize()

    # the public one-call step: the executor issues the same copies and calls
    # from native code and waits for the step; in graph mode it captured the
    # sequence once and each run is one graph launch, in stream mode each
    # run launches the kernels one by one (programmatic dependent launch kept
    # in both)
    def make_executor(graph):
        return m.StepExecutor(
            h=run.h, W1=run.W1, b1=run.b1, W2=run.W2, top_s=cfg.top_s, topk=(run.ids, run.logp),
            root=run.root, s=cfg.s, n=cfg.n, prefix_len=run.prefix, tree=run.tree, q=run.q,
            k_ptrs=run.kptr, v_ptrs=run.vptr, P_max=cfg.P_max, attn_out=run.out,
            logits=run.logits, post=host_post, K=K, mode=run.mode, eps=cfg.eps, delta=cfg.delta,
            temperature=cfg.temperature, ws=run.ws, early=[(run.start, host_in["start"])],
            late=[(run.q, host_in["q"]), (run.kc[0][P0:], host_in["k_tree"]),
                  (run.vc[0][P0:], host_in["v_tree"]), (run.logits, host_in["logits"])],
            graph=graph)

    executor = make_executor(graph=True)
    executor_stream = make_executor(graph=False)

    def e2e_native():
        executor.run(synchronize=True)

    def e2e_native_stream():
        executor_stream.run(synchronize=True)

    e2e_steps = max(3, min(args.steps, 50))

    def time_e2e(fn):
        for _ in range(2):
            fn()
        barrier()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            fn()
        return replica_throughput((time.perf_counter() - t0) / e2e_steps, nb["total"], dev)

    eager_s, eager_value = time_e2e(e2e_eager)
    graph_s, graph_value = time_e2e(e2e_graph)
    stream_s, stream_value = time_e2e(e2e_native_stream)
    e2e_s, e2e_value = time_e2e(e2e_native)
    executor_status = m.read_device_status(run.ws)
    if executor_status != 0:
        raise RuntimeError(f"device status {executor_status} set by the step executor")

    # where the end-to-end time goes: the native call that issues the step,
    # the step's span on the GPU (events on the stream around the call), and
    # what is left (launch latency to the GPU plus the host's wait for the
    # results); the input copy that gates the first kernel is timed alone
    ga, gz = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launch_us, span_us, wall_us = [], [], []
    for _ in range(e2e_steps):
        t0 = time.perf_counter()
        ga.record(stream)
        executor.run(synchronize=False)
        t1 = time.perf_counter()
        gz.record(stream)
        executor.wait()
        t2 = time.perf_counter()
        gz.synchronize()
        launch_us.append((t1 - t0) * 1e6)
        wall_us.append((t2 - t0) * 1e6)
        span_us.append(ga.elapsed_time(gz) * 1e3)

    def first_copy():
        run.start.copy_(host_in["start"], non_blocking=True)

    first_copy_us = timed_loop(first_copy)
    e2e_breakdown = {
        "wall_us": round(float(np.median(wall_us)), 2),
        "issue_call_us": round(float(np.median(launch_us)), 2),
        "gpu_span_us": round(float(np.median(span_us)), 2),
        "launch_and_sync_us": round(float(np.median(wall_us) - np.median(span_us)), 2),
        "device_resident_step_us": round(ms_step * 1e3, 2),
        "copies_on_gpu_us": round(float(np.median(span_us)) - ms_step * 1e3, 2),
        "first_input_copy_us": round(first_copy_us, 2),
        "first_input_copy_bytes": int(host_start.numel()),
    }

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return 0

    heads_ms = float(np.mean(per_call["heads"]))
    achieved = nb["heads"] / (heads_ms * 1e-3) / 1e9
    traffic = None
    tp = os.path.join(ROOT, "profiles", "heads_v7b_bs1_traffic.json")
    if os.path.exists(tp):
        try:
            traffic = json.load(open(tp)).get("bytes_per_launch")
        except Exception:
            traffic = None
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak_gbs,
                "unit": "GB/s", "frac": round(achieved / peak_gbs, 4), "traffic": traffic,
                "kernel": "medusa_heads (heads_w1 + heads_w2 + heads_reduce)",
                "peak_source": f"hbm_gbs of {peak_src}"}

    clocks = clk.summary()
    if clocks is not None:
        clocks["window"] = {"steps": args.steps + window_steps,
                            "seconds": round(win_ms * 1e-3, 3),
                            "us_per_step": round(win_ms / (args.steps + window_steps) * 1e3, 2),
                            "note": "the timed steps, continued without a break while the "
                                    "clocks are sampled"}
        clocks["step_kcycles"] = round(ms_step * clocks["sm_mhz"], 1)  # ms x MHz = k cycles

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "step_us": round(ms_step * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded, Vicuna-7B shapes: random weights, KV and logits)",
        "config": workload_config(cfg, world),
        "stages": run.stages(per_call, peak_gbs),
        **side,
        "next_rows": next_rows,
        "size_scan": size_scan,
        "roofline": roofline,
        "cpu_baseline": cpu_baseline(cfg, run.inp, nb["total"]),
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "us_per_step": round(e2e_s * 1e6, 2),
                "steps": e2e_steps,
                "api": "StepExecutor(graph=True).run = medusa_step_run (the step's input "
                       "copies from pinned memory and the four calls, captured once by the "
                       "executor as a CUDA graph, launched and awaited by one native call; the "
                       "posterior writes its results into pinned host memory)",
                "executor_stream_value": round(stream_value, 2),
                "executor_stream_us_per_step": round(stream_s * 1e6, 2),
                "torch_graph_value": round(graph_value, 2),
                "torch_graph_us_per_step": round(graph_s * 1e6, 2),
                "eager_value": round(eager_value, 2),
                "eager_us_per_step": round(eager_s * 1e6, 2),
                "breakdown": e2e_breakdown},
        "gpu_launches": int(launches),
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--clock-window-s", type=float, default=CLOCK_WINDOW_S,
                    help="seconds the headline's timed steps continue so that the clock "
                         "samples cover them (0: only the timed steps)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    cfg = synth.v7b().replace(mode="typical")
    if args.impl == "reference":
        return run_reference(args, cfg)
    return run_ours(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
