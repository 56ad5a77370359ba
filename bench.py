"""Benchmark one Medusa decoding step on synthetic Vicuna-7B-shaped inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one pass of the whole hot path on one batch of input:
    medusa_heads -> medusa_build_tree -> medusa_tree_attention -> medusa_evaluate_posterior
at the 7B shape, batch 1 (d=4096, V=32000, K=5 heads, s=(4,3,2,2,1) cut to 64
nodes, 32 x 128 attention heads, prefix 1024, typical acceptance eps=0.09,
delta=0.3).  Inputs are seeded random values of those shapes.

The metric is the step's achieved HBM bandwidth: algorithmic bytes of the step
(every weight, cache and logits byte the method must read once, plus its
outputs) divided by the device time of the step; the step time in microseconds
is reported beside it.  One JSON line goes to stdout.

Multi-GPU: the step does not shard (one sequence, one GPU); with N > 1 every
rank runs an independent replica and rank 0 reports the aggregate.

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


def scan_sizes(m, dev, T, timed_loop) -> dict:
    """Tree attention and the posterior alone on larger workloads than the bs1
    step (ragged batch of 8, prefix 8192), where their bytes, not the launch
    latency, set the time.  Trees come from seeded random top-s tables."""
    import torch
    out = {"attention": [], "posterior": []}
    for cfg in (synth.batch8(), synth.sweep(64, 8192), synth.sweep(128, 8192)):
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
        # enough copies that consecutive calls never find their inputs in L2
        copies = max(2, int(np.ceil(2 * L2_BYTES / nb["attention"])))
        sets = [synth.attention_inputs(cfg, rep=r) for r in range(copies)]
        q = T(sets[0].q)
        kc = [[T(x) for x in a.k_cache] for a in sets]
        vc = [[T(x) for x in a.v_cache] for a in sets]
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
        out["attention"].append({"config": cfg.name, "B": B, "prefix": list(cfg.prefix),
                                 "tree_rows": cfg.R, "us": round(us, 2),
                                 "bytes": int(nb["attention"]),
                                 "GB/s": round(nb["attention"] / (us * 1e-6) / 1e9, 1),
                                 "TFLOP/s": round(flops / (us * 1e-6) / 1e12, 1)})
        if B > 1:
            lcopies = max(2, int(np.ceil(2 * L2_BYTES / nb["posterior"])))
            lg0 = T(synth.cast(synth.base_logits(cfg), "bf16"))
            logits = [lg0] + [lg0.roll(r, dims=-1).contiguous() for r in range(1, lcopies)]
            post = m.Posterior.empty(B, cfg.R, K, dev, with_accept=False)

            def posterior():
                lg = logits[it[0] % lcopies]
                it[0] += 1
                m.evaluate_posterior(lg, tree.tokens, tree.parent, tree.depth, K, m.TYPICAL,
                                     ws=ws, out=post)

            us = timed_loop(posterior)
            out["posterior"].append({"config": cfg.name, "B": B, "tree_rows": cfg.R,
                                     "us": round(us, 2), "bytes": int(nb["posterior"]),
                                     "GB/s": round(nb["posterior"] / (us * 1e-6) / 1e9, 1)})
        if m.read_device_status(ws) != 0:
            raise RuntimeError(f"device status set in the size scan ({cfg.name})")
        out["attention"][-1]["input_copies"] = copies
        if B > 1:
            out["posterior"][-1]["input_copies"] = lcopies
            del logits
        del kc, vc, q, o, sets
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

    def T(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    inp = make_inputs(cfg)
    hi = inp["heads"]
    W1, b1, W2 = T(hi.W1), T(hi.b1), T(hi.W2)
    # h and the root share one device buffer, so that a step's first inputs
    # arrive in one copy
    h_bytes = cfg.B * cfg.d * 2
    start = torch.empty(h_bytes + 16 * ((cfg.B * 4 + 15) // 16), dtype=torch.uint8, device=dev)
    h = start[:h_bytes].view(torch.bfloat16).view(cfg.B, cfg.d)
    root = start[h_bytes:h_bytes + cfg.B * 4].view(torch.int32)
    h.copy_(T(hi.h))
    root.copy_(T(inp["root"]))
    ai = inp["attn"]
    q = T(ai.q)
    kc = [T(x) for x in ai.k_cache]
    vc = [T(x) for x in ai.v_cache]
    kptr, vptr = m.cache_pointers(kc, dev), m.cache_pointers(vc, dev)
    prefix = T(ai.prefix_len)
    B, K, S, R, n = cfg.B, cfg.K, cfg.top_s, cfg.R, cfg.n
    ws_bytes = max(m.heads_workspace_size(B, K, cfg.d, cfg.V, S),
                   m.build_tree_workspace_size(B, K, S, n),
                   m.tree_attention_workspace_size(m.BF16, B, R, cfg.H, cfg.dh, cfg.P_max),
                   m.posterior_workspace_size(B, R))
    ws = m.new_workspace(ws_bytes, dev)
    ids = torch.empty((B, K, S), dtype=torch.int32, device=dev)
    logp = torch.empty((B, K, S), dtype=torch.float32, device=dev)
    tree = m.Tree.empty(B, n, K, dev)
    out = torch.empty_like(q)
    # the posterior's results share one device buffer (one copy back per step)
    quad = lambda n: (n + 3) // 4 * 4  # int32 slots, 16-byte aligned pieces
    res_sizes = (B, B * (K + 1), B * (K + 1), B)
    results = torch.zeros(sum(quad(x) for x in res_sizes), dtype=torch.int32, device=dev)
    res_views, o = [], 0
    for x in res_sizes:
        res_views.append(results[o:o + x])
        o += quad(x)
    post = m.Posterior(res_views[0], res_views[1].view(B, K + 1), res_views[2].view(B, K + 1),
                       res_views[3], None)
    stream = torch.cuda.current_stream(dev)

    # the verification logits carry one planted chain on this step's tree
    m.heads(h, W1, b1, W2, S, ws=ws, out=(ids, logp))
    m.build_tree(root, ids, logp, cfg.s, n, prefix_len=prefix, ws=ws, out=tree)
    tnp = {k: getattr(tree, k).cpu().numpy() for k in ("tokens", "parent", "depth")}
    plant_on(inp, cfg, tnp)
    logits = T(inp["logits"])
    mode = m.TYPICAL if cfg.mode == "typical" else m.GREEDY

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]

    def step(record=None, before_attention=None):
        if record is not None:
            record[0].record(stream)
        m.heads(h, W1, b1, W2, S, ws=ws, out=(ids, logp))
        if record is not None:
            record[1].record(stream)
        m.build_tree(root, ids, logp, cfg.s, n, prefix_len=prefix, ws=ws, out=tree)
        if record is not None:
            record[2].record(stream)
        if before_attention is not None:
            before_attention()
        m.tree_attention(q, kptr, vptr, prefix, cfg.P_max, tree.anc_mask, out=out, ws=ws)
        if record is not None:
            record[3].record(stream)
        m.evaluate_posterior(logits, tree.tokens, tree.parent, tree.depth, K, mode, cfg.eps,
                             cfg.delta, cfg.temperature, ws=ws, out=post)
        if record is not None:
            record[4].record(stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if m.read_device_status(ws) != 0:
        raise RuntimeError("device status set during warm-up")

    # Region 1: the step as a user runs it, events only at the two ends (an
    # event between calls would cut the programmatic-dependent-launch overlap
    # of consecutive kernels).  Region 2: the same steps with an event around
    # every call, for the per-call breakdown and the heads roofline.
    per_call = {k: [] for k in ("heads", "tree", "attention", "posterior")}
    recs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    launches0 = m.launch_count()
    with ClockSampler(dev.index) as clk:
        barrier()
        torch.cuda.synchronize(dev)
        clk.begin()
        t_start.record(stream)
        for i in range(args.steps):
            step()
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        launches = m.launch_count() - launches0
        for i in range(args.steps):
            step(recs[i])
        torch.cuda.synchronize(dev)
        clk.end()
    total_ms = t_start.elapsed_time(t_end)
    for r in recs:
        per_call["heads"].append(r[0].elapsed_time(r[1]))
        per_call["tree"].append(r[1].elapsed_time(r[2]))
        per_call["attention"].append(r[2].elapsed_time(r[3]))
        per_call["posterior"].append(r[3].elapsed_time(r[4]))
    nb = step_bytes(cfg)
    s_step, value = replica_throughput(total_ms / args.steps * 1e-3, nb["total"], dev)
    ms_step = s_step * 1e3

    # ---- Region 3: the KV-cache commit (a row past the step proper), alone
    # and fused into the posterior, each timed over a loop with events at the
    # two ends.  The commit moves the accepted path's rows inside the tree
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
        m.heads(h, W1, b1, W2, S, ws=ws, out=(ids, logp))

    us_heads_lm = timed_loop(heads_lm)
    us_heads = timed_loop(heads_only)
    lm_bytes = nb["heads"] + cfg.V * cfg.d * 2 + B * 8

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
    chain[:, 0] = root
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
    size_scan = scan_sizes(m, dev, T, timed_loop)
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
            "frac_hbm": None, "heads_alone_us": round(us_heads, 2),
            "note": "LM head (32000 x 4096) + 5 Medusa heads in one weight pass"}}

    # ---- end to end through the public API with pinned host buffers
    host_start = torch.empty(start.numel(), dtype=torch.uint8).pin_memory()
    host_start.copy_(start.cpu())
    host_in = {
        "start": host_start,  # h and the root
        "q": torch.from_numpy(np.ascontiguousarray(ai.q).view(np.int16)).view(torch.bfloat16).pin_memory(),
        "k_tree": torch.from_numpy(ai.k_cache[0][cfg.prefix[0]:].view(np.int16)).view(torch.bfloat16).pin_memory(),
        "v_tree": torch.from_numpy(ai.v_cache[0][cfg.prefix[0]:].view(np.int16)).view(torch.bfloat16).pin_memory(),
        "logits": torch.from_numpy(inp["logits"].view(np.int16)).view(torch.bfloat16).pin_memory(),
    }
    host_out = {"results": torch.empty(results.shape, dtype=torch.int32).pin_memory()}
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())
    P0 = cfg.prefix[0]

    copy_stream = torch.cuda.Stream(dev)

    def e2e_issue():
        # h and the root start the step; q, the tree's K/V rows and the
        # verification logits are first read by the attention and the
        # posterior, so they travel on a second stream during the heads pass
        main = torch.cuda.current_stream(dev)
        copy_stream.wait_stream(main)
        start.copy_(host_in["start"], non_blocking=True)
        with torch.cuda.stream(copy_stream):
            q.copy_(host_in["q"], non_blocking=True)
            kc[0][P0:].copy_(host_in["k_tree"], non_blocking=True)
            vc[0][P0:].copy_(host_in["v_tree"], non_blocking=True)
            logits.copy_(host_in["logits"], non_blocking=True)
        step(before_attention=lambda: main.wait_stream(copy_stream))
        host_out["results"].copy_(results, non_blocking=True)

    def e2e_eager():
        e2e_issue()
        torch.cuda.current_stream(dev).synchronize()

    # the public step API: the whole step (input copies, calls, result
    # copies) captured once as a CUDA graph, replayed every step
    graph = m.StepGraph(e2e_issue)

    def e2e_graph():
        graph.replay()
        torch.cuda.current_stream(dev).synchronize()

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
    e2e_s, e2e_value = time_e2e(e2e_graph)

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return 0

    peaks, peak_src = measured_peaks()
    for rows in size_scan.values():
        for r in rows:
            r["frac_hbm"] = round(r["GB/s"] / peaks["hbm_gbs"], 4)
    next_rows["heads_lm"]["frac_hbm"] = round(
        next_rows["heads_lm"]["GB/s"] / peaks["hbm_gbs"], 4)
    heads_ms = float(np.mean(per_call["heads"]))
    achieved = nb["heads"] / (heads_ms * 1e-3) / 1e9
    traffic = None
    tp = os.path.join(ROOT, "profiles", "heads_v7b_bs1_traffic.json")
    if os.path.exists(tp):
        try:
            traffic = json.load(open(tp)).get("bytes_per_launch")
        except Exception:
            traffic = None
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                "kernel": "medusa_heads (heads_w1 + heads_w2 + heads_reduce)",
                "peak_source": f"hbm_gbs of {peak_src}"}

    # ---- CPU baseline: the oracle on the full step, ~10 s of host work
    import oracle
    oracle.build()
    cpu_secs = []
    tb = time.perf_counter()
    while True:
        cpu_secs.append(oracle_step(cfg, inp))
        if time.perf_counter() - tb > 10.0 or len(cpu_secs) >= 5:
            break
    cpu_value = nb["total"] / float(np.mean(cpu_secs)) / 1e9

    stages = {k: {"us": round(float(np.mean(v)) * 1e3, 2),
                  "us_median": round(float(np.median(v)) * 1e3, 2),
                  "us_p10": round(float(np.percentile(v, 10)) * 1e3, 2),
                  "us_p90": round(float(np.percentile(v, 90)) * 1e3, 2),
                  "GB/s": round(nb[k] / (float(np.mean(v)) * 1e-3) / 1e9, 1),
                  "frac_hbm": round(nb[k] / (float(np.mean(v)) * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}
              for k, v in per_call.items()}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "step_us": round(ms_step * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded, Vicuna-7B shapes: random weights, KV and logits)",
        "config": workload_config(cfg, world),
        "stages": stages,
        "next_rows": next_rows,
        "size_scan": size_scan,
        "roofline": roofline,
        "cpu_baseline": {"value": round(cpu_value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{len(cpu_secs)} full oracle steps of the same workload "
                                   f"(single-threaded float64 C), mean "
                                   f"{float(np.mean(cpu_secs)):.2f} s per step"},
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "us_per_step": round(e2e_s * 1e6, 2),
                "steps": e2e_steps, "api": "StepGraph.replay (copies + calls in one CUDA graph)",
                "eager_value": round(eager_value, 2),
                "eager_us_per_step": round(eager_s * 1e6, 2)},
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    cfg = synth.v7b().replace(mode="typical")
    if args.impl == "reference":
        return run_reference(args, cfg)
    return run_ours(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
