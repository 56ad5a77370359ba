"""Seeded synthetic inputs for one Medusa decoding step.

This module draws random numbers and lays them out; it holds none of the
method's arithmetic (no heads, no tree, no attention, no acceptance).  Where a
recipe needs a quantity the method defines -- the entropy of a softmax row for
the entropy-targeted logits -- the caller passes that function in.

Both the CUDA path (tests, bench) and the oracle (tests) take their inputs from
here.  bf16 tensors are returned as ``uint16`` bit patterns, produced from
float32 draws by round-to-nearest-even.

The workloads stand in for the pages' Vicuna-7B/13B decoding on MT-Bench
(neither weights nor dataset are available): same shapes (hidden size, vocab,
five heads, tree sizes, attention heads, context lengths), random values.
"""
from __future__ import annotations

import concurrent.futures as cf
import dataclasses
import os
from dataclasses import dataclass
from typing import Callable

import numpy as np

# --------------------------------------------------------------------------
# bf16 bit conversion (data layout only)
# --------------------------------------------------------------------------


def f32_to_bf16_bits(x: np.ndarray, chunk: int = 1 << 26) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); return the uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    flat = x.reshape(-1)
    out = np.empty(flat.size, np.uint16)
    for s in range(0, flat.size, chunk):
        u = flat[s:s + chunk].view(np.uint32)
        bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
        out[s:s + chunk] = ((u + bias) >> np.uint32(16)).astype(np.uint16)
    return out.reshape(x.shape)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------


@dataclass(frozen=True)
class StepConfig:
    """One workload: shapes, value distributions and acceptance settings."""
    name: str
    seed: int
    dtype: str                  # "f32" or "bf16"
    B: int                      # sequences
    d: int                      # hidden size
    V: int                      # vocabulary
    K: int                      # Medusa heads
    s: tuple                    # top-s per head
    n: int                      # tree nodes besides the root
    H: int                      # attention heads
    dh: int                     # attention head dim
    prefix: tuple               # prefix length per sequence
    w1_std: float = 0.01
    w2_std: float = 0.02
    h_std: float = 1.0
    logit_std: float = 3.0
    mode: str = "greedy"        # "greedy" or "typical"
    eps: float = 0.09
    delta: float = 0.3
    temperature: float = 1.0
    lm_head_variant: bool = False

    @property
    def R(self) -> int:
        return self.n + 1

    @property
    def top_s(self) -> int:
        return max(self.s)

    @property
    def P_max(self) -> int:
        return max(self.prefix)

    def replace(self, **kw) -> "StepConfig":
        return dataclasses.replace(self, **kw)


def tiny() -> StepConfig:
    """Tiny float32 step: d=64, V=1000, K=3, s=(2,2,2) -> 14 nodes; one
    attention head of dim 64 over 32 prefix slots."""
    return StepConfig(name="tiny", seed=0, dtype="f32", B=1, d=64, V=1000, K=3, s=(2, 2, 2),
                      n=14, H=1, dh=64, prefix=(32,), w1_std=0.02, w2_std=0.05,
                      logit_std=2.0, mode="typical")


def v7b(lm_head_variant: bool = False) -> StepConfig:
    """Vicuna-7B shape at batch 1: d=4096, V=32000, K=5, s=(4,3,2,2,1) cut to
    64 nodes, 32 heads x 128, prefix 1024."""
    return StepConfig(name="v7b" + ("_lmhead" if lm_head_variant else ""), seed=1, dtype="bf16",
                      B=1, d=4096, V=32000, K=5, s=(4, 3, 2, 2, 1), n=64, H=32, dh=128,
                      prefix=(1024,), w1_std=0.01, w2_std=0.02, logit_std=3.0, mode="greedy",
                      lm_head_variant=lm_head_variant)


def v13b() -> StepConfig:
    """Vicuna-13B shape at batch 1: d=5120, 40 heads x 128, prefix 4096,
    typical acceptance on entropy-targeted logits."""
    return StepConfig(name="v13b", seed=2, dtype="bf16", B=1, d=5120, V=32000, K=5,
                      s=(4, 3, 2, 2, 1), n=64, H=40, dh=128, prefix=(4096,), logit_std=1.0,
                      mode="typical")


def sweep(n: int, P: int, mode: str = "greedy") -> StepConfig:
    """7B shape, s=(8,4,4,2,2) cut to n nodes, prefix P."""
    return StepConfig(name=f"sweep_n{n}_P{P}_{mode}", seed=3, dtype="bf16", B=1, d=4096,
                      V=32000, K=5, s=(8, 4, 4, 2, 2), n=n, H=32, dh=128, prefix=(P,),
                      mode=mode)


def batch8() -> StepConfig:
    """7B shape, 8 independent sequences, ragged prefixes U{256..4096}."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([4, 7])))
    prefix = tuple(int(x) for x in rng.integers(256, 4096, size=8, endpoint=True))
    return StepConfig(name="batch8", seed=4, dtype="bf16", B=8, d=4096, V=32000, K=5,
                      s=(4, 3, 2, 2, 1), n=64, H=32, dh=128, prefix=prefix, mode="typical")


SWEEP_N = (16, 32, 64, 128)
SWEEP_P = (512, 2048, 8192)

# component streams: each input part has its own child generator so that any
# subset of parts can be drawn alone and still match.
_STREAMS = {"h": 1, "w1": 2, "b1": 3, "w2": 4, "root": 5, "q": 6, "kv": 7, "logits": 8,
            "plant": 9, "uniform": 10}


def rng_for(cfg: StepConfig, part: str, rep: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([cfg.seed, _STREAMS[part], rep])))


_CHUNK = 1 << 22
_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        _POOL = cf.ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1)))
    return _POOL


def _normal_keyed(key: tuple, shape, std: float, dtype: str) -> np.ndarray:
    """N(0, std) array drawn in fixed chunks of 2^22 elements; chunk c comes from
    its own PCG64 stream seeded by (key, c), so the values do not depend on how
    many threads fill the chunks."""
    size = int(np.prod(shape))
    out = np.empty(size, np.uint16 if dtype == "bf16" else np.float32)

    def fill(c):
        lo, hi = c * _CHUNK, min(size, (c + 1) * _CHUNK)
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([*key, c])))
        x = g.standard_normal(size=hi - lo, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[lo:hi] = f32_to_bf16_bits(x) if dtype == "bf16" else x

    list(_pool().map(fill, range((size + _CHUNK - 1) // _CHUNK)))
    return out.reshape(shape)


def _normal(cfg: StepConfig, part: str, rep: int, shape, std, dtype, *sub) -> np.ndarray:
    return _normal_keyed((cfg.seed, _STREAMS[part], rep, *sub), shape, std, dtype)


def _zeros(shape, dtype) -> np.ndarray:
    return np.zeros(shape, np.uint16 if dtype == "bf16" else np.float32)


@dataclass
class HeadsInputs:
    h: np.ndarray      # [B,d]
    W1: np.ndarray     # [K,d,d]
    b1: np.ndarray     # [K,d]
    W2: np.ndarray     # [K,V,d]


def heads_inputs(cfg: StepConfig, rep: int = 0) -> HeadsInputs:
    """h ~ N(0, h_std); W1 ~ N(0, w1_std); b1 = 0; W2 ~ N(0, w2_std).  The
    LM-head variant sets W1 = 0, b1 = 0 and every head's W2 to one shared
    LM-head matrix W_lm ~ N(0, w2_std)."""
    h = hidden_states(cfg, rep)
    b1 = _zeros((cfg.K, cfg.d), cfg.dtype)
    if cfg.lm_head_variant:
        W1 = _zeros((cfg.K, cfg.d, cfg.d), cfg.dtype)
        w_lm = lm_head_weight(cfg, rep)
        W2 = np.empty((cfg.K, cfg.V, cfg.d), w_lm.dtype)
        W2[:] = w_lm[None]
    else:
        W1 = _normal(cfg, "w1", rep, (cfg.K, cfg.d, cfg.d), cfg.w1_std, cfg.dtype)
        W2 = _normal(cfg, "w2", rep, (cfg.K, cfg.V, cfg.d), cfg.w2_std, cfg.dtype)
    return HeadsInputs(h=h, W1=W1, b1=b1, W2=W2)


def hidden_states(cfg: StepConfig, rep: int = 0) -> np.ndarray:
    """h [B,d] ~ N(0, h_std) alone (the same values heads_inputs returns)."""
    return _normal(cfg, "h", rep, (cfg.B, cfg.d), cfg.h_std, cfg.dtype)


def lm_head_weight(cfg: StepConfig, rep: int = 0) -> np.ndarray:
    """The base model's LM head W_lm [V,d] ~ N(0, w2_std) (the same matrix the
    LM-head variant copies into every head's W2)."""
    return _normal(cfg, "w2", rep, (cfg.V, cfg.d), cfg.w2_std, cfg.dtype, 1)


def root_tokens(cfg: StepConfig, rep: int = 0) -> np.ndarray:
    """The LM head's greedy token per sequence (an input: the base model is not run)."""
    return rng_for(cfg, "root", rep).integers(0, cfg.V, size=cfg.B).astype(np.int32)


@dataclass
class AttentionInputs:
    q: np.ndarray              # [B,R,H,dh]
    k_cache: list              # B arrays [P_b+R,H,dh]
    v_cache: list
    prefix_len: np.ndarray     # [B] int32


def attention_inputs(cfg: StepConfig, rep: int = 0, extra_slots: int = 0) -> AttentionInputs:
    """q and every K/V slot ~ N(0,1).  Sequence b's cache holds P_b prefix slots
    followed by R tree slots (plus ``extra_slots`` spare rows)."""
    q = _normal(cfg, "q", rep, (cfg.B, cfg.R, cfg.H, cfg.dh), 1.0, cfg.dtype)
    ks, vs = [], []
    for b in range(cfg.B):
        rows = cfg.prefix[b] + cfg.R + extra_slots
        ks.append(_normal(cfg, "kv", rep, (rows, cfg.H, cfg.dh), 1.0, cfg.dtype, b, 0))
        vs.append(_normal(cfg, "kv", rep, (rows, cfg.H, cfg.dh), 1.0, cfg.dtype, b, 1))
    return AttentionInputs(q=q, k_cache=ks, v_cache=vs,
                           prefix_len=np.asarray(cfg.prefix, np.int32))


def base_logits(cfg: StepConfig, rep: int = 0) -> np.ndarray:
    """Verification logits [B,R,V] ~ N(0, logit_std) as float32 (not yet cast)."""
    return _normal(cfg, "logits", rep, (cfg.B, cfg.R, cfg.V), cfg.logit_std, "f32")


def plant_bernoulli(logits: np.ndarray, tokens: np.ndarray, parent: np.ndarray,
                    rng: np.random.Generator, prob: float = 0.5, amount: float = 6.0) -> np.ndarray:
    """For every non-root node, with probability ``prob`` add ``amount`` to the
    logit of its token in its parent's row.  In place on float32 [B,R,V]."""
    B, R = tokens.shape
    for b in range(B):
        for i in range(1, R):
            if rng.random() < prob:
                logits[b, parent[b, i], tokens[b, i]] += np.float32(amount)
    return logits


def plant_chain(logits: np.ndarray, tokens: np.ndarray, parent: np.ndarray, depth: np.ndarray,
                L_star: int, rng: np.random.Generator, lift: float = 4.0) -> np.ndarray:
    """Plant one accepted chain of length ``L_star`` per sequence: pick a node u
    at depth L_star uniformly (the deepest available depth if none), and for
    every edge on root -> u set the child's logit in the parent's row to the
    row maximum plus ``lift``.  Children of u are left alone.  In place."""
    B, R = tokens.shape
    for b in range(B):
        L = min(L_star, int(depth[b].max()))
        if L <= 0:
            continue
        cand = np.nonzero(depth[b] == L)[0]
        u = int(cand[rng.integers(0, cand.size)])
        chain = []
        while u > 0:
            chain.append(u)
            u = int(parent[b, u])
        for c in reversed(chain):
            p = int(parent[b, c])
            row = logits[b, p]
            row[tokens[b, c]] = row.max() + np.float32(lift)
    return logits


def scale_rows_to_entropy(logits: np.ndarray, target: float,
                          entropy_fn: Callable[[np.ndarray, float], float],
                          tol: float = 1e-6) -> np.ndarray:
    """Divide every row by a temperature found by bisection (in float64) so that
    ``entropy_fn(row, T) == target`` within ``tol``.  Returns float32 rows.
    ``entropy_fn(row_float64, T)`` is supplied by the caller."""
    out = np.empty_like(logits, dtype=np.float32)
    flat_in = logits.reshape(-1, logits.shape[-1]).astype(np.float64)
    flat_out = out.reshape(-1, logits.shape[-1])
    for r in range(flat_in.shape[0]):
        row = flat_in[r]
        lo, hi = 1e-4, 1e4          # entropy rises with T
        T = 1.0
        for _ in range(200):
            T = np.sqrt(lo * hi)
            e = entropy_fn(row, T)
            if abs(e - target) <= tol:
                break
            if e < target:
                lo = T
            else:
                hi = T
        flat_out[r] = (row / T).astype(np.float32)
    return out


def cast(x: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16_bits(x) if dtype == "bf16" else np.ascontiguousarray(x, np.float32)


def uniforms(cfg: StepConfig, shape, rep: int = 0) -> np.ndarray:
    """U[0,1) float32 draws (for the sampling-based acceptance rule)."""
    return rng_for(cfg, "uniform", rep).random(size=shape, dtype=np.float32)
