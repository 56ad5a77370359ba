"""GPU-vs-oracle parity of exact speculative sampling (medusa_heads_sample and
medusa_speculative_posterior), through the C ABI, plus distribution checks
of the GPU samples themselves.

Both sides draw from the same counter-based Philox4x64-10 streams, so a
sampled token is a deterministic argmax and is compared bit-exactly, except
where the oracle's Gumbel keys of the GPU's choice and its own differ by
less than 1e-3 (the sides compute in fp32 and fp64).  An acceptance decision
whose oracle margin |log p - log q - log u| is below 1e-3 is exempt the same
way; after an exemption the oracle is re-run with the GPU's decisions.
Floats (the drafts' logits) within max-abs 1e-2 and relative 2e-2.
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp
from scipy.stats import chisquare

import oracle
import synth
import medusa_speculative_decoding_02_gb300 as m
from medusa_speculative_decoding_02_gb300 import build as mbuild

pytestmark = pytest.mark.gpu

GAP = 1e-3


@pytest.fixture(scope="module")
def dev():
    mbuild.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def T(a, dev):
    a = np.ascontiguousarray(a)
    if not a.flags.writeable:
        a = a.copy()
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(a).to(dev)


def N(t):
    return t.detach().cpu().numpy()


def chi2_pvalue(counts, probs):
    counts = np.asarray(counts, np.float64)
    probs = np.asarray(probs, np.float64)
    exp = probs / probs.sum() * counts.sum()
    keep = exp > 1e-12
    assert counts[~keep].sum() == 0
    return chisquare(counts[keep], exp[keep]).pvalue


# ------------------------------------------------------------------ drafts ---

@pytest.mark.parametrize("dtype,B,d,V,K,temp", [
    ("f32", 1, 64, 1000, 3, 1.0), ("bf16", 2, 72, 1031, 2, 0.7), ("bf16", 1, 4096, 32000, 5, 1.0),
    ("f32", 8, 136, 999, 5, 2.0), ("bf16", 3, 256, 4000, 8, 0.5)])
def test_heads_sample_matches_oracle(dev, dtype, B, d, V, K, temp):
    cfg = synth.tiny().replace(name=f"smp{dtype}{B}{d}{V}{K}", dtype=dtype, B=B, d=d, V=V, K=K,
                               s=(1,) * K, w1_std=0.05, w2_std=0.05 if d < 4096 else 0.02)
    hi = synth.heads_inputs(cfg)
    seed, step = 1234 + B, 17
    drafts, dl = m.heads_sample(T(hi.h, dev), T(hi.W1, dev), T(hi.b1, dev), T(hi.W2, dev), temp,
                                seed, step)
    torch.cuda.synchronize()
    g_dr, g_dl = N(drafts), N(dl)
    o_dr, o_lg, o_keys = oracle.draft_sample(hi.h, hi.W1, hi.b1, hi.W2, temp, seed, step,
                                             want_keys=True)
    err = np.abs(g_dl - o_lg)
    assert err.max() <= 1e-2, err.max()
    assert np.linalg.norm(g_dl - o_lg) <= 2e-2 * np.linalg.norm(o_lg)
    for b in range(B):
        for k in range(K):
            a, o = int(g_dr[b, k]), int(o_dr[b, k])
            if a != o:
                gap = o_keys[b, k, o] - o_keys[b, k, a]
                assert gap < GAP, (b, k, a, o, gap)


def test_heads_sample_frequencies(dev):
    """The GPU drafts follow softmax(logits / T): heads whose logits are set
    by scaled one-hot rows, 8 sequences x 400 steps, chi-square per head."""
    rng = np.random.default_rng(21)
    K, V, d, B, temp = 3, 16, 8, 8, 0.8
    c = rng.uniform(-2, 2, size=(K, V)).astype(np.float32)
    W1 = np.zeros((K, d, d), np.float32)
    W2 = np.zeros((K, V, d), np.float32)
    W2[:, :, 2] = c
    h = np.zeros((B, d), np.float32)
    h[:, 2] = 1.0
    hd, W1d, W2d = T(h, dev), T(W1, dev), T(W2, dev)
    ws = m.new_workspace(m.heads_workspace_size(B, K, d, V, 1), dev)
    out = (torch.empty((B, K), dtype=torch.int32, device=dev),
           torch.empty((B, K, V), dtype=torch.float32, device=dev))
    counts = np.zeros((K, V), np.int64)
    for step in range(400):
        m.heads_sample(hd, W1d, None, W2d, temp, 77, step, ws=ws, out=out)
        dr = N(out[0])
        for k in range(K):
            counts[k] += np.bincount(dr[:, k], minlength=V)
    for k in range(K):
        p = np.exp(c[k].astype(np.float64) / temp - logsumexp(c[k].astype(np.float64) / temp))
        assert chi2_pvalue(counts[k], p) > 1e-4, (k, counts[k])


# --------------------------------------------------------------- posterior ---

def run_spec(dev, logits, tokens, dl, temp, seed, step):
    out = m.speculative_posterior(T(logits, dev), T(tokens, dev), T(dl, dev), temp, seed, step)
    torch.cuda.synchronize()
    return {k: N(getattr(out, k)) for k in ("accept_len", "path_tokens", "next_token", "accept")}


def check_spec(g, logits, tokens, dl, temp, seed, step):
    o = oracle.speculative_posterior(logits, tokens, dl, temp, seed, step)
    mism = g["accept"] != o["accept"]
    near = np.abs(o["margin"]) < GAP
    # a decision past the oracle's own rejection is -1 there; compare reached ones
    reached = (o["accept"] >= 0) & (g["accept"] >= 0)
    assert not (mism & reached & ~near).any(), np.argwhere(mism & reached & ~near)
    if mism.any():
        fa = np.where(g["accept"] >= 0, g["accept"], 1)
        o = oracle.speculative_posterior(logits, tokens, dl, temp, seed, step, forced_accept=fa)
    assert np.array_equal(g["accept_len"], o["accept_len"])
    assert np.array_equal(g["path_tokens"], o["path_tokens"])
    assert np.array_equal(g["accept"], o["accept"])
    for b in range(len(g["next_token"])):
        a, e = int(g["next_token"][b]), int(o["next_token"][b])
        if a != e:
            keys = o["sample_keys"][b]
            assert keys[e] - keys[a] < GAP, (b, a, e, keys[e], keys[a])
    return o


@pytest.mark.parametrize("dtype,B,V,K,temp", [
    ("f32", 4, 1000, 3, 1.0), ("bf16", 2, 32000, 5, 1.0), ("bf16", 8, 4000, 5, 0.7),
    ("f32", 3, 1024, 8, 1.5), ("bf16", 1, 32000, 1, 0.5)])
def test_speculative_matches_oracle(dev, dtype, B, V, K, temp):
    """Random verification rows and draft logits, drafts sampled by the
    oracle's draft sampler from those draft logits (so that rejections and
    acceptances both occur); tokens, decisions and the next token against
    the oracle."""
    rng = np.random.default_rng(V + K)
    p_f = rng.normal(0, 2.0, size=(B, K + 1, V)).astype(np.float32)
    q = rng.normal(0, 2.0, size=(B, K, V)).astype(np.float32)
    # make p and q overlap so that some drafts pass: p rows share half of q's mass
    p_f[:, :K] = 0.5 * p_f[:, :K] + q
    logits = synth.cast(p_f, dtype)
    seed, step = 99, 5
    tokens = np.zeros((B, K + 1), np.int32)
    tokens[:, 0] = rng.integers(0, V, size=B)
    for b in range(B):
        for k in range(K):
            g = np.array([-math.log(-math.log(oracle.uniform(seed, step + 1, 1, b, k, v)))
                          for v in range(V)])
            tokens[b, k + 1] = int(np.argmax(q[b, k].astype(np.float64) / temp + g))
    g = run_spec(dev, logits, tokens, q, temp, seed, step)
    check_spec(g, logits, tokens, q, temp, seed, step)


def test_speculative_gpu_distribution(dev):
    """The GPU's emitted tokens follow p exactly: 4096 sequences with the same
    p and q (each its own random streams), drafts sampled by the GPU's heads
    from q; the first emitted token (draft if accepted, else the
    replacement) against p_0, the second (after an accepted first draft)
    against p_1, and the first acceptance rate against sum_v min(p_0, q_1)."""
    rng = np.random.default_rng(31)
    K, V, d, B = 2, 16, 8, 4096
    temp = 1.0
    qc = rng.normal(0, 1.0, size=(K, V)).astype(np.float32)
    pc = rng.normal(0, 1.0, size=(K + 1, V)).astype(np.float32)
    W1 = np.zeros((K, d, d), np.float32)
    W2 = np.zeros((K, V, d), np.float32)
    W2[:, :, 3] = qc
    # heads_sample takes at most 8 sequences per call: sample in blocks of 8
    drafts = np.zeros((B, K), np.int32)
    hb = np.zeros((8, d), np.float32)
    hb[:, 3] = 1.0
    hd, W1d, W2d = T(hb, dev), T(W1, dev), T(W2, dev)
    for blk in range(B // 8):
        dr, _ = m.heads_sample(hd, W1d, None, W2d, temp, 5, 1000 + blk)
        drafts[blk * 8:(blk + 1) * 8] = N(dr)
    tokens = np.concatenate([np.zeros((B, 1), np.int32), drafts], axis=1)
    logits = np.ascontiguousarray(np.broadcast_to(pc, (B, K + 1, V)))
    dl = np.ascontiguousarray(np.broadcast_to(qc, (B, K, V)))
    g = run_spec(dev, logits, tokens, dl, temp, 6, 0)
    p = np.exp(pc - logsumexp(pc, axis=1, keepdims=True))
    q = np.exp(qc - logsumexp(qc, axis=1, keepdims=True))
    L = g["accept_len"]
    first = np.where(L >= 1, tokens[:, 1], g["next_token"])
    assert chi2_pvalue(np.bincount(first, minlength=V), p[0]) > 1e-4
    sel = L >= 1
    second = np.where(L[sel] >= 2, tokens[sel, 2], g["next_token"][sel])
    assert chi2_pvalue(np.bincount(second, minlength=V), p[1]) > 1e-4
    rate = np.minimum(p[0], q[0]).sum()
    assert abs(sel.mean() - rate) < 5 * math.sqrt(rate * (1 - rate) / B)


def test_speculative_full_chain_v7b(dev):
    """Vicuna-7B shapes: drafts sampled on the GPU, a chain tree through the
    tree builder (s = 1 per level), verification rows with the drafts made
    likely, then the exact posterior; each stage against the oracle fed the
    GPU's previous stage."""
    cfg = synth.v7b()
    hi = synth.heads_inputs(cfg)
    temp, seed, step = 0.9, 2024, 3
    drafts, dl = m.heads_sample(T(hi.h, dev), T(hi.W1, dev), T(hi.b1, dev), T(hi.W2, dev), temp,
                                seed, step)
    torch.cuda.synchronize()
    g_dr, g_dl = N(drafts), N(dl)
    # the oracle on two heads (each head is independent)
    for k in (0, cfg.K - 1):
        o_dr, o_lg, o_keys = oracle.draft_sample(hi.h, hi.W1[k:k + 1], hi.b1[k:k + 1],
                                                 hi.W2[k:k + 1], temp, seed, step, want_keys=True)
        assert np.abs(g_dl[:, k] - o_lg[:, 0]).max() <= 1e-2
        # the oracle's stream row is the head index: compare on head 0 only
        if k == 0 and int(g_dr[0, 0]) != int(o_dr[0, 0]):
            assert o_keys[0, 0, o_dr[0, 0]] - o_keys[0, 0, g_dr[0, 0]] < GAP
    root = synth.root_tokens(cfg)
    ids = g_dr.reshape(1, cfg.K, 1).astype(np.int32)
    tree = m.build_tree(T(root, dev), T(ids, dev), T(np.zeros((1, cfg.K, 1), np.float32), dev),
                        (1,) * cfg.K, cfg.K, prefix_len=T(np.array([1024], np.int32), dev))
    torch.cuda.synchronize()
    tokens = N(tree.tokens)
    assert list(tokens[0]) == [int(root[0])] + [int(x) for x in g_dr[0]]
    assert list(N(tree.parent)[0]) == list(range(-1, cfg.K))
    rng = np.random.default_rng(7)
    lg = rng.normal(0, 3.0, size=(1, cfg.K + 1, cfg.V)).astype(np.float32)
    for k in range(cfg.K):  # verification rows that like the drafts
        lg[0, k, tokens[0, k + 1]] += 9.0
    l16 = synth.cast(lg, "bf16")
    g = run_spec(dev, l16, tokens, g_dl, temp, seed, step)
    check_spec(g, l16, tokens, g_dl, temp, seed, step)


def test_speculative_bad_draft_token_status(dev):
    B, K, V = 2, 3, 1000
    rng = np.random.default_rng(2)
    logits = rng.normal(size=(B, K + 1, V)).astype(np.float32)
    dl = rng.normal(size=(B, K, V)).astype(np.float32)
    tokens = rng.integers(0, V, size=(B, K + 1)).astype(np.int32)
    tokens[1, 2] = V + 3
    ws = m.new_workspace(m.speculative_workspace_size(B, K), dev)
    out = m.speculative_posterior(T(logits, dev), T(tokens, dev), T(dl, dev), 1.0, 1, 1, ws=ws)
    torch.cuda.synchronize()
    assert m.read_device_status(ws) == 1
    assert int(N(out.accept_len)[1]) <= 1
