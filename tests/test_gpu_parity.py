"""GPU-vs-oracle parity for every stage of the Medusa step, through the C ABI.

Tolerances (fixed by the acceptance bar for this path):
  * ids, tree arrays, accepted length, path and next token: bit-exact, except
    a top-s / argmax decision whose oracle logit gap is < 1e-3, or a typical
    decision whose oracle margin |log p - log threshold| is < 1e-3; after such
    an exemption the later stage is compared with the oracle re-run on the
    GPU's choice.
  * floats (attention output, log-probs): max-abs <= 1e-2 and relative L2
    error <= 2e-2.
"""
import contextlib
import math

import numpy as np
import pytest
import torch

import oracle
import synth
import medusa_speculative_decoding_02_gb300 as m
from medusa_speculative_decoding_02_gb300 import build as mbuild

pytestmark = pytest.mark.gpu

GAP = 1e-3
ATOL, RTOL = 1e-2, 2e-2


# ---------------------------------------------------------------- helpers ---

@pytest.fixture(scope="session")
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


_cache = {}


def cached(key, fn):
    if key not in _cache:
        _cache[key] = fn()
    return _cache[key]


def check_topk(g_ids, g_logp, o_ids, o_logits, o_logz):
    """Bit-exact ids except near-ties (oracle gap < 1e-3); log-probs within
    tolerance.  Returns the number of exempted positions."""
    B, K, S = g_ids.shape
    exempt = 0
    for b in range(B):
        for k in range(K):
            assert len(set(g_ids[b, k].tolist())) == S, (b, k)
            for j in range(S):
                a, o = int(g_ids[b, k, j]), int(o_ids[b, k, j])
                if a != o:
                    gap = abs(o_logits[b, k, a] - o_logits[b, k, o])
                    assert gap < GAP, (b, k, j, a, o, gap)
                    exempt += 1
                ref = o_logits[b, k, a] - o_logz[b, k]
                assert abs(g_logp[b, k, j] - ref) <= ATOL + RTOL * abs(ref), (b, k, j)
    return exempt


def check_close(g, o, what="", bf16_out=True):
    """Max-abs <= 1e-2 and relative L2 <= 2e-2.  A bf16 result also carries
    its own rounding: the nearest bf16 to an exact value o can be up to half
    a unit in the last place, 2^-9 |o|, away (0.0156 for |o| in [4, 8)), so
    that allowance is added element by element for bf16 outputs."""
    g = np.asarray(g, np.float64)
    o = np.asarray(o, np.float64)
    err = np.abs(g - o)
    bound = ATOL + (np.abs(o) * 2.0 ** -9 if bf16_out else 0.0)
    assert (err <= bound).all(), f"{what} max-abs {err.max()} (worst excess {(err - bound).max()})"
    rel = np.linalg.norm(g - o) / max(np.linalg.norm(o), 1e-30)
    assert rel <= RTOL, f"{what} relative {rel}"
    return float(err.max()), float(rel)


def tree_np(t: m.Tree):
    return dict(tokens=N(t.tokens), parent=N(t.parent), depth=N(t.depth), pos_id=N(t.pos_id),
                anc_mask=N(t.anc_mask).view(np.uint64), paths=N(t.paths), n_leaf=N(t.n_leaf))


def check_tree(gt: dict, ot: dict):
    for key in ("tokens", "parent", "depth", "pos_id", "anc_mask", "paths", "n_leaf"):
        assert np.array_equal(gt[key], ot[key]), key


def check_posterior(gp: m.Posterior, logits_np, ot, K, mode, eps, delta, temp):
    op = oracle.posterior(logits_np, ot["tokens"], ot["parent"], ot["depth"], K, mode, eps, delta,
                          temp)
    g_acc = N(gp.accept)
    mism = g_acc != op["accept"]
    near = np.abs(op["margin"]) < GAP
    assert not (mism & ~near).any(), np.argwhere(mism & ~near)
    if mism.any():
        op = oracle.posterior(logits_np, ot["tokens"], ot["parent"], ot["depth"], K, mode, eps,
                              delta, temp, forced_accept=g_acc)
    for key in ("accept_len", "path", "path_tokens", "next_token"):
        assert np.array_equal(N(getattr(gp, key)), op[key]), key
    return op


def random_topk(rng, B, K, S, V=32000):
    """Top-s tables shaped like the heads' output: distinct ids, log-probs
    sorted descending."""
    ids = np.stack([np.stack([rng.choice(V, size=S, replace=False) for _ in range(K)])
                    for _ in range(B)]).astype(np.int32)
    p = rng.dirichlet(np.ones(S + 1), size=(B, K))[..., :S]
    logp = np.log(-np.sort(-p, axis=-1)).astype(np.float32)
    return ids, logp


def oracle_tree_for(rng, s, n, B, prefix, V=32000):
    ids, logp = random_topk(rng, B, len(s), max(s), V)
    return oracle.build_tree(np.arange(B, dtype=np.int32) + 7, ids, logp.astype(np.float64), s, n,
                             prefix_len=np.asarray(prefix, np.int32))


# ------------------------------------------------------------------ heads ---

def run_heads(cfg, dev, hi=None):
    hi = hi or cached(("heads", cfg.name), lambda: synth.heads_inputs(cfg))
    ids, logp = m.heads(T(hi.h, dev), T(hi.W1, dev), T(hi.b1, dev), T(hi.W2, dev), cfg.top_s)
    torch.cuda.synchronize()
    return hi, N(ids), N(logp)


def oracle_heads_for(cfg, hi):
    return cached(("oheads", cfg.name), lambda: oracle.heads(hi.h, hi.W1, hi.b1, hi.W2, cfg.top_s,
                                                             want_logits=True))


def test_heads_tiny_f32(dev):
    cfg = synth.tiny()
    hi, ids, logp = run_heads(cfg, dev)
    o_ids, _, o_logits, o_logz = oracle.heads(hi.h, hi.W1, hi.b1, hi.W2, cfg.top_s, want_logits=True)
    check_topk(ids, logp, o_ids, o_logits, o_logz)


@pytest.mark.parametrize("dtype,B,d,V,K,S", [
    ("bf16", 1, 64, 1000, 3, 2), ("bf16", 3, 72, 1031, 2, 16), ("f32", 2, 128, 1031, 4, 5),
    ("bf16", 8, 136, 999, 5, 8), ("bf16", 5, 256, 4000, 8, 16), ("f32", 1, 8, 17, 1, 16),
    ("bf16", 2, 520, 20011, 3, 4)])
def test_heads_ragged_shapes(dev, dtype, B, d, V, K, S):
    """Ragged d (partial vector loops), prime V (uneven CTA slices), B inside a
    larger batch bucket, non-zero bias."""
    cfg = synth.tiny().replace(name=f"r{dtype}{B}{d}{V}{K}{S}", dtype=dtype, B=B, d=d, V=V, K=K,
                               s=(S,) * K, w1_std=0.05, w2_std=0.05)
    hi = synth.heads_inputs(cfg)
    rng = np.random.default_rng(d + V)
    b1 = rng.standard_normal((K, d)).astype(np.float32) * 0.5
    hi.b1 = synth.cast(b1, dtype)
    _, ids, logp = run_heads(cfg, dev, hi)
    o_ids, _, o_logits, o_logz = oracle.heads(hi.h, hi.W1, hi.b1, hi.W2, S, want_logits=True)
    check_topk(ids, logp, o_ids, o_logits, o_logz)


@pytest.mark.parametrize("dtype,B", [("bf16", 1), ("bf16", 2), ("f32", 1)])
def test_heads_bias_many_rows_per_warp(dev, dtype, B):
    """Full-width W1 (K = 5, d = 4096: about four rows per phase-1 warp) with a
    non-zero bias, so the per-warp bias fetch is used at every row position;
    a small vocabulary keeps the oracle quick."""
    cfg = synth.v7b().replace(name=f"bias{dtype}{B}", dtype=dtype, B=B, V=1000, w1_std=0.02,
                              w2_std=0.05)
    hi = synth.heads_inputs(cfg)
    rng = np.random.default_rng(41 + B)
    hi.b1 = synth.cast(rng.standard_normal((cfg.K, cfg.d)).astype(np.float32) * 0.5, dtype)
    _, ids, logp = run_heads(cfg, dev, hi)
    o_ids, _, o_logits, o_logz = oracle.heads(hi.h, hi.W1, hi.b1, hi.W2, cfg.top_s,
                                              want_logits=True)
    check_topk(ids, logp, o_ids, o_logits, o_logz)


@pytest.mark.parametrize("cfg_fn", [synth.v7b, synth.v13b, synth.batch8],
                         ids=["v7b", "v13b", "batch8"])
def test_heads_full_size(dev, cfg_fn):
    cfg = cfg_fn()
    hi, ids, logp = run_heads(cfg, dev)
    o_ids, _, o_logits, o_logz = oracle_heads_for(cfg, hi)
    check_topk(ids, logp, o_ids, o_logits, o_logz)


def test_heads_identity_init_variant(dev):
    """W1 = 0, b1 = 0, every W2 = the LM head: every head returns the same
    top-s, equal to the LM head's (oracle) top-s."""
    cfg = synth.v7b(lm_head_variant=True)
    hi, ids, logp = run_heads(cfg, dev)
    for k in range(1, cfg.K):
        assert np.array_equal(ids[0, k], ids[0, 0])
        assert np.array_equal(logp[0, k], logp[0, 0])
    sub = synth.HeadsInputs(h=hi.h, W1=hi.W1[:1], b1=hi.b1[:1], W2=hi.W2[:1])
    o_ids, _, o_logits, o_logz = oracle.heads(sub.h, sub.W1, sub.b1, sub.W2, cfg.top_s,
                                              want_logits=True)
    check_topk(ids[:, :1], logp[:, :1], o_ids, o_logits, o_logz)


# ------------------------------------------------------------------- tree ---

def run_tree(dev, root, ids, logp, s, n, prefix):
    t = m.build_tree(T(root, dev), T(ids, dev), T(logp, dev), s, n,
                     prefix_len=T(np.asarray(prefix, np.int32), dev))
    torch.cuda.synchronize()
    return tree_np(t)


@pytest.mark.parametrize("s,n,B", [
    ((2, 2, 2), 14, 1), ((4, 3, 2, 2, 1), 64, 2), ((8, 4, 4, 2, 2), 16, 1),
    ((8, 4, 4, 2, 2), 32, 1), ((8, 4, 4, 2, 2), 64, 3), ((8, 4, 4, 2, 2), 128, 1),
    ((16, 16), 255, 3), ((1, 1, 1, 1, 1), 5, 1), ((3,) * 8, 200, 2), ((4, 3, 2, 2, 1), 136, 1),
    ((16,), 16, 1), ((2, 3), 8, 8)])
def test_tree_parity(dev, s, n, B):
    rng = np.random.default_rng(n * 31 + B)
    ids, logp = random_topk(rng, B, len(s), max(s))
    root = rng.integers(0, 32000, size=B).astype(np.int32)
    prefix = rng.integers(0, 5000, size=B).astype(np.int32)
    gt = run_tree(dev, root, ids, logp, s, n, prefix)
    ot = oracle.build_tree(root, ids, logp.astype(np.float64), s, n, prefix_len=prefix)
    check_tree(gt, ot)


def test_tree_ties(dev):
    """Equal scores: smaller depth first, then the smaller rank path; also
    log-probability exactly 0 (a child ties its parent)."""
    s, n = (3, 3, 3), 20
    ids = np.arange(27, dtype=np.int32).reshape(1, 3, 9)[:, :, :3].copy()
    for logp_val in (np.log(0.25), 0.0):
        logp = np.full((1, 3, 3), logp_val, np.float32)
        gt = run_tree(dev, np.array([5], np.int32), ids, logp, s, n, [0])
        ot = oracle.build_tree([5], ids, logp.astype(np.float64), s, n, prefix_len=[0])
        check_tree(gt, ot)


def test_tree_worked_example_on_gpu(dev):
    """The sparse-tree worked example (three heads, two ranks each, budget 6)
    through the GPU builder: the same six nodes, E[L_cover] = 1.9325."""
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                    "sparse_tree_worked_example.json")))
    a = g["a"]
    ids = np.array([[[100 * (k + 1) + r for r in range(2)] for k in range(3)]], np.int32)
    logp = np.log(np.array([a], np.float64)).astype(np.float32)
    gt = run_tree(dev, np.array([1], np.int32), ids, logp, (2, 2, 2), g["budget"], [0])
    paths = set()
    for i in range(1, g["budget"] + 1):
        p, x = [], i
        while x > 0:
            p.append(int(gt["tokens"][0, x]) % 100)
            x = int(gt["parent"][0, x])
        paths.add(tuple(reversed(p)))
    assert paths == {tuple(r - 1 for r in p) for p in g["picks_in_order"]}
    cover = sum(math.prod(a[k][r] for k, r in enumerate(p)) for p in paths)
    assert cover == pytest.approx(g["expected_cover_depth"], abs=1e-6)


def run_tree_static(dev, root, ids, log_a, s, n, prefix):
    t = m.build_tree_static(T(root, dev), T(ids, dev), T(log_a.astype(np.float32), dev), s, n,
                            prefix_len=T(np.asarray(prefix, np.int32), dev))
    torch.cuda.synchronize()
    return tree_np(t)


def test_tree_static_worked_example(dev):
    """The calibrated table of the sparse-tree worked example drives the
    shape for three sequences with different top-s tokens: every sequence
    gets the six worked-example nodes, its own tokens, and the arrays equal
    the oracle's tree built from the same table."""
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                    "sparse_tree_worked_example.json")))
    a = np.array(g["a"], np.float64)
    B = 3
    ids = np.array([[[1000 * b + 100 * (k + 1) + r for r in range(2)] for k in range(3)]
                    for b in range(B)], np.int32)
    log_a = np.log(a).astype(np.float32)
    root = np.array([5, 6, 7], np.int32)
    gt = run_tree_static(dev, root, ids, log_a, (2, 2, 2), g["budget"], [0, 3, 9])
    ot = oracle.build_tree(root, ids, np.broadcast_to(log_a.astype(np.float64), (B, 3, 2)),
                           (2, 2, 2), g["budget"], prefix_len=np.array([0, 3, 9], np.int32))
    check_tree(gt, ot)
    for b in range(B):
        paths = set()
        for i in range(1, g["budget"] + 1):
            p, x = [], i
            while x > 0:
                assert int(gt["tokens"][b, x]) // 1000 == b
                p.append(int(gt["tokens"][b, x]) % 100)
                x = int(gt["parent"][b, x])
            paths.add(tuple(reversed(p)))
        assert paths == {tuple(r - 1 for r in p) for p in g["picks_in_order"]}


@pytest.mark.parametrize("s,n,B", [((4, 3, 2, 2, 1), 64, 8), ((8, 4, 4, 2, 2), 128, 2),
                                   ((16, 16), 255, 1), ((3, 3, 3), 10, 4)])
def test_tree_static_random_tables(dev, s, n, B):
    """Random calibrated tables (accuracies decreasing with rank): the shape is
    the same for every sequence and the arrays equal both the oracle's and
    the dynamic builder's on the table broadcast to every sequence."""
    rng = np.random.default_rng(n + B)
    K, S = len(s), max(s)
    acc = np.sort(rng.uniform(0.05, 0.9, size=(K, S)), axis=1)[:, ::-1]
    log_a = np.log(acc).astype(np.float32)
    ids = np.stack([np.stack([rng.choice(32000, size=S, replace=False) for _ in range(K)])
                    for _ in range(B)]).astype(np.int32)
    root = rng.integers(0, 32000, size=B).astype(np.int32)
    prefix = rng.integers(0, 2000, size=B).astype(np.int32)
    gt = run_tree_static(dev, root, ids, log_a, s, n, prefix)
    full = np.ascontiguousarray(np.broadcast_to(log_a, (B, K, S)))
    ot = oracle.build_tree(root, ids, full.astype(np.float64), s, n, prefix_len=prefix)
    check_tree(gt, ot)
    gd = run_tree(dev, root, ids, full, s, n, prefix)
    check_tree(gt, gd)
    for b in range(1, B):
        assert np.array_equal(gt["parent"][b], gt["parent"][0])
        assert np.array_equal(gt["depth"][b], gt["depth"][0])


def test_tree_from_heads_v7b(dev):
    cfg = synth.v7b()
    _, ids, logp = run_heads(cfg, dev)
    root = synth.root_tokens(cfg)
    gt = run_tree(dev, root, ids, logp, cfg.s, cfg.n, cfg.prefix)
    ot = oracle.build_tree(root, ids, logp.astype(np.float64), cfg.s, cfg.n,
                           prefix_len=np.asarray(cfg.prefix))
    check_tree(gt, ot)


# -------------------------------------------------------------- attention ---

def run_attention(dev, ai, anc_mask, P_max, dh):
    kc = [T(x, dev) for x in ai.k_cache]
    vc = [T(x, dev) for x in ai.v_cache]
    out = m.tree_attention(T(ai.q, dev), m.cache_pointers(kc, dev), m.cache_pointers(vc, dev),
                           T(ai.prefix_len, dev), P_max, T(anc_mask.view(np.int64), dev),
                           1.0 / math.sqrt(dh))
    torch.cuda.synchronize()
    o = out.float() if out.dtype == torch.bfloat16 else out
    return N(o)


@contextlib.contextmanager
def all_cores():
    """Full-size attention checks run the oracle's OpenMP build (the same
    source and the same bits as the serial build, tests/test_oracle_parallel.py)
    when it exists, so that checking every head stays within seconds."""
    on = oracle.parallel_available()
    if on:
        oracle.set_parallel(True)
    try:
        yield
    finally:
        oracle.set_parallel(False)


def oracle_attention_heads(ai, anc_mask, dh, heads, seqs=None):
    """Oracle on a subset of attention heads (the others are independent),
    optionally on a subset of the sequences."""
    sl = lambda x: np.ascontiguousarray(x[..., heads, :])
    bs = list(range(len(ai.k_cache))) if seqs is None else list(seqs)
    with all_cores():
        return oracle.tree_attention(sl(ai.q[bs]), [sl(ai.k_cache[b]) for b in bs],
                                     [sl(ai.v_cache[b]) for b in bs], ai.prefix_len[bs],
                                     anc_mask[bs], 1.0 / math.sqrt(dh))


def test_attention_tiny_f32(dev):
    cfg = synth.tiny()
    ot = oracle_tree_for(np.random.default_rng(0), cfg.s, cfg.n, 1, cfg.prefix)
    ai = synth.attention_inputs(cfg)
    g = run_attention(dev, ai, ot["anc_mask"], cfg.P_max, cfg.dh)
    o = oracle.tree_attention(ai.q, ai.k_cache, ai.v_cache, ai.prefix_len, ot["anc_mask"],
                              1.0 / math.sqrt(cfg.dh))
    check_close(g, o, "tiny", bf16_out=False)


@pytest.mark.parametrize("B,s,n,H,dh,prefix", [
    (1, (2, 2, 2), 14, 2, 64, (0,)), (2, (4, 4), 16, 3, 128, (1, 70)),
    (1, (4, 3, 2, 2, 1), 64, 4, 128, (1023,)), (3, (8, 4, 4), 128, 2, 128, (5, 300, 64)),
    (1, (16, 16), 255, 1, 128, (100,)), (2, (4, 4, 2), 32, 2, 64, (128, 0)),
    (1, (1,), 1, 2, 128, (10,)), (2, (8, 4, 4, 2, 2), 200, 1, 64, (65, 1)),
    (1, (4, 3, 2, 2, 1), 64, 2, 64, (3000,)), (3, (4, 4, 2), 32, 3, 128, (2500, 40, 1700)),
    (2, (8, 4, 4, 2, 2), 129, 3, 128, (77, 1)), (1, (8, 4, 4, 2, 2), 130, 2, 128, (200,)),
    (2, (8, 4, 4), 128, 2, 64, (90, 3))])
def test_attention_shapes(dev, B, s, n, H, dh, prefix):
    """Ragged prefixes (0, 1, non-multiples of the 64-key tile), tree sizes
    from 2 to 256 rows (both warp-count instantiations), dh 64 and 128;
    129, 130 and 131 rows here take two 128-row tiles (short key ranges)."""
    cfg = synth.v7b().replace(name=f"att{B}{n}{H}{dh}{prefix}", B=B, s=s, n=n, H=H, dh=dh,
                              prefix=prefix)
    ot = oracle_tree_for(np.random.default_rng(n + dh), s, n, B, prefix)
    ai = synth.attention_inputs(cfg)
    g = run_attention(dev, ai, ot["anc_mask"], cfg.P_max, dh)
    o = oracle.tree_attention(ai.q, ai.k_cache, ai.v_cache, ai.prefix_len, ot["anc_mask"],
                              1.0 / math.sqrt(dh))
    check_close(g, o, cfg.name)


@pytest.mark.parametrize("cfg_fn", [synth.v7b, synth.v13b, synth.batch8],
                         ids=["v7b", "v13b", "batch8"])
def test_attention_full_size(dev, cfg_fn):
    """Every attention head of every sequence against the oracle, so that a
    slip in the (sequence, head) decode of the grid cannot hide."""
    cfg = cfg_fn()
    ot = oracle_tree_for(np.random.default_rng(cfg.seed), cfg.s, cfg.n, cfg.B, cfg.prefix)
    ai = synth.attention_inputs(cfg)
    g = run_attention(dev, ai, ot["anc_mask"], cfg.P_max, cfg.dh)
    heads = list(range(cfg.H))
    o = oracle_attention_heads(ai, ot["anc_mask"], cfg.dh, heads)
    check_close(g, o, cfg.name)


@pytest.mark.parametrize("n", synth.SWEEP_N)
@pytest.mark.parametrize("P", synth.SWEEP_P)
def test_attention_sweep(dev, n, P):
    """Every head at every point of the tree-size x context sweep."""
    cfg = synth.sweep(n, P)
    ot = oracle_tree_for(np.random.default_rng(n + P), cfg.s, cfg.n, 1, cfg.prefix)
    ai = synth.attention_inputs(cfg)
    g = run_attention(dev, ai, ot["anc_mask"], cfg.P_max, cfg.dh)
    o = oracle_attention_heads(ai, ot["anc_mask"], cfg.dh, list(range(cfg.H)))
    check_close(g, o, cfg.name)


@pytest.mark.parametrize("P,growth,n,H", [(1024, 0.02, 64, 4), (8192, 0.004, 64, 4),
                                           (700, -0.03, 64, 4), (8192, 0.004, 128, 32),
                                           (900, -0.03, 128, 4)])
def test_attention_growing_scores(dev, P, growth, n, H):
    """Key rows scaled by exp(growth * slot): the scores' row maxima grow (or
    shrink) steadily along the prefix, so later 64-key sub-chunks raise the
    softmax reference by more than 2^8 many times and the O accumulator is
    rescaled in tensor memory (growth > 0), or the first sub-chunk dominates
    (growth < 0).  With n = 128 (129 rows) at prefix 8192 and 32 heads the
    row past the tensor-core tile is computed on the CUDA cores and moves its
    own reference by the same rule; at prefix 900 the tree takes two tiles."""
    s = (4, 3, 2, 2, 1) if n == 64 else (8, 4, 4, 2, 2)
    cfg = synth.v7b().replace(name=f"grow{P}{growth}{n}", H=H, prefix=(P,), s=s, n=n)
    ot = oracle_tree_for(np.random.default_rng(P), cfg.s, cfg.n, 1, cfg.prefix)
    ai = synth.attention_inputs(cfg)
    k = synth.bf16_bits_to_f32(ai.k_cache[0])
    slot = np.arange(k.shape[0], dtype=np.float64)
    f = np.exp(np.clip(growth * slot, -4.0, 4.0)).astype(np.float32)
    ai.k_cache[0] = synth.cast(k * f[:, None, None], "bf16")
    g = run_attention(dev, ai, ot["anc_mask"], cfg.P_max, cfg.dh)
    o = oracle_attention_heads(ai, ot["anc_mask"], cfg.dh, list(range(cfg.H)))
    check_close(g, o, cfg.name)


@pytest.mark.parametrize("prefix", [(8192,), (4100, 8192), (8192, 5, 6000), (0, 8192)],
                         ids=["one", "two", "three", "empty_prefix"])
def test_attention_tail_row(dev, prefix):
    """Trees of 129 rows over long prefixes (32 heads of 128): one 128-row
    tensor-core tile per key range, the last row on the CUDA cores of the
    same CTAs.  Every head of every sequence against the oracle; ragged
    prefixes, a 5-slot prefix whose later key ranges are empty, and an empty
    prefix (the tree's own slots are the only keys)."""
    cfg = synth.v7b().replace(name=f"tail{len(prefix)}", B=len(prefix), s=(8, 4, 4, 2, 2), n=128,
                              prefix=prefix)
    ot = oracle_tree_for(np.random.default_rng(len(prefix)), cfg.s, cfg.n, cfg.B, cfg.prefix)
    ai = synth.attention_inputs(cfg)
    g = run_attention(dev, ai, ot["anc_mask"], cfg.P_max, cfg.dh)
    o = oracle_attention_heads(ai, ot["anc_mask"], cfg.dh, list(range(cfg.H)))
    check_close(g, o, cfg.name)


# -------------------------------------------------------------- posterior ---

def run_posterior(dev, logits_np, ot, K, mode, eps=0.09, delta=0.3, temp=1.0):
    gp = m.evaluate_posterior(T(logits_np, dev), T(ot["tokens"], dev), T(ot["parent"], dev),
                              T(ot["depth"], dev), K, mode, eps, delta, temp)
    torch.cuda.synchronize()
    return gp


@pytest.mark.parametrize("mode", [m.GREEDY, m.TYPICAL])
def test_posterior_tiny(dev, mode):
    cfg = synth.tiny()
    ot = oracle_tree_for(np.random.default_rng(1), cfg.s, cfg.n, 1, cfg.prefix, cfg.V)
    logits = synth.base_logits(cfg)
    synth.plant_bernoulli(logits, ot["tokens"], ot["parent"], synth.rng_for(cfg, "plant"))
    gp = run_posterior(dev, logits, ot, cfg.K, mode, cfg.eps, cfg.delta)
    check_posterior(gp, logits, ot, cfg.K, mode, cfg.eps, cfg.delta, 1.0)


@pytest.mark.parametrize("L_star", range(6))
@pytest.mark.parametrize("mode", [m.GREEDY, m.TYPICAL])
def test_posterior_v7b_planted_chain(dev, L_star, mode):
    cfg = synth.v7b()
    ot = oracle_tree_for(np.random.default_rng(L_star), cfg.s, cfg.n, 1, cfg.prefix)
    logits = synth.base_logits(cfg, rep=L_star)
    synth.plant_chain(logits, ot["tokens"], ot["parent"], ot["depth"], L_star,
                      synth.rng_for(cfg, "plant", L_star))
    l16 = synth.cast(logits, "bf16")
    gp = run_posterior(dev, l16, ot, cfg.K, mode)
    op = check_posterior(gp, l16, ot, cfg.K, mode, 0.09, 0.3, 1.0)
    assert int(op["accept_len"][0]) >= min(L_star, int(ot["depth"].max()))


@pytest.mark.parametrize("target", [1.0, 3.0, 6.0])
def test_posterior_v13b_entropy(dev, target):
    cfg = synth.v13b()
    ot = oracle_tree_for(np.random.default_rng(13), cfg.s, cfg.n, 1, cfg.prefix)
    logits = synth.base_logits(cfg, rep=int(target))
    synth.plant_chain(logits, ot["tokens"], ot["parent"], ot["depth"], 3,
                      synth.rng_for(cfg, "plant", int(target)))
    scaled = synth.scale_rows_to_entropy(logits, target, oracle.softmax_entropy)
    l16 = synth.cast(scaled, "bf16")
    gp = run_posterior(dev, l16, ot, cfg.K, m.TYPICAL, cfg.eps, cfg.delta)
    check_posterior(gp, l16, ot, cfg.K, m.TYPICAL, cfg.eps, cfg.delta, 1.0)


def test_posterior_batch8(dev):
    cfg = synth.batch8()
    ot = oracle_tree_for(np.random.default_rng(8), cfg.s, cfg.n, cfg.B, cfg.prefix)
    logits = synth.base_logits(cfg)
    for b in range(cfg.B):
        sl = slice(b, b + 1)
        synth.plant_chain(logits[sl], ot["tokens"][sl], ot["parent"][sl], ot["depth"][sl], b % 6,
                          synth.rng_for(cfg, "plant", b))
    l16 = synth.cast(logits, "bf16")
    for mode in (m.GREEDY, m.TYPICAL):
        gp = run_posterior(dev, l16, ot, cfg.K, mode, cfg.eps, cfg.delta)
        check_posterior(gp, l16, ot, cfg.K, mode, cfg.eps, cfg.delta, 1.0)


def test_posterior_many_sequences_one_workspace(dev):
    """Batches past the heads' limit of 8 (the posterior takes any B): 53,
    3, 49 and 53 sequences through one workspace, each checked against the
    oracle; the status word stays 0."""
    cfg = synth.tiny()
    ws = m.new_workspace(m.posterior_workspace_size(53, cfg.R), dev)
    for B in (53, 3, 49, 53):
        c = cfg.replace(name=f"many{B}", B=B, prefix=(0,) * B)
        rng = np.random.default_rng(B)
        ot = oracle_tree_for(rng, c.s, c.n, B, c.prefix, c.V)
        logits = synth.plant_bernoulli(synth.base_logits(c), ot["tokens"], ot["parent"], rng,
                                       prob=0.8, amount=9.0)
        for mode in (m.GREEDY, m.TYPICAL):
            gp = m.evaluate_posterior(T(logits, dev), T(ot["tokens"], dev), T(ot["parent"], dev),
                                      T(ot["depth"], dev), c.K, mode, c.eps, c.delta, 1.0, ws=ws)
            torch.cuda.synchronize()
            check_posterior(gp, logits, ot, c.K, mode, c.eps, c.delta, 1.0)
            assert m.read_device_status(ws) == 0
    assert (N(gp.accept_len) > 0).any()


@pytest.mark.parametrize("dtype,V,s,n,temp", [
    ("f32", 1000, (2, 2, 2), 14, 0.7), ("bf16", 1008, (4, 3), 15, 1.0),
    ("bf16", 32000, (16, 16), 255, 0.7), ("bf16", 8, (2,), 1, 2.0), ("f32", 4, (4, 4), 20, 1.0),
    ("bf16", 1000, (2,) * 8, 255, 1.0), ("f32", 64, (3,) * 8, 100, 0.5)])
def test_posterior_shapes(dev, dtype, V, s, n, temp):
    """Small and odd vocabularies, 2..256 rows, temperature != 1, and the
    deepest trees (8 heads: paths of 9 nodes)."""
    cfg = synth.tiny().replace(name=f"post{dtype}{V}{n}", dtype=dtype, V=V, s=s, n=n, K=len(s))
    ot = oracle_tree_for(np.random.default_rng(V + n), s, n, 1, (0,))
    ot["tokens"][:, 1:] %= V
    logits = synth.base_logits(cfg)
    synth.plant_bernoulli(logits, ot["tokens"], ot["parent"], synth.rng_for(cfg, "plant"))
    lg = synth.cast(logits, dtype)
    for mode in (m.GREEDY, m.TYPICAL):
        gp = run_posterior(dev, lg, ot, len(s), mode, 0.09, 0.3, temp)
        check_posterior(gp, lg, ot, len(s), mode, 0.09, 0.3, temp)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_posterior_masked_vocabulary(dev, dtype):
    """-inf logits (a masked vocabulary: every fifth token, a whole block, and
    some of the tree's own tokens) add nothing to the softmax sums and are
    never accepted; the entropy and decisions match the oracle."""
    cfg = synth.v7b().replace(name=f"mask{dtype}", dtype=dtype, V=4000)
    ot = oracle_tree_for(np.random.default_rng(5), cfg.s, cfg.n, 1, cfg.prefix, cfg.V)
    logits = synth.base_logits(cfg)
    synth.plant_bernoulli(logits, ot["tokens"], ot["parent"], synth.rng_for(cfg, "plant"))
    logits[..., 3::5] = -np.inf
    logits[..., 1200:1900] = -np.inf
    for i in range(1, cfg.R, 9):
        logits[0, ot["parent"][0, i], ot["tokens"][0, i]] = -np.inf
    lg = synth.cast(logits, dtype)
    for mode in (m.GREEDY, m.TYPICAL):
        gp = run_posterior(dev, lg, ot, cfg.K, mode)
        check_posterior(gp, lg, ot, cfg.K, mode, 0.09, 0.3, 1.0)


@pytest.mark.parametrize("ties", [
    [31999, 7, 12345],       # maxima far apart (different threads and slices)
    [13, 10, 2058, 4106],    # two in one 16-byte group, more in later groups
    [5001, 5000],            # adjacent ids in one group
    [16007, 16000, 8]])      # both ends of a group, and an early id
def test_posterior_argmax_ties_and_all_rejected(dev, ties):
    """bf16 rows with repeated maxima (argmax -> smallest id) and every
    candidate rejected (L = 0, path = [root], next = argmax of row 0)."""
    cfg = synth.v7b()
    ot = oracle_tree_for(np.random.default_rng(99), cfg.s, cfg.n, 1, cfg.prefix)
    logits = synth.base_logits(cfg)
    for r in range(cfg.R):
        top = logits[0, r].max() + 1.0
        logits[0, r, ties] = top
    for i in range(1, cfg.R):
        logits[0, ot["parent"][0, i], ot["tokens"][0, i]] = -30.0
    l16 = synth.cast(logits, "bf16")
    for mode in (m.GREEDY, m.TYPICAL):
        gp = run_posterior(dev, l16, ot, cfg.K, mode)
        op = check_posterior(gp, l16, ot, cfg.K, mode, 0.09, 0.3, 1.0)
        assert int(op["accept_len"][0]) == 0 and int(N(gp.next_token)[0]) == min(ties)


# ------------------------------------------------------------ whole step ---

def test_full_step_v7b_chain(dev):
    """heads -> tree -> tree attention -> posterior, all on the GPU, each stage
    checked against the oracle fed the GPU's previous-stage output."""
    cfg = synth.v7b()
    hi, ids, logp = run_heads(cfg, dev)
    o_ids, _, o_logits, o_logz = oracle_heads_for(cfg, hi)
    check_topk(ids, logp, o_ids, o_logits, o_logz)
    root = synth.root_tokens(cfg)
    gt = run_tree(dev, root, ids, logp, cfg.s, cfg.n, cfg.prefix)
    ot = oracle.build_tree(root, ids, logp.astype(np.float64), cfg.s, cfg.n,
                           prefix_len=np.asarray(cfg.prefix))
    check_tree(gt, ot)
    ai = synth.attention_inputs(cfg)
    g = run_attention(dev, ai, gt["anc_mask"], cfg.P_max, cfg.dh)
    o = oracle_attention_heads(ai, ot["anc_mask"], cfg.dh, [0, 9, 31])
    check_close(g[..., [0, 9, 31], :], o, "v7b step")
    logits = synth.base_logits(cfg)
    synth.plant_chain(logits, gt["tokens"], gt["parent"], gt["depth"], 4, synth.rng_for(cfg, "plant"))
    l16 = synth.cast(logits, "bf16")
    gp = run_posterior(dev, l16, gt, cfg.K, m.GREEDY)
    op = check_posterior(gp, l16, ot, cfg.K, m.GREEDY, 0.09, 0.3, 1.0)
    assert int(op["accept_len"][0]) >= 4


def test_full_step_batch8_chain(dev):
    """The same chain on 8 independent sequences: ragged prefixes (635 to
    3990 slots, each cache its own allocation), one planted chain per
    sequence, typical acceptance."""
    cfg = synth.batch8()
    hi, ids, logp = run_heads(cfg, dev)
    o_ids, _, o_logits, o_logz = oracle_heads_for(cfg, hi)
    check_topk(ids, logp, o_ids, o_logits, o_logz)
    root = synth.root_tokens(cfg)
    gt = run_tree(dev, root, ids, logp, cfg.s, cfg.n, cfg.prefix)
    ot = oracle.build_tree(root, ids, logp.astype(np.float64), cfg.s, cfg.n,
                           prefix_len=np.asarray(cfg.prefix))
    check_tree(gt, ot)
    ai = synth.attention_inputs(cfg)
    g = run_attention(dev, ai, gt["anc_mask"], cfg.P_max, cfg.dh)
    o = oracle_attention_heads(ai, ot["anc_mask"], cfg.dh, [0, 31])
    check_close(g[..., [0, 31], :], o, "batch8 step")
    logits = synth.base_logits(cfg)
    for b in range(cfg.B):
        sl = slice(b, b + 1)
        synth.plant_chain(logits[sl], gt["tokens"][sl], gt["parent"][sl], gt["depth"][sl], b % 6,
                          synth.rng_for(cfg, "plant", b))
    l16 = synth.cast(logits, "bf16")
    gp = run_posterior(dev, l16, gt, cfg.K, m.TYPICAL, cfg.eps, cfg.delta)
    op = check_posterior(gp, l16, ot, cfg.K, m.TYPICAL, cfg.eps, cfg.delta, 1.0)
    assert (op["accept_len"] >= np.minimum(np.arange(cfg.B) % 6, gt["depth"].max(1))).all()


# ---------------------------------------------------- device-side checks ---

def test_device_status_reports_bad_data(dev):
    """Data only the device can see is reported in the workspace status word
    (first error wins) and cleared on request; nothing faults."""
    cfg = synth.tiny()
    ot = oracle_tree_for(np.random.default_rng(3), cfg.s, cfg.n, 1, cfg.prefix, cfg.V)
    logits = synth.base_logits(cfg)
    ws = m.new_workspace(m.posterior_workspace_size(1, cfg.R), dev)
    bad = ot["tokens"].copy()
    bad[0, 3] = cfg.V + 5
    m.evaluate_posterior(T(logits, dev), T(bad, dev), T(ot["parent"], dev), T(ot["depth"], dev),
                         cfg.K, m.TYPICAL, ws=ws)
    assert m.read_device_status(ws) == 1
    m.clear_device_status(ws)
    assert m.read_device_status(ws) == 0
    # prefix longer than the stated maximum
    ai = synth.attention_inputs(cfg)
    kc = [T(x, dev) for x in ai.k_cache]
    vc = [T(x, dev) for x in ai.v_cache]
    wsa = m.new_workspace(m.tree_attention_workspace_size(m.F32, 1, cfg.R, 1, cfg.dh, 16), dev)
    m.tree_attention(T(ai.q, dev), m.cache_pointers(kc, dev), m.cache_pointers(vc, dev),
                     T(ai.prefix_len, dev), 16, T(ot["anc_mask"].view(np.int64), dev), ws=wsa)
    assert m.read_device_status(wsa) == 3
    # a positive "log-probability" fed to the tree builder
    ids, lp = random_topk(np.random.default_rng(4), 1, 3, 2)
    lp[0, 1, 0] = 0.5
    wst = m.new_workspace(m.build_tree_workspace_size(1, 3, 2, 5), dev)
    m.build_tree(T(np.array([1], np.int32), dev), T(ids, dev), T(lp, dev), (2, 2, 2), 5, ws=wst)
    assert m.read_device_status(wst) == 4


def test_launch_count(dev):
    cfg = synth.tiny()
    hi = synth.heads_inputs(cfg)
    before = m.launch_count()
    m.heads(T(hi.h, dev), T(hi.W1, dev), T(hi.b1, dev), T(hi.W2, dev), cfg.top_s)
    assert m.launch_count() - before == 3
