"""Pins for the float64 oracle: checks against what the pages and mathematics
fix, independent of the oracle's own code (CPU only)."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit, logsumexp

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- tree ----

def _rank_tables(a):
    """Per-level tables where token id encodes (level, rank): 100*(k+1) + r."""
    K = len(a)
    s = max(len(x) for x in a)
    ids = np.full((1, K, s), -1, np.int32)
    logp = np.full((1, K, s), -np.inf)
    for k, row in enumerate(a):
        for r, w in enumerate(row):
            ids[0, k, r] = 100 * (k + 1) + r
            logp[0, k, r] = math.log(w)
    return ids, logp


def _rank_path(t, i):
    """Rank path (0-based) of node i from the token encoding."""
    out = []
    while i > 0:
        out.append(int(t["tokens"][0, i]) % 100)
        i = int(t["parent"][0, i])
    return tuple(reversed(out))


def test_worked_example_sparse_tree():
    """[P2] §6.2 worked example: exact picks in order and E[L_cover] = 1.9325."""
    g = json.load(open(os.path.join(GOLDEN, "sparse_tree_worked_example.json")))
    a = g["a"]
    ids, logp = _rank_tables(a)
    s = [len(x) for x in a]
    picks = [tuple(r - 1 for r in p) for p in g["picks_in_order"]]
    prev = set()
    for n in range(1, g["budget"] + 1):
        t = oracle.build_tree([7], ids, logp, s, n)
        got = {_rank_path(t, i) for i in range(1, n + 1)}
        assert len(got) == n
        added = got - prev
        assert added == {picks[n - 1]}, (n, added)
        prev = got
    weights = [math.prod(a[k][r] for k, r in enumerate(p)) for p in sorted(prev)]
    assert sum(weights) == pytest.approx(g["expected_cover_depth"], abs=1e-12)
    for p, w in zip(picks, g["weights_in_order"]):
        assert math.prod(a[k][r] for k, r in enumerate(p)) == pytest.approx(w, abs=1e-15)


@pytest.mark.parametrize("s,count,seqs", [((2, 3), 8, 6), ((2, 2, 2), 14, 8),
                                          ((4, 3, 2, 2, 1), 136, 48),
                                          ((8, 4, 4, 2, 2), 936, 512)])
def test_full_cartesian_tree_node_count(s, count, seqs):
    """[P2] §6.1: new nodes = sum_k prod_{j<=k} s_j; candidate sequences =
    prod s_k (one leaf per sequence when the whole Cartesian tree is kept)."""
    rng = np.random.default_rng(5)
    a = [sorted(rng.uniform(0.01, 1.0, size=sk), reverse=True) for sk in s]
    ids, logp = _rank_tables(a)
    t = oracle.build_tree([1], ids, logp, list(s), count)
    assert t["tokens"].shape[1] == count + 1
    assert int(t["n_leaf"][0]) == seqs
    per_depth = np.bincount(t["depth"][0], minlength=len(s) + 1)
    assert list(per_depth[1:]) == list(np.cumprod(s))
    with pytest.raises(RuntimeError):
        oracle.build_tree([1], ids, logp, list(s), count + 1)


def _all_nodes(s):
    nodes = []
    for k in range(1, len(s) + 1):
        nodes += list(itertools.product(*[range(x) for x in s[:k]]))
    return nodes


@pytest.mark.parametrize("s,n,seed", [((2, 2), 3, 0), ((2, 2, 2), 5, 1), ((3, 2), 4, 2),
                                      ((2, 3, 2), 6, 3), ((3, 3), 7, 4)])
def test_greedy_tree_maximises_cover(s, n, seed):
    """[P2] §6.2: E[L_cover] = sum of node weights over the tree; the greedy
    tree attains the maximum over every prefix-closed tree of n nodes
    (brute force)."""
    rng = np.random.default_rng(seed)
    a = [sorted(rng.dirichlet(np.ones(x + 1))[:x], reverse=True) for x in s]
    ids, logp = _rank_tables(a)
    t = oracle.build_tree([0], ids, logp, list(s), n)
    w = lambda p: math.prod(a[k][r] for k, r in enumerate(p))
    greedy = sum(w(_rank_path(t, i)) for i in range(1, n + 1))
    best = 0.0
    for sub in itertools.combinations(_all_nodes(s), n):
        ss = set(sub)
        if all(len(p) == 1 or p[:-1] in ss for p in sub):
            best = max(best, sum(w(p) for p in sub))
    assert greedy == pytest.approx(best, abs=1e-12)


def test_tree_structure_invariants():
    """[P2] §6.1: a node sees the root and its own ancestors; nodes of one depth
    share one position index; canonical order puts parents first."""
    cfg = synth.sweep(128, 512)
    rng = np.random.default_rng(11)
    B = 3
    ids = rng.integers(0, 32000, size=(B, cfg.K, cfg.top_s)).astype(np.int32)
    logp = np.log(np.sort(rng.dirichlet(np.ones(cfg.top_s + 1), size=(B, cfg.K))[..., :cfg.top_s], -1)[..., ::-1])
    P = np.array([5, 100, 0], np.int32)
    t = oracle.build_tree([3, 4, 5], ids, logp, cfg.s, cfg.n, prefix_len=P)
    R = cfg.R
    for b in range(B):
        par, de = t["parent"][b], t["depth"][b]
        assert par[0] == -1 and de[0] == 0
        assert t["tokens"][b, 0] == [3, 4, 5][b]
        for i in range(1, R):
            assert 0 <= par[i] < i
            assert de[i] == de[par[i]] + 1
        assert np.all(np.diff(de) >= 0)
        assert np.all(t["pos_id"][b] == P[b] + de)
        for i in range(R):
            anc = set()
            a = i
            while a >= 0:
                anc.add(a)
                a = par[a]
            bits = {j for j in range(R) if (int(t["anc_mask"][b, i, j // 64]) >> (j % 64)) & 1}
            assert bits == anc
        nl = int(t["n_leaf"][b])
        leaves = [i for i in range(R) if i not in set(par[1:].tolist())]
        assert nl == len(leaves)
        for li, leaf in enumerate(leaves):
            row = t["paths"][b, li]
            assert row[de[leaf]] == leaf and row[0] == 0
            assert np.all(row[de[leaf] + 1:] == -1)
        assert np.all(t["paths"][b, nl:] == -1)


# --------------------------------------------------------------- heads ----

def _ref_topk(logits, s):
    order = sorted(range(len(logits)), key=lambda v: (-logits[v], v))
    return order[:s]


def test_heads_identity_init_reproduces_lm_head():
    """[P2] §3.1 initialisation: W1 = 0 (and b1 = 0) makes the residual branch
    the identity; with W2 = the LM head every head reproduces the LM-head
    distribution softmax(W_lm h)."""
    cfg = synth.tiny().replace(lm_head_variant=True)
    hi = synth.heads_inputs(cfg)
    ids, logp, logits, logz = oracle.heads(hi.h, hi.W1, hi.b1, hi.W2, 4, want_logits=True)
    w_lm = hi.W2[0].astype(np.float64)
    ref = w_lm @ hi.h[0].astype(np.float64)
    ref_lp = ref - logsumexp(ref)
    for k in range(cfg.K):
        np.testing.assert_allclose(logits[0, k], ref, rtol=0, atol=1e-12)
        assert list(ids[0, k]) == _ref_topk(ref, 4)
        np.testing.assert_allclose(logp[0, k], ref_lp[ids[0, k]], atol=1e-12)
        assert list(ids[0, k]) == list(ids[0, 0])


def test_heads_residual_silu_and_orientation():
    """[P3] Part 3 residual block z = h + SiLU(W1 h + b1), vocab projection
    W2 z without bias.  W1 = a permutation and W2 = scaled one-hot rows turn
    both products into index gathers, so the expected logits have a closed
    form; transposed operands, a dropped residual, bias or SiLU term all
    change them."""
    rng = np.random.default_rng(3)
    d, V, K, B = 16, 40, 2, 2
    h = rng.standard_normal((B, d)).astype(np.float32)
    perm = np.stack([rng.permutation(d) for _ in range(K)])
    W1 = np.zeros((K, d, d), np.float32)
    for k in range(K):
        W1[k, np.arange(d), perm[k]] = 1.0
    b1 = rng.standard_normal((K, d)).astype(np.float32)
    col = rng.integers(0, d, size=(K, V))
    scale = rng.uniform(0.5, 2.0, size=(K, V)).astype(np.float32)
    W2 = np.zeros((K, V, d), np.float32)
    for k in range(K):
        W2[k, np.arange(V), col[k]] = scale[k]
    ids, logp, logits, logz = oracle.heads(h, W1, b1, W2, 5, want_logits=True)
    for b in range(B):
        for k in range(K):
            u = h[b, perm[k]].astype(np.float64) + b1[k]
            z = h[b].astype(np.float64) + u * expit(u)
            ref = scale[k].astype(np.float64) * z[col[k]]
            np.testing.assert_allclose(logits[b, k], ref, atol=1e-12)
            assert logz[b, k] == pytest.approx(logsumexp(ref), abs=1e-12)
            assert list(ids[b, k]) == _ref_topk(ref, 5)


def test_heads_tie_rule_lowest_id():
    """Equal logits rank the smaller token id first (convention)."""
    d, V = 4, 10
    h = np.ones((1, d), np.float32)
    W1 = np.zeros((1, d, d), np.float32)
    W2 = np.zeros((1, V, d), np.float32)
    W2[0, [7, 2, 5], 0] = 1.0
    ids, _, _, _ = oracle.heads(h, W1, None, W2, 4)
    assert list(ids[0, 0]) == [2, 5, 7, 0]


def test_heads_bf16_widening_exact():
    """bf16 inputs are widened exactly: bf16 data gives the same result as the
    same values passed as float32."""
    cfg = synth.tiny()
    hi = synth.heads_inputs(cfg)
    to16 = synth.f32_to_bf16_bits
    to32 = synth.bf16_bits_to_f32
    a = oracle.heads(to16(hi.h), to16(hi.W1), to16(hi.b1), to16(hi.W2), 3, want_logits=True)
    b = oracle.heads(to32(to16(hi.h)), to32(to16(hi.W1)), to32(to16(hi.b1)), to32(to16(hi.W2)), 3,
                     want_logits=True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[2], b[2])


def test_lm_head_equals_identity_initialised_head():
    """A Medusa head with W1 = 0 and b1 = 0 has z = h + SiLU(0) = h ([P2] §3.1
    initialisation), so with W2 = W_lm it is the LM head: the separately
    written LM-head oracle must agree with the heads oracle (itself pinned)
    logit for logit, in top-s order and log Z."""
    cfg = synth.tiny().replace(lm_head_variant=True, B=2)
    hi = synth.heads_inputs(cfg)
    w_lm = hi.W2[0]
    ids, logp, logits, logz = oracle.lm_head(hi.h, w_lm, 5, want_logits=True)
    hids, hlogp, hlogits, hlogz = oracle.heads(hi.h, hi.W1[:1], hi.b1[:1], hi.W2[:1], 5,
                                               want_logits=True)
    np.testing.assert_allclose(logits, hlogits[:, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(logz, hlogz[:, 0], rtol=0, atol=1e-12)
    assert np.array_equal(ids, hids[:, 0])
    np.testing.assert_allclose(logp, hlogp[:, 0], rtol=0, atol=1e-12)


def test_lm_head_one_hot_rows_closed_form():
    """W_lm row v = c_v e_{j_v} makes logit v = c_v h[j_v]: closed-form logits,
    log Z and greedy root.  A transposed W_lm, a dropped term or a wrong
    normaliser changes them.  Equal logits rank the smaller id first."""
    rng = np.random.default_rng(11)
    d, V, B = 8, 30, 3
    h = rng.standard_normal((B, d)).astype(np.float32)
    col = rng.integers(0, d, size=V)
    c = rng.uniform(0.5, 3.0, size=V).astype(np.float32)
    col[17], c[17] = col[4], c[4] = col[4], 10.0   # tokens 4 and 17 tie at the top
    h[:, col[4]] = np.abs(h[:, col[4]]) + 1.0
    W = np.zeros((V, d), np.float32)
    W[np.arange(V), col] = c
    ids, logp, logits, logz = oracle.lm_head(h, W, 6, want_logits=True)
    for b in range(B):
        ref = c.astype(np.float64) * h[b, col].astype(np.float64)
        np.testing.assert_allclose(logits[b], ref, atol=1e-12)
        assert logz[b] == pytest.approx(logsumexp(ref), abs=1e-12)
        assert list(ids[b]) == _ref_topk(ref, 6)
        np.testing.assert_allclose(logp[b], ref[ids[b]] - logsumexp(ref), atol=1e-12)
    # the tie at the top: the greedy root is the smaller id, the other is next
    assert (ids[:, 0] == 4).all() and (ids[:, 1] == 17).all()


# ----------------------------------------------------------- attention ----

def _sdpa_path(q_rows, k_rows, v_rows, P, scale):
    """Textbook causal attention (torch float64) of the path queries over
    [prefix ; path]: query t sits at position P+t and sees positions <= P+t."""
    L = q_rows.shape[0]
    qt = torch.from_numpy(q_rows).permute(1, 0, 2)[None]      # [1,H,L,dh]
    kt = torch.from_numpy(k_rows).permute(1, 0, 2)[None]      # [1,H,P+L,dh]
    vt = torch.from_numpy(v_rows).permute(1, 0, 2)[None]
    pos_q = P + torch.arange(L)[:, None]
    pos_k = torch.arange(P + L)[None, :]
    mask = pos_k <= pos_q
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("s,n,P,H,dh", [((2, 2, 2), 14, 32, 1, 64), ((3, 2, 2), 10, 7, 2, 16),
                                        ((4, 3, 2, 2, 1), 40, 0, 3, 8), ((1, 1, 1, 1), 4, 12, 2, 8)])
def test_tree_attention_equals_per_path_causal(s, n, P, H, dh):
    """[P2] §6.1: with the tree mask every root-to-leaf path is exactly an
    independent causal sequence over [prefix ; path]."""
    rng = np.random.default_rng(n + P)
    K = len(s)
    ids = rng.integers(0, 1000, size=(1, K, max(s))).astype(np.int32)
    logp = np.log(np.sort(rng.dirichlet(np.ones(max(s) + 1), size=(1, K))[..., :max(s)], -1)[..., ::-1])
    t = oracle.build_tree([9], ids, logp, list(s), n, prefix_len=[P])
    R = n + 1
    q = rng.standard_normal((1, R, H, dh)).astype(np.float32)
    kc = rng.standard_normal((P + R, H, dh)).astype(np.float32)
    vc = rng.standard_normal((P + R, H, dh)).astype(np.float32)
    scale = 1.0 / math.sqrt(dh)
    out = oracle.tree_attention(q, [kc], [vc], [P], t["anc_mask"], scale)
    for li in range(int(t["n_leaf"][0])):
        path = [int(x) for x in t["paths"][0, li] if x >= 0]
        rows = np.array(path)
        kk = np.concatenate([kc[:P], kc[P + rows]]).astype(np.float64)
        vv = np.concatenate([vc[:P], vc[P + rows]]).astype(np.float64)
        ref = _sdpa_path(q[0, rows].astype(np.float64), kk, vv, P, scale)
        np.testing.assert_allclose(out[0, rows], ref, atol=1e-12, rtol=0)


# ----------------------------------------------------------- posterior ----

def _chain_tree(L, root=0):
    """Chain tree root -> 1 -> ... -> L with tokens 10+i."""
    R = L + 1
    tokens = np.array([[root] + [10 + i for i in range(1, R)]], np.int32)
    parent = np.array([[-1] + list(range(R - 1))], np.int32)
    depth = np.array([list(range(R))], np.int32)
    return tokens, parent, depth


@pytest.mark.parametrize("L_true", [0, 1, 3, 5])
def test_greedy_stops_at_first_mismatch(L_true):
    """[P3] Part 2: greedy verification accepts while the candidate equals the
    target argmax; the first mismatch ends the prefix, even if later
    candidates would match."""
    K, V = 5, 50
    tokens, parent, depth = _chain_tree(K)
    logits = np.zeros((1, K + 1, V), np.float32)
    for i in range(1, K + 1):
        p = parent[0, i]
        if i != L_true + 1:
            logits[0, p, tokens[0, i]] = 5.0          # match
        else:
            logits[0, p, 3] = 5.0                     # mismatch
    logits[0, K, 42] = 9.0
    o = oracle.posterior(logits, tokens, parent, depth, K, oracle.GREEDY)
    assert int(o["accept_len"][0]) == L_true
    assert list(o["path"][0, :L_true + 1]) == list(range(L_true + 1))
    assert np.all(o["path"][0, L_true + 1:] == -1)
    assert list(o["path_tokens"][0, :L_true + 1]) == list(tokens[0, :L_true + 1])
    exp_next = 42 if L_true == K else 0
    if L_true < K:
        exp_next = int(np.argmax(logits[0, L_true]))
    assert int(o["next_token"][0]) == exp_next


@pytest.mark.parametrize("seed", range(8))
def test_longest_path_brute_force_on_random_trees(seed):
    """[P3] Part 2 and [P2] §5: a node counts only if every node of its
    branch is accepted; the deepest such node (the smallest canonical index
    among equals) ends the path, and the next token is the argmax of its
    row.  On random trees with random per-node decisions (given to the
    oracle as forced decisions, so that only its path logic is under test),
    every root-to-node branch is enumerated, and the oracle's accept_len,
    path, path_tokens and next_token must equal the enumeration's."""
    rng = np.random.default_rng(100 + seed)
    K = int(rng.integers(1, 6))
    s = tuple(int(x) for x in rng.integers(1, 4, size=K))
    full = sum(math.prod(s[:k + 1]) for k in range(K))
    n = int(rng.integers(1, full + 1))
    B, V, S = 2, 500, max(s)
    ids = np.stack([np.stack([rng.choice(V, size=S, replace=False) for _ in range(K)])
                    for _ in range(B)]).astype(np.int32)
    p = rng.dirichlet(np.ones(S + 1), size=(B, K))[..., :S]
    t = oracle.build_tree(np.array([7, 9], np.int32), ids, np.log(-np.sort(-p, axis=-1)), s, n)
    R = n + 1
    logits = rng.standard_normal((B, R, V)).astype(np.float32)
    acc = (rng.random((B, R)) < 0.7).astype(np.int32)
    acc[:, 0] = 1
    o = oracle.posterior(logits, t["tokens"], t["parent"], t["depth"], K, oracle.GREEDY,
                         forced_accept=acc)
    assert np.array_equal(o["accept"], acc)
    for b in range(B):
        best, L = 0, 0
        for i in range(1, R):  # ascending: the first node of a depth wins ties
            branch, x = [], i
            while x > 0:
                branch.append(x)
                x = int(t["parent"][b, x])
            assert len(branch) == int(t["depth"][b, i])
            if all(acc[b, y] for y in branch) and len(branch) > L:
                best, L = i, len(branch)
        path, x = [], best
        while x > 0:
            path.append(x)
            x = int(t["parent"][b, x])
        path = [0] + path[::-1]
        pad = [-1] * (K + 1 - len(path))
        assert int(o["accept_len"][b]) == L
        assert list(o["path"][b]) == path + pad
        assert list(o["path_tokens"][b]) == [int(t["tokens"][b, x]) for x in path] + pad
        assert int(o["next_token"][b]) == int(np.argmax(logits[b, best]))


def test_progress_guarantee_all_rejected():
    """[P3] Part 2 / [P2] §5: with every candidate wrong the step still commits
    the root and yields the next greedy token (L = 0, path = [root])."""
    cfg = synth.tiny()
    rng = np.random.default_rng(2)
    ids = rng.integers(0, cfg.V, size=(1, cfg.K, 2)).astype(np.int32)
    logp = np.log(np.full((1, cfg.K, 2), 0.4))
    t = oracle.build_tree([17], ids, logp, cfg.s, cfg.n)
    logits = rng.standard_normal((1, cfg.R, cfg.V)).astype(np.float32)
    for i in range(1, cfg.R):
        logits[0, t["parent"][0, i], t["tokens"][0, i]] = -50.0
    for mode in (oracle.GREEDY, oracle.TYPICAL):
        o = oracle.posterior(logits, t["tokens"], t["parent"], t["depth"], cfg.K, mode)
        assert int(o["accept_len"][0]) == 0
        assert list(o["path"][0]) == [0] + [-1] * cfg.K
        assert list(o["path_tokens"][0]) == [17] + [-1] * cfg.K
        assert int(o["next_token"][0]) == int(np.argmax(logits[0, 0]))


def test_entropy_closed_forms():
    """H of a uniform row is ln V; H of a two-level row has a closed form."""
    V = 1000
    assert oracle.softmax_entropy(np.zeros(V)) == pytest.approx(math.log(V), abs=1e-12)
    m, a = 7, 3.0
    x = np.zeros(V)
    x[:m] = a
    Z = m * math.exp(a) + (V - m)
    ph, pl = math.exp(a) / Z, 1.0 / Z
    Href = -m * ph * math.log(ph) - (V - m) * pl * math.log(pl)
    assert oracle.softmax_entropy(x) == pytest.approx(Href, abs=1e-12)
    # temperature: softmax(x/T) equals softmax of the pre-divided row
    assert oracle.softmax_entropy(x, 2.5) == pytest.approx(oracle.softmax_entropy(x / 2.5), abs=1e-12)


@pytest.mark.parametrize("V,scale,T", [(8, 1.0, 1.0), (1000, 3.0, 0.7), (32000, 3.0, 1.0),
                                        (32000, 30.0, 1.0), (4096, 0.01, 2.0)])
def test_entropy_random_rows_against_scipy(V, scale, T):
    """[P2] §5 uses H(p) = -sum p ln p of p = softmax(logits / T): on random
    rows, from nearly uniform to nearly one-hot, the oracle's entropy equals
    SciPy's softmax and entropy routines (an independent implementation)."""
    from scipy.special import softmax
    from scipy.stats import entropy
    rng = np.random.default_rng(V + int(scale * 10))
    for _ in range(3):
        x = rng.standard_normal(V) * scale
        assert oracle.softmax_entropy(x, T) == pytest.approx(entropy(softmax(x / T)), rel=1e-10,
                                                             abs=1e-12)


@pytest.mark.parametrize("m,a", [(1, 12.0), (2, 6.0), (20, 4.0), (300, 1.0), (900, 2.0)])
def test_typical_threshold_closed_form(m, a):
    """[P2] §5: accept x iff p(x) > min(eps, delta * exp(-H)).  Rows with two
    probability levels give p and H in closed form; the oracle's margin is
    log p - log threshold for tokens of both levels."""
    V, eps, delta = 1000, 0.09, 0.3
    x = np.zeros(V, np.float32)
    x[:m] = a
    Z = m * math.exp(a) + (V - m)
    ph, pl = math.exp(a) / Z, 1.0 / Z
    H = -m * ph * math.log(ph) - (V - m) * pl * math.log(pl)
    thr = min(eps, delta * math.exp(-H))
    tokens = np.array([[0, 0, V - 1]], np.int32)
    parent = np.array([[-1, 0, 0]], np.int32)
    depth = np.array([[0, 1, 1]], np.int32)
    logits = np.stack([x, x, x])[None]
    o = oracle.posterior(logits, tokens, parent, depth, 1, oracle.TYPICAL, eps, delta)
    assert o["margin"][0, 1] == pytest.approx(math.log(ph) - math.log(thr), abs=1e-9)
    assert o["margin"][0, 2] == pytest.approx(math.log(pl) - math.log(thr), abs=1e-9)
    assert o["accept"][0, 1] == int(ph > thr) and o["accept"][0, 2] == int(pl > thr)


def test_typical_threshold_values_and_monotone():
    """min(eps, delta e^{-H}) with eps=.09, delta=.3: switch-over at
    H* = ln(delta/eps); values at H = 1, 3, 6 nats; non-increasing in H."""
    eps, delta = 0.09, 0.3
    thr = lambda H: min(eps, delta * math.exp(-H))
    assert math.log(delta / eps) == pytest.approx(1.2039728, abs=1e-6)
    assert thr(1.0) == pytest.approx(0.09, abs=1e-12)
    assert thr(3.0) == pytest.approx(0.0149361, abs=1e-7)
    assert thr(6.0) == pytest.approx(7.43626e-4, abs=1e-9)
    # the oracle's decision flips exactly where p crosses the threshold:
    # build rows of rising entropy (larger uniform support) with one token at
    # fixed probability 0.05 and check accept <-> 0.05 > thr(H)
    V = 2000
    for m in (1, 3, 10, 100, 1000):
        x = np.full(V, -1e4)
        x[1:m + 1] = 0.0
        # token 0 gets probability 0.05 exactly: e^{x0} / (e^{x0} + m) = 0.05
        x[0] = math.log(0.05 * m / 0.95)
        p = np.exp(x - x.max())
        p /= p.sum()
        H = float(-(p[p > 0] * np.log(p[p > 0])).sum())
        tokens = np.array([[0, 0]], np.int32)
        parent = np.array([[-1, 0]], np.int32)
        depth = np.array([[0, 1]], np.int32)
        o = oracle.posterior(np.stack([x, x]).astype(np.float32)[None], tokens, parent, depth, 1,
                             oracle.TYPICAL, eps, delta)
        assert o["accept"][0, 1] == int(0.05 > thr(H)), (m, H)


def test_longest_path_tie_lowest_index():
    """Two fully accepted branches of the same depth: the lower canonical index
    wins (convention); a deeper accepted branch beats both."""
    # root -> 1, 2 ; 1 -> 3 ; 2 -> 4 ; 4 -> 5
    tokens = np.array([[0, 11, 12, 13, 14, 15]], np.int32)
    parent = np.array([[-1, 0, 0, 1, 2, 4]], np.int32)
    depth = np.array([[0, 1, 1, 2, 2, 3]], np.int32)
    forced = np.array([[1, 1, 1, 1, 1, 0]], np.int32)
    logits = np.zeros((1, 6, 20), np.float32)
    o = oracle.posterior(logits, tokens, parent, depth, 3, oracle.GREEDY, forced_accept=forced)
    assert int(o["accept_len"][0]) == 2 and list(o["path"][0]) == [0, 1, 3, -1]
    forced[0, 5] = 1
    o = oracle.posterior(logits, tokens, parent, depth, 3, oracle.GREEDY, forced_accept=forced)
    assert int(o["accept_len"][0]) == 3 and list(o["path"][0]) == [0, 2, 4, 5]


def test_argmax_tie_lowest_id():
    V = 10
    x = np.zeros(V, np.float32)
    x[[6, 3, 8]] = 2.0
    tokens = np.array([[0, 6]], np.int32)
    parent = np.array([[-1, 0]], np.int32)
    depth = np.array([[0, 1]], np.int32)
    o = oracle.posterior(np.stack([x, x])[None], tokens, parent, depth, 1, oracle.GREEDY)
    assert int(o["accept_len"][0]) == 0 and int(o["next_token"][0]) == 3


# -------------------------------------------------------------- commit ----

def test_commit_kv_gathers_path():
    """The accepted path's rows move to slots P..P+L; new prefix = P+L+1."""
    P, R, H, dh = 4, 6, 2, 3
    kc = np.arange((P + R) * H * dh, dtype=np.float32).reshape(P + R, H, dh)
    vc = -kc.copy()
    k0, v0 = kc.copy(), vc.copy()
    path = np.array([[0, 2, 5, -1]], np.int32)
    new = oracle.commit_kv([kc], [vc], [P], path, [2])
    assert int(new[0]) == P + 3
    assert np.array_equal(kc[:P], k0[:P])
    for q, node in enumerate([0, 2, 5]):
        assert np.array_equal(kc[P + q], k0[P + node]) and np.array_equal(vc[P + q], v0[P + node])


def test_typical_decision_at_the_crossing():
    """[P2] §5 strict rule p(x) > min(eps, delta e^{-H}).  In a two-level row
    (m tokens at logit a, the rest at 0) the low-level token's margin
    log p_low + H - log delta falls through zero as a grows; the float32
    logits just before and just after the closed-form crossing must be
    accepted and rejected respectively."""
    V, m, eps, delta = 1000, 5, 0.09, 0.3

    def f(a):
        Z = m * math.exp(a) + (V - m)
        ph, pl = math.exp(a) / Z, 1.0 / Z
        H = -m * ph * math.log(ph) - (V - m) * pl * math.log(pl)
        thr = min(eps, delta * math.exp(-H))
        return math.log(pl) - math.log(thr), H

    lo, hi = 0.0, 30.0
    assert f(lo)[0] > 0 > f(hi)[0]
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if f(mid)[0] > 0:
            lo = mid
        else:
            hi = mid
    assert f(lo)[1] > math.log(delta / eps)        # entropy branch of the min
    a_below = np.float32(lo)
    while f(float(a_below))[0] <= 0:
        a_below = np.nextafter(a_below, np.float32(-np.inf))
    a_above = np.nextafter(a_below, np.float32(np.inf))
    while f(float(a_above))[0] > 0:
        a_above = np.nextafter(a_above, np.float32(np.inf))
    for a, want in ((a_below, 1), (a_above, 0)):
        x = np.zeros(V, np.float32)
        x[:m] = a
        tokens = np.array([[0, V - 1]], np.int32)
        parent = np.array([[-1, 0]], np.int32)
        depth = np.array([[0, 1]], np.int32)
        o = oracle.posterior(np.stack([x, x])[None], tokens, parent, depth, 1, oracle.TYPICAL,
                             eps, delta)
        assert int(o["accept"][0, 1]) == want, (a, f(float(a)))


# ------------------------------------------------------- exact sampling ----

def _chi2_pvalue(counts, probs):
    from scipy.stats import chisquare
    counts = np.asarray(counts, np.float64)
    probs = np.asarray(probs, np.float64)
    exp = probs / probs.sum() * counts.sum()
    keep = exp > 0
    assert counts[~keep].sum() == 0, "a zero-probability outcome occurred"
    return chisquare(counts[keep], exp[keep]).pvalue


@pytest.mark.parametrize("ctr,key", [
    ([1, 0, 0, 0], [0, 0]), ([6, 7, 9, 11], [123, 456]), ([2 ** 64 - 1, 3, 0, 0], [99, 2 ** 63]),
    ([12345, 2 ** 40, 77, 3], [2 ** 64 - 1, 1])])
def test_philox_matches_numpy(ctr, key):
    """Philox4x64-10 (Salmon et al., SC 2011) against numpy's implementation of
    the same generator (which advances its counter once before the first
    block)."""
    prev = list(ctr)
    if prev[0] == 0:
        prev[0] = 2 ** 64 - 1
        prev[1] -= 1
    else:
        prev[0] -= 1
    g = np.random.Philox(counter=np.array(prev, np.uint64), key=np.array(key, np.uint64))
    assert np.array_equal(oracle.philox4x64(ctr, key), g.random_raw(4).astype(np.uint64))


def test_uniforms_open_interval_float32_exact():
    us = [oracle.uniform(7, 3, p, b, r, v) for p in (1, 2, 3) for b in (0, 5) for r in (0, 2)
          for v in range(9)]
    for u in us:
        assert 0.0 < u < 1.0
        assert float(np.float32(u)) == u
        assert (u * 2 ** 23 - 0.5) == int(u * 2 ** 23 - 0.5)
    # word v % 4 of the block for counter (v // 4, row, b, purpose)
    w = oracle.philox4x64([2, 1, 4, 3], [11, 12])
    for j in range(4):
        assert oracle.uniform(11, 12, 3, 4, 1, 8 + j) == ((int(w[j]) >> 41) + 0.5) / 2 ** 23


def _onehot_heads(c, d=4, j=1):
    """Heads whose logits are c[k][v] * h[j] (W1 = 0, so z = h; W2 rows are
    scaled unit vectors)."""
    K, V = c.shape
    W1 = np.zeros((K, d, d), np.float32)
    W2 = np.zeros((K, V, d), np.float32)
    W2[:, :, j] = c
    return W1, W2


def test_draft_sampling_frequencies():
    """Gumbel-max drafts follow softmax(logits / T): 40000 independent
    sequences, chi-square against the closed-form probabilities per head."""
    rng = np.random.default_rng(5)
    c = rng.uniform(-2, 2, size=(2, 6)).astype(np.float32)
    W1, W2 = _onehot_heads(c)
    B = 40000
    h = np.zeros((B, 4), np.float32)
    h[:, 1] = 1.0
    T = 0.7
    drafts, logits, _ = oracle.draft_sample(h, W1, None, W2, T, seed=123, step=4)
    for k in range(2):
        np.testing.assert_allclose(logits[0, k], c[k], atol=1e-7)
        ck = c[k].astype(np.float64)
        p = np.exp(ck / T - logsumexp(ck / T))
        counts = np.bincount(drafts[:, k], minlength=6)
        assert _chi2_pvalue(counts, p) > 1e-4, (k, counts, p)


def _spec_case(p_logits, q_logits, B, T=1.0, seed=9, step=2):
    """Chain of K drafts x_k ~ q_k (oracle's draft sampler) verified against
    fixed rows p_0..p_K; every sequence has its own random streams."""
    K, V = q_logits.shape
    W1, W2 = _onehot_heads(q_logits.astype(np.float32))
    h = np.zeros((B, 4), np.float32)
    h[:, 1] = 1.0
    drafts, _, _ = oracle.draft_sample(h, W1, None, W2, T, seed=seed, step=step)
    tokens = np.concatenate([np.full((B, 1), 0, np.int32), drafts], axis=1)
    logits = np.broadcast_to(p_logits.astype(np.float32), (B, K + 1, V))
    dl = np.broadcast_to(q_logits.astype(np.float32), (B, K, V))
    return tokens, oracle.speculative_posterior(logits, tokens, dl, T, seed, step)


def test_speculative_emits_target_distribution():
    """[P1] Acceptance rules / [P2] §3: accepting x ~ q with probability
    min(1, p/q) and resampling from (p - q)+ at the first rejection yields
    tokens distributed exactly as p.  K = 2 over 60000 sequences: the first
    emitted token follows p_0; after an accepted first draft the second
    follows p_1; with both accepted the bonus follows p_2.  The acceptance
    rate of the first draft is sum_v min(p_0, q_1)."""
    rng = np.random.default_rng(8)
    V, K, B = 7, 2, 60000
    p_logits = rng.normal(0, 1.2, size=(K + 1, V))
    q_logits = rng.normal(0, 1.2, size=(K, V))
    tokens, o = _spec_case(p_logits, q_logits, B)
    p = np.exp(p_logits - logsumexp(p_logits, axis=1, keepdims=True))
    q = np.exp(q_logits - logsumexp(q_logits, axis=1, keepdims=True))
    L = o["accept_len"]
    first = np.where(L >= 1, tokens[:, 1], o["next_token"])
    assert _chi2_pvalue(np.bincount(first, minlength=V), p[0]) > 1e-4
    sel = L >= 1
    second = np.where(L[sel] >= 2, tokens[sel, 2], o["next_token"][sel])
    assert _chi2_pvalue(np.bincount(second, minlength=V), p[1]) > 1e-4
    both = L == 2
    assert _chi2_pvalue(np.bincount(o["next_token"][both], minlength=V), p[2]) > 1e-4
    rate = np.minimum(p[0], q[0]).sum()
    n1 = (L >= 1).sum()
    assert abs(n1 / B - rate) < 5 * math.sqrt(rate * (1 - rate) / B)
    # bookkeeping: accept flags, path tokens and margins agree with L
    for b in range(50):
        assert list(o["path_tokens"][b, :L[b] + 1]) == list(tokens[b, :L[b] + 1])
        assert (o["path_tokens"][b, L[b] + 1:] == -1).all()
        assert all(o["accept"][b, :L[b]] == 1) and (L[b] == K or o["accept"][b, L[b]] == 0)
        assert all((o["margin"][b, :L[b]] > 0))


def test_speculative_q_equal_p_accepts_everything():
    """q = p makes p/q = 1 > u for every u in (0, 1): all K drafts are
    accepted and the next token is the bonus sample from the last row."""
    rng = np.random.default_rng(3)
    V, K, B = 5, 3, 2000
    lg = rng.normal(0, 1, size=(K, V))
    p_logits = np.concatenate([lg, rng.normal(0, 1, size=(1, V))])
    _, o = _spec_case(p_logits, lg, B)
    assert (o["accept_len"] == K).all()
    assert (o["sample_row"] == K).all()


def test_speculative_replacement_has_positive_residual():
    """A rejected draft is replaced by a token where p > q (the normalised
    positive residual puts no mass elsewhere), and T divides both sides'
    logits."""
    rng = np.random.default_rng(4)
    V, K, B, T = 6, 1, 5000, 1.7
    p_logits = rng.normal(0, 2, size=(K + 1, V))
    q_logits = rng.normal(0, 2, size=(K, V))
    tokens, o = _spec_case(p_logits, q_logits, B, T=T)
    p = np.exp(p_logits[0] / T - logsumexp(p_logits[0] / T))
    q = np.exp(q_logits[0] / T - logsumexp(q_logits[0] / T))
    rej = o["accept_len"] == 0
    assert rej.any()
    assert (p[o["next_token"][rej]] > q[o["next_token"][rej]]).all()
    first = np.where(o["accept_len"] >= 1, tokens[:, 1], o["next_token"])
    assert _chi2_pvalue(np.bincount(first, minlength=V), p) > 1e-4
