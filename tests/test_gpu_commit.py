"""GPU-vs-oracle parity of the KV-cache commit (medusa_commit_kv and the fused
medusa_evaluate_posterior_commit), through the C ABI.

The commit moves bytes, so the bar is bit-exact: every byte of every cache
and every new prefix length must equal the oracle's.  Paths come from the
oracle's posterior on planted logits, or are drawn directly from the tree
(any root-to-node walk), so that both short and full-depth paths occur.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import medusa_speculative_decoding_02_gb300 as m
from medusa_speculative_decoding_02_gb300 import build as mbuild

pytestmark = pytest.mark.gpu


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
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(a).to(dev)


def N(t):
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def tree_for(rng, s, n, prefix, V=32000):
    B = len(prefix)
    ids = np.stack([np.stack([rng.choice(V, size=max(s), replace=False) for _ in s])
                    for _ in range(B)]).astype(np.int32)
    p = rng.dirichlet(np.ones(max(s) + 1), size=(B, len(s)))[..., :max(s)]
    logp = np.log(-np.sort(-p, axis=-1))
    return oracle.build_tree(np.arange(B, dtype=np.int32) + 3, ids, logp, s, n,
                             prefix_len=np.asarray(prefix, np.int32))


def random_paths(rng, ot, K):
    """A root-to-node walk per sequence: a uniformly drawn node and its
    ancestors, padded with -1 (the layout medusa_evaluate_posterior writes)."""
    B, R = ot["tokens"].shape
    path = np.full((B, K + 1), -1, np.int32)
    L = np.zeros(B, np.int32)
    for b in range(B):
        x = int(rng.integers(0, R))
        d = int(ot["depth"][b, x])
        L[b] = d
        for q in range(d, -1, -1):
            path[b, q] = x
            x = int(ot["parent"][b, x])
    return path, L


def device_caches(cfg, dev, extra_slots=0):
    ai = synth.attention_inputs(cfg, extra_slots=extra_slots)
    kc = [T(x, dev) for x in ai.k_cache]
    vc = [T(x, dev) for x in ai.v_cache]
    return ai, kc, vc


def check_caches(kc, vc, ok, ov):
    for b in range(len(kc)):
        assert np.array_equal(N(kc[b]), ok[b]), f"K cache of sequence {b}"
        assert np.array_equal(N(vc[b]), ov[b]), f"V cache of sequence {b}"


CASES = [
    # name, dtype, s, n, H, dh, prefix
    ("tiny", "f32", (2, 2, 2), 14, 1, 64, (32,)),
    ("v7b", "bf16", (4, 3, 2, 2, 1), 64, 32, 128, (1024,)),
    ("ragged", "bf16", (4, 4, 2), 32, 3, 64, (0, 1, 77)),
    ("wide", "bf16", (16, 16), 255, 2, 128, (5, 300)),
    ("deep", "f32", (1,) * 8, 8, 2, 64, (9,)),
    ("odd_row", "f32", (3, 2), 6, 1, 4, (2, 17)),
]


@pytest.mark.parametrize("name,dtype,s,n,H,dh,prefix", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_commit_kv_matches_oracle(dev, name, dtype, s, n, H, dh, prefix, seed):
    """Random accepted paths (L from 0 to the tree's depth) on ragged
    prefixes: caches and new prefix lengths bit-exact against the oracle."""
    cfg = synth.v7b().replace(name=f"commit_{name}", dtype=dtype, B=len(prefix), s=s, n=n, H=H,
                              dh=dh, prefix=prefix, K=len(s))
    rng = np.random.default_rng(100 * seed + len(name))
    ot = tree_for(rng, s, n, prefix)
    path, L = random_paths(rng, ot, len(s))
    ai, kc, vc = device_caches(cfg, dev, extra_slots=seed)
    g_npl = m.commit_kv(m.F32 if dtype == "f32" else m.BF16, m.cache_pointers(kc, dev),
                        m.cache_pointers(vc, dev), T(ai.prefix_len, dev), T(path, dev),
                        T(L, dev), cfg.R, H, dh)
    torch.cuda.synchronize()
    ok = [x.copy() for x in ai.k_cache]
    ov = [x.copy() for x in ai.v_cache]
    o_npl = oracle.commit_kv(ok, ov, ai.prefix_len, path, L)
    assert np.array_equal(N(g_npl), o_npl)
    check_caches(kc, vc, ok, ov)


def test_commit_full_depth_and_root_only(dev):
    """L = K (the deepest node of a chain tree: every row moves) and L = 0
    (only the root, already in place: nothing moves)."""
    s = (1, 1, 1, 1, 1)
    cfg = synth.v7b().replace(name="commit_edges", B=2, s=s, n=5, H=4, dh=128, prefix=(64, 3))
    rng = np.random.default_rng(9)
    ot = tree_for(rng, s, 5, cfg.prefix)
    path = np.array([[0, 1, 2, 3, 4, 5], [0, -1, -1, -1, -1, -1]], np.int32)
    L = np.array([5, 0], np.int32)
    assert (ot["parent"][0, 1:] == np.arange(5)).all()
    ai, kc, vc = device_caches(cfg, dev)
    g = m.commit_kv(m.BF16, m.cache_pointers(kc, dev), m.cache_pointers(vc, dev),
                    T(ai.prefix_len, dev), T(path, dev), T(L, dev), cfg.R, 4, 128)
    ok = [x.copy() for x in ai.k_cache]
    ov = [x.copy() for x in ai.v_cache]
    o = oracle.commit_kv(ok, ov, ai.prefix_len, path, L)
    assert np.array_equal(N(g), o) and list(o) == [70, 4]
    check_caches(kc, vc, ok, ov)
    # a chain tree's path is already in place: the caches are unchanged
    check_caches(kc, vc, ai.k_cache, ai.v_cache)


@pytest.mark.parametrize("mode", [m.GREEDY, m.TYPICAL])
@pytest.mark.parametrize("cfg_fn", [synth.v7b, synth.batch8], ids=["v7b", "batch8"])
def test_posterior_commit_fused(dev, cfg_fn, mode):
    """The fused call: posterior outputs equal medusa_evaluate_posterior's and
    the caches equal the oracle's posterior followed by the oracle's commit.
    Three steps in a row, each starting from the previous new prefix (the
    tree slots of step t+1 are the rows just past the new prefix)."""
    cfg = cfg_fn()
    K = cfg.K
    ai, kc, vc = device_caches(cfg, dev, extra_slots=2 * K + 2)
    ok = [x.copy() for x in ai.k_cache]
    ov = [x.copy() for x in ai.v_cache]
    prefix = ai.prefix_len.copy()
    kp, vp = m.cache_pointers(kc, dev), m.cache_pointers(vc, dev)
    for step in range(3):
        rng = np.random.default_rng(7 + step)
        ot = tree_for(rng, cfg.s, cfg.n, prefix)
        logits = synth.base_logits(cfg, rep=step)
        for b in range(cfg.B):
            lb = logits[b:b + 1]
            synth.plant_chain(lb, ot["tokens"][b:b + 1], ot["parent"][b:b + 1],
                              ot["depth"][b:b + 1], (step + b) % (K + 1),
                              synth.rng_for(cfg, "plant", 10 * step + b))
        l16 = synth.cast(logits, "bf16")
        lg = T(l16, dev)
        args = (T(ot["tokens"], dev), T(ot["parent"], dev), T(ot["depth"], dev))
        ref = m.evaluate_posterior(lg, *args, K, mode)
        gp, g_npl = m.evaluate_posterior_commit(lg, *args, K, kp, vp, T(prefix, dev), cfg.H,
                                                cfg.dh, mode=mode)
        torch.cuda.synchronize()
        for key in ("accept_len", "path", "path_tokens", "next_token", "accept"):
            assert torch.equal(getattr(gp, key), getattr(ref, key)), key
        op = oracle.posterior(l16, ot["tokens"], ot["parent"], ot["depth"], K, mode, 0.09, 0.3,
                              1.0)
        g_acc = N(gp.accept)
        mism = g_acc != op["accept"]
        assert not (mism & ~(np.abs(op["margin"]) < 1e-3)).any()
        if mism.any():
            op = oracle.posterior(l16, ot["tokens"], ot["parent"], ot["depth"], K, mode, 0.09,
                                  0.3, 1.0, forced_accept=g_acc)
        path, L = N(gp.path), N(gp.accept_len)
        assert np.array_equal(path, op["path"]) and np.array_equal(L, op["accept_len"])
        o_npl = oracle.commit_kv(ok, ov, prefix, path, L)
        assert np.array_equal(N(g_npl), o_npl)
        check_caches(kc, vc, ok, ov)
        prefix = o_npl


def test_commit_device_checks(dev):
    """Bad data the host cannot see sets the status word, leaves the sequence
    untouched and returns its old prefix; the other sequences commit."""
    s = (4, 3, 2)
    cfg = synth.v7b().replace(name="commit_bad", B=3, s=s, n=20, H=2, dh=64, prefix=(10, 20, 30),
                              K=3)
    rng = np.random.default_rng(5)
    ot = tree_for(rng, s, 20, cfg.prefix)
    path, L = random_paths(rng, ot, 3)
    cases = []
    p1 = path.copy(); l1 = L.copy(); l1[1] = 4                 # accept_len > K
    cases.append((p1, l1, None, 7))
    p2 = path.copy(); l2 = L.copy(); l2[1] = 2; p2[1, :3] = [0, 2, cfg.R]  # node index R
    cases.append((p2, l2, None, 7))
    p3 = path.copy(); l3 = L.copy(); l3[1] = 1; p3[1, :2] = [0, -1]        # negative index
    cases.append((p3, l3, None, 7))
    cases.append((path, L, np.array([10, -1, 30], np.int32), 3))           # negative prefix
    for pth, acc, pre, code in cases:
        ai, kc, vc = device_caches(cfg, dev)
        pl = ai.prefix_len if pre is None else pre
        ws = m.new_workspace(m.WS_HEADER, dev)
        g = m.commit_kv(m.BF16, m.cache_pointers(kc, dev), m.cache_pointers(vc, dev), T(pl, dev),
                        T(pth, dev), T(acc, dev), cfg.R, 2, 64, ws=ws)
        assert m.read_device_status(ws) == code
        ok = [x.copy() for x in ai.k_cache]
        ov = [x.copy() for x in ai.v_cache]
        good = [0, 2]
        o = oracle.commit_kv([ok[b] for b in good], [ov[b] for b in good], pl[good], pth[good],
                             acc[good])
        assert np.array_equal(N(g)[good], o)
        assert int(N(g)[1]) == int(pl[1])
        check_caches(kc, vc, ok, ov)


def test_cache_pointer_checks(dev):
    """A cache pointer that is not 16-byte aligned is reported (status 8) by
    the commit, the fused commit and the attention, none of which touches
    memory through it."""
    cfg = synth.v7b().replace(name="commit_ptr", B=2, s=(2, 2), n=6, H=1, dh=64, prefix=(8, 8),
                              K=2)
    rng = np.random.default_rng(6)
    ot = tree_for(rng, cfg.s, cfg.n, cfg.prefix)
    path, L = random_paths(rng, ot, 2)
    ai, kc, vc = device_caches(cfg, dev)
    kp = m.cache_pointers(kc, dev)
    vp = m.cache_pointers(vc, dev)
    kp_bad = kp.clone()
    kp_bad[1] += 2                       # misaligned: rejected before any access
    ws = m.new_workspace(m.WS_HEADER, dev)
    g = m.commit_kv(m.BF16, kp_bad, vp, T(ai.prefix_len, dev), T(path, dev), T(L, dev), cfg.R, 1,
                    64, ws=ws)
    assert m.read_device_status(ws) == 8
    assert int(N(g)[1]) == 8
    ok = [x.copy() for x in ai.k_cache]
    ov = [x.copy() for x in ai.v_cache]
    oracle.commit_kv(ok[:1], ov[:1], ai.prefix_len[:1], path[:1], L[:1])
    check_caches(kc, vc, ok[:1] + [ai.k_cache[1]], ov[:1] + [ai.v_cache[1]])
    # the fused commit
    logits = T(synth.cast(synth.base_logits(cfg.replace(B=2)), "bf16"), dev)
    wsp = m.new_workspace(m.posterior_workspace_size(2, cfg.R), dev)
    vp_bad = vp.clone()
    vp_bad += 8                          # 8-byte aligned only
    m.evaluate_posterior_commit(logits, T(ot["tokens"], dev), T(ot["parent"], dev),
                                T(ot["depth"], dev), 2, kp, vp_bad, T(ai.prefix_len, dev), 1, 64,
                                ws=wsp)
    assert m.read_device_status(wsp) == 8
    # attention
    wsa = m.new_workspace(m.tree_attention_workspace_size(m.BF16, 2, cfg.R, 1, 64, 8), dev)
    out = m.tree_attention(T(ai.q, dev), kp_bad, vp, T(ai.prefix_len, dev), 8,
                           T(ot["anc_mask"].view(np.int64), dev), ws=wsa)
    assert m.read_device_status(wsa) == 8
    assert not out[1].float().abs().sum().item()
    assert torch.isfinite(out[0].float()).all()
