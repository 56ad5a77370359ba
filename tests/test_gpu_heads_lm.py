"""GPU-vs-oracle parity of the fused LM-head + Medusa-heads pass
(medusa_heads_lm), through the C ABI.

Bar: the root token is bit-exact unless the oracle's gap between the GPU's
choice and its own is < 1e-3 (near-tie exemption); root log-probabilities
and the heads' log-probs within max-abs 1e-2 + relative 2e-2; the Medusa
heads' top-s lists match the oracle as in the heads parity tests, and are
the same candidates as medusa_heads on the same inputs (the LM head shares
the pass but not the arithmetic of any other head).
"""
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
    return t.detach().cpu().numpy()


def check_root(g_root, g_lp, o_ids, o_logits, o_logz):
    for b in range(len(g_root)):
        a, o = int(g_root[b]), int(o_ids[b, 0])
        if a != o:
            gap = abs(o_logits[b, a] - o_logits[b, o])
            assert gap < GAP, (b, a, o, gap)
        ref = o_logits[b, a] - o_logz[b]
        assert abs(g_lp[b] - ref) <= ATOL + RTOL * abs(ref), (b, g_lp[b], ref)


def check_topk(g_ids, g_logp, o_ids, o_logits, o_logz):
    B, K, S = g_ids.shape
    for b in range(B):
        for k in range(K):
            assert len(set(g_ids[b, k].tolist())) == S
            for j in range(S):
                a, o = int(g_ids[b, k, j]), int(o_ids[b, k, j])
                if a != o:
                    assert abs(o_logits[b, k, a] - o_logits[b, k, o]) < GAP, (b, k, j)
                ref = o_logits[b, k, a] - o_logz[b, k]
                assert abs(g_logp[b, k, j] - ref) <= ATOL + RTOL * abs(ref), (b, k, j)


def run(cfg, dev, hi, w_lm):
    """heads_lm, and the plain heads call on the same inputs.  The two may
    take different paths (several bf16 sequences run the plain heads on the
    tensor cores), so each is compared with the oracle, not with the other."""
    args = (T(hi.h, dev), T(w_lm, dev), T(hi.W1, dev), T(hi.b1, dev), T(hi.W2, dev))
    root, root_lp, ids, logp = m.heads_lm(*args, cfg.top_s)
    ids_ref, logp_ref = m.heads(args[0], *args[2:], cfg.top_s)
    torch.cuda.synchronize()
    return N(root), N(root_lp), N(ids), N(logp), N(ids_ref), N(logp_ref)


CASES = [
    # dtype, B, d, V, K, S
    ("f32", 1, 64, 1000, 3, 2), ("bf16", 1, 64, 1000, 3, 4), ("bf16", 3, 72, 1031, 2, 16),
    ("f32", 2, 128, 1031, 4, 5), ("bf16", 8, 136, 999, 5, 8), ("bf16", 5, 256, 4000, 8, 16),
    ("f32", 1, 8, 17, 1, 16), ("bf16", 2, 520, 20011, 3, 4), ("bf16", 1, 1024, 32000, 8, 4),
]


@pytest.mark.parametrize("dtype,B,d,V,K,S", CASES)
def test_heads_lm_shapes(dev, dtype, B, d, V, K, S):
    """Ragged d and V, every batch bucket, K up to 8 (nine heads in the pass,
    two head groups per CTA at batch 1)."""
    cfg = synth.tiny().replace(name=f"lm{dtype}{B}{d}{V}{K}{S}", dtype=dtype, B=B, d=d, V=V, K=K,
                               s=(S,) * K, w1_std=0.05, w2_std=0.05)
    hi = synth.heads_inputs(cfg)
    w_lm = synth.lm_head_weight(cfg)
    root, root_lp, ids, logp, ids_ref, logp_ref = run(cfg, dev, hi, w_lm)
    o_ids, _, o_logits, o_logz = oracle.lm_head(hi.h, w_lm, 1, want_logits=True)
    check_root(root, root_lp, o_ids, o_logits, o_logz)
    h_ids, _, h_logits, h_logz = oracle.heads(hi.h, hi.W1, hi.b1, hi.W2, S, want_logits=True)
    check_topk(ids, logp, h_ids, h_logits, h_logz)
    check_topk(ids_ref, logp_ref, h_ids, h_logits, h_logz)


@pytest.mark.parametrize("cfg_fn", [synth.v7b, synth.batch8], ids=["v7b", "batch8"])
def test_heads_lm_full_size(dev, cfg_fn):
    """Vicuna-7B shapes: the root over the 32000-token LM head; the heads'
    top-s against the oracle on two of the five heads (each head is an
    independent computation)."""
    cfg = cfg_fn()
    hi = synth.heads_inputs(cfg)
    w_lm = synth.lm_head_weight(cfg)
    root, root_lp, ids, logp, ids_ref, logp_ref = run(cfg, dev, hi, w_lm)
    o_ids, _, o_logits, o_logz = oracle.lm_head(hi.h, w_lm, 1, want_logits=True)
    check_root(root, root_lp, o_ids, o_logits, o_logz)
    for k in (0, cfg.K - 1):
        h_ids, _, h_logits, h_logz = oracle.heads(hi.h, hi.W1[k:k + 1], hi.b1[k:k + 1],
                                                  hi.W2[k:k + 1], cfg.top_s, want_logits=True)
        check_topk(ids[:, k:k + 1], logp[:, k:k + 1], h_ids, h_logits, h_logz)
        check_topk(ids_ref[:, k:k + 1], logp_ref[:, k:k + 1], h_ids, h_logits, h_logz)


def test_heads_lm_identity_variant(dev):
    """W1 = 0, b1 = 0 and every W2 = W_lm: every Medusa head is the LM head,
    so each head's best token is the root and its log-prob the root's."""
    cfg = synth.v7b(lm_head_variant=True)
    hi = synth.heads_inputs(cfg)
    w_lm = synth.lm_head_weight(cfg)
    root, root_lp, ids, logp, _, _ = run(cfg, dev, hi, w_lm)
    for k in range(cfg.K):
        assert np.array_equal(ids[:, k, 0], root)
        np.testing.assert_array_equal(logp[:, k, 0], root_lp)


def test_heads_lm_root_ties(dev):
    """Equal logits: the root is the smaller token id."""
    d, V = 64, 1000
    cfg = synth.tiny().replace(name="lmtie", d=d, V=V, K=1, s=(2,))
    hi = synth.heads_inputs(cfg)
    w_lm = np.zeros((V, d), np.float32)
    w_lm[[811, 90, 433], 0] = 3.0
    hi.h[:] = 1.0
    root, root_lp, _, _, _, _ = run(cfg, dev, hi, w_lm)
    assert int(root[0]) == 90
    ref = 3.0 - np.log(3 * np.exp(3.0) + (V - 3))
    assert abs(float(root_lp[0]) - ref) < 1e-5
