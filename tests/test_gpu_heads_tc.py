"""The heads on the tensor cores (several bf16 sequences), against the oracle.

The path takes batches of 2..8 bf16 sequences with d a multiple of 256 and V
a multiple of 8: phase 1 (W1 h, bias, SiLU, residual) and phase 2 (W2 z,
running softmax normaliser and top-s) as tcgen05 MMAs fed by TMA, then the
same merge of the per-CTA partials as the CUDA-core path.  Shapes below
cover: batches that do not fill the 8 sequence columns, one head and eight
heads, vocabularies whose per-CTA shares are not multiples of 128 rows,
hidden sizes at and above 4096, top-1 and top-16, and a non-zero bias.

Tolerances as in test_gpu_parity: ids bit-exact except where the oracle's
logit gap is < 1e-3; log-probabilities within 1e-2 + 2e-2 relative.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import medusa_speculative_decoding_02_gb300 as m
from medusa_speculative_decoding_02_gb300 import build as mbuild
from test_gpu_parity import N, T, check_topk

pytestmark = pytest.mark.gpu

TIMEOUT = 6  # MEDUSA_DEV_TIMEOUT


@pytest.fixture(scope="module")
def dev():
    mbuild.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def case(B, d, V, K, S, bias_std, seed):
    cfg = synth.tiny().replace(name=f"tc{B}_{d}_{V}_{K}_{S}", dtype="bf16", B=B, d=d, V=V, K=K,
                               s=(S,) * K, w1_std=1.0 / np.sqrt(d), w2_std=0.05, seed=seed)
    hi = synth.heads_inputs(cfg)
    if bias_std:
        rng = np.random.default_rng(seed)
        hi.b1 = synth.cast(rng.standard_normal((K, d)).astype(np.float32) * bias_std, "bf16")
    return cfg, hi


def run(dev, hi, S, ws=None):
    ids, logp = m.heads(T(hi.h, dev), T(hi.W1, dev), T(hi.b1, dev), T(hi.W2, dev), S, ws=ws)
    torch.cuda.synchronize()
    return N(ids), N(logp)


@pytest.mark.parametrize("B,d,V,K,S,bias", [
    (8, 1024, 4000, 5, 4, 0.5),     # V/8 = 500 units over 30 CTAs a head: ragged tiles
    (3, 2048, 2000, 1, 16, 0.0),    # one head: all 152 CTAs on it; top-16
    (5, 512, 8000, 8, 1, 0.3),      # eight heads (19 CTAs each); top-1
    (7, 4096, 1216, 4, 8, 0.5),     # d = 4096; eight 8-row units per phase-2 CTA
    (4, 1536, 32000, 3, 3, 0.2),    # the full vocabulary
    (2, 1024, 4000, 5, 4, 0.5),     # two sequences (the smallest batch on this path)
])
def test_heads_tc_shapes(dev, B, d, V, K, S, bias):
    cfg, hi = case(B, d, V, K, S, bias, seed=B * 1000 + K)
    ids, logp = run(dev, hi, S)
    o_ids, _, o_logits, o_logz = oracle.heads(hi.h, hi.W1, hi.b1, hi.W2, S, want_logits=True)
    check_topk(ids, logp, o_ids, o_logits, o_logz)


def test_heads_tc_repeat_same_bits(dev):
    """Two calls on the same inputs give the same bits (the partials and
    their merge have a fixed order)."""
    cfg, hi = case(6, 1024, 4096, 5, 4, 0.5, seed=7)
    a = run(dev, hi, 4)
    b = run(dev, hi, 4)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1].view(np.uint32), b[1].view(np.uint32))


def test_heads_tc_batch_columns_independent(dev):
    """Each sequence's result equals the batch-1 (CUDA-core) result for that
    sequence up to the tolerance: no column of the MMA leaks into another."""
    cfg, hi = case(8, 1024, 4000, 2, 4, 0.5, seed=11)
    ids8, logp8 = run(dev, hi, 4)
    for b in (0, 5, 7):
        one = synth.HeadsInputs(h=hi.h[b:b + 1], W1=hi.W1, b1=hi.b1, W2=hi.W2)
        ids1, logp1 = run(dev, one, 4)
        o_ids, _, o_logits, o_logz = oracle.heads(one.h, one.W1, one.b1, one.W2, 4,
                                                  want_logits=True)
        check_topk(ids8[b:b + 1], logp8[b:b + 1], o_ids, o_logits, o_logz)
        check_topk(ids1, logp1, o_ids, o_logits, o_logz)


def test_heads_tc_wait_timeout_sets_status_and_context_survives(dev):
    """With the wait budget at 0 every bounded wait of the tensor-core heads
    gives up at once: the status word reads "timeout", the kernel drains its
    copies and MMAs and frees its tensor memory, and the context stays
    usable: with the budget restored the same call matches the oracle."""
    cfg, hi = case(8, 1024, 4000, 5, 4, 0.5, seed=3)
    ws = m.new_workspace(m.heads_workspace_size(8, 5, 1024, 4000, 4), dev)
    default = m.wait_budget()
    m.set_wait_budget(0)
    try:
        run(dev, hi, 4, ws=ws)
        assert m.read_device_status(ws) == TIMEOUT
    finally:
        m.set_wait_budget(default)
    m.clear_device_status(ws)
    ids, logp = run(dev, hi, 4, ws=ws)
    assert m.read_device_status(ws) == 0
    o_ids, _, o_logits, o_logz = oracle.heads(hi.h, hi.W1, hi.b1, hi.W2, 4, want_logits=True)
    check_topk(ids, logp, o_ids, o_logits, o_logz)


@pytest.mark.parametrize("B", [2, 8])
def test_heads_tc_lm_head(dev, B):
    """The LM head in the same tensor-core pass (head 0 multiplies h itself,
    from its own weight matrix): the root and its log-probability against
    the oracle's LM head, the Medusa heads' top-s against the oracle."""
    from test_gpu_heads_lm import check_root
    K, d, V, S = 5, 1024, 4000, 4
    cfg, hi = case(B, d, V, K, S, 0.5, seed=50 + B)
    w_lm = synth.lm_head_weight(cfg)
    root, root_lp, ids, logp = m.heads_lm(T(hi.h, dev), T(w_lm, dev), T(hi.W1, dev),
                                          T(hi.b1, dev), T(hi.W2, dev), S)
    torch.cuda.synchronize()
    o_ids, _, o_logits, o_logz = oracle.lm_head(hi.h, w_lm, 1, want_logits=True)
    check_root(N(root), N(root_lp), o_ids, o_logits, o_logz)
    h_ids, _, h_logits, h_logz = oracle.heads(hi.h, hi.W1, hi.b1, hi.W2, S, want_logits=True)
    check_topk(N(ids), N(logp), h_ids, h_logits, h_logz)


@pytest.mark.parametrize("B,temp", [(2, 0.7), (8, 1.0)])
def test_heads_tc_sampling(dev, B, temp):
    """Drafts sampled in the tensor-core pass (top-1 of logit / T plus the
    Gumbel noise of the library's Philox streams): ids equal the oracle's
    outside a key gap of 1e-3, and the raw logits written out match."""
    K, d, V = 5, 1024, 4000
    cfg, hi = case(B, d, V, K, 1, 0.5, seed=70 + B)
    seed, step = 99 + B, 5
    drafts, dl = m.heads_sample(T(hi.h, dev), T(hi.W1, dev), T(hi.b1, dev), T(hi.W2, dev), temp,
                                seed, step)
    torch.cuda.synchronize()
    g_dr, g_dl = N(drafts), N(dl)
    o_dr, o_lg, o_keys = oracle.draft_sample(hi.h, hi.W1, hi.b1, hi.W2, temp, seed, step,
                                             want_keys=True)
    err = np.abs(g_dl - o_lg)
    assert err.max() <= 1e-2, err.max()
    for b in range(B):
        for k in range(K):
            a, o = int(g_dr[b, k]), int(o_dr[b, k])
            if a != o:
                assert o_keys[b, k, o] - o_keys[b, k, a] < 1e-3, (b, k, a, o)
