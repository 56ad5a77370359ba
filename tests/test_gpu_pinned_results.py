"""Posterior results written straight into page-locked host memory.

medusa_evaluate_posterior and the fused posterior + commit accept pinned
host buffers as outputs: the select kernel writes the results there, so a
decoding step needs no copy back.  Each case runs the same call once with
device outputs and once with pinned outputs and compares every result (the
commit case also compares the caches, bit for bit).  Pageable host memory is
refused before anything is launched.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
import medusa_speculative_decoding_02_gb300 as m
from medusa_speculative_decoding_02_gb300 import build as mbuild
from test_gpu_commit import N, T, device_caches, tree_for

pytestmark = pytest.mark.gpu

KEYS = ("accept_len", "path", "path_tokens", "next_token", "accept")


@pytest.fixture(scope="module")
def dev():
    mbuild.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def case(cfg, dev, seed):
    """A tree from the oracle's builder and logits with a planted chain per
    sequence (lengths 0..K across the batch)."""
    rng = np.random.default_rng(seed)
    prefix = np.asarray(cfg.prefix, np.int32)
    ot = tree_for(rng, cfg.s, cfg.n, prefix)
    logits = synth.base_logits(cfg, rep=seed)
    for b in range(cfg.B):
        synth.plant_chain(logits[b:b + 1], ot["tokens"][b:b + 1], ot["parent"][b:b + 1],
                          ot["depth"][b:b + 1], b % (cfg.K + 1),
                          synth.rng_for(cfg, "plant", seed * 10 + b))
    lg = T(synth.cast(logits, "bf16"), dev)
    args = (T(ot["tokens"], dev), T(ot["parent"], dev), T(ot["depth"], dev))
    return lg, args


@pytest.mark.parametrize("mode", [m.GREEDY, m.TYPICAL])
@pytest.mark.parametrize("cfg_fn", [synth.v7b, synth.batch8], ids=["v7b", "batch8"])
def test_posterior_pinned_equals_device(dev, cfg_fn, mode):
    cfg = cfg_fn()
    lg, args = case(cfg, dev, seed=3)
    ref = m.evaluate_posterior(lg, *args, cfg.K, mode)
    pin = m.Posterior.pinned(cfg.B, cfg.R, cfg.K)
    for t in (pin.accept_len, pin.path, pin.path_tokens, pin.next_token, pin.accept):
        t.fill_(-7)  # every slot must be written
    m.evaluate_posterior(lg, *args, cfg.K, mode, out=pin)
    torch.cuda.synchronize()
    for key in KEYS:
        assert torch.equal(getattr(pin, key), getattr(ref, key).cpu()), key


def test_posterior_commit_pinned_equals_device(dev):
    """The fused commit with pinned results: results and caches equal those of
    the same call with device results, each on its own copy of the caches."""
    cfg = synth.batch8()
    lg, args = case(cfg, dev, seed=5)
    prefix = T(np.asarray(cfg.prefix, np.int32), dev)
    _, kc_a, vc_a = device_caches(cfg, dev, extra_slots=cfg.K + 1)
    _, kc_b, vc_b = device_caches(cfg, dev, extra_slots=cfg.K + 1)
    ptrs_a = (m.cache_pointers(kc_a, dev), m.cache_pointers(vc_a, dev))
    ptrs_b = (m.cache_pointers(kc_b, dev), m.cache_pointers(vc_b, dev))
    ref, npl_a = m.evaluate_posterior_commit(lg, *args, cfg.K, *ptrs_a, prefix, cfg.H, cfg.dh,
                                             mode=m.TYPICAL)
    pin = m.Posterior.pinned(cfg.B, cfg.R, cfg.K)
    _, npl_b = m.evaluate_posterior_commit(lg, *args, cfg.K, *ptrs_b, prefix, cfg.H, cfg.dh,
                                           mode=m.TYPICAL, out=pin)
    torch.cuda.synchronize()
    for key in KEYS:
        assert torch.equal(getattr(pin, key), getattr(ref, key).cpu()), key
    assert torch.equal(npl_a, npl_b)
    for b in range(cfg.B):
        assert np.array_equal(N(kc_a[b]), N(kc_b[b])) and np.array_equal(N(vc_a[b]), N(vc_b[b]))


def test_pageable_results_refused(dev):
    """A pageable host buffer as a result is refused (MEDUSA_ERR_INVALID_ARG)
    by the C ABI and by the binding, and nothing is launched."""
    cfg = synth.v7b()
    lg, args = case(cfg, dev, seed=2)
    B, R, V, K = cfg.B, cfg.R, cfg.V, cfg.K
    ws = m.new_workspace(m.posterior_workspace_size(B, R), dev)
    dev_out = m.Posterior.empty(B, R, K, dev)
    pageable = np.zeros(B, np.int32)
    L = m.lib()
    before = L.medusa_launch_count()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = L.medusa_evaluate_posterior(
        m.BF16, p(lg), p(args[0]), p(args[1]), p(args[2]), B, R, V, K, m.GREEDY, 0.09, 0.3, 1.0,
        ctypes.c_void_p(pageable.ctypes.data), p(dev_out.path), p(dev_out.path_tokens),
        p(dev_out.next_token), p(dev_out.accept), p(ws), ws.numel(), None)
    assert rc == 1
    assert "pageable" in m.lib().medusa_last_error().decode()
    assert L.medusa_launch_count() == before
    bad = m.Posterior(torch.zeros(B, dtype=torch.int32), dev_out.path, dev_out.path_tokens,
                      dev_out.next_token, None)
    with pytest.raises(ValueError):
        m.evaluate_posterior(lg, *args, K, m.GREEDY, out=bad)
