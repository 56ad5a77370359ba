"""The OpenMP build of the oracle (used only to time the CPU baseline on all
host cores) gives the same bits as the serial build the parity tests use."""
import math

import numpy as np
import pytest

import oracle
import synth


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()
    if not oracle.parallel_available():
        pytest.skip("no OpenMP compiler support on this host")
    yield
    oracle.set_parallel(False)


def _both(fn):
    oracle.set_parallel(False)
    a = fn()
    oracle.set_parallel(True)
    try:
        b = fn()
    finally:
        oracle.set_parallel(False)
    return a, b


def _same(a, b):
    if isinstance(a, dict):
        assert a.keys() == b.keys()
        for k in a:
            _same(a[k], b[k])
    elif isinstance(a, (tuple, list)):
        assert len(a) == len(b)
        for x, y in zip(a, b):
            _same(x, y)
    elif a is None:
        assert b is None
    else:
        x, y = np.asarray(a), np.asarray(b)
        assert x.dtype == y.dtype and x.shape == y.shape
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_parallel_build_same_bits(dtype):
    cfg = synth.tiny().replace(name="omp", dtype=dtype, B=2, d=128, V=3000, H=4,
                               prefix=(40, 7))
    hi = synth.heads_inputs(cfg)
    heads = _both(lambda: oracle.heads(hi.h, hi.W1, hi.b1, hi.W2, cfg.top_s, want_logits=True))
    _same(*heads)
    ids, logp = heads[0][0], heads[0][1]
    root = synth.root_tokens(cfg)
    t = oracle.build_tree(root, ids, logp, cfg.s, cfg.n, prefix_len=np.asarray(cfg.prefix))
    ai = synth.attention_inputs(cfg)
    _same(*_both(lambda: oracle.tree_attention(ai.q, ai.k_cache, ai.v_cache, ai.prefix_len,
                                               t["anc_mask"], 1.0 / math.sqrt(cfg.dh))))
    lg = synth.base_logits(cfg)
    synth.plant_bernoulli(lg, t["tokens"], t["parent"], synth.rng_for(cfg, "plant"))
    lg = synth.cast(lg, dtype)
    for mode in (oracle.GREEDY, oracle.TYPICAL):
        _same(*_both(lambda: oracle.posterior(lg, t["tokens"], t["parent"], t["depth"], cfg.K,
                                              mode, cfg.eps, cfg.delta, cfg.temperature)))


def test_posterior_rejects_bad_parent_in_both_builds():
    lg = np.zeros((1, 3, 10), np.float32)
    tokens = np.array([[0, 1, 2]], np.int32)
    parent = np.array([[-1, 0, 2]], np.int32)   # node 2 names itself
    depth = np.array([[0, 1, 2]], np.int32)
    for par in (False, True):
        oracle.set_parallel(par)
        with pytest.raises(RuntimeError):
            oracle.posterior(lg, tokens, parent, depth, 2, oracle.GREEDY, 0.09, 0.3, 1.0)
    oracle.set_parallel(False)
