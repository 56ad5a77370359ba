"""Fault injection for the bounded device waits, on the GPU, without a hung
or faulted GPU.

The tensor-core attention waits on mbarriers for its own MMAs.  With the wait
budget at 0 every such wait in the key loop gives up at once: the kernel must
record the "timeout" device status, stop its key loop, drain its MMAs and
copies with its fixed limit, free its tensor memory and return.  The context
must stay usable: after the budget is restored and the status cleared, the
same call on the same buffers matches the oracle again.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
import medusa_speculative_decoding_02_gb300 as m
from medusa_speculative_decoding_02_gb300 import build as mbuild

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


def T(a, dev):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(a).to(dev)


def attention_case(dev, n, prefix, H=2):
    cfg = synth.v7b().replace(name=f"fault{n}_{prefix}_{H}", H=H, n=n,
                              s=(8, 4, 4, 2, 2) if n > 64 else (4, 3, 2, 2, 1), prefix=(prefix,))
    rng = np.random.default_rng(n + prefix)
    S = max(cfg.s)
    ids = np.stack([rng.choice(cfg.V, size=S, replace=False) for _ in cfg.s])[None].astype(np.int32)
    p = rng.dirichlet(np.ones(S + 1), size=(1, len(cfg.s)))[..., :S]
    logp = np.log(-np.sort(-p, axis=-1))
    ot = oracle.build_tree(np.array([7], np.int32), ids, logp, cfg.s, cfg.n,
                           prefix_len=np.asarray(cfg.prefix, np.int32))
    ai = synth.attention_inputs(cfg)
    kc = [T(x, dev) for x in ai.k_cache]
    vc = [T(x, dev) for x in ai.v_cache]
    args = dict(q=T(ai.q, dev), k_ptrs=m.cache_pointers(kc, dev), v_ptrs=m.cache_pointers(vc, dev),
                prefix_len=T(ai.prefix_len, dev), P_max=cfg.P_max,
                anc_mask=T(ot["anc_mask"].view(np.int64), dev))
    ws = m.new_workspace(m.tree_attention_workspace_size(m.BF16, 1, cfg.R, cfg.H, cfg.dh,
                                                         cfg.P_max), dev)
    from test_gpu_parity import oracle_attention_heads
    ref = oracle_attention_heads(ai, ot["anc_mask"], cfg.dh, list(range(cfg.H)))
    return args, ws, ref, (kc, vc)


def run(args, ws):
    out = m.tree_attention(args["q"], args["k_ptrs"], args["v_ptrs"], args["prefix_len"],
                           args["P_max"], args["anc_mask"], ws=ws)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


@pytest.mark.parametrize("n,prefix,H", [(64, 1024, 2), (64, 0, 2), (128, 3000, 2), (200, 700, 2),
                                         (128, 8192, 32)])
def test_attention_wait_timeout_sets_status_and_context_survives(dev, n, prefix, H):
    """Every (head, key range) CTA times out: the status word reads "timeout"
    and every output row is zero (no key range survives the merge); then,
    with the default budget back, the same buffers give the oracle's result.
    The last case (129 rows over prefix 8192, 32 heads) runs the one-tile
    variant whose last row is computed on the CUDA cores."""
    args, ws, ref, _keep = attention_case(dev, n, prefix, H)
    default = m.wait_budget()
    assert default > 0
    m.set_wait_budget(0)
    try:
        assert m.wait_budget() == 0
        out = run(args, ws)
        assert m.read_device_status(ws) == TIMEOUT
        assert np.all(out == 0.0)
    finally:
        m.set_wait_budget(default)
    m.clear_device_status(ws)
    out = run(args, ws)
    assert m.read_device_status(ws) == 0
    err = np.abs(out - ref)
    assert (err <= 1e-2 + np.abs(ref) * 2.0 ** -9).all(), err.max()
