"""StepGraph: a full decoding step (input copies, heads, tree, tree
attention, posterior, result copy) captured once and replayed.  Each replay
reads the pinned inputs afresh and equals the same calls issued eagerly."""
import math

import numpy as np
import pytest
import torch

import synth
import medusa_speculative_decoding_02_gb300 as m
from medusa_speculative_decoding_02_gb300 import build as mbuild

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    mbuild.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def test_step_graph_replays_with_new_inputs(dev):
    cfg = synth.tiny()
    hi = synth.heads_inputs(cfg)
    ai = synth.attention_inputs(cfg)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32))
    W1, b1, W2 = f32(hi.W1).to(dev), f32(hi.b1).to(dev), f32(hi.W2).to(dev)
    kc, vc = f32(ai.k_cache[0]).to(dev), f32(ai.v_cache[0]).to(dev)
    kp, vp = m.cache_pointers([kc], dev), m.cache_pointers([vc], dev)
    prefix = torch.tensor(ai.prefix_len, dtype=torch.int32, device=dev)
    B, K, S, n, R, V = cfg.B, cfg.K, cfg.top_s, cfg.n, cfg.R, cfg.V
    # device inputs the graph reads, and their pinned host sources
    h = torch.empty((B, cfg.d), device=dev)
    root = torch.empty((B,), dtype=torch.int32, device=dev)
    q = torch.empty((B, R, 1, cfg.dh), device=dev)
    logits = torch.empty((B, R, V), device=dev)
    host = dict(h=torch.empty(h.shape).pin_memory(),
                root=torch.empty(root.shape, dtype=torch.int32).pin_memory(),
                q=torch.empty(q.shape).pin_memory(), logits=torch.empty(logits.shape).pin_memory())
    ws = m.new_workspace(max(m.heads_workspace_size(B, K, cfg.d, V, S),
                             m.build_tree_workspace_size(B, K, S, n),
                             m.tree_attention_workspace_size(m.F32, B, R, 1, cfg.dh, cfg.P_max),
                             m.posterior_workspace_size(B, R)), dev)
    ids = torch.empty((B, K, S), dtype=torch.int32, device=dev)
    logp = torch.empty((B, K, S), device=dev)
    tree = m.Tree.empty(B, n, K, dev)
    out = torch.empty_like(q)
    post = m.Posterior.empty(B, R, K, dev, with_accept=False)
    host_next = torch.empty((B,), dtype=torch.int32).pin_memory()
    host_out = torch.empty(out.shape).pin_memory()

    def issue():
        for name, t in (("h", h), ("root", root), ("q", q), ("logits", logits)):
            t.copy_(host[name], non_blocking=True)
        m.heads(h, W1, b1, W2, S, ws=ws, out=(ids, logp))
        m.build_tree(root, ids, logp, cfg.s, n, prefix_len=prefix, ws=ws, out=tree)
        m.tree_attention(q, kp, vp, prefix, cfg.P_max, tree.anc_mask, out=out, ws=ws)
        m.evaluate_posterior(logits, tree.tokens, tree.parent, tree.depth, K, m.TYPICAL, ws=ws,
                             out=post)
        host_next.copy_(post.next_token, non_blocking=True)
        host_out.copy_(out, non_blocking=True)

    def fill(rep):
        host["h"].copy_(f32(synth.heads_inputs(cfg, rep=rep).h))
        host["root"].copy_(torch.from_numpy(synth.root_tokens(cfg, rep=rep)))
        host["q"].copy_(f32(synth.attention_inputs(cfg, rep=rep).q))
        host["logits"].copy_(f32(synth.base_logits(cfg, rep=rep)))

    fill(0)
    graph = m.StepGraph(issue)
    for rep in (1, 2, 3):
        fill(rep)
        graph.replay()
        torch.cuda.synchronize()
        g_next, g_out = host_next.clone(), host_out.clone()
        g_tokens = tree.tokens.clone()
        issue()  # the same step, eagerly
        torch.cuda.synchronize()
        assert torch.equal(g_next, host_next)
        assert torch.equal(g_out, host_out)
        assert torch.equal(g_tokens, tree.tokens)
        assert int(g_tokens[0, 0]) == int(synth.root_tokens(cfg, rep=rep)[0])
    assert m.read_device_status(ws) == 0
