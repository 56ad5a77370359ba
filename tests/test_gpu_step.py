"""The step executor (medusa_step_create / medusa_step_run): one native call
issues a whole decoding step -- the input copies from pinned host memory,
heads, tree, tree attention and posterior (with the fused commit) -- and its
results equal those of the separate calls on the same inputs, bit for bit,
and the oracle's posterior on the executor's tree."""
import numpy as np
import pytest
import torch

import oracle
import synth
import medusa_speculative_decoding_02_gb300 as m
from medusa_speculative_decoding_02_gb300 import build as mbuild
from test_gpu_parity import N, check_posterior

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    mbuild.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _t(a, dev=None):
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16 \
        else torch.from_numpy(a)
    return t if dev is None else t.to(dev)


class Step:
    """Device buffers of one step on `cfg`, the pinned host sources of its
    inputs, and the same step issued as separate calls."""

    def __init__(self, cfg, dev, commit=False, pinned_results=True, graph=False):
        self.cfg, self.dev = cfg, dev
        hi = synth.heads_inputs(cfg)
        ai = synth.attention_inputs(cfg)
        B, K, S, n, R, V = cfg.B, cfg.K, cfg.top_s, cfg.n, cfg.R, cfg.V
        self.W1, self.b1, self.W2 = _t(hi.W1, dev), _t(hi.b1, dev), _t(hi.W2, dev)
        self.kc = [_t(x, dev) for x in ai.k_cache]
        self.vc = [_t(x, dev) for x in ai.v_cache]
        self.kp, self.vp = m.cache_pointers(self.kc, dev), m.cache_pointers(self.vc, dev)
        self.prefix = torch.tensor(ai.prefix_len, dtype=torch.int32, device=dev)
        dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
        self.h = torch.empty((B, cfg.d), dtype=dt, device=dev)
        self.root = torch.empty((B,), dtype=torch.int32, device=dev)
        self.q = torch.empty((B, R, cfg.H, cfg.dh), dtype=dt, device=dev)
        self.logits = torch.empty((B, R, V), dtype=dt, device=dev)
        pin = lambda t: torch.empty(t.shape, dtype=t.dtype).pin_memory()
        self.host = {"h": pin(self.h), "root": pin(self.root), "q": pin(self.q),
                     "logits": pin(self.logits)}
        # the tree's own K/V rows (slots P_b .. P_b+R-1) arrive from the host too
        P = [int(x) for x in ai.prefix_len]
        self.kv_rows = [(self.kc[b][P[b]:P[b] + R], self.vc[b][P[b]:P[b] + R]) for b in range(B)]
        self.host_kv = [(pin(k), pin(v)) for k, v in self.kv_rows]
        self.mode = m.TYPICAL if cfg.mode == "typical" else m.GREEDY
        self.ws = m.new_workspace(max(
            m.heads_workspace_size(B, K, cfg.d, V, S), m.build_tree_workspace_size(B, K, S, n),
            m.tree_attention_workspace_size(m.BF16 if dt == torch.bfloat16 else m.F32, B, R,
                                            cfg.H, cfg.dh, cfg.P_max),
            m.posterior_workspace_size(B, R)), dev)
        self.ids = torch.empty((B, K, S), dtype=torch.int32, device=dev)
        self.logp = torch.empty((B, K, S), dtype=torch.float32, device=dev)
        self.tree = m.Tree.empty(B, n, K, dev)
        self.out = torch.empty_like(self.q)
        self.post = m.Posterior.pinned(B, R, K) if pinned_results else \
            m.Posterior.empty(B, R, K, dev)
        self.new_prefix = torch.empty((B,), dtype=torch.int32, device=dev) if commit else None
        self.ex = self.make_executor(graph)

    def make_executor(self, graph):
        cfg = self.cfg
        late = [(self.q, self.host["q"]), (self.logits, self.host["logits"])]
        for (k, v), (hk, hv) in zip(self.kv_rows, self.host_kv):
            late += [(k, hk), (v, hv)]
        return m.StepExecutor(
            h=self.h, W1=self.W1, b1=self.b1, W2=self.W2, top_s=cfg.top_s,
            topk=(self.ids, self.logp), root=self.root, s=cfg.s, n=cfg.n,
            prefix_len=self.prefix, tree=self.tree, q=self.q, k_ptrs=self.kp, v_ptrs=self.vp,
            P_max=cfg.P_max, attn_out=self.out, logits=self.logits, post=self.post, K=cfg.K,
            mode=self.mode, eps=cfg.eps, delta=cfg.delta, temperature=cfg.temperature,
            ws=self.ws, early=[(self.h, self.host["h"]), (self.root, self.host["root"])],
            late=late, new_prefix_len=self.new_prefix, graph=graph)

    def fill(self, rep):
        cfg = self.cfg
        self.host["h"].copy_(_t(synth.hidden_states(cfg, rep=rep)))
        self.host["root"].copy_(torch.from_numpy(synth.root_tokens(cfg, rep=rep)))
        ai = synth.attention_inputs(cfg, rep=rep)
        self.host["q"].copy_(_t(ai.q))
        self.host["logits"].copy_(_t(synth.cast(synth.base_logits(cfg, rep=rep), cfg.dtype)))
        R = cfg.R
        for b, (hk, hv) in enumerate(self.host_kv):
            P = int(ai.prefix_len[b])
            hk.copy_(_t(ai.k_cache[b][P:P + R]))
            hv.copy_(_t(ai.v_cache[b][P:P + R]))

    def results(self):
        t = self.tree
        r = {"ids": self.ids, "logp": self.logp, "tokens": t.tokens, "parent": t.parent,
             "depth": t.depth, "pos_id": t.pos_id, "anc_mask": t.anc_mask, "paths": t.paths,
             "n_leaf": t.n_leaf, "out": self.out, "accept_len": self.post.accept_len,
             "path": self.post.path, "path_tokens": self.post.path_tokens,
             "next_token": self.post.next_token, "accept": self.post.accept}
        if self.new_prefix is not None:
            r["new_prefix"] = self.new_prefix
        return {k: v.detach().clone().cpu() for k, v in r.items()}

    def separate_calls(self):
        """The same step as the individual public calls (inputs already on
        the device)."""
        cfg = self.cfg
        m.heads(self.h, self.W1, self.b1, self.W2, cfg.top_s, ws=self.ws,
                out=(self.ids, self.logp))
        m.build_tree(self.root, self.ids, self.logp, cfg.s, cfg.n, prefix_len=self.prefix,
                     ws=self.ws, out=self.tree)
        m.tree_attention(self.q, self.kp, self.vp, self.prefix, cfg.P_max, self.tree.anc_mask,
                         out=self.out, ws=self.ws)
        if self.new_prefix is None:
            m.evaluate_posterior(self.logits, self.tree.tokens, self.tree.parent, self.tree.depth,
                                 cfg.K, self.mode, cfg.eps, cfg.delta, cfg.temperature, ws=self.ws,
                                 out=self.post)
        else:
            m.evaluate_posterior_commit(self.logits, self.tree.tokens, self.tree.parent,
                                        self.tree.depth, cfg.K, self.kp, self.vp, self.prefix,
                                        cfg.H, cfg.dh, new_prefix_len=self.new_prefix,
                                        mode=self.mode, eps=cfg.eps, delta=cfg.delta,
                                        temperature=cfg.temperature, ws=self.ws, out=self.post)
        torch.cuda.synchronize()


def _same(a: dict, b: dict):
    assert a.keys() == b.keys()
    for k in a:
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("graph", [False, True])
def test_step_executor_tiny_matches_calls_and_oracle(dev, graph):
    cfg = synth.tiny()
    st = Step(cfg, dev, graph=graph)
    for rep in (0, 1, 2):
        st.fill(rep)
        st.ex.run()
        got = st.results()
        # the root is the host's, the posterior the oracle's on the executor's tree
        assert int(got["tokens"][0, 0]) == int(synth.root_tokens(cfg, rep=rep)[0])
        ot = {k: N(getattr(st.tree, k)) for k in ("tokens", "parent", "depth")}
        check_posterior(st.post, synth.base_logits(cfg, rep=rep), ot, cfg.K,
                        st.mode, cfg.eps, cfg.delta, cfg.temperature)
        st.separate_calls()
        _same(got, st.results())
    assert m.read_device_status(st.ws) == 0


@pytest.mark.parametrize("graph", [False, True])
def test_step_executor_v7b_commit_matches_calls(dev, graph):
    """Vicuna-7B shape, bf16, typical acceptance, tree K/V rows from the
    host and the fused commit: caches, prefix lengths and every output equal
    the separate calls' from the same starting state."""
    cfg = synth.v7b().replace(mode="typical")
    st = Step(cfg, dev, commit=True, graph=graph)
    for rep in (0, 1):
        st.fill(rep)
        k0 = [k.clone() for k in st.kc]
        v0 = [v.clone() for v in st.vc]
        st.ex.run()
        got = st.results()
        gk = [k.clone() for k in st.kc]
        gv = [v.clone() for v in st.vc]
        assert int(got["new_prefix"][0]) == int(st.prefix[0]) + int(got["accept_len"][0]) + 1
        for b in range(cfg.B):  # the executor's starting state, then the separate calls
            st.kc[b].copy_(k0[b])
            st.vc[b].copy_(v0[b])
            k, v = st.kv_rows[b]
            k.copy_(st.host_kv[b][0])
            v.copy_(st.host_kv[b][1])
        for name in ("h", "root", "q", "logits"):
            getattr(st, name).copy_(st.host[name])
        st.separate_calls()
        _same(got, st.results())
        for b in range(cfg.B):
            assert torch.equal(gk[b], st.kc[b]) and torch.equal(gv[b], st.vc[b])
    assert m.read_device_status(st.ws) == 0


@pytest.mark.parametrize("graph", [False, True])
def test_step_executor_runs_without_waiting_then_waits(dev, graph):
    """Steps issued without waiting, then one waited for: the wait covers
    the last step (the completion words count every run issued), and the
    results equal the separate calls'."""
    cfg = synth.v7b().replace(mode="typical")
    st = Step(cfg, dev, graph=graph)
    st.fill(4)
    for _ in range(3):
        st.ex.run(synchronize=False)
    st.ex.run()
    got = st.results()
    st.ex.run(synchronize=False)
    st.ex.wait()  # the wait of run() on its own
    _same(got, st.results())
    st.separate_calls()
    _same(got, st.results())
    assert m.read_device_status(st.ws) == 0


@pytest.mark.parametrize("graph", [False, True])
def test_step_executor_batch8_matches_calls(dev, graph):
    """Eight ragged 7B sequences: the heads run on the tensor cores (tensor
    maps built on the host at issue, or once at capture in graph mode); the
    executor equals the separate calls bit for bit over two steps."""
    cfg = synth.batch8()
    st = Step(cfg, dev, graph=graph)
    for rep in (0, 1):
        st.fill(rep)
        st.ex.run()
        got = st.results()
        assert torch.equal(got["tokens"][:, 0], torch.from_numpy(synth.root_tokens(cfg, rep=rep)))
        st.separate_calls()
        _same(got, st.results())
    assert m.read_device_status(st.ws) == 0


@pytest.mark.parametrize("graph", [False, True])
def test_step_executor_on_a_side_stream_with_device_results(dev, graph):
    """Issued on a non-default stream without waiting, with device-resident
    results, the step completes in stream order like the separate calls."""
    cfg = synth.tiny()
    st = Step(cfg, dev, pinned_results=False, graph=graph)
    st.fill(3)
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    st.ex.run(stream=s, synchronize=False)
    s.synchronize()
    got = st.results()
    st.separate_calls()
    _same(got, st.results())


def test_step_executor_reports_a_call_error(dev):
    """A call that fails its host checks ends the run with that call's
    status, and nothing is launched."""
    cfg = synth.tiny()
    st = Step(cfg, dev)
    st.fill(0)
    small = m.new_workspace(m.WS_HEADER, dev)
    ex = m.StepExecutor(
        h=st.h, W1=st.W1, b1=st.b1, W2=st.W2, top_s=cfg.top_s, topk=(st.ids, st.logp),
        root=st.root, s=cfg.s, n=cfg.n, prefix_len=st.prefix, tree=st.tree, q=st.q,
        k_ptrs=st.kp, v_ptrs=st.vp, P_max=cfg.P_max, attn_out=st.out, logits=st.logits,
        post=st.post, K=cfg.K, ws=small, early=[(st.h, st.host["h"])])
    before = m.launch_count()
    with pytest.raises(m.MedusaError) as e:
        ex.run()
    assert e.value.status == 3  # MEDUSA_ERR_WORKSPACE, from medusa_heads
    assert m.launch_count() == before
    ex.close()
    with pytest.raises(m.MedusaError):
        ex.run()


def test_step_executor_graph_mode_reports_a_call_error_at_create(dev):
    """In graph mode the calls' host checks run while capturing: a failing
    call makes the construction fail with its status and leaves no
    executor."""
    cfg = synth.tiny()
    st = Step(cfg, dev)
    small = m.new_workspace(m.WS_HEADER, dev)
    before = m.launch_count()
    with pytest.raises(m.MedusaError) as e:
        m.StepExecutor(
            h=st.h, W1=st.W1, b1=st.b1, W2=st.W2, top_s=cfg.top_s, topk=(st.ids, st.logp),
            root=st.root, s=cfg.s, n=cfg.n, prefix_len=st.prefix, tree=st.tree, q=st.q,
            k_ptrs=st.kp, v_ptrs=st.vp, P_max=cfg.P_max, attn_out=st.out, logits=st.logits,
            post=st.post, K=cfg.K, ws=small, early=[(st.h, st.host["h"])],
            late=[(st.q, st.host["q"])], graph=True)
    assert e.value.status == 3
    assert m.launch_count() == before
    # the stream and the context stay usable
    st.fill(1)
    st.ex.run()
    got = st.results()
    st.separate_calls()
    _same(got, st.results())


def test_step_executor_refuses_pageable_sources(dev):
    """The executor resolves each copy's direction at create: a pageable
    host source, or a host destination, is refused before any work (the
    binding refuses pageable tensors itself, so the descriptor is built
    here by hand)."""
    import ctypes
    cfg = synth.tiny()
    st = Step(cfg, dev)
    nb = st.h.numel() * st.h.element_size()
    pageable = torch.empty(st.h.shape, dtype=st.h.dtype)
    copies = (m._Copy * 1)(m._Copy(st.h.data_ptr(), pageable.data_ptr(), nb))
    s_host = (ctypes.c_int32 * cfg.K)(*cfg.s)
    t, p = st.tree, st.post
    fields = dict(early=ctypes.addressof(copies), n_early=1, dtype=m.F32, h=st.h, W1=st.W1,
                  b1=st.b1, W2=st.W2, B=cfg.B, d=cfg.d, V=cfg.V, K=cfg.K, top_s=cfg.top_s,
                  topk_ids=st.ids, topk_logp=st.logp, root=st.root,
                  s_host=ctypes.addressof(s_host), n=cfg.n, prefix_len=st.prefix,
                  tokens=t.tokens, parent=t.parent, depth=t.depth, pos_id=t.pos_id,
                  anc_mask=t.anc_mask, paths=t.paths, n_leaf=t.n_leaf, q=st.q, k_cache=st.kp,
                  v_cache=st.vp, P_max=cfg.P_max, H=cfg.H, dh=cfg.dh, scale=0.125,
                  attn_out=st.out, logits=st.logits, mode=m.GREEDY, eps=0.09, delta=0.3,
                  temperature=1.0, accept_len=p.accept_len, path=p.path,
                  path_tokens=p.path_tokens, next_token=p.next_token, ws=st.ws,
                  ws_bytes=st.ws.numel())
    d = m._StepDesc()
    for k, v in fields.items():
        setattr(d, k, v.data_ptr() if isinstance(v, torch.Tensor) else v)
    lib = m.lib()
    h = ctypes.c_void_p()
    assert lib.medusa_step_create(ctypes.byref(d), ctypes.byref(h)) == 1
    assert "source is neither" in lib.medusa_last_error().decode()
    assert h.value is None
    copies[0] = m._Copy(st.host["h"].data_ptr(), st.h.data_ptr(), nb)  # host destination
    assert lib.medusa_step_create(ctypes.byref(d), ctypes.byref(h)) == 1
    assert "destination is not device memory" in lib.medusa_last_error().decode()
    copies[0] = m._Copy(st.h.data_ptr(), st.host["h"].data_ptr(), nb)  # pinned source
    assert lib.medusa_step_create(ctypes.byref(d), ctypes.byref(h)) == 0
    lib.medusa_step_destroy(h)


def test_step_executor_graph_keeps_the_wait_budget_of_create(dev):
    """In graph mode the attention's wait budget is the one in force at
    create.  Captured with a budget of 0 (fault injection: every mbarrier
    wait of the tensor-core attention gives up at once), each replay reports
    "timeout" with zero attention rows even after the budget is restored; a
    stream-mode executor made afterwards uses the restored budget and equals
    the separate calls, so the context stays usable."""
    cfg = synth.v7b().replace(mode="typical")
    default = m.wait_budget()
    assert default > 0
    m.set_wait_budget(0)
    try:
        st = Step(cfg, dev, graph=True)
    finally:
        m.set_wait_budget(default)
    st.fill(0)
    for _ in range(2):
        st.ex.run()
        assert m.read_device_status(st.ws) == 6  # MEDUSA_DEV_TIMEOUT
        assert torch.count_nonzero(st.out) == 0
        m.clear_device_status(st.ws)
    st.ex.close()
    ex = st.make_executor(graph=False)
    ex.run()
    assert m.read_device_status(st.ws) == 0
    got = st.results()
    assert torch.count_nonzero(got["out"]) > 0
    st.separate_calls()
    _same(got, st.results())
