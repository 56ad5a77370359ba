"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments before launching anything."""
import ctypes
import os
import re

import pytest

import medusa_speculative_decoding_02_gb300 as m
from medusa_speculative_decoding_02_gb300 import build as mbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
P = ctypes.c_void_p
A = P(4096)          # fake, 16-byte aligned device address: never dereferenced
MISALIGNED = P(4100)
WS = P(1 << 20)      # fake 256-byte aligned workspace


@pytest.fixture(scope="module")
def L():
    mbuild.build()
    return m.lib()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"MEDUSA_API[^;(]*?\b(medusa_\w+)\s*\(", txt, flags=re.S))
    return names


def test_exports_every_declared_symbol(L):
    names = declared_symbols()
    assert len(names) >= 13
    for n in names:
        assert hasattr(L, n), n
    assert set(m.EXPORTS) <= names


def test_wait_budget_roundtrip(L):
    default = m.wait_budget()
    assert default == 1 << 16 or "MEDUSA_FAULT_WAIT_BUDGET" in os.environ
    try:
        m.set_wait_budget(123)
        assert m.wait_budget() == 123
        m.set_wait_budget(0)
        assert m.wait_budget() == 0
    finally:
        m.set_wait_budget(default)
    assert m.wait_budget() == default


@pytest.mark.parametrize("value,expect", [("7", 7), ("0", 0), ("junk", 1 << 16), ("", 1 << 16)])
def test_wait_budget_from_environment(L, value, expect):
    """MEDUSA_FAULT_WAIT_BUDGET sets the budget a process starts with; a value
    that is not a whole number leaves the default."""
    import subprocess
    import sys
    env = dict(os.environ, MEDUSA_FAULT_WAIT_BUDGET=value)
    r = subprocess.run([sys.executable, "-c",
                        "import medusa_speculative_decoding_02_gb300 as m; print(m.wait_budget())"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert int(r.stdout.strip().splitlines()[-1]) == expect


def test_status_strings(L):
    for code, name in m.STATUS.items():
        assert L.medusa_status_string(code).decode() == name


def _heads(L, **kw):
    a = dict(dtype=m.BF16, h=A, W1=A, b1=None, W2=A, B=1, d=4096, V=32000, K=5, s=4, ids=A,
             logp=A, ws=WS, ws_bytes=1 << 30)
    a.update(kw)
    return L.medusa_heads(a["dtype"], a["h"], a["W1"], a["b1"], a["W2"], a["B"], a["d"], a["V"],
                          a["K"], a["s"], a["ids"], a["logp"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(h=None), 1), (dict(W2=None), 1), (dict(dtype=7), 1), (dict(B=0), 2), (dict(B=9), 2),
    (dict(K=0), 1), (dict(K=9), 1), (dict(d=12), 1), (dict(s=0), 1), (dict(s=17), 1),
    (dict(V=3, s=4), 1), (dict(B=8, d=8192), 2), (dict(W1=MISALIGNED), 1), (dict(ws=None), 3),
    (dict(ws=P((1 << 20) + 16)), 3), (dict(ws_bytes=100), 3)])
def test_heads_rejects(L, kw, code):
    before = L.medusa_launch_count()
    assert _heads(L, **kw) == code
    assert L.medusa_launch_count() == before
    assert L.medusa_last_error().decode()


def _tree(L, s=(4, 3, 2, 2, 1), n=64, **kw):
    a = dict(root=A, ids=A, logp=A, B=1, K=len(s), S=max(s), ws=WS, ws_bytes=1 << 20)
    a.update(kw)
    sh = (ctypes.c_int32 * len(s))(*s)
    return L.medusa_build_tree(a["root"], a["ids"], a["logp"], a["B"], a["K"], sh, a["S"], n, None,
                               A, A, A, A, A, A, A, a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("args,code", [
    (dict(n=137), 1), (dict(n=0), 1), (dict(n=256, s=(16, 16)), 1), (dict(s=(4, 3, 2, 2, 1), S=3), 1),
    (dict(K=9, s=(1,) * 9), 1), (dict(root=None), 1), (dict(ws=None), 3), (dict(B=0), 1)])
def test_tree_rejects(L, args, code):
    before = L.medusa_launch_count()
    assert _tree(L, **args) == code
    assert L.medusa_launch_count() == before


@pytest.mark.parametrize("args,code", [
    (dict(n=137), 1), (dict(n=0), 1), (dict(K=9, s=(1,) * 9), 1), (dict(root=None), 1),
    (dict(ws=None), 3), (dict(B=0), 1), (dict(logp=None), 1)])
def test_tree_static_rejects(L, args, code):
    s = args.pop("s", (4, 3, 2, 2, 1))
    n = args.pop("n", 64)
    a = dict(root=A, ids=A, logp=A, B=1, K=len(s), S=max(s), ws=WS, ws_bytes=1 << 20)
    a.update(args)
    sh = (ctypes.c_int32 * len(s))(*s)
    before = L.medusa_launch_count()
    rc = L.medusa_build_tree_static(a["root"], a["ids"], a["logp"], a["B"], a["K"], sh, a["S"], n,
                                    None, A, A, A, A, A, A, A, a["ws"], a["ws_bytes"], None)
    assert rc == code
    assert L.medusa_launch_count() == before


def test_tree_full_cartesian_budget_accepted_by_validation(L):
    # n equal to the full node count passes validation; with a NULL output the
    # call must still be rejected before any launch.
    sh = (ctypes.c_int32 * 5)(4, 3, 2, 2, 1)
    rc = L.medusa_build_tree(A, A, A, 1, 5, sh, 4, 136, None, None, A, A, A, A, A, A, WS, 1 << 20,
                             None)
    assert rc == 1


def _attn(L, **kw):
    a = dict(dtype=m.BF16, q=A, k=A, v=A, pl=A, P_max=1024, mask=A, B=1, R=65, H=32, dh=128,
             scale=0.088, out=A, ws=WS, ws_bytes=1 << 30)
    a.update(kw)
    return L.medusa_tree_attention(a["dtype"], a["q"], a["k"], a["v"], a["pl"], a["P_max"],
                                   a["mask"], a["B"], a["R"], a["H"], a["dh"],
                                   ctypes.c_float(a["scale"]), a["out"], a["ws"], a["ws_bytes"],
                                   None)


@pytest.mark.parametrize("kw,code", [
    (dict(dh=96), 2), (dict(R=0), 1), (dict(R=257), 1), (dict(P_max=-1), 1), (dict(q=None), 1),
    (dict(scale=0.0), 1), (dict(out=MISALIGNED), 1), (dict(dtype=m.F32, P_max=16384), 2),
    (dict(ws_bytes=1000), 3)])
def test_attention_rejects(L, kw, code):
    before = L.medusa_launch_count()
    assert _attn(L, **kw) == code
    assert L.medusa_launch_count() == before


def _post(L, **kw):
    a = dict(dtype=m.BF16, logits=A, B=1, R=65, V=32000, K=5, mode=m.TYPICAL, eps=0.09, delta=0.3,
             T=1.0, ws=WS, ws_bytes=1 << 20)
    a.update(kw)
    f = ctypes.c_float
    return L.medusa_evaluate_posterior(a["dtype"], a["logits"], A, A, A, a["B"], a["R"], a["V"],
                                       a["K"], a["mode"], f(a["eps"]), f(a["delta"]), f(a["T"]), A, A,
                                       A, A, None, a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(V=32001), 1), (dict(dtype=m.F32, V=1002), 1), (dict(R=257), 1), (dict(K=9), 1),
    (dict(mode=2), 1), (dict(T=0.0), 1), (dict(eps=-1.0), 1), (dict(delta=0.0), 1),
    (dict(logits=MISALIGNED), 1), (dict(ws_bytes=64), 3)])
def test_posterior_rejects(L, kw, code):
    before = L.medusa_launch_count()
    assert _post(L, **kw) == code
    assert L.medusa_launch_count() == before


A2 = P(8192)         # a second fake address, for the no-alias rule


def _commit(L, **kw):
    a = dict(dtype=m.BF16, k=A, v=A, pl=A, path=A, al=A, B=1, K=5, R=65, H=32, dh=128, npl=A2,
             ws=WS, ws_bytes=256)
    a.update(kw)
    return L.medusa_commit_kv(a["dtype"], a["k"], a["v"], a["pl"], a["path"], a["al"], a["B"],
                              a["K"], a["R"], a["H"], a["dh"], a["npl"], a["ws"], a["ws_bytes"],
                              None)


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=5), 1), (dict(k=None), 1), (dict(v=None), 1), (dict(path=None), 1),
    (dict(al=None), 1), (dict(npl=None), 1), (dict(npl=A), 1), (dict(k=MISALIGNED), 1),
    (dict(B=0), 1), (dict(K=9), 1), (dict(K=-1), 1), (dict(R=0), 1), (dict(R=257), 1),
    (dict(H=0), 1), (dict(H=1, dh=7), 1), (dict(dtype=m.F32, H=1, dh=2), 1), (dict(ws=None), 3),
    (dict(ws_bytes=255), 3)])
def test_commit_rejects(L, kw, code):
    before = L.medusa_launch_count()
    assert _commit(L, **kw) == code
    assert L.medusa_launch_count() == before
    assert L.medusa_last_error().decode()


def _post_commit(L, **kw):
    a = dict(dtype=m.BF16, logits=A, B=1, R=65, V=32000, K=5, mode=m.GREEDY, k=A, v=A, pl=A, H=32,
             dh=128, npl=A2, ws=WS, ws_bytes=1 << 20)
    a.update(kw)
    f = ctypes.c_float
    return L.medusa_evaluate_posterior_commit(
        a["dtype"], a["logits"], A, A, A, a["B"], a["R"], a["V"], a["K"], a["mode"], f(0.09),
        f(0.3), f(1.0), A, A, A, A, None, a["k"], a["v"], a["pl"], a["H"], a["dh"], a["npl"],
        a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(V=32001), 1), (dict(K=9), 1), (dict(k=None), 1), (dict(pl=None), 1), (dict(npl=A), 1),
    (dict(H=1, dh=4), 1), (dict(v=MISALIGNED), 1), (dict(ws_bytes=64), 3)])
def test_posterior_commit_rejects(L, kw, code):
    before = L.medusa_launch_count()
    assert _post_commit(L, **kw) == code
    assert L.medusa_launch_count() == before


def test_workspace_sizes(L):
    hs = m.heads_workspace_size(1, 5, 4096, 32000, 4)
    assert hs >= 256 + 5 * 4096 * 4
    assert m.heads_workspace_size(8, 5, 4096, 32000, 4) > hs
    assert m.build_tree_workspace_size(1, 5, 4, 64) >= 256
    a1 = m.tree_attention_workspace_size(m.BF16, 1, 65, 32, 128, 1024)
    assert a1 > 65 * 32 * 128 * 4
    assert m.tree_attention_workspace_size(m.F32, 1, 15, 1, 64, 32) >= 256
    assert m.posterior_workspace_size(8, 65) >= 256 + 8 * 65 * 16
    assert L.medusa_heads_workspace_size(0, 5, 4096, 32000, 4) == 0


def test_device_status_helpers_reject_null(L):
    assert L.medusa_read_device_status(None, None, None) == 1
    assert L.medusa_clear_device_status(None, None) == 1


def test_binding_refuses_pageable_result_buffers():
    """The binding passes a posterior result as a CUDA tensor or pinned host
    memory only; an ordinary CPU tensor is refused before any call."""
    import torch
    with pytest.raises(ValueError):
        m._result_ptr(torch.zeros(3, dtype=torch.int32), "accept_len")
    assert m._result_ptr(None, "accept") is None


def test_attention_plan_tail_rule():
    """The attention's workspace follows its plan: one partial row (dh
    floats and an (m, l) pair) per (sequence, head, key range, tree row), so
    its size shows how many key ranges the plan took.  A 129-row tree at dh 128
    takes one 128-row tile when every CTA then runs at least 8 sub-chunks of
    64 keys (long prefixes), two tiles otherwise; 130 rows and dh 64 always
    take two.  Checked with the 152-SM plan the library uses without a
    device."""
    def ws(R, dh, P, ns):
        rows = 32 * ns * R
        a256 = lambda x: (x + 255) // 256 * 256
        return m.WS_HEADER + a256(rows * dh * 4) + a256(rows * 8)

    def ns_for(R, P, tiles):
        nsub = (P + R + 63) // 64
        per_head = max(1, 2 * 152 // (32 * tiles))
        cps = max(2, -(-nsub // per_head))
        return -(-nsub // cps), cps

    for P in (512, 2048, 4096, 8192):
        ns1, cps1 = ns_for(129, P, 1)
        ns2, _ = ns_for(129, P, 2)
        expect = ws(129, 128, P, ns1 if cps1 >= 8 else ns2)
        assert m.tree_attention_workspace_size(m.BF16, 1, 129, 32, 128, P) == expect, P
        assert m.tree_attention_workspace_size(m.BF16, 1, 129, 32, 64, P) == ws(129, 64, P, ns2), P
        assert m.tree_attention_workspace_size(m.BF16, 1, 130, 32, 128, P) == \
            ws(130, 128, P, ns_for(130, P, 2)[0]), P
    # the switch point: one tile from prefix 4096 on, two below
    assert ns_for(129, 2048, 1)[1] < 8 <= ns_for(129, 4096, 1)[1]


def test_step_desc_layout_matches_header(tmp_path):
    """The binding's mirror of medusa_step_desc has every field at the offset
    the C compiler gives it (gcc on include/medusa.h), and the same size."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    names = [f[0] for f in m._StepDesc._fields_]
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stddef.h>\n#include <stdio.h>\n#include "medusa.h"\nint main(void) {\n'
        + "".join(f'  printf("{n} %zu\\n", offsetof(medusa_step_desc, {n}));\n' for n in names)
        + '  printf("sizeof %zu\\n", sizeof(medusa_step_desc));\n'
        + '  printf("copy %zu\\n", sizeof(medusa_copy));\n  return 0;\n}\n')
    exe = tmp_path / "layout"
    subprocess.run([gcc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    got = dict(line.split() for line in subprocess.run(
        [str(exe)], check=True, capture_output=True, text=True).stdout.splitlines())
    for n in names:
        assert int(got[n]) == getattr(m._StepDesc, n).offset, n
    assert int(got["sizeof"]) == ctypes.sizeof(m._StepDesc)
    assert int(got["copy"]) == ctypes.sizeof(m._Copy)


def _step_desc(**kw):
    """A structurally valid descriptor with fake device addresses."""
    d = m._StepDesc()
    for name, typ in m._StepDesc._fields_:
        if typ is ctypes.c_void_p:
            setattr(d, name, 4096)
    s = (ctypes.c_int32 * 5)(4, 3, 2, 2, 1)
    d.s_host = ctypes.addressof(s)
    d.b1 = d.accept = d.new_prefix_len = None
    d.dtype, d.B, d.d, d.V, d.K, d.top_s, d.n = m.BF16, 1, 4096, 32000, 5, 4, 64
    d.P_max, d.H, d.dh, d.scale = 1024, 32, 128, 0.088
    d.mode, d.eps, d.delta, d.temperature = m.TYPICAL, 0.09, 0.3, 1.0
    d.ws_bytes = 1 << 24
    d.early = d.late = None
    for k, v in kw.items():
        setattr(d, k, v)
    return d, s


@pytest.mark.parametrize("kw,msg", [
    (dict(B=0), "B outside"), (dict(B=9), "B outside"), (dict(K=9), "K outside"),
    (dict(top_s=17), "top_s"), (dict(n=256), "n + 1"), (dict(n=0), "n + 1"),
    (dict(dtype=7), "dtype"), (dict(s_host=None), "s_host"), (dict(q=None), "required"),
    (dict(logits=None), "required"), (dict(ws=None), "required"),
    (dict(n_early=1), "early copy list"), (dict(n_late=65), "late copy count"),
    (dict(P_max=-1), "P_max"), (dict(flags=2), "unknown flags"),
])
def test_step_create_rejects_before_cuda(L, kw, msg):
    d, _s = _step_desc(**kw)
    ex = ctypes.c_void_p(1234)
    rc = L.medusa_step_create(ctypes.byref(d), ctypes.byref(ex))
    assert rc == 1, m.STATUS.get(rc)
    assert msg in L.medusa_last_error().decode()
    assert ex.value is None  # the output is cleared on failure


def test_step_create_rejects_bad_copies_and_s(L):
    bad = (m._Copy * 2)(m._Copy(4096, 8192, 64), m._Copy(4096, None, 64))
    d, _s = _step_desc(early=ctypes.addressof(bad), n_early=2)
    ex = ctypes.c_void_p()
    assert L.medusa_step_create(ctypes.byref(d), ctypes.byref(ex)) == 1
    assert "early copy 1" in L.medusa_last_error().decode()
    zero = (m._Copy * 1)(m._Copy(4096, 8192, 0))
    d, _s = _step_desc(late=ctypes.addressof(zero), n_late=1)
    assert L.medusa_step_create(ctypes.byref(d), ctypes.byref(ex)) == 1
    assert "late copy 0" in L.medusa_last_error().decode()
    s = (ctypes.c_int32 * 5)(4, 3, 5, 2, 1)  # s_k > top_s
    d, _ = _step_desc(s_host=ctypes.addressof(s))
    assert L.medusa_step_create(ctypes.byref(d), ctypes.byref(ex)) == 1
    assert "s_host[k]" in L.medusa_last_error().decode()
    assert L.medusa_step_create(None, ctypes.byref(ex)) == 1
    assert L.medusa_step_run(None, None, 1) == 1
    assert L.medusa_step_wait(None, None) == 1
    L.medusa_step_destroy(None)  # a no-op


def test_step_create_without_a_device_fails_cleanly(L):
    """A valid descriptor on a machine without a GPU fails at the side
    stream's creation with MEDUSA_ERR_CUDA and returns no executor."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    d, _s = _step_desc()
    ex = ctypes.c_void_p(1234)
    assert L.medusa_step_create(ctypes.byref(d), ctypes.byref(ex)) == 4
    assert ex.value is None
