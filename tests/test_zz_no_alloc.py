"""medusa_heads_noalloc: the Medusa heads with the library's own static device
scratch, for callers that cannot allocate device memory when they run the
heads (a serving runtime that gave all free HBM to its KV-cache pool, or a
decode loop that cannot pay for cudaMalloc's device-wide synchronisation).

The GPU test calls the entry point through the C ABI twice in a row, with
different inputs, and checks each result against medusa_heads (caller
workspace) on the same inputs: identical token ids, log-probs within the
parity tolerance (max-abs 1e-2, relative 2e-2).  This file is collected last
on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
import medusa_speculative_decoding_02_gb300 as m
from medusa_speculative_decoding_02_gb300 import build as mbuild

ATOL, RTOL = 1e-2, 2e-2


def _sig(L):
    fn = L.medusa_heads_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [I, P, P, P, P, I, I, I, I, I, P, P, P]
    fn.restype = I
    return fn


def _T(a, dev):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(a).to(dev)


@pytest.mark.gpu
@pytest.mark.parametrize("cfg_fn", [synth.tiny, synth.v7b], ids=["tiny", "v7b"])
def test_noalloc_matches_workspace_heads_twice(cfg_fn):
    mbuild.build()
    assert torch.cuda.is_available()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    cfg = cfg_fn()
    fn = _sig(m.lib())
    hi = synth.heads_inputs(cfg)
    W1, b1, W2 = _T(hi.W1, dev), _T(hi.b1, dev), _T(hi.W2, dev)
    dt = m.BF16 if cfg.dtype == "bf16" else m.F32
    S = cfg.top_s
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    for call in range(2):
        h = _T(synth.heads_inputs(cfg, rep=call).h, dev)
        ref_ids, ref_logp = m.heads(h, W1, b1, W2, S)
        ids = torch.full((cfg.B, cfg.K, S), -7, dtype=torch.int32, device=dev)
        logp = torch.full((cfg.B, cfg.K, S), float("nan"), dtype=torch.float32, device=dev)
        rc = fn(dt, h.data_ptr(), W1.data_ptr(), b1.data_ptr(), W2.data_ptr(), cfg.B, cfg.d, cfg.V,
                cfg.K, S, ids.data_ptr(), logp.data_ptr(), stream)
        assert rc == 0, m.lib().medusa_last_error()
        torch.cuda.synchronize(dev)
        assert torch.equal(ids, ref_ids), f"call {call}: ids differ"
        err = (logp - ref_logp).abs()
        assert bool(torch.all(err <= ATOL + RTOL * ref_logp.abs())), f"call {call}: logp differ"


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """B=8, K=8, d=4096, top-16 needs ~10 MB of scratch, more than the 4 MiB
    the library holds: rejected before any launch, with a message."""
    mbuild.build()
    L = m.lib()
    fn = _sig(L)
    assert m.heads_workspace_size(8, 8, 4096, 32000, 16) > (4 << 20)
    A = ctypes.c_void_p(4096)
    before = L.medusa_launch_count()
    rc = fn(m.BF16, A, A, None, A, 8, 4096, 32000, 8, 16, A, A, None)
    assert rc == 2
    assert L.medusa_launch_count() == before
    assert b"static scratch" in L.medusa_last_error()
