"""Thin Python binding over libmedusa_gb300.so (ctypes).

Every step of the Medusa decoding step runs in the library's CUDA kernels;
this module only turns torch tensors into device pointers, sizes and the
current CUDA stream, allocates outputs and workspaces with torch, and raises
``MedusaError`` on a non-OK status.  There is no CPU or PyTorch fallback: if
the compiled library is missing, importing the calls fails loudly.

Public calls (same names as the C ABI in include/medusa.h):
    heads, heads_lm, heads_sample, heads_noalloc, build_tree, build_tree_static, tree_attention, evaluate_posterior,
    speculative_posterior, commit_kv, evaluate_posterior_commit
plus workspace-size queries, device-status helpers, launch_count,
``StepExecutor`` (medusa_step_create / medusa_step_run: the whole step, input
copies included, issued by one native call), and ``StepGraph``, which
captures a whole decoding step (copies and calls) into a CUDA graph once and
replays it per step.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmedusa_gb300.so")

F32, BF16 = 0, 1
GREEDY, TYPICAL = 0, 1
WS_HEADER = 256
STEP_GRAPH = 1
MAX_TOP_S = 16
MAX_TREE_ROWS = 256

STATUS = {0: "MEDUSA_OK", 1: "MEDUSA_ERR_INVALID_ARG", 2: "MEDUSA_ERR_UNSUPPORTED",
          3: "MEDUSA_ERR_WORKSPACE", 4: "MEDUSA_ERR_CUDA", 5: "MEDUSA_ERR_TIMEOUT",
          6: "MEDUSA_ERR_DEVICE_CHECK"}
DEVICE_STATUS = {0: "ok", 1: "bad token", 2: "bad parent", 3: "bad prefix", 4: "bad score",
                 5: "bad depth", 6: "timeout", 7: "bad path", 8: "bad cache",
                 9: "drain timeout"}

EXPORTS = ("medusa_status_string", "medusa_last_error", "medusa_launch_count",
           "medusa_wait_budget", "medusa_set_wait_budget",
           "medusa_read_device_status", "medusa_clear_device_status",
           "medusa_heads_workspace_size", "medusa_heads",
           "medusa_heads_lm_workspace_size", "medusa_heads_lm",
           "medusa_build_tree_workspace_size", "medusa_build_tree", "medusa_build_tree_static",
           "medusa_tree_attention_workspace_size", "medusa_tree_attention",
           "medusa_posterior_workspace_size", "medusa_evaluate_posterior",
           "medusa_evaluate_posterior_commit", "medusa_commit_kv", "medusa_heads_sample",
           "medusa_speculative_workspace_size", "medusa_speculative_posterior",
           "medusa_step_desc_size", "medusa_step_create", "medusa_step_run",
           "medusa_step_wait", "medusa_step_destroy")


class _Copy(ctypes.Structure):
    """medusa_copy"""
    _fields_ = [("dst", ctypes.c_void_p), ("src", ctypes.c_void_p), ("bytes", ctypes.c_size_t)]


class _StepDesc(ctypes.Structure):
    """medusa_step_desc, field for field (checked against medusa_step_desc_size)."""
    _P, _I, _F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
    _fields_ = [("early", _P), ("n_early", _I), ("late", _P), ("n_late", _I), ("dtype", _I),
                ("h", _P), ("W1", _P), ("b1", _P), ("W2", _P),
                ("B", _I), ("d", _I), ("V", _I), ("K", _I), ("top_s", _I),
                ("topk_ids", _P), ("topk_logp", _P),
                ("root", _P), ("s_host", _P), ("n", _I), ("prefix_len", _P),
                ("tokens", _P), ("parent", _P), ("depth", _P), ("pos_id", _P), ("anc_mask", _P),
                ("paths", _P), ("n_leaf", _P),
                ("q", _P), ("k_cache", _P), ("v_cache", _P), ("P_max", _I), ("H", _I), ("dh", _I),
                ("scale", _F), ("attn_out", _P),
                ("logits", _P), ("mode", _I), ("eps", _F), ("delta", _F), ("temperature", _F),
                ("accept_len", _P), ("path", _P), ("path_tokens", _P), ("next_token", _P),
                ("accept", _P), ("new_prefix_len", _P), ("ws", _P), ("ws_bytes", ctypes.c_size_t),
                ("flags", _I)]


class MedusaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """Load libmedusa_gb300.so (built by ``build.build()``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc, sm_103a)")
    L = ctypes.CDLL(LIB_PATH)
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    U64 = ctypes.c_uint64
    sig = {
        "medusa_status_string": ([I], ctypes.c_char_p),
        "medusa_last_error": ([], ctypes.c_char_p),
        "medusa_launch_count": ([], ctypes.c_uint64),
        "medusa_wait_budget": ([], ctypes.c_uint32),
        "medusa_set_wait_budget": ([ctypes.c_uint32], None),
        "medusa_read_device_status": ([P, P, P], I),
        "medusa_clear_device_status": ([P, P], I),
        "medusa_heads_workspace_size": ([I, I, I, I, I], S),
        "medusa_heads": ([I, P, P, P, P, I, I, I, I, I, P, P, P, S, P], I),
        "medusa_heads_lm_workspace_size": ([I, I, I, I, I], S),
        "medusa_heads_lm": ([I, P, P, P, P, P, I, I, I, I, I, P, P, P, P, P, S, P], I),
        "medusa_build_tree_workspace_size": ([I, I, I, I], S),
        "medusa_build_tree": ([P, P, P, I, I, P, I, I, P, P, P, P, P, P, P, P, P, S, P], I),
        "medusa_build_tree_static": ([P, P, P, I, I, P, I, I, P, P, P, P, P, P, P, P, P, S, P], I),
        "medusa_tree_attention_workspace_size": ([I, I, I, I, I, I], S),
        "medusa_tree_attention": ([I, P, P, P, P, I, P, I, I, I, I, F, P, P, S, P], I),
        "medusa_posterior_workspace_size": ([I, I], S),
        "medusa_evaluate_posterior": ([I, P, P, P, P, I, I, I, I, I, F, F, F, P, P, P, P, P, P, S, P], I),
        "medusa_evaluate_posterior_commit": ([I, P, P, P, P, I, I, I, I, I, F, F, F, P, P, P, P, P,
                                              P, P, P, I, I, P, P, S, P], I),
        "medusa_commit_kv": ([I, P, P, P, P, P, I, I, I, I, I, P, P, S, P], I),
        "medusa_heads_sample": ([I, P, P, P, P, I, I, I, I, F, U64, U64, P, P, P, S, P], I),
        "medusa_speculative_workspace_size": ([I, I], S),
        "medusa_speculative_posterior": ([I, P, P, P, I, I, I, F, U64, U64, P, P, P, P, P, S, P],
                                         I),
        "medusa_step_desc_size": ([], S),
        "medusa_step_create": ([ctypes.POINTER(_StepDesc), ctypes.POINTER(P)], I),
        "medusa_step_run": ([P, P, I], I),
        "medusa_step_wait": ([P, P], I),
        "medusa_step_destroy": ([P], None),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


def _check(rc: int):
    if rc != 0:
        msg = lib().medusa_last_error().decode(errors="replace")
        raise MedusaError(rc, msg)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def _need(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _result_ptr(t: Optional[torch.Tensor], name: str):
    """Pointer of a posterior output: a CUDA tensor, or a pinned CPU tensor
    that the kernel writes directly (no copy back)."""
    if t is None:
        return None
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return _ptr(t)


def launch_count() -> int:
    return int(lib().medusa_launch_count())


def wait_budget() -> int:
    """Poll limit of the bounded device waits (fault injection: 0 makes
    them time out at once and set the "timeout" device status)."""
    return int(lib().medusa_wait_budget())


def set_wait_budget(polls: int) -> None:
    lib().medusa_set_wait_budget(int(polls))


def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    """Zeroed device workspace (the status word must start at 0)."""
    n = (max(int(nbytes), WS_HEADER) + 255) // 256 * 256
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def read_device_status(ws: torch.Tensor, stream=None) -> int:
    out = ctypes.c_int32(0)
    _check(lib().medusa_read_device_status(_ptr(ws), ctypes.byref(out), _stream(stream)))
    return int(out.value)


def clear_device_status(ws: torch.Tensor, stream=None):
    _check(lib().medusa_clear_device_status(_ptr(ws), _stream(stream)))


# ------------------------------------------------------------------ heads ---

def heads_workspace_size(B: int, K: int, d: int, V: int, top_s: int) -> int:
    return int(lib().medusa_heads_workspace_size(B, K, d, V, top_s))


def heads(h, W1, b1, W2, top_s: int, ws=None, out=None, stream=None):
    """Top-s token ids [B,K,s] (int32) and log-probs (fp32) of the K heads."""
    for t, n in ((h, "h"), (W1, "W1"), (W2, "W2")):
        _need(t, n)
    if b1 is not None:
        _need(b1, "b1")
    B, d = h.shape
    K, V = W2.shape[0], W2.shape[1]
    if ws is None:
        ws = new_workspace(heads_workspace_size(B, K, d, V, top_s), h.device)
    if out is None:
        out = (torch.empty((B, K, top_s), dtype=torch.int32, device=h.device),
               torch.empty((B, K, top_s), dtype=torch.float32, device=h.device))
    ids, logp = out
    _check(lib().medusa_heads(_dtype(h), _ptr(h), _ptr(W1), _ptr(b1), _ptr(W2), B, d, V, K, top_s,
                              _ptr(ids), _ptr(logp), _ptr(ws), ws.numel(), _stream(stream)))
    return ids, logp


def heads_lm_workspace_size(B: int, K: int, d: int, V: int, top_s: int) -> int:
    return int(lib().medusa_heads_lm_workspace_size(B, K, d, V, top_s))


def heads_lm(h, W_lm, W1, b1, W2, top_s: int, ws=None, out=None, stream=None):
    """The LM head and the Medusa heads in one weight pass.  Returns
    (root int32 [B], root_logp fp32 [B], topk_ids int32 [B,K,top_s],
    topk_logp fp32 [B,K,top_s])."""
    for t, name in ((h, "h"), (W_lm, "W_lm"), (W1, "W1"), (W2, "W2")):
        _need(t, name)
    B, d = h.shape
    K, V = W2.shape[0], W2.shape[1]
    dev = h.device
    if ws is None:
        ws = new_workspace(heads_lm_workspace_size(B, K, d, V, top_s), dev)
    if out is None:
        out = (torch.empty((B,), dtype=torch.int32, device=dev),
               torch.empty((B,), dtype=torch.float32, device=dev),
               torch.empty((B, K, top_s), dtype=torch.int32, device=dev),
               torch.empty((B, K, top_s), dtype=torch.float32, device=dev))
    root, root_logp, ids, logp = out
    _check(lib().medusa_heads_lm(_dtype(h), _ptr(h), _ptr(W_lm), _ptr(W1), _ptr(b1), _ptr(W2), B, d,
                                 V, K, int(top_s), _ptr(root), _ptr(root_logp), _ptr(ids),
                                 _ptr(logp), _ptr(ws), ws.numel(), _stream(stream)))
    return root, root_logp, ids, logp


def heads_noalloc(h, W1, b1, W2, top_s: int, out=None, stream=None):
    """medusa_heads with the library's own 4 MiB device scratch: for callers
    that cannot allocate device memory when they run the heads.  Calls that
    overlap on the GPU share the scratch and must be serialised."""
    for t, n in ((h, "h"), (W1, "W1"), (W2, "W2")):
        _need(t, n)
    fn = lib().medusa_heads_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [I, P, P, P, P, I, I, I, I, I, P, P, P]
    fn.restype = I
    B, d = h.shape
    K, V = W2.shape[0], W2.shape[1]
    if out is None:
        out = (torch.empty((B, K, top_s), dtype=torch.int32, device=h.device),
               torch.empty((B, K, top_s), dtype=torch.float32, device=h.device))
    ids, logp = out
    _check(fn(_dtype(h), _ptr(h), _ptr(W1), _ptr(b1), _ptr(W2), B, d, V, K, top_s, _ptr(ids),
              _ptr(logp), _stream(stream)))
    return ids, logp


# ------------------------------------------------------------------- tree ---

@dataclass
class Tree:
    tokens: torch.Tensor
    parent: torch.Tensor
    depth: torch.Tensor
    pos_id: torch.Tensor
    anc_mask: torch.Tensor
    paths: torch.Tensor
    n_leaf: torch.Tensor

    @staticmethod
    def empty(B: int, n: int, K: int, device) -> "Tree":
        R = n + 1
        W = (R + 63) // 64
        i32 = dict(dtype=torch.int32, device=device)
        return Tree(torch.empty((B, R), **i32), torch.empty((B, R), **i32),
                    torch.empty((B, R), **i32), torch.empty((B, R), **i32),
                    torch.empty((B, R, W), dtype=torch.int64, device=device),
                    torch.empty((B, n, K + 1), **i32), torch.empty((B,), **i32))


def build_tree_workspace_size(B: int, K: int, top_s: int, n: int) -> int:
    return int(lib().medusa_build_tree_workspace_size(B, K, top_s, n))


def build_tree(root, topk_ids, topk_logp, s: Sequence[int], n: int, prefix_len=None, ws=None,
               out: Optional[Tree] = None, stream=None) -> Tree:
    """Budgeted candidate tree (canonical order) from the heads' top-s lists."""
    for t, nm in ((root, "root"), (topk_ids, "topk_ids"), (topk_logp, "topk_logp")):
        _need(t, nm)
    B, K, S = topk_ids.shape
    s_host = (ctypes.c_int32 * K)(*[int(x) for x in s])
    if ws is None:
        ws = new_workspace(build_tree_workspace_size(B, K, S, n), root.device)
    t = out or Tree.empty(B, n, K, root.device)
    _check(lib().medusa_build_tree(_ptr(root), _ptr(topk_ids), _ptr(topk_logp), B, K, s_host, S, n,
                                   _ptr(prefix_len), _ptr(t.tokens), _ptr(t.parent), _ptr(t.depth),
                                   _ptr(t.pos_id), _ptr(t.anc_mask), _ptr(t.paths), _ptr(t.n_leaf),
                                   _ptr(ws), ws.numel(), _stream(stream)))
    return t


def build_tree_static(root, topk_ids, log_a, s: Sequence[int], n: int, prefix_len=None, ws=None,
                      out: Optional[Tree] = None, stream=None) -> Tree:
    """Candidate tree whose shape comes from a calibrated table log_a [K, top_s]
    (shared by every sequence); tokens from each sequence's top-s lists."""
    for t, nm in ((root, "root"), (topk_ids, "topk_ids"), (log_a, "log_a")):
        _need(t, nm)
    B, K, S = topk_ids.shape
    if tuple(log_a.shape) != (K, S) or log_a.dtype != torch.float32:
        raise ValueError(f"log_a must be float32 [{K}, {S}], got {log_a.dtype} {tuple(log_a.shape)}")
    s_host = (ctypes.c_int32 * K)(*[int(x) for x in s])
    if ws is None:
        ws = new_workspace(build_tree_workspace_size(B, K, S, n), root.device)
    t = out or Tree.empty(B, n, K, root.device)
    _check(lib().medusa_build_tree_static(_ptr(root), _ptr(topk_ids), _ptr(log_a), B, K, s_host, S,
                                          n, _ptr(prefix_len), _ptr(t.tokens), _ptr(t.parent),
                                          _ptr(t.depth), _ptr(t.pos_id), _ptr(t.anc_mask),
                                          _ptr(t.paths), _ptr(t.n_leaf), _ptr(ws), ws.numel(),
                                          _stream(stream)))
    return t


# -------------------------------------------------------------- attention ---

def tree_attention_workspace_size(dtype: int, B: int, R: int, H: int, dh: int, P_max: int) -> int:
    return int(lib().medusa_tree_attention_workspace_size(dtype, B, R, H, dh, P_max))


def cache_pointers(caches: Sequence[torch.Tensor], device) -> torch.Tensor:
    """Device array of the per-sequence cache base pointers."""
    for c in caches:
        _need(c, "cache")
    return torch.tensor([c.data_ptr() for c in caches], dtype=torch.int64, device=device)


def tree_attention(q, k_ptrs, v_ptrs, prefix_len, P_max: int, anc_mask, scale=None, out=None,
                   ws=None, stream=None):
    """Tree-masked attention.  q [B,R,H,dh]; k_ptrs/v_ptrs: int64 device arrays of
    per-sequence cache pointers (see cache_pointers); prefix_len int32 [B]."""
    _need(q, "q")
    B, R, H, dh = q.shape
    dt = _dtype(q)
    if scale is None:
        scale = 1.0 / math.sqrt(dh)
    if ws is None:
        ws = new_workspace(tree_attention_workspace_size(dt, B, R, H, dh, P_max), q.device)
    if out is None:
        out = torch.empty_like(q)
    _check(lib().medusa_tree_attention(dt, _ptr(q), _ptr(k_ptrs), _ptr(v_ptrs), _ptr(prefix_len),
                                       int(P_max), _ptr(anc_mask), B, R, H, dh, float(scale),
                                       _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))
    return out


# -------------------------------------------------------------- posterior ---

@dataclass
class Posterior:
    accept_len: torch.Tensor
    path: torch.Tensor
    path_tokens: torch.Tensor
    next_token: torch.Tensor
    accept: Optional[torch.Tensor]

    @staticmethod
    def empty(B: int, R: int, K: int, device, with_accept: bool = True) -> "Posterior":
        i32 = dict(dtype=torch.int32, device=device)
        return Posterior(torch.empty((B,), **i32), torch.empty((B, K + 1), **i32),
                         torch.empty((B, K + 1), **i32), torch.empty((B,), **i32),
                         torch.empty((B, R), **i32) if with_accept else None)

    @staticmethod
    def pinned(B: int, R: int, K: int, with_accept: bool = True) -> "Posterior":
        """Results in page-locked host memory: the posterior kernel writes
        them there directly; read them after the stream has synchronised."""
        i32 = dict(dtype=torch.int32)
        mk = lambda shape: torch.empty(shape, **i32).pin_memory()
        return Posterior(mk((B,)), mk((B, K + 1)), mk((B, K + 1)), mk((B,)),
                         mk((B, R)) if with_accept else None)


def posterior_workspace_size(B: int, R: int) -> int:
    return int(lib().medusa_posterior_workspace_size(B, R))


def evaluate_posterior(logits, tokens, parent, depth, K: int, mode: int = GREEDY, eps=0.09,
                       delta=0.3, temperature=1.0, ws=None, out: Optional[Posterior] = None,
                       with_accept: bool = True, stream=None) -> Posterior:
    """Acceptance + longest accepted path.  logits [B,R,V] bf16 or fp32."""
    _need(logits, "logits")
    B, R, V = logits.shape
    if ws is None:
        ws = new_workspace(posterior_workspace_size(B, R), logits.device)
    o = out or Posterior.empty(B, R, K, logits.device, with_accept)
    _check(lib().medusa_evaluate_posterior(_dtype(logits), _ptr(logits), _ptr(tokens), _ptr(parent),
                                           _ptr(depth), B, R, V, K, int(mode), float(eps),
                                           float(delta), float(temperature),
                                           _result_ptr(o.accept_len, "accept_len"),
                                           _result_ptr(o.path, "path"),
                                           _result_ptr(o.path_tokens, "path_tokens"),
                                           _result_ptr(o.next_token, "next_token"),
                                           _result_ptr(o.accept, "accept"), _ptr(ws), ws.numel(),
                                           _stream(stream)))
    return o


def evaluate_posterior_commit(logits, tokens, parent, depth, K: int, k_ptrs, v_ptrs, prefix_len,
                              H: int, dh: int, new_prefix_len=None, mode: int = GREEDY, eps=0.09,
                              delta=0.3, temperature=1.0, ws=None,
                              out: Optional[Posterior] = None, with_accept: bool = True,
                              stream=None):
    """evaluate_posterior, then the commit of commit_kv in the same kernel.
    The caches hold logits.dtype elements.  Returns (Posterior, new_prefix_len)."""
    _need(logits, "logits")
    B, R, V = logits.shape
    if ws is None:
        ws = new_workspace(posterior_workspace_size(B, R), logits.device)
    o = out or Posterior.empty(B, R, K, logits.device, with_accept)
    if new_prefix_len is None:
        new_prefix_len = torch.empty((B,), dtype=torch.int32, device=logits.device)
    _check(lib().medusa_evaluate_posterior_commit(
        _dtype(logits), _ptr(logits), _ptr(tokens), _ptr(parent), _ptr(depth), B, R, V, K,
        int(mode), float(eps), float(delta), float(temperature),
        _result_ptr(o.accept_len, "accept_len"), _result_ptr(o.path, "path"),
        _result_ptr(o.path_tokens, "path_tokens"), _result_ptr(o.next_token, "next_token"),
        _result_ptr(o.accept, "accept"), _ptr(k_ptrs), _ptr(v_ptrs),
        _ptr(prefix_len), int(H), int(dh), _ptr(new_prefix_len), _ptr(ws), ws.numel(),
        _stream(stream)))
    return o, new_prefix_len


# ----------------------------------------------------------------- commit ---

def commit_kv(dtype: int, k_ptrs, v_ptrs, prefix_len, path, accept_len, R: int, H: int, dh: int,
              new_prefix_len=None, ws=None, stream=None):
    """Move the accepted path's K/V rows into slots P_b..P_b+L (in place in the
    caches behind k_ptrs/v_ptrs); return new_prefix_len = P_b + L + 1."""
    B, K1 = path.shape
    dev = path.device
    if ws is None:
        ws = new_workspace(WS_HEADER, dev)
    if new_prefix_len is None:
        new_prefix_len = torch.empty((B,), dtype=torch.int32, device=dev)
    _check(lib().medusa_commit_kv(int(dtype), _ptr(k_ptrs), _ptr(v_ptrs), _ptr(prefix_len),
                                  _ptr(path), _ptr(accept_len), B, K1 - 1, int(R), int(H), int(dh),
                                  _ptr(new_prefix_len), _ptr(ws), ws.numel(), _stream(stream)))
    return new_prefix_len


# --------------------------------------------------------------- sampling ---

def heads_sample(h, W1, b1, W2, temperature: float, seed: int, step: int, ws=None, out=None,
                 stream=None):
    """One draft per head sampled from softmax(logits / T) (Gumbel-max with the
    library's Philox streams).  Returns (drafts int32 [B,K], draft_logits fp32
    [B,K,V])."""
    for t, name in ((h, "h"), (W1, "W1"), (W2, "W2")):
        _need(t, name)
    B, d = h.shape
    K, V = W2.shape[0], W2.shape[1]
    dev = h.device
    if ws is None:
        ws = new_workspace(heads_workspace_size(B, K, d, V, 1), dev)
    if out is None:
        out = (torch.empty((B, K), dtype=torch.int32, device=dev),
               torch.empty((B, K, V), dtype=torch.float32, device=dev))
    drafts, dl = out
    _check(lib().medusa_heads_sample(_dtype(h), _ptr(h), _ptr(W1), _ptr(b1), _ptr(W2), B, d, V, K,
                                     float(temperature), int(seed), int(step), _ptr(drafts),
                                     _ptr(dl), _ptr(ws), ws.numel(), _stream(stream)))
    return drafts, dl


@dataclass
class Speculative:
    accept_len: torch.Tensor
    path_tokens: torch.Tensor
    next_token: torch.Tensor
    accept: Optional[torch.Tensor]


def speculative_workspace_size(B: int, K: int) -> int:
    return int(lib().medusa_speculative_workspace_size(B, K))


def speculative_posterior(logits, tokens, draft_logits, temperature: float, seed: int, step: int,
                          ws=None, out: Optional[Speculative] = None, with_accept: bool = True,
                          stream=None) -> Speculative:
    """Exact speculative sampling on a chain: logits [B,K+1,V], tokens [B,K+1]
    (root then drafts), draft_logits fp32 [B,K,V]."""
    _need(logits, "logits")
    B, R, V = logits.shape
    K = R - 1
    dev = logits.device
    if ws is None:
        ws = new_workspace(speculative_workspace_size(B, K), dev)
    if out is None:
        i32 = dict(dtype=torch.int32, device=dev)
        out = Speculative(torch.empty((B,), **i32), torch.empty((B, K + 1), **i32),
                          torch.empty((B,), **i32),
                          torch.empty((B, K), **i32) if with_accept else None)
    _check(lib().medusa_speculative_posterior(
        _dtype(logits), _ptr(logits), _ptr(tokens), _ptr(draft_logits), B, V, K,
        float(temperature), int(seed), int(step), _ptr(out.accept_len), _ptr(out.path_tokens),
        _ptr(out.next_token), _ptr(out.accept), _ptr(ws), ws.numel(), _stream(stream)))
    return out


# ------------------------------------------------------------- step graph ---

class StepGraph:
    """A decoding step captured once into a CUDA graph and replayed.

    ``fn`` issues the step on the current stream: copies of the step's
    inputs from pinned host buffers, the library calls (heads, tree,
    attention, posterior, ...), and the results' way back to the host: copies
    into pinned buffers, or a posterior whose outputs are pinned host memory
    (``Posterior.pinned``), which its kernel writes directly.  Every buffer it touches must stay allocated and at the
    same address while the graph lives; new inputs are written into the same
    pinned host buffers before each ``replay``.  The launches keep their
    programmatic-dependent-launch edges inside the graph.
    """

    def __init__(self, fn, warmup: int = 2):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(warmup):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            fn()
        torch.cuda.synchronize()

    def replay(self):
        self.graph.replay()


# ---------------------------------------------------------- step executor ---

def _copy_pair(dst: torch.Tensor, src: torch.Tensor, name: str):
    _need(dst, f"{name} destination")
    if not (src.is_cuda or src.is_pinned()):
        raise ValueError(f"{name} source must be pinned host memory or a CUDA tensor")
    if not src.is_contiguous():
        raise ValueError(f"{name} source must be contiguous")
    nb = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != nb or nb == 0:
        raise ValueError(f"{name}: source and destination sizes differ or are empty")
    return _Copy(dst.data_ptr(), src.data_ptr(), nb)


class StepExecutor:
    """One decoding step issued by one native call (medusa_step_run).

    The executor holds the step's buffers (the descriptor of
    medusa_step_create): ``early`` and ``late`` are lists of (device
    destination, pinned-host or device source) tensor pairs copied at the
    start of every run -- early ones before the heads on the caller's stream,
    late ones on the executor's side stream during the heads pass.  Then
    heads, tree, attention and posterior (with the fused commit when
    ``new_prefix_len`` is given) run as the separate calls do.  Every tensor
    must keep its address while the executor lives; write new inputs into
    the same host buffers before each ``run``.  With ``graph=True`` the
    sequence is captured once at construction as a CUDA graph and each run
    is one graph launch.
    """

    def __init__(self, *, h, W1, b1, W2, top_s: int, topk: tuple, root, s: Sequence[int], n: int,
                 prefix_len, tree: "Tree", q, k_ptrs, v_ptrs, P_max: int, attn_out, logits,
                 post: "Posterior", K: int, mode: int = GREEDY, eps=0.09, delta=0.3,
                 temperature=1.0, ws=None, early=(), late=(), new_prefix_len=None, scale=None,
                 graph: bool = False):
        L = lib()
        if ctypes.sizeof(_StepDesc) != L.medusa_step_desc_size():
            raise MedusaError(1, "medusa_step_desc layout differs from the binding's")
        for t, nm in ((h, "h"), (W1, "W1"), (W2, "W2"), (root, "root"), (prefix_len, "prefix_len"),
                      (q, "q"), (attn_out, "attn_out"), (logits, "logits"), (k_ptrs, "k_ptrs"),
                      (v_ptrs, "v_ptrs")):
            _need(t, nm)
        B, d = h.shape
        V = W2.shape[1]
        H, dh = q.shape[2], q.shape[3]
        ids, logp = topk
        if ws is None:
            R = n + 1
            need = max(heads_workspace_size(B, K, d, V, top_s),
                       build_tree_workspace_size(B, K, top_s, n),
                       tree_attention_workspace_size(_dtype(q), B, R, H, dh, P_max),
                       posterior_workspace_size(B, R))
            ws = new_workspace(need, h.device)
        self._early = (_Copy * max(1, len(early)))(
            *[_copy_pair(a, b, f"early[{i}]") for i, (a, b) in enumerate(early)])
        self._late = (_Copy * max(1, len(late)))(
            *[_copy_pair(a, b, f"late[{i}]") for i, (a, b) in enumerate(late)])
        self._s = (ctypes.c_int32 * K)(*[int(x) for x in s])
        pv = lambda t: None if t is None else t.data_ptr()
        res = lambda t, nm: None if t is None else _result_ptr(t, nm).value
        desc = _StepDesc(
            early=ctypes.addressof(self._early), n_early=len(early),
            late=ctypes.addressof(self._late), n_late=len(late), dtype=_dtype(h),
            h=pv(h), W1=pv(W1), b1=pv(b1), W2=pv(W2), B=B, d=d, V=V, K=K, top_s=int(top_s),
            topk_ids=pv(ids), topk_logp=pv(logp), root=pv(root),
            s_host=ctypes.addressof(self._s), n=int(n), prefix_len=pv(prefix_len),
            tokens=pv(tree.tokens), parent=pv(tree.parent), depth=pv(tree.depth),
            pos_id=pv(tree.pos_id), anc_mask=pv(tree.anc_mask), paths=pv(tree.paths),
            n_leaf=pv(tree.n_leaf), q=pv(q), k_cache=pv(k_ptrs), v_cache=pv(v_ptrs),
            P_max=int(P_max), H=H, dh=dh,
            scale=float(1.0 / math.sqrt(dh) if scale is None else scale), attn_out=pv(attn_out),
            logits=pv(logits), mode=int(mode), eps=float(eps), delta=float(delta),
            temperature=float(temperature),
            accept_len=res(post.accept_len, "accept_len"), path=res(post.path, "path"),
            path_tokens=res(post.path_tokens, "path_tokens"),
            next_token=res(post.next_token, "next_token"), accept=res(post.accept, "accept"),
            new_prefix_len=pv(new_prefix_len), ws=pv(ws), ws_bytes=ws.numel(),
            flags=STEP_GRAPH if graph else 0)
        # every buffer the descriptor names stays referenced while the executor lives
        self._keep = (h, W1, b1, W2, ids, logp, root, prefix_len, tree, q, k_ptrs, v_ptrs,
                      attn_out, logits, post, new_prefix_len, ws, tuple(early), tuple(late))
        self.ws = ws
        handle = ctypes.c_void_p()
        _check(L.medusa_step_create(ctypes.byref(desc), ctypes.byref(handle)))
        self._handle = handle
        self._h = handle.value  # plain integers keep the per-step call short
        self._run = L.medusa_step_run

    def run(self, stream=None, synchronize: bool = True):
        """Issue one step on ``stream`` (the current stream by default); with
        ``synchronize`` wait for it, so results in pinned memory are ready."""
        if self._handle is None:
            raise MedusaError(1, "StepExecutor is closed")
        s = (torch.cuda.current_stream() if stream is None else stream).cuda_stream
        rc = self._run(self._h, s, 1 if synchronize else 0)
        if rc:
            _check(rc)

    def wait(self, stream=None):
        """Wait for every step issued so far (the wait of ``run``)."""
        if self._handle is None:
            raise MedusaError(1, "StepExecutor is closed")
        s = (torch.cuda.current_stream() if stream is None else stream).cuda_stream
        _check(lib().medusa_step_wait(self._h, s))

    def close(self):
        if getattr(self, "_handle", None) is not None:
            lib().medusa_step_destroy(self._handle)
            self._handle = None
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
