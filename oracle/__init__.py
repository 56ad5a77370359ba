"""Float64 CPU oracle for one Medusa decoding step -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never loads it and
has no fallback to it.  The arithmetic lives in ``oracle.c`` (plain loops in
IEEE double, compiled with ``-ffp-contract=off``); this module only compiles
it and marshals numpy arrays through ctypes.

bf16 arrays travel as ``uint16`` bit patterns, float32 arrays as ``float32``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_LIB_OMP = os.path.join(_HERE, "liboracle_omp.so")
_lock = threading.Lock()
_libs = {}
_parallel = False

F32, BF16 = 0, 1
GREEDY, TYPICAL = 0, 1

_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-Wall",
           "-Wno-unknown-pragmas", "-shared", "-fPIC"]


def _compile(out: str, extra, force: bool) -> None:
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(_SRC):
        tmp = out + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", *_CFLAGS, *extra, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, out)


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (plain gcc, no BLAS), and
    into liboracle_omp.so with OpenMP when the compiler supports it."""
    _compile(_LIB, [], force)
    try:
        _compile(_LIB_OMP, ["-fopenmp"], force)
    except (subprocess.CalledProcessError, OSError):
        pass  # parallel_available() reports False
    return _LIB


def parallel_available() -> bool:
    """True if the OpenMP build of the oracle exists."""
    return os.path.exists(_LIB_OMP)


def set_parallel(on: bool) -> None:
    """Route later calls to the OpenMP build (all host cores) or back to the
    serial build.  The benchmark's all-core CPU baseline turns this on, and so
    do the parity tests' full-size attention checks, which would otherwise
    take minutes; every other test uses the serial build.  Both builds give
    the same bits (tests/test_oracle_parallel.py)."""
    global _parallel
    if on and not parallel_available():
        raise RuntimeError("the OpenMP build of the oracle is not available")
    _parallel = bool(on)


def threads() -> int:
    """Threads the current build's parallel loops use (1 for the serial build)."""
    return int(_load().oracle_threads())


def _load():
    path = _LIB_OMP if _parallel else _LIB
    with _lock:
        if path not in _libs:
            build()
            lib = ctypes.CDLL(path)
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            lib.oracle_heads.argtypes = [I, P, P, P, P, I, I, I, I, I, P, P, P, P]
            lib.oracle_heads.restype = I
            lib.oracle_lm_head.argtypes = [I, P, P, I, I, I, I, P, P, P, P]
            lib.oracle_lm_head.restype = I
            lib.oracle_build_tree.argtypes = [P, P, P, I, I, P, I, I, P, P, P, P, P, P, P, P, P]
            lib.oracle_build_tree.restype = I
            lib.oracle_tree_attention.argtypes = [I, P, P, P, P, P, I, I, I, I, D, P]
            lib.oracle_tree_attention.restype = I
            lib.oracle_softmax_entropy.argtypes = [P, I, D]
            lib.oracle_softmax_entropy.restype = D
            lib.oracle_posterior.argtypes = [I, P, P, P, P, I, I, I, I, I, D, D, D, P, P, P, P, P, P, P]
            lib.oracle_posterior.restype = I
            U64 = ctypes.c_uint64
            lib.oracle_philox4x64.argtypes = [P, P, P]
            lib.oracle_philox4x64.restype = None
            lib.oracle_uniform.argtypes = [U64, U64, I, I, I, I]
            lib.oracle_uniform.restype = D
            lib.oracle_draft_sample.argtypes = [I, P, P, P, P, I, I, I, I, D, U64, U64, P, P, P]
            lib.oracle_draft_sample.restype = I
            lib.oracle_speculative_posterior.argtypes = [I, P, P, P, I, I, I, D, U64, U64, P, P,
                                                         P, P, P, P, P, P, P]
            lib.oracle_speculative_posterior.restype = I
            lib.oracle_commit_kv.argtypes = [P, P, P, P, P, I, I, ctypes.c_size_t, P]
            lib.oracle_commit_kv.restype = I
            lib.oracle_threads.argtypes = []
            lib.oracle_threads.restype = I
            _libs[path] = lib
    return _libs[path]


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype=None):
    a = np.asarray(a) if dtype is None else np.asarray(a, dtype=dtype)
    return np.ascontiguousarray(a)


def _dt(a) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle takes float32 or bf16-bits (uint16) arrays, got {a.dtype}")


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def heads(h, W1, b1, W2, top_s: int, want_logits: bool = False):
    """Medusa heads: top-s ids and log-probs per (sequence, head).

    h [B,d], W1 [K,d,d], b1 [K,d] or None, W2 [K,V,d], all float32 or all bf16 bits.
    Returns (ids int32 [B,K,s], logp float64 [B,K,s], logits [B,K,V] or None,
    logz [B,K]).
    """
    lib = _load()
    h, W1, W2 = _c(h), _c(W1), _c(W2)
    b1 = None if b1 is None else _c(b1)
    dt = _dt(h)
    for a in (W1, W2) + (() if b1 is None else (b1,)):
        if _dt(a) != dt:
            raise TypeError("mixed dtypes")
    B, d = h.shape
    K, V = W2.shape[0], W2.shape[1]
    ids = np.zeros((B, K, top_s), np.int32)
    logp = np.zeros((B, K, top_s), np.float64)
    logits = np.zeros((B, K, V), np.float64) if want_logits else None
    logz = np.zeros((B, K), np.float64)
    rc = lib.oracle_heads(dt, _ptr(h), _ptr(W1), _ptr(b1), _ptr(W2), B, d, V, K, top_s,
                          _ptr(ids), _ptr(logp), _ptr(logits), _ptr(logz))
    _check(rc, "heads")
    return ids, logp, logits, logz


def lm_head(h, W_lm, top_s: int = 1, want_logits: bool = False):
    """The base model's LM head on h: top-s ids and log-probs per sequence;
    entry 0 is the greedy root token.

    h [B,d], W_lm [V,d], float32 or bf16 bits.  Returns (ids int32 [B,s],
    logp float64 [B,s], logits [B,V] or None, logz [B]).
    """
    lib = _load()
    h, W_lm = _c(h), _c(W_lm)
    dt = _dt(h)
    if _dt(W_lm) != dt:
        raise TypeError("mixed dtypes")
    B, d = h.shape
    V = W_lm.shape[0]
    ids = np.zeros((B, top_s), np.int32)
    logp = np.zeros((B, top_s), np.float64)
    logits = np.zeros((B, V), np.float64) if want_logits else None
    logz = np.zeros(B, np.float64)
    rc = lib.oracle_lm_head(dt, _ptr(h), _ptr(W_lm), B, d, V, top_s, _ptr(ids), _ptr(logp),
                            _ptr(logits), _ptr(logz))
    _check(rc, "lm_head")
    return ids, logp, logits, logz


def build_tree(root, topk_ids, topk_logp, s, n: int, prefix_len=None):
    """Greedy budgeted candidate tree in canonical order (see oracle.c, O2).

    Returns a dict of numpy arrays: tokens, parent, depth, pos_id [B,R],
    anc_mask uint64 [B,R,W], paths [B,n,K+1], n_leaf [B], cut_gap [B].
    """
    lib = _load()
    root = _c(root, np.int32)
    topk_ids = _c(topk_ids, np.int32)
    topk_logp = _c(topk_logp, np.float64)
    s = _c(s, np.int32)
    B, K, s_stride = topk_ids.shape
    R = n + 1
    W = (R + 63) // 64
    pl = _c(np.zeros(B) if prefix_len is None else prefix_len, np.int32)
    out = dict(
        tokens=np.zeros((B, R), np.int32), parent=np.zeros((B, R), np.int32),
        depth=np.zeros((B, R), np.int32), pos_id=np.zeros((B, R), np.int32),
        anc_mask=np.zeros((B, R, W), np.uint64), paths=np.zeros((B, n, K + 1), np.int32),
        n_leaf=np.zeros(B, np.int32), cut_gap=np.zeros(B, np.float64),
    )
    rc = lib.oracle_build_tree(_ptr(root), _ptr(topk_ids), _ptr(topk_logp), B, K, _ptr(s),
                               s_stride, n, _ptr(pl), _ptr(out["tokens"]), _ptr(out["parent"]),
                               _ptr(out["depth"]), _ptr(out["pos_id"]), _ptr(out["anc_mask"]),
                               _ptr(out["paths"]), _ptr(out["n_leaf"]), _ptr(out["cut_gap"]))
    _check(rc, "build_tree")
    return out


def tree_attention(q, k_caches, v_caches, prefix_len, anc_mask, scale: float):
    """Tree-masked attention, direct definition.  q [B,R,H,dh]; k/v caches: lists
    of B arrays [P_b+R,H,dh].  Returns float64 [B,R,H,dh]."""
    lib = _load()
    q = _c(q)
    dt = _dt(q)
    B, R, H, dh = q.shape
    ks = [_c(k) for k in k_caches]
    vs = [_c(v) for v in v_caches]
    for a in ks + vs:
        if _dt(a) != dt:
            raise TypeError("mixed dtypes")
    pl = _c(prefix_len, np.int32)
    for b in range(B):
        need = (int(pl[b]) + R) * H * dh
        if ks[b].size < need or vs[b].size < need:
            raise ValueError("cache too small")
    kp = (ctypes.c_void_p * B)(*[k.ctypes.data for k in ks])
    vp = (ctypes.c_void_p * B)(*[v.ctypes.data for v in vs])
    am = _c(anc_mask, np.uint64)
    out = np.zeros((B, R, H, dh), np.float64)
    rc = lib.oracle_tree_attention(dt, _ptr(q), ctypes.cast(kp, ctypes.c_void_p),
                                   ctypes.cast(vp, ctypes.c_void_p), _ptr(pl), _ptr(am),
                                   B, R, H, dh, float(scale), _ptr(out))
    _check(rc, "tree_attention")
    return out


def softmax_entropy(x, T: float = 1.0) -> float:
    """Natural-log entropy of softmax(x / T) for one float64 row."""
    lib = _load()
    x = _c(x, np.float64)
    return float(lib.oracle_softmax_entropy(_ptr(x), x.size, float(T)))


def posterior(logits, tokens, parent, depth, K: int, mode: int, eps=0.09, delta=0.3,
              temperature=1.0, forced_accept=None):
    """Acceptance + longest accepted path.  logits [B,R,V] float32 or bf16 bits.
    Returns dict: accept_len [B], path/path_tokens [B,K+1], next_token [B],
    accept [B,R], margin [B,R]."""
    lib = _load()
    logits = _c(logits)
    dt = _dt(logits)
    B, R, V = logits.shape
    tokens = _c(tokens, np.int32)
    parent = _c(parent, np.int32)
    depth = _c(depth, np.int32)
    fa = None if forced_accept is None else _c(forced_accept, np.int32)
    out = dict(
        accept_len=np.zeros(B, np.int32), path=np.zeros((B, K + 1), np.int32),
        path_tokens=np.zeros((B, K + 1), np.int32), next_token=np.zeros(B, np.int32),
        accept=np.zeros((B, R), np.int32), margin=np.zeros((B, R), np.float64),
    )
    rc = lib.oracle_posterior(dt, _ptr(logits), _ptr(tokens), _ptr(parent), _ptr(depth),
                              B, R, V, K, int(mode), float(eps), float(delta), float(temperature),
                              _ptr(fa), _ptr(out["accept_len"]), _ptr(out["path"]),
                              _ptr(out["path_tokens"]), _ptr(out["next_token"]),
                              _ptr(out["accept"]), _ptr(out["margin"]))
    _check(rc, "posterior")
    return out


def commit_kv(k_caches, v_caches, prefix_len, path, accept_len):
    """Gather the accepted path's K/V rows into contiguous slots (in place on the
    given numpy caches).  Returns the new prefix lengths."""
    lib = _load()
    B = len(k_caches)
    path = _c(path, np.int32)
    K = path.shape[1] - 1
    pl = _c(prefix_len, np.int32)
    al = _c(accept_len, np.int32)
    for a in list(k_caches) + list(v_caches):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("caches must be contiguous")
    row_bytes = k_caches[0][0].nbytes
    kp = (ctypes.c_void_p * B)(*[k.ctypes.data for k in k_caches])
    vp = (ctypes.c_void_p * B)(*[v.ctypes.data for v in v_caches])
    new_pl = np.zeros(B, np.int32)
    rc = lib.oracle_commit_kv(ctypes.cast(kp, ctypes.c_void_p), ctypes.cast(vp, ctypes.c_void_p),
                              _ptr(pl), _ptr(path), _ptr(al), B, K, row_bytes, _ptr(new_pl))
    _check(rc, "commit_kv")
    return new_pl


# ------------------------------------------------------- exact sampling ---

RNG_DRAFT, RNG_ACCEPT, RNG_RESAMPLE = 1, 2, 3


def philox4x64(ctr, key):
    """Philox4x64-10 block: four 64-bit words for a 4-word counter and a
    2-word key."""
    lib = _load()
    c = _c(ctr, np.uint64)
    k = _c(key, np.uint64)
    out = np.zeros(4, np.uint64)
    lib.oracle_philox4x64(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, step: int, purpose: int, b: int, row: int, v: int) -> float:
    return float(_load().oracle_uniform(seed, step, purpose, b, row, v))


def draft_sample(h, W1, b1, W2, temperature: float, seed: int, step: int,
                 want_logits: bool = True, want_keys: bool = False):
    """Drafts x_k ~ softmax(head logits / T) by Gumbel-max (see oracle.c, O5).
    Returns (drafts int32 [B,K], logits [B,K,V] or None, keys [B,K,V] or None)."""
    lib = _load()
    h, W1, W2 = _c(h), _c(W1), _c(W2)
    b1 = None if b1 is None else _c(b1)
    dt = _dt(h)
    B, d = h.shape
    K, V = W2.shape[0], W2.shape[1]
    drafts = np.zeros((B, K), np.int32)
    logits = np.zeros((B, K, V), np.float64) if want_logits else None
    keys = np.zeros((B, K, V), np.float64) if want_keys else None
    rc = lib.oracle_draft_sample(dt, _ptr(h), _ptr(W1), _ptr(b1), _ptr(W2), B, d, V, K,
                                 float(temperature), int(seed), int(step), _ptr(drafts),
                                 _ptr(logits), _ptr(keys))
    _check(rc, "draft_sample")
    return drafts, logits, keys


def speculative_posterior(logits, tokens, draft_logits, temperature: float, seed: int, step: int,
                          forced_accept=None, forced_next=None):
    """Exact speculative sampling on a chain (see oracle.c, O5).  logits
    [B,K+1,V] float32 or bf16 bits, tokens [B,K+1], draft_logits [B,K,V]
    float32.  Returns a dict of numpy arrays."""
    lib = _load()
    logits = _c(logits)
    dt = _dt(logits)
    tokens = _c(tokens, np.int32)
    dl = _c(draft_logits, np.float32)
    B, R, V = logits.shape
    K = R - 1
    fa = None if forced_accept is None else _c(forced_accept, np.int32)
    fn = None if forced_next is None else _c(forced_next, np.int32)
    out = dict(accept_len=np.zeros(B, np.int32), path_tokens=np.zeros((B, K + 1), np.int32),
               next_token=np.zeros(B, np.int32), accept=np.zeros((B, max(K, 1)), np.int32),
               margin=np.zeros((B, max(K, 1)), np.float64), sample_row=np.zeros(B, np.int32),
               sample_keys=np.zeros((B, V), np.float64))
    rc = lib.oracle_speculative_posterior(
        dt, _ptr(logits), _ptr(tokens), _ptr(dl), B, V, K, float(temperature), int(seed),
        int(step), _ptr(fa), _ptr(fn), _ptr(out["accept_len"]), _ptr(out["path_tokens"]),
        _ptr(out["next_token"]), _ptr(out["accept"]), _ptr(out["margin"]),
        _ptr(out["sample_row"]), _ptr(out["sample_keys"]))
    _check(rc, "speculative_posterior")
    out["accept"] = out["accept"][:, :K]
    out["margin"] = out["margin"][:, :K]
    return out
