"""CPU oracle for the speculative-decoding verification step.

TEST INFRASTRUCTURE ONLY.  This package wraps ``oracle.c`` (plain C, double
precision, single-threaded) through ctypes.  Only the tests, the smoke check
and the benchmark's CPU-baseline leg may import it; the product library never
does, and shares no code with it.

Each wrapper takes numpy arrays holding the same bytes the GPU path gets
(bf16 as raw ``uint16`` bits) and returns numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

OK = 0
ERR_INVALID_ARG = 1
ERR_BAD_INPUT = 6

FLAG_ACCEPT_NEAR_TIE = 1
FLAG_SAMPLE_NEAR_TIE = 2
FLAG_DEGENERATE_RESIDUAL = 4

F32 = 0
BF16 = 1


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (gcc, no fast-math, no FMA contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call([
        "gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
        "-shared", "-fPIC", _SRC, "-o", tmp, "-lm",
    ])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        _lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I = ctypes.c_int
        _lib.orc_ancestor_mask.argtypes = [P, I, P, P]
        _lib.orc_tree_attention.argtypes = [P, P, P, P, P, I, I, I, I, I, I, ctypes.c_double, P, I, P]
        _lib.orc_row_stats.argtypes = [P, I, I, P, P, P]
        _lib.orc_row_stats.restype = None
        _lib.orc_verify_chain.argtypes = [P, P, I, P, P, P, I, I, I, P, P, P, P, P]
        _lib.orc_verify_tree_greedy.argtypes = [P, I, P, P, I, I, I, P, P, P, P]
        _lib.orc_verify_tree_stochastic.argtypes = [P, P, I, P, P, P, P, I, I, I, P, P, P, P, P]
        _lib.orc_compact_kv.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, P, P]
        for name in ("orc_ancestor_mask", "orc_tree_attention", "orc_verify_chain",
                     "orc_verify_tree_greedy", "orc_verify_tree_stochastic", "orc_compact_kv"):
            getattr(_lib, name).restype = ctypes.c_int
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _logits_dtype(arr):
    if arr.dtype == np.float32:
        return F32
    if arr.dtype == np.uint16:
        return BF16
    raise TypeError("logits must be float32 or uint16 (bf16 bits)")


def ancestor_mask(parents, T):
    """(mask [T,T] uint8, depth [T] int32) for one parent array (None = chain)."""
    mask = np.zeros((T, T), np.uint8)
    depth = np.zeros(T, np.int32)
    par = None if parents is None else _c(parents, np.int32)
    rc = lib().orc_ancestor_mask(_ptr(par), T, _ptr(mask), _ptr(depth))
    if rc != OK:
        raise ValueError(f"orc_ancestor_mask status {rc}")
    return mask, depth


def tree_attention(q, k, v, prefix_lens, parents, Hkv, S_max, scale=None, sel=None):
    """Dense masked attention, float64 output [B,T,Hq,D].

    q: uint16 [B,T,Hq,D]; k, v: uint16 [B,Hkv,S_max,D]; parents int32 [B,T] or None
    (chain).  sel: optional int array [n,3] of (b,t,h) rows to compute (others NaN).
    """
    q = _c(q, np.uint16)
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    B, T, Hq, D = q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    pl = _c(prefix_lens, np.int32)
    par = None if parents is None else _c(parents, np.int32)
    out = np.full((B, T, Hq, D), np.nan, np.float64)
    s = None if sel is None else _c(sel, np.int32).reshape(-1, 3)
    rc = lib().orc_tree_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(pl), _ptr(par),
                                  B, T, Hq, Hkv, D, S_max, float(scale),
                                  _ptr(s), 0 if s is None else s.shape[0], _ptr(out))
    if rc != OK:
        raise ValueError(f"orc_tree_attention status {rc}")
    return out


def row_stats(row):
    """(m, s, argmax) of one logits row (float32 or bf16 bits)."""
    row = np.ascontiguousarray(row)
    m = ctypes.c_double()
    s = ctypes.c_double()
    am = ctypes.c_int32()
    lib().orc_row_stats(_ptr(row), _logits_dtype(row), row.shape[-1],
                        ctypes.byref(m), ctypes.byref(s), ctypes.byref(am))
    return m.value, s.value, am.value


def verify_chain(target, draft, draft_tokens, u_accept, u_sample):
    """Stochastic chain acceptance.  Returns dict of accepted_len [B],
    out_tokens [B,N+1], probs [B,N,2], flags [B], status [B]."""
    target = np.ascontiguousarray(target)
    draft = np.ascontiguousarray(draft)
    dt = _logits_dtype(target)
    assert _logits_dtype(draft) == dt
    B, N1, V = target.shape
    N = N1 - 1
    assert draft.shape == (B, N, V)
    tok = _c(draft_tokens, np.int32).reshape(B, N)
    ua = _c(u_accept, np.float32).reshape(B, N)
    us = _c(u_sample, np.float32).reshape(B)
    acc = np.zeros(B, np.int32)
    out = np.zeros((B, N + 1), np.int32)
    probs = np.zeros((B, N, 2), np.float64)
    flags = np.zeros(B, np.int32)
    status = np.zeros(B, np.int32)
    rc = lib().orc_verify_chain(_ptr(target), _ptr(draft), dt, _ptr(tok), _ptr(ua), _ptr(us),
                                B, N, V, _ptr(acc), _ptr(out), _ptr(probs), _ptr(flags),
                                _ptr(status))
    if rc != OK:
        raise ValueError(f"orc_verify_chain status {rc}")
    return dict(accepted_len=acc, out_tokens=out, probs=probs, flags=flags, status=status)


def verify_tree_greedy(target, node_tokens, parents):
    """Greedy longest agreeing path.  Returns dict of accepted_len [B],
    path_nodes [B,T], out_tokens [B,T], status [B]."""
    target = np.ascontiguousarray(target)
    dt = _logits_dtype(target)
    B, T, V = target.shape
    tok = _c(node_tokens, np.int32).reshape(B, T)
    par = _c(parents, np.int32).reshape(B, T)
    acc = np.zeros(B, np.int32)
    path = np.zeros((B, T), np.int32)
    out = np.zeros((B, T), np.int32)
    status = np.zeros(B, np.int32)
    rc = lib().orc_verify_tree_greedy(_ptr(target), dt, _ptr(tok), _ptr(par), B, T, V,
                                      _ptr(acc), _ptr(path), _ptr(out), _ptr(status))
    if rc != OK:
        raise ValueError(f"orc_verify_tree_greedy status {rc}")
    return dict(accepted_len=acc, path_nodes=path, out_tokens=out, status=status)


def verify_tree_stochastic(target, draft, node_tokens, parents, u_accept, u_sample):
    """Multi-draft stochastic acceptance on a tree.  Returns dict of
    accepted_len [B], path_nodes [B,T], out_tokens [B,T], flags [B], status [B]."""
    target = np.ascontiguousarray(target)
    draft = np.ascontiguousarray(draft)
    dt = _logits_dtype(target)
    assert _logits_dtype(draft) == dt
    B, T, V = target.shape
    assert draft.shape == (B, T, V)
    tok = _c(node_tokens, np.int32).reshape(B, T)
    par = _c(parents, np.int32).reshape(B, T)
    ua = _c(u_accept, np.float32).reshape(B, T)
    us = _c(u_sample, np.float32).reshape(B)
    acc = np.zeros(B, np.int32)
    path = np.zeros((B, T), np.int32)
    out = np.zeros((B, T), np.int32)
    flags = np.zeros(B, np.int32)
    status = np.zeros(B, np.int32)
    rc = lib().orc_verify_tree_stochastic(_ptr(target), _ptr(draft), dt, _ptr(tok), _ptr(par),
                                          _ptr(ua), _ptr(us), B, T, V, _ptr(acc), _ptr(path),
                                          _ptr(out), _ptr(flags), _ptr(status))
    if rc != OK:
        raise ValueError(f"orc_verify_tree_stochastic status {rc}")
    return dict(accepted_len=acc, path_nodes=path, out_tokens=out, flags=flags, status=status)


def compact_kv(k, v, prefix_lens, path_nodes, accepted_len):
    """Out-of-place compaction.  Returns dict of k, v, new_kv_lens, status."""
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    B, Hkv, S_max, D = k.shape
    pl = _c(prefix_lens, np.int32)
    acc = _c(accepted_len, np.int32)
    path = None if path_nodes is None else _c(path_nodes, np.int32)
    stride = 0 if path is None else path.shape[-1]
    k_out = np.empty_like(k)
    v_out = np.empty_like(v)
    lens = np.zeros(B, np.int32)
    status = np.zeros(B, np.int32)
    rc = lib().orc_compact_kv(_ptr(k), _ptr(v), _ptr(k_out), _ptr(v_out), _ptr(pl), _ptr(path),
                              _ptr(acc), B, Hkv, D, S_max, stride, _ptr(lens), _ptr(status))
    if rc != OK:
        raise ValueError(f"orc_compact_kv status {rc}")
    return dict(k=k_out, v=v_out, new_kv_lens=lens, status=status)
