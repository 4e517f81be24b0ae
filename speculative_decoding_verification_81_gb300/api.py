"""Thin Python binding of libspecverify (ctypes).

Each function has the name of the C entry point it calls and only marshals
arguments: torch tensors on the GPU become device pointers, the current torch
stream becomes the launch stream, and a non-OK status becomes an exception.
Every step of the computation runs in the library's CUDA kernels; there is no
fallback.  If the library is missing the first call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

from . import build as _build

SV_OK = 0
SV_ERR_INVALID_ARG = 1
SV_ERR_WORKSPACE = 2
SV_ERR_UNSUPPORTED = 3
SV_ERR_CUDA = 4
SV_ERR_TIMEOUT = 5
SV_ERR_BAD_INPUT = 6

SV_F32 = 0
SV_BF16 = 1

SV_OP_TREE_ATTENTION = 0
SV_OP_VERIFY_CHAIN = 1
SV_OP_VERIFY_TREE_GREEDY = 2
SV_OP_VERIFY_TREE_STOCHASTIC = 3
SV_OP_VERIFY_STEP_CHAIN = 4
SV_OP_VERIFY_STEP_TREE_GREEDY = 5

EXPORTS = ("sv_workspace_size", "sv_tree_attention", "sv_verify_chain", "sv_verify_tree_greedy",
           "sv_compact_kv", "sv_status_string", "sv_version", "sv_verify_chain_noalloc",
           "sv_tree_attention_paged", "sv_compact_kv_paged", "sv_verify_tree_stochastic",
           "sv_verify_step_chain", "sv_verify_step_tree_greedy")

# Length of the fixed scratch array behind sv_verify_chain_noalloc.
SV_NOALLOC_SCRATCH_BYTES = 4 << 20


class SpecVerifyError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)}")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB_PATH):
            raise ImportError(f"libspecverify.so is not built ({_build.LIB_PATH}); "
                              "run __graft_entry__.build() or python -m "
                              "speculative_decoding_verification_81_gb300.build")
        _lib = load(_build.LIB_PATH)
    return _lib


def use_library(path: str) -> ctypes.CDLL:
    """Route every call of this module to the library at `path` (a build of
    the same sources, e.g. the phase-stamped one of the ``phases`` tool)."""
    global _lib
    _lib = load(path)
    return _lib


def load(path: str) -> ctypes.CDLL:
    """Load a build of libspecverify and declare its entry points' C types."""
    L = ctypes.CDLL(path)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.sv_workspace_size.argtypes = [I, I, I, I, I, I, I, I]
    L.sv_workspace_size.restype = Z
    L.sv_tree_attention.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, ctypes.c_float, P, P, P,
                                    Z, P]
    L.sv_verify_chain.argtypes = [P, P, I, P, P, P, P, I, I, I, P, P, P, P, P, Z, P]
    L.sv_verify_tree_greedy.argtypes = [P, I, P, P, P, I, I, I, P, P, P, P, P, Z, P]
    L.sv_verify_chain_noalloc.argtypes = [P, P, I, P, P, P, I, I, I, P, P, P, P, P]
    L.sv_compact_kv.argtypes = [P, P, P, P, P, I, P, I, I, I, I, P, P]
    L.sv_tree_attention_paged.argtypes = [P, P, P, P, I, I, I, P, P, P, I, I, I, I, I,
                                          ctypes.c_float, P, P, P, Z, P]
    L.sv_compact_kv_paged.argtypes = [P, P, P, I, I, I, P, P, P, I, P, I, I, I, P, P]
    L.sv_verify_tree_stochastic.argtypes = [P, P, I, P, P, P, P, P, I, I, I, P, P, P, P, P, Z,
                                            P]
    F = ctypes.c_float
    L.sv_verify_step_chain.argtypes = [P, P, P, P, I, I, I, I, F, P, P, P, P, I, P, P, P, P, I, I,
                                       I, P, P, P, P, P, P, Z, P]
    L.sv_verify_step_tree_greedy.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, F, P, P, P, I, P,
                                             I, P, P, P, P, P, P, Z, P]
    for fn in ("sv_tree_attention", "sv_verify_chain", "sv_verify_tree_greedy", "sv_compact_kv",
               "sv_verify_chain_noalloc", "sv_tree_attention_paged", "sv_compact_kv_paged",
               "sv_verify_tree_stochastic", "sv_verify_step_chain", "sv_verify_step_tree_greedy"):
        getattr(L, fn).restype = I
    L.sv_status_string.argtypes = [I]
    L.sv_status_string.restype = ctypes.c_char_p
    L.sv_version.argtypes = []
    L.sv_version.restype = I
    return L


def status_string(status: int) -> str:
    return lib().sv_status_string(int(status)).decode()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, rc):
    if rc != SV_OK:
        raise SpecVerifyError(fn, rc)


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return SV_BF16
    if t.dtype == torch.float32:
        return SV_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _on_device(t):
    return t.is_cuda


def _req(t, name, dtype=None, ndim=None):
    if not _on_device(t) or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    return t


def _shape(t, name, shape):
    """The kernels index every array by the call's sizes: a tensor of another
    shape would be read or written out of bounds, so it is refused here."""
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _opt(t, name, dtype, shape):
    """An optional array (an input or a caller-provided output): checked when given."""
    if t is not None:
        _shape(_req(t, name, dtype, len(shape)), name, shape)
    return t


def sv_workspace_size(op: int, B: int, T_or_N: int, V: int = 0, dtype: int = SV_BF16, Hq: int = 0,
                      Hkv: int = 0, D: int = 0) -> int:
    return int(lib().sv_workspace_size(op, B, T_or_N, V, dtype, Hq, Hkv, D))


_ws_cache: dict = {}


def workspace(op: int, B: int, T_or_N: int, V: int = 0, dtype: int = SV_BF16, Hq: int = 0,
              Hkv: int = 0, D: int = 0, device=None) -> torch.Tensor:
    """A zero-filled workspace for one call shape, cached per (shape, device).
    Calls sharing it must not overlap on the GPU."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    key = (op, B, T_or_N, V, dtype, Hq, Hkv, D, str(device))
    ws = _ws_cache.get(key)
    if ws is None:
        n = sv_workspace_size(op, B, T_or_N, V, dtype, Hq, Hkv, D)
        if n == 0:
            raise SpecVerifyError("sv_workspace_size", SV_ERR_UNSUPPORTED)
        ws = torch.zeros(n, dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def sv_tree_attention(q, k_cache, v_cache, prefix_lens, parents=None, scale=None, out=None,
                      seq_status=None, ws=None, stream=None, node_counts=None):
    """q [B,T,Hq,D] bf16; k_cache/v_cache [B,Hkv,S_max,D] bf16; prefix_lens [B] int32;
    parents [B,T] int32 or None (chain); node_counts [B] int32 or None (every
    sequence has T nodes).  Returns out [B,T,Hq,D] bf16."""
    _req(q, "q", torch.bfloat16, 4)
    _req(k_cache, "k_cache", torch.bfloat16, 4)
    _req(v_cache, "v_cache", torch.bfloat16, 4)
    _req(prefix_lens, "prefix_lens", torch.int32, 1)
    B, T, Hq, D = q.shape
    _, Hkv, S_max, _ = k_cache.shape
    _shape(k_cache, "k_cache", (B, Hkv, S_max, D))
    _shape(v_cache, "v_cache", k_cache.shape)
    _shape(prefix_lens, "prefix_lens", (B,))
    _opt(parents, "parents", torch.int32, (B, T))
    _opt(node_counts, "node_counts", torch.int32, (B,))
    _opt(out, "out", torch.bfloat16, q.shape)
    _opt(seq_status, "seq_status", torch.int32, (B,))
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if ws is None:
        ws = workspace(SV_OP_TREE_ATTENTION, B, T, Hq=Hq, Hkv=Hkv, D=D, device=q.device)
    rc = lib().sv_tree_attention(_p(q), _p(k_cache), _p(v_cache), _p(prefix_lens), _p(parents),
                                 _p(node_counts), B, T, Hq, Hkv, D, S_max, float(scale), _p(out),
                                 _p(seq_status), _p(ws), ws.numel(), _stream(stream))
    _check("sv_tree_attention", rc)
    return out


def sv_tree_attention_paged(q, k_pages, v_pages, block_table, prefix_lens, parents=None,
                            scale=None, out=None, seq_status=None, ws=None, stream=None,
                            node_counts=None):
    """q [B,T,Hq,D] bf16; k_pages/v_pages [num_pages,Hkv,page_size,D] bf16;
    block_table [B,max_pages] int32; prefix_lens [B] int32; parents [B,T] int32
    or None (chain).  Returns out [B,T,Hq,D] bf16."""
    _req(q, "q", torch.bfloat16, 4)
    _req(k_pages, "k_pages", torch.bfloat16, 4)
    _req(v_pages, "v_pages", torch.bfloat16, 4)
    _req(block_table, "block_table", torch.int32, 2)
    _req(prefix_lens, "prefix_lens", torch.int32, 1)
    B, T, Hq, D = q.shape
    num_pages, Hkv, page_size, _ = k_pages.shape
    max_pages = block_table.shape[1]
    _shape(k_pages, "k_pages", (num_pages, Hkv, page_size, D))
    _shape(v_pages, "v_pages", k_pages.shape)
    _shape(block_table, "block_table", (B, max_pages))
    _shape(prefix_lens, "prefix_lens", (B,))
    _opt(parents, "parents", torch.int32, (B, T))
    _opt(node_counts, "node_counts", torch.int32, (B,))
    _opt(out, "out", torch.bfloat16, q.shape)
    _opt(seq_status, "seq_status", torch.int32, (B,))
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if ws is None:
        ws = workspace(SV_OP_TREE_ATTENTION, B, T, Hq=Hq, Hkv=Hkv, D=D, device=q.device)
    rc = lib().sv_tree_attention_paged(_p(q), _p(k_pages), _p(v_pages), _p(block_table), max_pages,
                                       num_pages, page_size, _p(prefix_lens), _p(parents),
                                       _p(node_counts), B, T, Hq, Hkv, D, float(scale), _p(out),
                                       _p(seq_status), _p(ws), ws.numel(), _stream(stream))
    _check("sv_tree_attention_paged", rc)
    return out


def _chain_shapes(B, N, V, draft_logits, draft_tokens, u_accept, u_sample, accepted_len,
                  out_tokens, probs_out, seq_status):
    _shape(draft_logits, "draft_logits", (B, N, V))
    _shape(draft_tokens, "draft_tokens", (B, N))
    _shape(u_accept, "u_accept", (B, N))
    _shape(u_sample, "u_sample", (B,))
    _opt(accepted_len, "accepted_len", torch.int32, (B,))
    _opt(out_tokens, "out_tokens", torch.int32, (B, N + 1))
    _opt(probs_out, "probs_out", torch.float32, (B, N, 2))
    _opt(seq_status, "seq_status", torch.int32, (B,))


def sv_verify_chain(target_logits, draft_logits, draft_tokens, u_accept, u_sample,
                    accepted_len=None, out_tokens=None, probs_out=None, seq_status=None, ws=None,
                    stream=None, draft_lens=None):
    """target [B,N+1,V], draft [B,N,V] (bf16 or f32); draft_tokens [B,N] int32;
    u_accept [B,N] f32; u_sample [B] f32; draft_lens [B] int32 or None (every
    sequence drafted N tokens).  Returns (accepted_len [B], out_tokens [B,N+1])."""
    _req(target_logits, "target_logits", None, 3)
    _req(draft_logits, "draft_logits", target_logits.dtype, 3)
    _req(draft_tokens, "draft_tokens", torch.int32, 2)
    _req(u_accept, "u_accept", torch.float32, 2)
    _req(u_sample, "u_sample", torch.float32, 1)
    dt = _dtype_code(target_logits)
    B, N1, V = target_logits.shape
    N = N1 - 1
    _chain_shapes(B, N, V, draft_logits, draft_tokens, u_accept, u_sample, accepted_len,
                  out_tokens, probs_out, seq_status)
    _opt(draft_lens, "draft_lens", torch.int32, (B,))
    dev = target_logits.device
    if accepted_len is None:
        accepted_len = torch.empty(B, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty(B, N + 1, dtype=torch.int32, device=dev)
    if ws is None:
        ws = workspace(SV_OP_VERIFY_CHAIN, B, N, V, dt, device=dev)
    rc = lib().sv_verify_chain(_p(target_logits), _p(draft_logits), dt, _p(draft_tokens),
                               _p(draft_lens), _p(u_accept), _p(u_sample), B, N, V, _p(accepted_len),
                               _p(out_tokens), _p(probs_out), _p(seq_status), _p(ws), ws.numel(),
                               _stream(stream))
    _check("sv_verify_chain", rc)
    return accepted_len, out_tokens


def _tree_shapes(B, T, node_tokens, parents, node_counts, accepted_len, path_nodes, out_tokens,
                 seq_status):
    _shape(node_tokens, "node_tokens", (B, T))
    _opt(parents, "parents", torch.int32, (B, T))
    _opt(node_counts, "node_counts", torch.int32, (B,))
    _opt(accepted_len, "accepted_len", torch.int32, (B,))
    _opt(path_nodes, "path_nodes", torch.int32, (B, T))
    _opt(out_tokens, "out_tokens", torch.int32, (B, T))
    _opt(seq_status, "seq_status", torch.int32, (B,))


def sv_verify_tree_greedy(target_logits, node_tokens, parents, accepted_len=None, path_nodes=None,
                          out_tokens=None, seq_status=None, ws=None, stream=None,
                          node_counts=None):
    """target [B,T,V] (bf16 or f32); node_tokens, parents [B,T] int32 (parents
    None: a chain, i.e. greedy chain verification); node_counts [B] int32 or
    None (every sequence has T nodes).
    Returns (accepted_len [B], path_nodes [B,T], out_tokens [B,T])."""
    _req(target_logits, "target_logits", None, 3)
    _req(node_tokens, "node_tokens", torch.int32, 2)
    dt = _dtype_code(target_logits)
    B, T, V = target_logits.shape
    _tree_shapes(B, T, node_tokens, parents, node_counts, accepted_len, path_nodes, out_tokens,
                 seq_status)
    dev = target_logits.device
    if accepted_len is None:
        accepted_len = torch.empty(B, dtype=torch.int32, device=dev)
    if path_nodes is None:
        path_nodes = torch.empty(B, T, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty(B, T, dtype=torch.int32, device=dev)
    if ws is None:
        ws = workspace(SV_OP_VERIFY_TREE_GREEDY, B, T, V, dt, device=dev)
    rc = lib().sv_verify_tree_greedy(_p(target_logits), dt, _p(node_tokens), _p(parents),
                                     _p(node_counts), B, T, V,
                                     _p(accepted_len), _p(path_nodes), _p(out_tokens),
                                     _p(seq_status), _p(ws), ws.numel(), _stream(stream))
    _check("sv_verify_tree_greedy", rc)
    return accepted_len, path_nodes, out_tokens


def sv_verify_tree_stochastic(target_logits, draft_logits, node_tokens, parents, u_accept,
                              u_sample, accepted_len=None, path_nodes=None, out_tokens=None,
                              seq_status=None, ws=None, stream=None, node_counts=None):
    """target, draft [B,T,V] (bf16 or f32; draft row u: the distribution u's
    children were drawn from); node_tokens, parents [B,T] int32 (parents None:
    a chain); u_accept [B,T] f32; u_sample [B] f32; node_counts [B] int32 or
    None (every sequence has T nodes).
    Returns (accepted_len [B], path_nodes [B,T], out_tokens [B,T])."""
    _req(target_logits, "target_logits", None, 3)
    _req(draft_logits, "draft_logits", target_logits.dtype, 3)
    _req(node_tokens, "node_tokens", torch.int32, 2)
    _req(u_accept, "u_accept", torch.float32, 2)
    _req(u_sample, "u_sample", torch.float32, 1)
    dt = _dtype_code(target_logits)
    B, T, V = target_logits.shape
    _shape(draft_logits, "draft_logits", (B, T, V))
    _shape(u_accept, "u_accept", (B, T))
    _shape(u_sample, "u_sample", (B,))
    _tree_shapes(B, T, node_tokens, parents, node_counts, accepted_len, path_nodes, out_tokens,
                 seq_status)
    dev = target_logits.device
    if accepted_len is None:
        accepted_len = torch.empty(B, dtype=torch.int32, device=dev)
    if path_nodes is None:
        path_nodes = torch.empty(B, T, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty(B, T, dtype=torch.int32, device=dev)
    if ws is None:
        ws = workspace(SV_OP_VERIFY_TREE_STOCHASTIC, B, T, V, dt, device=dev)
    rc = lib().sv_verify_tree_stochastic(_p(target_logits), _p(draft_logits), dt, _p(node_tokens),
                                         _p(parents), _p(node_counts), _p(u_accept),
                                         _p(u_sample), B, T, V,
                                         _p(accepted_len), _p(path_nodes), _p(out_tokens),
                                         _p(seq_status), _p(ws), ws.numel(), _stream(stream))
    _check("sv_verify_tree_stochastic", rc)
    return accepted_len, path_nodes, out_tokens


def _attn_shapes(q, k_cache, v_cache, prefix_lens, out, seq_status):
    _req(q, "q", torch.bfloat16, 4)
    _req(k_cache, "k_cache", torch.bfloat16, 4)
    _req(v_cache, "v_cache", torch.bfloat16, 4)
    _req(prefix_lens, "prefix_lens", torch.int32, 1)
    B, T, Hq, D = q.shape
    _, Hkv, S_max, _ = k_cache.shape
    _shape(k_cache, "k_cache", (B, Hkv, S_max, D))
    _shape(v_cache, "v_cache", k_cache.shape)
    _shape(prefix_lens, "prefix_lens", (B,))
    _opt(out, "attn_out", torch.bfloat16, q.shape)
    _opt(seq_status, "attn_status", torch.int32, (B,))
    return B, T, Hq, D, Hkv, S_max


def sv_verify_step_chain(q, k_cache, v_cache, prefix_lens, target_logits, draft_logits,
                         draft_tokens, u_accept, u_sample, attn_out=None, accepted_len=None,
                         out_tokens=None, new_kv_lens=None, probs_out=None, attn_status=None,
                         verify_status=None, draft_lens=None, scale=None, ws=None, stream=None):
    """The fused chain step.  q [B,N+1,Hq,D] bf16; caches [B,Hkv,S_max,D] bf16;
    prefix_lens [B] int32; logits and draws as sv_verify_chain.
    Returns (attn_out, accepted_len, out_tokens, new_kv_lens)."""
    B, T, Hq, D, Hkv, S_max = _attn_shapes(q, k_cache, v_cache, prefix_lens, attn_out,
                                            attn_status)
    _req(target_logits, "target_logits", None, 3)
    _req(draft_logits, "draft_logits", target_logits.dtype, 3)
    _req(draft_tokens, "draft_tokens", torch.int32, 2)
    _req(u_accept, "u_accept", torch.float32, 2)
    _req(u_sample, "u_sample", torch.float32, 1)
    dt = _dtype_code(target_logits)
    N = T - 1
    V = target_logits.shape[2]
    _shape(target_logits, "target_logits", (B, T, V))
    _chain_shapes(B, N, V, draft_logits, draft_tokens, u_accept, u_sample, accepted_len,
                  out_tokens, probs_out, verify_status)
    _opt(draft_lens, "draft_lens", torch.int32, (B,))
    _opt(new_kv_lens, "new_kv_lens", torch.int32, (B,))
    dev = q.device
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if attn_out is None:
        attn_out = torch.empty_like(q)
    if accepted_len is None:
        accepted_len = torch.empty(B, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty(B, N + 1, dtype=torch.int32, device=dev)
    if new_kv_lens is None:
        new_kv_lens = torch.empty_like(prefix_lens)
    if ws is None:
        ws = workspace(SV_OP_VERIFY_STEP_CHAIN, B, N, V, dt, Hq, Hkv, D, device=dev)
    rc = lib().sv_verify_step_chain(
        _p(q), _p(k_cache), _p(v_cache), _p(prefix_lens), Hq, Hkv, D, S_max, float(scale),
        _p(attn_out), _p(attn_status), _p(target_logits), _p(draft_logits), dt, _p(draft_tokens),
        _p(draft_lens), _p(u_accept), _p(u_sample), B, N, V, _p(accepted_len), _p(out_tokens),
        _p(probs_out), _p(verify_status), _p(new_kv_lens), _p(ws), ws.numel(), _stream(stream))
    _check("sv_verify_step_chain", rc)
    return attn_out, accepted_len, out_tokens, new_kv_lens


def sv_verify_step_tree_greedy(q, k_cache, v_cache, prefix_lens, parents, target_logits,
                               node_tokens, attn_out=None, accepted_len=None, path_nodes=None,
                               out_tokens=None, new_kv_lens=None, attn_status=None,
                               verify_status=None, node_counts=None, scale=None, ws=None,
                               stream=None):
    """The fused tree step (greedy acceptance; the caches are compacted in
    place).  q [B,T,Hq,D] bf16; caches [B,Hkv,S_max,D] bf16; parents [B,T]
    int32 or None (a chain); logits [B,T,V]; node_tokens [B,T] int32.
    Returns (attn_out, accepted_len, path_nodes, out_tokens, new_kv_lens)."""
    B, T, Hq, D, Hkv, S_max = _attn_shapes(q, k_cache, v_cache, prefix_lens, attn_out,
                                            attn_status)
    _req(target_logits, "target_logits", None, 3)
    _req(node_tokens, "node_tokens", torch.int32, 2)
    dt = _dtype_code(target_logits)
    V = target_logits.shape[2]
    _shape(target_logits, "target_logits", (B, T, V))
    _tree_shapes(B, T, node_tokens, parents, node_counts, accepted_len, path_nodes, out_tokens,
                 verify_status)
    _opt(new_kv_lens, "new_kv_lens", torch.int32, (B,))
    dev = q.device
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if attn_out is None:
        attn_out = torch.empty_like(q)
    if accepted_len is None:
        accepted_len = torch.empty(B, dtype=torch.int32, device=dev)
    if path_nodes is None:
        path_nodes = torch.empty(B, T, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty(B, T, dtype=torch.int32, device=dev)
    if new_kv_lens is None:
        new_kv_lens = torch.empty_like(prefix_lens)
    if ws is None:
        ws = workspace(SV_OP_VERIFY_STEP_TREE_GREEDY, B, T, V, dt, Hq, Hkv, D, device=dev)
    rc = lib().sv_verify_step_tree_greedy(
        _p(q), _p(k_cache), _p(v_cache), _p(prefix_lens), _p(parents), _p(node_counts), B, T, Hq,
        Hkv, D, S_max, float(scale), _p(attn_out), _p(attn_status), _p(target_logits), dt,
        _p(node_tokens), V, _p(accepted_len), _p(path_nodes), _p(out_tokens), _p(verify_status),
        _p(new_kv_lens), _p(ws), ws.numel(), _stream(stream))
    _check("sv_verify_step_tree_greedy", rc)
    return attn_out, accepted_len, path_nodes, out_tokens, new_kv_lens


def sv_compact_kv(k_cache, v_cache, prefix_lens, accepted_len, path_nodes=None, new_kv_lens=None,
                  seq_status=None, stream=None):
    """In place on k_cache/v_cache [B,Hkv,S_max,D] bf16.  path_nodes [B,P] int32 or
    None (chain).  Returns new_kv_lens [B] int32 (may be prefix_lens itself)."""
    _req(k_cache, "k_cache", torch.bfloat16, 4)
    _req(v_cache, "v_cache", torch.bfloat16, 4)
    _req(prefix_lens, "prefix_lens", torch.int32, 1)
    _req(accepted_len, "accepted_len", torch.int32, 1)
    B, Hkv, S_max, D = k_cache.shape
    _shape(v_cache, "v_cache", k_cache.shape)
    _shape(prefix_lens, "prefix_lens", (B,))
    _shape(accepted_len, "accepted_len", (B,))
    _opt(new_kv_lens, "new_kv_lens", torch.int32, (B,))
    _opt(seq_status, "seq_status", torch.int32, (B,))
    stride = 0
    if path_nodes is not None:
        _req(path_nodes, "path_nodes", torch.int32, 2)
        _shape(path_nodes, "path_nodes", (B, path_nodes.shape[1]))
        stride = path_nodes.shape[1]
    if new_kv_lens is None:
        new_kv_lens = torch.empty_like(prefix_lens)
    rc = lib().sv_compact_kv(_p(k_cache), _p(v_cache), _p(prefix_lens), _p(new_kv_lens),
                             _p(path_nodes), stride, _p(accepted_len), B, Hkv, D, S_max,
                             _p(seq_status), _stream(stream))
    _check("sv_compact_kv", rc)
    return new_kv_lens


def sv_compact_kv_paged(k_pages, v_pages, block_table, prefix_lens, accepted_len,
                        path_nodes=None, new_kv_lens=None, seq_status=None, stream=None):
    """In place on k_pages/v_pages [num_pages,Hkv,page_size,D] bf16 through
    block_table [B,max_pages] int32.  path_nodes [B,P] int32 or None (chain).
    Returns new_kv_lens [B] int32 (may be prefix_lens itself)."""
    _req(k_pages, "k_pages", torch.bfloat16, 4)
    _req(v_pages, "v_pages", torch.bfloat16, 4)
    _req(block_table, "block_table", torch.int32, 2)
    _req(prefix_lens, "prefix_lens", torch.int32, 1)
    _req(accepted_len, "accepted_len", torch.int32, 1)
    num_pages, Hkv, page_size, D = k_pages.shape
    B, max_pages = block_table.shape
    _shape(v_pages, "v_pages", k_pages.shape)
    _shape(prefix_lens, "prefix_lens", (B,))
    _shape(accepted_len, "accepted_len", (B,))
    _opt(new_kv_lens, "new_kv_lens", torch.int32, (B,))
    _opt(seq_status, "seq_status", torch.int32, (B,))
    stride = 0
    if path_nodes is not None:
        _req(path_nodes, "path_nodes", torch.int32, 2)
        _shape(path_nodes, "path_nodes", (B, path_nodes.shape[1]))
        stride = path_nodes.shape[1]
    if new_kv_lens is None:
        new_kv_lens = torch.empty_like(prefix_lens)
    rc = lib().sv_compact_kv_paged(_p(k_pages), _p(v_pages), _p(block_table), max_pages, num_pages,
                                   page_size, _p(prefix_lens), _p(new_kv_lens), _p(path_nodes),
                                   stride, _p(accepted_len), B, Hkv, D, _p(seq_status),
                                   _stream(stream))
    _check("sv_compact_kv_paged", rc)
    return new_kv_lens


def sv_verify_chain_noalloc(target_logits, draft_logits, draft_tokens, u_accept, u_sample,
                            accepted_len, out_tokens, probs_out=None, seq_status=None, stream=None):
    """sv_verify_chain without a workspace, for callers that cannot allocate
    device memory at the call site; the outputs must be passed in.  Uses the
    library's fixed scratch array: calls must not overlap on the GPU."""
    _req(target_logits, "target_logits", None, 3)
    _req(draft_logits, "draft_logits", target_logits.dtype, 3)
    _req(draft_tokens, "draft_tokens", torch.int32, 2)
    _req(u_accept, "u_accept", torch.float32, 2)
    _req(u_sample, "u_sample", torch.float32, 1)
    _req(accepted_len, "accepted_len", torch.int32, 1)
    _req(out_tokens, "out_tokens", torch.int32, 2)
    dt = _dtype_code(target_logits)
    B, N1, V = target_logits.shape
    _chain_shapes(B, N1 - 1, V, draft_logits, draft_tokens, u_accept, u_sample, accepted_len,
                  out_tokens, probs_out, seq_status)
    rc = lib().sv_verify_chain_noalloc(_p(target_logits), _p(draft_logits), dt, _p(draft_tokens),
                                       _p(u_accept), _p(u_sample), B, N1 - 1, V,
                                       _p(accepted_len), _p(out_tokens), _p(probs_out),
                                       _p(seq_status), _stream(stream))
    _check("sv_verify_chain_noalloc", rc)
    return accepted_len, out_tokens
