"""Seeded synthetic inputs for the verification step.

This module draws the inputs only; it holds none of the verification
arithmetic.  Both the CUDA path and the CPU oracle are fed the same bytes it
produces (bf16 tensors are returned as raw ``uint16`` bit patterns).

Shapes and distributions follow the workloads the pages describe: N = 4..8
draft tokens, trees of tens of nodes, Llama-scale vocabularies (32000,
128256) and grouped-query heads (32 query / 8 KV heads of dimension 128).
No public dataset is involved; these synthetic tensors stand in for model
activations.

Every tensor has its own random stream, ``numpy.random.default_rng([seed,
tag])``, so changing one shape does not perturb the others.  The drafter's
token choice (sampling from softmax of the draft logits) and the tree node
tokens (a fraction copied from the target's argmax at the parent) are part
of the input recipe: they play the drafter, which the step under test does
not contain.
"""
from __future__ import annotations

import itertools

import numpy as np

BF16_NAN = np.uint16(0x7FC0)

# tags for the per-tensor streams
_T_TARGET, _T_BOOST, _T_DRAFT, _T_DTOK, _T_UACC, _T_USAMP = 1, 2, 3, 4, 5, 6
_T_Q, _T_K, _T_V, _T_TREE, _T_NTOK, _T_NMATCH, _T_TLOG = 11, 12, 13, 14, 15, 16, 17


def _rng(seed, tag):
    return np.random.default_rng([int(seed), int(tag)])


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to the nearest bf16 (ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal(rng, shape, sigma, chunk=1 << 24):
    """float32 N(0, sigma^2) samples, drawn in chunks to bound temporaries."""
    n = int(np.prod(shape))
    out = np.empty(n, np.float32)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = rng.standard_normal(e - s, dtype=np.float32)
    if sigma != 1.0:
        out *= np.float32(sigma)
    return out.reshape(shape)


# --------------------------------------------------------------------------
# tree shapes


def medusa_tree(keep=26, branching=(4, 3, 2, 1)):
    """Parent array of a Medusa-style top-k candidate tree.

    Reading of "a fixed Medusa-style tree of 26 nodes (branching top-4, then
    3, 2, 1 along each path; depth 4)": the full 4*3*2*1 tree has 65 nodes, so
    the 26 best-ranked nodes are kept.  A node reached through ranks
    (r1, ..., rd) scores prod 1/(r_i + 1); the root scores 1.  Ties go to the
    shallower node, then to the lexicographically smaller rank path.  Every
    kept node's ancestors score at least as high, so the kept set is a tree.
    Nodes are numbered in breadth-first order (depth, then rank path).
    """
    paths = [()]
    for depth in range(1, len(branching) + 1):
        for ranks in itertools.product(*[range(b) for b in branching[:depth]]):
            paths.append(tuple(ranks))

    def score(p):
        s = 1.0
        for r in p:
            s /= (r + 1)
        return s

    kept = sorted(paths, key=lambda p: (-score(p), len(p), p))[:keep]
    kept = sorted(kept, key=lambda p: (len(p), p))
    index = {p: i for i, p in enumerate(kept)}
    parents = np.array([-1] + [index[p[:-1]] for p in kept[1:]], np.int32)
    return parents


def random_tree(T, max_depth, rng):
    """Random topologically ordered tree: node i's parent is uniform over the
    earlier nodes whose depth is below max_depth (so no node is deeper than
    max_depth).  Node 0 is the root."""
    parents = np.full(T, -1, np.int32)
    depth = np.zeros(T, np.int32)
    for i in range(1, T):
        cand = np.nonzero(depth[:i] < max_depth)[0]
        p = int(cand[rng.integers(0, len(cand))])
        parents[i] = p
        depth[i] = depth[p] + 1
    return parents


def chain_parents(T):
    return np.arange(-1, T - 1, dtype=np.int32)


# --------------------------------------------------------------------------
# logits and acceptance inputs


def _sample_from_logits(logits_f32, u):
    """Drafter's token draw: inverse CDF of softmax(logits) with uniform u."""
    x = logits_f32.astype(np.float64)
    w = np.exp(x - x.max())
    c = np.cumsum(w)
    k = int(np.searchsorted(c, u * c[-1], side="right"))
    return min(k, len(w) - 1)


def chain_inputs(B, N, V, dtype="bf16", target_sigma=3.0, draft_sigma=1.0, boost=8.0,
                 seed=0):
    """Inputs of stochastic chain verification.

    target logits [B, N+1, V] ~ N(0, target_sigma^2), plus `boost` on one
    random token per row; draft logits [B, N, V] = target[:, :N] + N(0,
    draft_sigma^2); draft token x_i sampled from softmax(draft_i); seeded
    uniforms u_accept [B, N] and u_sample [B] in [0, 1).
    """
    t = _normal(_rng(seed, _T_TARGET), (B, N + 1, V), target_sigma)
    if boost:
        idx = _rng(seed, _T_BOOST).integers(0, V, size=(B, N + 1))
        np.add.at(t, (np.arange(B)[:, None], np.arange(N + 1)[None, :], idx), np.float32(boost))
    if dtype == "bf16":
        t_store = f32_to_bf16_bits(t)
        t_val = bf16_bits_to_f32(t_store)
    else:
        t_store = t
        t_val = t
    d = t_val[:, :N] + _normal(_rng(seed, _T_DRAFT), (B, N, V), draft_sigma)
    if dtype == "bf16":
        d_store = f32_to_bf16_bits(d)
        d_val = bf16_bits_to_f32(d_store)
    else:
        d_store = d.astype(np.float32)
        d_val = d_store
    ud = _rng(seed, _T_DTOK).random((B, N))
    tok = np.empty((B, N), np.int32)
    for b in range(B):
        for i in range(N):
            tok[b, i] = _sample_from_logits(d_val[b, i], ud[b, i])
    u_accept = _rng(seed, _T_UACC).random((B, N), dtype=np.float32)
    u_sample = _rng(seed, _T_USAMP).random(B, dtype=np.float32)
    return dict(target=t_store, draft=d_store, draft_tokens=tok, u_accept=u_accept,
                u_sample=u_sample, B=B, N=N, V=V, dtype=dtype)


def stree_inputs(B, T, V, parents, dtype="bf16", target_sigma=3.0, draft_sigma=1.0, boost=8.0,
                 seed=0):
    """Inputs of stochastic tree verification.

    target logits [B, T, V] ~ N(0, target_sigma^2) plus `boost` on one random
    token per row; draft logits [B, T, V] = target + N(0, draft_sigma^2) (row
    u: the drafter at node u); the children of node u drawn independently
    from softmax(draft_u) (node 0's token: 0); seeded uniforms u_accept
    [B, T] and u_sample [B].  parents: [T] (shared) or [B, T].
    """
    par = np.broadcast_to(np.asarray(parents, np.int32), (B, T)).copy()
    t = _normal(_rng(seed, _T_TARGET), (B, T, V), target_sigma)
    if boost:
        idx = _rng(seed, _T_BOOST).integers(0, V, size=(B, T))
        np.add.at(t, (np.arange(B)[:, None], np.arange(T)[None, :], idx), np.float32(boost))
    if dtype == "bf16":
        t_store = f32_to_bf16_bits(t)
        t_val = bf16_bits_to_f32(t_store)
    else:
        t_store = t
        t_val = t
    d = t_val + _normal(_rng(seed, _T_DRAFT), (B, T, V), draft_sigma)
    if dtype == "bf16":
        d_store = f32_to_bf16_bits(d)
        d_val = bf16_bits_to_f32(d_store)
    else:
        d_store = d.astype(np.float32)
        d_val = d_store
    ud = _rng(seed, _T_DTOK).random((B, T))
    tok = np.zeros((B, T), np.int32)
    for b in range(B):
        for v in range(1, T):
            tok[b, v] = _sample_from_logits(d_val[b, par[b, v]], ud[b, v])
    u_accept = _rng(seed, _T_UACC).random((B, T), dtype=np.float32)
    u_sample = _rng(seed, _T_USAMP).random(B, dtype=np.float32)
    return dict(target=t_store, draft=d_store, node_tokens=tok, parents=par, u_accept=u_accept,
                u_sample=u_sample, B=B, T=T, V=V, dtype=dtype)


def tree_logit_inputs(B, T, V, parents, p_match, sigma=3.0, dtype="bf16", seed=0):
    """Inputs of greedy tree verification: target logits [B, T, V] ~ N(0,
    sigma^2); node tokens where each non-root node independently copies the
    target's argmax at its parent with probability p_match, else a uniform
    token.  parents: [T] (shared) or [B, T]."""
    par = np.broadcast_to(np.asarray(parents, np.int32), (B, T)).copy()
    t = _normal(_rng(seed, _T_TLOG), (B, T, V), sigma)
    if dtype == "bf16":
        t_store = f32_to_bf16_bits(t)
        t_val = bf16_bits_to_f32(t_store)
    else:
        t_store = t
        t_val = t
    amax = t_val.argmax(axis=-1)
    r = _rng(seed, _T_NTOK)
    tok = r.integers(0, V, size=(B, T)).astype(np.int32)
    match = _rng(seed, _T_NMATCH).random((B, T)) < p_match
    for b in range(B):
        for i in range(1, T):
            if match[b, i]:
                tok[b, i] = amax[b, par[b, i]]
    return dict(target=t_store, node_tokens=tok, parents=par, B=B, T=T, V=V, dtype=dtype)


def attention_inputs(B, T, Hq, Hkv, D, prefix_lens, S_max=None, parents=None, seed=0,
                     unused_fill="nan"):
    """Q [B,T,Hq,D], K/V caches [B,Hkv,S_max,D] (bf16 bits, N(0,1)) with the
    prefix in slots [0, L_b) and node j's row in slot L_b + j; slots at and
    beyond L_b + T hold NaN (or zeros) so that any read past the valid range
    shows up.  prefix_lens: int or [B]."""
    pl = np.broadcast_to(np.asarray(prefix_lens, np.int32), (B,)).copy()
    if S_max is None:
        S_max = int(pl.max()) + 64
    assert int(pl.max()) + T <= S_max
    q = f32_to_bf16_bits(_normal(_rng(seed, _T_Q), (B, T, Hq, D), 1.0))
    k = f32_to_bf16_bits(_normal(_rng(seed, _T_K), (B, Hkv, S_max, D), 1.0))
    v = f32_to_bf16_bits(_normal(_rng(seed, _T_V), (B, Hkv, S_max, D), 1.0))
    fill = BF16_NAN if unused_fill == "nan" else np.uint16(0)
    for b in range(B):
        k[b, :, pl[b] + T:, :] = fill
        v[b, :, pl[b] + T:, :] = fill
    par = None if parents is None else np.broadcast_to(np.asarray(parents, np.int32), (B, T)).copy()
    return dict(q=q, k=k, v=v, prefix_lens=pl, parents=par, B=B, T=T, Hq=Hq, Hkv=Hkv, D=D,
                S_max=S_max)


# --------------------------------------------------------------------------
# the five named workloads

_T_PAGES = 18


def paged_cache(k, v, page_size, seed=0, spare_pages=3, nan_fill=True):
    """Scatter contiguous caches k, v [B, Hkv, S_max, D] (bf16 bits) into pages
    [num_pages, Hkv, page_size, D] under a random page table: logical page j
    of sequence b is physical page block_table[b, j].  Page slots past S_max
    and the spare pages that no sequence uses hold NaN (zeros without
    nan_fill), so that a stray read shows.  Returns (k_pages, v_pages,
    block_table)."""
    B, Hkv, S_max, D = k.shape
    max_pages = -(-S_max // page_size)
    num_pages = B * max_pages + spare_pages
    r = _rng(seed, _T_PAGES)
    perm = r.permutation(num_pages).astype(np.int32)
    table = perm[:B * max_pages].reshape(B, max_pages)
    fill = 0x7FC0 if nan_fill else 0
    kp = np.full((num_pages, Hkv, page_size, D), fill, np.uint16)
    vp = np.full((num_pages, Hkv, page_size, D), fill, np.uint16)
    for b in range(B):
        for j in range(max_pages):
            s0, s1 = j * page_size, min(S_max, (j + 1) * page_size)
            kp[table[b, j], :, :s1 - s0] = k[b, :, s0:s1]
            vp[table[b, j], :, :s1 - s0] = v[b, :, s0:s1]
    return kp, vp, table


def gather_paged(pages, block_table, S_max):
    """Inverse of paged_cache for one cache: [B, Hkv, S_max, D] from the pages."""
    num_pages, Hkv, page_size, D = pages.shape
    B, max_pages = block_table.shape
    out = np.empty((B, Hkv, max_pages * page_size, D), pages.dtype)
    for b in range(B):
        for j in range(max_pages):
            out[b, :, j * page_size:(j + 1) * page_size] = pages[block_table[b, j]]
    return out[:, :, :S_max]


WORKLOADS = {
    1: dict(name="chain rejection-sampling verify, B=1 N=4 V=1024 fp32",
            kind="chain", B=1, N=4, V=1024, dtype="f32", target_sigma=2.0, draft_sigma=0.5,
            boost=0.0),
    2: dict(name="chain verify at Llama vocab, B=8 N=5 V=32000 bf16",
            kind="chain", B=8, N=5, V=32000, dtype="bf16", target_sigma=3.0, draft_sigma=1.0,
            boost=8.0),
    3: dict(name="tree attention + greedy, B=4 L=2048 Medusa tree T=26 32q/8kv D=128 V=32000",
            kind="tree_step", B=4, L=2048, T=26, tree="medusa", Hq=32, Hkv=8, D=128, V=32000,
            p_match=0.5),
    4: dict(name="fused chain step, B=32 N=8 L=4096 32q/8kv D=128 V=128256",
            kind="chain_step", B=32, N=8, L=4096, Hq=32, Hkv=8, D=128, V=128256,
            target_sigma=3.0, draft_sigma=1.0, boost=8.0),
    5: dict(name="EAGLE-2-style random tree, B=16 T=64 L=8192 32q/8kv D=128 V=128256",
            kind="tree_step", B=16, L=8192, T=64, tree="random", max_depth=8, Hq=32, Hkv=8,
            D=128, V=128256, p_match=0.6),
}


def workload(k, seed=None, **overrides):
    """Inputs for named workload k (1..5).  overrides replace shape fields
    (e.g. B, L, V) to get a smaller case with the same recipe."""
    cfg = dict(WORKLOADS[k])
    cfg.update(overrides)
    seed = 1000 + k if seed is None else seed
    out = dict(cfg=cfg, seed=seed)
    if cfg["kind"] == "chain":
        out.update(chain_inputs(cfg["B"], cfg["N"], cfg["V"], cfg["dtype"], cfg["target_sigma"],
                                cfg["draft_sigma"], cfg["boost"], seed))
        return out
    if cfg["kind"] == "chain_step":
        T = cfg["N"] + 1
        out["chain"] = chain_inputs(cfg["B"], cfg["N"], cfg["V"], "bf16", cfg["target_sigma"],
                                    cfg["draft_sigma"], cfg["boost"], seed)
        out["attn"] = attention_inputs(cfg["B"], T, cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["L"],
                                       parents=None, seed=seed)
        return out
    if cfg["kind"] == "tree_step":
        if cfg["tree"] == "medusa":
            parents = medusa_tree(cfg["T"])
            par_b = np.broadcast_to(parents, (cfg["B"], cfg["T"])).copy()
        else:
            r = _rng(seed, _T_TREE)
            par_b = np.stack([random_tree(cfg["T"], cfg["max_depth"], r) for _ in range(cfg["B"])])
        out["tree"] = tree_logit_inputs(cfg["B"], cfg["T"], cfg["V"], par_b, cfg["p_match"],
                                        seed=seed)
        out["attn"] = attention_inputs(cfg["B"], cfg["T"], cfg["Hq"], cfg["Hkv"], cfg["D"],
                                       cfg["L"], parents=par_b, seed=seed)
        return out
    raise ValueError(cfg["kind"])
