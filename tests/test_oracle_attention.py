"""Pins for the oracle's verification attention and ancestor mask.

Each test checks the oracle against something other than its own formula:
torch's scaled_dot_product_attention on special cases that reduce to plain
decode / causal attention, a per-node gather of the root->node path (a
different formulation of the tree mask), relabelling invariance and closed
forms.  Source: "Parallel Decoding" glossary, Medusa "Tree attention" and
"L'attention en arbre : la brique commune"; "Chapitre 9 -- Décodage
spéculatif" §9.1 (one pass over prefix + candidates) and §9.2 (EAGLE-2 tree
verified in one attention pass with a custom mask).
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from speculative_decoding_verification_81_gb300 import workloads as W


def _f64(bits):
    return torch.from_numpy(W.bf16_bits_to_f32(bits).astype(np.float64))


def _sdpa(qrows, krows, vrows, mask=None):
    """qrows [M,D], krows/vrows [K,D] float64 -> [M,D] via torch SDPA."""
    return F.scaled_dot_product_attention(qrows[None, None], krows[None, None], vrows[None, None],
                                          attn_mask=None if mask is None else mask[None, None])[0, 0]


def _gqa_kv(h, Hq, Hkv):
    return h // (Hq // Hkv)


def test_ancestor_mask_chain_is_causal(orc):
    T = 9
    m, depth = orc.ancestor_mask(None, T)
    assert np.array_equal(m, np.tril(np.ones((T, T), np.uint8)))
    assert depth.tolist() == list(range(T))
    m2, _ = orc.ancestor_mask(W.chain_parents(T), T)
    assert np.array_equal(m, m2)


def test_ancestor_mask_star_and_medusa(orc):
    T = 6
    star = np.array([-1, 0, 0, 0, 0, 0], np.int32)
    m, depth = orc.ancestor_mask(star, T)
    expect = np.eye(T, dtype=np.uint8)
    expect[:, 0] = 1
    assert np.array_equal(m, expect)
    assert depth.tolist() == [0, 1, 1, 1, 1, 1]
    par = W.medusa_tree(26)
    m, depth = orc.ancestor_mask(par, 26)
    # depth histogram of the 26-node tree: 1, 4, 7, 8, 6 nodes at depths 0..4
    assert np.bincount(depth).tolist() == [1, 4, 7, 8, 6]
    # row t has exactly depth+1 ones
    assert (m.sum(1) == depth + 1).all()


@pytest.mark.parametrize("bad", [[0, 0, 1], [-1, 1, 0], [-1, 0, 3], [-1, -1, 0]])
def test_ancestor_mask_rejects_bad_parents(orc, bad):
    with pytest.raises(ValueError):
        orc.ancestor_mask(np.array(bad, np.int32), 3)


def test_single_query_is_plain_decode_attention(orc):
    """T = 1: the step degenerates to ordinary decode attention over L+1 keys."""
    inp = W.attention_inputs(B=2, T=1, Hq=4, Hkv=2, D=64, prefix_lens=[37, 5], seed=3)
    out = orc.tree_attention(inp["q"], inp["k"], inp["v"], inp["prefix_lens"], None, 2,
                             inp["S_max"])
    for b in range(2):
        L = int(inp["prefix_lens"][b])
        for h in range(4):
            kv = _gqa_kv(h, 4, 2)
            ref = _sdpa(_f64(inp["q"][b, :, h]), _f64(inp["k"][b, kv, :L + 1]),
                        _f64(inp["v"][b, kv, :L + 1]))
            np.testing.assert_allclose(out[b, :, h], ref.numpy(), rtol=0, atol=1e-12)


def test_chain_equals_causal_attention(orc):
    """Chain parents => prefix fully visible plus a causal mask over the N+1 new rows."""
    B, T, Hq, Hkv, D = 2, 9, 8, 2, 32
    inp = W.attention_inputs(B, T, Hq, Hkv, D, prefix_lens=[70, 0], seed=4)
    out_null = orc.tree_attention(inp["q"], inp["k"], inp["v"], inp["prefix_lens"], None, Hkv,
                                  inp["S_max"])
    par = np.broadcast_to(W.chain_parents(T), (B, T))
    out_par = orc.tree_attention(inp["q"], inp["k"], inp["v"], inp["prefix_lens"], par, Hkv,
                                 inp["S_max"])
    np.testing.assert_array_equal(out_null, out_par)
    for b in range(B):
        L = int(inp["prefix_lens"][b])
        causal = torch.ones(T, L + T, dtype=torch.bool).tril(diagonal=L)
        for h in range(Hq):
            kv = _gqa_kv(h, Hq, Hkv)
            ref = _sdpa(_f64(inp["q"][b, :, h]), _f64(inp["k"][b, kv, :L + T]),
                        _f64(inp["v"][b, kv, :L + T]), causal)
            np.testing.assert_allclose(out_null[b, :, h], ref.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("tree", ["medusa", "random"])
def test_tree_node_equals_attention_over_its_own_path(orc, tree):
    """Each node's output equals causal attention of that node alone over
    [prefix || the K/V rows of its root->node path, in path order]."""
    rng = np.random.default_rng(5)
    T = 26 if tree == "medusa" else 20
    B, Hq, Hkv, D = 2, 8, 4, 64
    if tree == "medusa":
        par = np.broadcast_to(W.medusa_tree(26), (B, T)).copy()
    else:
        par = np.stack([W.random_tree(T, 5, rng) for _ in range(B)])
    inp = W.attention_inputs(B, T, Hq, Hkv, D, prefix_lens=[51, 130], parents=par, seed=6)
    out = orc.tree_attention(inp["q"], inp["k"], inp["v"], inp["prefix_lens"], par, Hkv,
                             inp["S_max"])
    for b in range(B):
        L = int(inp["prefix_lens"][b])
        for t in range(T):
            path = []
            n = t
            while n >= 0:
                path.append(n)
                n = int(par[b, n])
            path = path[::-1]
            slots = list(range(L)) + [L + j for j in path]
            for h in range(Hq):
                kv = _gqa_kv(h, Hq, Hkv)
                ref = _sdpa(_f64(inp["q"][b, t:t + 1, h]), _f64(inp["k"][b, kv, slots]),
                            _f64(inp["v"][b, kv, slots]))
                np.testing.assert_allclose(out[b, t, h], ref[0].numpy(), rtol=0, atol=1e-12)


def test_relabelling_permutes_outputs(orc):
    """A different topological numbering of the same tree permutes the outputs."""
    B, T, Hq, Hkv, D = 1, 12, 4, 1, 32
    rng = np.random.default_rng(7)
    par = W.random_tree(T, 4, rng)
    inp = W.attention_inputs(B, T, Hq, Hkv, D, prefix_lens=[40], parents=par[None], seed=8)
    out = orc.tree_attention(inp["q"], inp["k"], inp["v"], inp["prefix_lens"], par[None], Hkv,
                             inp["S_max"])
    # new numbering: sort nodes by (depth, -old index): still topological
    _, depth = orc.ancestor_mask(par, T)
    order = sorted(range(T), key=lambda i: (depth[i], -i))  # order[new] = old
    new_of = {old: new for new, old in enumerate(order)}
    par2 = np.array([-1 if par[o] < 0 else new_of[int(par[o])] for o in order], np.int32)
    L = 40
    q2 = inp["q"][:, order]
    k2 = inp["k"].copy()
    v2 = inp["v"].copy()
    k2[:, :, L:L + T] = inp["k"][:, :, [L + o for o in order]]
    v2[:, :, L:L + T] = inp["v"][:, :, [L + o for o in order]]
    out2 = orc.tree_attention(q2, k2, v2, inp["prefix_lens"], par2[None], Hkv, inp["S_max"])
    np.testing.assert_allclose(out2, out[:, order], rtol=0, atol=1e-13)


def test_gqa_head_mapping(orc):
    """Query head h reads KV head h // (Hq/Hkv): consecutive query heads share."""
    B, T, Hq, Hkv, D = 1, 3, 8, 4, 16
    inp = W.attention_inputs(B, T, Hq, Hkv, D, prefix_lens=[10], seed=9)
    out = orc.tree_attention(inp["q"], inp["k"], inp["v"], inp["prefix_lens"], None, Hkv,
                             inp["S_max"])
    L = 10
    kx = torch.repeat_interleave(_f64(inp["k"][0, :, :L + T]), Hq // Hkv, dim=0)
    vx = torch.repeat_interleave(_f64(inp["v"][0, :, :L + T]), Hq // Hkv, dim=0)
    qx = _f64(inp["q"][0]).permute(1, 0, 2)  # [Hq, T, D]
    causal = torch.ones(T, L + T, dtype=torch.bool).tril(diagonal=L)
    ref = F.scaled_dot_product_attention(qx[None], kx[None], vx[None], attn_mask=causal)[0]
    np.testing.assert_allclose(out[0], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_closed_forms(orc):
    """Constant V rows => output is that constant; K = 0 => uniform mean of allowed V."""
    B, T, Hq, Hkv, D = 1, 5, 2, 1, 8
    par = np.array([[-1, 0, 0, 1, 2]], np.int32)
    inp = W.attention_inputs(B, T, Hq, Hkv, D, prefix_lens=[6], parents=par, seed=10,
                             unused_fill="zero")
    L = 6
    v = inp["v"].copy()
    v[:, :, :L + T] = W.f32_to_bf16_bits(np.full((1, 1, L + T, D), 0.75, np.float32))
    out = orc.tree_attention(inp["q"], inp["k"], v, inp["prefix_lens"], par, Hkv, inp["S_max"])
    np.testing.assert_allclose(out, 0.75, rtol=0, atol=1e-14)
    k0 = np.zeros_like(inp["k"])
    out = orc.tree_attention(inp["q"], k0, inp["v"], inp["prefix_lens"], par, Hkv, inp["S_max"])
    vf = W.bf16_bits_to_f32(inp["v"]).astype(np.float64)
    paths = {0: [0], 1: [0, 1], 2: [0, 2], 3: [0, 1, 3], 4: [0, 2, 4]}
    for t, p in paths.items():
        rows = list(range(L)) + [L + j for j in p]
        expect = vf[0, 0, rows].mean(0)
        for h in range(Hq):
            np.testing.assert_allclose(out[0, t, h], expect, rtol=0, atol=1e-13)


def test_selected_rows_match_full(orc):
    inp = W.attention_inputs(B=2, T=4, Hq=4, Hkv=2, D=32, prefix_lens=[20, 9], seed=11)
    full = orc.tree_attention(inp["q"], inp["k"], inp["v"], inp["prefix_lens"], None, 2,
                              inp["S_max"])
    sel = np.array([[1, 3, 2], [0, 0, 0]], np.int32)
    part = orc.tree_attention(inp["q"], inp["k"], inp["v"], inp["prefix_lens"], None, 2,
                              inp["S_max"], sel=sel)
    for b, t, h in sel:
        np.testing.assert_array_equal(part[b, t, h], full[b, t, h])
    assert np.isnan(part[0, 1, 1]).all()
