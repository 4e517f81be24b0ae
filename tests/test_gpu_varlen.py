"""GPU parity of variable-length batches: per-sequence node counts T_b
(attention, greedy verification) and draft lengths N_b (chain acceptance).

Each sequence of a ragged batch must give exactly what the oracle gives for
that sequence alone, cut to its own T_b nodes or N_b drafts.  Everything past
a sequence's length is padding filled with values that would show if read:
NaN logits and K/V rows, out-of-range tokens and parents, uniforms >= 1.
"""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_81_gb300 as sv
from speculative_decoding_verification_81_gb300 import workloads as W
from gpu_util import bf16_to_f64, dev, host

pytestmark = pytest.mark.gpu
ATTN_TOL = 1e-2
BF16_NAN = np.uint16(0x7FC0)


def _nan_of(a):
    return BF16_NAN if a.dtype == np.uint16 else np.float32(np.nan)


# ------------------------------------------------------------------ attention

def _pad_attention(inp, counts):
    """NaN in the Q rows and the K/V slots of padding nodes."""
    for b, tb in enumerate(counts):
        L = int(inp["prefix_lens"][b])
        inp["q"][b, tb:] = BF16_NAN
        inp["k"][b, :, L + tb:] = BF16_NAN
        inp["v"][b, :, L + tb:] = BF16_NAN


def _check_attention_rows(orc, inp, par, counts, got):
    for b, tb in enumerate(counts):
        p_b = None if par is None else par[b:b + 1, :tb]
        ref = orc.tree_attention(inp["q"][b:b + 1, :tb], inp["k"][b:b + 1], inp["v"][b:b + 1],
                                 inp["prefix_lens"][b:b + 1], p_b, inp["Hkv"], inp["S_max"])
        err = np.abs(got[b, :tb] - ref[0]).max()
        assert np.isfinite(err) and err <= ATTN_TOL, (b, tb, err)


@pytest.mark.parametrize("B,T,Hq,Hkv,L,counts,tree,seed", [
    (4, 13, 16, 4, [100, 300, 0, 129], [13, 1, 7, 5], "random", 1),
    (3, 9, 32, 8, [4000, 77, 128], [9, 2, 8], "chain", 2),      # a tile edge at L + T_b
    (2, 64, 8, 1, [130, 500], [10, 64], "random", 3),          # whole row groups of padding
    (5, 26, 32, 8, [257, 1000, 3, 64, 2048], [26, 11, 1, 25, 20], "medusa", 4),
])
def test_attention_node_counts(orc, B, T, Hq, Hkv, L, counts, tree, seed):
    rng = np.random.default_rng(seed)
    if tree == "chain":
        par = None
    elif tree == "medusa":
        par = np.broadcast_to(W.medusa_tree(26), (B, T)).copy()
    else:
        par = np.stack([W.random_tree(T, 6, rng) for _ in range(B)])
    inp = W.attention_inputs(B, T, Hq, Hkv, 128, L, parents=par, seed=seed)
    _pad_attention(inp, counts)
    if par is not None:
        for b, tb in enumerate(counts):
            par[b, tb:] = 999  # padding parents: never looked at
    st = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    out = sv.sv_tree_attention(dev(inp["q"]), dev(inp["k"]), dev(inp["v"]),
                               dev(inp["prefix_lens"]), None if par is None else dev(par),
                               seq_status=st, node_counts=dev(np.asarray(counts, np.int32)))
    torch.cuda.synchronize()
    assert (host(st) == 0).all()
    _check_attention_rows(orc, inp, par, counts, bf16_to_f64(host(out)))


def test_attention_node_counts_all_full_equals_null(orc):
    """node_counts all equal to T is the NULL case, bit for bit."""
    inp = W.attention_inputs(3, 9, 32, 8, 128, [500, 33, 129], seed=9)
    args = [dev(inp[n]) for n in ("q", "k", "v", "prefix_lens")]
    a = host(sv.sv_tree_attention(*args))
    b = host(sv.sv_tree_attention(*args, node_counts=dev(np.full(3, 9, np.int32))))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(a, b)


def test_attention_bad_node_counts_reported():
    inp = W.attention_inputs(4, 5, 16, 4, 128, [10, 20, 30, 40], seed=10)
    st = torch.full((4,), -7, dtype=torch.int32, device="cuda")
    sv.sv_tree_attention(dev(inp["q"]), dev(inp["k"]), dev(inp["v"]), dev(inp["prefix_lens"]),
                         seq_status=st, node_counts=dev(np.array([5, 0, 6, -1], np.int32)))
    torch.cuda.synchronize()
    assert host(st).tolist() == [0, sv.SV_ERR_BAD_INPUT, sv.SV_ERR_BAD_INPUT, sv.SV_ERR_BAD_INPUT]


@pytest.mark.parametrize("page_size", [128, 16])
def test_attention_paged_node_counts(orc, page_size):
    B, T, Hq, Hkv = 3, 13, 16, 4
    counts = [4, 13, 1]
    rng = np.random.default_rng(11)
    par = np.stack([W.random_tree(T, 5, rng) for _ in range(B)])
    inp = W.attention_inputs(B, T, Hq, Hkv, 128, [700, 128, 33], parents=par, seed=11)
    _pad_attention(inp, counts)
    kp, vp, table = W.paged_cache(inp["k"], inp["v"], page_size, seed=11)
    st = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    out = sv.sv_tree_attention_paged(dev(inp["q"]), dev(kp), dev(vp), dev(table),
                                     dev(inp["prefix_lens"]), dev(par), seq_status=st,
                                     node_counts=dev(np.asarray(counts, np.int32)))
    torch.cuda.synchronize()
    assert (host(st) == 0).all()
    _check_attention_rows(orc, inp, par, counts, bf16_to_f64(host(out)))


# ------------------------------------------------------------------ chain

def _pad_chain(inp, lens):
    N = inp["draft_tokens"].shape[1]
    for b, nb in enumerate(lens):
        inp["target"][b, nb + 1:] = _nan_of(inp["target"])
        inp["draft"][b, nb:] = _nan_of(inp["draft"])
        inp["draft_tokens"][b, nb:] = -3
        inp["u_accept"][b, nb:] = np.float32(7.0)
    assert N >= max(lens)


def _run_chain_lens(inp, lens):
    B, N = inp["draft_tokens"].shape
    probs = torch.full((B, N, 2), -1.0, dtype=torch.float32, device="cuda")
    st = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    acc, out = sv.sv_verify_chain(dev(inp["target"]), dev(inp["draft"]), dev(inp["draft_tokens"]),
                                  dev(inp["u_accept"]), dev(inp["u_sample"]), probs_out=probs,
                                  seq_status=st, draft_lens=dev(np.asarray(lens, np.int32)))
    torch.cuda.synchronize()
    return host(acc), host(out), host(probs), host(st)


@pytest.mark.parametrize("B,N,V,dtype,lens,seed", [
    (6, 8, 5000, "bf16", [8, 0, 3, 1, 7, 5], 21),
    (4, 8, 128256, "bf16", [2, 8, 0, 6], 22),      # the Llama-3 vocabulary
    (5, 5, 4097, "f32", [5, 4, 0, 2, 1], 23),       # unaligned f32 rows
    (3, 63, 700, "f32", [63, 31, 0], 24),           # maximum N
])
def test_chain_draft_lens(orc, B, N, V, dtype, lens, seed):
    inp = W.chain_inputs(B, N, V, dtype, target_sigma=2.0, draft_sigma=1.0, boost=4.0, seed=seed)
    clean = {k: np.copy(v) for k, v in inp.items()}
    _pad_chain(inp, lens)
    acc, out, probs, st = _run_chain_lens(inp, lens)
    assert (st == 0).all()
    flagged = 0
    for b, nb in enumerate(lens):
        ref = orc.verify_chain(clean["target"][b:b + 1, :nb + 1], clean["draft"][b:b + 1, :nb],
                               clean["draft_tokens"][b:b + 1, :nb],
                               clean["u_accept"][b:b + 1, :nb], clean["u_sample"][b:b + 1])
        assert (out[b, nb + 1:] == -1).all()
        assert (probs[b, nb:] == 0).all()
        if nb:
            rp = ref["probs"][0]
            rel = np.abs(probs[b, :nb].astype(np.float64) - rp) / np.maximum(rp, 1e-30)
            assert rel.max() <= 1e-5, (b, rel.max())
        if ref["flags"][0] & 1:  # an acceptance decision at a near-tie: not compared
            flagged += 1
            continue
        assert acc[b] == ref["accepted_len"][0], b
        a = int(acc[b])
        # the drawn token is compared unless u * S sits at a cumulative-sum
        # boundary (a near-tie, frequent at a flat residual over 128k tokens)
        n_cmp = a if ref["flags"][0] & 2 else a + 1
        np.testing.assert_array_equal(out[b, :n_cmp], ref["out_tokens"][0, :n_cmp])
    assert flagged <= 1


def test_chain_draft_lens_all_full_equals_null():
    inp = W.chain_inputs(8, 6, 3000, "bf16", 2.0, 1.0, 4.0, seed=25)
    args = [dev(inp[n]) for n in ("target", "draft", "draft_tokens", "u_accept", "u_sample")]
    a = [host(x) for x in sv.sv_verify_chain(*args)]
    b = [host(x) for x in sv.sv_verify_chain(*args, draft_lens=dev(np.full(8, 6, np.int32)))]
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_chain_bad_draft_lens_reported():
    inp = W.chain_inputs(4, 3, 700, "f32", 2.0, 1.0, 0.0, seed=26)
    acc, out, probs, st = _run_chain_lens(inp, [3, -1, 4, 0])
    assert st.tolist() == [0, sv.SV_ERR_BAD_INPUT, sv.SV_ERR_BAD_INPUT, 0]
    assert (acc[[1, 2]] == -1).all() and (out[[1, 2]] == -1).all()


# ------------------------------------------------------------------ tree greedy

@pytest.mark.parametrize("B,T,V,dtype,counts,chain,seed", [
    (5, 40, 3000, "bf16", [40, 1, 17, 2, 33], False, 31),
    (4, 26, 128256, "bf16", [26, 9, 1, 14], False, 32),
    (3, 9, 1001, "f32", [9, 5, 1], True, 33),        # greedy chain, parents NULL
    (2, 1024, 64, "bf16", [1024, 500], False, 34),   # maximum T
])
def test_tree_node_counts(orc, B, T, V, dtype, counts, chain, seed):
    rng = np.random.default_rng(seed)
    par = (np.broadcast_to(W.chain_parents(T), (B, T)).copy() if chain else
           np.stack([W.random_tree(T, 8, rng) for _ in range(B)]))
    inp = W.tree_logit_inputs(B, T, V, par, p_match=0.85, sigma=2.0, dtype=dtype, seed=seed)
    clean = {k: np.copy(v) for k, v in inp.items()}
    for b, tb in enumerate(counts):
        inp["target"][b, tb:] = _nan_of(inp["target"])
        inp["node_tokens"][b, tb:] = -5
        inp["parents"][b, tb:] = T + 3
    st = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    acc, path, out = sv.sv_verify_tree_greedy(
        dev(inp["target"]), dev(inp["node_tokens"]), None if chain else dev(inp["parents"]),
        seq_status=st, node_counts=dev(np.asarray(counts, np.int32)))
    torch.cuda.synchronize()
    acc, path, out = host(acc), host(path), host(out)
    assert (host(st) == 0).all()
    for b, tb in enumerate(counts):
        ref = orc.verify_tree_greedy(clean["target"][b:b + 1, :tb],
                                     clean["node_tokens"][b:b + 1, :tb],
                                     clean["parents"][b:b + 1, :tb])
        assert acc[b] == ref["accepted_len"][0], b
        np.testing.assert_array_equal(path[b, :tb], ref["path_nodes"][0])
        np.testing.assert_array_equal(out[b, :tb], ref["out_tokens"][0])
        assert (path[b, tb:] == -1).all() and (out[b, tb:] == -1).all()


def test_tree_bad_node_counts_reported():
    inp = W.tree_logit_inputs(3, 5, 100, W.chain_parents(5), 0.9, seed=35)
    st = torch.full((3,), -7, dtype=torch.int32, device="cuda")
    acc, _, _ = sv.sv_verify_tree_greedy(dev(inp["target"]), dev(inp["node_tokens"]),
                                         dev(inp["parents"]), seq_status=st,
                                         node_counts=dev(np.array([5, 0, 6], np.int32)))
    torch.cuda.synchronize()
    assert host(st).tolist() == [0, sv.SV_ERR_BAD_INPUT, sv.SV_ERR_BAD_INPUT]
    assert (host(acc)[1:] == -1).all()


# ------------------------------------------------------------------ stochastic tree

@pytest.mark.parametrize("B,T,V,dtype,counts,seed", [
    (5, 20, 3000, "bf16", [20, 1, 9, 2, 14], 41),
    (3, 26, 32000, "bf16", [26, 5, 13], 42),
    (4, 12, 1001, "f32", [12, 7, 1, 3], 43),
])
def test_stochastic_tree_node_counts(orc, B, T, V, dtype, counts, seed):
    rng = np.random.default_rng(seed)
    par = np.stack([W.random_tree(T, 6, rng) for _ in range(B)])
    inp = W.stree_inputs(B, T, V, par, dtype, target_sigma=2.0, draft_sigma=1.0, boost=4.0,
                         seed=seed)
    clean = {k: np.copy(v) for k, v in inp.items()}
    for b, tb in enumerate(counts):
        inp["target"][b, tb:] = _nan_of(inp["target"])
        inp["draft"][b, tb:] = _nan_of(inp["draft"])
        inp["node_tokens"][b, tb:] = -5
        inp["parents"][b, tb:] = T + 3
    st = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    acc, path, out = sv.sv_verify_tree_stochastic(
        dev(inp["target"]), dev(inp["draft"]), dev(inp["node_tokens"]), dev(inp["parents"]),
        dev(inp["u_accept"]), dev(inp["u_sample"]), seq_status=st,
        node_counts=dev(np.asarray(counts, np.int32)))
    torch.cuda.synchronize()
    acc, path, out = host(acc), host(path), host(out)
    assert (host(st) == 0).all()
    for b, tb in enumerate(counts):
        ref = orc.verify_tree_stochastic(clean["target"][b:b + 1, :tb], clean["draft"][b:b + 1, :tb],
                                         clean["node_tokens"][b:b + 1, :tb],
                                         clean["parents"][b:b + 1, :tb],
                                         clean["u_accept"][b:b + 1, :tb], clean["u_sample"][b:b + 1])
        assert (path[b, tb:] == -1).all() and (out[b, tb:] == -1).all()
        f = ref["flags"][0]
        if f & 1:
            continue
        assert acc[b] == ref["accepted_len"][0], b
        np.testing.assert_array_equal(path[b, :tb], ref["path_nodes"][0])
        n_cmp = int(acc[b]) if f & 2 else tb
        np.testing.assert_array_equal(out[b, :n_cmp], ref["out_tokens"][0, :n_cmp])
