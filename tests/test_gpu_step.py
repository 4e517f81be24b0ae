"""GPU parity of the fused verification step (sv_verify_step_chain,
sv_verify_step_tree_greedy) against the oracle: the attention rows (sampled
at full size, within 1e-2 max-abs), the acceptance (bit-exact except the
oracle's flagged near-ties; p, q within 1e-5 relative), the compacted caches
and the new lengths (bit-exact), all from one call on one set of inputs.
"""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_81_gb300 as sv
from speculative_decoding_verification_81_gb300 import workloads as W
from gpu_util import bf16_to_f64, dev, host

pytestmark = pytest.mark.gpu


def _sample_rows(rng, B, T, Hq, n, counts=None):
    rows = []
    for _ in range(n):
        b = int(rng.integers(0, B))
        t = int(rng.integers(0, T if counts is None else counts[b]))
        rows.append((b, t, int(rng.integers(0, Hq))))
    return np.array(sorted(set(rows)), np.int32)


def _check_attention(orc, a, out, parents, sel=None):
    ref = orc.tree_attention(a["q"], a["k"], a["v"], a["prefix_lens"], parents, a["Hkv"],
                             a["S_max"], sel=sel)
    got = bf16_to_f64(host(out))
    if sel is None:
        err = np.abs(got - ref).max()
    else:
        err = max(np.abs(got[b, t, h] - ref[b, t, h]).max() for b, t, h in sel)
    assert err <= 1e-2, err


def _check_chain(ref, acc, toks, probs, status, max_flag_frac=0.02):
    np.testing.assert_array_equal(status, ref["status"])
    ok = ref["flags"] == 0
    np.testing.assert_array_equal(acc[ok], ref["accepted_len"][ok])
    np.testing.assert_array_equal(toks[ok], ref["out_tokens"][ok])
    good = ref["status"] == 0
    rp, gp = ref["probs"][good], probs[good].astype(np.float64)
    big = rp > 1e-30
    assert (np.abs(gp[big] - rp[big]) / rp[big]).max(initial=0.0) <= 1e-5
    assert (~ok).mean() <= max_flag_frac
    return ok


def _chain_step(inp, draft_lens=None):
    a, c = inp["attn"], inp["chain"]
    B, N = c["draft_tokens"].shape
    k, v = dev(a["k"]), dev(a["v"])
    k0, v0 = k.clone(), v.clone()
    probs = torch.full((B, N, 2), -1.0, dtype=torch.float32, device="cuda")
    ast = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    vst = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    out, acc, toks, newl = sv.sv_verify_step_chain(
        dev(a["q"]), k, v, dev(a["prefix_lens"]), dev(c["target"]), dev(c["draft"]),
        dev(c["draft_tokens"]), dev(c["u_accept"]), dev(c["u_sample"]), probs_out=probs,
        attn_status=ast, verify_status=vst,
        draft_lens=None if draft_lens is None else dev(draft_lens))
    torch.cuda.synchronize()
    # a chain moves no rows (bits compared: the unused slots hold NaN)
    assert torch.equal(k.view(torch.int16), k0.view(torch.int16))
    assert torch.equal(v.view(torch.int16), v0.view(torch.int16))
    return out, host(acc), host(toks), host(probs), host(ast), host(vst), host(newl)


def test_chain_step_full_size(orc):
    """The bench's whole step -- B=32, N=8, L=4096, 32q/8kv heads, V=128256 --
    on one set of inputs: sampled attention rows, the acceptance and the new
    lengths against the oracle."""
    inp = W.workload(4)
    a, c = inp["attn"], inp["chain"]
    out, acc, toks, probs, ast, vst, newl = _chain_step(inp)
    sel = _sample_rows(np.random.default_rng(4), a["B"], a["T"], a["Hq"], 96)
    _check_attention(orc, a, out, None, sel)
    assert (ast == 0).all()
    ref = orc.verify_chain(c["target"], c["draft"], c["draft_tokens"], c["u_accept"],
                           c["u_sample"])
    ok = _check_chain(ref, acc, toks, probs, vst)
    # a chain's compaction moves nothing (checked in _chain_step) and sets L + a + 1
    np.testing.assert_array_equal(newl[ok], a["prefix_lens"][ok] + ref["accepted_len"][ok] + 1)
    np.testing.assert_array_equal(newl[~ok], a["prefix_lens"][~ok] + acc[~ok] + 1)


def test_chain_step_small_cluster_mode(orc):
    """A small chain step (the attention in cluster mode), every row checked."""
    c = W.chain_inputs(3, 5, 4000, "bf16", 3.0, 1.0, 8.0, seed=12)
    a = W.attention_inputs(3, 6, 16, 4, 128, [700, 1, 129], seed=12)
    out, acc, toks, probs, ast, vst, newl = _chain_step(dict(attn=a, chain=c))
    _check_attention(orc, a, out, None)
    ref = orc.verify_chain(c["target"], c["draft"], c["draft_tokens"], c["u_accept"],
                           c["u_sample"])
    ok = _check_chain(ref, acc, toks, probs, vst, max_flag_frac=1.0)
    np.testing.assert_array_equal(newl[ok], a["prefix_lens"][ok] + ref["accepted_len"][ok] + 1)


def test_chain_step_ragged_draft_lengths(orc):
    """Draft lengths N_b < N: each sequence equals the oracle on that sequence
    alone, cut to N_b drafts (N_b + 1 attention rows)."""
    B, N, V = 4, 6, 3000
    lens = np.array([6, 0, 3, 1], np.int32)
    c = W.chain_inputs(B, N, V, "bf16", 3.0, 1.0, 8.0, seed=21)
    a = W.attention_inputs(B, N + 1, 8, 2, 128, [50, 300, 0, 1000], seed=21)
    out, acc, toks, probs, ast, vst, newl = _chain_step(dict(attn=a, chain=c), draft_lens=lens)
    got = bf16_to_f64(host(out))
    for b in range(B):
        nb = int(lens[b])
        sub = dict(q=a["q"][b:b + 1, :nb + 1], k=a["k"][b:b + 1], v=a["v"][b:b + 1],
                   prefix_lens=a["prefix_lens"][b:b + 1], Hkv=a["Hkv"], S_max=a["S_max"])
        ref_o = orc.tree_attention(sub["q"], sub["k"], sub["v"], sub["prefix_lens"], None,
                                   sub["Hkv"], sub["S_max"])
        assert np.abs(got[b:b + 1, :nb + 1] - ref_o).max() <= 1e-2
        if nb == 0:  # no drafts: only the bonus token, drawn from target row 0
            assert acc[b] == 0 and vst[b] == 0
            assert 0 <= toks[b, 0] < V and (toks[b, 1:] == -1).all()
            assert newl[b] == a["prefix_lens"][b] + 1
            continue
        ref = orc.verify_chain(c["target"][b:b + 1, :nb + 1], c["draft"][b:b + 1, :nb],
                               c["draft_tokens"][b:b + 1, :nb], c["u_accept"][b:b + 1, :nb],
                               c["u_sample"][b:b + 1])
        if ref["flags"][0]:
            continue
        assert acc[b] == ref["accepted_len"][0]
        np.testing.assert_array_equal(toks[b, :nb + 1], ref["out_tokens"][0])
        assert (toks[b, nb + 1:] == -1).all()
        assert newl[b] == a["prefix_lens"][b] + acc[b] + 1


def _tree_step(a, tr, node_counts=None, seed=0):
    B, T = tr["node_tokens"].shape
    k, v = dev(a["k"]), dev(a["v"])
    ast = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    vst = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    out, acc, path, toks, newl = sv.sv_verify_step_tree_greedy(
        dev(a["q"]), k, v, dev(a["prefix_lens"]), dev(tr["parents"]), dev(tr["target"]),
        dev(tr["node_tokens"]), attn_status=ast, verify_status=vst,
        node_counts=None if node_counts is None else dev(node_counts))
    torch.cuda.synchronize()
    return (out, host(acc), host(path), host(toks), host(newl), host(k), host(v), host(ast),
            host(vst))


def _check_tree(orc, a, tr, res, sel=None):
    out, acc, path, toks, newl, k, v, ast, vst = res
    _check_attention(orc, a, out, tr["parents"], sel)
    ref = orc.verify_tree_greedy(tr["target"], tr["node_tokens"], tr["parents"])
    np.testing.assert_array_equal(acc, ref["accepted_len"])
    np.testing.assert_array_equal(path, ref["path_nodes"])
    np.testing.assert_array_equal(toks, ref["out_tokens"])
    np.testing.assert_array_equal(vst, ref["status"])
    rc = orc.compact_kv(a["k"], a["v"], a["prefix_lens"], ref["path_nodes"], ref["accepted_len"])
    np.testing.assert_array_equal(k, rc["k"])
    np.testing.assert_array_equal(v, rc["v"])
    np.testing.assert_array_equal(newl, rc["new_kv_lens"])
    return ref


def test_tree_step_medusa_full_size(orc):
    """The Medusa-tree step (B=4, L=2048, T=26, 32q/8kv, V=32000): attention in
    cluster mode, compaction inside the attention and walk kernels; every
    attention row, the paths and the compacted caches against the oracle."""
    inp = W.workload(3)
    a, tr = inp["attn"], inp["tree"]
    res = _tree_step(a, tr)
    ref = _check_tree(orc, a, tr, res)
    assert (res[7] == 0).all()
    assert ref["accepted_len"].max() > 0  # rows moved


def test_tree_step_flat_split_side_by_side(orc):
    """Many single row groups (B=24, T=16, 8 KV heads: 192 groups of 64 rows):
    the attention's flat split beside the greedy pass, and a compaction
    kernel after the join."""
    rng = np.random.default_rng(6)
    B, T = 24, 16
    par = np.stack([W.random_tree(T, 6, rng) for _ in range(B)])
    tr = W.tree_logit_inputs(B, T, 8000, par, 0.7, seed=6)
    a = W.attention_inputs(B, T, 32, 8, 128, rng.integers(0, 700, B), parents=par, seed=6,
                           unused_fill="zero")
    res = _tree_step(a, tr)
    sel = _sample_rows(rng, B, T, 32, 256)
    ref = _check_tree(orc, a, tr, res, sel)
    assert ref["accepted_len"].max() > 0


def test_tree_step_flat_split(orc):
    """Many row groups (B=16, T=64, 8 KV heads: 256 groups, two per KV head):
    the attention's flat split, the kernels one after another, and a
    compaction kernel at the end."""
    rng = np.random.default_rng(5)
    B, T = 16, 64
    par = np.stack([W.random_tree(T, 8, rng) for _ in range(B)])
    tr = W.tree_logit_inputs(B, T, 32000, par, 0.7, seed=5)
    a = W.attention_inputs(B, T, 32, 8, 128, rng.integers(0, 400, B), parents=par, seed=5,
                           unused_fill="zero")
    res = _tree_step(a, tr)
    sel = _sample_rows(rng, B, T, 32, 256)
    ref = _check_tree(orc, a, tr, res, sel)
    assert ref["accepted_len"].max() > 0


def test_tree_step_repeat_and_bad_sequence(orc):
    """Two steps in a row through one workspace (the arrival counters come
    back to zero), the second with a sequence whose tree is invalid: it is
    reported, keeps its rows and its length; the others are exact."""
    par = W.medusa_tree(26)
    for rep in range(2):
        B = 3
        pb = np.broadcast_to(par, (B, 26)).copy()
        tr = W.tree_logit_inputs(B, 26, 5000, pb, 0.8, seed=30 + rep)
        a = W.attention_inputs(B, 26, 16, 4, 128, [200, 64, 1], parents=pb, seed=30 + rep,
                               unused_fill="zero")
        if rep == 1:
            tr["parents"] = tr["parents"].copy()
            tr["parents"][1, 5] = 7  # a parent after its child
            a["parents"] = tr["parents"]
        res = _tree_step(a, tr)
        out, acc, path, toks, newl, k, v, ast, vst = res
        good = np.arange(B) != 1 if rep == 1 else np.ones(B, bool)
        ref = orc.verify_tree_greedy(tr["target"][good], tr["node_tokens"][good],
                                     tr["parents"][good])
        np.testing.assert_array_equal(acc[good], ref["accepted_len"])
        np.testing.assert_array_equal(path[good], ref["path_nodes"])
        rc = orc.compact_kv(a["k"][good], a["v"][good], a["prefix_lens"][good],
                            ref["path_nodes"], ref["accepted_len"])
        np.testing.assert_array_equal(k[good], rc["k"])
        np.testing.assert_array_equal(v[good], rc["v"])
        np.testing.assert_array_equal(newl[good], rc["new_kv_lens"])
        if rep == 1:
            assert acc[1] == -1 and vst[1] == sv.SV_ERR_BAD_INPUT and ast[1] == sv.SV_ERR_BAD_INPUT
            assert newl[1] == a["prefix_lens"][1]
            np.testing.assert_array_equal(k[1], a["k"][1])
            np.testing.assert_array_equal(v[1], a["v"][1])


def test_tree_step_ragged_node_counts(orc):
    """Node counts T_b < T: each sequence equals the oracle on its first T_b
    nodes alone (attention rows, path, compacted rows)."""
    B, T = 4, 26
    par = W.medusa_tree(T)
    pb = np.broadcast_to(par, (B, T)).copy()
    counts = np.array([26, 1, 9, 17], np.int32)
    tr = W.tree_logit_inputs(B, T, 7000, pb, 0.8, seed=40)
    a = W.attention_inputs(B, T, 32, 8, 128, [100, 5, 900, 33], parents=pb, seed=40,
                           unused_fill="zero")
    out, acc, path, toks, newl, k, v, ast, vst = _tree_step(a, tr, node_counts=counts)
    got = bf16_to_f64(host(out))
    for b in range(B):
        n = int(counts[b])
        ref_o = orc.tree_attention(a["q"][b:b + 1, :n], a["k"][b:b + 1], a["v"][b:b + 1],
                                   a["prefix_lens"][b:b + 1], pb[b:b + 1, :n], a["Hkv"],
                                   a["S_max"])
        assert np.abs(got[b:b + 1, :n] - ref_o).max() <= 1e-2
        ref = orc.verify_tree_greedy(tr["target"][b:b + 1, :n], tr["node_tokens"][b:b + 1, :n],
                                     pb[b:b + 1, :n])
        assert acc[b] == ref["accepted_len"][0]
        np.testing.assert_array_equal(path[b, :n], ref["path_nodes"][0])
        rc = orc.compact_kv(a["k"][b:b + 1], a["v"][b:b + 1], a["prefix_lens"][b:b + 1],
                            ref["path_nodes"], ref["accepted_len"])
        np.testing.assert_array_equal(k[b:b + 1], rc["k"])
        np.testing.assert_array_equal(v[b:b + 1], rc["v"])
        assert newl[b] == rc["new_kv_lens"][0]


def test_tree_step_flat_split_ragged_node_counts(orc):
    """The flat split's kernels in sequence (B=16, T=64: two row groups per KV
    head) with node counts T_b < T and NaN logits on the padding nodes' rows:
    each sequence's paths, tokens and compacted rows equal the oracle on its
    first T_b nodes alone."""
    rng = np.random.default_rng(41)
    B, T, V = 16, 64, 5000
    par = np.stack([W.random_tree(T, 8, rng) for _ in range(B)])
    counts = rng.integers(1, T + 1, B).astype(np.int32)
    counts[0], counts[1] = T, 1
    tr = W.tree_logit_inputs(B, T, V, par, 0.7, seed=41)
    for b in range(B):
        tr["target"][b, counts[b]:] = 0x7FC0  # bf16 NaN: padding rows are never read
    a = W.attention_inputs(B, T, 32, 8, 128, rng.integers(0, 300, B), parents=par, seed=41,
                           unused_fill="zero")
    out, acc, path, toks, newl, k, v, ast, vst = _tree_step(a, tr, node_counts=counts)
    for b in range(B):
        n = int(counts[b])
        ref = orc.verify_tree_greedy(tr["target"][b:b + 1, :n], tr["node_tokens"][b:b + 1, :n],
                                     par[b:b + 1, :n])
        assert acc[b] == ref["accepted_len"][0]
        np.testing.assert_array_equal(path[b, :n], ref["path_nodes"][0])
        np.testing.assert_array_equal(toks[b, :n], ref["out_tokens"][0])
        rc = orc.compact_kv(a["k"][b:b + 1], a["v"][b:b + 1], a["prefix_lens"][b:b + 1],
                            ref["path_nodes"], ref["accepted_len"])
        np.testing.assert_array_equal(k[b:b + 1], rc["k"])
        np.testing.assert_array_equal(v[b:b + 1], rc["v"])
        assert newl[b] == rc["new_kv_lens"][0]
    assert acc.max() > 0
