"""Pins for the oracle's greedy tree acceptance and KV compaction.

Greedy acceptance keeps the longest path of the draft tree on which every
candidate equals the target's own choice at its parent, then appends the
target's choice at the end of that path ("Parallel Decoding" glossary,
"L'attention en arbre : la brique commune": the longest accepted path becomes
the generated sequence; "Chapitre 9 -- Décodage spéculatif" §9.1: longest
agreeing prefix, then the target's own choice).  The tests compare against a
brute force over every root->node path, the chain special case written as a
left-to-right prefix scan, and the compaction invariants (glossary, "Limites
du parallel decoding": the enlarged KV cache of the branches).
"""
import itertools

import numpy as np
import pytest

from speculative_decoding_verification_81_gb300 import workloads as W


def _brute_force(target_vals, tokens, parents):
    """Enumerate every node's root->node path; keep paths whose every edge
    agrees; the deepest wins, smallest node index among equal depths."""
    T = len(parents)
    amax = target_vals.argmax(-1)
    best = None
    for node in range(T):
        path = [node]
        while parents[path[-1]] >= 0:
            path.append(int(parents[path[-1]]))
        path = path[::-1]
        if all(tokens[path[d]] == amax[path[d - 1]] for d in range(1, len(path))):
            key = (-(len(path) - 1), node)
            if best is None or key < best[0]:
                best = (key, path)
    path = best[1]
    out = [int(tokens[n]) for n in path[1:]] + [int(amax[path[-1]])]
    return len(path) - 1, path, out


@pytest.mark.parametrize("seed", range(6))
def test_greedy_matches_brute_force(orc, seed):
    rng = np.random.default_rng(seed)
    B, V = 8, 5  # tiny vocabulary: many agreements and many argmax ties
    T = int(rng.integers(2, 13))
    par = np.stack([W.random_tree(T, int(rng.integers(1, 6)), rng) for _ in range(B)])
    inp = W.tree_logit_inputs(B, T, V, par, p_match=0.7, sigma=1.0, seed=seed)
    r = orc.verify_tree_greedy(inp["target"], inp["node_tokens"], par)
    vals = W.bf16_bits_to_f32(inp["target"])
    _, depth = orc.ancestor_mask(par[0], T)
    for b in range(B):
        a, path, out = _brute_force(vals[b], inp["node_tokens"][b], par[b])
        assert r["accepted_len"][b] == a
        assert r["path_nodes"][b, :a + 1].tolist() == path
        assert (r["path_nodes"][b, a + 1:] == -1).all()
        assert r["out_tokens"][b, :a + 1].tolist() == out
        assert (r["out_tokens"][b, a + 1:] == -1).all()


def test_exhaustive_tiny_trees(orc):
    """Every parent array with T = 4, every token assignment over V = 2."""
    V, T = 2, 4
    target = np.array([[0.0, 1.0], [1.0, 0.0], [0.0, 1.0], [1.0, 1.0]], np.float32)
    trees = [np.array((-1,) + p, np.int32) for p in itertools.product(*[range(i) for i in range(1, T)])]
    toks = [np.array((0,) + t, np.int32) for t in itertools.product(range(V), repeat=T - 1)]
    for par in trees:
        for tok in toks:
            r = orc.verify_tree_greedy(target[None], tok[None], par[None])
            a, path, out = _brute_force(target, tok, par)
            assert r["accepted_len"][0] == a
            assert r["path_nodes"][0, :a + 1].tolist() == path
            assert r["out_tokens"][0, :a + 1].tolist() == out


def test_chain_is_longest_agreeing_prefix(orc):
    rng = np.random.default_rng(3)
    B, T, V = 16, 9, 4
    par = np.broadcast_to(W.chain_parents(T), (B, T)).copy()
    inp = W.tree_logit_inputs(B, T, V, par, p_match=0.8, seed=3)
    r = orc.verify_tree_greedy(inp["target"], inp["node_tokens"], par)
    amax = W.bf16_bits_to_f32(inp["target"]).argmax(-1)
    for b in range(B):
        a = 0
        while a + 1 < T and inp["node_tokens"][b, a + 1] == amax[b, a]:
            a += 1
        assert r["accepted_len"][b] == a
        assert r["path_nodes"][b, :a + 1].tolist() == list(range(a + 1))
        expect = inp["node_tokens"][b, 1:a + 1].tolist() + [int(amax[b, a])]
        assert r["out_tokens"][b, :a + 1].tolist() == expect


def test_greedy_invariants_on_workload_trees(orc):
    for k in (3, 5):
        cfg = W.WORKLOADS[k]
        inp = W.workload(k, B=4, V=300, L=8)
        par = inp["tree"]["parents"]
        r = orc.verify_tree_greedy(inp["tree"]["target"], inp["tree"]["node_tokens"], par)
        for b in range(4):
            _, depth = orc.ancestor_mask(par[b], cfg["T"])
            a = r["accepted_len"][b]
            assert 0 <= a <= depth.max()
            path = r["path_nodes"][b, :a + 1]
            assert path[0] == 0 and all(par[b, path[d]] == path[d - 1] for d in range(1, a + 1))
            assert (r["out_tokens"][b, :a] == inp["tree"]["node_tokens"][b, path[1:]]).all()


def test_greedy_bad_parents_status(orc):
    target = np.zeros((2, 3, 4), np.float32)
    r = orc.verify_tree_greedy(target, np.zeros((2, 3), np.int32),
                               np.array([[-1, 0, 2], [-1, 0, 0]], np.int32))
    assert r["status"].tolist() == [orc.ERR_BAD_INPUT, orc.OK]
    assert r["accepted_len"][0] == -1


# -------------------------------------------------------------- compaction

def test_compaction_invariants(orc):
    rng = np.random.default_rng(4)
    B, Hkv, D, T = 3, 2, 16, 10
    pl = np.array([5, 0, 17], np.int32)
    inp = W.attention_inputs(B, T, 4, Hkv, D, pl, parents=None, seed=4, unused_fill="zero")
    paths = np.full((B, T), -1, np.int32)
    acc = np.array([3, 0, 6], np.int32)
    paths[0, :4] = [0, 2, 5, 9]
    paths[1, :1] = [0]
    paths[2, :7] = [0, 1, 2, 4, 5, 7, 8]
    r = orc.compact_kv(inp["k"], inp["v"], pl, paths, acc)
    assert r["new_kv_lens"].tolist() == [9, 1, 24]
    for b in range(B):
        L, a = int(pl[b]), int(acc[b])
        for name in ("k", "v"):
            before, after = inp[name][b], r[name][b]
            assert np.array_equal(after[:, :L], before[:, :L])
            for d in range(a + 1):
                assert np.array_equal(after[:, L + d], before[:, L + paths[b, d]])
            assert np.array_equal(after[:, L + a + 1:], before[:, L + a + 1:])


def test_compaction_chain_moves_nothing(orc):
    inp = W.attention_inputs(2, 9, 4, 2, 16, [7, 3], seed=5, unused_fill="zero")
    r = orc.compact_kv(inp["k"], inp["v"], inp["prefix_lens"], None, np.array([4, 8], np.int32))
    assert np.array_equal(r["k"], inp["k"]) and np.array_equal(r["v"], inp["v"])
    assert r["new_kv_lens"].tolist() == [12, 12]


def test_compaction_rejects_bad_paths(orc):
    inp = W.attention_inputs(3, 4, 2, 1, 8, [2, 2, 2], S_max=8, seed=6, unused_fill="zero")
    paths = np.array([[0, 2, 1, -1], [0, 6, -1, -1], [0, 1, -1, -1], [1, 2, -1, -1]], np.int32)
    acc = np.array([2, 1, -1, 1], np.int32)
    inp = W.attention_inputs(4, 4, 2, 1, 8, [2, 2, 2, 2], S_max=8, seed=6, unused_fill="zero")
    r = orc.compact_kv(inp["k"], inp["v"], inp["prefix_lens"], paths, acc)
    assert r["status"].tolist() == [orc.ERR_BAD_INPUT, orc.ERR_BAD_INPUT, orc.OK, orc.ERR_BAD_INPUT]
    assert r["new_kv_lens"].tolist() == [2, 2, 2, 2]
    assert np.array_equal(r["k"], inp["k"])


def test_medusa_tree_fixture():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "medusa_tree_26.txt")
    rows = [ln for ln in open(path) if ln.strip() and not ln.startswith("#")]
    fixture = [int(x) for x in rows[0].split()]
    assert W.medusa_tree(26).tolist() == fixture
