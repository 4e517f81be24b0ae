"""Pins of the oracle's stochastic tree acceptance (multi-draft speculative
sampling, the SpecInfer rule; "Chapitre 9 -- Décodage spéculatif" §9.2 has the
target choose among drafted paths without a rule):

- a chain-shaped tree is the chain rule, checked against the separately
  pinned chain oracle;
- the first emitted token is distributed as the target's p at the root when
  the root's children are drawn i.i.d. from q (chi-square over 2e5 trials):
  a residual that is not updated between siblings fails it;
- below the root, given the accepted path so far, the next emitted token is
  distributed as the target's p at the accepted node (a two-level tree): a
  residual carried over from the parent node fails it;
- a draft equal to the target accepts the first child at every node;
- structural invariants of the outputs."""
import numpy as np
import pytest
from scipy import special, stats

import oracle
from speculative_decoding_verification_81_gb300 import workloads as W


def _chain_as_tree(inp):
    B, N = inp["draft_tokens"].shape
    V = inp["target"].shape[-1]
    draft = np.concatenate([inp["draft"], inp["draft"][:, :1]], axis=1)  # row N: a leaf's, unused
    tok = np.concatenate([np.zeros((B, 1), np.int32), inp["draft_tokens"]], axis=1)
    ua = np.concatenate([np.full((B, 1), 0.5, np.float32), inp["u_accept"]], axis=1)
    par = np.broadcast_to(W.chain_parents(N + 1), (B, N + 1)).copy()
    return draft, tok, par, ua


@pytest.mark.parametrize("B,N,V,dtype,seed", [(64, 4, 300, "f32", 1), (40, 6, 1000, "bf16", 2)])
def test_chain_tree_equals_chain_rule(B, N, V, dtype, seed):
    inp = W.chain_inputs(B, N, V, dtype, target_sigma=2.0, draft_sigma=1.0, boost=3.0, seed=seed)
    ch = oracle.verify_chain(inp["target"], inp["draft"], inp["draft_tokens"], inp["u_accept"],
                             inp["u_sample"])
    draft, tok, par, ua = _chain_as_tree(inp)
    tr = oracle.verify_tree_stochastic(inp["target"], draft, tok, par, ua, inp["u_sample"])
    ok = (ch["flags"] == 0) & (tr["flags"] == 0)
    assert ok.mean() > 0.9
    np.testing.assert_array_equal(tr["accepted_len"][ok], ch["accepted_len"][ok])
    np.testing.assert_array_equal(tr["out_tokens"][ok], ch["out_tokens"][ok])
    for b in np.nonzero(ok)[0]:
        a = tr["accepted_len"][b]
        assert tr["path_nodes"][b, :a + 1].tolist() == list(range(a + 1))
    assert 0 < ch["accepted_len"].mean() < N


@pytest.mark.parametrize("k,draft_sigma", [(1, 1.0), (3, 1.0), (3, 3.0)])
def test_first_token_follows_target_at_root(k, draft_sigma):
    rng = np.random.default_rng(7 + k)
    V, n = 8, 200_000
    T = 1 + k  # the root and k leaf children
    z = (rng.standard_normal(V) * 1.5).astype(np.float32)
    d = (z + rng.standard_normal(V) * draft_sigma).astype(np.float32)
    p = special.softmax(z.astype(np.float64))
    q = special.softmax(d.astype(np.float64))
    target = np.broadcast_to(np.tile(z, (T, 1)), (n, T, V)).copy()
    draft = np.broadcast_to(np.tile(d, (T, 1)), (n, T, V)).copy()
    par = np.broadcast_to(np.array([-1] + [0] * k, np.int32), (n, T)).copy()
    tok = np.zeros((n, T), np.int32)
    tok[:, 1:] = rng.choice(V, size=(n, k), p=q)  # children drawn i.i.d. from q
    ua = rng.random((n, T), dtype=np.float32)
    us = rng.random(n, dtype=np.float32)
    r = oracle.verify_tree_stochastic(target, draft, tok, par, ua, us)
    first = r["out_tokens"][:, 0]
    obs = np.bincount(first, minlength=V)
    chi = stats.chisquare(obs, p * n)
    assert chi.pvalue > 1e-3, (chi, obs / n, p)
    if k > 1:  # some draws come after several rejected siblings
        assert (r["accepted_len"] == 0).mean() > 0.01


def test_equal_draft_accepts_first_children():
    rng = np.random.default_rng(3)
    B, T, V = 20, 12, 50
    par = np.stack([W.random_tree(T, 5, rng) for _ in range(B)])
    target = (rng.standard_normal((B, T, V)) * 2).astype(np.float32)
    tok = rng.integers(0, V, (B, T), dtype=np.int32)
    ua = rng.random((B, T), dtype=np.float32) * np.float32(0.999)
    r = oracle.verify_tree_stochastic(target, target, tok, par, ua,
                                      rng.random(B, dtype=np.float32))
    for b in range(B):
        node, path = 0, [0]
        while True:  # the first child of every node on the way, down to a leaf
            kids = [v for v in range(T) if par[b, v] == node]
            if not kids:
                break
            node = kids[0]
            path.append(node)
        a = r["accepted_len"][b]
        assert a == len(path) - 1
        assert r["path_nodes"][b, :a + 1].tolist() == path


def test_outputs_are_a_valid_path():
    rng = np.random.default_rng(4)
    B, T, V = 30, 20, 200
    par = np.stack([W.random_tree(T, 6, rng) for _ in range(B)])
    target = (rng.standard_normal((B, T, V)) * 2).astype(np.float32)
    draft = (target + rng.standard_normal((B, T, V))).astype(np.float32)
    tok = rng.integers(0, V, (B, T), dtype=np.int32)
    r = oracle.verify_tree_stochastic(target, draft, tok, par, rng.random((B, T), np.float32),
                                      rng.random(B, dtype=np.float32))
    for b in range(B):
        a = r["accepted_len"][b]
        path = r["path_nodes"][b]
        assert path[0] == 0 and (path[a + 1:] == -1).all()
        for d in range(1, a + 1):
            assert par[b, path[d]] == path[d - 1]
            assert r["out_tokens"][b, d - 1] == tok[b, path[d]]
        assert 0 <= r["out_tokens"][b, a] < V and (r["out_tokens"][b, a + 1:] == -1).all()


def test_bad_inputs_reported():
    rng = np.random.default_rng(5)
    B, T, V = 3, 6, 40
    par = np.broadcast_to(W.chain_parents(T), (B, T)).copy()
    target = rng.standard_normal((B, T, V)).astype(np.float32)
    draft = rng.standard_normal((B, T, V)).astype(np.float32)
    tok = rng.integers(0, V, (B, T), dtype=np.int32)
    par[1, 3] = 4          # a parent after its child
    draft[2, 2, 7] = np.nan  # a used draft row that defines no distribution
    r = oracle.verify_tree_stochastic(target, draft, tok, par, rng.random((B, T), np.float32),
                                      rng.random(B, dtype=np.float32))
    assert r["status"].tolist() == [0, 6, 6]
    assert (r["accepted_len"][1:] == -1).all()


def test_later_tokens_follow_target_below_the_root():
    """A two-level tree, two children a node, each node's children drawn
    i.i.d. from the drafter at that node, every node of a level with the same
    rows.  Given that a first-level child was accepted, the second emitted
    token follows the target at the first level, and given a second-level
    child, the third follows the target at the leaves: the residual restarts
    at every accepted node (chi-square over 2e5 trials)."""
    rng = np.random.default_rng(31)
    V, n = 6, 200_000
    par = np.array([-1, 0, 0, 1, 1, 2, 2], np.int32)
    T = len(par)
    z = [(rng.standard_normal(V) * 1.5).astype(np.float32) for _ in range(3)]
    d = [(z[k] + rng.standard_normal(V)).astype(np.float32) for k in range(2)]
    level = [0, 1, 1, 2, 2, 2, 2]
    rows_t = np.stack([z[lv] for lv in level])
    rows_d = np.stack([d[min(lv, 1)] for lv in level])  # the leaves' draft rows are not used
    p = [special.softmax(zk.astype(np.float64)) for zk in z]
    q = [special.softmax(dk.astype(np.float64)) for dk in d]
    tok = np.zeros((n, T), np.int32)
    tok[:, 1:3] = rng.choice(V, size=(n, 2), p=q[0])
    tok[:, 3:7] = rng.choice(V, size=(n, 4), p=q[1])
    r = oracle.verify_tree_stochastic(np.broadcast_to(rows_t, (n, T, V)).copy(),
                                      np.broadcast_to(rows_d, (n, T, V)).copy(), tok,
                                      np.broadcast_to(par, (n, T)).copy(),
                                      rng.random((n, T), dtype=np.float32),
                                      rng.random(n, dtype=np.float32))
    acc = r["accepted_len"]
    assert (r["status"] == 0).all() and acc.max() == 2
    for depth in (1, 2):
        sel = acc >= depth
        assert sel.mean() > 0.1, (depth, sel.mean())
        obs = np.bincount(r["out_tokens"][sel, depth], minlength=V)
        chi = stats.chisquare(obs, p[depth] * sel.sum())
        assert chi.pvalue > 1e-3, (depth, chi, obs / sel.sum(), p[depth])
