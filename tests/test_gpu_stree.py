"""GPU parity of sv_verify_tree_stochastic against the oracle.

Bar: accepted lengths, paths and emitted tokens bit-exact, except sequences
the oracle flags: an acceptance near-tie (|u q N - r| < 1e-5 of the larger)
is not compared; after a sampling near-tie (u S within 1e-6 S of a
cumulative-sum boundary) the path is compared and the drawn token is not.
"""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_81_gb300 as sv
from speculative_decoding_verification_81_gb300 import workloads as W
from gpu_util import dev, host

pytestmark = pytest.mark.gpu


def _run(inp, parents=True):
    B = inp["node_tokens"].shape[0]
    st = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    acc, path, out = sv.sv_verify_tree_stochastic(
        dev(inp["target"]), dev(inp["draft"]), dev(inp["node_tokens"]),
        dev(inp["parents"]) if parents else None, dev(inp["u_accept"]), dev(inp["u_sample"]),
        seq_status=st)
    torch.cuda.synchronize()
    return host(acc), host(path), host(out), host(st)


def _check(orc, inp, max_flag_frac=0.25):
    ref = orc.verify_tree_stochastic(inp["target"], inp["draft"], inp["node_tokens"],
                                     inp["parents"], inp["u_accept"], inp["u_sample"])
    acc, path, out, st = _run(inp)
    np.testing.assert_array_equal(st, ref["status"])
    compared = 0
    for b in range(len(acc)):
        f = ref["flags"][b]
        if f & 1:  # an acceptance near-tie
            continue
        assert acc[b] == ref["accepted_len"][b], b
        np.testing.assert_array_equal(path[b], ref["path_nodes"][b])
        a = max(int(acc[b]), 0)
        n_cmp = a if f & 2 else out.shape[1]
        np.testing.assert_array_equal(out[b, :n_cmp], ref["out_tokens"][b, :n_cmp])
        compared += 1
    assert compared >= (1 - max_flag_frac) * len(acc)
    return ref, acc


@pytest.mark.parametrize("B,T,V,dtype,tree,seed", [
    (6, 12, 1000, "bf16", "random", 1),
    (4, 26, 32000, "bf16", "medusa", 2),    # the Medusa tree at the Llama-2 vocabulary
    (5, 9, 1001, "f32", "random", 3),       # unaligned f32 rows
    (3, 64, 128256, "bf16", "random", 4),   # EAGLE-style: 64 nodes, the Llama-3 vocabulary
    (2, 40, 20000, "f32", "wide", 5),       # eight children at the root: many sibling passes
])
def test_stochastic_tree_matches_oracle(orc, B, T, V, dtype, tree, seed):
    rng = np.random.default_rng(seed)
    if tree == "medusa":
        par = W.medusa_tree(T)
    elif tree == "wide":
        par = np.array([-1] + [0] * 8 + [1 + (i % 8) for i in range(T - 9)], np.int32)
    else:
        par = np.stack([W.random_tree(T, 8, rng) for _ in range(B)])
    inp = W.stree_inputs(B, T, V, par, dtype, target_sigma=2.0, draft_sigma=1.0, boost=4.0,
                         seed=seed)
    ref, acc = _check(orc, inp)
    assert (ref["status"] == 0).all()


def test_chain_shaped_tree_equals_chain_call():
    """A chain-shaped tree (parents NULL) gives sv_verify_chain's outputs."""
    B, N, V = 16, 6, 5000
    c = W.chain_inputs(B, N, V, "bf16", target_sigma=2.0, draft_sigma=1.0, boost=4.0, seed=8)
    t, d = dev(c["target"]), dev(c["draft"])
    acc_c, out_c = sv.sv_verify_chain(t, d, dev(c["draft_tokens"]), dev(c["u_accept"]),
                                      dev(c["u_sample"]))
    draft_tree = np.concatenate([c["draft"], c["draft"][:, :1]], axis=1)
    tok = np.concatenate([np.zeros((B, 1), np.int32), c["draft_tokens"]], axis=1)
    ua = np.concatenate([np.full((B, 1), 0.5, np.float32), c["u_accept"]], axis=1)
    acc_t, path_t, out_t = sv.sv_verify_tree_stochastic(t, dev(draft_tree), dev(tok), None,
                                                       dev(ua), dev(c["u_sample"]))
    torch.cuda.synchronize()
    acc_c, out_c, acc_t, out_t = host(acc_c), host(out_c), host(acc_t), host(out_t)
    np.testing.assert_array_equal(acc_t, acc_c)
    # the drawn token comes from the same weights through a different summation
    # order; every accepted prefix is identical
    for b in range(B):
        a = acc_c[b]
        np.testing.assert_array_equal(out_t[b, :a], out_c[b, :a])
        assert host(path_t)[b, :a + 1].tolist() == list(range(a + 1))


def test_first_token_follows_target_on_gpu():
    """Independent of the oracle: 100k GPU trials, a root with three children
    drawn i.i.d. from q; the first emitted token follows p (chi-square)."""
    from scipy import special, stats
    rng = np.random.default_rng(21)
    V, n, k = 64, 100_000, 3
    T = 1 + k
    z = (rng.standard_normal(V) * 1.5).astype(np.float32)
    dd = (z + rng.standard_normal(V)).astype(np.float32)
    p = special.softmax(z.astype(np.float64))
    q = special.softmax(dd.astype(np.float64))
    inp = dict(target=np.broadcast_to(np.tile(z, (T, 1)), (n, T, V)).copy(),
               draft=np.broadcast_to(np.tile(dd, (T, 1)), (n, T, V)).copy(),
               parents=np.broadcast_to(np.array([-1, 0, 0, 0], np.int32), (n, T)).copy(),
               node_tokens=np.concatenate([np.zeros((n, 1), np.int32),
                                           rng.choice(V, size=(n, k), p=q).astype(np.int32)], 1),
               u_accept=rng.random((n, T), dtype=np.float32),
               u_sample=rng.random(n, dtype=np.float32))
    acc, path, out, st = _run(inp)
    assert (st == 0).all()
    obs = np.bincount(out[:, 0], minlength=V)
    e = p * n
    big = e >= 5
    o_b, e_b = obs[big], e[big]
    if (~big).any():  # the rare tokens pooled into one bin
        o_b, e_b = np.append(o_b, obs[~big].sum()), np.append(e_b, e[~big].sum())
    pv = stats.chisquare(o_b, e_b * (o_b.sum() / e_b.sum())).pvalue
    assert pv > 1e-3, pv


def test_bad_inputs_reported(orc):
    rng = np.random.default_rng(9)
    B, T, V = 4, 8, 700
    par = np.stack([W.random_tree(T, 4, rng) for _ in range(B)])
    inp = W.stree_inputs(B, T, V, par, "f32", seed=9)
    inp["parents"][1, 5] = 6                      # a parent after its child
    inp["node_tokens"][2, 3] = V                  # a token out of range
    inp["draft"][3, 0, 5] = np.nan                # the root's draft row is used
    ref = orc.verify_tree_stochastic(inp["target"], inp["draft"], inp["node_tokens"],
                                     inp["parents"], inp["u_accept"], inp["u_sample"])
    acc, path, out, st = _run(inp)
    assert st.tolist() == ref["status"].tolist() == [0, 6, 6, 6]
    assert (acc[1:] == -1).all() and (path[1:] == -1).all() and (out[1:] == -1).all()
