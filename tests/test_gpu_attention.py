"""GPU parity of sv_tree_attention against the oracle: max-abs error at most
1e-2 against the double-precision oracle on bf16 inputs."""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_81_gb300 as sv
from speculative_decoding_verification_81_gb300 import workloads as W
from gpu_util import bf16_to_f64, dev, host

pytestmark = pytest.mark.gpu
TOL = 1e-2


def _gpu(inp, parents):
    st = torch.full((inp["B"],), -7, dtype=torch.int32, device="cuda")
    out = sv.sv_tree_attention(dev(inp["q"]), dev(inp["k"]), dev(inp["v"]),
                               dev(inp["prefix_lens"]),
                               None if parents is None else dev(parents), seq_status=st)
    torch.cuda.synchronize()
    return bf16_to_f64(host(out)), host(st)


def _check(orc, inp, parents, sel=None):
    got, st = _gpu(inp, parents)
    ref = orc.tree_attention(inp["q"], inp["k"], inp["v"], inp["prefix_lens"], parents,
                             inp["Hkv"], inp["S_max"], sel=sel)
    if sel is None:
        err = np.abs(got - ref).max()
    else:
        s = np.asarray(sel)
        err = np.abs(got[s[:, 0], s[:, 1], s[:, 2]] - ref[s[:, 0], s[:, 1], s[:, 2]]).max()
    assert np.isfinite(err) and err <= TOL, err
    return got, st


@pytest.mark.parametrize("B,T,Hq,Hkv,L,tree,seed", [
    (2, 9, 32, 8, [300, 77], "chain", 1),      # chain, ragged prefixes
    (3, 13, 8, 2, [200, 64, 0], "random", 2),  # empty prefix, tile-aligned prefix
    (1, 1, 8, 8, [1000], "chain", 3),          # plain decode, G = 1
    (2, 64, 8, 1, [130, 5], "random", 4),      # T = 64, G = 8: two row groups
    (2, 26, 32, 8, [257, 1000], "medusa", 5),  # Medusa tree
    (4, 5, 16, 4, [63, 64, 65, 129], "random", 6),  # prefixes around a tile edge
])
def test_attention_small(orc, B, T, Hq, Hkv, L, tree, seed):
    rng = np.random.default_rng(seed)
    if tree == "chain":
        par = None
    elif tree == "medusa":
        par = np.broadcast_to(W.medusa_tree(26), (B, T)).copy()
    else:
        par = np.stack([W.random_tree(T, 6, rng) for _ in range(B)])
    inp = W.attention_inputs(B, T, Hq, Hkv, 128, L, parents=par, seed=seed)
    got, st = _check(orc, inp, par)
    assert (st == 0).all()


def test_attention_chain_equals_explicit_chain_parents(orc):
    inp = W.attention_inputs(2, 9, 32, 8, 128, [500, 33], seed=7)
    a, _ = _gpu(inp, None)
    b, _ = _gpu(inp, np.broadcast_to(W.chain_parents(9), (2, 9)).copy())
    np.testing.assert_array_equal(a, b)


def test_attention_bad_sequences_skipped(orc):
    inp = W.attention_inputs(3, 4, 8, 2, 128, [10, 20, 30], S_max=64, seed=8)
    inp["prefix_lens"][1] = 61                   # 61 + 4 > S_max
    par = np.broadcast_to(W.chain_parents(4), (3, 4)).copy()
    par[2, 2] = 3                                # parent after child
    got, st = _gpu(inp, par)
    assert st.tolist() == [0, sv.SV_ERR_BAD_INPUT, sv.SV_ERR_BAD_INPUT]
    ref = orc.tree_attention(inp["q"][:1], inp["k"][:1], inp["v"][:1], inp["prefix_lens"][:1],
                             par[:1], 2, 64)
    assert np.abs(got[:1] - ref).max() <= TOL


def _sample(rng, B, T, Hq, n):
    return np.stack([rng.integers(0, B, n), rng.integers(0, T, n), rng.integers(0, Hq, n)], 1)


def test_attention_workload3_full(orc):
    inp = W.workload(3)["attn"]
    _check(orc, inp, inp["parents"])


def test_attention_workload4_sampled(orc):
    inp = W.workload(4)["attn"]
    rng = np.random.default_rng(4)
    sel = np.concatenate([_sample(rng, 32, 9, 32, 96),
                          np.array([[31, 8, 31], [0, 0, 0], [17, 4, 12]])])
    _check(orc, inp, None, sel)


def test_attention_flat_split_128_row_groups_sampled(orc):
    """26 chain nodes x 4 heads = 104 query rows per KV head: one 128-row group
    per (sequence, KV head) with padding rows, and enough groups (256) for the
    flat split over persistent CTAs, whose groups straddle CTAs and merge."""
    rng = np.random.default_rng(11)
    B, T = 32, 26
    L = [int(x) for x in rng.integers(900, 1100, B)]
    inp = W.attention_inputs(B, T, 32, 8, 128, L, seed=11)
    sel = np.concatenate([_sample(rng, B, T, 32, 64),
                          np.array([[B - 1, T - 1, 31], [0, 0, 0], [5, 25, 3]])])
    _check(orc, inp, None, sel)


def test_attention_workload5_sampled(orc):
    inp = W.workload(5)["attn"]
    rng = np.random.default_rng(5)
    _check(orc, inp, inp["parents"], _sample(rng, 16, 64, 32, 48))


def test_attention_repeatable():
    inp = W.attention_inputs(2, 9, 32, 8, 128, [1000, 2000], seed=9)
    a, _ = _gpu(inp, None)
    b, _ = _gpu(inp, None)
    np.testing.assert_array_equal(a, b)
