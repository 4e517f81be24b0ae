"""Paged KV cache (a per-sequence page table over fixed-size pages): the
paged attention gives bitwise the results of the contiguous one and matches
the oracle on the gathered cache; paged compaction moves the same rows."""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_81_gb300 as sv
from speculative_decoding_verification_81_gb300 import workloads as W
from gpu_util import bf16_to_f64, dev, host

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.mark.parametrize("page_size,B,T,Hq,Hkv,L,tree,seed", [
    (16, 3, 9, 32, 8, [300, 1000, 77], "chain", 1),    # small pages: several per key tile
    (64, 2, 26, 32, 8, [257, 640], "medusa", 2),
    (128, 3, 13, 8, 2, [200, 0, 129], "random", 3),    # one page per key tile
    (256, 2, 64, 8, 1, [700, 5], "random", 4),         # pages larger than a tile, two row groups
    (8, 2, 5, 16, 4, [63, 130], "chain", 5),           # smallest page
])
def test_paged_attention_matches_contiguous_and_oracle(orc, page_size, B, T, Hq, Hkv, L, tree,
                                                       seed):
    rng = np.random.default_rng(seed)
    if tree == "chain":
        par = None
    elif tree == "medusa":
        par = np.broadcast_to(W.medusa_tree(26), (B, T)).copy()
    else:
        par = np.stack([W.random_tree(T, 6, rng) for _ in range(B)])
    inp = W.attention_inputs(B, T, Hq, Hkv, 128, L, parents=par, seed=seed)
    kp, vp, table = W.paged_cache(inp["k"], inp["v"], page_size, seed=seed)
    table = table.copy()
    for b in range(B):  # entries past the pages a sequence uses may hold anything
        table[b, -(-(L[b] + T) // page_size):] = -1 - b
    st = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    got = sv.sv_tree_attention_paged(dev(inp["q"]), dev(kp), dev(vp), dev(table),
                                     dev(inp["prefix_lens"]), None if par is None else dev(par),
                                     seq_status=st)
    ref_gpu = sv.sv_tree_attention(dev(inp["q"]), dev(inp["k"]), dev(inp["v"]),
                                   dev(inp["prefix_lens"]), None if par is None else dev(par))
    torch.cuda.synchronize()
    assert (host(st) == 0).all()
    np.testing.assert_array_equal(host(got), host(ref_gpu))
    ref = orc.tree_attention(inp["q"], inp["k"], inp["v"], inp["prefix_lens"], par, Hkv,
                             inp["S_max"])
    err = np.abs(bf16_to_f64(host(got)) - ref).max()
    assert np.isfinite(err) and err <= TOL, err


def test_paged_attention_bad_page_id_reported():
    B, T = 2, 9
    inp = W.attention_inputs(B, T, 8, 2, 128, [300, 100], seed=6)
    kp, vp, table = W.paged_cache(inp["k"], inp["v"], 64, seed=6)
    table = table.copy()
    table[1, 0] = kp.shape[0] + 5  # sequence 1's first page does not exist
    st = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    sv.sv_tree_attention_paged(dev(inp["q"]), dev(kp), dev(vp), dev(table),
                               dev(inp["prefix_lens"]), seq_status=st)
    torch.cuda.synchronize()
    assert host(st).tolist() == [sv.SV_OK, sv.SV_ERR_BAD_INPUT]


@pytest.mark.parametrize("page_size", [16, 128])
def test_paged_compaction_moves_the_same_rows(orc, page_size):
    B, Hkv, D, T = 4, 2, 128, 12
    rng = np.random.default_rng(7)
    par = np.stack([W.random_tree(T, 5, rng) for _ in range(B)])
    inp = W.attention_inputs(B, T, 8, Hkv, D, [100, 255, 0, 31], parents=par, seed=7,
                             unused_fill="zero")
    # accepted paths: root to a random node of each tree
    path = np.full((B, T), -1, np.int32)
    acc = np.zeros(B, np.int32)
    for b in range(B):
        node = int(rng.integers(0, T))
        chain = []
        while node >= 0:
            chain.append(node)
            node = int(par[b, node])
        chain = chain[::-1]
        path[b, :len(chain)] = chain
        acc[b] = len(chain) - 1
    kp, vp, table = W.paged_cache(inp["k"], inp["v"], page_size, seed=8, nan_fill=False)
    kc, vc = dev(inp["k"]), dev(inp["v"])
    kpd, vpd = dev(kp), dev(vp)
    st = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    new_c = sv.sv_compact_kv(kc, vc, dev(inp["prefix_lens"]), dev(acc), dev(path))
    new_p = sv.sv_compact_kv_paged(kpd, vpd, dev(table), dev(inp["prefix_lens"]), dev(acc),
                                   dev(path), seq_status=st)
    torch.cuda.synchronize()
    assert (host(st) == 0).all()
    np.testing.assert_array_equal(host(new_p), host(new_c))
    S_max = inp["S_max"]
    np.testing.assert_array_equal(W.gather_paged(host(kpd), table, S_max), host(kc))
    np.testing.assert_array_equal(W.gather_paged(host(vpd), table, S_max), host(vc))
    ref = orc.compact_kv(inp["k"], inp["v"], inp["prefix_lens"], path, acc)
    for b in range(B):
        n = int(ref["new_kv_lens"][b])
        np.testing.assert_array_equal(host(kc)[b, :, :n], ref["k"][b, :, :n])
