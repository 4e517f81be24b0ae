"""GPU parity of sv_compact_kv against the oracle: bit-exact caches and lengths."""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_81_gb300 as sv
from speculative_decoding_verification_81_gb300 import workloads as W
from gpu_util import dev, host

pytestmark = pytest.mark.gpu


def _run(orc, inp, paths, acc, alias=False):
    ref = orc.compact_kv(inp["k"], inp["v"], inp["prefix_lens"], paths, acc)
    k, v = dev(inp["k"]), dev(inp["v"])
    pl = dev(inp["prefix_lens"])
    st = torch.full((len(acc),), -7, dtype=torch.int32, device="cuda")
    newl = sv.sv_compact_kv(k, v, pl, dev(acc), None if paths is None else dev(paths),
                            new_kv_lens=pl if alias else None, seq_status=st)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(k), ref["k"])
    np.testing.assert_array_equal(host(v), ref["v"])
    np.testing.assert_array_equal(host(newl), ref["new_kv_lens"])
    np.testing.assert_array_equal(host(st), ref["status"])
    return ref


def _random_paths(rng, B, T, par):
    acc = np.zeros(B, np.int32)
    paths = np.full((B, T), -1, np.int32)
    for b in range(B):
        node = int(rng.integers(0, T))
        path = [node]
        while par[b, path[-1]] >= 0:
            path.append(int(par[b, path[-1]]))
        path = path[::-1]
        acc[b] = len(path) - 1
        paths[b, :len(path)] = path
    return paths, acc


@pytest.mark.parametrize("alias", [False, True])
def test_compact_tree_paths(orc, alias):
    rng = np.random.default_rng(1)
    B, T, Hkv, D = 6, 64, 4, 128
    par = np.stack([W.random_tree(T, 12, rng) for _ in range(B)])
    inp = W.attention_inputs(B, T, 8, Hkv, D, rng.integers(0, 300, B), parents=par, seed=1,
                             unused_fill="zero")
    paths, acc = _random_paths(rng, B, T, par)
    _run(orc, inp, paths, acc, alias)


def test_compact_long_path_spans_batches(orc):
    """A 50-row path (more than one staged batch) with rows moving far."""
    B, T, Hkv, D = 2, 64, 2, 64
    inp = W.attention_inputs(B, T, 2, Hkv, D, [100, 3], seed=2, unused_fill="zero")
    paths = np.full((B, T), -1, np.int32)
    paths[0, :50] = [0] + list(range(14, 63))
    paths[1, :40] = [0] + list(range(3, 42))
    _run(orc, inp, paths, np.array([49, 39], np.int32))


def test_compact_chain_and_errors(orc):
    inp = W.attention_inputs(4, 9, 4, 2, 128, [10, 20, 0, 5], seed=3, unused_fill="zero")
    _run(orc, inp, None, np.array([8, 0, 3, -1], np.int32))
    paths = np.array([[0, 2, 1, -1], [0, 1, 2, 3], [1, 2, -1, -1], [0, 3, -1, -1]], np.int32)
    ref = _run(orc, inp, paths, np.array([2, 3, 1, 1], np.int32))
    assert ref["status"].tolist() == [sv.SV_ERR_BAD_INPUT, 0, sv.SV_ERR_BAD_INPUT, 0]


def test_compact_workload3_full(orc):
    inp = W.workload(3)
    a = inp["attn"]
    rng = np.random.default_rng(3)
    paths, acc = _random_paths(rng, a["B"], a["T"], a["parents"])
    _run(orc, a, paths, acc)
