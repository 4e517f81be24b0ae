"""The seeded input recipe (workloads.py) checked against facts that do not
come from the module itself: torch's bf16 conversion, closed-form sampling
probabilities, the Medusa tree's depth profile and the workload table."""
import numpy as np
import pytest
import torch
from scipy import stats

from speculative_decoding_verification_81_gb300 import workloads as W


def _depths(par):
    d = np.zeros(len(par), np.int64)
    for i in range(1, len(par)):
        d[i] = d[par[i]] + 1
    return d


def _within(frac, p, n, k=5.0):
    return abs(frac - p) < k * np.sqrt(p * (1 - p) / n)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(100_000).astype(np.float32) * np.float32(3.0),
        (rng.standard_normal(10_000) * 1e30).astype(np.float32),
        (rng.standard_normal(10_000) * 1e-39).astype(np.float32),  # subnormals
        np.array([0.0, -0.0, np.inf, -np.inf, 3.4e38, -3.4e38], np.float32),
        # halfway cases between neighbouring bf16 values: ties go to even
        np.array([0x3F808000, 0x3F818000, 0xBF808000, 0x3F808001], np.uint32).view(np.float32),
    ])
    ours = W.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    assert ours[-4:].tolist() == [0x3F80, 0x3F82, 0xBF80, 0x3F81]
    back = torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(W.bf16_bits_to_f32(ours), back)


def test_medusa_tree_depth_profile_and_branching():
    """26 kept nodes of the 4-3-2-1 tree: 1, 4, 7, 8 and 6 nodes at depths
    0..4, at most 4, 3, 2, 1 children at depths 0..3, breadth-first order."""
    par = W.medusa_tree(26)
    d = _depths(par)
    assert np.bincount(d).tolist() == [1, 4, 7, 8, 6]
    kids = np.bincount(par[1:], minlength=26)
    for u in range(26):
        assert kids[u] <= (4, 3, 2, 1, 0)[d[u]]
    assert (np.diff(d) >= 0).all()


def test_random_tree_structure_and_uniform_parent():
    rng = np.random.default_rng(2)
    for _ in range(200):
        par = W.random_tree(64, 8, rng)
        assert par[0] == -1 and all(0 <= par[i] < i for i in range(1, 64))
        assert _depths(par).max() <= 8
    assert (W.random_tree(20, 1, rng)[1:] == 0).all()  # depth 1: a star
    # node 3's parent is uniform over nodes 0..2 when no depth bound binds
    n = 6000
    obs = np.bincount([W.random_tree(4, 8, rng)[3] for _ in range(n)], minlength=3)
    assert stats.chisquare(obs, np.full(3, n / 3)).pvalue > 1e-3
    # node 2 may hang under node 1 only while depth 1 is below the bound
    assert all(W.random_tree(3, 1, rng)[2] == 0 for _ in range(50))
    obs = np.bincount([W.random_tree(3, 2, rng)[2] for _ in range(n)], minlength=2)
    assert stats.chisquare(obs, np.full(2, n / 2)).pvalue > 1e-3


def test_drafter_draws_from_softmax_of_the_draft_row():
    """Zero noise and one token boosted by b: the drafter picks the boosted
    token with probability e^b / (e^b + V - 1)."""
    B, V, b = 20_000, 50, 3.0
    c = W.chain_inputs(B, 1, V, "f32", target_sigma=0.0, draft_sigma=0.0, boost=b, seed=3)
    boosted = c["draft"][:, 0].argmax(-1)
    frac = (c["draft_tokens"][:, 0] == boosted).mean()
    assert _within(frac, np.exp(b) / (np.exp(b) + V - 1), B)


def test_tree_children_are_drawn_at_their_parent():
    """Each node's draft row has its own boosted token; children follow
    their parent's row, not their own."""
    B, V, b = 10_000, 40, 3.0
    s = W.stree_inputs(B, 3, V, np.array([-1, 0, 0], np.int32), "f32", target_sigma=0.0,
                       draft_sigma=0.0, boost=b, seed=4)
    p_boost = np.exp(b) / (np.exp(b) + V - 1)
    at_parent = s["draft"][:, 0].argmax(-1)
    for v in (1, 2):
        own = s["draft"][:, v].argmax(-1)
        tok = s["node_tokens"][:, v]
        assert _within((tok == at_parent).mean(), p_boost, B)
        differ = own != at_parent
        assert (tok[differ] == own[differ]).mean() < 2 * (1 - p_boost) / (V - 1)
    assert (s["node_tokens"][:, 0] == 0).all()


def test_tree_node_tokens_copy_the_parent_argmax_with_p_match():
    rng = np.random.default_rng(5)
    par = np.stack([W.random_tree(12, 4, rng) for _ in range(300)])
    all_match = W.tree_logit_inputs(300, 12, 16, par, p_match=1.0, dtype="f32", seed=6)
    am = all_match["target"].argmax(-1)
    for bb in range(300):
        for i in range(1, 12):
            assert all_match["node_tokens"][bb, i] == am[bb, par[bb, i]]
    none = W.tree_logit_inputs(300, 12, 16, par, p_match=0.0, dtype="f32", seed=7)
    obs = np.bincount(none["node_tokens"][:, 1:].ravel(), minlength=16)
    assert stats.chisquare(obs).pvalue > 1e-3


def test_attention_inputs_poison_unused_slots():
    a = W.attention_inputs(3, 5, 8, 2, 128, [7, 0, 20], S_max=40, seed=8)
    f = W.bf16_bits_to_f32
    for b, L in enumerate([7, 0, 20]):
        assert np.isnan(f(a["k"][b, :, L + 5:])).all() and np.isnan(f(a["v"][b, :, L + 5:])).all()
        assert np.isfinite(f(a["k"][b, :, :L + 5])).all() and np.isfinite(f(a["v"][b, :, :L + 5])).all()
    assert np.isfinite(f(a["q"])).all() and a["q"].shape == (3, 5, 8, 128)


@pytest.mark.parametrize("k,fields", [
    (3, dict(B=4, L=2048, T=26, V=32000, Hq=32, Hkv=8, D=128, tree="medusa")),
    (4, dict(B=32, N=8, L=4096, V=128256, Hq=32, Hkv=8, D=128)),
    (5, dict(B=16, L=8192, T=64, V=128256, Hq=32, Hkv=8, D=128, tree="random", max_depth=8)),
])
def test_workload_table(k, fields):
    cfg = W.WORKLOADS[k]
    for key, val in fields.items():
        assert cfg[key] == val, (k, key)


def test_workloads_are_deterministic_and_seeded():
    a, b = W.workload(2, B=2, V=3000), W.workload(2, B=2, V=3000)
    c = W.workload(2, B=2, V=3000, seed=1)
    for key in ("target", "draft", "draft_tokens", "u_accept", "u_sample"):
        np.testing.assert_array_equal(a[key], b[key])
    assert not np.array_equal(a["target"], c["target"])
    assert a["seed"] == 1002
    # sigma of the recipe: target ~ N(0, 3^2) away from the boosted token
    t = W.bf16_bits_to_f32(a["target"]).astype(np.float64)
    assert abs(np.median(np.abs(t)) / 0.6745 - 3.0) < 0.05


@pytest.mark.parametrize("page_size", [8, 16, 128])
def test_paged_cache_round_trip(page_size):
    """Scattering a cache into pages and gathering it back is the identity;
    the page table is a permutation of distinct pages; spare pages and page
    slots past S_max stay NaN."""
    a = W.attention_inputs(3, 4, 8, 2, 128, [30, 5, 50], S_max=70, seed=9, unused_fill="zero")
    kp, vp, table = W.paged_cache(a["k"], a["v"], page_size, seed=10, spare_pages=3)
    np.testing.assert_array_equal(W.gather_paged(kp, table, 70), a["k"])
    np.testing.assert_array_equal(W.gather_paged(vp, table, 70), a["v"])
    assert len(np.unique(table)) == table.size and table.min() >= 0 and table.max() < len(kp)
    spare = np.setdiff1d(np.arange(len(kp)), table.ravel())
    assert len(spare) == 3 and np.isnan(W.bf16_bits_to_f32(kp[spare])).all()
    tail = 70 % page_size
    if tail:  # the last page of each sequence holds S_max's remainder, then NaN
        last = table[:, -1]
        assert np.isnan(W.bf16_bits_to_f32(kp[last][:, :, tail:])).all()
