"""Pins for the oracle's softmax statistics and stochastic chain acceptance.

The acceptance rule (accept draft x ~ q with probability min(1, p(x)/q(x)),
else draw from the normalised residual (p - q)+, bonus from the last
distribution) makes the emitted tokens distributed exactly as the target's
own sampling ("Chapitre 9 -- Décodage spéculatif" §9.1; "Parallel Decoding"
glossary, "Garantie de qualité").  These tests pin the oracle to that
guarantee by exact enumeration over a low-discrepancy grid of uniforms, by a
chi-square test on random trials, by the closed form of the acceptance
probability, and by special cases whose outcome is forced.
"""
import numpy as np
import pytest
from scipy import special, stats

from speculative_decoding_verification_81_gb300 import workloads as W


def _softmax64(x):
    return special.softmax(np.asarray(x, np.float64), axis=-1)


def _vals(arr):
    return W.bf16_bits_to_f32(arr) if arr.dtype == np.uint16 else arr


# ---------------------------------------------------------------- row stats

def test_row_stats_constant_row(orc):
    for V in (1, 7, 1024):
        m, s, am = orc.row_stats(np.full(V, 1.25, np.float32))
        assert m == 1.25 and am == 0
        assert s == pytest.approx(V, rel=0, abs=0)  # exp(0) summed V times


def test_row_stats_against_library(orc):
    rng = np.random.default_rng(1)
    for V, dt in ((1024, "f32"), (32000, "bf16"), (5, "bf16")):
        x = (rng.standard_normal(V) * 3).astype(np.float32)
        row = W.f32_to_bf16_bits(x) if dt == "bf16" else x
        xv = _vals(row).astype(np.float64)
        m, s, am = orc.row_stats(row)
        assert m == xv.max()
        assert am == int(np.argmax(xv))  # numpy returns the first maximum
        assert np.log(s) + m == pytest.approx(special.logsumexp(xv), rel=1e-14)


def test_row_stats_argmax_ties_take_smallest_index(orc):
    row = np.zeros(40, np.float32)
    row[[7, 13, 31]] = 2.0
    assert orc.row_stats(row)[2] == 7
    bits = W.f32_to_bf16_bits(np.array([0.5, 3.0, 3.0, -1.0], np.float32))
    assert orc.row_stats(bits)[2] == 1


# ------------------------------------------------- acceptance: enumeration

def _fib_lattice(n_index=26):
    """Rank-1 Fibonacci lattice in [0,1)^2 shifted to cell midpoints."""
    f = [1, 1]
    while len(f) < n_index + 1:
        f.append(f[-1] + f[-2])
    M, g = f[n_index], f[n_index - 1]
    k = np.arange(M, dtype=np.int64)
    u1 = (k + 0.5) / M
    u2 = (((k * g) % M) + 0.5) / M
    return u1.astype(np.float32), u2.astype(np.float32), M


def _enumerate_chain_n1(orc, target, draft):
    """Run the oracle over every draft token x (weight q(x)) and every point
    of a 2-D lattice of (u_accept, u_sample).  Returns the exact weighted
    distribution of out[0], the acceptance probability and the distribution
    of out[1] given acceptance."""
    V = target.shape[-1]
    q = _softmax64(_vals(draft)[0])
    ua, us, M = _fib_lattice()
    p_out0 = np.zeros(V)
    p_acc = 0.0
    p_bonus = np.zeros(V)
    for x in range(V):
        if q[x] == 0.0:
            continue
        B = M
        res = orc.verify_chain(np.broadcast_to(target, (B,) + target.shape),
                               np.broadcast_to(draft, (B,) + draft.shape),
                               np.full((B, 1), x, np.int32), ua[:, None], us)
        assert ((res["accepted_len"] >= 0) & (res["accepted_len"] <= 1)).all()
        w = q[x] / M
        p_out0 += w * np.bincount(res["out_tokens"][:, 0], minlength=V)
        acc = res["accepted_len"] == 1
        p_acc += w * acc.sum()
        p_bonus += w * np.bincount(res["out_tokens"][acc, 1], minlength=V)
    return p_out0, p_acc, p_bonus / max(p_acc, 1e-300)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_enumeration_emitted_token_is_target_distribution(orc, seed):
    """Exhaustive over draft tokens, lattice over uniforms (V = 6, N = 1):
    out[0] ~ p_0 (accept-or-resample), P(accept) = sum_v min(p_0, q_0), and
    the bonus after acceptance ~ p_1."""
    rng = np.random.default_rng(seed)
    V = 6
    target = (rng.standard_normal((2, V)) * 1.5).astype(np.float32)
    draft = (target[:1] + rng.standard_normal((1, V)) * 1.0).astype(np.float32)
    p0, p1 = _softmax64(target[0]), _softmax64(target[1])
    q0 = _softmax64(draft[0])
    out0, pacc, bonus = _enumerate_chain_n1(orc, target, draft)
    # lattice discrepancy is O(log M / M) with M = 121393; observed errors
    # are below 1e-5
    np.testing.assert_allclose(out0, p0, rtol=0, atol=5e-5)
    assert pacc == pytest.approx(np.minimum(p0, q0).sum(), abs=2e-5)
    np.testing.assert_allclose(bonus, p1, rtol=0, atol=1e-4)


def test_enumeration_detects_wrong_rules(orc):
    """Sanity check of the enumeration's power: the plausible wrong rules
    (residual p instead of (p-q)+, or resampling from q) move out[0] by far
    more than the tolerance used above."""
    rng = np.random.default_rng(0)
    V = 6
    target = (rng.standard_normal((2, V)) * 1.5).astype(np.float64)
    draft = target[:1] + rng.standard_normal((1, V))
    p0, q0 = _softmax64(target[0]), _softmax64(draft[0])
    beta = np.minimum(p0, q0).sum()
    accepted_part = np.minimum(p0, q0)
    wrong_p = accepted_part + (1 - beta) * p0
    wrong_q = accepted_part + (1 - beta) * q0
    assert np.abs(wrong_p - p0).max() > 2e-2
    assert np.abs(wrong_q - p0).max() > 2e-2


# ------------------------------------------------- acceptance: statistics

def _trials(orc, target, draft, n, seed, batch=20000):
    """n independent speculative iterations with fresh draft tokens x_i ~ q_i
    and fresh uniforms.  Returns accepted_len [n] and out_tokens [n, N+1]."""
    rng = np.random.default_rng(seed)
    N, V = draft.shape
    q = _softmax64(_vals(draft))
    accs, outs = [], []
    for s in range(0, n, batch):
        B = min(batch, n - s)
        tok = np.stack([rng.choice(V, size=B, p=q[i]) for i in range(N)], 1).astype(np.int32)
        ua = rng.random((B, N), dtype=np.float32)
        us = rng.random(B, dtype=np.float32)
        r = orc.verify_chain(np.broadcast_to(target, (B,) + target.shape),
                             np.broadcast_to(draft, (B,) + draft.shape), tok, ua, us)
        accs.append(r["accepted_len"])
        outs.append(r["out_tokens"])
    return np.concatenate(accs), np.concatenate(outs)


def _chisq_pvalue(tokens, p):
    V = len(p)
    obs = np.bincount(tokens, minlength=V).astype(np.float64)
    exp = p * len(tokens)
    big = exp >= 5
    o = np.append(obs[big], obs[~big].sum())
    e = np.append(exp[big], exp[~big].sum())
    if e[-1] == 0:
        o, e = o[:-1], e[:-1]
    return stats.chisquare(o, e).pvalue


def test_chi_square_v64(orc):
    """10^6 speculative iterations at V = 64, N = 2: at every position the
    emitted token (accepted draft or resample/bonus) follows p_i, and the
    acceptance rate matches sum_v min(p, q) within 5 sigma."""
    rng = np.random.default_rng(11)
    V, N, n = 64, 2, 1_000_000
    target = (rng.standard_normal((N + 1, V)) * 2.0).astype(np.float32)
    draft = (target[:N] + rng.standard_normal((N, V)) * 1.0).astype(np.float32)
    acc, out = _trials(orc, target, draft, n, seed=12)
    assert ((acc >= 0) & (acc <= N)).all()
    p = _softmax64(target)
    q = _softmax64(draft)
    reached = np.ones(n, bool)
    for i in range(N + 1):
        pv = _chisq_pvalue(out[reached, i], p[i])
        assert pv > 1e-3, (i, pv)
        if i < N:
            beta = np.minimum(p[i], q[i]).sum()
            k = reached.sum()
            rate = (acc[reached] > i).mean()
            assert abs(rate - beta) < 5 * np.sqrt(beta * (1 - beta) / k), (i, rate, beta)
            reached = acc > i
    # layout invariant: x_0..x_{a-1}, the final token, then -1 padding
    for a in range(N + 1):
        rows = out[acc == a]
        assert (rows[:, :a + 1] >= 0).all() and (rows[:, a + 1:] == -1).all()


def test_identical_distributions_accept_everything(orc):
    """p = q => every draft is accepted (u*q < p for u < 1), a = N, and the
    bonus token follows p_N."""
    rng = np.random.default_rng(21)
    V, N = 32, 4
    target = W.f32_to_bf16_bits((rng.standard_normal((N + 1, V)) * 2).astype(np.float32))
    draft = target[:N].copy()
    acc, out = _trials(orc, target, draft, 200_000, seed=22)
    assert (acc == N).all()
    assert _chisq_pvalue(out[:, N], _softmax64(_vals(target)[N])) > 1e-3


def test_disjoint_supports_always_reject(orc):
    """q puts no mass where p does => a = 0 and the resample follows p_0."""
    V, N = 8, 3
    target = np.full((N + 1, V), -1.0e4, np.float32)
    draft = np.full((N, V), -1.0e4, np.float32)
    target[:, :4] = np.array([0.3, -0.7, 1.1, 0.0], np.float32)
    draft[:, 4:] = np.array([0.2, 0.9, -0.4, 0.5], np.float32)
    acc, out = _trials(orc, target, draft, 200_000, seed=23)
    assert (acc == 0).all()
    assert _chisq_pvalue(out[:, 0], _softmax64(target[0])) > 1e-3


def test_one_hot_target_is_deterministic(orc):
    """A one-hot p at every position forces the output to the target's token."""
    V, N = 16, 4
    rng = np.random.default_rng(24)
    hot = rng.integers(0, V, N + 1)
    target = np.zeros((N + 1, V), np.float32)
    target[np.arange(N + 1), hot] = 1.0e4
    draft = (rng.standard_normal((N, V)) * 2).astype(np.float32)
    acc, out = _trials(orc, target, draft, 20_000, seed=25)
    for n in range(len(acc)):
        a = acc[n]
        assert (out[n, :a + 1] == hot[:a + 1]).all()


def test_near_tie_and_degenerate_flags(orc):
    # q = (1/2, 1/2); p(0) = 1/4 up to float rounding; u = 1/2 => u*q(0) ~ p(0)
    target = np.array([[[np.log(1.0 / 3.0), 0.0], [0.0, 0.0]]], np.float32)
    draft = np.array([[[0.0, 0.0]]], np.float32)
    r = orc.verify_chain(target, draft, np.array([[0]]), np.array([[0.5]], np.float32),
                         np.array([0.3], np.float32))
    assert r["flags"][0] & orc.FLAG_ACCEPT_NEAR_TIE
    assert r["probs"][0, 0, 0] == pytest.approx(0.25, rel=1e-6)
    assert r["probs"][0, 0, 1] == 0.5
    # draft token with p = q = 0: rejected, residual is zero, fall back to p
    target = np.array([[[0.0, 1.0, -1e4], [0.0, 0.0, 0.0]]], np.float32)
    draft = np.array([[[0.0, 1.0, -1e4]]], np.float32)
    r = orc.verify_chain(target, draft, np.array([[2]]), np.array([[0.9]], np.float32),
                         np.array([0.99], np.float32))
    assert r["accepted_len"][0] == 0
    assert r["flags"][0] & orc.FLAG_DEGENERATE_RESIDUAL
    assert r["out_tokens"][0].tolist() == [1, -1]


def test_bad_draft_token_sets_status(orc):
    target = np.zeros((2, 3, 4), np.float32)
    draft = np.zeros((2, 2, 4), np.float32)
    r = orc.verify_chain(target, draft, np.array([[0, 4], [1, 2]]),
                         np.full((2, 2), 0.5, np.float32), np.full(2, 0.5, np.float32))
    assert r["status"].tolist() == [orc.ERR_BAD_INPUT, orc.OK]
    assert r["accepted_len"][0] == -1 and (r["out_tokens"][0] == -1).all()
    assert r["accepted_len"][1] == 2  # p = q: all accepted


def test_probabilities_definition(orc):
    """probs = (p_i(x_i), q_i(x_i)) match softmax from scipy."""
    inp = W.chain_inputs(B=3, N=4, V=500, dtype="bf16", seed=31)
    r = orc.verify_chain(inp["target"], inp["draft"], inp["draft_tokens"], inp["u_accept"],
                         inp["u_sample"])
    p = _softmax64(_vals(inp["target"]))
    q = _softmax64(_vals(inp["draft"]))
    for b in range(3):
        for i in range(4):
            x = inp["draft_tokens"][b, i]
            assert r["probs"][b, i, 0] == pytest.approx(p[b, i, x], rel=1e-12)
            assert r["probs"][b, i, 1] == pytest.approx(q[b, i, x], rel=1e-12)


def test_non_finite_rows_are_bad_input(orc):
    """A row with NaN, +inf or only -inf logits defines no distribution."""
    target = np.zeros((4, 3, 5), np.float32)
    draft = np.zeros((4, 2, 5), np.float32)
    target[0, 1, 2] = np.nan
    draft[1, 0, 4] = np.inf
    target[2, 2, :] = -np.inf
    r = orc.verify_chain(target, draft, np.zeros((4, 2), np.int32),
                         np.full((4, 2), 0.5, np.float32), np.full(4, 0.5, np.float32))
    assert r["status"].tolist() == [orc.ERR_BAD_INPUT] * 3 + [orc.OK]
    assert (r["accepted_len"][:3] == -1).all() and (r["out_tokens"][:3] == -1).all()
