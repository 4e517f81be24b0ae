"""GPU parity of sv_verify_chain and sv_verify_tree_greedy against the oracle.

Bar: accepted lengths, emitted tokens and tree paths bit-exact, except
sequences the oracle flags as near-ties (|u*q - p| < 1e-6 p at a decision,
or u*S within 1e-6 S of a cumulative-sum boundary), which are counted, not
failed; p(x_i), q(x_i) within 1e-5 relative in fp32.
"""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_81_gb300 as sv
from speculative_decoding_verification_81_gb300 import workloads as W
from gpu_util import dev, host

pytestmark = pytest.mark.gpu


def _run_chain(inp):
    t, d = dev(inp["target"]), dev(inp["draft"])
    B, N = inp["draft_tokens"].shape
    probs = torch.full((B, N, 2), -1.0, dtype=torch.float32, device="cuda")
    status = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    acc, out = sv.sv_verify_chain(t, d, dev(inp["draft_tokens"]), dev(inp["u_accept"]),
                                  dev(inp["u_sample"]), probs_out=probs, seq_status=status)
    torch.cuda.synchronize()
    return host(acc), host(out), host(probs), host(status)


def _check_chain(orc, inp, max_flag_frac=0.02):
    ref = orc.verify_chain(inp["target"], inp["draft"], inp["draft_tokens"], inp["u_accept"],
                           inp["u_sample"])
    acc, out, probs, status = _run_chain(inp)
    assert (status == ref["status"]).all()
    flagged = ref["flags"] != 0
    ok = ~flagged
    np.testing.assert_array_equal(acc[ok], ref["accepted_len"][ok])
    np.testing.assert_array_equal(out[ok], ref["out_tokens"][ok])
    good = ref["status"] == 0
    rp = ref["probs"][good]
    gp = probs[good].astype(np.float64)
    big = rp > 1e-30
    rel = np.abs(gp[big] - rp[big]) / rp[big]
    assert rel.max(initial=0.0) <= 1e-5, rel.max()
    assert np.abs(gp[~big] - rp[~big]).max(initial=0.0) <= 1e-30
    assert flagged.mean() <= max_flag_frac, flagged.sum()
    return ref, acc, out


def test_chain_workload1_fp32(orc):
    inp = W.workload(1)
    _check_chain(orc, inp)


def test_chain_workload2_llama_vocab(orc):
    inp = W.workload(2)
    _check_chain(orc, inp)


def test_chain_workload4_logits_full_size(orc):
    """The chain-verification half of the fused step at full size:
    B=32, N=8, V=128256 bf16."""
    cfg = W.WORKLOADS[4]
    inp = W.chain_inputs(cfg["B"], cfg["N"], cfg["V"], "bf16", cfg["target_sigma"],
                         cfg["draft_sigma"], cfg["boost"], seed=1004)
    ref, acc, _ = _check_chain(orc, inp)
    assert 0 <= acc.min() and acc.max() <= cfg["N"]


@pytest.mark.parametrize("B,N,V,dtype,seed", [
    (3, 1, 8, "f32", 1),            # tiny vocabulary, single draft
    (5, 7, 1000, "bf16", 2),        # V*2 not a multiple of 16: scalar row path
    (4, 3, 16389, "bf16", 3),       # one element past a streaming chunk
    (2, 63, 3000, "f32", 4),        # maximum N
    (17, 4, 50000, "bf16", 5),      # ragged batch, several residual chunks
    (6, 5, 4097, "f32", 6),         # f32, unaligned rows
])
def test_chain_random_shapes(orc, B, N, V, dtype, seed):
    inp = W.chain_inputs(B, N, V, dtype, target_sigma=2.0, draft_sigma=1.0, boost=4.0, seed=seed)
    _check_chain(orc, inp)


def test_chain_residual_forms_agree_bitwise():
    """The residual draw's two forms -- a thread-block cluster per sequence
    (whole-GPU calls whose clusters fit with room: B = 8 here) and the arrival
    counter with the last CTA (B = 32 sequences of 16 chunks, near the
    device's cluster capacity; and the fused step's acceptance) -- take the
    same arithmetic, so the same sequences give the same bits whichever runs.
    Sequences 8..15 of a B = 32 batch against the same 8 sequences alone."""
    cfg = W.WORKLOADS[4]
    inp = W.chain_inputs(32, cfg["N"], cfg["V"], "bf16", cfg["target_sigma"], cfg["draft_sigma"],
                         cfg["boost"], seed=1011)
    # rejections at every position, and bonus draws where all are accepted
    inp["u_accept"][8:12] = np.float32(1.0 - 2.0 ** -24)
    inp["draft"][12:14] = inp["target"][12:14, :cfg["N"]]
    full = _run_chain(inp)
    part = _run_chain({k: inp[k][8:16] for k in ("target", "draft", "draft_tokens", "u_accept",
                                                 "u_sample")})
    for a, b in zip(full, part):
        np.testing.assert_array_equal(a[8:16], b)


def test_chain_all_accepted_and_all_rejected(orc):
    inp = W.chain_inputs(8, 4, 2000, "bf16", target_sigma=2.0, draft_sigma=1.0, boost=0.0, seed=9)
    same = dict(inp, draft=inp["target"][:, :4].copy())          # p = q: every draft accepted
    ref, acc, out = _check_chain(orc, same)
    assert (acc == 4).all()
    far = dict(inp)                                               # u = 1 - 2^-24: rejections
    far["u_accept"] = np.full_like(inp["u_accept"], np.float32(1.0 - 2.0 ** -24))
    _check_chain(orc, far)


def test_chain_bad_inputs_reported_per_sequence(orc):
    inp = W.chain_inputs(4, 3, 700, "f32", 2.0, 1.0, 0.0, seed=10)
    inp["draft_tokens"][1, 2] = 700                     # token out of range
    inp["target"][2, 1, 5] = np.nan                      # non-finite row
    acc, out, probs, status = _run_chain(inp)
    assert status.tolist() == [0, sv.SV_ERR_BAD_INPUT, sv.SV_ERR_BAD_INPUT, 0]
    assert (acc[[1, 2]] == -1).all() and (out[[1, 2]] == -1).all()
    _check_chain(orc, inp)


def test_chain_distribution_on_gpu():
    """Independent of the oracle: 200k GPU trials at V = 64, N = 2; the first
    emitted token follows p_0 (chi-square) and P(accept_0) = sum min(p, q)."""
    from scipy import special, stats
    rng = np.random.default_rng(77)
    V, N, n = 64, 2, 200_000
    target = (rng.standard_normal((N + 1, V)) * 2.0).astype(np.float32)
    draft = (target[:N] + rng.standard_normal((N, V))).astype(np.float32)
    p = special.softmax(target.astype(np.float64), -1)
    q = special.softmax(draft.astype(np.float64), -1)
    tok = np.stack([rng.choice(V, size=n, p=q[i]) for i in range(N)], 1).astype(np.int32)
    inp = dict(target=np.broadcast_to(target, (n, N + 1, V)).copy(),
               draft=np.broadcast_to(draft, (n, N, V)).copy(), draft_tokens=tok,
               u_accept=rng.random((n, N), dtype=np.float32), u_sample=rng.random(n, dtype=np.float32))
    acc, out, _, _ = _run_chain(inp)
    obs = np.bincount(out[:, 0], minlength=V)
    e = p[0] * n
    big = e >= 5
    pv = stats.chisquare(np.append(obs[big], obs[~big].sum()), np.append(e[big], e[~big].sum())).pvalue
    assert pv > 1e-3
    beta = np.minimum(p[0], q[0]).sum()
    assert abs((acc > 0).mean() - beta) < 5 * np.sqrt(beta * (1 - beta) / n)


# ------------------------------------------------------------------ tree greedy

def _check_tree(orc, tinp):
    ref = orc.verify_tree_greedy(tinp["target"], tinp["node_tokens"], tinp["parents"])
    status = torch.full((tinp["target"].shape[0],), -7, dtype=torch.int32, device="cuda")
    acc, path, out = sv.sv_verify_tree_greedy(dev(tinp["target"]), dev(tinp["node_tokens"]),
                                              dev(tinp["parents"]), seq_status=status)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(status), ref["status"])
    np.testing.assert_array_equal(host(acc), ref["accepted_len"])
    np.testing.assert_array_equal(host(path), ref["path_nodes"])
    np.testing.assert_array_equal(host(out), ref["out_tokens"])
    return ref


@pytest.mark.parametrize("B,N,V,dtype,seed", [
    (8, 8, 32000, "bf16", 11),     # the chain workload's draft length, Llama vocabulary
    (32, 8, 128256, "bf16", 12),   # the fused chain step's shapes
    (5, 63, 1000, "f32", 13),      # longest chain, unaligned f32 rows
])
def test_greedy_chain_parents_null(orc, B, N, V, dtype, seed):
    """Greedy chain verification: parents NULL is the chain parent_i = i - 1
    (the oracle gets the explicit chain)."""
    inp = W.tree_logit_inputs(B, N + 1, V, W.chain_parents(N + 1), p_match=0.85, sigma=2.0,
                              dtype=dtype, seed=seed)
    ref = orc.verify_tree_greedy(inp["target"], inp["node_tokens"], inp["parents"])
    acc, path, out = sv.sv_verify_tree_greedy(dev(inp["target"]), dev(inp["node_tokens"]), None)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(acc), ref["accepted_len"])
    np.testing.assert_array_equal(host(path), ref["path_nodes"])
    np.testing.assert_array_equal(host(out), ref["out_tokens"])
    assert 0 < ref["accepted_len"].max()


def test_tree_workload3_logits(orc):
    inp = W.workload(3)
    ref = _check_tree(orc, inp["tree"])
    assert ref["accepted_len"].max() >= 1


def test_tree_workload5_logits_full_size(orc):
    inp = W.tree_logit_inputs(16, 64, 128256,
                              np.stack([W.random_tree(64, 8, np.random.default_rng([1005, i]))
                                        for i in range(16)]), 0.6, seed=1005)
    _check_tree(orc, inp)


@pytest.mark.parametrize("B,T,V,dtype,seed", [
    (6, 1, 50, "bf16", 1),       # root only
    (9, 12, 5, "bf16", 2),       # tiny vocabulary: argmax ties everywhere
    (4, 40, 1001, "f32", 3),     # unaligned f32 rows
    (3, 1024, 64, "bf16", 4),    # maximum T
    (5, 30, 40000, "bf16", 5),   # several chunks per row
])
def test_tree_random_shapes(orc, B, T, V, dtype, seed):
    rng = np.random.default_rng(seed)
    par = np.stack([W.random_tree(T, int(rng.integers(1, 10)), rng) for _ in range(B)])
    inp = W.tree_logit_inputs(B, T, V, par, p_match=0.8, sigma=1.0, dtype=dtype, seed=seed)
    _check_tree(orc, inp)


def test_tree_bf16_ties_take_smallest_index(orc):
    T, V = 4, 300
    target = np.zeros((1, T, V), np.uint16)
    target[0, :, [17, 250]] = W.f32_to_bf16_bits(np.array([5.0], np.float32))[0]
    inp = dict(target=target, node_tokens=np.array([[0, 17, 17, 250]], np.int32),
               parents=np.array([[-1, 0, 1, 2]], np.int32))
    ref = _check_tree(orc, inp)
    assert ref["accepted_len"][0] == 2


def test_tree_bad_parents_reported(orc):
    inp = W.tree_logit_inputs(3, 5, 100, W.chain_parents(5), 0.9, seed=11)
    inp["parents"][1, 3] = 3
    inp["node_tokens"][2, 4] = -5
    ref = _check_tree(orc, inp)
    assert ref["status"].tolist() == [0, sv.SV_ERR_BAD_INPUT, sv.SV_ERR_BAD_INPUT]


def test_repeated_calls_reuse_workspace(orc):
    """Counters in the workspace return to zero: back-to-back calls agree."""
    inp = W.workload(2)
    r1 = _run_chain(inp)
    r2 = _run_chain(inp)
    for a, b in zip(r1, r2):
        np.testing.assert_array_equal(a, b)


def test_chain_statistics_timeout_reported():
    """A statistics pass whose bounded wait gave up raises a flag in the
    workspace (after the per-sequence arrival counters); the decisions then
    report SV_ERR_TIMEOUT for every sequence instead of deciding on records
    that were never written.  The flag is raised here by the host, no wait is
    made to run out; re-zeroing the workspace clears it."""
    inp = W.chain_inputs(4, 3, 5000, "bf16", 2.0, 1.0, 4.0, seed=41)
    B, N = inp["draft_tokens"].shape
    ws = torch.zeros(sv.sv_workspace_size(sv.SV_OP_VERIFY_CHAIN, B, N, 5000, sv.SV_BF16, 0, 0),
                     dtype=torch.uint8, device="cuda")
    ws.view(torch.int32)[2 * B] = 1
    st = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    args = [dev(inp[n]) for n in ("target", "draft", "draft_tokens", "u_accept", "u_sample")]
    acc, out = sv.sv_verify_chain(*args, seq_status=st, ws=ws)
    torch.cuda.synchronize()
    assert (host(st) == sv.SV_ERR_TIMEOUT).all()
    assert (host(acc) == -1).all() and (host(out) == -1).all()
    ws.zero_()
    acc, out = sv.sv_verify_chain(*args, seq_status=st, ws=ws)
    torch.cuda.synchronize()
    assert (host(st) == 0).all() and (host(acc) >= 0).all()


def test_tree_statistics_timeout_reported():
    """The same flag for greedy tree verification (aligned rows: the streaming
    argmax pass): every sequence reports SV_ERR_TIMEOUT with -1 outputs."""
    B, T, V = 3, 9, 4096
    inp = W.tree_logit_inputs(B, T, V, W.chain_parents(T), 0.9, seed=42)
    ws = torch.zeros(sv.sv_workspace_size(sv.SV_OP_VERIFY_TREE_GREEDY, B, T, V, sv.SV_BF16, 0, 0),
                     dtype=torch.uint8, device="cuda")
    ws.view(torch.int32)[2 * B] = 1
    st = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    args = [dev(inp[n]) for n in ("target", "node_tokens", "parents")]
    acc, path, out = sv.sv_verify_tree_greedy(*args, seq_status=st, ws=ws)
    torch.cuda.synchronize()
    assert (host(st) == sv.SV_ERR_TIMEOUT).all()
    assert (host(acc) == -1).all() and (host(path) == -1).all() and (host(out) == -1).all()
    ws.zero_()
    acc, path, out = sv.sv_verify_tree_greedy(*args, seq_status=st, ws=ws)
    torch.cuda.synchronize()
    assert (host(st) == 0).all() and (host(acc) >= 0).all()
