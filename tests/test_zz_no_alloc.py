"""sv_verify_chain_noalloc, the chain-acceptance entry point for callers that
cannot allocate device memory where they call the library (a plugin whose
host owns all device memory and exposes no allocator, a real-time loop that
must not take the device-wide synchronisation of cudaMalloc and cudaFree).
It takes no workspace and keeps its scratch in a fixed array of the library.

Checked through the C ABI: two calls in a row give exactly the outputs of
sv_verify_chain on the same inputs (the same kernels run) and agree with the
oracle (tokens and lengths bit-exact except the oracle's flagged near-ties,
p and q within 1e-5 relative), and a shape whose scratch exceeds the fixed
array is refused before anything is launched.  This file is collected last
so that a failure here leaves every other test already run; it also passes
on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import speculative_decoding_verification_81_gb300 as sv
from speculative_decoding_verification_81_gb300 import workloads as W
from speculative_decoding_verification_81_gb300 import api

pytestmark = pytest.mark.gpu


def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def _noalloc_call(t, d, tok, ua, us, acc, out, probs, status):
    """Direct C ABI call: the caller passes every output, the library allocates nothing."""
    L = sv.lib()
    B, N1, V = t.shape
    dt = sv.SV_BF16 if t.dtype == torch.bfloat16 else sv.SV_F32
    P = lambda x: ctypes.c_void_p(x.data_ptr())
    return L.sv_verify_chain_noalloc(P(t), P(d), dt, P(tok), P(ua), P(us), B, N1 - 1, V, P(acc),
                                     P(out), P(probs), P(status),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("case", ["llama_vocab", "fused_step_logits", "fp32_small"])
def test_noalloc_matches_workspace_entry_point(orc, case):
    if case == "llama_vocab":
        inp = W.workload(2)
    elif case == "fused_step_logits":
        inp = W.chain_inputs(32, 8, 128256, "bf16", 3.0, 1.0, 8.0, seed=1004)
    else:
        inp = W.chain_inputs(5, 6, 1000, "f32", 2.0, 1.0, 0.0, seed=3)
    t, d = _dev(inp["target"]), _dev(inp["draft"])
    tok, ua, us = _dev(inp["draft_tokens"]), _dev(inp["u_accept"]), _dev(inp["u_sample"])
    B, N = inp["draft_tokens"].shape
    assert sv.sv_workspace_size(sv.SV_OP_VERIFY_CHAIN, B, N, t.shape[2],
                                sv.SV_BF16 if t.dtype == torch.bfloat16 else sv.SV_F32) \
        <= api.SV_NOALLOC_SCRATCH_BYTES

    ref_probs = torch.zeros(B, N, 2, dtype=torch.float32, device="cuda")
    ref_status = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    ref_acc, ref_out = sv.sv_verify_chain(t, d, tok, ua, us, probs_out=ref_probs,
                                          seq_status=ref_status)
    torch.cuda.synchronize()
    for call in range(2):  # the fixed array keeps the previous call's contents
        acc = torch.full((B,), -9, dtype=torch.int32, device="cuda")
        out = torch.full((B, N + 1), -9, dtype=torch.int32, device="cuda")
        probs = torch.zeros(B, N, 2, dtype=torch.float32, device="cuda")
        status = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        rc = _noalloc_call(t, d, tok, ua, us, acc, out, probs, status)
        assert rc == sv.SV_OK, sv.status_string(rc)
        torch.cuda.synchronize()
        assert torch.equal(acc, ref_acc), call
        assert torch.equal(out, ref_out), call
        assert torch.equal(status, ref_status), call
        rel = ((probs - ref_probs).abs() / ref_probs.abs().clamp_min(1e-30)).max().item()
        assert rel <= 1e-5, (call, rel)
        # and against the oracle itself
        o = orc.verify_chain(inp["target"], inp["draft"], inp["draft_tokens"], inp["u_accept"],
                             inp["u_sample"])
        ok = o["flags"] == 0
        np.testing.assert_array_equal(acc.cpu().numpy()[ok], o["accepted_len"][ok])
        np.testing.assert_array_equal(out.cpu().numpy()[ok], o["out_tokens"][ok])
        np.testing.assert_array_equal(status.cpu().numpy(), o["status"])
        good = o["status"] == 0
        rp, gp = o["probs"][good], probs.cpu().numpy()[good].astype(np.float64)
        big = rp > 1e-30
        assert (np.abs(gp[big] - rp[big]) / rp[big]).max(initial=0.0) <= 1e-5, call


def test_noalloc_binding_and_oversize_refusal():
    inp = W.workload(1)
    t, d = _dev(inp["target"]), _dev(inp["draft"])
    B, N = inp["draft_tokens"].shape
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, N + 1, dtype=torch.int32, device="cuda")
    sv.api.sv_verify_chain_noalloc(t, d, _dev(inp["draft_tokens"]), _dev(inp["u_accept"]),
                                   _dev(inp["u_sample"]), acc, out)
    ref_acc, ref_out = sv.sv_verify_chain(t, d, _dev(inp["draft_tokens"]), _dev(inp["u_accept"]),
                                          _dev(inp["u_sample"]))
    torch.cuda.synchronize()
    assert torch.equal(acc, ref_acc) and torch.equal(out, ref_out)
    # a shape whose scratch exceeds the fixed array: refused, nothing launched
    Bbig, Nbig, Vbig = 4096, 8, 128256
    assert sv.sv_workspace_size(sv.SV_OP_VERIFY_CHAIN, Bbig, Nbig, Vbig, sv.SV_BF16) > \
        api.SV_NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: the size check comes first
    rc = sv.lib().sv_verify_chain_noalloc(fake, fake, sv.SV_BF16, fake, fake, fake, Bbig, Nbig,
                                          Vbig, fake, fake, None, None, None)
    assert rc == sv.SV_ERR_WORKSPACE
