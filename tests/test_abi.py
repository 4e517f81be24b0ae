"""The C ABI without a GPU: the library loads, exports every entry point its
header declares, and rejects invalid host arguments with the documented
status before launching anything."""
import ctypes
import os
import re

import pytest

import speculative_decoding_verification_81_gb300 as sv
from speculative_decoding_verification_81_gb300 import build as svbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specverify.h")


@pytest.fixture(scope="module")
def L():
    svbuild.build()
    return sv.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sv_[a-z_]+)\s*\(", text)))


def test_header_declares_the_api():
    names = _declared()
    assert set(names) == set(sv.api.EXPORTS), names


def test_library_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), name
        assert isinstance(getattr(L, name), ctypes._CFuncPtr)


def test_version_and_status_strings(L):
    assert L.sv_version() >= 100
    for code in range(7):
        assert sv.status_string(code).startswith("SV_")
    assert "unknown" in sv.status_string(99)


FAKE = ctypes.c_void_p(0x10000)        # never dereferenced: every case fails validation first
MISALIGNED = ctypes.c_void_p(0x10004)


def _chain(L, **kw):
    a = dict(t=FAKE, d=FAKE, dt=sv.SV_BF16, tok=FAKE, lens=None, ua=FAKE, us=FAKE, B=2, N=4,
             V=1000, acc=FAKE, out=FAKE, probs=None, st=None, ws=None, wsb=0)
    a.update(kw)
    return L.sv_verify_chain(a["t"], a["d"], a["dt"], a["tok"], a["lens"], a["ua"], a["us"],
                             a["B"], a["N"],
                             a["V"], a["acc"], a["out"], a["probs"], a["st"], a["ws"], a["wsb"],
                             None)


def test_verify_chain_host_validation(L):
    assert _chain(L, t=None) == sv.SV_ERR_INVALID_ARG
    assert _chain(L, out=None) == sv.SV_ERR_INVALID_ARG
    assert _chain(L, B=0) == sv.SV_ERR_INVALID_ARG
    assert _chain(L, N=0) == sv.SV_ERR_INVALID_ARG
    assert _chain(L, V=-3) == sv.SV_ERR_INVALID_ARG
    assert _chain(L, dt=7) == sv.SV_ERR_INVALID_ARG
    assert _chain(L, t=MISALIGNED) == sv.SV_ERR_INVALID_ARG
    assert _chain(L, N=64) == sv.SV_ERR_UNSUPPORTED
    assert _chain(L) == sv.SV_ERR_WORKSPACE  # no workspace
    assert _chain(L, lens=FAKE) == sv.SV_ERR_WORKSPACE  # draft lengths are checked on the device
    need = L.sv_workspace_size(sv.SV_OP_VERIFY_CHAIN, 2, 4, 1000, sv.SV_BF16, 0, 0, 0)
    assert need > 0
    assert _chain(L, ws=FAKE, wsb=need - 1) == sv.SV_ERR_WORKSPACE
    assert _chain(L, ws=MISALIGNED, wsb=need) == sv.SV_ERR_WORKSPACE


def test_verify_tree_host_validation(L):
    def call(**kw):
        a = dict(t=FAKE, dt=sv.SV_BF16, tok=FAKE, par=FAKE, cnt=None, B=2, T=26, V=32000,
                 acc=FAKE, path=FAKE, out=FAKE, ws=None, wsb=0)
        a.update(kw)
        return L.sv_verify_tree_greedy(a["t"], a["dt"], a["tok"], a["par"], a["cnt"], a["B"],
                                       a["T"], a["V"],
                                       a["acc"], a["path"], a["out"], None, a["ws"], a["wsb"], None)
    assert call(tok=None) == sv.SV_ERR_INVALID_ARG
    assert call(par=None) == sv.SV_ERR_WORKSPACE  # NULL parents: a chain, valid
    assert call(T=0) == sv.SV_ERR_INVALID_ARG
    assert call(T=1025) == sv.SV_ERR_UNSUPPORTED
    assert call() == sv.SV_ERR_WORKSPACE
    assert call(cnt=FAKE) == sv.SV_ERR_WORKSPACE  # node counts are checked on the device
    need = L.sv_workspace_size(sv.SV_OP_VERIFY_TREE_GREEDY, 2, 26, 32000, sv.SV_BF16, 0, 0, 0)
    assert call(ws=FAKE, wsb=need - 16) == sv.SV_ERR_WORKSPACE


def test_verify_tree_stochastic_host_validation(L):
    def call(**kw):
        a = dict(t=FAKE, d=FAKE, dt=sv.SV_BF16, tok=FAKE, par=FAKE, cnt=None, ua=FAKE, us=FAKE, B=2,
                 T=26, V=32000, acc=FAKE, path=FAKE, out=FAKE, ws=None, wsb=0)
        a.update(kw)
        return L.sv_verify_tree_stochastic(a["t"], a["d"], a["dt"], a["tok"], a["par"], a["cnt"],
                                           a["ua"], a["us"], a["B"], a["T"], a["V"], a["acc"],
                                           a["path"], a["out"], None, a["ws"], a["wsb"], None)
    assert call(d=None) == sv.SV_ERR_INVALID_ARG
    assert call(ua=None) == sv.SV_ERR_INVALID_ARG
    assert call(dt=9) == sv.SV_ERR_INVALID_ARG
    assert call(T=0) == sv.SV_ERR_INVALID_ARG
    assert call(d=MISALIGNED) == sv.SV_ERR_INVALID_ARG
    assert call(T=1025) == sv.SV_ERR_UNSUPPORTED
    assert call(V=(1 << 22) + 1) == sv.SV_ERR_UNSUPPORTED
    assert call(par=None) == sv.SV_ERR_WORKSPACE  # NULL parents: a chain, valid
    assert call(cnt=FAKE) == sv.SV_ERR_WORKSPACE  # node counts are checked on the device
    need = L.sv_workspace_size(sv.SV_OP_VERIFY_TREE_STOCHASTIC, 2, 26, 32000, sv.SV_BF16, 0, 0, 0)
    assert need > 0
    assert call(ws=FAKE, wsb=need - 16) == sv.SV_ERR_WORKSPACE
    assert call(ws=MISALIGNED, wsb=need) == sv.SV_ERR_WORKSPACE


def test_attention_host_validation(L):
    def call(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, pl=FAKE, par=None, cnt=None, B=2, T=9, Hq=32, Hkv=8,
                 D=128, S=4160, scale=0.088, out=FAKE)
        a.update(kw)
        return L.sv_tree_attention(a["q"], a["k"], a["v"], a["pl"], a["par"], a["cnt"], a["B"],
                                   a["T"],
                                   a["Hq"], a["Hkv"], a["D"], a["S"], a["scale"], a["out"], None,
                                   None, 0, None)
    assert call(q=None) == sv.SV_ERR_INVALID_ARG
    assert call(pl=None) == sv.SV_ERR_INVALID_ARG
    assert call(Hq=30) == sv.SV_ERR_INVALID_ARG      # Hq % Hkv
    assert call(S=8) == sv.SV_ERR_INVALID_ARG        # S_max < T
    assert call(scale=0.0) == sv.SV_ERR_INVALID_ARG
    assert call(scale=float("nan")) == sv.SV_ERR_INVALID_ARG
    assert call(k=MISALIGNED) == sv.SV_ERR_INVALID_ARG
    assert call(B=1 << 20, Hkv=8, Hq=32, S=4160) == sv.SV_ERR_UNSUPPORTED  # rows >= 2^31


def test_compact_host_validation(L):
    def call(**kw):
        a = dict(k=FAKE, v=FAKE, pl=FAKE, nl=FAKE, path=None, stride=0, acc=FAKE, B=2, Hkv=8,
                 D=128, S=4160)
        a.update(kw)
        return L.sv_compact_kv(a["k"], a["v"], a["pl"], a["nl"], a["path"], a["stride"], a["acc"],
                               a["B"], a["Hkv"], a["D"], a["S"], None, None)
    assert call(acc=None) == sv.SV_ERR_INVALID_ARG
    assert call(path=FAKE, stride=0) == sv.SV_ERR_INVALID_ARG
    assert call(D=100) == sv.SV_ERR_UNSUPPORTED
    assert call(D=512) == sv.SV_ERR_UNSUPPORTED
    assert call(v=MISALIGNED) == sv.SV_ERR_INVALID_ARG


def test_workspace_sizes_scale_with_shape(L):
    a = L.sv_workspace_size(sv.SV_OP_VERIFY_CHAIN, 32, 8, 128256, sv.SV_BF16, 0, 0, 0)
    b = L.sv_workspace_size(sv.SV_OP_VERIFY_CHAIN, 64, 8, 128256, sv.SV_BF16, 0, 0, 0)
    assert 0 < a < b
    assert L.sv_workspace_size(sv.SV_OP_VERIFY_CHAIN, 0, 8, 1000, sv.SV_BF16, 0, 0, 0) == 0
    assert L.sv_workspace_size(sv.SV_OP_VERIFY_CHAIN, 1, 8, 1000, 5, 0, 0, 0) == 0


@pytest.mark.parametrize("op,T,V", [
    (sv.SV_OP_VERIFY_CHAIN, 64, 1000),                   # N > 63
    (sv.SV_OP_VERIFY_CHAIN, 8, 1 << 30),
    (sv.SV_OP_VERIFY_TREE_GREEDY, 1025, 1000),
    (sv.SV_OP_VERIFY_TREE_GREEDY, (1 << 31) - 1, 1000),  # 2T would overflow an int
    (sv.SV_OP_VERIFY_TREE_STOCHASTIC, 1025, 1000),
    (sv.SV_OP_VERIFY_TREE_STOCHASTIC, (1 << 31) - 1, 1000),
    (sv.SV_OP_VERIFY_TREE_STOCHASTIC, 8, (1 << 22) + 1),
])
def test_workspace_size_is_zero_for_unsupported_shapes(L, op, T, V):
    assert L.sv_workspace_size(op, 2, T, V, sv.SV_BF16, 0, 0, 0) == 0
    # the largest supported sizes still get a workspace
    top = {sv.SV_OP_VERIFY_CHAIN: (63, (1 << 30) - 1), sv.SV_OP_VERIFY_TREE_GREEDY: (1024, 1 << 22),
           sv.SV_OP_VERIFY_TREE_STOCHASTIC: (1024, 1 << 22)}[op]
    assert L.sv_workspace_size(op, 1, top[0], top[1], sv.SV_BF16, 0, 0, 0) > 0


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "specverify.h"

int main(void) {
    int32_t acc[2], out[10];
    size_t ws;
    if (sv_version() < 100) return 1;
    if (strncmp(sv_status_string(SV_ERR_BAD_INPUT), "SV_ERR_BAD_INPUT", 16) != 0) return 2;
    ws = sv_workspace_size(SV_OP_VERIFY_TREE_STOCHASTIC, 2, 26, 32000, SV_BF16, 0, 0, 0);
    if (ws == 0 || sv_workspace_size(SV_OP_VERIFY_CHAIN, 0, 4, 1000, SV_BF16, 0, 0, 0) != 0) return 3;
    /* host-side validation answers before any launch: no GPU is needed */
    if (sv_verify_chain(NULL, NULL, SV_BF16, NULL, NULL, NULL, NULL, 2, 4, 1000, acc, out, NULL,
                        NULL, NULL, 0, (sv_stream_t)0) != SV_ERR_INVALID_ARG) return 4;
    if (sv_compact_kv(NULL, NULL, NULL, NULL, NULL, 0, NULL, 1, 1, 128, 16, NULL,
                      (sv_stream_t)0) != SV_ERR_INVALID_ARG) return 5;
    printf("ok %zu\n", ws);
    return 0;
}
"""


def test_plain_c_program_uses_the_header_and_library(L, tmp_path):
    """The header is plain C99 (no C++ and no CUDA headers needed), and a C
    program links against the library and gets the documented answers."""
    import subprocess
    src = tmp_path / "use_api.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "use_api"
    libdir = os.path.dirname(svbuild.LIB_PATH)
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                           f"-I{os.path.dirname(HEADER)}", str(src), f"-L{libdir}", "-lspecverify",
                           f"-Wl,-rpath,{libdir}", "-o", str(exe)])
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.startswith("ok ")


def _step_chain(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, pl=FAKE, Hq=32, Hkv=8, D=128, S=4160, scale=0.088, out=FAKE,
             ast=None, t=FAKE, d=FAKE, dt=sv.SV_BF16, tok=FAKE, lens=None, ua=FAKE, us=FAKE, B=2,
             N=8, V=1000, acc=FAKE, otok=FAKE, probs=None, vst=None, newl=MISALIGNED, ws=None,
             wsb=0)
    a.update(kw)
    return L.sv_verify_step_chain(a["q"], a["k"], a["v"], a["pl"], a["Hq"], a["Hkv"], a["D"],
                                  a["S"], a["scale"], a["out"], a["ast"], a["t"], a["d"], a["dt"],
                                  a["tok"], a["lens"], a["ua"], a["us"], a["B"], a["N"], a["V"],
                                  a["acc"], a["otok"], a["probs"], a["vst"], a["newl"], a["ws"],
                                  a["wsb"], None)


def _step_tree(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, pl=FAKE, par=None, cnt=None, B=2, T=26, Hq=32, Hkv=8, D=128,
             S=2112, scale=0.088, out=FAKE, ast=None, t=FAKE, dt=sv.SV_BF16, tok=FAKE, V=32000,
             acc=FAKE, path=FAKE, otok=FAKE, vst=None, newl=MISALIGNED, ws=None, wsb=0)
    a.update(kw)
    return L.sv_verify_step_tree_greedy(a["q"], a["k"], a["v"], a["pl"], a["par"], a["cnt"],
                                        a["B"], a["T"], a["Hq"], a["Hkv"], a["D"], a["S"],
                                        a["scale"], a["out"], a["ast"], a["t"], a["dt"], a["tok"],
                                        a["V"], a["acc"], a["path"], a["otok"], a["vst"], a["newl"],
                                        a["ws"], a["wsb"], None)


def test_fused_step_host_validation(L):
    """The fused steps refuse, before any launch: NULL or misaligned tensors,
    bad sizes, new lengths written over the prefix lengths the attention is
    reading, and shapes outside the calls' ranges."""
    for call in (_step_chain, _step_tree):
        assert call(L, q=None) == sv.SV_ERR_INVALID_ARG
        assert call(L, newl=None) == sv.SV_ERR_INVALID_ARG
        assert call(L, newl=FAKE) == sv.SV_ERR_INVALID_ARG  # the same pointer as prefix_lens
        assert call(L, q=MISALIGNED) == sv.SV_ERR_INVALID_ARG
        assert call(L, B=0) == sv.SV_ERR_INVALID_ARG
        assert call(L, Hkv=5) == sv.SV_ERR_INVALID_ARG  # Hq % Hkv
        assert call(L, scale=0.0) == sv.SV_ERR_INVALID_ARG
        assert call(L, dt=9) == sv.SV_ERR_INVALID_ARG
    assert _step_chain(L, N=64, S=5000) == sv.SV_ERR_UNSUPPORTED
    assert _step_tree(L, Hq=512, Hkv=512) == sv.SV_ERR_UNSUPPORTED


@pytest.mark.gpu
def test_fused_step_workspace_sizes(L):
    """A fused step's workspace holds its attention's and its acceptance's
    (attention sizes follow the device's SM count: a GPU is needed)."""
    bf = sv.SV_BF16
    a = L.sv_workspace_size(sv.SV_OP_TREE_ATTENTION, 32, 9, 0, bf, 32, 8, 128)
    c = L.sv_workspace_size(sv.SV_OP_VERIFY_CHAIN, 32, 8, 128256, bf, 0, 0, 0)
    s = L.sv_workspace_size(sv.SV_OP_VERIFY_STEP_CHAIN, 32, 8, 128256, bf, 32, 8, 128)
    assert a > 0 and c > 0 and s >= a + c
    a = L.sv_workspace_size(sv.SV_OP_TREE_ATTENTION, 4, 26, 0, bf, 32, 8, 128)
    g = L.sv_workspace_size(sv.SV_OP_VERIFY_TREE_GREEDY, 4, 26, 32000, bf, 0, 0, 0)
    s = L.sv_workspace_size(sv.SV_OP_VERIFY_STEP_TREE_GREEDY, 4, 26, 32000, bf, 32, 8, 128)
    assert s >= a + g + 4 * 8 * 4
    assert L.sv_workspace_size(sv.SV_OP_VERIFY_STEP_CHAIN, 32, 8, 128256, bf, 32, 5, 128) == 0
    assert L.sv_workspace_size(sv.SV_OP_VERIFY_STEP_TREE_GREEDY, 4, 65, 32000, bf, 32, 8, 128) == 0
