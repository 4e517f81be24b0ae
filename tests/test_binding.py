"""The Python binding's marshalling, on the CPU.  Every wrapper, called with
tensors of the documented shapes, hands the library the call's sizes,
dtype code and pointers; a tensor of another shape is refused before the
library is called (the kernels index every array by the call's sizes).  The
library is replaced by a recorder and the device check by a stub."""
import ctypes
import types

import pytest
import torch

from speculative_decoding_verification_81_gb300 import api


class Recorder:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        if name.startswith("__"):
            raise AttributeError(name)

        def fn(*args):
            self.calls.append((name, args))
            return 0
        return fn


@pytest.fixture
def rec(monkeypatch):
    r = Recorder()
    monkeypatch.setattr(api, "_lib", r)
    monkeypatch.setattr(api, "_on_device", lambda t: True)
    return r


STREAM = types.SimpleNamespace(cuda_stream=0)


def _ws():
    return torch.zeros(256, dtype=torch.uint8)


def _addr(x):
    return x.value if isinstance(x, ctypes.c_void_p) else x


def _i32(*shape):
    return torch.zeros(shape, dtype=torch.int32)


def _bf(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def _f32(*shape):
    return torch.zeros(shape, dtype=torch.float32)


def _refused(rec, fn, **kw):
    n = len(rec.calls)
    with pytest.raises(ValueError):
        fn(**kw)
    assert len(rec.calls) == n


# ---------------------------------------------------------------- attention

def _attn_kw():
    B, T, Hq, Hkv, D, S = 2, 3, 4, 2, 8, 16
    return dict(q=_bf(B, T, Hq, D), k_cache=_bf(B, Hkv, S, D), v_cache=_bf(B, Hkv, S, D),
                prefix_lens=_i32(B), parents=_i32(B, T), out=_bf(B, T, Hq, D), seq_status=_i32(B),
                node_counts=_i32(B), ws=_ws(), stream=STREAM)


def test_tree_attention_marshalling(rec):
    kw = _attn_kw()
    out = api.sv_tree_attention(**kw)
    name, a = rec.calls[-1]
    assert name == "sv_tree_attention" and out is kw["out"]
    assert a[6:12] == (2, 3, 4, 2, 8, 16)                  # B, T, Hq, Hkv, D, S_max
    assert a[12] == pytest.approx(8 ** -0.5)               # default scale 1/sqrt(D)
    ptrs = [_addr(a[i]) for i in (0, 1, 2, 3, 4, 5, 13, 14, 15)]
    assert ptrs == [kw[n].data_ptr() for n in ("q", "k_cache", "v_cache", "prefix_lens", "parents",
                                                 "node_counts", "out", "seq_status", "ws")]
    assert a[16] == 256 and _addr(a[17]) is None


@pytest.mark.parametrize("name,bad", [
    ("v_cache", _bf(2, 2, 17, 8)), ("k_cache", _bf(3, 2, 16, 8)), ("prefix_lens", _i32(3)),
    ("parents", _i32(2, 4)), ("node_counts", _i32(1)), ("out", _bf(2, 3, 4, 4)),
    ("seq_status", _i32(3)),
])
def test_tree_attention_refuses_shapes(rec, name, bad):
    kw = _attn_kw()
    kw[name] = bad
    _refused(rec, api.sv_tree_attention, **kw)


def _paged_kw():
    B, T, Hq, Hkv, D, P, ps, mp = 2, 3, 4, 2, 8, 7, 8, 3
    return dict(q=_bf(B, T, Hq, D), k_pages=_bf(P, Hkv, ps, D), v_pages=_bf(P, Hkv, ps, D),
                block_table=_i32(B, mp), prefix_lens=_i32(B), parents=_i32(B, T),
                out=_bf(B, T, Hq, D), seq_status=_i32(B), node_counts=_i32(B), ws=_ws(),
                stream=STREAM)


def test_paged_attention_marshalling(rec):
    kw = _paged_kw()
    api.sv_tree_attention_paged(**kw)
    name, a = rec.calls[-1]
    assert name == "sv_tree_attention_paged"
    assert a[4:7] == (3, 7, 8)                             # max_pages, num_pages, page_size
    assert a[10:15] == (2, 3, 4, 2, 8)                     # B, T, Hq, Hkv, D
    assert _addr(a[3]) == kw["block_table"].data_ptr() and _addr(a[16]) == kw["out"].data_ptr()


@pytest.mark.parametrize("name,bad", [
    ("v_pages", _bf(8, 2, 8, 8)), ("block_table", _i32(3, 3)), ("prefix_lens", _i32(1)),
    ("parents", _i32(2, 2)), ("out", _bf(2, 3, 4, 16)), ("seq_status", _i32(1)),
])
def test_paged_attention_refuses_shapes(rec, name, bad):
    kw = _paged_kw()
    kw[name] = bad
    _refused(rec, api.sv_tree_attention_paged, **kw)


# ---------------------------------------------------------------- chain

def _chain_kw(dtype=torch.float32):
    B, N, V = 2, 3, 10
    return dict(target_logits=torch.zeros(B, N + 1, V, dtype=dtype),
                draft_logits=torch.zeros(B, N, V, dtype=dtype), draft_tokens=_i32(B, N),
                u_accept=_f32(B, N), u_sample=_f32(B), accepted_len=_i32(B),
                out_tokens=_i32(B, N + 1), probs_out=_f32(B, N, 2), seq_status=_i32(B),
                stream=STREAM)


@pytest.mark.parametrize("dtype,code", [(torch.float32, api.SV_F32), (torch.bfloat16, api.SV_BF16)])
def test_verify_chain_marshalling(rec, dtype, code):
    kw = _chain_kw(dtype)
    acc, out = api.sv_verify_chain(**kw, ws=_ws(), draft_lens=_i32(2))
    name, a = rec.calls[-1]
    assert name == "sv_verify_chain" and a[2] == code and a[7:10] == (2, 3, 10)
    assert acc is kw["accepted_len"] and out is kw["out_tokens"]
    assert _addr(a[12]) == kw["probs_out"].data_ptr()


def test_verify_chain_allocates_outputs(rec):
    kw = _chain_kw()
    for n in ("accepted_len", "out_tokens", "probs_out", "seq_status"):
        kw.pop(n)
    acc, out = api.sv_verify_chain(**kw, ws=_ws())
    assert acc.shape == (2,) and out.shape == (2, 4) and acc.dtype == out.dtype == torch.int32


@pytest.mark.parametrize("name,bad", [
    ("draft_logits", _f32(2, 4, 10)), ("draft_tokens", _i32(2, 4)), ("u_accept", _f32(2, 2)),
    ("u_sample", _f32(3)), ("accepted_len", _i32(3)), ("out_tokens", _i32(2, 3)),
    ("probs_out", _f32(2, 3, 1)), ("seq_status", _i32(1)),
])
def test_verify_chain_refuses_shapes(rec, name, bad):
    kw = _chain_kw()
    kw[name] = bad
    _refused(rec, api.sv_verify_chain, **kw, ws=_ws())
    _refused(rec, api.sv_verify_chain_noalloc, **kw)


def test_verify_chain_refuses_draft_lens_shape(rec):
    _refused(rec, api.sv_verify_chain, **_chain_kw(), ws=_ws(), draft_lens=_i32(3))


def test_verify_chain_noalloc_marshalling(rec):
    kw = _chain_kw()
    api.sv_verify_chain_noalloc(**kw)
    name, a = rec.calls[-1]
    assert name == "sv_verify_chain_noalloc" and a[6:9] == (2, 3, 10)


# ---------------------------------------------------------------- trees

def _tree_kw(stochastic):
    B, T, V = 2, 5, 12
    kw = dict(target_logits=_bf(B, T, V), node_tokens=_i32(B, T), parents=_i32(B, T),
              node_counts=_i32(B), accepted_len=_i32(B), path_nodes=_i32(B, T),
              out_tokens=_i32(B, T), seq_status=_i32(B), ws=_ws(), stream=STREAM)
    if stochastic:
        kw.update(draft_logits=_bf(B, T, V), u_accept=_f32(B, T), u_sample=_f32(B))
    return kw


def test_verify_tree_greedy_marshalling(rec):
    kw = _tree_kw(False)
    api.sv_verify_tree_greedy(**kw)
    name, a = rec.calls[-1]
    assert name == "sv_verify_tree_greedy" and a[1] == api.SV_BF16 and a[5:8] == (2, 5, 12)
    assert [_addr(a[i]) for i in (2, 3, 4, 8, 9, 10, 11)] == [
        kw[n].data_ptr() for n in ("node_tokens", "parents", "node_counts", "accepted_len",
                                   "path_nodes", "out_tokens", "seq_status")]


def test_verify_tree_stochastic_marshalling(rec):
    kw = _tree_kw(True)
    api.sv_verify_tree_stochastic(**kw)
    name, a = rec.calls[-1]
    assert name == "sv_verify_tree_stochastic" and a[2] == api.SV_BF16 and a[8:11] == (2, 5, 12)
    assert [_addr(a[i]) for i in (1, 6, 7)] == [kw[n].data_ptr()
                                                for n in ("draft_logits", "u_accept", "u_sample")]


@pytest.mark.parametrize("stochastic", [False, True])
@pytest.mark.parametrize("name,bad", [
    ("node_tokens", _i32(2, 4)), ("parents", _i32(3, 5)), ("node_counts", _i32(5)),
    ("accepted_len", _i32(1)), ("path_nodes", _i32(2, 6)), ("out_tokens", _i32(2, 4)),
    ("seq_status", _i32(3)),
])
def test_verify_tree_refuses_shapes(rec, stochastic, name, bad):
    kw = _tree_kw(stochastic)
    kw[name] = bad
    fn = api.sv_verify_tree_stochastic if stochastic else api.sv_verify_tree_greedy
    _refused(rec, fn, **kw)


@pytest.mark.parametrize("name,bad", [
    ("draft_logits", _bf(2, 5, 13)), ("u_accept", _f32(2, 4)), ("u_sample", _f32(1)),
])
def test_verify_tree_stochastic_refuses_shapes(rec, name, bad):
    kw = _tree_kw(True)
    kw[name] = bad
    _refused(rec, api.sv_verify_tree_stochastic, **kw)


# ---------------------------------------------------------------- compaction

def _compact_kw():
    B, Hkv, S, D = 3, 2, 20, 8
    return dict(k_cache=_bf(B, Hkv, S, D), v_cache=_bf(B, Hkv, S, D), prefix_lens=_i32(B),
                accepted_len=_i32(B), path_nodes=_i32(B, 6), new_kv_lens=_i32(B),
                seq_status=_i32(B), stream=STREAM)


def test_compact_kv_marshalling(rec):
    kw = _compact_kw()
    newl = api.sv_compact_kv(**kw)
    name, a = rec.calls[-1]
    assert name == "sv_compact_kv" and newl is kw["new_kv_lens"]
    assert a[5] == 6 and a[7:11] == (3, 2, 8, 20)          # path stride; B, Hkv, D, S_max
    kw["path_nodes"] = None
    api.sv_compact_kv(**kw)
    assert rec.calls[-1][1][5] == 0 and _addr(rec.calls[-1][1][4]) is None


@pytest.mark.parametrize("name,bad", [
    ("v_cache", _bf(3, 2, 21, 8)), ("prefix_lens", _i32(2)), ("accepted_len", _i32(4)),
    ("path_nodes", _i32(2, 6)), ("new_kv_lens", _i32(2)), ("seq_status", _i32(4)),
])
def test_compact_kv_refuses_shapes(rec, name, bad):
    kw = _compact_kw()
    kw[name] = bad
    _refused(rec, api.sv_compact_kv, **kw)


def _compact_paged_kw():
    B, Hkv, D, P, ps, mp = 3, 2, 8, 10, 8, 3
    return dict(k_pages=_bf(P, Hkv, ps, D), v_pages=_bf(P, Hkv, ps, D), block_table=_i32(B, mp),
                prefix_lens=_i32(B), accepted_len=_i32(B), path_nodes=_i32(B, 6),
                new_kv_lens=_i32(B), seq_status=_i32(B), stream=STREAM)


def test_compact_kv_paged_marshalling(rec):
    kw = _compact_paged_kw()
    api.sv_compact_kv_paged(**kw)
    name, a = rec.calls[-1]
    assert name == "sv_compact_kv_paged"
    assert a[3:6] == (3, 10, 8) and a[9] == 6 and a[11:14] == (3, 2, 8)


@pytest.mark.parametrize("name,bad", [
    ("v_pages", _bf(10, 2, 16, 8)), ("prefix_lens", _i32(4)), ("accepted_len", _i32(2)),
    ("path_nodes", _i32(4, 6)), ("new_kv_lens", _i32(1)),
])
def test_compact_kv_paged_refuses_shapes(rec, name, bad):
    kw = _compact_paged_kw()
    kw[name] = bad
    _refused(rec, api.sv_compact_kv_paged, **kw)


def test_library_status_becomes_an_exception(monkeypatch, rec):
    monkeypatch.setattr(Recorder, "__getattr__", lambda self, n: (lambda *a: api.SV_ERR_WORKSPACE))
    monkeypatch.setattr(api, "status_string", lambda s: f"status {s}")
    with pytest.raises(api.SpecVerifyError) as e:
        api.sv_compact_kv(**_compact_kw())
    assert e.value.status == api.SV_ERR_WORKSPACE
