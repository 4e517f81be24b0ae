"""Phase timeline of the verification attention kernel (a diagnostic tool).

Builds the library a second time with -DSV_PHASE_STAMPS (into _build/phases/,
beside the product library, which stays stamp-free), runs one attention
shape through it and prints, for each stamped point of a CTA's run, the
spread over the CTAs of its globaltimer reading, in microseconds from the
moment the kernel was allowed to start (the earliest return from the wait
for the previous kernel).

    python -m speculative_decoding_verification_81_gb300.phases [--shape medusa|chain|small|eagle]
        [--reps N] [--behind N]
    python -m speculative_decoding_verification_81_gb300.phases --step chain|medusa|eagle
        [--side-ctas N]

--behind N: the stamped launch is the last of N + 1 calls in one CUDA graph,
as in a stream of steps; its CTAs may be placed while the call before it
still runs.  --copies C: the calls cycle through C input sets, so that with
enough of them (C * the inputs' bytes > 3 x L2) each call reads its K/V from
HBM rather than from L2.
"""
from __future__ import annotations

import argparse
import ctypes
import os

import numpy as np

from . import build as _build

PHASES_DIR = os.path.join(_build.BUILD_DIR, "phases")
PHASES_LIB = os.path.join(PHASES_DIR, "libspecverify_phases.so")
SLOTS = 32
# slot 0: globaltimer at CTA entry; slot 1: the SM clock there; the others:
# the SM clock at the point (slot 17: tiles the CTA processed)
POINTS = [
    (1, "CTA entry (placed on its SM)"),
    (2, "wait for the previous kernel returned"),
    (3, "prologue + unit range done"),
    (4, "K producer: cursor ready"),
    (5, "first Q rows requested"),
    (6, "first K tile requested"),
    (18, "first V tile requested"),
    (7, "first K tile landed (S lane)"),
    (8, "first S product ready (softmax warp)"),
    (19, "first V tile landed (PV lane)"),
    (9, "last S product ready (softmax warp)"),
    (10, "last K tile requested"),
    (11, "last PV product done (segment end)"),
    (12, "O staged / written out"),
    (13, "cluster barrier 1 passed"),
    (20, "cluster merge done (stamped build: once more)"),
    (21, "cluster merge done a second time (warm code)"),
    (15, "cluster merge done"),
    (16, "CTA end (thread 0)"),
    (22, "CTA end (its last warp)"),
]

def step_timeline(args):
    """The kernels of one fused step on a time line: for the attention, its
    CTAs' first entry, first return from the wait for the previous kernel and
    last end; for the acceptance's kernels, their first start and last end.
    The step is the only node of its graph, replayed once after a warm one;
    the inputs are cycled (3 x L2) as in the bench."""
    import torch

    from . import api
    from . import workloads as W

    if args.side_ctas:
        os.environ["SV_STEP_SIDE_CTAS"] = str(args.side_ctas)
    L_ = api.use_library(build_phases_lib())
    for fn in ("sv_debug_attention_stamps", "sv_debug_vocab_spans"):
        getattr(L_, fn).restype = ctypes.c_int
    L_.sv_debug_attention_stamps.argtypes = [ctypes.c_void_p, ctypes.c_int]
    L_.sv_debug_vocab_spans.argtypes = [ctypes.c_void_p]
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(9)
    Hq, Hkv, D = 32, 8, 128
    if args.step == "chain":
        cfg = W.WORKLOADS[4]
        B, L, T, V = cfg["B"], cfg["L"], cfg["N"] + 1, cfg["V"]
    else:
        cfg = W.WORKLOADS[3 if args.step == "medusa" else 5]
        B, L, T, V = cfg["B"], cfg["L"], cfg["T"], cfg["V"]
    S = L + 64
    rows = (2 * T - 1) if args.step == "chain" else T
    one = B * Hkv * S * D * 4 + B * rows * V * 2
    copies = max(1, -(-3 * 126 * 2**20 // one))
    sets = []
    for _ in range(copies):
        x = dict(q=torch.randn(B, T, Hq, D, device=dev, generator=g).to(torch.bfloat16),
                 k=torch.randn(B, Hkv, S, D, device=dev, generator=g).to(torch.bfloat16),
                 v=torch.randn(B, Hkv, S, D, device=dev, generator=g).to(torch.bfloat16),
                 t=(torch.randn(B, T, V, device=dev, generator=g) * 3).to(torch.bfloat16))
        if args.step == "chain":
            x["d"] = (x["t"][:, :T - 1].float() + torch.randn(B, T - 1, V, device=dev,
                                                               generator=g)).to(torch.bfloat16)
            x["tok"] = torch.randint(0, V, (B, T - 1), device=dev, generator=g, dtype=torch.int32)
        else:
            x["tok"] = torch.randint(0, V, (B, T), device=dev, generator=g, dtype=torch.int32)
        sets.append(x)
    pl = torch.full((B,), L, dtype=torch.int32, device=dev)
    newl = torch.empty_like(pl)
    ua = torch.rand(B, T, device=dev, generator=g)
    us = torch.rand(B, device=dev, generator=g)
    if args.step == "medusa":
        par = torch.from_numpy(np.broadcast_to(W.medusa_tree(T), (B, T)).copy()).to(dev)
    elif args.step == "eagle":
        r = np.random.default_rng(5)
        par = torch.from_numpy(np.stack([W.random_tree(T, 8, r) for _ in range(B)])).to(dev)

    def step(i):
        x = sets[i % copies]
        if args.step == "chain":
            api.sv_verify_step_chain(x["q"], x["k"], x["v"], pl, x["t"], x["d"], x["tok"],
                                     ua_c, us,
                                     new_kv_lens=newl)
        else:
            api.sv_verify_step_tree_greedy(x["q"], x["k"], x["v"], pl, par, x["t"], x["tok"],
                                           new_kv_lens=newl)
    ua_c = ua[:, :T - 1].contiguous()
    stream = torch.cuda.current_stream()
    for i in range(copies):
        step(i)
    torch.cuda.synchronize()
    graphs = []
    for i in range(copies):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            step(i)
        graphs.append(gr)
    rows_out = []
    for rep_i in range(args.reps):
        for gr in graphs[:-1]:
            gr.replay()
        torch.cuda.synchronize()
        L_.sv_debug_attention_clear()
        L_.sv_debug_vocab_clear()
        graphs[-1].replay()
        torch.cuda.synchronize()
        buf = np.zeros(1024 * SLOTS, np.int64)
        assert L_.sv_debug_attention_stamps(buf.ctypes.data, 1024) == 0
        raw = buf.reshape(1024, SLOTS)
        raw = raw[raw[:, 0] > 0]
        ghz = args.sm_ghz
        entry = raw[:, 0].astype(np.float64)
        waited = entry + (raw[:, 2] - raw[:, 1]) / ghz
        end = entry + (np.maximum(raw[:, 16], raw[:, 22]) - raw[:, 1]) / ghz
        spans = np.zeros(2 * len(SPAN_NAMES), np.uint64)
        assert L_.sv_debug_vocab_spans(spans.ctypes.data) == 0
        spans = spans.reshape(len(SPAN_NAMES), 2).astype(np.float64)
        t0 = min(entry.min(), spans[spans[:, 1] > 0, 0].min())
        row = {"attention: first CTA entry": entry.min() - t0,
               "attention: first wait return": waited.min() - t0,
               "attention: last CTA end": end.max() - t0}
        names = SPAN_NAMES
        for i, nm in enumerate(names):
            if spans[i, 1] > 0:
                row[f"{nm}: start"] = spans[i, 0] - t0
                row[f"{nm}: end"] = spans[i, 1] - t0
        rows_out.append(row)
    print(f"step {args.step}: B={B} L={L} T={T} V={V}; {copies} input sets; "
          f"side CTAs override {args.side_ctas or 'none'}; median of {args.reps} steps; "
          f"us from the first kernel start")
    for k in rows_out[0]:
        vals = [r[k] for r in rows_out if k in r]
        print(f"{k:44s} {np.median(vals) / 1e3:8.2f}")


# the vocabulary kernels' spans, in the library's order
SPAN_NAMES = ["chain statistics", "chain decisions + residual draw", "tree argmax pass",
              "tree walk (+ compaction)"]

SHAPES = {
    # name: (B, L, T, tree)
    "medusa": (4, 2048, 26, "medusa"),
    "chain": (32, 4096, 9, None),
    "small": (2, 300, 9, None),
    "eagle": (16, 8192, 64, "random"),
}


def build_phases_lib(force: bool = False) -> str:
    return _build.build(force=force, defines=("SV_PHASE_STAMPS",), lib_path=PHASES_LIB,
                        build_dir=PHASES_DIR)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--shape", choices=sorted(SHAPES), default="medusa")
    ap.add_argument("--step", choices=["chain", "medusa", "eagle"], default=None,
                    help="time line of one fused step instead of the attention's phases")
    ap.add_argument("--side-ctas", type=int, default=0,
                    help="chain step: SMs left to the acceptance (default: the library's split)")
    ap.add_argument("--reps", type=int, default=5, help="stamped runs (the table is their median)")
    ap.add_argument("--behind", type=int, default=3)
    ap.add_argument("--sm-ghz", type=float, default=2.07,
                    help="SM clock under load, to turn clock ticks into time")
    ap.add_argument("--copies", type=int, default=0,
                    help="input sets cycled (default: enough for 3 x 126 MB)")
    args = ap.parse_args()
    if args.step:
        step_timeline(args)
        return

    import torch

    from . import api
    from . import workloads as W

    path = build_phases_lib()
    L_ = api.use_library(path)
    L_.sv_debug_attention_stamps.argtypes = [ctypes.c_void_p, ctypes.c_int]
    ghz = args.sm_ghz
    L_.sv_debug_attention_stamps.restype = ctypes.c_int
    L_.sv_debug_attention_clear.restype = ctypes.c_int

    B, L, T, tree = SHAPES[args.shape]
    Hq, Hkv, D = 32, 8, 128
    S = L + 64
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(3)
    one = B * Hkv * S * D * 4 + 2 * B * T * Hq * D * 2
    copies = args.copies or max(1, -(-3 * 126 * 2**20 // one))
    sets = []
    for _ in range(copies):
        q = torch.randn(B, T, Hq, D, device=dev, generator=g).to(torch.bfloat16)
        k = torch.randn(B, Hkv, S, D, device=dev, generator=g).to(torch.bfloat16)
        v = torch.randn(B, Hkv, S, D, device=dev, generator=g).to(torch.bfloat16)
        sets.append((q, k, v, torch.empty_like(q)))
    pl = torch.full((B,), L, dtype=torch.int32, device=dev)
    if tree == "medusa":
        par = torch.from_numpy(np.broadcast_to(W.medusa_tree(T), (B, T)).copy()).to(dev)
    elif tree == "random":  # EAGLE-style trees, as the bench draws them
        rng = np.random.default_rng(5)
        par = torch.from_numpy(np.stack([W.random_tree(T, 8, rng) for _ in range(B)])).to(dev)
    else:
        par = None
    ws = api.workspace(api.SV_OP_TREE_ATTENTION, B, T, Hq=Hq, Hkv=Hkv, D=D, device=dev)

    # every set is read once per replay, the stamped (last) call's set least recently
    ncalls = max(args.behind + 1, copies)

    def call(i=0):
        q, k, v, out = sets[i % copies]
        api.sv_tree_attention(q, k, v, pl, par, out=out, ws=ws)

    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        call()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(ncalls):
            call(i)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()

    ctas = 1024
    runs = []
    for _ in range(args.reps):
        assert L_.sv_debug_attention_clear() == 0
        graph.replay()
        torch.cuda.synchronize()
        buf = np.zeros(ctas * SLOTS, np.int64)
        assert L_.sv_debug_attention_stamps(buf.ctypes.data, ctas) == 0
        raw = buf.reshape(ctas, SLOTS)
        raw = raw[raw[:, 0] > 0]
        # every point on the globaltimer line (ns): entry time + clock ticks since entry
        st = np.zeros(raw.shape, np.float64)
        for slot in range(SLOTS):
            if slot in (0, 17):
                continue
            ok = raw[:, slot] != 0
            st[ok, slot] = raw[ok, 0] + (raw[ok, slot] - raw[ok, 1]) / ghz
        st[:, 17] = raw[:, 17]
        t0 = st[:, 2][st[:, 2] > 0].min()
        runs.append((st, t0))
    n = runs[0][0].shape[0]
    print(f"shape {args.shape}: B={B} L={L} T={T} tree={tree or 'chain'}; {n} CTAs; "
          f"SM clock taken as {ghz} GHz; "
          f"{copies} input sets, the last of {ncalls} calls stamped; median of {args.reps} runs; "
          f"us from the earliest return of the wait for the previous kernel")
    print(f"{'point':44s} {'min':>8s} {'median':>8s} {'max':>8s}")
    for slot, name in POINTS:
        rows = []
        for st, t0 in runs:
            col = st[:, slot]
            col = col[col > 0]
            if col.size == 0:
                continue
            rel = (col - t0) / 1e3
            rows.append((rel.min(), np.median(rel), rel.max()))
        if not rows:
            continue
        a = np.median(np.array(rows), axis=0)
        print(f"{name:44s} {a[0]:8.2f} {a[1]:8.2f} {a[2]:8.2f}")
    tiles = runs[0][0][:, 17]
    print(f"tiles per CTA: min {tiles.min():.0f} max {tiles.max():.0f}")


if __name__ == "__main__":
    main()
